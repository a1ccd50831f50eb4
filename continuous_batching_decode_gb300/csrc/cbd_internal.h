// Internal declarations shared by the libcbd translation units.
#pragma once

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "../../include/cbd.h"

#include <cuda.h>
#include <cuda_runtime.h>

namespace cbd {

// Thread-local message of the last failure; returns `code`.
cbd_status fail(cbd_status code, const char* fmt, ...);
void clear_error();

// One-time set-up per CUDA device (kernel attributes, occupancy queries):
// run(fn) calls fn(device) for the current device until it succeeds once,
// under a mutex, so two host threads launching first at once, or engines on
// several devices of one process, each see a finished set-up; *dev receives
// the current device ordinal.  Later calls cost one cudaGetDevice and one
// atomic load.
constexpr int kMaxDevices = 64;
class DeviceOnce {
 public:
  template <class F>
  cudaError_t run(F&& fn, int* dev = nullptr) {
    int d = 0;
    cudaError_t ce = cudaGetDevice(&d);
    if (ce != cudaSuccess) return ce;
    if (d < 0 || d >= kMaxDevices) return cudaErrorInvalidDevice;
    if (dev) *dev = d;
    if (done_[d].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lk(mu_);
    if (done_[d].load(std::memory_order_relaxed)) return cudaSuccess;
    ce = fn(d);
    if (ce == cudaSuccess) done_[d].store(true, std::memory_order_release);
    return ce;
  }

 private:
  std::mutex mu_;
  std::atomic<bool> done_[kMaxDevices] = {};
};

// Makes `dev` the calling thread's current device for the guard's lifetime
// (entry points that enqueue work for an engine of another device than the
// current one); ok() is false if the switch failed.
class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) { ok_ = false; prev_ = -1; return; }
    if (prev_ != dev) ok_ = cudaSetDevice(dev) == cudaSuccess;
    else prev_ = -1;
  }
  ~DeviceGuard() {
    if (prev_ >= 0) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;

 private:
  int prev_ = -1;
  bool ok_ = true;
};

// Sets a kernel's dynamic shared-memory limit once per device.
template <class K>
inline cudaError_t set_smem_once(DeviceOnce& once, K kernel, int bytes) {
  return once.run([&](int) { return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes); });
}

constexpr int kBlock = 32;          // positions per KV block
constexpr int kAttnChunk = 128;     // positions per attention split (4 blocks)
constexpr int kMaxVocab = 65536;

// Device error codes written to the engine's error word (first one wins).
enum DeviceError : int32_t {
  kDevOk = 0,
  kDevBadRow = 1,        // a row index or position outside the staged tables
  kDevBadBlock = 2,      // a block id outside the pool
  kDevWaitTimeout = 3,   // a bounded wait gave up
  kDevSampler = 4,       // sampler found no token (should not happen)
};

// Per-step row record as the kernels read it.
struct RowDev {
  int32_t slot, token, pos, flags;   // flags: bit0 prefill, bit1 sample
};

// Sampling parameters as the sampler kernel reads them.
struct SampDev {
  float temperature, top_p, presence, frequency, decay;
  int32_t top_k;
  uint32_t seed_lo, seed_hi, req_lo, req_hi, token_index;
  float uniform;                     // >= 0: use it; < 0: draw with Philox
};

// One attention work item: a row's chunk of positions [start, end) (at
// most kAttnChunk), its index wi among the step's chunks (a row's chunks are
// consecutive, chunk c at wi = first + c) and the row's chunk count packed
// as wn = wi << 16 | nch, and the physical KV blocks of the chunk (-1 past
// its end), resolved through the block table on the host.  The list is
// stored largest chunk first, so dynamically scheduled warps finish on the
// smallest ones.
struct AttnWork {
  int32_t row, start, end, wn;
  int32_t blk[kAttnChunk / kBlock];
};
static_assert(sizeof(AttnWork) == 32, "two 16-byte loads per record");

// A block of prompt rows for the prefill attention kernel: positions
// pos0 .. pos0 + npos - 1 of `slot`, held by the step's rows
// pf_rows[idx0 .. idx0 + npos - 1] (in position order).
struct PfBlock {
  int32_t idx0, npos, pos0, slot;
};
// runs of at least this many consecutive positions of one slot (wherever
// their rows sit in the step) go to the prefill attention kernel
constexpr int kPfMinRun = 16;

struct LayerDev {
  const float* attn_norm;            // [d] fp32
  const float* ffn_norm;             // [d] fp32
  const uint16_t* w_qkv;             // [(Hq+2Hkv)*hd][d], q/k rows rope-interleaved (bf16 engines)
  const uint16_t* w_o;               // [d][Hq*hd]
  const uint16_t* w_gu;              // [2F][d], rows (gate_i, up_i) interleaved
  const uint16_t* w_down;            // [d][F]
  // int8 engines (cbd_config.weights_int8): the same matrices, same row
  // orders and tiling, one signed byte per weight, and per-row fp32 scales
  const uint8_t* q_qkv;
  const uint8_t* q_o;
  const uint8_t* q_gu;
  const uint8_t* q_down;
  const float* s_qkv;
  const float* s_o;
  const float* s_gu;
  const float* s_down;
};

// One weight matrix as the tcgen05 GEMM sees it: tensor maps of the
// weights and of the hi / lo activation matrices it multiplies.
struct TcGemm {
  const CUtensorMap* w;
  const CUtensorMap* hi;
  const CUtensorMap* lo;
  int M, K;
  int N;                  // weight rows per tile (the weights' tiling)
  const float* scale;     // int8 weights: per-row scales (null: bf16 weights)
  const uint8_t* w8;      // int8 weights: the tiled bytes (tile (t, kb) is one N x 64-byte run)
};
// Pre-tiled weights: with a tile width of N rows (chosen per matrix), tile
// (t, kb) -- N output features x 64 k -- is one contiguous N * 128-byte run
// at byte offset (t * KB + kb) * N * 128; element (r, k) sits at
// ((r / N) * KB + k / 64) * N * 64 + (r % N) * 64 + k % 64.
__host__ __device__ inline size_t tiled_off(int r, int k, int N, int KB) {
  return ((size_t)(r / N) * KB + (k >> 6)) * (size_t)N * 64 + (size_t)(r % N) * 64 + (k & 63);
}

// L2 prefetch of an upcoming tcgen05 GEMM's weights: the first P k-blocks
// of each of its T x S (feature tile, K split) work units, so that HBM keeps
// streaming while a kernel boundary drains and the next kernel starts.  A
// prefetch is only a hint to the cache; it never changes a result.
struct PfSpec {
  const uint8_t* w;          // the GEMM's pre-tiled weights; null: nothing
  int32_t N, T, KB, S, P;    // tile width, tiles, k-blocks, K split, k-blocks per unit to fetch
};

// A GEMM of the step: weights W [M][K] times activations (hi + lo) [n][lda].
struct GemmOp {
  const uint16_t* W;
  int M, K;
  const uint16_t* a_hi;
  const uint16_t* a_lo;
  int lda;
  TcGemm tc;
};

struct Dims {
  int L, d, hq, hkv, hd, F, V, qkv_out, max_rows, max_slots, max_blocks_per_seq;
  float rope_base, eps;
};

}  // namespace cbd

struct cbd_engine {
  cbd::Dims dm{};
  cbd_config cfg{};
  int device = 0;
  int sm_count = 0;
  // weights
  void* arena = nullptr;
  size_t arena_bytes = 0;
  std::vector<cbd::LayerDev> layers;
  const uint16_t* embed = nullptr;
  const uint16_t* lm_head = nullptr;
  bool w_int8 = false;                // streamed matrices stored as int8 + per-row scales
  const uint8_t* lm_q = nullptr;      // int8 LM head (tiled) and its scales
  const float* lm_scale = nullptr;
  const float* final_norm = nullptr;
  const float* rope_cs = nullptr;     // [max_pos][hd/2][2] fp32 (cos, sin)
  int max_pos = 0;
  // activations / workspaces
  void* work = nullptr;
  size_t work_bytes = 0;
  float* x = nullptr;                 // [max_rows][d] residual
  uint16_t* act_hi = nullptr;         // [max_rows][max(d, Hq*hd)] bf16
  uint16_t* act_lo = nullptr;
  uint16_t* norm_hi = nullptr;        // [max_rows][d] bf16 split(x * g): fused-RMSNorm GEMM input
  uint16_t* norm_lo = nullptr;
  float* ssq = nullptr;               // [max_rows][kMaxSsqParts] partial sums of x^2
  uint16_t* ffn_hi = nullptr;         // [max_rows][F] bf16 SwiGLU output
  uint16_t* ffn_lo = nullptr;
  float* q = nullptr;                 // [max_rows][Hq*hd]
  float* attn_o = nullptr;            // [max_work][Hq][hd] partial outputs
  float* attn_ml = nullptr;           // [max_work][Hq][2] (max, sum)
  int32_t* attn_next = nullptr;       // [L] attention task counters, zeroed at the start of each step
  uint32_t* chain_sync = nullptr;     // [L][kChainMaxPhases] GEMM-chain grid barriers, zeroed with attn_next
  int max_work = 0;
  float* logits = nullptr;            // [max_slots][V] internal logits
  float* samp_scratch = nullptr;      // [max_slots][V] sampler scratch
  float* counters = nullptr;          // [max_slots][V]
  int32_t* last_tok = nullptr;        // [max_slots] the token last sampled for each slot (CBD_TOKEN_LAST)
  uint32_t* forbid = nullptr;         // [ceil(V/32)] bitmap of token ids the sampler never draws
  int32_t n_forbidden = 0;            // ids set in `forbid` (0: mask off)
  int32_t* err = nullptr;             // device error word
  // staging for cbd_step (pinned host + device), double-buffered
  struct Stage {
    void* host = nullptr;
    void* dev = nullptr;
    size_t bytes = 0;
    cudaEvent_t done{};
  } stage[2];
  int stage_idx = 0;
  cbd_batch* step_batch = nullptr;    // batch object reused by cbd_step
  // cbd_step as CUDA graphs (cbd_engine_set_step_graph): per staging buffer,
  // a few graphs keyed by everything their launches bake in
  static constexpr int kStepGraphKey = 14;
  static constexpr size_t kStepGraphCache = 8;
  struct StepGraph {
    uint64_t key[kStepGraphKey];
    cudaGraphExec_t exec;
    uint64_t last_use;
  };
  bool step_graph = false;
  std::vector<StepGraph> step_graphs[2];
  uint64_t step_graph_clock = 0;
  int32_t step_graph_captures = 0;
  // tcgen05 GEMM: tensor maps (built once), partial tiles, counters
  std::vector<CUtensorMap> tmaps;     // per layer: qkv, o, gu, down; then lm_head; then activations
  int tile_qkv = 256, tile_o = 256, tile_gu = 256, tile_dn = 256, tile_lm = 256;   // weight tile widths
  int gemm_path = 0;                  // 0 auto, 1 CUDA-core GEMV, 2 tcgen05
  size_t l2_prefetch = 0;             // bytes of the next GEMM's weights each kernel prefetches to L2 (off)
  bool fuse_norm = true;              // RMSNorm folded into the GEMM epilogues (tcgen05 path)
  bool gemm_chain = false;            // decode: O, gate/up, down and the next QKV as one persistent launch
  int gemv_max_rows = 0;              // auto: GEMV up to this many rows
  int rows_gemm_min = 256;            // tcgen05 path: 128-row-tile kernel from this many rows (0 = never)
  bool rows_gemm_force = false;       // ... for every GEMM of such a step, however it fills the GPU
  int attn_path = 0;                  // 0 tensor cores (mma.sync), 1 CUDA cores
  bool prefill_attn = true;           // path 0, bf16 K/V: prefill runs on the prefill attention kernel
  uint64_t epoch = 1;                 // bumped by every setting that changes the launch sequence
  bool kv_fp8 = false;                // K/V stored as E4M3 bytes (cbd_config.kv_fp8)
  cudaStream_t cap_stream = nullptr;  // private stream for graph capture
  // optional per-launch timing (cbd_engine_profile)
  bool prof = false;
  struct ProfRec { int cls; cudaEvent_t a, b; };
  std::vector<ProfRec> prof_recs;
  std::vector<cudaEvent_t> prof_free;
};

struct cbd_kv_pool {
  cbd_engine* e = nullptr;
  int device = 0;                     // the engine's device
  uint16_t* base = nullptr;           // bf16 elements, or E4M3 bytes when the engine's KV is FP8
  int32_t n_blocks = 0;
  size_t bytes = 0;
};

struct cbd_batch {
  int device = 0;                     // the engine's device
  bool owns_dev = true;
  void* dev = nullptr;                // device copy of everything below
  size_t dev_bytes = 0;
  int32_t n_rows = 0, m = 0, n_work = 0, table_slots = 0, max_chunks = 0;
  int32_t n_dec = 0;                  // work items of rows outside prefill runs (they come first)
  int32_t n_pfb = 0;                  // prefill attention blocks
  // device pointers into `dev`
  cbd::RowDev* rows = nullptr;
  int32_t* sampled_rows = nullptr;    // [m] row index of each sampled row
  int32_t* sampled_slots = nullptr;   // [m]
  cbd::SampDev* samp = nullptr;       // [m]
  int32_t* tables = nullptr;          // [table_slots][max_blocks_per_seq]
  cbd::AttnWork* work = nullptr;      // [n_work]: rows outside prefill runs, then rows inside
  cbd::PfBlock* pfb = nullptr;        // [n_pfb], longest context first
  int32_t* pf_rows = nullptr;         // rows of the prefill runs, by slot and position
  // rows whose chunk partials the merge kernel combines (more than one
  // chunk): those outside prefill runs first (n_comb_dec), then the rest
  int32_t* comb_rows = nullptr;
  int32_t n_comb_dec = 0, n_comb_all = 0;
  int32_t* row_work = nullptr;        // [n_rows + 1] prefix: first work item of each row
  int32_t launches = 0;
  // CUDA graph of one run's launch sequence (cbd_batch_set_graph)
  bool graph_on = false;
  cudaGraphExec_t exec = nullptr;
  uint64_t g_epoch = 0;               // engine settings epoch the graph was captured under
  const void* g_pool = nullptr;
  const void* g_tok = nullptr;
  const void* g_lg = nullptr;
  int32_t captures = 0;
};

namespace cbd {

// Host-side builder: validates a step's inputs and lays out the staging
// image (host buffer `img`) with its offsets.  Returns CBD_OK or CBD_EINVAL.
struct BatchImage {
  std::vector<uint8_t> bytes;
  size_t off_rows, off_sr, off_ss, off_samp, off_tables, off_work, off_row_work, off_pfb, off_pf_rows, off_comb;
  int32_t n_rows, m, n_work, table_slots, max_chunks, n_dec, n_pfb, n_comb_dec, n_comb_all;
};
cbd_status build_batch_image(const cbd_engine* e, const cbd_kv_pool* pool, const cbd_row* rows,
                             int32_t n_rows, const int32_t* tables, int32_t table_slots,
                             const int32_t* nbps, const cbd_sampling* sp, const float* uniforms,
                             BatchImage* img);
void bind_batch(cbd_batch* b, const BatchImage& img, void* dev);

#ifdef __CUDACC__
// Launch with programmatic stream serialisation (the kernel may start while
// the previous kernel on the stream finishes; it synchronises with
// griddepcontrol.wait).
template <typename... P, typename... A>
inline cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}
// Kernel launchers (stream-ordered).  Each returns cudaGetLastError().
// Embedding gather; with fused RMSNorm (g != null) also writes split(x * g)
// to norm_hi / norm_lo and each row's sum of x^2 as its single partial.
cudaError_t launch_embed(const cbd_engine* e, const cbd_batch* b, const float* g, cudaStream_t s);
cudaError_t launch_rmsnorm(const cbd_engine* e, const float* x, const float* g, int n_rows,
                           const int32_t* gather, uint16_t* hi, uint16_t* lo, cudaStream_t s);
enum Epilogue : int { kEpiQKV = 0, kEpiResid = 1, kEpiSwiGLU = 2, kEpiLogits = 3, kEpiResidNorm = 4 };
// Fused RMSNorm (tcgen05 path): a residual-norm epilogue writes x += Y and
// also the next norm's input without its 1/rms factor, split(x * g) as hi +
// lo bf16, plus one partial sum of x^2 per row and CTA feature range; the
// GEMM that consumes it multiplies its sums by 1/sqrt(sum of the row's
// partials / d + eps) (RMSNorm(x) W^T = (1/rms) (x * g) W^T).
constexpr int kMaxSsqParts = 256;   // partials per row: feature tiles x K splits of the producing GEMM
struct EpiArgs {
  int kind;
  float* out_f32;            // logits [n][ld]; residual x [n][ld]; q [n][Hq*hd]
  int ld;
  uint16_t* out_hi;          // SwiGLU output split
  uint16_t* out_lo;
  int ld_act;
  // QKV epilogue
  uint16_t* pool;            // layer-0 base of the pool (E4M3 bytes when kv_fp8)
  int kv_fp8;
  int layer, n_blocks, hq, hkv, hd, max_blocks_per_seq, max_pos;
  const float* rope_cs;
  const RowDev* rows;
  const int32_t* tables;
  int32_t* err;
  // residual-norm epilogue (kEpiResidNorm)
  const float* norm_g;       // [d] gain of the next RMSNorm
  uint16_t* norm_hi;         // [n][d] split(x * g)
  uint16_t* norm_lo;
  float* ssq_out;            // [n][kMaxSsqParts] partial sums of x^2
  // consumer of a fused norm: ssq_in != null scales every sum of row r by
  // 1/sqrt(sum(ssq_in[r][0..n_parts_in)) / d_norm + eps)
  const float* ssq_in;
  int n_parts_in, d_norm;
  float eps;
  // int8 weights: every sum of feature f is multiplied by w_scale[f] first
  const float* w_scale;
};
cudaError_t launch_gemv(const uint16_t* W, int M, int K, int N, const uint16_t* a_hi, const uint16_t* a_lo, int lda,
                        int n, const EpiArgs& ep, cudaStream_t s);
cudaError_t launch_gemm_tc(const TcGemm& g, int n, const EpiArgs& ep, const PfSpec& pf, cudaStream_t s);
// The tcgen05 GEMM's work split for M x K weights and n rows, RT row tiles
// of 64 per CTA: feature tiles, row tiles, k-blocks and the cluster (K
// split) size.
void gemm_tc_plan(int M, int K, int N, int n, int RT, int* T, int* NR, int* KB, int* S);
// Row tiles per CTA the tcgen05 GEMM takes for n rows (2 above 64 rows with
// bf16 weights, else 1).
int gemm_tc_row_tiles(int n, bool int8);
// Weight tiles (of N rows) per unit of the tcgen05 GEMM for n rows: 2 for
// 128-row tiles in steps of more than 128 rows (256-wide units), else 1.
// The unit width N * P is what gemm_tc_plan takes.
int gemm_tc_pair(int M, int N, int n, bool int8);
// Tile width (weight rows per tile) for an M x K weight matrix on this GPU.
int gemm_tc_pick_tile(int M, int K);
// Activation matrices (hi / lo bf16 GEMM inputs) are read by the GEMMs in
// boxes of 64 rows x 64 k: one TMA instruction per row tile and half, since
// each tiled copy has a fixed issue cost (on GB300 a 128-row-tile weight
// stream fed by four 16-row boxes per half ran at 4.3 TB/s, by one box at
// 4.9 TB/s).  The buffers hold a multiple of 64 rows so that a box never
// leaves them; rows past a step's last row hold stale values and land in
// accumulator lanes no epilogue reads.
constexpr int kActBoxRows = 64;
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t stride_elems,
                    uint32_t box_rows);
// Tensor map of tiled int8 weights [rows][64] bytes, box 64 x box_rows, no swizzle.
bool make_tmap_i8(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows);
cudaError_t launch_gemm(const cbd_engine* e, const GemmOp& op, int n, const EpiArgs& epi, const PfSpec& pf,
                        cudaStream_t s);
// The L2 prefetch a kernel issues for the GEMM `op` that follows it on n rows
// (nothing when that GEMM takes the CUDA-core path or prefetch is off).
PfSpec next_prefetch(const cbd_engine* e, const GemmOp& op, int n);
// Whether a GEMM of M x K weights on n rows takes the tcgen05 path, and
// its number of (feature tile x K split) units.
bool gemm_uses_tc(const cbd_engine* e, int n);
// the 128-row-tile persistent kernel (k_gemm_rows.cu) runs this step's GEMMs
bool gemm_uses_rows(const cbd_engine* e, int n);
bool gemm_rows_supports(const EpiArgs& ep);
// the 128-row-tile kernel fills the GPU well enough for this GEMM and row count
bool gemm_rows_preferred(const TcGemm& g, int n);
cudaError_t launch_gemm_rows(const TcGemm& g, int n, const EpiArgs& ep, cudaStream_t s);
// Persistent chain of up to kChainMaxPhases decode GEMMs in one launch
// (k_gemm_chain.cu): the phases run in order, separated by grid barriers on
// the counters sync[0 .. n_phases - 2] (zero at launch), each with the
// per-launch kernel's K split and epilogue, so the sums are the same.
// Possible for 1..64 rows, bf16 weights, 128- or 256-row tiles, K splits
// of 1, 2 or 4 and at most as many CTAs as fit on the GPU at once.
constexpr int kChainMaxPhases = 4;
// pf_bytes: weights of each phase after the first prefetched into L2 (spread
// over its CTAs) while the previous phase finishes; 0: none.
bool gemm_chain_possible(const TcGemm* g, int n_phases, int n);
cudaError_t launch_gemm_chain(const TcGemm* g, const EpiArgs* ep, int n_phases, int n, uint32_t* sync,
                              size_t pf_bytes, cudaStream_t s);
int gemm_tc_units(int M, int K, int N, int n, bool int8);
cudaError_t launch_attn_stream_fp8(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                                   int n_items, const PfSpec& pf, cudaStream_t s);
// Prefill attention kernel (k_attn_pf.cu): query positions per block for a
// KV group of G heads, and the launch over b's blocks.
int prefill_block_positions(int G);
cudaError_t launch_attn_prefill(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                                cudaStream_t s);
// kernel launches launch_attention makes for b
int attention_launches(const cbd_engine* e, const cbd_batch* b);
cudaError_t launch_attention(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                             const PfSpec& pf, cudaStream_t s);
cudaError_t launch_sampler(const cbd_engine* e, const float* logits, int m, const int32_t* slots,
                           const SampDev* samp, int32_t* out_tokens, cudaStream_t s);
// One CTA whose bounded mbarrier wait runs out after `limit` cycles and
// records kDevWaitTimeout in `err` (k_misc.cu).
cudaError_t launch_wait_probe(long long limit, int32_t* err, cudaStream_t s);
#endif

}  // namespace cbd
