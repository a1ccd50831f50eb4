// Weight contraction for steps with many rows (prefill chunks: "20.3 服务、
// 批处理与流式" section 20.3.2, chunked prefill shares the step with decode
// rows; "大模型推理为什么需要 Continuous Batching" section 2.2: prefill is
// compute-bound).  Same sums as gemm_tc_kernel -- fp32 accumulation of the
// bf16 weights times the hi + lo bf16 halves of each activation -- laid out
// for throughput instead of for one weight stream:
//   * a tile is 128 activation rows x N weight rows; hi and lo are two MMAs
//     (M = 128) into the same TMEM accumulator, so each TMEM lane already
//     holds a row's full sum and no fold through shared memory is needed;
//   * CTAs are persistent over (feature tile, row tile) units, and two TMEM
//     accumulators alternate: the epilogue warps drain one (TMEM -> registers
//     -> the kind's epilogue -> global) while the MMA warp fills the other,
//     so a unit's epilogue overlaps the next unit's mainloop;
//   * K is not split (there are enough units), so there is no exchange;
//   * every CTA copies its own activation boxes (one CTA per SM, no
//     clusters);
//   * weights tiled at 128 rows pair two tiles into one 256-wide unit, so
//     each activation stage feeds N = 256.
// Epilogues: QKV (RoPE, KV append through the block table), SwiGLU,
// residual add and logits, four features at a time (epi_quad, shared with
// the 64-row-tile kernel).  A step that may route a GEMM here runs the
// RMSNorm as its own kernel: folding it into these epilogues (the residual
// epilogue writing x * g and partial sums of x^2, the consumers scaling by
// 1/rms) measured no faster, the heavier residual epilogue costing what the
// norm launches saved.
#include <algorithm>

#include "gemm_epi.cuh"

namespace cbd {

constexpr int kRwRows = 128;                        // activation rows per tile (MMA M)
constexpr int kRwBK = 64;                           // k per stage (one 128-byte swizzle row)
constexpr int kRwABytes = kRwRows * kRwBK * 2;      // 16 KB: the hi (or lo) tile of one stage
constexpr uint32_t kABox = kActBoxRows * kRwBK * 2;  // 8 KB: one activation box (64 rows x 64 k)
static_assert(kRwRows % kActBoxRows == 0, "whole activation boxes per row tile");
constexpr int kRwRing = 192 * 1024;
constexpr int kRwSmem = kRwRing + 1024;
constexpr int kRwEpiWarps = 8;
constexpr int kRwThreads = 64 + 32 * kRwEpiWarps;
constexpr int kRwMaxStages = 8;

struct RwArgs {
  int n, KB, NRT;                                   // rows, k blocks, row tiles
  int units;                                        // (feature tile, row tile) units = T * NRT
  int32_t* err;
};


template <int N>
__host__ __device__ constexpr int rw_stages() {
  return kRwRing / (N * kRwBK * 2 + 2 * kRwABytes) < kRwMaxStages ? kRwRing / (N * kRwBK * 2 + 2 * kRwABytes)
                                                                    : kRwMaxStages;
}

// Epilogue of one accumulator for one thread: its TMEM lane is tile row
// `row`, its columns [c0, c0 + N/2) of feature tile t.  Four quads (16
// columns) at a time; the global operands of the next four are loaded
// before this four are stored, so the loads' round trips overlap instead of
// queueing behind one another.
template <int KIND, int N>
__device__ __forceinline__ void rw_epilogue(const EpiArgs& ep, uint32_t taddr, int t, int c0, int row, bool valid) {
  constexpr int HALF = N / 2;
  int2 ri[1] = {make_int2(0, 0)};
  if constexpr (KIND == kEpiQKV) {
    if (valid) {
      const RowDev rw = ep.rows[row];
      ri[0] = make_int2(rw.pos, ep.tables[(size_t)rw.slot * ep.max_blocks_per_seq + (rw.pos >> 5)]);
    }
  }
  const int fb = t * N + c0;
  float4 pre[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    pre[j] = valid ? epi_preload<KIND>(ep, row, fb + 4 * j, ri, 0) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
  for (int c = 0; c < HALF; c += 16) {
    float v[16];
    tc::tmem_ld16(taddr + (uint32_t)c, v);
    float4 nxt[4];
    const bool more = valid && c + 16 < HALF;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      nxt[j] = more ? epi_preload<KIND>(ep, row, fb + c + 16 + 4 * j, ri, 0) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        epi_quad<KIND>(ep, row, fb + c + 4 * j, make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]),
                       pre[j], ri, 0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) pre[j] = nxt[j];
  }
}

// N = MMA N: the features of a unit; TP = weight tiles (of N / TP rows, the
// weights' tiling) stacked into its B operand -- two 128-row tiles make one
// 256-wide unit, so each activation stage feeds twice the MMA work.
template <int N, int TP>
__global__ void __launch_bounds__(kRwThreads, 1)
    gemm_rows_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                     const __grid_constant__ CUtensorMap tmL, const RwArgs a, const EpiArgs ep) {
  static_assert(N % 32 == 0 && N >= 64 && N <= 256, "tile width");
  constexpr uint32_t idesc = tc::idesc_bf16(kRwRows, N);
  constexpr int ST = rw_stages<N>();
  static_assert(ST >= 2, "pipeline stages");
  constexpr uint32_t w_bytes = (uint32_t)N * kRwBK * 2;
  constexpr uint32_t stage_bytes = w_bytes + 2 * kRwABytes;      // weights, hi rows, lo rows
  constexpr uint32_t kCols = 512;                                  // two accumulators, 256 columns apart
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kRwMaxStages], empty_bar[kRwMaxStages];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  // units (feature tile t, row tile rt), t-major, go to CTAs round-robin
  const int cta = (int)blockIdx.x, ncta = (int)gridDim.x;
  const int nu = (a.units - cta + ncta - 1) / ncta;
  const int KB = a.KB;
  auto tile_of = [&](int i, int& t, int& rt) {
    const int u = cta + i * ncta;
    t = u / a.NRT;
    rt = u - t * a.NRT;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], kRwEpiWarps);
    }
    tc::mbar_init(&mma_done, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmW);
    tc::prefetch_tmap(&tmH);
    tc::prefetch_tmap(&tmL);
  }
  pdl_trigger();
  if (warp == 1) tc::tmem_alloc(&tmem_base, kCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort_p = &abort_flag;
  if (warp != 0) pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const long long total = (long long)nu * KB;
      // stage g = (unit i, k block q) of this CTA
      auto unit_of = [&](long long g, int& t, int& rt, int& q) {
        const int i = (int)(g / KB);
        q = (int)(g - (long long)i * KB);
        tile_of(i, t, rt);
      };
      auto issue_w = [&](long long g) {
        int t, rt, q;
        unit_of(g, t, rt, q);
        const int s = (int)(g % ST);
        const int nbox = (min(kRwRows, a.n - rt * kRwRows) + kActBoxRows - 1) / kActBoxRows;
        tc::mbar_arrive_expect_tx(&full_bar[s], w_bytes + 2u * nbox * kABox);
        // (no evict-first hint: the NRT units of a feature tile each read it)
        constexpr int NT = N / TP;                  // rows of one weight tile
#pragma unroll
        for (int tp = 0; tp < TP; ++tp)
          tc::tma_load_2d(ring + (size_t)s * stage_bytes + tp * NT * 128, &tmW, 0, ((t * TP + tp) * KB + q) * NT,
                          &full_bar[s]);
      };
      auto issue_a = [&](long long g) {
        int t, rt, q;
        unit_of(g, t, rt, q);
        const int s = (int)(g % ST);
        const int nbox = (min(kRwRows, a.n - rt * kRwRows) + kActBoxRows - 1) / kActBoxRows;
        uint8_t* st = ring + (size_t)s * stage_bytes + w_bytes;
        for (int j = 0; j < nbox; ++j) {
          tc::tma_load_2d(st + j * kABox, &tmH, q * kRwBK, rt * kRwRows + j * kActBoxRows, &full_bar[s]);
          tc::tma_load_2d(st + kRwABytes + j * kABox, &tmL, q * kRwBK, rt * kRwRows + j * kActBoxRows, &full_bar[s]);
        }
      };
      // weights do not depend on the previous kernel: start them first
      const long long npre = total < ST ? total : ST;
      for (long long g = 0; g < npre; ++g) issue_w(g);
      pdl_wait();
      for (long long g = 0; g < npre; ++g) issue_a(g);
      long long g = npre;
      bool ok = true;
      for (; g < total; ++g) {
        const int s = (int)(g % ST);
        if (!tc::mbar_wait(&empty_bar[s], (uint32_t)(((g / ST) & 1) ^ 1), a.err, abort_p)) { ok = false; break; }
        issue_w(g);
        issue_a(g);
      }
      if (!ok) {    // every load issued must land before the CTA exits
        for (long long r = g > ST ? g - ST : 0; r < g; ++r) {
          int no_abort = 0;
          tc::mbar_wait(&full_bar[r % ST], (uint32_t)((r / ST) & 1), nullptr, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      long long g = 0;
      for (int i = 0; i < nu && ok; ++i) {
        const int b = i & 1;
        if (!tc::mbar_wait(&acc_empty[b], (uint32_t)(((i >> 1) & 1) ^ 1), a.err, abort_p)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(b * 256);
        for (int q = 0; q < KB; ++q, ++g) {
          const int s = (int)(g % ST);
          if (!tc::mbar_wait(&full_bar[s], (uint32_t)((g / ST) & 1), a.err, abort_p)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t st = tc::smem_u32(ring + (size_t)s * stage_bytes);
          const uint64_t dW = tc::sdesc_sw128(st);
          const uint64_t dH = tc::sdesc_sw128(st + w_bytes);
          const uint64_t dL = tc::sdesc_sw128(st + w_bytes + kRwABytes);
#pragma unroll
          for (int k = 0; k < kRwBK / 16; ++k) {
            tc::mma_bf16(acc, dH + 2 * k, dW + 2 * k, idesc, (q > 0 || k > 0) ? 1u : 0u);
            tc::mma_bf16(acc, dL + 2 * k, dW + 2 * k, idesc, 1u);
          }
          tc::mma_commit(&empty_bar[s]);
        }
        if (ok) tc::mma_commit(&acc_full[b]);
      }
      // every MMA issued completes before TMEM is released
      tc::mma_commit(&mma_done);
      int no_abort = 0;
      tc::mbar_wait(&mma_done, 0, a.err, &no_abort);
    }
  } else {
    // ------------------------------------------------ epilogue: TMEM lane quarter x column half
    // warp w reads TMEM lanes 32 (w % 4) .. + 31 (tile rows; lane = row) and
    // half of the columns; a warp whose rows are all past n only hands the
    // accumulator back
    const int lq = warp & 3;
    const int c0 = ((warp - 2) >> 2) * (N / 2);
    for (int i = 0; i < nu; ++i) {
      const int b = i & 1;
      int t, rt;
      tile_of(i, t, rt);
      const int row0 = rt * kRwRows + lq * 32;
      const int row = row0 + lane;
      const bool ready = tc::mbar_wait(&acc_full[b], (uint32_t)((i >> 1) & 1), a.err, abort_p);
      __syncwarp();
      tc::tc_fence_after();
      if (ready && row0 < a.n) {
        const uint32_t taddr = tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)(b * 256 + c0);
        const bool valid = row < a.n;
        switch (ep.kind) {
          case kEpiQKV: rw_epilogue<kEpiQKV, N>(ep, taddr, t, c0, row, valid); break;
          case kEpiSwiGLU: rw_epilogue<kEpiSwiGLU, N>(ep, taddr, t, c0, row, valid); break;
          case kEpiResid: rw_epilogue<kEpiResid, N>(ep, taddr, t, c0, row, valid); break;
          default: rw_epilogue<kEpiLogits, N>(ep, taddr, t, c0, row, valid); break;
        }
      }
      // this warp's columns of the accumulator are read: hand it back
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[b]);
      if (!ready) break;
    }
  }
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kCols);
  }
}

// ---------------------------------------------------------------- host side
// CTAs (one per SM) that can be resident at once, on the current device;
// also sets the kernels' shared-memory limit there.  0 if the query fails.
static int max_ctas() {
  static DeviceOnce once;
  static int cache[kMaxDevices] = {0};
  int dev = -1;
  const cudaError_t ce = once.run([](int d) -> cudaError_t {
    for (auto k : {gemm_rows_kernel<256, 1>, gemm_rows_kernel<224, 1>, gemm_rows_kernel<192, 1>,
                   gemm_rows_kernel<160, 1>, gemm_rows_kernel<128, 1>, gemm_rows_kernel<256, 2>}) {
      const cudaError_t e1 = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kRwSmem);
      if (e1 != cudaSuccess) return e1;
    }
    int per_sm = 0, sms = 0;
    cudaError_t e2 = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_rows_kernel<256, 1>, kRwThreads,
                                                                    kRwSmem);
    if (e2 == cudaSuccess) e2 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    if (e2 != cudaSuccess) return e2;
    cache[d] = per_sm * sms;
    return cudaSuccess;
  }, &dev);
  if (ce != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return cache[dev];
}

// Weight tiles per unit: 128-row tiles pair up into 256-wide units.
static int rows_tp(const TcGemm& g) { return g.N == 128 && g.M % 256 == 0 ? 2 : 1; }

bool gemm_rows_preferred(const TcGemm& g, int n) {
  if (g.N <= 0 || g.M % g.N || g.K % kRwBK) return false;
  // matrices tiled 256 rows wide (the 7B shape's QKV and gate/up) stream
  // faster through the 64-row-tile kernel with two row tiles per CTA, which
  // also splits K (GB300, 7B, 2080 rows: gate/up 23.1 vs 28.6 ms, QKV 6.6 vs
  // 7.0 ms per step)
  if (g.N > 128) return false;
  const int T = g.M / (g.N * rows_tp(g));
  const long long units = (long long)T * ((n + kRwRows - 1) / kRwRows);
  const int resident = max_ctas();
  if (resident <= 0) return false;
  // whole units per CTA: a last wave that is mostly empty makes this kernel
  // slower than the 64-row-tile kernel (which splits K to fill SMs and, past
  // 128 rows, pairs these tiles into 256-wide units).  Measured on GB300
  // (7B): 544 rows, 80 units on 152 SMs, 17.66 ms against 16.40 with the
  // other kernel; 1056 and 2080 rows (144 and 272 units) 24.15 / 43.68 ms
  // against 24.65 / 44.90.
  const long long waves = (units + resident - 1) / resident;
  return (double)units / (double)(waves * resident) >= 0.6;
}

bool gemm_rows_supports(const EpiArgs& ep) {
  return (ep.kind == kEpiQKV || ep.kind == kEpiSwiGLU || ep.kind == kEpiResid || ep.kind == kEpiLogits) &&
         ep.ssq_in == nullptr;
}

cudaError_t launch_gemm_rows(const TcGemm& g, int n, const EpiArgs& ep, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (g.M % g.N || g.K % kRwBK || !gemm_rows_supports(ep)) return cudaErrorInvalidValue;
  RwArgs a{};
  a.n = n;
  a.KB = g.K / kRwBK;
  a.NRT = (n + kRwRows - 1) / kRwRows;
  const int TP = rows_tp(g);
  const int T = g.M / (g.N * TP);
  a.units = T * a.NRT;
  a.err = ep.err;
  const int resident = max_ctas();
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(a.units, resident));
  cfg.blockDim = dim3(kRwThreads);
  cfg.dynamicSmemBytes = kRwSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (TP == 2) return cudaLaunchKernelEx(&cfg, gemm_rows_kernel<256, 2>, *g.w, *g.hi, *g.lo, a, ep);
  switch (g.N) {
    case 256: return cudaLaunchKernelEx(&cfg, gemm_rows_kernel<256, 1>, *g.w, *g.hi, *g.lo, a, ep);
    case 224: return cudaLaunchKernelEx(&cfg, gemm_rows_kernel<224, 1>, *g.w, *g.hi, *g.lo, a, ep);
    case 192: return cudaLaunchKernelEx(&cfg, gemm_rows_kernel<192, 1>, *g.w, *g.hi, *g.lo, a, ep);
    case 160: return cudaLaunchKernelEx(&cfg, gemm_rows_kernel<160, 1>, *g.w, *g.hi, *g.lo, a, ep);
    case 128: return cudaLaunchKernelEx(&cfg, gemm_rows_kernel<128, 1>, *g.w, *g.hi, *g.lo, a, ep);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cbd
