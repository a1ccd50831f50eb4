// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMA).
//
//   Y[n][m] = sum_k W[m][k] * (a_hi[n][k] + a_lo[n][k])    (fp32 accumulate)
//
// then one of the shared epilogues (RoPE + paged KV append, residual add,
// SwiGLU, logits).  The decode step reads every weight once for all rows
// ("0.8MB 跑通 Qwen 第 14-1 篇", section 1; "20.3 服务、批处理与流式", section
// 20.3.2: step cost (W + B*A)/beta).
//
// Orientation.  The MMA's A operand is the activation tile -- 64 rows of
// a_hi stacked on the same 64 rows of a_lo (M = 128) -- and its B operand
// is a tile of 256 weight rows (N = 256), K = 16 per instruction.  Each MMA
// instruction costs about the same for any N, so putting 256 weight rows on
// N makes one instruction cover 8 KB of weights; with the weights on M
// (N = row count) the same stream needs 4x the instructions and the tensor
// pipe, not HBM, becomes the limit.  D[row][feature] lands in TMEM lane
// `row` (hi rows 0-63, lo rows 64-127), column `feature`; the epilogue adds
// the hi and lo lanes, which keeps ~16 significant bits of the fp32
// activations (bf16 alone puts 32-layer logits far outside the accuracy
// bound).
//
// Weights are stored pre-tiled, [M/256][K/64][256][64] bf16, so the box a
// pipeline stage loads is one contiguous 32 KB read.
//
// Split-K inside a thread-block cluster.  A cluster of S CTAs owns one
// (256-feature tile, 64-row tile); CTA rank r accumulates k-blocks
// [r*KB/S, (r+1)*KB/S).  Each CTA folds its hi and lo lanes into a 64 x 256
// fp32 partial in its own shared memory; after a cluster barrier, CTA r
// finalises feature pairs [r*128/S, (r+1)*128/S) by reading all S partials
// over distributed shared memory in rank order (fixed, so results do not
// depend on timing) and runs the epilogue.  No partials go to global memory
// and no CTA waits on a flag.
//
// CTA = 6 warps: warp 0 issues TMA loads into a ring of shared-memory
// stages; warp 1 owns TMEM and issues the MMAs (one thread); warps 2-5 read
// the accumulator back (warp w owns TMEM lanes 32*(w%4)..+31) and run the
// epilogue.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tc.cuh"

namespace cbd {

constexpr int kTcBN = 256;          // weight rows per tile (MMA N)
constexpr int kTcRows = 64;         // activation rows per tile (MMA M = 2 x 64: hi, lo)
constexpr int kTcBK = 64;           // k per stage: one 128-byte swizzle row of bf16
constexpr int kTcThreads = 192;
constexpr int kTcStages = 4;
constexpr int kTcWBytes = kTcBN * kTcBK * 2;            // 32 KB
constexpr int kTcABytes = 2 * kTcRows * kTcBK * 2;      // 16 KB (hi rows, then lo rows)
constexpr int kTcStageBytes = kTcWBytes + kTcABytes;
constexpr int kTcPStride = kTcBN + 4;                   // fp32 partial row stride (padded)
constexpr int kTcLoStride = 32 + 4;
constexpr int kTcSmem = kTcStages * kTcStageBytes + 1024;
constexpr int kTcMaxCluster = 8;

struct TcArgs {
  int M, K, n;                       // weight rows, reduction length, activation rows
  int T, NR, KB, S;                  // feature tiles, row tiles, k blocks, cluster size
  int32_t* err;
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 ld_peer_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
// Load 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  float a[16], b[16];
  tc::tmem_ld16(taddr, a);
  tc::tmem_ld16(taddr + 16, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) { v[i] = a[i]; v[16 + i] = b[i]; }
}

// Epilogue for NB (row, feature pair) items: features f, f+1 (f even) of
// row `row` with values a, b.  Same arithmetic as epi_pair / epi_single;
// all global reads of the batch are issued before any is used.
template <int NB>
__device__ __forceinline__ void epi_pairs(const EpiArgs& ep, const int (&row)[NB], const int (&f)[NB],
                                          const bool (&ok)[NB], const float (&a)[NB], const float (&b)[NB]) {
  if (ep.kind == kEpiLogits) {
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (ok[j]) *reinterpret_cast<float2*>(ep.out_f32 + (size_t)row[j] * ep.ld + f[j]) = make_float2(a[j], b[j]);
    return;
  }
  if (ep.kind == kEpiResid) {
    float2 x[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (ok[j]) x[j] = *reinterpret_cast<const float2*>(ep.out_f32 + (size_t)row[j] * ep.ld + f[j]);
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (ok[j])
        *reinterpret_cast<float2*>(ep.out_f32 + (size_t)row[j] * ep.ld + f[j]) = make_float2(x[j].x + a[j], x[j].y + b[j]);
    return;
  }
  if (ep.kind == kEpiSwiGLU) {
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (ok[j]) epi_pair(ep, f[j], row[j], a[j], b[j]);
    return;
  }
  // QKV: row records, then RoPE factors and block ids, then compute + store
  const int hd = ep.hd, half = hd >> 1, nq = ep.hq * hd, nk = ep.hkv * hd;
  int pos[NB], slot[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j)
    if (ok[j]) {
      const RowDev rw = ep.rows[row[j]];
      pos[j] = rw.pos;
      slot[j] = rw.slot;
    }
  int blk[NB];
  float2 cs[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j)
    if (ok[j]) {
      if (f[j] >= nq) blk[j] = ep.tables[(size_t)slot[j] * ep.max_blocks_per_seq + (pos[j] >> 5)];
      if (f[j] < nq + nk) {
        const int i = ((f[j] < nq ? f[j] : f[j] - nq) % hd) >> 1;
        cs[j] = reinterpret_cast<const float2*>(ep.rope_cs)[(size_t)pos[j] * half + i];
      }
    }
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    if (!ok[j]) continue;
    const int fj = f[j];
    if (fj < nq) {
      const int head = fj / hd, i = (fj % hd) >> 1;
      float* qrow = ep.out_f32 + (size_t)row[j] * nq + head * hd;
      qrow[i] = a[j] * cs[j].x - b[j] * cs[j].y;
      qrow[i + half] = b[j] * cs[j].x + a[j] * cs[j].y;
      continue;
    }
    if (blk[j] < 0 || blk[j] >= ep.n_blocks) { set_err(ep.err, kDevBadBlock); continue; }
    if (fj < nq + nk) {
      const int head = (fj - nq) / hd, i = ((fj - nq) % hd) >> 1;
      const size_t t0 = pool_tile(ep.layer, ep.n_blocks, blk[j], ep.hkv, head, 0, hd);
      ep.pool[t0 + tile_elem(pos[j] & 31, i)] = f32_to_bf16(a[j] * cs[j].x - b[j] * cs[j].y);
      ep.pool[t0 + tile_elem(pos[j] & 31, i + half)] = f32_to_bf16(b[j] * cs[j].x + a[j] * cs[j].y);
    } else {
      const int fv = fj - nq - nk, head = fv / hd, jd = fv % hd;
      const size_t o = pool_off(ep.layer, 1, ep.n_blocks, blk[j], ep.hkv, head, hd, pos[j] & 31, jd);
      ep.pool[o] = f32_to_bf16(a[j]);
      ep.pool[o + 1] = f32_to_bf16(b[j]);
    }
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                   const __grid_constant__ CUtensorMap tmL, const TcArgs a, const EpiArgs ep) {
  constexpr uint32_t kIdesc = tc::idesc_bf16(2 * kTcRows, kTcBN);
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kTcStages], empty_bar[kTcStages];
  __shared__ __align__(8) uint64_t accum_full, mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int decision;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  // unit = (feature tile t, row tile nr); the cluster's ranks split K
  const int S = a.S;
  const int rank = S > 1 ? (int)cluster_rank() : 0;
  const int unit = blockIdx.x / S;
  const int nr = unit % a.NR, t = unit / a.NR;
  const int kb0 = rank * a.KB / S, kb1 = (rank + 1) * a.KB / S;
  const int n_it = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    tc::mbar_init(&accum_full, 1);
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
  if (warp == 1) tc::tmem_alloc(&tmem_base, kTcBN);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort_p = &abort_flag;
  if (warp != 0) pdl_wait();          // the producer waits after prefetching weights

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      auto issue_w = [&](int q) {
        const int s = q % kTcStages;
        uint8_t* st = ring + (size_t)s * kTcStageBytes;
        tc::mbar_arrive_expect_tx(&full_bar[s], kTcStageBytes);
        tc::tma_load_2d(st, &tmW, 0, (t * a.KB + kb0 + q) * kTcBN, &full_bar[s]);
      };
      auto issue_a = [&](int q) {
        const int s = q % kTcStages;
        uint8_t* st = ring + (size_t)s * kTcStageBytes + kTcWBytes;
        const int kx = (kb0 + q) * kTcBK;
#pragma unroll
        for (int j = 0; j < kTcRows / 16; ++j) {
          tc::tma_load_2d(st + j * 2048, &tmH, kx, nr * kTcRows + j * 16, &full_bar[s]);
          tc::tma_load_2d(st + kTcABytes / 2 + j * 2048, &tmL, kx, nr * kTcRows + j * 16, &full_bar[s]);
        }
      };
      // weights do not depend on the previous kernel: start streaming them
      // before waiting for it, then add the activations
      const int npre = n_it < kTcStages ? n_it : kTcStages;
      for (int q = 0; q < npre; ++q) issue_w(q);
      pdl_wait();
      for (int q = 0; q < npre; ++q) issue_a(q);
      int q = npre;
      bool ok = true;
      for (; q < n_it; ++q) {
        const int s = q % kTcStages;
        if (!tc::mbar_wait(&empty_bar[s], ((q / kTcStages) & 1) ^ 1, a.err, abort_p)) { ok = false; break; }
        issue_w(q);
        issue_a(q);
      }
      if (!ok) {     // every load issued must land before the CTA exits
        for (int r = q > kTcStages ? q - kTcStages : 0; r < q; ++r) {
          int no_abort = 0;
          tc::mbar_wait(&full_bar[r % kTcStages], (r / kTcStages) & 1, nullptr, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int q = 0; q < n_it; ++q) {
        const int s = q % kTcStages;
        if (!tc::mbar_wait(&full_bar[s], (q / kTcStages) & 1, a.err, abort_p)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t st = tc::smem_u32(ring + (size_t)s * kTcStageBytes);
        const uint64_t dW = tc::sdesc_sw128(st);
        const uint64_t dA = tc::sdesc_sw128(st + kTcWBytes);
#pragma unroll
        for (int k = 0; k < kTcBK / 16; ++k)   // 16 bf16 = 32 bytes along K inside the swizzled rows
          tc::mma_bf16(tmem, dA + 2 * k, dW + 2 * k, kIdesc, (q > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&empty_bar[s]);
      }
      if (ok && n_it > 0) tc::mma_commit(&accum_full);
      // every MMA issued completes before TMEM is released
      tc::mma_commit(&mma_done);
      int no_abort = 0;
      tc::mbar_wait(&mma_done, 0, a.err, &no_abort);
    }
  } else {
    // ------------------------------------------------ epilogue phase 1: fold hi + lo into the partial
    const int lg = warp & 3;                       // TMEM lane group: rows 32*lg..+31
    const int r = lg * 32 + lane;                  // row of the hi|lo tile
    const uint32_t taddr = tmem + ((uint32_t)(lg * 32) << 16);
    float* P = reinterpret_cast<float*>(ring);                                // [64][kTcPStride]
    float* LO = reinterpret_cast<float*>(ring + 64 * kTcPStride * 4);          // [64][kTcLoStride]
    if (n_it > 0) tc::mbar_wait(&accum_full, 0, a.err, abort_p);
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (threadIdx.x == 64) decision = *abort_p || n_it == 0;
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const bool skip = decision != 0;
    tc::tc_fence_after();
#pragma unroll 1
    for (int c0 = 0; c0 < kTcBN; c0 += 32) {
      float v[32];
      if (!skip) {
        tmem_ld32(taddr + c0, v);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
      if (r >= 64) {
        float4* lo = reinterpret_cast<float4*>(LO + (r - 64) * kTcLoStride);
#pragma unroll
        for (int j = 0; j < 8; ++j) lo[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (r < 64) {
        const float4* lo = reinterpret_cast<const float4*>(LO + r * kTcLoStride);
        float4* p = reinterpret_cast<float4*>(P + r * kTcPStride + c0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 l4 = lo[j];
          p[j] = make_float4(v[4 * j] + l4.x, v[4 * j + 1] + l4.y, v[4 * j + 2] + l4.z, v[4 * j + 3] + l4.w);
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }
    tc::tc_fence_before();
  }
  // ------------------------------------------------ cluster: every partial is in shared memory
  __syncwarp();
  if (S > 1) cluster_sync_all();
  else __syncthreads();
  if (warp >= 2) {
    // ------------------------------------------------ epilogue phase 2: reduce over ranks, finish
    const int et = threadIdx.x - 64;                            // 0..127
    const int p0 = rank * (kTcBN / 2) / S, p1 = (rank + 1) * (kTcBN / 2) / S;   // feature pairs
    const int np = p1 - p0;
    const int rows_here = min(kTcRows, a.n - nr * kTcRows);
    const int items = rows_here * np;
    const uint32_t Pbase = tc::smem_u32(ring);
    constexpr int NB = 4;
#pragma unroll 1
    for (int i0 = et; i0 < items; i0 += 128 * NB) {
      int row[NB], f[NB];
      bool ok[NB];
      float va[NB], vb[NB];
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const int it = i0 + j * 128;
        ok[j] = it < items;
        const int i = ok[j] ? it / np : 0, pp = ok[j] ? it - (it / np) * np : 0;
        row[j] = nr * kTcRows + i;
        f[j] = 2 * (p0 + pp);                    // feature within the tile
        va[j] = 0.f;
        vb[j] = 0.f;
      }
#pragma unroll 1
      for (int qr = 0; qr < S; ++qr) {
        float2 pv[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          if (!ok[j]) continue;
          const uint32_t off = (uint32_t)((row[j] - nr * kTcRows) * kTcPStride + f[j]) * 4u;
          pv[j] = S > 1 ? ld_peer_f2(map_peer(Pbase + off, (uint32_t)qr))
                        : *reinterpret_cast<const float2*>(ring + off);
        }
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (ok[j]) { va[j] += pv[j].x; vb[j] += pv[j].y; }
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) f[j] += t * kTcBN;
      epi_pairs<NB>(ep, row, f, ok, va, vb);
    }
  }
  // peers keep their partials alive until every rank has read them
  __syncwarp();
  if (S > 1) cluster_sync_all();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTcBN);
  }
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map of a row-major bf16 matrix [rows][inner] (row stride in
// elements) with a box of box_rows x 64 and the 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t stride_elems,
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {stride_elems * 2};
  cuuint32_t box[2] = {(cuuint32_t)kTcBK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Co-resident clusters of each size (queried once per process).
static int max_clusters(int S) {
  static int cache[kTcMaxCluster + 1] = {0};
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    for (int s = 1; s <= kTcMaxCluster; ++s) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(s * 64);
      cfg.blockDim = dim3(kTcThreads);
      cfg.dynamicSmemBytes = kTcSmem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = s;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel, &cfg) != cudaSuccess) n = 0;
      cache[s] = n;
    }
    cudaGetLastError();
  });
  return cache[S];
}

// Cluster size for U units of KB k-blocks: fewest estimated waves x (k-blocks
// per CTA + a fixed per-CTA cost of ~6 k-blocks).
static int choose_cluster(long long U, int KB) {
  int best = 1;
  double best_cost = 1e30;
  for (int S = 1; S <= kTcMaxCluster; ++S) {
    if (S > KB) break;
    const int C = max_clusters(S);
    if (C <= 0) continue;
    const long long waves = (U + C - 1) / C;
    const double cost = (double)waves * ((double)(KB + S - 1) / S + 6.0);
    if (cost < best_cost - 1e-9) { best_cost = cost; best = S; }
  }
  return best;
}

cudaError_t launch_gemm_tc(const TcGemm& g, int n, const EpiArgs& ep, const TcWork& w, int sm_count,
                           cudaStream_t s) {
  (void)w;
  (void)sm_count;
  if (n <= 0) return cudaSuccess;
  if (g.M % kTcBN || g.K % kTcBK) return cudaErrorInvalidValue;
  TcArgs a{};
  a.M = g.M; a.K = g.K; a.n = n;
  a.T = g.M / kTcBN; a.NR = (n + kTcRows - 1) / kTcRows; a.KB = g.K / kTcBK;
  a.err = ep.err;
  const long long U = (long long)a.T * a.NR;
  a.S = choose_cluster(U, a.KB);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(U * a.S));
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (a.S > 1) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = a.S;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, *g.w, *g.hi, *g.lo, a, ep);
}

}  // namespace cbd
