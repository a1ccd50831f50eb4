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
//   * clusters of S <= 4 CTAs take adjacent feature tiles of the same row
//     tile; each copies 1/S of every stage's activation boxes and multicasts
//     them to all S, so L2 serves fewer bytes per MMA (the copies, not the
//     tensor pipe, were the limit with one CTA per unit);
//   * weights tiled at 128 rows pair two tiles into one 256-wide unit.
// Epilogues: QKV (RoPE, KV append through the block table), SwiGLU,
// residual add and logits, four features at a time (epi_quad, shared with
// the 64-row-tile kernel).  A step that may route a GEMM here runs the
// RMSNorm as its own kernel: folding it into these epilogues (the residual
// epilogue writing x * g and partial sums of x^2, the consumers scaling by
// 1/rms) measured no faster, the heavier residual epilogue costing what the
// norm launches saved.
#include <algorithm>
#include <mutex>

#include "gemm_epi.cuh"

namespace cbd {

constexpr int kRwRows = 128;                        // activation rows per tile (MMA M)
constexpr int kRwBK = 64;                           // k per stage (one 128-byte swizzle row)
constexpr int kRwABytes = kRwRows * kRwBK * 2;      // 16 KB: the hi (or lo) tile of one stage
constexpr int kRwRing = 192 * 1024;
constexpr int kRwSmem = kRwRing + 1024;
constexpr int kRwEpiWarps = 8;
constexpr int kRwThreads = 64 + 32 * kRwEpiWarps;
constexpr int kRwMaxStages = 8;

constexpr int kRwMaxCluster = 4;

struct RwArgs {
  int n, KB, NRT;                                   // rows, k blocks, row tiles
  int S;                                            // cluster size: CTAs that share each A tile
  int units;                                        // cluster units = (T / S) * NRT
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
  // Cluster units (feature tiles S tq .. S tq + S - 1, row tile rt) go to
  // clusters round-robin; rank r of the cluster owns feature tile S tq + r.
  // The S CTAs of a cluster work on the same row tile in lockstep, so each
  // issues 1/S of every stage's activation boxes and multicasts them to all.
  const int S = a.S;
  const int rank = S > 1 ? (int)cluster_rank() : 0;
  const int cl = (int)blockIdx.x / S, ncl = (int)gridDim.x / S;
  const int nu = (a.units - cl + ncl - 1) / ncl;
  const int KB = a.KB;
  const uint16_t cmask = (uint16_t)((1u << S) - 1u);
  auto tile_of = [&](int i, int& t, int& rt) {
    const int cu = cl + i * ncl;
    const int tq = cu / a.NRT;
    rt = cu - tq * a.NRT;
    t = tq * S + rank;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], (uint32_t)S);     // every CTA of the cluster frees it
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
  if (S > 1) cluster_sync_all();        // peers' barriers are initialised before any multicast
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
        const int nbox = (min(kRwRows, a.n - rt * kRwRows) + 15) / 16;
        tc::mbar_arrive_expect_tx(&full_bar[s], w_bytes + 2u * nbox * 2048u);
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
        const int nbox = (min(kRwRows, a.n - rt * kRwRows) + 15) / 16;
        uint8_t* st = ring + (size_t)s * stage_bytes + w_bytes;
        if (S == 1) {
          for (int j = 0; j < nbox; ++j) {
            tc::tma_load_2d(st + j * 2048, &tmH, q * kRwBK, rt * kRwRows + j * 16, &full_bar[s]);
            tc::tma_load_2d(st + kRwABytes + j * 2048, &tmL, q * kRwBK, rt * kRwRows + j * 16, &full_bar[s]);
          }
        } else {
          // box j of the 2 nbox (hi boxes, then lo boxes) comes from rank j % S
          for (int j = rank; j < 2 * nbox; j += S) {
            const bool lo = j >= nbox;
            const int jb = lo ? j - nbox : j;
            tc::tma_load_2d_mc(st + (lo ? kRwABytes : 0) + jb * 2048, lo ? &tmL : &tmH, q * kRwBK,
                               rt * kRwRows + jb * 16, &full_bar[s], cmask);
          }
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
          if (S == 1) tc::mma_commit(&empty_bar[s]);
          else tc::mma_commit_mc(&empty_bar[s], cmask);   // the stage's boxes came from every CTA
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
  // no CTA leaves while a peer may still multicast into it or arrive on its
  // barriers (every CTA's MMAs, hence its commits, are complete here)
  if (S > 1) cluster_sync_all();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kCols);
  }
}

// ---------------------------------------------------------------- host side
// Clusters of S CTAs (one per SM) that can be resident at once, S = 1, 2, 4.
static int max_clusters(int S) {
  static int cache[kRwMaxCluster + 1] = {0};
  static std::once_flag once;
  std::call_once(once, [] {
    for (auto k : {gemm_rows_kernel<256, 1>, gemm_rows_kernel<224, 1>, gemm_rows_kernel<192, 1>,
                   gemm_rows_kernel<160, 1>, gemm_rows_kernel<128, 1>, gemm_rows_kernel<256, 2>})
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kRwSmem);
    for (int c = 1; c <= kRwMaxCluster; c *= 2) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c * 64);
      cfg.blockDim = dim3(kRwThreads);
      cfg.dynamicSmemBytes = kRwSmem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = c;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_rows_kernel<256, 1>, &cfg) != cudaSuccess) n = 0;
      cache[c] = n;
    }
    cudaGetLastError();
  });
  return cache[S];
}

// Cluster size for a GEMM of T feature tiles: the largest (<= 4) that
// divides T and can be resident.
static int rows_cluster(int T) {
  for (int c = kRwMaxCluster; c > 1; c /= 2)
    if (T % c == 0 && max_clusters(c) > 0) return c;
  return 1;
}

// Weight tiles per unit: 128-row tiles pair up into 256-wide units.
static int rows_tp(const TcGemm& g) { return g.N == 128 && g.M % 256 == 0 ? 2 : 1; }

bool gemm_rows_preferred(const TcGemm& g, int n) {
  if (g.N <= 0 || g.M % g.N || g.K % kRwBK) return false;
  const int T = g.M / (g.N * rows_tp(g)), S = rows_cluster(T);
  const long long units = (long long)(T / S) * ((n + kRwRows - 1) / kRwRows);
  const int resident = max_clusters(S);
  if (resident <= 0) return false;
  // whole units per cluster: a last wave that is mostly empty makes this
  // kernel slower than the 64-row-tile kernel (which splits K to fill SMs).
  // Measured (7B, 544 rows): O and down with 20 units for 36 resident
  // clusters still ran faster here (2.06 vs 2.24, 5.64 vs 6.49 ms per step).
  const long long waves = (units + resident - 1) / resident;
  return (double)units / (double)(waves * resident) >= 0.5;
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
  a.S = rows_cluster(T);
  a.units = (T / a.S) * a.NRT;
  a.err = ep.err;
  const int resident = max_clusters(a.S);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.S * std::min(a.units, resident)));
  cfg.blockDim = dim3(kRwThreads);
  cfg.dynamicSmemBytes = kRwSmem;
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
