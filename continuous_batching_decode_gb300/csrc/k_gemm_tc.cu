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
// finalises feature quads [r*64/S, (r+1)*64/S) by reading all S partials
// over distributed shared memory in rank order (fixed, so results do not
// depend on timing) and runs the epilogue.  No partials go to global memory
// and no CTA waits on a flag.
//
// Two row tiles per CTA (RT = 2, bf16 weights, more than 64 rows): a stage
// holds one weight tile and the activation tiles of rows 0-63 and 64-127,
// and each k-step issues two MMAs into two TMEM accumulators (columns 0..N-1
// and N..2N-1), so a weight tile is read once for 128 rows instead of once
// per 64; the hi/lo fold runs in place over both, and phase 2 covers all 128
// rows.  Per row the sums are those of the one-tile kernel with the same K
// split.  In steps of more than 128 rows, weights tiled 128 rows wide run as
// 256-wide units of two tiles (two weight boxes per stage stacked along the
// MMA's N), as the 256-row-tiled matrices do.
//
// CTA = 10 warps: warp 0 issues TMA loads into a ring of shared-memory
// stages; warp 1 owns TMEM and issues the MMAs (one thread); warps 2-9 read
// the accumulator back (warp w owns TMEM lanes 32*(w%4)..+31, warps w and
// w+4 split the columns) and run the epilogue.
//
// Int8 weights (I8; "RWKV Runner Albatross 后端", 边界与后续路线): a stage
// holds the int8 weight tile (N rows x 64 bytes, one contiguous run of the
// tiled layout) and the activation tile.  While the mainloop runs, the eight
// epilogue warps convert each int8 tile into bf16 (exact: every int8 value
// is a bf16 value) in one of two 128-byte-swizzled buffers that the
// unchanged bf16 MMA reads as its B operand; the first two tiles are
// converted before the dependency wait, since weights do not depend on the
// previous kernel.  The per-row scale multiplies each finished sum in the
// epilogue: y = s_f * sum_k q[f][k] * (a_hi + a_lo)[k].
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "gemm_epi.cuh"

namespace cbd {

constexpr int kTcMaxBN = 256;       // weight rows per tile (MMA N) at most; TMEM columns allocated
constexpr int kTcRows = 64;         // activation rows per tile (MMA M = 2 x 64: hi, lo)
constexpr int kTcBK = 64;           // k per stage: one 128-byte swizzle row of bf16
constexpr int kEpiThreads = 256;    // 8 epilogue warps (two per TMEM lane quarter)
constexpr int kTcThreads = 64 + kEpiThreads;
constexpr int kTcABytes = 2 * kTcRows * kTcBK * 2;      // 16 KB (hi rows, then lo rows)
// Pipeline stages: 4 at N = 256 (6 at 128).  A larger ring (224 KB) cost
// ~2% of the step on GB300: shared memory and L1 share 256 KB per SM, and
// the epilogue's residual / RoPE reads hit L1.
constexpr int kTcRing = 4 * (kTcMaxBN * kTcBK * 2 + kTcABytes);
constexpr int kTcMaxStages = 8;
constexpr int kTcSmem = kTcRing + 1024;
constexpr int kTcMaxCluster = 8;

struct TcArgs {
  int M, K, n;                       // weight rows, reduction length, activation rows
  int N;                             // weight rows per unit (MMA N)
  int P;                             // weight tiles per unit (2: two 128-row tiles side by side)
  int T, NR, KB, S;                  // feature units, row tiles, k blocks, cluster size
  int32_t* err;
  const uint8_t* w8;                 // int8 weights: tiled bytes, fetched by 1-D bulk copies
};

__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_peer_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Epilogue phase 2 for one epilogue kind (256 threads, et = 0..255).  CTA
// rank r of the cluster finalises feature quads [r*64/S, (r+1)*64/S) of the
// tile for every row: the S partials are read (over distributed shared
// memory when S > 1) and summed in rank order, then the epilogue runs.
// Item it = (row it / nq, quad it % nq) belongs to thread it % 256.
// A norm consumer (ep.ssq_in) scales each row's sums by rinv[row] first; a
// residual-norm producer collects each quad's sum of x^2 in sq[row][quad]
// and then writes the row's partial for this CTA (quads in order).
template <int KIND, int N, bool I8>
__device__ __forceinline__ void epi_phase2(const EpiArgs& ep, int S, int rank, int t, int nr, int rows_here,
                                           int et, uint32_t Pbase, const int2* rinfo, const float* rinv, float* sq) {
  const int q0 = rank * (N / 4) / S, q1 = (rank + 1) * (N / 4) / S;
  constexpr int PS = N + 4;                    // fp32 partial row stride (padded)
  const int nq = q1 - q0;
  const int items = rows_here * nq;
  const bool scale = ep.ssq_in != nullptr;
  // Rolled loop: this code runs once per CTA, and fetching a larger
  // (unrolled) body while HBM is saturated costs more than it saves.
#pragma unroll 1
  for (int it = et; it < items; it += kEpiThreads) {
    const int i = it / nq;
    const int f = 4 * (q0 + it - i * nq);      // feature within the tile
    const uint32_t off = (uint32_t)(i * PS + f) * 4u;
    const int fg = t * N + f;
    const float4 pre = epi_preload<KIND>(ep, nr * kTcRows + i, fg, rinfo, i);
    float4 acc;
    if (S == 1) {
      acc = ld_shared_f4(Pbase + off);
    } else {
      float4 pv[kTcMaxCluster];
#pragma unroll
      for (int qr = 0; qr < kTcMaxCluster; ++qr)
        if (qr < S) pv[qr] = ld_peer_f4(map_peer(Pbase + off, (uint32_t)qr));
      acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int qr = 0; qr < kTcMaxCluster; ++qr)
        if (qr < S) {
          acc.x += pv[qr].x; acc.y += pv[qr].y;
          acc.z += pv[qr].z; acc.w += pv[qr].w;
        }
    }
    if constexpr (I8) {
      const float4 ws = *reinterpret_cast<const float4*>(ep.w_scale + fg);
      acc.x *= ws.x; acc.y *= ws.y; acc.z *= ws.z; acc.w *= ws.w;
    }
    if (scale) {
      const float r = rinv[i];
      acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
    }
    const float q2 = epi_quad<KIND>(ep, nr * kTcRows + i, fg, acc, pre, rinfo, i);
    if constexpr (KIND == kEpiResidNorm) sq[i * 64 + (it - i * nq)] = q2;
  }
  if constexpr (KIND == kEpiResidNorm) {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    if (et < rows_here) {
      float acc = 0.f;
      for (int j = 0; j < nq; ++j) acc += sq[et * 64 + j];
      ep.ssq_out[(size_t)(nr * kTcRows + et) * kMaxSsqParts + t * S + rank] = acc;
    }
  }
}

// While the mainloop runs: pull each epilogue thread's global operands
// (residual x, RoPE factors) into L1 so phase 2 does not wait on memory
// round trips that are long while HBM is saturated.
template <int KIND, int N>
__device__ __forceinline__ void epi_prefetch(const EpiArgs& ep, int S, int rank, int t, int nr, int rows_here,
                                             int et, const int2* rinfo) {
  if constexpr (KIND == kEpiResid || KIND == kEpiResidNorm || KIND == kEpiQKV) {
    const int q0 = rank * (N / 4) / S, q1 = (rank + 1) * (N / 4) / S;
    const int nq = q1 - q0;
    const int items = rows_here * nq;
    for (int it = et; it < items; it += kEpiThreads) {
      const int i = it / nq;
      const float* p = epi_pre_addr<KIND>(ep, nr * kTcRows + i, t * N + 4 * (q0 + it - i * nq), rinfo, i);
      if (p) asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
    }
  }
}

template <int N, int RT = 1>
__host__ __device__ constexpr int tc_stages() {
  return kTcRing / (N * kTcBK * 2 + RT * kTcABytes) < kTcMaxStages ? kTcRing / (N * kTcBK * 2 + RT * kTcABytes)
                                                                     : kTcMaxStages;
}
// Int8 weights: kConvBufs bf16 conversion buffers of N x 128 bytes, then
// stages of (int8 tile, activation tile) in the rest of the ring.
constexpr int kConvBufs = 2;   // 2: one more int8 stage at N = 256 (7B step 5.61 -> 5.49 ms) than with 3
template <int N>
__host__ __device__ constexpr int tc_stages8() {
  return (kTcRing - kConvBufs * N * 128) / (N * kTcBK + kTcABytes) < kTcMaxStages
             ? (kTcRing - kConvBufs * N * 128) / (N * kTcBK + kTcABytes)
             : kTcMaxStages;
}
// Two int8 weights (bytes j, j + 1 of w) -> bf16x2, exactly, the byte j
// value in the low half.  For a byte b = s|m (sign bit s, low bits m) the
// permute builds the bf16 words 0x43|b, from which one mask keeps
// 0x4300|m = 128 + m and the other 0x4300|(s << 7) = 128 or 256; their
// difference, m - 128 s, is the two's-complement value, and every number
// involved is an integer below 2^8, exact in bf16.
__device__ __forceinline__ uint32_t i8pair_bf16x2(uint32_t w, int j) {
  const uint32_t t = __byte_perm(w, 0x43434343u, 0x5140u + j + (j << 8));
  const uint32_t val = t & 0xFF7FFF7Fu, sub = t & 0xFF80FF80u;
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(val), "r"(sub));
  return r;
}
// 16 int8 weights -> 16 bf16, as two 16-byte chunks (8 k each, the lower k
// in the lower half of each 32-bit word).
__device__ __forceinline__ void i8x16_bf16(uint4 v, uint4& c0, uint4& c1) {
  c0 = make_uint4(i8pair_bf16x2(v.x, 0), i8pair_bf16x2(v.x, 2), i8pair_bf16x2(v.y, 0), i8pair_bf16x2(v.y, 2));
  c1 = make_uint4(i8pair_bf16x2(v.z, 0), i8pair_bf16x2(v.z, 2), i8pair_bf16x2(v.w, 0), i8pair_bf16x2(v.w, 2));
}

// One instantiation per tile width N (weight rows per tile, MMA N), weight
// type (I8: int8 weights with per-row scales) and row tiles per CTA (RT).
template <int N, bool I8, int RT>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                   const __grid_constant__ CUtensorMap tmL, const TcArgs a, const EpiArgs ep, const PfSpec pf) {
  static_assert(N % 32 == 0 && N >= 64 && N <= kTcMaxBN, "tile width");
  static_assert(RT == 1 || (RT == 2 && !I8), "two row tiles: bf16 weights");
  constexpr uint32_t idesc = tc::idesc_bf16(2 * kTcRows, N);
  constexpr int ST0 = I8 ? tc_stages8<N>() : tc_stages<N, RT>();
  constexpr uint32_t tmem_cols = RT == 2 ? 2 * kTcMaxBN : kTcMaxBN;
  // bf16: a stage is (weight tile, RT activation tiles); int8: (int8 tile,
  // activation tile), and the two bf16 conversion buffers follow the stages
  constexpr uint32_t w_bytes = (uint32_t)N * kTcBK * (I8 ? 1 : 2);   // one weight tile per stage
  constexpr uint32_t stage_bytes = w_bytes + RT * kTcABytes;
  constexpr uint32_t conv_off0 = (uint32_t)ST0 * stage_bytes;       // int8: bf16 buffer b at conv_off + b * N * 128
  static_assert(!I8 || (conv_off0 % 1024 == 0 && conv_off0 + kConvBufs * N * 128u <= (uint32_t)kTcRing),
                "int8 ring layout");
  static_assert(stage_bytes % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
  constexpr int PS = N + 4;                                     // fp32 partial row stride (padded)
  TR_DECL;
#ifdef CBD_TRACE
  unsigned long long _e0 = 0, _e1 = 0;    // epilogue: accumulator ready, hi + lo folded
#endif
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kTcMaxStages], empty_bar[kTcMaxStages];
  __shared__ __align__(8) uint64_t accum_full, mma_done;
  // int8 weights: int8 tile landed; bf16 buffer converted; bf16 buffer free
  __shared__ __align__(8) uint64_t w8_full[I8 ? kTcMaxStages : 1], conv_full[I8 ? kConvBufs : 1],
      conv_free[I8 ? kConvBufs : 1];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int decision;
  __shared__ int2 rinfo[kTcRows * RT];      // QKV epilogue: (position, KV block) of each tile row
  __shared__ float rinv[kTcRows * RT];      // fused RMSNorm consumer: 1/rms of each tile row

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  // unit = (feature tile t, row tiles nr .. nr + RT - 1); the cluster's
  // ranks split K
  const int S = a.S;
  const int rank = S > 1 ? (int)cluster_rank() : 0;
  const int unit = blockIdx.x / S;
  const int NP = (a.NR + RT - 1) / RT;
  const int nr = (unit % NP) * RT, t = unit / NP;
  const int rows_cta = min(kTcRows * RT, a.n - nr * kTcRows);   // activation rows of this CTA
  const int kb0 = rank * a.KB / S, kb1 = (rank + 1) * a.KB / S;
  const int n_it = kb1 - kb0;
  // stage s: weight (or int8) tile at w_off(s), activation tiles from a_off(s)
  constexpr int ST = ST0;
  constexpr uint32_t conv_off = conv_off0;
  auto w_off = [](int s) -> uint32_t { return (uint32_t)s * stage_bytes; };
  auto a_off = [](int s) -> uint32_t { return (uint32_t)s * stage_bytes + w_bytes; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    tc::mbar_init(&accum_full, 1);
    tc::mbar_init(&mma_done, 1);
    if constexpr (I8) {
      for (int s = 0; s < ST; ++s) tc::mbar_init(&w8_full[s], 1);
      for (int b = 0; b < kConvBufs; ++b) {
        tc::mbar_init(&conv_full[b], kEpiThreads / 32);
        tc::mbar_init(&conv_free[b], 1);
      }
    }
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::prefetch_tmap(&tmW);
    tc::prefetch_tmap(&tmH);
    tc::prefetch_tmap(&tmL);
  }
  pdl_trigger();
  if (warp == 1) tc::tmem_alloc(&tmem_base, tmem_cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort_p = &abort_flag;
  // the producer waits after prefetching weights; int8 converters after
  // converting the first weight tiles
  if (warp == 1 || (warp >= 2 && !I8)) pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      // activation rows: one 64-row box per row tile and half (hi, lo);
      // rows past the tile's last row carry stale values into TMEM lanes
      // the epilogue never reads
      static_assert(kActBoxRows == kTcRows, "one activation box per row tile");
      constexpr uint32_t abox = kTcABytes / 2;
      const int nbox1 = RT == 2 && rows_cta > kTcRows ? 1 : 0;   // second row tile
      const uint32_t stage_tx = w_bytes + 2u * (1 + nbox1) * abox;
      const uint64_t w_policy = tc::policy_evict_first();   // weights are read once per step
      // weight tiles 2t and 2t + 1 of N / 2 rows form a unit only with two
      // row tiles per CTA (steps of more than 128 rows)
      const bool paired = RT == 2 && a.P == 2;
      auto issue_w = [&](int q) {
        const int s = q % ST;
        uint8_t* st = ring + w_off(s);
        if constexpr (I8) {
          // the tile is one contiguous N x 64-byte run: one bulk copy
          tc::mbar_arrive_expect_tx(&w8_full[s], w_bytes);
          tc::bulk_load_hint(st, a.w8 + (size_t)(t * a.KB + kb0 + q) * w_bytes, w_bytes, &w8_full[s], w_policy);
        } else {
          tc::mbar_arrive_expect_tx(&full_bar[s], stage_tx);
          if (RT == 2 && paired) {
            // the two tiles stacked along the MMA's N
            tc::tma_load_2d_hint(st, &tmW, 0, ((2 * t) * a.KB + kb0 + q) * (N / 2), &full_bar[s], w_policy);
            tc::tma_load_2d_hint(st + (N / 2) * 128, &tmW, 0, ((2 * t + 1) * a.KB + kb0 + q) * (N / 2),
                                 &full_bar[s], w_policy);
          } else {
            tc::tma_load_2d_hint(st, &tmW, 0, (t * a.KB + kb0 + q) * N, &full_bar[s], w_policy);
          }
        }
      };
      auto issue_a = [&](int q) {
        const int s = q % ST;
        uint8_t* st = ring + a_off(s);
        const int kx = (kb0 + q) * kTcBK;
        if constexpr (I8) tc::mbar_arrive_expect_tx(&full_bar[s], 2u * abox);
        tc::tma_load_2d(st, &tmH, kx, nr * kTcRows, &full_bar[s]);
        tc::tma_load_2d(st + abox, &tmL, kx, nr * kTcRows, &full_bar[s]);
        if (nbox1) {
          tc::tma_load_2d(st + kTcABytes, &tmH, kx, (nr + 1) * kTcRows, &full_bar[s]);
          tc::tma_load_2d(st + kTcABytes + abox, &tmL, kx, (nr + 1) * kTcRows, &full_bar[s]);
        }
      };
      // weights do not depend on the previous kernel: start streaming them
      // before waiting for it, then add the activations
      const int npre = n_it < ST ? n_it : ST;
      for (int q = 0; q < npre; ++q) issue_w(q);
      pdl_wait();
      TR_MARK1;
      for (int q = 0; q < npre; ++q) issue_a(q);
      int q = npre;
      bool ok = true;
      for (; q < n_it; ++q) {
        const int s = q % ST;
        if (!tc::mbar_wait(&empty_bar[s], ((q / ST) & 1) ^ 1, a.err, abort_p)) { ok = false; break; }
        issue_w(q);
        issue_a(q);
      }
      // this CTA's stream is fully issued: start pulling the next GEMM's
      // first k-blocks into L2 while the last stages, the epilogue and the
      // kernel boundary drain
      TR_MARK2;
      if (ok) tc::pf_issue(pf, blockIdx.x, gridDim.x);
      if (!ok) {     // every load issued must land before the CTA exits
        for (int r = q > ST ? q - ST : 0; r < q; ++r) {
          int no_abort = 0;
          tc::mbar_wait(&full_bar[r % ST], (r / ST) & 1, nullptr, &no_abort);
          if constexpr (I8) tc::mbar_wait(&w8_full[r % ST], (r / ST) & 1, nullptr, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      const bool two = RT == 2 && rows_cta > kTcRows;    // the second row tile has rows
      for (int q = 0; q < n_it; ++q) {
        const int s = q % ST;
        if constexpr (I8)
          if (!tc::mbar_wait(&conv_full[q % kConvBufs], (q / kConvBufs) & 1, a.err, abort_p)) { ok = false; break; }
        if (!tc::mbar_wait(&full_bar[s], (q / ST) & 1, a.err, abort_p)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t rb = tc::smem_u32(ring);
        const uint64_t dW = I8 ? tc::sdesc_sw128(rb + conv_off + (uint32_t)(q % kConvBufs) * N * 128u)
                               : tc::sdesc_sw128(rb + w_off(s));
        const uint64_t dA = tc::sdesc_sw128(rb + a_off(s));
#pragma unroll
        for (int k = 0; k < kTcBK / 16; ++k)   // 16 bf16 = 32 bytes along K inside the swizzled rows
          tc::mma_bf16(tmem, dA + 2 * k, dW + 2 * k, idesc, (q > 0 || k > 0) ? 1u : 0u);
        if (RT == 2 && two) {
          const uint64_t dA1 = tc::sdesc_sw128(rb + a_off(s) + kTcABytes);   // second row tile (never packed)
#pragma unroll
          for (int k = 0; k < kTcBK / 16; ++k)
            tc::mma_bf16(tmem + (uint32_t)N, dA1 + 2 * k, dW + 2 * k, idesc, (q > 0 || k > 0) ? 1u : 0u);
        }
        tc::mma_commit(&empty_bar[s]);
        if constexpr (I8) tc::mma_commit(&conv_free[q % kConvBufs]);
      }
      if (ok && n_it > 0) tc::mma_commit(&accum_full);
      // every MMA issued completes before TMEM is released
      tc::mma_commit(&mma_done);
      int no_abort = 0;
      tc::mbar_wait(&mma_done, 0, a.err, &no_abort);
    }
  } else {
    // ------------------------------------------------ epilogue phase 1: fold hi + lo into the partial
    // TMEM lane group lg = warp % 4 holds tile rows 32 * (lg % 2) + lane,
    // hi halves for lg < 2 and lo halves for lg >= 2; two warps share each
    // lane group, one per half of the columns.  The lo warps copy their
    // lanes to shared memory, then the hi warps add them to their own (hi +
    // lo per element) and write the partial P; warps whose lanes hold no row
    // of this tile skip their loads.
    const int lg = warp & 3;
    // column halves on 32-column boundaries
    constexpr int c_mid = ((N / 2 + 31) / 32) * 32;
    const int c_lo = (warp - 2) < 4 ? 0 : c_mid, c_hi = (warp - 2) < 4 ? c_mid : N;
    const int rows_here = rows_cta;
    const int rl = (lg & 1) * 32 + lane;           // tile row of this lane
    const bool has_rows = (lg & 1) * 32 < rows_here;
    const uint32_t taddr = tmem + ((uint32_t)(lg * 32) << 16);
    float* P = reinterpret_cast<float*>(ring);                  // [64][PS] hi + lo
    float* LO = reinterpret_cast<float*>(ring + 64 * PS * 4);    // [64][PS] lo
    const int et = threadIdx.x - 64;
    if constexpr (I8) {
      // what the epilogue reads from the previous kernel and the staged
      // batch, fetched while the mainloop runs, after the first weight
      // tiles are converted (they need no dependency)
      auto prologue = [&]() {
        pdl_wait();
        if (ep.kind == kEpiQKV) {
          // the rows' positions and KV blocks, read while the mainloop runs
          for (int i = et; i < rows_here; i += kEpiThreads) {
            const RowDev rw = ep.rows[nr * kTcRows + i];
            rinfo[i] = make_int2(rw.pos, ep.tables[(size_t)rw.slot * ep.max_blocks_per_seq + (rw.pos >> 5)]);
          }
          asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
          epi_prefetch<kEpiQKV, N>(ep, S, rank, t, nr, rows_here, et, rinfo);
        } else if (ep.kind == kEpiResid) {
          epi_prefetch<kEpiResid, N>(ep, S, rank, t, nr, rows_here, et, rinfo);
        } else if (ep.kind == kEpiResidNorm) {
          epi_prefetch<kEpiResidNorm, N>(ep, S, rank, t, nr, rows_here, et, rinfo);
        }
        if (ep.ssq_in) {
          // fused RMSNorm: 1/rms of each row from the producer's partials; a
          // warp per row, lanes over the partials (all loads in flight), then a
          // fixed shuffle tree
          for (int i = warp - 2; i < rows_here; i += kEpiThreads / 32) {
            const float* sp = ep.ssq_in + (size_t)(nr * kTcRows + i) * kMaxSsqParts;
            float v[kMaxSsqParts / 32];
#pragma unroll
            for (int j = 0; j < kMaxSsqParts / 32; ++j) v[j] = lane + 32 * j < ep.n_parts_in ? sp[lane + 32 * j] : 0.f;
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxSsqParts / 32; ++j) acc += v[j];
            acc = warp_sum(acc);
            if (lane == 0) rinv[i] = 1.0f / sqrtf(acc / (float)ep.d_norm + ep.eps);
          }
        }
      };
      // convert each stage's int8 tile into a bf16 buffer the MMA reads;
      // the prologue runs once every buffer holds a tile
      bool conv_ok = true;
      const uint32_t conv_base = tc::smem_u32(ring) + conv_off;
      for (int q = 0; q < n_it; ++q) {
        const int s = q % ST, b = q % kConvBufs;
        if (conv_ok && (!tc::mbar_wait(&w8_full[s], (q / ST) & 1, a.err, abort_p) ||
                        !tc::mbar_wait(&conv_free[b], ((q / kConvBufs) & 1) ^ 1, a.err, abort_p)))
          conv_ok = false;
        conv_ok = __all_sync(0xffffffffu, conv_ok);    // warp-uniform before the warp's arrive
        if (conv_ok) {
          const uint8_t* src = ring + w_off(s);
          const uint32_t dst = conv_base + (uint32_t)b * N * 128u;
          // task i: row i / 4, 16-byte int8 chunk i % 4 -> bf16 chunks 2c, 2c + 1
#pragma unroll
          for (int j = 0; j < (N * 4 + kEpiThreads - 1) / kEpiThreads; ++j) {
            const int i = et + j * kEpiThreads;
            if (i < N * 4) {
              const int r = i >> 2, c = i & 3;
              const uint4 v = *reinterpret_cast<const uint4*>(src + r * 64 + c * 16);
              uint4 c0, c1;
              i8x16_bf16(v, c0, c1);
              const uint32_t row = dst + (uint32_t)r * 128u;
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((((2 * c) ^ (r & 7))) << 4)),
                           "r"(c0.x), "r"(c0.y), "r"(c0.z), "r"(c0.w) : "memory");
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((((2 * c + 1) ^ (r & 7))) << 4)),
                           "r"(c1.x), "r"(c1.y), "r"(c1.z), "r"(c1.w) : "memory");
            }
          }
          // the MMA (async proxy) reads what these threads wrote
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&conv_full[b]);
        }
        if (q == (n_it < kConvBufs ? n_it : kConvBufs) - 1) prologue();
      }
      if (n_it == 0) prologue();
    } else {
      if (ep.kind == kEpiQKV) {
        // the rows' positions and KV blocks, read while the mainloop runs
        for (int i = et; i < rows_here; i += kEpiThreads) {
          const RowDev rw = ep.rows[nr * kTcRows + i];
          rinfo[i] = make_int2(rw.pos, ep.tables[(size_t)rw.slot * ep.max_blocks_per_seq + (rw.pos >> 5)]);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
        epi_prefetch<kEpiQKV, N>(ep, S, rank, t, nr, rows_here, et, rinfo);
      } else if (ep.kind == kEpiResid) {
        epi_prefetch<kEpiResid, N>(ep, S, rank, t, nr, rows_here, et, rinfo);
      } else if (ep.kind == kEpiResidNorm) {
        epi_prefetch<kEpiResidNorm, N>(ep, S, rank, t, nr, rows_here, et, rinfo);
      }
      if (ep.ssq_in) {
        // fused RMSNorm: 1/rms of each row from the producer's partials; a
        // warp per row, lanes over the partials (all loads in flight), then a
        // fixed shuffle tree
        for (int i = warp - 2; i < rows_here; i += kEpiThreads / 32) {
          const float* sp = ep.ssq_in + (size_t)(nr * kTcRows + i) * kMaxSsqParts;
          float v[kMaxSsqParts / 32];
#pragma unroll
          for (int j = 0; j < kMaxSsqParts / 32; ++j) v[j] = lane + 32 * j < ep.n_parts_in ? sp[lane + 32 * j] : 0.f;
          float acc = 0.f;
#pragma unroll
          for (int j = 0; j < kMaxSsqParts / 32; ++j) acc += v[j];
          acc = warp_sum(acc);
          if (lane == 0) rinv[i] = 1.0f / sqrtf(acc / (float)ep.d_norm + ep.eps);
        }
      }
    }
    if (n_it > 0) tc::mbar_wait(&accum_full, 0, a.err, abort_p);
#ifdef CBD_TRACE
    _e0 = gtimer();
#endif
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    if (threadIdx.x == 64) decision = *abort_p || n_it == 0;
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    const bool skip = decision != 0;
    tc::tc_fence_after();
    // 64 columns per TMEM wait where two 32-column chunks remain, else 32
    auto load64 = [&](int c0, bool two, float (&v)[64]) {
      if (skip) {
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = 0.f;
        return;
      }
      uint32_t x0[32], x1[32];
      tc::tmem_ld32_nowait(taddr + c0, x0);
      if (two) tc::tmem_ld32_nowait(taddr + c0 + 32, x1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) { v[j] = __uint_as_float(x0[j]); v[32 + j] = two ? __uint_as_float(x1[j]) : 0.f; }
    };
    if constexpr (RT == 2) {
      // both accumulators, in place: P [128][PS]; the lo warps store their
      // lanes, then the hi warps add their own to them (hi + lo per element)
      for (int pass = 0; pass < 2; ++pass) {
        if ((pass == 0) == (lg >= 2)) {
#pragma unroll 1
          for (int acc = 0; acc < 2; ++acc) {
            if (acc * kTcRows + (lg & 1) * 32 >= rows_here) continue;
            float* prow = P + (acc * kTcRows + rl) * PS;
#pragma unroll 1
            for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
              uint32_t x[32];
              if (!skip) {
                tc::tmem_ld32_nowait(taddr + (uint32_t)(acc * N + c0), x);
                tc::tmem_wait_ld();
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = 0u;
              }
              float4* dst = reinterpret_cast<float4*>(prow + c0);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float4 v = make_float4(__uint_as_float(x[4 * j]), __uint_as_float(x[4 * j + 1]),
                                       __uint_as_float(x[4 * j + 2]), __uint_as_float(x[4 * j + 3]));
                if (pass == 1) {
                  const float4 l4 = dst[j];
                  v = make_float4(v.x + l4.x, v.y + l4.y, v.z + l4.z, v.w + l4.w);
                }
                dst[j] = v;
              }
            }
          }
        }
        if (pass == 0) asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
      }
    } else {
    if (lg >= 2 && has_rows) {
#pragma unroll 1
      for (int c0 = c_lo; c0 < c_hi; c0 += 64) {
        const bool two = c0 + 64 <= c_hi;
        float v[64];
        load64(c0, two, v);
        float4* lo = reinterpret_cast<float4*>(LO + rl * PS + c0);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < 8 || two) lo[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    if (lg < 2 && has_rows) {
#pragma unroll 1
      for (int c0 = c_lo; c0 < c_hi; c0 += 64) {
        const bool two = c0 + 64 <= c_hi;
        float v[64];
        load64(c0, two, v);
        const float4* lo = reinterpret_cast<const float4*>(LO + rl * PS + c0);
        float4* p = reinterpret_cast<float4*>(P + rl * PS + c0);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < 8 || two) {
            const float4 l4 = lo[j];
            p[j] = make_float4(v[4 * j] + l4.x, v[4 * j + 1] + l4.y, v[4 * j + 2] + l4.z, v[4 * j + 3] + l4.w);
          }
      }
    }
    }
#ifdef CBD_TRACE
    _e1 = gtimer();
#endif
    tc::tc_fence_before();
  }
  // ------------------------------------------------ cluster: every partial is in shared memory
  __syncwarp();
  if (S > 1) cluster_sync_all();
  else __syncthreads();
#ifdef CBD_TRACE
  const unsigned long long _e_sync = gtimer();
#endif
  if (warp >= 2) {
    // ------------------------------------------------ epilogue phase 2: reduce over ranks, finish
    const int et = threadIdx.x - 64;
    const int rows_here = rows_cta;
    const uint32_t Pbase = tc::smem_u32(ring);
    // the residual-norm sums: after P (the LO area, free after phase 1, when RT = 1)
    float* sq = reinterpret_cast<float*>(ring + kTcRows * RT * PS * 4);
    switch (ep.kind) {
      case kEpiQKV: epi_phase2<kEpiQKV, N, I8>(ep, S, rank, t, nr, rows_here, et, Pbase, rinfo, rinv, sq); break;
      case kEpiResid: epi_phase2<kEpiResid, N, I8>(ep, S, rank, t, nr, rows_here, et, Pbase, rinfo, rinv, sq); break;
      case kEpiResidNorm: epi_phase2<kEpiResidNorm, N, I8>(ep, S, rank, t, nr, rows_here, et, Pbase, rinfo, rinv, sq); break;
      case kEpiSwiGLU: epi_phase2<kEpiSwiGLU, N, I8>(ep, S, rank, t, nr, rows_here, et, Pbase, rinfo, rinv, sq); break;
      default: epi_phase2<kEpiLogits, N, I8>(ep, S, rank, t, nr, rows_here, et, Pbase, rinfo, rinv, sq); break;
    }
  }
#ifdef CBD_TRACE
  if (threadIdx.x == 64) {
    const unsigned long long te = gtimer();
    trace_put((17u << 12) | (unsigned)(a.M >> 8), _e0, _e1, _e_sync, te);
  }
#endif
  // peers keep their partials alive until every rank has read them
  __syncwarp();
  if (S > 1) cluster_sync_all();
  tc::tc_fence_before();
  __syncthreads();
  TR_END((16u << 12) | (unsigned)(a.M >> 8));
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tmem_cols);
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

bool make_tmap_i8(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {64, rows};
  cuuint64_t strides[1] = {64};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Co-resident clusters of each size on the current device (queried once per
// device; also sets the kernels' shared-memory limit there).  0 if the
// query fails.
static int max_clusters(int S) {
  static DeviceOnce once;
  static int cache[kMaxDevices][kTcMaxCluster + 1] = {};
  int dev = -1;
  const cudaError_t ce = once.run([](int d) -> cudaError_t {
    for (auto k : {gemm_tc_kernel<256, false, 1>, gemm_tc_kernel<224, false, 1>, gemm_tc_kernel<192, false, 1>,
                   gemm_tc_kernel<160, false, 1>, gemm_tc_kernel<128, false, 1>, gemm_tc_kernel<256, true, 1>,
                   gemm_tc_kernel<224, true, 1>, gemm_tc_kernel<192, true, 1>, gemm_tc_kernel<160, true, 1>,
                   gemm_tc_kernel<128, true, 1>, gemm_tc_kernel<256, false, 2>, gemm_tc_kernel<224, false, 2>,
                   gemm_tc_kernel<192, false, 2>, gemm_tc_kernel<160, false, 2>, gemm_tc_kernel<128, false, 2>}) {
      const cudaError_t e1 = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
      if (e1 != cudaSuccess) return e1;
    }
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
      if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<kTcMaxBN, false, 1>, &cfg) != cudaSuccess) {
        n = 0;
        cudaGetLastError();
      }
      cache[d][s] = n;
    }
    return cudaSuccess;
  }, &dev);
  if (ce != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return cache[dev][S];
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

int gemm_tc_row_tiles(int n, bool int8) { return !int8 && n > kTcRows ? 2 : 1; }

// Weight tiles per unit: in steps of more than 128 rows (two row tiles per
// CTA, at least two pairs of them), matrices tiled 128 rows wide (the 7B O
// and down projections) run as 256-wide units of two tiles, as the
// 256-row-tiled matrices do: a stage then carries as many weight bytes per
// activation byte, and each MMA covers 256 features.  Measured on GB300
// (7B): the 544-row mixed step 16.40 ms against 18.58 with 128-wide units
// (and 17.66 with the 128-row-tile kernel for O and down); B = 128 decode
// (one pair of row tiles) 10.71 against 10.41, hence not there.
int gemm_tc_pair(int M, int N, int n, bool int8) {
  return !int8 && n > 2 * kTcRows && N == 128 && (M / N) % 2 == 0 ? 2 : 1;
}

void gemm_tc_plan(int M, int K, int N, int n, int RT, int* T, int* NR, int* KB, int* S) {
  *T = M / N;
  *NR = (n + kTcRows - 1) / kTcRows;
  *KB = K / kTcBK;
  *S = choose_cluster((long long)*T * ((*NR + RT - 1) / RT), *KB);
}

// Weight rows per tile for an M x K matrix: the widest tile that divides M,
// except that a matrix with fewer than 20 such tiles (the 4096-row O and down
// projections of a 7B model) takes 128-row tiles.  Measured on GB300 (7B
// decode step, B = 32): 128-row tiles for O and down let 128 CTAs stream
// instead of 96 (4.79 vs 4.81 ms per step); narrower tiles for the wide
// matrices ran slower (QKV 4.94, gate/up 5.20 ms): HBM is already saturated
// while their weights stream, and the per-stage cost and the activation
// traffic per weight byte grow as the tile narrows.  Tiles that only fill
// more SMs (224 rows for gate/up: 128 CTAs instead of 112; 192 for QKV: 128
// instead of 120) gained 0.7-1.2 % on decode steps of 32-128 rows but lost
// 11 % at 544 rows and 1.4 % at 2080 (more units per tile row, and a last
// wave that is mostly empty), so the widest tile stays.
int gemm_tc_pick_tile(int M, int K) {
  (void)K;
  int best = kTcMaxBN;
  for (int N : {256, 224, 192, 160, 128})
    if (M % N == 0) { best = N; break; }
  if (M / best < 20 && M % 128 == 0) best = 128;
  return best;
}

cudaError_t launch_gemm_tc(const TcGemm& g, int n, const EpiArgs& ep, const PfSpec& pf, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (g.M % g.N || g.K % kTcBK) return cudaErrorInvalidValue;
  TcArgs a{};
  a.M = g.M; a.K = g.K; a.n = n;
  a.w8 = g.w8;
  if (g.scale && !g.w8) return cudaErrorInvalidValue;
  const int RT = gemm_tc_row_tiles(n, g.scale != nullptr);
  a.P = gemm_tc_pair(g.M, g.N, n, g.scale != nullptr);
  a.N = g.N * a.P;
  gemm_tc_plan(g.M, g.K, a.N, n, RT, &a.T, &a.NR, &a.KB, &a.S);
  a.err = ep.err;
  const long long U = (long long)a.T * ((a.NR + RT - 1) / RT);
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
  if (max_clusters(1) <= 0) return cudaErrorInvalidConfiguration;   // also sets the shared-memory limit
  // bf16 weights: RT row tiles per CTA; int8: one
#define CBD_TC_LAUNCH(NN)                                                                                  \
  return g.scale ? cudaLaunchKernelEx(&cfg, gemm_tc_kernel<NN, true, 1>, *g.w, *g.hi, *g.lo, a, ep, pf)    \
                 : (RT == 2 ? cudaLaunchKernelEx(&cfg, gemm_tc_kernel<NN, false, 2>, *g.w, *g.hi, *g.lo, a, ep, pf) \
                            : cudaLaunchKernelEx(&cfg, gemm_tc_kernel<NN, false, 1>, *g.w, *g.hi, *g.lo, a, ep, pf))
  switch (a.N) {
    case 256: CBD_TC_LAUNCH(256);
    case 224: CBD_TC_LAUNCH(224);
    case 192: CBD_TC_LAUNCH(192);
    case 160: CBD_TC_LAUNCH(160);
    case 128: CBD_TC_LAUNCH(128);
    default: return cudaErrorInvalidValue;
  }
#undef CBD_TC_LAUNCH
}

CBD_TRACE_BIND(gemm_tc)

}  // namespace cbd
