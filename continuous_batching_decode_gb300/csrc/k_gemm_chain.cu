// Persistent chain of decode weight contractions: the O projection, the
// gate/up projection and the down projection of one layer, and the QKV
// projection of the next, as the phases of one kernel launch.  Each phase
// computes exactly what gemm_tc_kernel computes for it -- fp32 sums of the
// bf16 weights times the hi + lo bf16 activations, split over K inside a
// group of CTAs and reduced in rank order, then the same epilogue -- so the
// results are bit-identical to the per-launch path; what goes is the kernel
// boundary between the phases: a CTA's producer starts streaming the next
// phase's weights (which do not depend on the previous phase) while the
// current phase's epilogue runs, and the phases are separated by a
// grid-wide barrier instead of a launch.  The decode step reads every
// weight once for all rows ("0.8MB 跑通 Qwen 第 14-1 篇", section 1;
// "20.3 服务、批处理与流式", section 20.3.2: step cost (W + B*A)/beta), and
// this removes most of the fixed time that sits between those streams.
//
// Layout.  Clusters of C CTAs, C = 4 or 8 (the largest K split among the
// phases, at least 4); in a phase with K split S (1, 2, 4 or 8, the
// per-launch kernel's choice) the cluster's CTAs form C / S groups of S
// consecutive ranks; a group owns one feature tile of the single 64-row
// activation tile and its ranks take consecutive k-ranges.  The ring holds
// 192 KB of stages (weight tile + activation tile, sized by the phase's tile
// width N = 128 or 256); a phase's fp32 partial tile and its residual-norm
// partial sums sit at the end of the ring, so the next phase's first stages,
// which lie below them, can be filled while the epilogue runs.
//
// Synchronisation, every wait bounded (a wait that runs out records
// kDevWaitTimeout and the kernel winds down):
//   * full / empty mbarriers per stage slot, parity tracked per slot across
//     phases; the producer drains a phase's stages before the next phase
//     lays the ring out again with another stage size;
//   * accum_full (a unit's MMAs are done) and acc_free (the fold has read
//     TMEM) between the MMA thread and the epilogue warps;
//   * part_ready / part_done: once per phase every CTA of the cluster
//     arrives on all C CTAs' barriers, after publishing its partial and
//     after reading its group's partials; every CTA, busy or idle in the
//     phase, passes both in phase order, so an arrival always counts toward
//     the phase it belongs to;
//   * sync[p]: after phase p's stores a CTA adds 1 to a global counter
//     (zeroed by the step's first kernel); a CTA loads phase p+1's
//     activations, and its epilogue reads phase p's outputs, once the
//     counter holds the grid size.  The grid is at most the number of
//     co-resident clusters, and the next kernel of the stream launches only
//     once every CTA of this one has started, so every CTA is resident.
#include <cudaTypedefs.h>

#include <algorithm>

#include "gemm_epi.cuh"

namespace cbd {

constexpr int kChMaxCluster = 8;
constexpr int kChRows = 64;                              // activation rows per tile (MMA M = 2 x 64: hi, lo)
constexpr int kChBK = 64;                                // k per stage
constexpr int kChEpiThreads = 256;                       // 8 epilogue warps
constexpr int kChThreads = 64 + kChEpiThreads;
constexpr int kChABytes = 2 * kChRows * kChBK * 2;       // 16 KB activation tile (hi rows, then lo rows)
constexpr int kChRing = 192 * 1024;
constexpr int kChSmem = kChRing + 1024;
constexpr int kChMaxStages = 8;

struct ChainPhase {
  int N;                  // weight rows per tile (128 or 256)
  int T, KB, S;           // feature tiles, k-blocks, K split
  int pf;                 // k-blocks per CTA prefetched into L2 before the phase (beyond the staged ones)
  EpiArgs ep;
};
struct ChainArgs {
  int n_phases, n;        // phases, activation rows (<= 64)
  int C;                  // cluster size (4 or 8)
  ChainPhase ph[kChainMaxPhases];
  uint32_t* sync;         // [kChainMaxPhases] grid-barrier counters, zero at launch
  int32_t* err;
};
struct ChainMaps {
  CUtensorMap m[kChainMaxPhases][3];   // weights, activation hi, activation lo of each phase
};

__host__ __device__ constexpr int ch_stage_bytes(int N) { return N * kChBK * 2 + kChABytes; }
__host__ __device__ constexpr int ch_stages(int N) {
  return kChRing / ch_stage_bytes(N) < kChMaxStages ? kChRing / ch_stage_bytes(N) : kChMaxStages;
}
// A phase's partial area at the end of the ring: P [64][N + 4] fp32 (hi +
// lo sums), then the residual-norm partial sums [64][64] fp32.
__host__ __device__ constexpr int ch_part_bytes(int N) {
  return ((64 * (N + 4) + 64 * 64) * 4 + 1023) / 1024 * 1024;
}
static_assert(ch_part_bytes(256) + ch_stage_bytes(256) <= kChRing, "a stage fits below every partial area");

__device__ __forceinline__ uint32_t ch_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ch_ld_peer_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// Arrive on the mbarrier at this shared-memory offset in cluster CTA `rank`
// (release at cluster scope).
__device__ __forceinline__ void ch_arrive_remote(uint64_t* bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ch_map(tc::smem_u32(bar), rank))
               : "memory");
}
// Wait for the phase with this parity of a barrier that peers arrive on
// (acquire at cluster scope).
__device__ __forceinline__ bool ch_wait_cluster(uint64_t* bar, uint32_t parity, int32_t* err, volatile int* abort) {
  const long long t0 = clock64();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(tc::smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if (*abort) return false;
    if (clock64() - t0 > tc::kWaitLimit) {
      set_err(err, kDevWaitTimeout);
      *abort = 1;
      return false;
    }
  }
}
// L2 prefetch of one weight tile (box of the tensor map at x, y).
__device__ __forceinline__ void ch_prefetch_tile(const CUtensorMap* m, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y)
               : "memory");
}
// Grid barrier: wait until the counter holds `target` (acquire at GPU
// scope), then order what the other CTAs wrote before this thread's
// bulk-copy (async proxy) reads.
__device__ __forceinline__ bool ch_wait_grid(const uint32_t* ctr, uint32_t target, int32_t* err, volatile int* abort) {
  const long long t0 = clock64();
  while (true) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) break;
    if (*abort) return false;
    if (clock64() - t0 > tc::kWaitLimit) {
      set_err(err, kDevWaitTimeout);
      *abort = 1;
      return false;
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}
// Named barrier 1 over the 256 epilogue threads that also ANDs a flag: every
// thread leaves with the same value, true only if every thread passed true.
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kChEpiThreads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kChEpiThreads) : "memory"); }

// Epilogue phase 2 of one phase, the arithmetic of gemm_tc_kernel's: rank
// r of a group of S (cluster ranks r0 .. r0 + S - 1) finalises feature
// quads [r*N/4/S, (r+1)*N/4/S) of its tile for every row, reading the S
// partials (over distributed shared memory) and adding them in rank order.
// The tile width N is a run-time value: one copy of each epilogue kind
// keeps the kernel within its registers.
template <int KIND>
__device__ __forceinline__ void ch_phase2(int N, const EpiArgs& ep, int S, int r0, int rank, int t, int rows_here,
                                          int et, uint32_t Pbase, const int2* rinfo, const float* rinv, float* sq) {
  const int q0 = rank * (N / 4) / S, q1 = (rank + 1) * (N / 4) / S;
  const int PS = N + 4;
  const int nq = q1 - q0;
  const int items = rows_here * nq;
  const bool scale = ep.ssq_in != nullptr;
#pragma unroll 1
  for (int it = et; it < items; it += kChEpiThreads) {
    const int i = it / nq;
    const int f = 4 * (q0 + it - i * nq);
    const uint32_t off = (uint32_t)(i * PS + f) * 4u;
    const int fg = t * N + f;
    const float4 pre = epi_preload<KIND>(ep, i, fg, rinfo, i);
    float4 acc;
    if (S == 1) {
      acc = ch_ld_peer_f4(ch_map(Pbase + off, (uint32_t)r0));
    } else {
      // ranks in batches of four: the loads of a batch are in flight together
      acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int b0 = 0; b0 < kChMaxCluster; b0 += 4) {
        if (b0 < S) {
          float4 pv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (b0 + j < S) pv[j] = ch_ld_peer_f4(ch_map(Pbase + off, (uint32_t)(r0 + b0 + j)));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (b0 + j < S) {
              acc.x += pv[j].x; acc.y += pv[j].y;
              acc.z += pv[j].z; acc.w += pv[j].w;
            }
        }
      }
    }
    if (scale) {
      const float r = rinv[i];
      acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
    }
    const float q2 = epi_quad<KIND>(ep, i, fg, acc, pre, rinfo, i);
    if constexpr (KIND == kEpiResidNorm) sq[i * 64 + (it - i * nq)] = q2;
  }
  if constexpr (KIND == kEpiResidNorm) {
    epi_sync();
    if (et < rows_here) {
      float acc = 0.f;
      for (int j = 0; j < nq; ++j) acc += sq[et * 64 + j];
      ep.ssq_out[(size_t)et * kMaxSsqParts + t * S + rank] = acc;
    }
  }
}

__device__ __forceinline__ void ch_phase2_kind(int N, const EpiArgs& ep, int S, int r0, int rank, int t,
                                               int rows_here, int et, uint32_t Pbase, const int2* rinfo,
                                               const float* rinv, float* sq) {
  switch (ep.kind) {
    case kEpiQKV: ch_phase2<kEpiQKV>(N, ep, S, r0, rank, t, rows_here, et, Pbase, rinfo, rinv, sq); break;
    case kEpiResid: ch_phase2<kEpiResid>(N, ep, S, r0, rank, t, rows_here, et, Pbase, rinfo, rinv, sq); break;
    case kEpiResidNorm: ch_phase2<kEpiResidNorm>(N, ep, S, r0, rank, t, rows_here, et, Pbase, rinfo, rinv, sq); break;
    case kEpiSwiGLU: ch_phase2<kEpiSwiGLU>(N, ep, S, r0, rank, t, rows_here, et, Pbase, rinfo, rinv, sq); break;
    default: ch_phase2<kEpiLogits>(N, ep, S, r0, rank, t, rows_here, et, Pbase, rinfo, rinv, sq); break;
  }
}

// This CTA's share of phase p: group gi of S CTAs owns feature tile gi;
// false if the CTA is idle in the phase.
__device__ __forceinline__ bool ch_unit(const ChainArgs& a, int p, uint32_t crank, int& t, int& rank, int& r0) {
  const int S = a.ph[p].S;
  rank = (int)crank % S;
  r0 = (int)crank - rank;
  t = (int)(blockIdx.x / a.C) * (a.C / S) + (int)crank / S;
  return t < a.ph[p].T;
}

__global__ void __launch_bounds__(kChThreads, 1)
    gemm_chain_kernel(const __grid_constant__ ChainMaps maps, const __grid_constant__ ChainArgs a) {
  TR_DECL;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kChMaxStages], empty_bar[kChMaxStages];
  __shared__ __align__(8) uint64_t accum_full, acc_free, mma_done, part_ready, part_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int2 rinfo[kChRows];           // QKV epilogue: (position, KV block) of each row
  __shared__ float rinv[kChRows];           // fused RMSNorm consumer: 1/rms of each row

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = tc::smem_u32(smem_raw);
  uint8_t* ring = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const uint32_t crank = cluster_rank();
  const int rows_here = min(kChRows, a.n);
  const uint32_t grid = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kChMaxStages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    tc::mbar_init(&accum_full, 1);
    tc::mbar_init(&acc_free, kChEpiThreads / 32);
    tc::mbar_init(&mma_done, 1);
    tc::mbar_init(&part_ready, a.C);
    tc::mbar_init(&part_done, a.C);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0)
    for (int p = 0; p < a.n_phases; ++p)
      for (int j = 0; j < 3; ++j) tc::prefetch_tmap(&maps.m[p][j]);
  pdl_trigger();
  if (warp == 1) tc::tmem_alloc(&tmem_base, 256);
  tc::tc_fence_before();
  __syncthreads();
  cluster_sync_all();          // every peer's barriers are initialised before the first remote arrive
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort_p = &abort_flag;
  int32_t* err = a.err;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t w_policy = tc::policy_evict_first();   // weights are read once per step
      // activation rows: one 64-row box per half (hi, lo); rows past the
      // last one land in TMEM lanes no epilogue reads
      static_assert(kActBoxRows == kChRows, "one activation box per row tile");
      constexpr uint32_t abox = kChABytes / 2;
      uint32_t fpar = 0;                                     // per slot: fills so far, mod 2
      bool ok = true;
      for (int p = 0; p < a.n_phases && ok; ++p) {
        const ChainPhase& ph = a.ph[p];
        int t, rank, r0;
        const bool busy = ch_unit(a, p, crank, t, rank, r0);
        const int N = ph.N;
        const int ST = ch_stages(N);
        const uint32_t sb = (uint32_t)ch_stage_bytes(N);
        const uint32_t wb = (uint32_t)N * kChBK * 2;
        const int kb0 = rank * ph.KB / ph.S, kb1 = (rank + 1) * ph.KB / ph.S;
        const int n_it = busy ? kb1 - kb0 : 0;
        // stages below the previous phase's partial area are filled while
        // its epilogue runs; the rest once its partials are consumed
        const int pre = p == 0 ? ST : min(ST, (int)((kChRing - ch_part_bytes(a.ph[p - 1].N)) / sb));
        auto fill_w = [&](int q) -> bool {
          const int s = q % ST;
          if (!tc::mbar_wait(&empty_bar[s], ((fpar >> s) & 1u) ^ 1u, err, abort_p)) return false;
          fpar ^= 1u << s;
          tc::mbar_arrive_expect_tx(&full_bar[s], wb + 2u * abox);
          tc::tma_load_2d_hint(ring + (size_t)s * sb, &maps.m[p][0], 0, (t * ph.KB + kb0 + q) * N, &full_bar[s],
                               w_policy);
          return true;
        };
        auto fill_a = [&](int q) {
          const int s = q % ST;
          uint8_t* st = ring + (size_t)s * sb + wb;
          const int kx = (kb0 + q) * kChBK;
          tc::tma_load_2d(st, &maps.m[p][1], kx, 0, &full_bar[s]);
          tc::tma_load_2d(st + abox, &maps.m[p][2], kx, 0, &full_bar[s]);
        };
        const int npre = min(n_it, pre);
        int q = 0;
        for (; q < npre && ok; ++q) ok = fill_w(q);
        if (!ok) break;
        // the activations are the previous phase's (or kernel's) output;
        // the stages already armed get theirs even if the wait gave up, so
        // that every armed stage completes
        bool ready = true;
        if (p == 0) {
          pdl_wait();
          TR_MARK1;
        } else {
          ready = ch_wait_grid(a.sync + (p - 1), grid, err, abort_p);
        }
        for (int j = 0; j < q; ++j) fill_a(j);
        if (!ready) {
          ok = false;
          break;
        }
        if (p > 0 && q < n_it && !ch_wait_cluster(&part_done, (uint32_t)((p - 1) & 1), err, abort_p)) {
          ok = false;
          break;
        }
        for (; q < n_it && ok; ++q) {
          ok = fill_w(q);
          if (ok) fill_a(q);
        }
        // every load of this phase is issued: ask L2 for the next phase's
        // k-blocks that will not fit in the stages filled ahead of it, so
        // that HBM keeps streaming through the phase boundary
        if (ok && p + 1 < a.n_phases && a.ph[p + 1].pf > 0) {
          const ChainPhase& nx = a.ph[p + 1];
          int tn, rn, r0n;
          if (ch_unit(a, p + 1, crank, tn, rn, r0n)) {
            const int b0 = rn * nx.KB / nx.S, b1 = (rn + 1) * nx.KB / nx.S;
            const int pre_n = min(ch_stages(nx.N), (kChRing - ch_part_bytes(N)) / ch_stage_bytes(nx.N));
            for (int j = pre_n; j < min(b1 - b0, pre_n + nx.pf); ++j)
              ch_prefetch_tile(&maps.m[p + 1][0], 0, (tn * nx.KB + b0 + j) * nx.N);
          }
        }
        // drain: every stage of this phase is consumed before the next phase
        // lays the ring out again
        for (int s = 0; s < ST && ok && n_it > 0; ++s)
          ok = tc::mbar_wait(&empty_bar[s], ((fpar >> s) & 1u) ^ 1u, err, abort_p);
      }
      TR_MARK2;
      if (!ok) {       // every load issued must land before the CTA exits
        for (int s = 0; s < kChMaxStages; ++s) {
          int no_abort = 0;
          tc::mbar_wait(&full_bar[s], ((fpar >> s) & 1u) ^ 1u, nullptr, &no_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t cpar = 0;                                     // per slot: fills consumed so far, mod 2
      int units = 0;
      bool ok = true;
      for (int p = 0; p < a.n_phases && ok; ++p) {
        const ChainPhase& ph = a.ph[p];
        int t, rank, r0;
        if (!ch_unit(a, p, crank, t, rank, r0)) continue;
        const int N = ph.N;
        const int ST = ch_stages(N);
        const uint32_t sb = (uint32_t)ch_stage_bytes(N);
        const uint32_t wb = (uint32_t)N * kChBK * 2;
        const uint32_t idesc = N == 256 ? tc::idesc_bf16(2 * kChRows, 256) : tc::idesc_bf16(2 * kChRows, 128);
        const int n_it = (rank + 1) * ph.KB / ph.S - rank * ph.KB / ph.S;
        // the previous unit's fold has read the accumulator
        if (units > 0 && !tc::mbar_wait(&acc_free, (uint32_t)((units - 1) & 1), err, abort_p)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        for (int q = 0; q < n_it; ++q) {
          const int s = q % ST;
          if (!tc::mbar_wait(&full_bar[s], (cpar >> s) & 1u, err, abort_p)) { ok = false; break; }
          cpar ^= 1u << s;
          tc::tc_fence_after();
          const uint32_t st = tc::smem_u32(ring + (size_t)s * sb);
          const uint64_t dW = tc::sdesc_sw128(st);
          const uint64_t dA = tc::sdesc_sw128(st + wb);
#pragma unroll
          for (int k = 0; k < kChBK / 16; ++k)
            tc::mma_bf16(tmem, dA + 2 * k, dW + 2 * k, idesc, (q > 0 || k > 0) ? 1u : 0u);
          tc::mma_commit(&empty_bar[s]);
        }
        if (ok) tc::mma_commit(&accum_full);
        ++units;
      }
      // every MMA issued completes before TMEM is released
      tc::mma_commit(&mma_done);
      int no_abort = 0;
      tc::mbar_wait(&mma_done, 0, err, &no_abort);
    }
  } else {
    // ------------------------------------------------ epilogue warps
    // TMEM lane group lg = warp % 4 holds tile rows 32 * (lg % 2) + lane,
    // the hi halves for lg < 2 and the lo halves for lg >= 2; warps 2-5 take
    // the first half of the columns, warps 6-9 the second.
    const int et = threadIdx.x - 64;
    const int lg = warp & 3;
    const int rl = (lg & 1) * 32 + lane;
    const bool has_rows = (lg & 1) * 32 < rows_here;
    const uint32_t taddr = tmem + ((uint32_t)(lg * 32) << 16);
    int units = 0;
    bool ok = true;
    for (int p = 0; p < a.n_phases; ++p) {
      const ChainPhase& ph = a.ph[p];
      const EpiArgs& ep = ph.ep;
      int t = 0, rank = 0, r0 = 0;
      const bool busy = ch_unit(a, p, crank, t, rank, r0);
      const int N = ph.N;
      const int PS = N + 4;
      float* P = reinterpret_cast<float*>(ring + (kChRing - ch_part_bytes(N)));
      float* sq = P + 64 * PS;
      // what this phase's epilogue reads from the previous phase (or kernel)
      if (p == 0) pdl_wait();
      else if (et == 0 && ok) ok = ch_wait_grid(a.sync + (p - 1), grid, err, abort_p);
      ok = epi_all(ok && !*abort_p);
      if (busy && ok) {
        if (ep.kind == kEpiQKV) {
          for (int i = et; i < rows_here; i += kChEpiThreads) {
            const RowDev rw = ep.rows[i];
            rinfo[i] = make_int2(rw.pos, ep.tables[(size_t)rw.slot * ep.max_blocks_per_seq + (rw.pos >> 5)]);
          }
        }
        if (ep.ssq_in) {
          // 1/rms of each row from the producer's partials: a warp per row,
          // lanes over the partials, a fixed shuffle tree
          for (int i = warp - 2; i < rows_here; i += kChEpiThreads / 32) {
            const float* sp = ep.ssq_in + (size_t)i * kMaxSsqParts;
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
        ok = tc::mbar_wait(&accum_full, (uint32_t)(units & 1), err, abort_p);
      }
      // every peer has read the previous phase's partials before this
      // phase's fold overwrites the partial area
      if (p > 0 && ok) ok = ch_wait_cluster(&part_done, (uint32_t)((p - 1) & 1), err, abort_p);
      ok = epi_all(ok && !*abort_p);
      tc::tc_fence_after();
      if (busy && ok) {
        // fold hi + lo into P: the lo warps store their lanes, then the hi
        // warps add their own to them (hi + lo per element)
        const int c_mid = ((N / 2 + 31) / 32) * 32;
        const int c_lo = (warp - 2) < 4 ? 0 : c_mid, c_hi = (warp - 2) < 4 ? c_mid : N;
        for (int pass = 0; pass < 2; ++pass) {
          if ((pass == 0) == (lg >= 2) && has_rows) {
#pragma unroll 1
            for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
              uint32_t x[32];
              tc::tmem_ld32_nowait(taddr + c0, x);
              tc::tmem_wait_ld();
              float4* dst = reinterpret_cast<float4*>(P + rl * PS + c0);
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
          epi_sync();
        }
        // the accumulator is read: the MMA may start the next unit
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acc_free);
        ++units;
      }
      // publish this CTA's partial to the cluster (idle CTAs arrive too)
      asm volatile("fence.acq_rel.cluster;" ::: "memory");
      epi_sync();
      if (et == 0)
        for (uint32_t r = 0; r < (uint32_t)a.C; ++r) ch_arrive_remote(&part_ready, r);
      const bool ready = ch_wait_cluster(&part_ready, (uint32_t)(p & 1), err, abort_p);
      ok = epi_all(ok && ready && !*abort_p);
      if (busy && ok) {
        const uint32_t Pbase = tc::smem_u32(P);
        ch_phase2_kind(N, ep, ph.S, r0, rank, t, rows_here, et, Pbase, rinfo, rinv, sq);
      }
      // this CTA has read its group's partials and finished its stores: the
      // shared memory they used may be refilled by bulk copies, and the
      // outputs are published to the grid
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("fence.proxy.async.global;" ::: "memory");
      epi_sync();
      if (et == 0) {
        __threadfence();
        for (uint32_t r = 0; r < (uint32_t)a.C; ++r) ch_arrive_remote(&part_done, r);
        if (p + 1 < a.n_phases) atomicAdd(a.sync + p, 1u);
      }
    }
  }
  // every peer has read this CTA's last partial before it exits
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  TR_END(18u << 12);
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------- host side
// Co-resident clusters of C = 4 or 8 on the current device (queried once
// per device; also sets the kernel's shared-memory limit there).  0 if the
// query fails.
static int chain_max_clusters(int C) {
  static DeviceOnce once;
  static int cache[kMaxDevices][2] = {};
  int dev = -1;
  const cudaError_t ce = once.run([](int d) -> cudaError_t {
    cudaError_t e1 = cudaFuncSetAttribute(gemm_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kChSmem);
    if (e1 != cudaSuccess) return e1;
    for (int i = 0; i < 2; ++i) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(8 * 32);
      cfg.blockDim = dim3(kChThreads);
      cfg.dynamicSmemBytes = kChSmem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 4 << i;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_chain_kernel, &cfg) != cudaSuccess) {
        n = 0;
        cudaGetLastError();
      }
      cache[d][i] = n;
    }
    return cudaSuccess;
  }, &dev);
  if (ce != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return cache[dev][C == 8 ? 1 : 0];
}

// The chain's plan: each phase's tiles, k-blocks and K split (the
// per-launch kernel's), the cluster size and the clusters to launch; false
// if the chain cannot run these phases.
static bool chain_plan(const TcGemm* g, int n_phases, int n, ChainArgs* a, int* clusters) {
  if (n < 1 || n > kChRows || n_phases < 1 || n_phases > kChainMaxPhases) return false;
  int C = 4;
  long long ctas = 0;
  for (int p = 0; p < n_phases; ++p) {
    if ((g[p].N != 128 && g[p].N != 256) || g[p].M % g[p].N || g[p].K % kChBK || g[p].scale || g[p].w8) return false;
    ChainPhase& ph = a->ph[p];
    int NR;
    ph.N = g[p].N;
    gemm_tc_plan(g[p].M, g[p].K, g[p].N, n, 1, &ph.T, &NR, &ph.KB, &ph.S);
    // the per-launch kernel's K split (so the same sums), one that divides
    // the cluster, at least one k-block per rank
    if ((ph.S != 1 && ph.S != 2 && ph.S != 4 && ph.S != 8) || ph.KB < ph.S || NR != 1) return false;
    C = std::max(C, ph.S);
    ctas = std::max(ctas, (long long)ph.T * ph.S);
  }
  const long long need = (ctas + C - 1) / C;
  const int avail = chain_max_clusters(C);
  if (avail <= 0 || need > avail) return false;
  a->n_phases = n_phases;
  a->n = n;
  a->C = C;
  *clusters = (int)need;
  return true;
}

bool gemm_chain_possible(const TcGemm* g, int n_phases, int n) {
  ChainArgs a{};
  int clusters = 0;
  return chain_plan(g, n_phases, n, &a, &clusters);
}

cudaError_t launch_gemm_chain(const TcGemm* g, const EpiArgs* ep, int n_phases, int n, uint32_t* sync,
                              size_t pf_bytes, cudaStream_t s) {
  ChainMaps maps{};
  ChainArgs a{};
  int clusters = 0;
  if (!sync || !chain_plan(g, n_phases, n, &a, &clusters)) return cudaErrorInvalidValue;
  a.sync = sync;
  a.err = ep[0].err;
  for (int p = 0; p < n_phases; ++p) {
    ChainPhase& ph = a.ph[p];
    ph.ep = ep[p];
    // pf_bytes of each phase's weights, spread over its CTAs (whole tiles)
    const double per_cta = (double)pf_bytes / ((double)ph.T * ph.S) / ((double)ph.N * kChBK * 2);
    ph.pf = p == 0 ? 0 : (int)std::min<double>(per_cta, (double)ph.KB);
    maps.m[p][0] = *g[p].w;
    maps.m[p][1] = *g[p].hi;
    maps.m[p][2] = *g[p].lo;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(clusters * a.C));
  cfg.blockDim = dim3(kChThreads);
  cfg.dynamicSmemBytes = kChSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = a.C;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, gemm_chain_kernel, maps, a);
}

CBD_TRACE_BIND(gemm_chain)

}  // namespace cbd
