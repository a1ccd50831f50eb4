// The streaming attention kernel (attn_stream_kernel) and the tensor-core
// helpers it shares with the other attention kernels; included by the
// translation units that instantiate it (bf16 K/V and FP8 E4M3 K/V).
#pragma once

#include "tc.cuh"

namespace cbd {

// ---------------------------------------------------------------- tensor cores
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Two FP8 E4M3 values (byte 0, byte 1 of v) -> f16x2 (exact: every E4M3
// value is an f16 value); byte 0 lands in the low half.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
__device__ __forceinline__ uint32_t e4m3_lo(uint32_t w) { return e4m3x2_f16x2((uint16_t)(w & 0xffffu)); }
__device__ __forceinline__ uint32_t e4m3_hi(uint32_t w) { return e4m3x2_f16x2((uint16_t)(w >> 16)); }
// (a, b) -> packed f16x2 hi and lo halves (a in the low 16 bits): x = hi + lo
// to ~22 significant bits
__device__ __forceinline__ void split_pack_h(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half ah = __float2half_rn(a), bh = __float2half_rn(b);
  const __half al = __float2half_rn(a - __half2float(ah)), bl = __float2half_rn(b - __half2float(bh));
  hi = (uint32_t)__half_as_ushort(ah) | ((uint32_t)__half_as_ushort(bh) << 16);
  lo = (uint32_t)__half_as_ushort(al) | ((uint32_t)__half_as_ushort(bl) << 16);
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// (a, b) -> packed bf16x2 hi and lo halves (a in the low 16 bits)
__device__ __forceinline__ void split_pack(float a, float b, uint32_t& hi, uint32_t& lo) {
  uint16_t ah, al, bh, bl;
  split_bf16(a, ah, al);
  split_bf16(b, bh, bl);
  hi = (uint32_t)ah | ((uint32_t)bh << 16);
  lo = (uint32_t)al | ((uint32_t)bl << 16);
}
// Byte offset of (row, 16-byte chunk c) in a 128-byte-swizzled 32 x 64 bf16 tile.
__device__ __forceinline__ uint32_t swz(int row, int c) { return row * 128 + ((c ^ (row & 7)) << 4); }

constexpr int kStreamWarps = 8;
template <int HD>
__host__ __device__ constexpr int attn_stream_slots() { return HD == 128 ? 3 : 6; }
template <int HD>
__host__ __device__ constexpr int attn_stream_smem() {
  return kStreamWarps * attn_stream_slots<HD>() * (32 * HD * 2) + kStreamWarps * 8 * 32 * 4 + 1024;
}
// FP8 K/V: the same ring bytes per SM, spread over more warps (the kernel is
// latency-bound at half the bytes, and more warps per scheduler hide more):
// 12 warps of 16 KB rings instead of 8 of 24 KB.
constexpr int kStreamWarps8 = 12;
template <int HD, bool FP8>
__host__ __device__ constexpr int stream_warps() { return FP8 ? kStreamWarps8 : kStreamWarps; }
template <int HD, bool FP8>
__host__ __device__ constexpr int stream_slots() { return FP8 ? (HD == 128 ? 4 : 8) : attn_stream_slots<HD>(); }
template <int HD, bool FP8>
__host__ __device__ constexpr int stream_smem() {
  return stream_warps<HD, FP8>() * stream_slots<HD, FP8>() * (32 * HD * (FP8 ? 1 : 2)) +
         stream_warps<HD, FP8>() * 8 * 32 * 4 + 1024;
}

// FP8 = true: K and V are E4M3 bytes (tile layouts in common.cuh: K
// [pos][dim], V transposed [dim][pos], both 16-byte-chunk swizzled).  An
// ldmatrix over byte pairs gives each lane 4 consecutive bytes of a row;
// the MMA's k index is permuted accordingly -- fragment k pair (2t, 2t+1)
// takes bytes 4t, 4t+1 and pair (2t+8, 2t+9) bytes 4t+2, 4t+3 of the
// 16-byte chunk -- on both operands (q or P build the same permutation), so
// the sums are unchanged.  Products run as f16 MMAs, K/V converted exactly,
// q and P split into f16 hi + lo.
template <int HD, int G, bool FP8 = false>
__global__ void __launch_bounds__(stream_warps<HD, FP8>() * 32, 1) attn_stream_kernel(
    const uint16_t* __restrict__ pool, const float* __restrict__ q, const RowDev* __restrict__ rows,
    const int32_t* __restrict__ tables, const AttnWork* __restrict__ work, const int32_t* __restrict__ row_work,
    int n_tasks, int layer, int n_blocks, int hkv, int mbps, float* __restrict__ part_o, float* __restrict__ part_ml,
    uint16_t* __restrict__ out_hi, uint16_t* __restrict__ out_lo, int32_t* __restrict__ next_task, const PfSpec pf,
    int32_t* err) {
  static_assert(G >= 1 && G <= 8, "a KV group must fit the MMA's N = 8");
  constexpr int EB = FP8 ? 1 : 2;          // bytes per K / V element
  constexpr int TILE = 32 * HD * EB;
  constexpr int KS = HD / 16;
  constexpr int NS = stream_slots<HD, FP8>();   // ring slots per warp, one K or V tile each
  constexpr int NW = stream_warps<HD, FP8>();   // warps per CTA
  constexpr int QN = NS + 1 > 8 ? 16 : 8;   // task queue entries per warp (>= NS + 1)
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t bar[NW][NS];
  __shared__ int abort_flag;
  // tasks whose blocks this warp's producer has started issuing:
  // (row, start, end, kvh), (wi, task, -, -)
  __shared__ __align__(16) int tq[NW][QN][8];
  TR_DECL;
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid4 = lane & 3;
  const uint32_t raw = tc::smem_u32(sm_raw);
  uint8_t* base = sm_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* ring = base + warp * NS * TILE;               // slot s at s * TILE
  float* Pw = reinterpret_cast<float*>(base + NW * NS * TILE) + warp * 8 * 32;
  if (threadIdx.x == 0) {
    for (int w = 0; w < NW; ++w)
      for (int s = 0; s < NS; ++s) tc::mbar_init(&bar[w][s], 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  const int hq = hkv * G;
  const int gw = blockIdx.x * NW + warp, nwarps = gridDim.x * NW;
  const uint64_t kv_policy = tc::policy_evict_first();   // each K/V tile is read once per step
  // A task is one 128-position chunk (work item wi) for one KV head; its
  // record (row, positions, physical blocks) was built on the host.
  struct Rec {
    int row, start, end, nch, kvh, wi, b0, b1, b2, b3;
  };
  auto load_rec = [&](int t) {
    Rec r;
    const int k = t / hkv;                 // position in the (size-ordered) work list
    r.kvh = t - k * hkv;
    const int4* w = reinterpret_cast<const int4*>(work + k);
    const int4 h = w[0], bl = w[1];
    r.row = h.x; r.start = h.y; r.end = h.z; r.nch = h.w & 0xffff;
    r.wi = h.w >> 16;
    r.b0 = bl.x; r.b1 = bl.y; r.b2 = bl.z; r.b3 = bl.w;
    return r;
  };
  auto shfl_rec = [&](const Rec& r) {
    Rec o;
    o.row = __shfl_sync(0xffffffffu, r.row, 0); o.start = __shfl_sync(0xffffffffu, r.start, 0);
    o.end = __shfl_sync(0xffffffffu, r.end, 0); o.kvh = __shfl_sync(0xffffffffu, r.kvh, 0);
    o.nch = __shfl_sync(0xffffffffu, r.nch, 0);
    o.wi = __shfl_sync(0xffffffffu, r.wi, 0); o.b0 = __shfl_sync(0xffffffffu, r.b0, 0);
    o.b1 = __shfl_sync(0xffffffffu, r.b1, 0); o.b2 = __shfl_sync(0xffffffffu, r.b2, 0);
    o.b3 = __shfl_sync(0xffffffffu, r.b3, 0);
    return o;
  };
  // Tasks are handed out dynamically: every warp starts with task gw; later
  // tasks come from the per-launch counter (nwarps + ticket).  A warp holds
  // at most one claimed task beyond the one it is issuing (more would leave
  // whole tasks stranded on some warps at the end), and almost nothing it
  // waits for is a global-memory round trip: the next ticket is claimed when
  // a task starts issuing, its record is loaded at the next copy issue, block
  // ids come with the record, and the next task's query is prefetched into
  // registers.  Which warp computes a task does not change its result.
  // Producer (lane 0 issues the copies; all lanes track the cursor).  The
  // copy sequence is K(0), V(0), K(1), V(1), ... of the warp's tasks' blocks;
  // copy h goes to slot h % NS.
  int p_task = gw, p_blk = 0, p_half = 0;
  Rec pr{};
  uint32_t p_q = 0;
  bool pf_sent = false;
  int q_head = 0, q_tail = 0;              // tasks pushed / popped (warp-uniform)
  int n1 = n_tasks;                        // lane 0: next task id (ticket claimed)
  bool r1_pending = false;                 // its record still to be loaded (warp-uniform)
  bool lazy = false;                       // near the end: claim at the switch, not ahead
  Rec r1{};                                // lane 0: record of n1
  auto push = [&](int t, const Rec& r) {
    if (lane == 0) {
      int4* e = reinterpret_cast<int4*>(&tq[warp][q_head % QN][0]);
      e[0] = make_int4(r.row, r.start, r.end, r.kvh);
      e[1] = make_int4(r.wi, t, r.nch, 0);
    }
    ++q_head;
  };
  auto issue_next = [&]() {
    if (p_task >= n_tasks) {
      // this warp has issued its last K/V load: pull its share of the next
      // GEMM's weights into L2 while the remaining blocks and other warps drain
      if (!pf_sent && lane == 0) tc::pf_issue(pf, gw, nwarps);
      pf_sent = true;
      return;
    }
    if (r1_pending) {                      // the ticket claimed at the last task switch has arrived by now
      if (lane == 0 && n1 < n_tasks) r1 = load_rec(n1);
      r1_pending = false;
      // fewer tickets left than warps: stop claiming ahead, so no warp sits
      // on a task another warp could have run
      lazy = __shfl_sync(0xffffffffu, n1, 0) + nwarps >= n_tasks;
    }
    const int s = p_q % NS;
    if (lane == 0) {
      int blk = p_blk == 0 ? pr.b0 : p_blk == 1 ? pr.b1 : p_blk == 2 ? pr.b2 : pr.b3;
      if (blk < 0 || blk >= n_blocks) { set_err(err, kDevBadBlock); blk = 0; }
      tc::mbar_arrive_expect_tx(&bar[warp][s], TILE);
      tc::bulk_load_hint(ring + s * TILE,
                         reinterpret_cast<const uint8_t*>(pool) + pool_tile(layer, n_blocks, blk, hkv, pr.kvh, p_half, HD) * EB,
                         TILE,
                         &bar[warp][s], kv_policy);
    }
    ++p_q;
    if (p_half == 0) {
      p_half = 1;
      return;
    }
    p_half = 0;
    if (++p_blk == (pr.end - pr.start + 31) >> 5) {
      p_blk = 0;
      if (lazy && !r1_pending && n1 == -1) {
        // claim now (the warp waits two memory round trips, only at the end)
        if (lane == 0) {
          n1 = nwarps + atomicAdd(next_task, 1);
          if (n1 < n_tasks) r1 = load_rec(n1);
        }
      }
      p_task = __shfl_sync(0xffffffffu, n1, 0);
      if (p_task < n_tasks) {
        if (r1_pending) {                  // a one-block task: the record was not loaded yet
          if (lane == 0) r1 = load_rec(n1);
          r1_pending = false;
        }
        pr = shfl_rec(r1);
        push(p_task, pr);
        if (!lazy) {
          if (lane == 0) n1 = nwarps + atomicAdd(next_task, 1);
          r1_pending = true;
        } else {
          n1 = -1;                         // nothing claimed ahead
        }
      }
    }
  };
  pdl_wait();
  TR_MARK1;
  if (p_task < n_tasks) {
    if (lane == 0) n1 = nwarps + atomicAdd(next_task, 1);
    pr = load_rec(p_task);
    push(p_task, pr);
    r1_pending = true;
  }
  for (int i = 0; i < NS; ++i) issue_next();

  // Scores in log2 units: q is pre-scaled by log2(e) / sqrt(hd) and the
  // softmax uses exp2 (partials' maxima are log2-scaled for the merge).
  const float scale = 1.4426950408889634f / sqrtf((float)HD);
  const int mi = lane >> 3, ri = lane & 7;
  // With G <= 4 the MMA's 8 columns hold q hi (columns 0-3) and q lo
  // (columns 4-7) of the group's heads, so one MMA does both halves; column
  // n of a fragment is lane group gid = n: head gid & 3, half gid >> 2.
  // A head's hi and lo sums then sit in lanes tid4 and tid4 ^ 2.  With
  // G = 8, hi and lo take one MMA each.
  constexpr bool PK = G <= 4;
  const int qhead = PK ? (gid & 3) : gid;   // head whose q / P this lane's fragment column carries
  const bool qlo = PK && gid >= 4;          // ... and which half
  uint32_t c_q = 0;
  bool alive = true;
  // the next task's query (raw fp32, this lane's fragment elements)
  float qn[KS][2][2];
  bool qn_valid = false;
  auto load_q = [&](int row, int kvh, float (&d)[KS][2][2]) {
    const float* qrow = q + ((size_t)row * hq + kvh * G) * HD;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int dd = FP8 ? ks * 16 + tid4 * 4 + r * 2 : ks * 16 + r * 8 + tid4 * 2;
        if (qhead < G) {
          const float2 v = *reinterpret_cast<const float2*>(qrow + qhead * HD + dd);
          d[ks][r][0] = v.x;
          d[ks][r][1] = v.y;
        } else {
          d[ks][r][0] = 0.f;
          d[ks][r][1] = 0.f;
        }
      }
  };
  while (alive && q_tail < q_head) {
    __syncwarp();
    const int4 e0 = reinterpret_cast<const int4*>(&tq[warp][q_tail % QN][0])[0];
    const int4 e1 = reinterpret_cast<const int4*>(&tq[warp][q_tail % QN][0])[1];
    ++q_tail;
    struct {
      int row, start, end, kvh, wi, nb, nch;
    } tk{e0.x, e0.y, e0.z, e0.w, e1.x, (e0.z - e0.y + 31) >> 5, e1.z};
    if (!qn_valid) load_q(tk.row, tk.kvh, qn);
    qn_valid = false;
    // q of the group's heads (scaled) as B fragments: packed hi | lo, or
    // separate hi and lo
    uint32_t qh[KS][2], ql[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint32_t h, l;
        if constexpr (FP8) split_pack_h(qn[ks][r][0] * scale, qn[ks][r][1] * scale, h, l);
        else split_pack(qn[ks][r][0] * scale, qn[ks][r][1] * scale, h, l);
        qh[ks][r] = PK ? (qlo ? l : h) : h;
        ql[ks][r] = l;
      }
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[KS][4];
#pragma unroll
    for (int dt = 0; dt < KS; ++dt)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[dt][c] = 0.f;
    for (int b = 0; b < tk.nb; ++b) {
      const int nvalid = min(32, tk.end - (tk.start + b * 32));
      // ---- K tile of block b
      int s = c_q % NS;
      if (!tc::mbar_wait(&bar[warp][s], (c_q / NS) & 1, err, &abort_flag)) { alive = false; break; }
      const uint32_t ks_base = tc::smem_u32(ring + s * TILE);
      // q.K over independent accumulator chains (m-tile x [hi/lo] x k
      // parity) so consecutive MMAs never wait on each other; summed in a
      // fixed order afterwards
      constexpr int HL = PK ? 1 : 2;
      float acc[2][HL][2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hl = 0; hl < HL; ++hl)
#pragma unroll
          for (int par = 0; par < 2; ++par)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[mt][hl][par][c] = 0.f;
      if constexpr (FP8) {
        // one ldmatrix.x4 per m-tile covers 32 dims (two k16 steps):
        // matrices (pos 0-7 | 8-15) x (chunk 2j | 2j + 1)
#pragma unroll
        for (int j = 0; j < KS / 2; ++j) {
          uint32_t w[2][4];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const int r = mt * 16 + (mi & 1) * 8 + ri;
            ldsm_x4(ks_base + k8_off<HD>(r, 2 * j + (mi >> 1)), w[mt][0], w[mt][1], w[mt][2], w[mt][3]);
          }
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int ks = 2 * j + h2;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              const uint32_t a0 = e4m3_lo(w[mt][2 * h2]), a1 = e4m3_lo(w[mt][2 * h2 + 1]);
              const uint32_t a2 = e4m3_hi(w[mt][2 * h2]), a3 = e4m3_hi(w[mt][2 * h2 + 1]);
              mma_f16_16816(acc[mt][0][ks & 1], a0, a1, a2, a3, qh[ks][0], qh[ks][1]);
              if constexpr (!PK) mma_f16_16816(acc[mt][HL - 1][ks & 1], a0, a1, a2, a3, ql[ks][0], ql[ks][1]);
            }
          }
        }
      } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int dc = ks * 16 + (mi >> 1) * 8;
        uint32_t a[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          const int r = mt * 16 + (mi & 1) * 8 + ri;
          ldsm_x4(ks_base + (dc >> 6) * 4096 + swz(r, (dc & 63) >> 3), a[mt][0], a[mt][1], a[mt][2], a[mt][3]);
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          mma_bf16_16816(acc[mt][0][ks & 1], a[mt][0], a[mt][1], a[mt][2], a[mt][3], qh[ks][0], qh[ks][1]);
        if constexpr (!PK) {
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
            mma_bf16_16816(acc[mt][HL - 1][ks & 1], a[mt][0], a[mt][1], a[mt][2], a[mt][3], ql[ks][0], ql[ks][1]);
        }
      }
      }
      __syncwarp();          // every lane's K fragments are in registers
      issue_next();          // refill the K slot NS copies ahead
      ++c_q;
      float sc[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if constexpr (PK) {
            // this lane's column half plus the other half (lane ^ 2)
            const float own = acc[mt][0][0][c] + acc[mt][0][1][c];
            sc[mt][c] = own + __shfl_xor_sync(0xffffffffu, own, 2);
          } else {
            sc[mt][c] = (acc[mt][0][0][c] + acc[mt][0][1][c]) + (acc[mt][HL - 1][0][c] + acc[mt][HL - 1][1][c]);
          }
        }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v[4] = {sc[0][hh], sc[0][hh + 2], sc[1][hh], sc[1][hh + 2]};
        const int pos[4] = {gid, gid + 8, 16 + gid, 24 + gid};
        float bm = -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (pos[i] >= nvalid) v[i] = -INFINITY;
          bm = fmaxf(bm, v[i]);
        }
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        const float mn = fmaxf(m[hh], bm);
        float bs = 0.f;
        const int head = (PK ? (tid4 & 1) : tid4) * 2 + hh;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float pv = pos[i] < nvalid ? exp2f(v[i] - mn) : 0.f;
          bs += pv;
          if (!PK || tid4 < 2) Pw[head * 32 + pos[i]] = pv;
        }
        bs += __shfl_xor_sync(0xffffffffu, bs, 4);
        bs += __shfl_xor_sync(0xffffffffu, bs, 8);
        bs += __shfl_xor_sync(0xffffffffu, bs, 16);
        const float corr = m[hh] == -INFINITY ? 0.f : exp2f(m[hh] - mn);
        l[hh] = l[hh] * corr + bs;
        m[hh] = mn;
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) {
          o[dt][hh] *= corr;
          o[dt][hh + 2] *= corr;
        }
      }
      __syncwarp();
      uint32_t ph[2][2], pl[2][2];
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int j = FP8 ? k2 * 16 + tid4 * 4 + r * 2 : k2 * 16 + r * 8 + tid4 * 2;
          uint32_t h = 0, lo = 0;
          if (qhead < G) {
            if constexpr (FP8) split_pack_h(Pw[qhead * 32 + j], Pw[qhead * 32 + j + 1], h, lo);
            else split_pack(Pw[qhead * 32 + j], Pw[qhead * 32 + j + 1], h, lo);
          }
          ph[k2][r] = PK ? (qlo ? lo : h) : h;
          pl[k2][r] = lo;
        }
      // ---- V tile of block b (rows past the valid positions may hold stale
      // bits: zero them, P is 0 there)
      s = c_q % NS;
      if (!tc::mbar_wait(&bar[warp][s], (c_q / NS) & 1, err, &abort_flag)) { alive = false; break; }
      uint8_t* vt = ring + s * TILE;
      if constexpr (!FP8) {
        for (int i = lane; i < (32 - nvalid) * (HD / 8); i += 32) {
          const int r = nvalid + i / (HD / 8), ch = i % (HD / 8);
          *reinterpret_cast<uint4*>(vt + (ch >> 3) * 4096 + swz(r, ch & 7)) = make_uint4(0, 0, 0, 0);
        }
      }
      // (an FP8 pool is zeroed when created and E4M3 conversions saturate,
      // so a V byte past the valid positions is a finite value times P = 0)
      __syncwarp();
      const uint32_t vs_base = tc::smem_u32(vt);
      // P.V: the KS head-dim tiles are independent chains; issue them
      // interleaved (k2, then hi / lo, then tile) so no MMA waits on the last
      if constexpr (FP8) {
        // V^T rows are head dims: one ldmatrix.x4 per 16-dim tile covers all
        // 32 positions, matrices (dims 0-7 | 8-15) x (positions 0-15 | 16-31)
        uint32_t w4[KS][4];
#pragma unroll
        for (int dt = 0; dt < KS; ++dt)
          ldsm_x4(vs_base + v8_off(dt * 16 + (mi & 1) * 8 + ri, mi >> 1), w4[dt][0], w4[dt][1], w4[dt][2], w4[dt][3]);
        // tiles interleaved so no MMA waits on the previous one
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2)
#pragma unroll
          for (int hl = 0; hl < (PK ? 1 : 2); ++hl)
#pragma unroll
            for (int dt = 0; dt < KS; ++dt) {
              const uint32_t a0 = e4m3_lo(w4[dt][2 * k2]), a1 = e4m3_lo(w4[dt][2 * k2 + 1]);
              const uint32_t a2 = e4m3_hi(w4[dt][2 * k2]), a3 = e4m3_hi(w4[dt][2 * k2 + 1]);
              mma_f16_16816(o[dt], a0, a1, a2, a3, hl ? pl[k2][0] : ph[k2][0], hl ? pl[k2][1] : ph[k2][1]);
            }
      } else
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int r = k2 * 16 + (mi >> 1) * 8 + ri;
        uint32_t a[KS][4];
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) {
          const int dc = dt * 16 + (mi & 1) * 8;
          ldsm_x4_t(vs_base + (dc >> 6) * 4096 + swz(r, (dc & 63) >> 3), a[dt][0], a[dt][1], a[dt][2], a[dt][3]);
        }
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) mma_bf16_16816(o[dt], a[dt][0], a[dt][1], a[dt][2], a[dt][3], ph[k2][0], ph[k2][1]);
        if constexpr (!PK) {
#pragma unroll
          for (int dt = 0; dt < KS; ++dt)
            mma_bf16_16816(o[dt], a[dt][0], a[dt][1], a[dt][2], a[dt][3], pl[k2][0], pl[k2][1]);
        }
      }
      __syncwarp();          // every lane is done with the V slot (and Pw)
      issue_next();          // refill it NS copies ahead
      ++c_q;
      if (!qn_valid && q_tail < q_head) {
        // the next task is known: start loading its query now
        __syncwarp();
        const int4 n0 = reinterpret_cast<const int4*>(&tq[warp][q_tail % QN][0])[0];
        load_q(n0.x, n0.w, qn);
        qn_valid = true;
      }
    }
    if constexpr (PK) {
      // each head's output is its hi-column sum plus its lo-column sum
#pragma unroll
      for (int dt = 0; dt < KS; ++dt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[dt][c] += __shfl_xor_sync(0xffffffffu, o[dt][c], 2);
    }
    if (!alive) break;
    const int nch = tk.nch;
    if (nch == 1) {
      // the row's only chunk: normalise and write the output directly (the
      // merge kernel skips such rows; o * e^0 / (l * e^0) is the same value)
#pragma unroll
      for (int dt = 0; dt < KS; ++dt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int head = tid4 * 2 + (c & 1);
          if (head < G && (!PK || tid4 < 2)) {
            const int dim = dt * 16 + gid + (c >= 2 ? 8 : 0);
            uint16_t hi, lo;
            split_bf16(o[dt][c] / l[c & 1], hi, lo);
            const size_t oi = ((size_t)tk.row * hq + tk.kvh * G + head) * HD + dim;
            out_hi[oi] = hi;
            out_lo[oi] = lo;
          }
        }
      continue;
    }
    // the chunk's partial for the group's heads
#pragma unroll
    for (int dt = 0; dt < KS; ++dt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int head = tid4 * 2 + (c & 1);
        if (head < G && (!PK || tid4 < 2)) {
          const int dim = dt * 16 + gid + (c >= 2 ? 8 : 0);
          part_o[(((size_t)tk.wi * hq + tk.kvh * G + head) * HD) + dim] = o[dt][c];
        }
      }
    if (gid == 0 && (!PK || tid4 < 2)) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int head = tid4 * 2 + hh;
        if (head < G) {
          const size_t h = (size_t)tk.wi * hq + tk.kvh * G + head;
          part_ml[h * 2] = m[hh];
          part_ml[h * 2 + 1] = l[hh];
        }
      }
    }
  }
  TR_MARK2;
  // wind-down after a failed wait: let issued loads land before exiting
  if (!alive) {
    for (uint32_t r = c_q; r < p_q; ++r) {
      int no_abort = 0;
      tc::mbar_wait(&bar[warp][r % NS], (r / NS) & 1, nullptr, &no_abort);
    }
  }
#ifdef CBD_TRACE
  __syncthreads();
#endif
  TR_END(3);
}

// Merge the chunk partials of one (row, KV head) for the group's G heads,
// in chunk order: M = max of the chunk maxima, L = sum_c l_c e^(m_c - M)
// (2^(m_c - M) when the maxima are in log2 units, LOG2),
// O = sum_c o_c e^(m_c - M), output O / L as hi + lo bf16.  One CTA of
// G * HD / 4 threads per (row, KV head), each thread owning 4 dims of one
// head.  The (max, sum) pairs of all chunks are staged in shared memory in
// one pass; the partial outputs are independent loads, issued 8 chunks at
// a time.  Rows with a single chunk were finished by the attention kernel.
}  // namespace cbd
