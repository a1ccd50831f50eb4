// Attention for the prompt rows of a prefill chunk ("20.3 服务、批处理与流式"
// section 20.3.2: chunked prefill; "大模型推理为什么需要 Continuous Batching"
// section 2.2: prefill is compute-bound).  The rows of a chunk are
// consecutive positions of one sequence and read the same K/V blocks, so
// instead of one task per row (the streaming kernel's decode layout, where
// every row streams its blocks again) a CTA takes a block of consecutive
// query positions of one sequence for one KV head and streams each K/V block
// once for all of them:
//
//   * M = 64 query rows (BQ = 64 / G positions x the G query heads of the
//     KV head), 16 per consumer warp, on mma.sync m16n8k16;
//   * S = q K^T over a 32-position block (q split into bf16 hi + lo, scaled
//     to log2 units; f16 hi + lo over E4M3 K/V), causal mask (key position
//     <= query position), online softmax in exp2, then O += P V with P split
//     the same way -- the streaming kernel's arithmetic, summed in another
//     order (one pass over the row's blocks instead of 128-position chunks
//     merged afterwards);
//   * each consumer warp keeps its 16 rows of q in shared memory and reads
//     them back as ldmatrix A fragments (registers hold the output);
//   * one producer warp copies each block's K and V tiles (one contiguous
//     run in the pool) into a ring of stages; the consumer warps release a
//     stage once all four have used it.
//
// A row's whole context is one pass, so its output goes straight to the
// O-projection's input (split into bf16 hi + lo), with no partials.
#include <algorithm>

#include "attn_stream.cuh"

namespace cbd {

constexpr int kPfQRows = 64;                 // query rows (position x head) per CTA
constexpr int kPfWarps = kPfQRows / 16;      // consumer warps
constexpr int kPfStages = 4;
// K/V ring, then the consumer warps' q tiles (16 rows x HD, hi and lo)
template <int HD, bool FP8>
__host__ __device__ constexpr int pf_smem() {
  return kPfStages * 2 * (32 * HD * (FP8 ? 1 : 2)) + kPfWarps * 2 * 16 * HD * 2 + 128;
}

// FP8 = true: K and V are E4M3 bytes (K tiles [position][dim], V tiles
// transposed [dim][position], 16-byte chunks swizzled per row), converted
// exactly to f16 in registers; q and P are split into f16 hi + lo and the
// products are f16 MMAs.  An ldmatrix over byte pairs gives a lane 4
// consecutive bytes of a row, so the MMA's k index is permuted -- k pair
// (2t, 2t+1) takes bytes 4t, 4t+1 of the 16-byte chunk and (2t+8, 2t+9)
// bytes 4t+2, 4t+3 -- on both operands of each product: q is stored in that
// dim order, and the key rows of each q.K n-tile are loaded in the order that
// puts P's C fragment directly into the A fragment P.V needs (n-tile 2kk + h
// holds keys kk*16 + 4 (n >> 1) + 2 h + (n & 1), n = 0..7).
template <int HD, int G, bool FP8>
__global__ void __launch_bounds__((kPfWarps + 1) * 32, 2) attn_prefill_kernel(
    const uint16_t* __restrict__ pool, const float* __restrict__ q, const PfBlock* __restrict__ blocks,
    const int32_t* __restrict__ pf_rows, const int32_t* __restrict__ tables, int layer, int n_blocks, int hkv, int mbps, uint16_t* __restrict__ out_hi,
    uint16_t* __restrict__ out_lo, int32_t* err) {
  static_assert(kPfQRows % G == 0, "a position's heads share a warp");
  constexpr int TILE = 32 * HD * (FP8 ? 1 : 2);    // bytes of one K (or V) tile
  constexpr int KS = HD / 16;                // k-steps of q.K
  constexpr int DT = HD / 8;                 // n-tiles of P.V
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t full[kPfStages], empty[kPfStages];
  __shared__ int abort_flag;
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = tc::smem_u32(sm_raw);
  uint8_t* ring = sm_raw + (((raw + 127u) & ~127u) - raw);
  const PfBlock blk = blocks[blockIdx.x / hkv];
  const int kvh = (int)blockIdx.x % hkv;
  const int hq = hkv * G;
  const int nkeys = blk.pos0 + blk.npos;     // keys 0 .. nkeys - 1 (causal: the last row sees them all)
  const int ntiles = (nkeys + 31) >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], kPfWarps);
    }
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();                                // q and this step's K/V come from the previous kernels

  if (warp == kPfWarps) {
    // ------------------------------------------------ producer: K | V of block j -> stage j % kPfStages
    if (lane == 0) {
      const uint8_t* pb = reinterpret_cast<const uint8_t*>(pool);
      int j = 0;
      for (; j < ntiles; ++j) {
        const int s = j % kPfStages;
        if (j >= kPfStages && !tc::mbar_wait(&empty[s], ((j / kPfStages) & 1) ^ 1, err, &abort_flag)) break;
        int b = tables[(size_t)blk.slot * mbps + j];
        if (b < 0 || b >= n_blocks) {
          set_err(err, kDevBadBlock);
          b = 0;
        }
        tc::mbar_arrive_expect_tx(&full[s], 2 * TILE);
        tc::bulk_load(ring + s * 2 * TILE, pb + pool_tile(layer, n_blocks, b, hkv, kvh, 0, HD) * (FP8 ? 1 : 2),
                      2 * TILE, &full[s]);
      }
      if (j < ntiles) {     // gave up: the copies in flight land before the CTA exits
        for (int r = j > kPfStages ? j - kPfStages : 0; r < j; ++r) {
          int no_abort = 0;
          tc::mbar_wait(&full[r % kPfStages], (r / kPfStages) & 1, nullptr, &no_abort);
        }
      }
    }
    return;
  }

  // ------------------------------------------------ consumers: 16 query rows each
  const int gid = lane >> 2, tid4 = lane & 3;
  // MMA rows gid and gid + 8 of this warp: row m -> (position m / G, head m % G)
  int lp[2], hh[2], qpos[2], row[2];
  bool valid[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int mrow = warp * 16 + gid + 8 * i;
    lp[i] = mrow / G;
    hh[i] = mrow - lp[i] * G;
    valid[i] = lp[i] < blk.npos;
    // a row past the block's positions computes over every key and is not stored
    qpos[i] = valid[i] ? blk.pos0 + lp[i] : nkeys - 1;
    row[i] = valid[i] ? pf_rows[blk.idx0 + lp[i]] : 0;
  }
  // q (scaled to log2 units), split into bf16 hi and lo, into this warp's
  // shared tiles [16 rows][HD] (16-byte chunk c of row r at c ^ (r & 7));
  // the q.K loop reads them back as A fragments with ldmatrix
  const float scale = 1.4426950408889634f / sqrtf((float)HD);
  uint8_t* qt = ring + kPfStages * 2 * TILE + warp * 2 * (16 * HD * 2);
  const uint32_t qhb = tc::smem_u32(qt), qlb = qhb + 16 * HD * 2;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int f = 0; f < 4; ++f) {
      const int i = f & 1;                               // fragment rows gid and gid + 8
      // fragment k position ks*16 + (f >> 1) * 8 + tid4 * 2 (+1) holds that dim,
      // or for FP8 dims ks*16 + 4 tid4 + 2 (f >> 1) (+1)
      const int d = ks * 16 + (f >> 1) * 8 + tid4 * 2;
      const int dq = FP8 ? ks * 16 + tid4 * 4 + (f >> 1) * 2 : d;
      float2 v = make_float2(0.f, 0.f);
      if (valid[i])
        v = *reinterpret_cast<const float2*>(q + ((size_t)row[i] * hq + kvh * G + hh[i]) * HD + dq);
      uint32_t h, l;
      if constexpr (FP8) split_pack_h(v.x * scale, v.y * scale, h, l);
      else split_pack(v.x * scale, v.y * scale, h, l);
      const int rr = gid + 8 * i, chq = d >> 3;
      const uint32_t off = (uint32_t)(rr * HD * 2 + ((chq ^ (rr & 7)) << 4) + tid4 * 4);
      *reinterpret_cast<uint32_t*>(qt + off) = h;
      *reinterpret_cast<uint32_t*>(qt + 16 * HD * 2 + off) = l;
    }
  __syncwarp();
  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float o[DT][4];
#pragma unroll
  for (int dt = 0; dt < DT; ++dt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[dt][c] = 0.f;
  const int mi = lane >> 3, r8 = lane & 7;              // ldmatrix: this lane's matrix and row

  for (int j = 0; j < ntiles; ++j) {
    const int s = j % kPfStages;
    if (!tc::mbar_wait(&full[s], (j / kPfStages) & 1, err, &abort_flag)) break;
    const uint32_t kb = tc::smem_u32(ring + s * 2 * TILE), vb = kb + TILE;
    const int nv = min(32, nkeys - j * 32);      // positions of this block inside the sequence
    // ---- S = q K^T: 4 n-tiles of 8 key positions; the q hi and q lo
    // products accumulate in separate chains (so consecutive MMAs do not
    // wait on each other) and are added once, in a fixed order
    float sc[4][4], sl[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        sc[nt][c] = 0.f;
        sl[nt][c] = 0.f;
      }
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      // q's A fragments for dims ks*16 .. +15: matrices (rows 0-7, dims 0-7),
      // (rows 8-15, dims 0-7), (rows 0-7, dims 8-15), (rows 8-15, dims 8-15)
      uint32_t ah[4], al[4];
      {
        const int rq = (mi & 1) * 8 + r8, cq = ks * 2 + (mi >> 1);
        const uint32_t oq = (uint32_t)(rq * HD * 2 + ((cq ^ (rq & 7)) << 4));
        ldsm_x4(qhb + oq, ah[0], ah[1], ah[2], ah[3]);
        ldsm_x4(qlb + oq, al[0], al[1], al[2], al[3]);
      }
      if constexpr (FP8) {
        // matrix mi = n-tile mi: 8 key rows (permuted), the 16-byte chunk of dims ks*16..
        const int key = (mi >> 1) * 16 + 4 * (r8 >> 1) + 2 * (mi & 1) + (r8 & 1);
        uint32_t kr[4];
        ldsm_x4(kb + k8_off<HD>(key, ks), kr[0], kr[1], kr[2], kr[3]);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const uint32_t b0 = e4m3_lo(kr[nt]), b1 = e4m3_hi(kr[nt]);
          mma_f16_16816(sc[nt], ah[0], ah[1], ah[2], ah[3], b0, b1);
          mma_f16_16816(sl[nt], al[0], al[1], al[2], al[3], b0, b1);
        }
      } else {
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        // matrices: (n-tile 2np, dims ks*16 + 0..7), (2np, +8..15), (2np+1, +0..7), (2np+1, +8..15)
        const int r = (2 * np + (mi >> 1)) * 8 + r8;
        const int ch = ks * 2 + (mi & 1);
        uint32_t b0a, b1a, b0b, b1b;
        ldsm_x4(kb + (ch >> 3) * 4096 + swz(r, ch & 7), b0a, b1a, b0b, b1b);
        mma_bf16_16816(sc[2 * np], ah[0], ah[1], ah[2], ah[3], b0a, b1a);
        mma_bf16_16816(sl[2 * np], al[0], al[1], al[2], al[3], b0a, b1a);
        mma_bf16_16816(sc[2 * np + 1], ah[0], ah[1], ah[2], ah[3], b0b, b1b);
        mma_bf16_16816(sl[2 * np + 1], al[0], al[1], al[2], al[3], b0b, b1b);
      }
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[nt][c] += sl[nt][c];
    // ---- causal mask and online softmax (rows gid: c = 0, 1; gid + 8: c = 2, 3)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int kp = FP8 ? j * 32 + (nt >> 1) * 16 + tid4 * 4 + (nt & 1) * 2 + (c & 1)
                           : j * 32 + nt * 8 + tid4 * 2 + (c & 1);
        if (kp > qpos[c >> 1]) sc[nt][c] = -INFINITY;
        mx[c >> 1] = fmaxf(mx[c >> 1], sc[nt][c]);
      }
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      const float mn = fmaxf(m_r[i], mx[i]);          // finite: key 0 is in every row's first block
      alpha[i] = exp2f(m_r[i] - mn);
      m_r[i] = mn;
      l_r[i] *= alpha[i];
    }
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      o[dt][0] *= alpha[0]; o[dt][1] *= alpha[0];
      o[dt][2] *= alpha[1]; o[dt][3] *= alpha[1];
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float p = exp2f(sc[nt][c] - m_r[c >> 1]);   // masked: exp2(-inf) = 0
        sc[nt][c] = p;
        l_r[c >> 1] += p;
      }
    // ---- O += P V: two k-steps of 16 key positions
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t ph[4], pl[4];
      if constexpr (FP8) {
        split_pack_h(sc[2 * kk][0], sc[2 * kk][1], ph[0], pl[0]);
        split_pack_h(sc[2 * kk][2], sc[2 * kk][3], ph[1], pl[1]);
        split_pack_h(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[2], pl[2]);
        split_pack_h(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[3], pl[3]);
        // V tile rows are dims: matrix mi = dim tile 4 dq + mi, the 16-byte
        // chunk of positions kk*16..; lane bytes 0,1 / 2,3 are keys
        // kk*16 + 4 tid4 + 0,1 / + 2,3
        const int k0 = kk * 16 + tid4 * 4;
        const uint32_t m0 = (k0 < nv ? 0xffffu : 0u) | (k0 + 1 < nv ? 0xffff0000u : 0u);
        const uint32_t m1 = (k0 + 2 < nv ? 0xffffu : 0u) | (k0 + 3 < nv ? 0xffff0000u : 0u);
#pragma unroll
        for (int dq = 0; dq < DT / 4; ++dq) {
          uint32_t vr[4];
          ldsm_x4(vb + v8_off((4 * dq + mi) * 8 + r8, kk), vr[0], vr[1], vr[2], vr[3]);
#pragma unroll
          for (int t4 = 0; t4 < 4; ++t4) {
            // past the sequence (stale pool bytes): zero, since P is 0 there
            const uint32_t b0 = e4m3_lo(vr[t4]) & m0, b1 = e4m3_hi(vr[t4]) & m1;
            mma_f16_16816(o[4 * dq + t4], ph[0], ph[1], ph[2], ph[3], b0, b1);
            mma_f16_16816(o[4 * dq + t4], pl[0], pl[1], pl[2], pl[3], b0, b1);
          }
        }
      } else {
      split_pack(sc[2 * kk][0], sc[2 * kk][1], ph[0], pl[0]);
      split_pack(sc[2 * kk][2], sc[2 * kk][3], ph[1], pl[1]);
      split_pack(sc[2 * kk + 1][0], sc[2 * kk + 1][1], ph[2], pl[2]);
      split_pack(sc[2 * kk + 1][2], sc[2 * kk + 1][3], ph[3], pl[3]);
#pragma unroll
      for (int dp = 0; dp < DT / 2; ++dp) {
        // transposed matrices: (keys kk*16 + 0..7, dims dp*16 + 0..7), (keys +8..15, same dims),
        // (keys +0..7, dims +8..15), (keys +8..15, dims +8..15)
        const int r = kk * 16 + (mi & 1) * 8 + r8;
        const int ch = dp * 2 + (mi >> 1);
        uint32_t b0a, b1a, b0b, b1b;
        ldsm_x4_t(vb + (ch >> 3) * 4096 + swz(r, ch & 7), b0a, b1a, b0b, b1b);
        if (nv < 32) {
          // V rows past the sequence (stale pool contents) are zeroed in the
          // fragments: P is 0 there, and 0 times a stale value must stay 0
          const int k0 = kk * 16 + tid4 * 2;
          const uint32_t m0 = (k0 < nv ? 0xffffu : 0u) | (k0 + 1 < nv ? 0xffff0000u : 0u);
          const uint32_t m1 = (k0 + 8 < nv ? 0xffffu : 0u) | (k0 + 9 < nv ? 0xffff0000u : 0u);
          b0a &= m0; b0b &= m0;
          b1a &= m1; b1b &= m1;
        }
        mma_bf16_16816(o[2 * dp], ph[0], ph[1], ph[2], ph[3], b0a, b1a);
        mma_bf16_16816(o[2 * dp], pl[0], pl[1], pl[2], pl[3], b0a, b1a);
        mma_bf16_16816(o[2 * dp + 1], ph[0], ph[1], ph[2], ph[3], b0b, b1b);
        mma_bf16_16816(o[2 * dp + 1], pl[0], pl[1], pl[2], pl[3], b0b, b1b);
      }
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&empty[s]);
  }
  // ---- O / l -> bf16 hi + lo at [row][head][dim]
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 1);
    l_r[i] += __shfl_xor_sync(0xffffffffu, l_r[i], 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!valid[i]) continue;
    const float inv = 1.f / l_r[i];
    const size_t ob = ((size_t)row[i] * hq + kvh * G + hh[i]) * HD + tid4 * 2;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      uint32_t h, l;
      split_pack(o[dt][2 * i] * inv, o[dt][2 * i + 1] * inv, h, l);
      *reinterpret_cast<uint32_t*>(out_hi + ob + dt * 8) = h;
      *reinterpret_cast<uint32_t*>(out_lo + ob + dt * 8) = l;
    }
  }
}

template <int HD, int G, bool FP8>
static cudaError_t launch_pf_t(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                               cudaStream_t s) {
  constexpr int smem = pf_smem<HD, FP8>();
  static DeviceOnce attr;
  {
    const cudaError_t ce = set_smem_once(attr, attn_prefill_kernel<HD, G, FP8>, smem);
    if (ce != cudaSuccess) return ce;
  }
  const Dims& dm = e->dm;
  return launch_pdl(attn_prefill_kernel<HD, G, FP8>, dim3(b->n_pfb * dm.hkv), dim3((kPfWarps + 1) * 32), smem, s,
                    (const uint16_t*)p->base, (const float*)e->q, (const PfBlock*)b->pfb,
                    (const int32_t*)b->pf_rows, (const int32_t*)b->tables, layer, p->n_blocks, dm.hkv,
                    dm.max_blocks_per_seq, e->act_hi, e->act_lo, e->err);
}

template <bool FP8>
static cudaError_t launch_pf_kv(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                                cudaStream_t s) {
  const int G = e->dm.hq / e->dm.hkv;
  const int HD = e->dm.hd;
  if (HD == 64 && G == 1) return launch_pf_t<64, 1, FP8>(e, p, b, layer, s);
  if (HD == 64 && G == 2) return launch_pf_t<64, 2, FP8>(e, p, b, layer, s);
  if (HD == 64 && G == 4) return launch_pf_t<64, 4, FP8>(e, p, b, layer, s);
  if (HD == 64 && G == 8) return launch_pf_t<64, 8, FP8>(e, p, b, layer, s);
  if (HD == 128 && G == 1) return launch_pf_t<128, 1, FP8>(e, p, b, layer, s);
  if (HD == 128 && G == 2) return launch_pf_t<128, 2, FP8>(e, p, b, layer, s);
  if (HD == 128 && G == 4) return launch_pf_t<128, 4, FP8>(e, p, b, layer, s);
  if (HD == 128 && G == 8) return launch_pf_t<128, 8, FP8>(e, p, b, layer, s);
  return cudaErrorInvalidValue;
}

int prefill_block_positions(int G) { return kPfQRows / G; }

cudaError_t launch_attn_prefill(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                                cudaStream_t s) {
  if (b->n_pfb <= 0) return cudaSuccess;
  return e->kv_fp8 ? launch_pf_kv<true>(e, p, b, layer, s) : launch_pf_kv<false>(e, p, b, layer, s);
}

}  // namespace cbd
