// Paged grouped-query attention for every row of a step.
//
// A row (slot s, position p) attends to positions 0..p of its slot.  K/V
// live in the paged pool ("20.3 服务、批处理与流式" section 20.3.2: PagedAttention
// splits the KV cache into fixed-size blocks allocated on demand); the row
// reaches its blocks through the slot's block table.  Per (layer, block, KV
// head) the pool holds the K tile and then the V tile (32 positions each),
// each stored in 128-byte-swizzled shared-memory order, so one contiguous
// bulk copy brings a block into shared memory ready for ldmatrix.  Because
// every row's K/V of this layer has been stored by the QKV epilogue before
// this kernel runs, a prefill row sees the earlier rows of its own chunk
// (causal chunked prefill) with no separate mask.
//
// Split-K: each row's positions are cut into fixed 128-position chunks (a
// host-built work list); a chunk is computed for one KV head and the H_q /
// H_kv query heads that share it, keeping an online softmax (running max,
// running sum, unnormalised output).
//
// Three kernels compute the chunks.  attn_stream_kernel (default): every
// warp owns a strided sequence of chunks and streams their blocks through a
// private ring of shared-memory stages.  attn_mma_kernel: one CTA per chunk,
// one block per warp.  Both run q.K and P.V on the tensor cores with
// mma.sync in a swapped form -- positions (or head dims) on the MMA's M
// side, the <= 8 query heads of the KV group on its N side -- with q and P
// split into hi + lo bf16 halves so the products keep ~16 significant bits
// (K and V are bf16 already).  attn_partial_kernel is the CUDA-core
// version.  A second kernel merges the chunks of each (row, head) in chunk
// order and writes the output as hi + lo bf16 halves for the O projection.
// The chunking depends only on the row's position and the merge order is
// fixed, so a row's result does not depend on the other rows of the step or
// on block placement.
#include <algorithm>

#include "attn_stream.cuh"

namespace cbd {

template <int HD, int G>
__global__ void __launch_bounds__(128) attn_partial_kernel(
    const float* __restrict__ q, const uint16_t* __restrict__ pool, const RowDev* __restrict__ rows,
    const int32_t* __restrict__ tables, const AttnWork* __restrict__ work, int layer, int n_blocks,
    int hkv, int mbps, float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* err) {
  constexpr int NW = 4;          // warps
  constexpr int DPL = HD / 32;   // dims per lane in the PV accumulation
  __shared__ __align__(16) float qs[G][HD];
  __shared__ float wm[NW][G], wl[NW][G];
  __shared__ __align__(16) float wo[NW][G][HD];
  pdl_trigger();
  pdl_wait();
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnWork wk = work[blockIdx.x];
  const int wi = wk.wn >> 16;          // the chunk's index among the step's chunks
  const RowDev rw = rows[wk.row];
  const int hq = hkv * G;
  const int end = min(wk.start + kAttnChunk, rw.pos + 1);
  for (int i = threadIdx.x; i < G * HD; i += blockDim.x)
    qs[i / HD][i % HD] = q[((size_t)wk.row * hq + kvh * G) * HD + i];
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)HD);
  float m[G], l[G], o[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[g][e] = 0.f;
  }
  for (int b0 = wk.start + warp * kBlock; b0 < end; b0 += NW * kBlock) {
    const int bi = b0 >> 5;
    const int blk = tables[(size_t)rw.slot * mbps + bi];
    if (blk < 0 || blk >= n_blocks) { set_err(err, kDevBadBlock); break; }
    const int nvalid = min(kBlock, end - b0);
    const uint16_t* Kt = pool + pool_tile(layer, n_blocks, blk, hkv, kvh, 0, HD);
    const uint16_t* Vt = pool + pool_tile(layer, n_blocks, blk, hkv, kvh, 1, HD);
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = 0.f;
    if (lane < nvalid) {
#pragma unroll 4
      for (int c = 0; c < HD / 8; ++c) {
        const uint4 kv = __ldg(reinterpret_cast<const uint4*>(Kt + tile_elem(lane, c * 8)));
        const float kf[8] = {bf16lo_f32(kv.x), bf16hi_f32(kv.x), bf16lo_f32(kv.y), bf16hi_f32(kv.y),
                             bf16lo_f32(kv.z), bf16hi_f32(kv.z), bf16lo_f32(kv.w), bf16hi_f32(kv.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 q0 = *reinterpret_cast<const float4*>(&qs[g][c * 8]);
          const float4 q1 = *reinterpret_cast<const float4*>(&qs[g][c * 8 + 4]);
          float t = s[g];
          t = fmaf(q0.x, kf[0], t); t = fmaf(q0.y, kf[1], t);
          t = fmaf(q0.z, kf[2], t); t = fmaf(q0.w, kf[3], t);
          t = fmaf(q1.x, kf[4], t); t = fmaf(q1.y, kf[5], t);
          t = fmaf(q1.z, kf[6], t); t = fmaf(q1.w, kf[7], t);
          s[g] = t;
        }
      }
    }
    float p[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float sv = lane < nvalid ? s[g] * scale : -INFINITY;
      const float bm = warp_max(sv);
      const float mn = fmaxf(m[g], bm);
      p[g] = lane < nvalid ? expf(sv - mn) : 0.f;
      const float bs = warp_sum(p[g]);
      const float corr = m[g] == -INFINITY ? 0.f : expf(m[g] - mn);
      l[g] = l[g] * corr + bs;
#pragma unroll
      for (int e = 0; e < DPL; ++e) o[g][e] *= corr;
      m[g] = mn;
    }
    for (int j = 0; j < nvalid; ++j) {
      const uint16_t* vr = Vt + tile_elem(j, lane * DPL);
      float vf[DPL];
      if constexpr (DPL == 4) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(vr));
        vf[0] = bf16lo_f32(v.x); vf[1] = bf16hi_f32(v.x); vf[2] = bf16lo_f32(v.y); vf[3] = bf16hi_f32(v.y);
      } else {
        const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(vr));
        vf[0] = bf16lo_f32(v); vf[1] = bf16hi_f32(v);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pj = __shfl_sync(0xffffffffu, p[g], j);
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[g][e] = fmaf(pj, vf[e], o[g][e]);
      }
    }
  }
  // merge the warps in warp order
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) { wm[warp][g] = m[g]; wl[warp][g] = l[g]; }
#pragma unroll
    for (int e = 0; e < DPL; ++e) wo[warp][g][lane * DPL + e] = o[g][e];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * HD; i += blockDim.x) {
    const int g = i / HD, dd = i % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w][g]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float c = wm[w][g] == -INFINITY ? 0.f : expf(wm[w][g] - M);
      L += wl[w][g] * c;
      O += wo[w][g][dd] * c;
    }
    const size_t h = (size_t)wi * hq + kvh * G + g;
    part_o[h * HD + dd] = O;
    if (dd == 0) { part_ml[h * 2] = M; part_ml[h * 2 + 1] = L; }
  }
}

constexpr int kAttnWarps = 4;

template <int HD>
constexpr int attn_mma_smem() {
  return kAttnWarps * 2 * 32 * HD * 2 + kAttnWarps * 8 * 32 * 4 + 1024;
}

template <int HD, int G>
__global__ void __launch_bounds__(128) attn_mma_kernel(const uint16_t* __restrict__ pool,
                                                       const float* __restrict__ q, const RowDev* __restrict__ rows,
                                                       const int32_t* __restrict__ tables,
                                                       const AttnWork* __restrict__ work, int layer, int n_blocks,
                                                       int hkv, int mbps, float* __restrict__ part_o,
                                                       float* __restrict__ part_ml, int32_t* err) {
  static_assert(G >= 1 && G <= 8, "a KV group must fit the MMA's N = 8");
  constexpr int TILE = 32 * HD * 2;       // bytes of one 32-position K or V tile
  constexpr int KS = HD / 16;             // 16-dim steps
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t bar[kAttnWarps];
  __shared__ int abort_flag;
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid4 = lane & 3;
  const uint32_t raw = tc::smem_u32(sm_raw);
  uint8_t* base = sm_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* kt = base + warp * 2 * TILE;   // this warp's K tile, then V tile
  uint8_t* vt = kt + TILE;
  float* Pw = reinterpret_cast<float*>(base + kAttnWarps * 2 * TILE) + warp * 8 * 32;
  const AttnWork wk = work[blockIdx.x];
  const int kvh = blockIdx.y;
  const RowDev rw = rows[wk.row];
  const int hq = hkv * G;
  const int end = min(wk.start + kAttnChunk, rw.pos + 1);
  const int p0 = wk.start + warp * 32;
  int blk = -1;
  if (p0 < end) blk = tables[(size_t)rw.slot * mbps + (p0 >> 5)];
  const bool have = p0 < end && blk >= 0 && blk < n_blocks;
  if (p0 < end && !have && lane == 0) set_err(err, kDevBadBlock);
  const int nvalid = have ? min(32, end - p0) : 0;

  if (threadIdx.x == 0) {
    for (int w = 0; w < kAttnWarps; ++w) tc::mbar_init(&bar[w], 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (have && lane == 0) {
    tc::mbar_arrive_expect_tx(&bar[warp], 2 * TILE);
    tc::bulk_load(kt, pool + pool_tile(layer, n_blocks, blk, hkv, kvh, 0, HD), 2 * TILE, &bar[warp]);
  }
  // q of the group's heads (scaled by 1/sqrt(hd)) as hi / lo B fragments
  const float scale = 1.0f / sqrtf((float)HD);
  uint32_t qh[KS][2], ql[KS][2];
  const float* qrow = q + ((size_t)wk.row * hq + kvh * G) * HD;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int dd = ks * 16 + r * 8 + tid4 * 2;
      float a = 0.f, b = 0.f;
      if (gid < G) {
        a = qrow[gid * HD + dd] * scale;
        b = qrow[gid * HD + dd + 1] * scale;
      }
      split_pack(a, b, qh[ks][r], ql[ks][r]);
    }
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[KS][4];
#pragma unroll
  for (int dt = 0; dt < KS; ++dt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[dt][c] = 0.f;
  bool ok = have;
  if (have) ok = tc::mbar_wait(&bar[warp], 0, err, &abort_flag);
  if (ok) {
    // rows past the valid positions may hold stale bits: zero their V
    for (int i = lane; i < (32 - nvalid) * (HD / 8); i += 32) {
      const int r = nvalid + i / (HD / 8), ch = i % (HD / 8);
      *reinterpret_cast<uint4*>(vt + (ch >> 3) * 4096 + swz(r, ch & 7)) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
    const uint32_t ks_base = tc::smem_u32(kt), vs_base = tc::smem_u32(vt);
    const int mi = lane >> 3, ri = lane & 7;
    // S^T[pos][head] = K q^T
    float sc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[mt][c] = 0.f;
      const int r = mt * 16 + (mi & 1) * 8 + ri;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int dc = ks * 16 + (mi >> 1) * 8;
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ks_base + (dc >> 6) * 4096 + swz(r, (dc & 63) >> 3), a0, a1, a2, a3);
        mma_bf16_16816(sc[mt], a0, a1, a2, a3, qh[ks][0], qh[ks][1]);
        mma_bf16_16816(sc[mt], a0, a1, a2, a3, ql[ks][0], ql[ks][1]);
      }
    }
    // softmax over this block's positions, per head (heads tid4*2, tid4*2+1)
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
      float bs = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float pv = pos[i] < nvalid ? expf(v[i] - bm) : 0.f;
        bs += pv;
        Pw[(tid4 * 2 + hh) * 32 + pos[i]] = pv;
      }
      bs += __shfl_xor_sync(0xffffffffu, bs, 4);
      bs += __shfl_xor_sync(0xffffffffu, bs, 8);
      bs += __shfl_xor_sync(0xffffffffu, bs, 16);
      m[hh] = bm;
      l[hh] = bs;
    }
    __syncwarp();
    // P as hi / lo B fragments: B[pos][head] = P[head][pos]
    uint32_t ph[2][2], pl[2][2];
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = k2 * 16 + r * 8 + tid4 * 2;
        split_pack(Pw[gid * 32 + j], Pw[gid * 32 + j + 1], ph[k2][r], pl[k2][r]);
      }
    // O^T[dim][head] = V^T P^T
#pragma unroll
    for (int dt = 0; dt < KS; ++dt) {
      const int dc = dt * 16 + (mi & 1) * 8;
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int r = k2 * 16 + (mi >> 1) * 8 + ri;
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vs_base + (dc >> 6) * 4096 + swz(r, (dc & 63) >> 3), a0, a1, a2, a3);
        mma_bf16_16816(o[dt], a0, a1, a2, a3, ph[k2][0], ph[k2][1]);
        mma_bf16_16816(o[dt], a0, a1, a2, a3, pl[k2][0], pl[k2][1]);
      }
    }
  }
  // merge the four warps' blocks (fixed warp order) into the chunk's partial
  __syncthreads();
  float* mo = reinterpret_cast<float*>(base);            // [4][8][HD]
  float* mml = mo + kAttnWarps * 8 * HD;                  // [4][8][2]
#pragma unroll
  for (int dt = 0; dt < KS; ++dt)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int head = tid4 * 2 + (c & 1);
      const int dim = dt * 16 + gid + (c >= 2 ? 8 : 0);
      mo[(warp * 8 + head) * HD + dim] = o[dt][c];
    }
  if (gid == 0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      mml[(warp * 8 + tid4 * 2 + hh) * 2] = ok ? m[hh] : -INFINITY;
      mml[(warp * 8 + tid4 * 2 + hh) * 2 + 1] = ok ? l[hh] : 0.f;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * HD; i += blockDim.x) {
    const int g = i / HD, dd = i % HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mml[(w * 8 + g) * 2]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
      const float mw = mml[(w * 8 + g) * 2];
      const float c = mw == -INFINITY ? 0.f : expf(mw - M);
      L += mml[(w * 8 + g) * 2 + 1] * c;
      O += mo[(w * 8 + g) * HD + dd] * c;
    }
    const size_t h = (size_t)(wk.wn >> 16) * hq + kvh * G + g;
    part_o[h * HD + dd] = O;
    if (dd == 0) { part_ml[h * 2] = M; part_ml[h * 2 + 1] = L; }
  }
}

// ---------------------------------------------------------------- streaming
// Persistent form of the tensor-core kernel: eight warps per CTA (two per
// scheduler, so one warp's latencies overlap the other's work), each taking
// tasks (task = one 128-position chunk of one row for one KV head) and
// streaming their 32-position K and V tiles -- as separate 8 KB (hd 128)
// copies, K then V -- through a private ring of NS shared-memory slots
// filled by TMA, running ahead across task boundaries.  Within a task the
// warp keeps an online softmax over its blocks; at the task's end it writes
// the chunk's partial (max, sum, unnormalised output).  No warp waits for
// another.
template <int HD, int G, bool LOG2>
__global__ void attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                    const RowDev* __restrict__ rows, const int32_t* __restrict__ row_work,
                                    const int32_t* __restrict__ comb_rows, int hq, uint16_t* __restrict__ out_hi,
                                    uint16_t* __restrict__ out_lo) {
  extern __shared__ float2 sml[];          // [nch][G] (max, sum)
  TR_DECL;
  pdl_trigger();
  // the listed rows (more than one chunk, and not written by the prefill
  // kernel), or every row when there is no list
  const int r = comb_rows ? comb_rows[blockIdx.x] : (int)blockIdx.x, kvh = blockIdx.y;
  const int w0 = row_work[r], nch = rows[r].pos / kAttnChunk + 1;
  pdl_wait();
  TR_MARK1;
  for (int i = threadIdx.x; i < nch * G; i += blockDim.x) {
    const int c = i / G, g = i - c * G;
    sml[i] = reinterpret_cast<const float2*>(part_ml)[(size_t)(w0 + c) * hq + kvh * G + g];
  }
  __syncthreads();
  constexpr int Q = HD / 4;                // float4s per head
  const int g = threadIdx.x / Q, d4 = threadIdx.x - g * Q;
  float M = -INFINITY;
  for (int c = 0; c < nch; ++c) M = fmaxf(M, sml[c * G + g].x);
  float L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* po = reinterpret_cast<const float4*>(part_o) + ((size_t)w0 * hq + kvh * G + g) * Q + d4;
  const size_t cstride = (size_t)hq * Q;   // float4s between consecutive chunks
  // up to 32 chunks' partials in flight at once (one memory round trip for
  // rows up to 4096 positions), then accumulated in chunk order
  constexpr int CB = 32;
  for (int c0 = 0; c0 < nch; c0 += CB) {
    float4 v[CB];
#pragma unroll
    for (int j = 0; j < CB; ++j)
      if (c0 + j < nch) v[j] = po[(size_t)(c0 + j) * cstride];
#pragma unroll
    for (int j = 0; j < CB; ++j)
      if (c0 + j < nch) {
        const float2 ml = sml[(c0 + j) * G + g];
        const float sc = LOG2 ? exp2f(ml.x - M) : expf(ml.x - M);
        L += ml.y * sc;
        O.x += v[j].x * sc; O.y += v[j].y * sc; O.z += v[j].z * sc; O.w += v[j].w * sc;
      }
  }
  const float o4[4] = {O.x / L, O.y / L, O.z / L, O.w / L};
  uint16_t hi[4], lo[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) split_bf16(o4[j], hi[j], lo[j]);
  const size_t oi = ((size_t)r * hq + kvh * G + g) * HD + d4 * 4;
  *reinterpret_cast<uint2*>(out_hi + oi) = make_uint2(hi[0] | ((uint32_t)hi[1] << 16), hi[2] | ((uint32_t)hi[3] << 16));
  *reinterpret_cast<uint2*>(out_lo + oi) = make_uint2(lo[0] | ((uint32_t)lo[1] << 16), lo[2] | ((uint32_t)lo[3] << 16));
  TR_END(4);
}

// Prefill runs go to the prefill attention kernel (streaming path).
static bool uses_prefill_kernel(const cbd_engine* e, const cbd_batch* b) {
  return e->attn_path == 0 && e->prefill_attn && b->n_pfb > 0;
}

// Rows the merge kernel combines: on the streaming path the listed rows with
// more than one chunk (those outside prefill runs when the prefill kernel
// writes the runs); on the other paths every row (they write partials only).
static int merge_rows(const cbd_engine* e, const cbd_batch* b) {
  if (e->attn_path != 0) return b->n_rows;
  return uses_prefill_kernel(e, b) ? b->n_comb_dec : b->n_comb_all;
}

int attention_launches(const cbd_engine* e, const cbd_batch* b) {
  if (e->attn_path != 0) return 1 + (merge_rows(e, b) > 0 ? 1 : 0);
  const bool pf = uses_prefill_kernel(e, b);
  return ((pf ? b->n_dec : b->n_work) > 0 ? 1 : 0) + (pf ? 1 : 0) + (merge_rows(e, b) > 0 ? 1 : 0);
}

template <int HD, int G>
static cudaError_t launch_attn_t(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                                 const PfSpec& pf, cudaStream_t s) {
  const Dims& dm = e->dm;
  if (e->kv_fp8) {
    if (e->attn_path != 0) return cudaErrorNotSupported;
    cudaError_t ce = launch_attn_stream_fp8(e, p, b, layer, uses_prefill_kernel(e, b) ? b->n_dec : b->n_work, pf, s);
    if (ce != cudaSuccess) return ce;
    if (uses_prefill_kernel(e, b)) {
      ce = launch_attn_prefill(e, p, b, layer, s);
      if (ce != cudaSuccess) return ce;
    }
  } else if (e->attn_path == 0) {
    constexpr int smem = attn_stream_smem<HD>();
    static DeviceOnce attr;
    {
      const cudaError_t ce = set_smem_once(attr, attn_stream_kernel<HD, G>, smem);
      if (ce != cudaSuccess) return ce;
    }
    // with the prefill kernel, the streaming kernel takes the items of rows
    // outside prefill runs (they come first in the list)
    const int n_tasks = (uses_prefill_kernel(e, b) ? b->n_dec : b->n_work) * dm.hkv;
    if (n_tasks > 0) {
      const int grid = std::min(e->sm_count, (n_tasks + kStreamWarps - 1) / kStreamWarps);
      cudaError_t ce = launch_pdl(attn_stream_kernel<HD, G>, dim3(grid), dim3(kStreamWarps * 32), smem, s,
                                  (const uint16_t*)p->base,
                                  (const float*)e->q, (const RowDev*)b->rows, (const int32_t*)b->tables,
                                  (const AttnWork*)b->work, (const int32_t*)b->row_work, n_tasks, layer,
                                  p->n_blocks, dm.hkv, dm.max_blocks_per_seq, e->attn_o, e->attn_ml, e->act_hi,
                                  e->act_lo, e->attn_next + layer, pf, e->err);
      if (ce != cudaSuccess) return ce;
    }
    if (uses_prefill_kernel(e, b)) {
      cudaError_t ce = launch_attn_prefill(e, p, b, layer, s);
      if (ce != cudaSuccess) return ce;
    }
  } else if (e->attn_path == 2) {
    constexpr int smem = attn_mma_smem<HD>();
    static DeviceOnce attr;
    {
      const cudaError_t ce = set_smem_once(attr, attn_mma_kernel<HD, G>, smem);
      if (ce != cudaSuccess) return ce;
    }
    cudaError_t ce = launch_pdl(attn_mma_kernel<HD, G>, dim3(b->n_work, dm.hkv), dim3(128), smem, s,
                                (const uint16_t*)p->base, (const float*)e->q, (const RowDev*)b->rows, (const int32_t*)b->tables,
                                (const AttnWork*)b->work, layer, p->n_blocks, dm.hkv, dm.max_blocks_per_seq,
                                e->attn_o, e->attn_ml, e->err);
    if (ce != cudaSuccess) return ce;
  } else {
    cudaError_t ce = launch_pdl(attn_partial_kernel<HD, G>, dim3(b->n_work, dm.hkv), dim3(128), 0, s,
                                (const float*)e->q, (const uint16_t*)p->base, (const RowDev*)b->rows,
                                (const int32_t*)b->tables, (const AttnWork*)b->work, layer, p->n_blocks, dm.hkv,
                                dm.max_blocks_per_seq, e->attn_o, e->attn_ml, e->err);
    if (ce != cudaSuccess) return ce;
  }
  // the streaming kernels write single-chunk rows themselves (and the
  // prefill kernel its runs); the other paths write partials only.  The
  // streaming kernels keep their maxima in log2 units (exp2 softmax).
  const size_t csmem = (size_t)b->max_chunks * G * sizeof(float2);
  auto combine = e->attn_path == 0 ? attn_combine_kernel<HD, G, true> : attn_combine_kernel<HD, G, false>;
  if (csmem > 48 * 1024) {
    cudaError_t ce = cudaFuncSetAttribute(combine, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem);
    if (ce != cudaSuccess) return ce;
  }
  const int nm = merge_rows(e, b);
  if (nm <= 0) return cudaSuccess;
  return launch_pdl(combine, dim3(nm, dm.hkv), dim3(G * HD / 4), csmem, s, (const float*)e->attn_o,
                    (const float*)e->attn_ml, (const RowDev*)b->rows, (const int32_t*)b->row_work,
                    e->attn_path == 0 ? (const int32_t*)b->comb_rows : (const int32_t*)nullptr, dm.hq, e->act_hi,
                    e->act_lo);
}

cudaError_t launch_attention(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                             const PfSpec& pf, cudaStream_t s) {
  const int G = e->dm.hq / e->dm.hkv;
  const int HD = e->dm.hd;
  if (HD == 64 && G == 1) return launch_attn_t<64, 1>(e, p, b, layer, pf, s);
  if (HD == 64 && G == 2) return launch_attn_t<64, 2>(e, p, b, layer, pf, s);
  if (HD == 64 && G == 4) return launch_attn_t<64, 4>(e, p, b, layer, pf, s);
  if (HD == 64 && G == 8) return launch_attn_t<64, 8>(e, p, b, layer, pf, s);
  if (HD == 128 && G == 1) return launch_attn_t<128, 1>(e, p, b, layer, pf, s);
  if (HD == 128 && G == 2) return launch_attn_t<128, 2>(e, p, b, layer, pf, s);
  if (HD == 128 && G == 4) return launch_attn_t<128, 4>(e, p, b, layer, pf, s);
  if (HD == 128 && G == 8) return launch_attn_t<128, 8>(e, p, b, layer, pf, s);
  return cudaErrorInvalidValue;
}

CBD_TRACE_BIND(attn)

}  // namespace cbd
