// Paged grouped-query attention for every row of a step.
//
// A row (slot s, position p) attends to positions 0..p of its slot.  K/V
// live in the paged pool ("20.3 服务、批处理与流式" section 20.3.2: PagedAttention
// splits the KV cache into fixed-size blocks allocated on demand); the row
// reaches its blocks through the slot's block table, one 32-position tile
// per (layer, K|V, block, KV head).  Because every row's K/V of this layer
// has been stored by the QKV epilogue before this kernel runs, a prefill row
// sees the earlier rows of its own chunk (causal chunked prefill) with no
// separate mask.
//
// Split-K: each row's positions are cut into fixed 256-position chunks (a
// host-built work list); one CTA handles one (chunk, KV head) for the H_q /
// H_kv query heads that share the KV head, keeping an online softmax
// (running max, running sum, unnormalised output).  A second kernel merges
// the chunks of each (row, head) in chunk order and writes the output as
// hi + lo bf16 halves for the O projection.  The chunking depends only on
// the row's position, and the merge order is fixed, so a row's result does
// not depend on the other rows of the step or on block placement.
#include "common.cuh"

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
  const int wi = blockIdx.x, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const AttnWork wk = work[wi];
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
    const uint16_t* Kt = pool + pool_off(layer, 0, n_blocks, blk, hkv, kvh, HD, 0, 0);
    const uint16_t* Vt = pool + pool_off(layer, 1, n_blocks, blk, hkv, kvh, HD, 0, 0);
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = 0.f;
    if (lane < nvalid) {
      const uint4* kr = reinterpret_cast<const uint4*>(Kt + (size_t)lane * HD);
#pragma unroll 4
      for (int c = 0; c < HD / 8; ++c) {
        const uint4 kv = __ldg(kr + c);
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
      const uint16_t* vr = Vt + (size_t)j * HD + lane * DPL;
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

// Merge a row's chunks for one head (chunk order), normalise, split.
template <int HD>
__global__ void attn_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                    const int32_t* __restrict__ row_work, int hq,
                                    uint16_t* __restrict__ out_hi, uint16_t* __restrict__ out_lo) {
  const int r = blockIdx.x, h = blockIdx.y, dd = threadIdx.x;
  const int w0 = row_work[r], w1 = row_work[r + 1];
  float M = -INFINITY;
  for (int w = w0; w < w1; ++w) M = fmaxf(M, part_ml[((size_t)w * hq + h) * 2]);
  float L = 0.f, O = 0.f;
  for (int w = w0; w < w1; ++w) {
    const size_t i = (size_t)w * hq + h;
    const float c = expf(part_ml[i * 2] - M);
    L += part_ml[i * 2 + 1] * c;
    O += part_o[i * HD + dd] * c;
  }
  uint16_t hi, lo;
  split_bf16(O / L, hi, lo);
  const size_t o = ((size_t)r * hq + h) * HD + dd;
  out_hi[o] = hi;
  out_lo[o] = lo;
}

template <int HD, int G>
static cudaError_t launch_attn_t(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                                 cudaStream_t s) {
  const Dims& dm = e->dm;
  attn_partial_kernel<HD, G><<<dim3(b->n_work, dm.hkv), 128, 0, s>>>(
      e->q, p->base, b->rows, b->tables, b->work, layer, p->n_blocks, dm.hkv, dm.max_blocks_per_seq,
      e->attn_o, e->attn_ml, e->err);
  attn_combine_kernel<HD><<<dim3(b->n_rows, dm.hq), HD, 0, s>>>(e->attn_o, e->attn_ml, b->row_work, dm.hq,
                                                                 e->act_hi, e->act_lo);
  return cudaGetLastError();
}

cudaError_t launch_attention(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                             cudaStream_t s) {
  const int G = e->dm.hq / e->dm.hkv;
  const int HD = e->dm.hd;
  if (HD == 64 && G == 1) return launch_attn_t<64, 1>(e, p, b, layer, s);
  if (HD == 64 && G == 2) return launch_attn_t<64, 2>(e, p, b, layer, s);
  if (HD == 64 && G == 4) return launch_attn_t<64, 4>(e, p, b, layer, s);
  if (HD == 64 && G == 8) return launch_attn_t<64, 8>(e, p, b, layer, s);
  if (HD == 128 && G == 1) return launch_attn_t<128, 1>(e, p, b, layer, s);
  if (HD == 128 && G == 2) return launch_attn_t<128, 2>(e, p, b, layer, s);
  if (HD == 128 && G == 4) return launch_attn_t<128, 4>(e, p, b, layer, s);
  if (HD == 128 && G == 8) return launch_attn_t<128, 8>(e, p, b, layer, s);
  return cudaErrorInvalidValue;
}

}  // namespace cbd
