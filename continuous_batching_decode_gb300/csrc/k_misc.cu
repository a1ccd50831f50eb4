// Embedding gather and RMSNorm (with the hi/lo bf16 split of its output).
#include <algorithm>

#include "common.cuh"

namespace cbd {

// x[r][:] = E[token_r][:] as fp32 (the residual stream starts at the
// embedding row of the row's token).
// CTA 0 also zeroes the step's per-layer attention task counters (every
// kernel of the previous step has completed once this kernel passes its
// dependency wait).
// With g != null (fused RMSNorm of layer 0) it also writes split(x * g) to
// norm_hi / norm_lo and the row's sum of x^2 (per-thread sums, then a fixed
// tree) as the row's only partial in ssq.
__global__ void embed_kernel(const uint16_t* __restrict__ E, const RowDev* __restrict__ rows, int d,
                             float* __restrict__ x, int32_t* __restrict__ attn_next, int n_layers,
                             const float* __restrict__ g, uint16_t* __restrict__ norm_hi,
                             uint16_t* __restrict__ norm_lo, float* __restrict__ ssq) {
  __shared__ float red[32];
  TR_DECL;
  pdl_trigger();
  pdl_wait();
  TR_MARK1;
  const int r = blockIdx.x;
  if (r == 0)
    for (int i = threadIdx.x; i < n_layers; i += blockDim.x) attn_next[i] = 0;
  const uint16_t* src = E + (size_t)rows[r].token * d;
  float* dst = x + (size_t)r * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = bf16_to_f32(src[i]);
    dst[i] = v;
    if (g) {
      uint16_t h, l;
      split_bf16(v * g[i], h, l);
      norm_hi[(size_t)r * d + i] = h;
      norm_lo[(size_t)r * d + i] = l;
      ss += v * v;
    }
  }
  if (g) {
    ss = warp_sum(ss);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = ss;
    __syncthreads();
    if (w == 0) {
      float t = l < (int)(blockDim.x >> 5) ? red[l] : 0.f;
      t = warp_sum(t);
      if (l == 0) ssq[(size_t)r * kMaxSsqParts] = t;
    }
  }
  TR_END(1);
}

cudaError_t launch_embed(const cbd_engine* e, const cbd_batch* b, const float* g, cudaStream_t s) {
  return launch_pdl(embed_kernel, dim3(b->n_rows), dim3(256), 0, s, (const uint16_t*)e->embed,
                    (const RowDev*)b->rows, e->dm.d, e->x, e->attn_next, e->dm.L, g, e->norm_hi, e->norm_lo,
                    e->ssq);
}

// h = x / sqrt(mean(x^2) + eps) * g, written as hi + lo bf16 halves.
// One CTA per output row, one float4 per thread and pass; `gather`
// (optional) picks the source row.  The sum of squares is reduced in a fixed
// order (per-thread sums, then a fixed tree), so a row's result does not
// depend on the other rows.
__global__ void rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ g,
                               const int32_t* __restrict__ gather, int d, float eps,
                               uint16_t* __restrict__ hi, uint16_t* __restrict__ lo) {
  __shared__ float red[32];
  TR_DECL;
  pdl_trigger();
  pdl_wait();
  TR_MARK1;
  const int r = blockIdx.x;
  const int src = gather ? gather[r] : r;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)src * d);
  const int n4 = d >> 2;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = xr[i];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = warp_sum(ss);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = ss;
  __syncthreads();
  if (w == 0) {
    float t = l < (int)(blockDim.x >> 5) ? red[l] : 0.f;
    t = warp_sum(t);
    if (l == 0) red[0] = t;
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf(red[0] / (float)d + eps);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  uint2* h2 = reinterpret_cast<uint2*>(hi + (size_t)r * d);
  uint2* l2 = reinterpret_cast<uint2*>(lo + (size_t)r * d);
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = xr[i], gg = g4[i];
    uint16_t h[4], q[4];
    split_bf16(v.x * inv * gg.x, h[0], q[0]);
    split_bf16(v.y * inv * gg.y, h[1], q[1]);
    split_bf16(v.z * inv * gg.z, h[2], q[2]);
    split_bf16(v.w * inv * gg.w, h[3], q[3]);
    h2[i] = make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
    l2[i] = make_uint2(q[0] | ((uint32_t)q[1] << 16), q[2] | ((uint32_t)q[3] << 16));
  }
  TR_END(2);
}

cudaError_t launch_rmsnorm(const cbd_engine* e, const float* x, const float* g, int n_rows,
                           const int32_t* gather, uint16_t* hi, uint16_t* lo, cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  const int threads = std::min(1024, e->dm.d / 4);
  return launch_pdl(rmsnorm_kernel, dim3(n_rows), dim3(threads), 0, s, x, g, gather, e->dm.d, e->dm.eps, hi, lo);
}

}  // namespace cbd

namespace cbd {
CBD_TRACE_BIND(misc)
}  // namespace cbd
