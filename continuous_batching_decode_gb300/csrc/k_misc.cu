// Embedding gather and RMSNorm (with the hi/lo bf16 split of its output).
#include <algorithm>

#include "common.cuh"
#include "tc.cuh"

namespace cbd {

// x[r][:] = E[token_r][:] as fp32 (the residual stream starts at the
// embedding row of the row's token; CBD_TOKEN_LAST: the token last sampled
// for the row's slot, which the previous step's sampler stored).
// CTA 0 also zeroes the step's counters (per layer: the attention task
// counter and the GEMM chain's grid barriers, n_counters in all; every
// kernel of the previous step has completed once this kernel passes its
// dependency wait).
// With g != null (fused RMSNorm of layer 0) it also writes split(x * g) to
// norm_hi / norm_lo and the row's sum of x^2 (per-thread sums, then a fixed
// tree) as the row's only partial in ssq.
__global__ void embed_kernel(const uint16_t* __restrict__ E, const RowDev* __restrict__ rows, int d,
                             float* __restrict__ x, int32_t* __restrict__ counters, int n_counters,
                             const float* __restrict__ g, uint16_t* __restrict__ norm_hi,
                             uint16_t* __restrict__ norm_lo, float* __restrict__ ssq,
                             const int32_t* __restrict__ last_tok) {
  __shared__ float red[32];
  TR_DECL;
  pdl_trigger();
  pdl_wait();
  TR_MARK1;
  const int r = blockIdx.x;
  if (r == 0)
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
  const int tok = rows[r].token >= 0 ? rows[r].token : last_tok[rows[r].slot];
  // 8 elements (16 bytes of the bf16 row) per thread and round; d is a
  // multiple of 256, so every access is whole and aligned
  const uint4* src = reinterpret_cast<const uint4*>(E + (size_t)tok * d);
  float* dst = x + (size_t)r * d;
  float ss = 0.f;
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    const uint4 w = src[c];
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(wv[j] << 16);
      v[2 * j + 1] = __uint_as_float(wv[j] & 0xffff0000u);
    }
    float4* d4 = reinterpret_cast<float4*>(dst + 8 * c);
    d4[0] = make_float4(v[0], v[1], v[2], v[3]);
    d4[1] = make_float4(v[4], v[5], v[6], v[7]);
    if (g) {
      const float4 g0 = reinterpret_cast<const float4*>(g)[2 * c], g1 = reinterpret_cast<const float4*>(g)[2 * c + 1];
      const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
      uint16_t h[8], l[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        split_bf16(v[j] * gv[j], h[j], l[j]);
        ss += v[j] * v[j];
      }
      const size_t o = (size_t)r * d + 8 * c;
      *reinterpret_cast<uint4*>(norm_hi + o) =
          make_uint4(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16), h[4] | ((uint32_t)h[5] << 16),
                     h[6] | ((uint32_t)h[7] << 16));
      *reinterpret_cast<uint4*>(norm_lo + o) =
          make_uint4(l[0] | ((uint32_t)l[1] << 16), l[2] | ((uint32_t)l[3] << 16), l[4] | ((uint32_t)l[5] << 16),
                     l[6] | ((uint32_t)l[7] << 16));
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
                    (const RowDev*)b->rows, e->dm.d, e->x, e->attn_next, e->dm.L * (1 + kChainMaxPhases), g,
                    e->norm_hi, e->norm_lo,
                    e->ssq, (const int32_t*)e->last_tok);
}

// h = x / sqrt(mean(x^2) + eps) * g, written as hi + lo bf16 halves.
// Four warps per output row (32 when there are fewer rows than SMs), one
// or two rows per CTA (two when there are rows enough to fill the GPU twice
// over); `gather`
// (optional) picks the source row.  Each thread sums the squares of its
// float4s (i = t, t + threads per row, ...) in order, the warps reduce by a fixed
// shuffle tree and the four warp sums are added in warp order, so a row's
// result does not depend on the other rows.  The thread keeps its first 8
// float4s in registers for the second pass (all of a row of d <= 4096; the
// rest, if any, is read again).  (One 1024-thread CTA per
// row spent most of its time in barriers -- 0.68 ms per 544-row step; one
// warp per row left most SMs idle at 544 rows.)
constexpr int kNormWarpsPerRow = 4;
constexpr int kNormMaxWarpsPerRow = 32;
constexpr int kNormRowsPerCta = 2;
constexpr int kNormMaxV = 8;                 // float4s a thread keeps in registers
__global__ void rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ g,
                               const int32_t* __restrict__ gather, int n_rows, int d, float eps, int tpr,
                               uint16_t* __restrict__ hi, uint16_t* __restrict__ lo) {
  __shared__ float red[kNormRowsPerCta * kNormMaxWarpsPerRow];
  TR_DECL;
  pdl_trigger();
  pdl_wait();
  TR_MARK1;
  const int TPR = tpr;                                 // threads per row
  const int rr = threadIdx.x / TPR, t = threadIdx.x % TPR, wpr = TPR >> 5;
  const int r = blockIdx.x * (blockDim.x / TPR) + rr;
  const bool live = r < n_rows;
  const int n4 = d >> 2;
  float4 v[kNormMaxV];
  float ss = 0.f;
  const float4* xr = nullptr;
  if (live) {
    const int src = gather ? gather[r] : r;
    xr = reinterpret_cast<const float4*>(x + (size_t)src * d);
#pragma unroll
    for (int j = 0; j < kNormMaxV; ++j) {
      const int i = t + j * TPR;
      v[j] = i < n4 ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kNormMaxV; ++j) ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    for (int i = t + kNormMaxV * TPR; i < n4; i += TPR) {
      const float4 u = xr[i];
      ss += u.x * u.x + u.y * u.y + u.z * u.z + u.w * u.w;
    }
  }
  ss = warp_sum(ss);
  if ((t & 31) == 0) red[rr * wpr + (t >> 5)] = ss;
  __syncthreads();
  if (!live) return;
  float tot = 0.f;
  for (int w = 0; w < wpr; ++w) tot += red[rr * wpr + w];
  const float inv = 1.0f / sqrtf(tot / (float)d + eps);
  const float4* g4 = reinterpret_cast<const float4*>(g);
  uint2* h2 = reinterpret_cast<uint2*>(hi + (size_t)r * d);
  uint2* l2 = reinterpret_cast<uint2*>(lo + (size_t)r * d);
  auto put = [&](int i, const float4 u) {
    const float4 gg = g4[i];
    uint16_t h[4], q[4];
    split_bf16(u.x * inv * gg.x, h[0], q[0]);
    split_bf16(u.y * inv * gg.y, h[1], q[1]);
    split_bf16(u.z * inv * gg.z, h[2], q[2]);
    split_bf16(u.w * inv * gg.w, h[3], q[3]);
    h2[i] = make_uint2(h[0] | ((uint32_t)h[1] << 16), h[2] | ((uint32_t)h[3] << 16));
    l2[i] = make_uint2(q[0] | ((uint32_t)q[1] << 16), q[2] | ((uint32_t)q[3] << 16));
  };
#pragma unroll
  for (int j = 0; j < kNormMaxV; ++j)
    if (t + j * TPR < n4) put(t + j * TPR, v[j]);
  for (int i = t + kNormMaxV * TPR; i < n4; i += TPR) put(i, xr[i]);
  TR_END(2);
}

cudaError_t launch_rmsnorm(const cbd_engine* e, const float* x, const float* g, int n_rows,
                           const int32_t* gather, uint16_t* hi, uint16_t* lo, cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  if (e->dm.d % 4) return cudaErrorInvalidValue;
  const int rpc = n_rows >= 2 * e->sm_count * kNormRowsPerCta ? kNormRowsPerCta : 1;
  const int tpr = 32 * (n_rows < e->sm_count ? std::min(kNormMaxWarpsPerRow, std::max(1, e->dm.d / 128))
                                             : kNormWarpsPerRow);
  const int ctas = (n_rows + rpc - 1) / rpc;
  return launch_pdl(rmsnorm_kernel, dim3(ctas), dim3(tpr * rpc), 0, s, x, g, gather, n_rows, e->dm.d, e->dm.eps, tpr,
                    hi, lo);
}

// The bounded mbarrier wait that every pipeline of the step's kernels uses,
// on a barrier that nothing completes: thread 0 gives up after `limit` SM
// cycles, which records kDevWaitTimeout in the error word, and the kernel
// returns.  No copy is in flight, no TMEM is held and no peer CTA waits.
__global__ void wait_probe_kernel(long long limit, int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait(&bar, 0, err, &abort_flag, limit);
  __syncthreads();
}

cudaError_t launch_wait_probe(long long limit, int32_t* err, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(limit, err);
  return cudaGetLastError();
}

}  // namespace cbd

namespace cbd {
CBD_TRACE_BIND(misc)
}  // namespace cbd
