// Weight-streaming GEMM on CUDA cores ("skinny GEMV"): Y[n][m] =
// sum_k W[m][k] * (a_hi[n][k] + a_lo[n][k]), fp32 accumulation, followed by
// one of the shared epilogues.  Every weight byte is read once per group of
// NB rows, which is the whole step when n <= NB: the batched decode step
// reads each weight once for all rows ("0.8MB 跑通 Qwen 第 14-1 篇", section 1;
// "20.3 服务、批处理与流式" section 20.3.2, cost (W + B*A)/beta).
//
// Weights are read from the pre-tiled layout [M/N][K/64][N][64] that the
// tensor-core path uses (16-byte chunks stay contiguous).
// CTA = 8 warps; a warp owns 4 consecutive output features, so RoPE and
// SwiGLU partners (features 2i, 2i+1) live in one warp.  Activations for
// the CTA's NB rows are staged in shared memory 256 columns at a time as
// fp32 (hi + lo is exact in fp32); each lane streams 16-byte chunks of its
// four weight rows.
#include "common.cuh"

namespace cbd {

constexpr int kGemvWarps = 8;
constexpr int kGemvFeat = 4;   // features per warp
constexpr int kKTile = 256;    // k columns per shared-memory tile

template <int NB>
__global__ void __launch_bounds__(256) gemv_kernel(const uint16_t* __restrict__ W, int M, int K, int TN,
                                                   const uint16_t* __restrict__ a_hi,
                                                   const uint16_t* __restrict__ a_lo, int lda, int n,
                                                   EpiArgs ep) {
  __shared__ __align__(16) float act[NB][kKTile];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f0 = (blockIdx.x * kGemvWarps + warp) * kGemvFeat;
  const int r0 = blockIdx.y * NB;
  float acc[kGemvFeat][NB];
#pragma unroll
  for (int i = 0; i < kGemvFeat; ++i)
#pragma unroll
    for (int j = 0; j < NB; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kKTile) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < NB * kKTile; idx += blockDim.x) {
      const int j = idx / kKTile, c = idx % kKTile;
      const int r = r0 + j;
      float v = 0.f;
      if (r < n) {
        const size_t o = (size_t)r * lda + k0 + c;
        v = bf16_to_f32(a_hi[o]) + bf16_to_f32(a_lo[o]);
      }
      act[j][c] = v;
    }
    __syncthreads();
    if (f0 < M) {
      const int kc = lane * 8;
      uint4 w[kGemvFeat];
      const int kk = k0 + kc, KB = K / 64;
#pragma unroll
      for (int i = 0; i < kGemvFeat; ++i) {
        const int f = f0 + i;
        w[i] = __ldg(reinterpret_cast<const uint4*>(W + tiled_off(f, kk, TN, KB)));
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        const float4 x0 = *reinterpret_cast<const float4*>(&act[j][kc]);
        const float4 x1 = *reinterpret_cast<const float4*>(&act[j][kc + 4]);
#pragma unroll
        for (int i = 0; i < kGemvFeat; ++i) {
          float s = acc[i][j];
          s = fmaf(bf16lo_f32(w[i].x), x0.x, s);
          s = fmaf(bf16hi_f32(w[i].x), x0.y, s);
          s = fmaf(bf16lo_f32(w[i].y), x0.z, s);
          s = fmaf(bf16hi_f32(w[i].y), x0.w, s);
          s = fmaf(bf16lo_f32(w[i].z), x1.x, s);
          s = fmaf(bf16hi_f32(w[i].z), x1.y, s);
          s = fmaf(bf16lo_f32(w[i].w), x1.z, s);
          s = fmaf(bf16hi_f32(w[i].w), x1.w, s);
          acc[i][j] = s;
        }
      }
    }
  }
  if (f0 >= M) return;
#pragma unroll
  for (int i = 0; i < kGemvFeat; ++i)
#pragma unroll
    for (int j = 0; j < NB; ++j) acc[i][j] = warp_sum(acc[i][j]);
  // every lane now holds all sums; spread the stores over the lanes
  if (epi_is_pair(ep.kind)) {
#pragma unroll
    for (int p = 0; p < kGemvFeat / 2; ++p)
#pragma unroll
      for (int j = 0; j < NB; ++j)
        if (lane == p * NB + j && r0 + j < n) epi_pair(ep, f0 + 2 * p, r0 + j, acc[2 * p][j], acc[2 * p + 1][j]);
  } else {
#pragma unroll
    for (int i = 0; i < kGemvFeat; ++i)
#pragma unroll
      for (int j = 0; j < NB; ++j)
        if (lane == (i * NB + j) % 32 && r0 + j < n) epi_single(ep, f0 + i, r0 + j, acc[i][j]);
  }
}

cudaError_t launch_gemv(const uint16_t* W, int M, int K, int TN, const uint16_t* a_hi, const uint16_t* a_lo,
                        int lda, int n, const EpiArgs& ep, cudaStream_t s) {
  const int feat_per_cta = kGemvWarps * kGemvFeat;
  dim3 block(32 * kGemvWarps);
  cudaError_t ce = cudaSuccess;
  if (n <= 1) {
    ce = launch_pdl(gemv_kernel<1>, dim3((M + feat_per_cta - 1) / feat_per_cta, 1), block, 0, s, W, M, K, TN, a_hi, a_lo, lda, n, ep);
  } else if (n <= 2) {
    ce = launch_pdl(gemv_kernel<2>, dim3((M + feat_per_cta - 1) / feat_per_cta, 1), block, 0, s, W, M, K, TN, a_hi, a_lo, lda, n, ep);
  } else if (n <= 4) {
    ce = launch_pdl(gemv_kernel<4>, dim3((M + feat_per_cta - 1) / feat_per_cta, 1), block, 0, s, W, M, K, TN, a_hi, a_lo, lda, n, ep);
  } else {
    dim3 grid((M + feat_per_cta - 1) / feat_per_cta, (n + 7) / 8);
    ce = launch_pdl(gemv_kernel<8>, grid, block, 0, s, W, M, K, TN, a_hi, a_lo, lda, n, ep);
  }
  return ce;
}

// Path choice: the CUDA-core GEMV for a handful of rows, the tcgen05 GEMM
// above that (or as forced by cbd_engine_set_gemm_path).
// Int8-weight engines run every contraction on the tcgen05 kernel with
// 64-row tiles (the only one with the int8 -> bf16 conversion stage).
static bool uses_tc(const cbd_engine* e, int n) {
  return e->w_int8 || e->gemm_path == 2 || (e->gemm_path == 0 && n > e->gemv_max_rows);
}
bool gemm_uses_tc(const cbd_engine* e, int n) { return uses_tc(e, n); }
bool gemm_uses_rows(const cbd_engine* e, int n) {
  return !e->w_int8 && uses_tc(e, n) && e->rows_gemm_min > 0 && n >= e->rows_gemm_min;
}
int gemm_tc_units(int M, int K, int N, int n, bool int8) {
  int T, NR, KB, S;
  const int RT = gemm_tc_row_tiles(n, int8);
  gemm_tc_plan(M, K, N * gemm_tc_pair(M, N, n, int8), n, RT, &T, &NR, &KB, &S);
  return T * S;
}

cudaError_t launch_gemm(const cbd_engine* e, const GemmOp& op, int n, const EpiArgs& ep, const PfSpec& pf,
                        cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (gemm_uses_rows(e, n) && gemm_rows_supports(ep) && (e->rows_gemm_force || gemm_rows_preferred(op.tc, n)))
    return launch_gemm_rows(op.tc, n, ep, s);
  if (uses_tc(e, n)) {
    if (op.tc.scale) {
      EpiArgs e8 = ep;
      e8.w_scale = op.tc.scale;
      return launch_gemm_tc(op.tc, n, e8, PfSpec{}, s);
    }
    return launch_gemm_tc(op.tc, n, ep, pf, s);
  }
  return launch_gemv(op.W, op.M, op.K, op.tc.N, op.a_hi, op.a_lo, op.lda, n, ep, s);
}

PfSpec next_prefetch(const cbd_engine* e, const GemmOp& op, int n) {
  PfSpec pf{};
  if (n <= 0 || e->l2_prefetch == 0 || !uses_tc(e, n) || e->w_int8) return pf;
  int T, NR, KB, S;
  const int RT = gemm_tc_row_tiles(n, false), TP = gemm_tc_pair(op.tc.M, op.tc.N, n, false);
  gemm_tc_plan(op.tc.M, op.tc.K, op.tc.N * TP, n, RT, &T, &NR, &KB, &S);
  T *= TP;                           // per weight tile: a unit's tiles read the same k-blocks
  const long long units = (long long)T * S;
  const long long per_unit = (KB + S - 1) / S;
  long long P = (long long)(e->l2_prefetch / ((size_t)op.tc.N * 128)) / units;
  if (P < 1) P = 1;
  if (P > per_unit) P = per_unit;
  pf.w = reinterpret_cast<const uint8_t*>(op.W);
  pf.N = op.tc.N; pf.T = T; pf.KB = KB; pf.S = S; pf.P = (int32_t)P;
  return pf;
}

}  // namespace cbd
