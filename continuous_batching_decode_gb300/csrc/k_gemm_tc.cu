// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05 + TMA).
//
//   Y[n][m] = sum_k W[m][k] * (a_hi[n][k] + a_lo[n][k])    (fp32 accumulate)
//
// Weights are stored pre-tiled, [M/128][K/64][128][64] bf16, so the
// 128 x 64 box each pipeline stage loads is one contiguous 16 KB read.
//
// then one of the shared epilogues (RoPE + paged KV append, residual add,
// SwiGLU, logits).  The decode step reads every weight once for all rows
// ("0.8MB 跑通 Qwen 第 14-1 篇", section 1; "20.3 服务、批处理与流式", section
// 20.3.2: step cost (W + B*A)/beta), so the weights sit on the MMA's M side
// (128 output features per tile) and the step's rows on its N side (16..128
// per tile): each weight tile crosses HBM once and feeds every row.
//
// Activations enter as a pair of bf16 matrices (hi + lo) and both are
// multiplied into the same TMEM accumulator, which keeps ~16 significant
// bits of the fp32 activation (bf16 alone puts 32-layer logits far outside
// the accuracy bound).
//
// Work split ("stream-K"): the T*NT*KB (tile, k-block) iterations are cut
// into gridDim.x equal contiguous ranges, one per CTA (one CTA per SM), so
// every SM streams the same number of weight bytes whatever the matrix
// shape.  A tile whose k-range spans several CTAs is finished by the CTA
// that arrives last on its counter: it sums the partial tiles in k order
// (fixed, so results do not depend on timing) and applies the epilogue.  No
// CTA ever waits for another.
//
// CTA = 6 warps: warp 0 issues TMA loads into a ring of shared-memory
// stages; warp 1 owns TMEM and issues the MMAs (one thread); warps 2-5 read
// the accumulator back (warp w owns TMEM lanes 32*(w%4)..+31) and run the
// epilogue.  The ring keeps loading the next tile while the epilogue drains
// the accumulator.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "tc.cuh"

namespace cbd {

constexpr int kTcBM = 128;          // weight rows per tile (MMA M)
constexpr int kTcBK = 64;           // k per stage: one 128-byte swizzle row of bf16
constexpr int kTcThreads = 192;
constexpr int kTcMaxStages = 16;
constexpr int kTcSmemBudget = 200 * 1024;
constexpr int kTcMaxSegs = 256;     // partial slots a reduction reads from shared memory
constexpr int kTcSegBatch = 8;      // segments whose loads are in flight together

struct TcArgs {
  int M, K, n;                       // weight rows, reduction length, activation rows
  int T, NTILES, KB;                 // m tiles, n tiles, k blocks
  long long total;                   // T * NTILES * KB
  int G;                             // CTAs
  int stages;
  float* part;                       // [2G][NT][128] partial tiles
  int32_t* counters;                 // [T * NTILES]
  int32_t* err;
};

__device__ __forceinline__ long long tc_begin(long long c, long long total, long long G) { return c * total / G; }
__device__ __forceinline__ int tc_cta_of(long long i, long long total, long long G) {
  return (int)(((i + 1) * G + total - 1) / total - 1);
}
// End of the segment that starts at k-block kb0 with `left` iterations left.
__device__ __forceinline__ int tc_seg_end(int KB, int kb0, long long left) {
  return (int)((long long)KB < kb0 + left ? (long long)KB : kb0 + left);
}

template <int NT>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                   const __grid_constant__ CUtensorMap tmL, const TcArgs a, const EpiArgs ep) {
  constexpr uint32_t kTmemCols = NT <= 32 ? 32 : NT;
  constexpr uint32_t kWBytes = kTcBM * kTcBK * 2;   // 16 KB
  constexpr uint32_t kABytes = NT * kTcBK * 2;      // per hi / lo tile
  constexpr uint32_t kStageBytes = kWBytes + 2 * kABytes;
  constexpr uint32_t kIdesc = tc::idesc_bf16(kTcBM, NT);

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kTcMaxStages], empty_bar[kTcMaxStages];
  __shared__ __align__(8) uint64_t accum_full, tmem_empty, mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ int last_flag;
  __shared__ int seg_slot[kTcMaxSegs];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = tc::smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  uint8_t* ring = smem_raw + pad;

  const long long G = a.G, total = a.total;
  const long long begin = tc_begin(blockIdx.x, total, G), end = tc_begin(blockIdx.x + 1, total, G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      tc::mbar_init(&full_bar[s], 1);
      tc::mbar_init(&empty_bar[s], 1);
    }
    tc::mbar_init(&accum_full, 1);
    tc::mbar_init(&tmem_empty, 128);
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
  if (warp == 1) tc::tmem_alloc(&tmem_base, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  volatile int* abort_p = &abort_flag;
  if (warp != 0) pdl_wait();          // the producer waits after prefetching weights

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      // iteration it = (unit u, k-block kb), u = nt * T + t; ring slot q = it - begin
      const long long n_it = end - begin;
      auto issue_w = [&](long long q) {
        const long long it = begin + q;
        const int u = (int)(it / a.KB), kb = (int)(it - (long long)u * a.KB);
        const int s = (int)(q % a.stages);
        uint8_t* st = ring + (size_t)s * kStageBytes;
        tc::mbar_arrive_expect_tx(&full_bar[s], kStageBytes);
        tc::tma_load_2d(st, &tmW, 0, ((u % a.T) * a.KB + kb) * kTcBM, &full_bar[s]);
      };
      auto issue_a = [&](long long q) {
        const long long it = begin + q;
        const int u = (int)(it / a.KB), kb = (int)(it - (long long)u * a.KB);
        const int nt = u / a.T;
        const int s = (int)(q % a.stages);
        uint8_t* st = ring + (size_t)s * kStageBytes;
#pragma unroll
        for (int j = 0; j < NT / 16; ++j) {
          tc::tma_load_2d(st + kWBytes + j * 16 * 128, &tmH, kb * kTcBK, nt * NT + j * 16, &full_bar[s]);
          tc::tma_load_2d(st + kWBytes + kABytes + j * 16 * 128, &tmL, kb * kTcBK, nt * NT + j * 16, &full_bar[s]);
        }
      };
      // weights do not depend on the previous kernel: start streaming them
      // before waiting for it, then add the activations
      const long long npre = n_it < a.stages ? n_it : a.stages;
      for (long long q = 0; q < npre; ++q) issue_w(q);
      pdl_wait();
      for (long long q = 0; q < npre; ++q) issue_a(q);
      long long q = npre;
      bool ok = true;
      for (; q < n_it; ++q) {
        const int s = (int)(q % a.stages);
        const uint32_t ph = (uint32_t)((q / a.stages) & 1);
        if (!tc::mbar_wait(&empty_bar[s], ph ^ 1, a.err, abort_p)) { ok = false; break; }
        issue_w(q);
        issue_a(q);
      }
      // wind-down: every load issued must land before the CTA exits
      if (!ok) {
        const long long first = q > a.stages ? q - a.stages : 0;
        for (long long r = first; r < q; ++r) {
          int dummy_abort = 0;
          tc::mbar_wait(&full_bar[r % a.stages], (uint32_t)((r / a.stages) & 1), nullptr, &dummy_abort);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      long long it = begin;
      uint32_t q = 0, seg = 0;
      bool ok = true;
      while (it < end && ok) {
        const int u = (int)(it / a.KB);
        const int kb0 = (int)(it - (long long)u * a.KB);
        const int kb1 = tc_seg_end(a.KB, kb0, end - it);
        if (seg > 0) {
          if (!tc::mbar_wait(&tmem_empty, (seg - 1) & 1, a.err, abort_p)) break;
          tc::tc_fence_after();
        }
        for (int kb = kb0; kb < kb1; ++kb, ++q) {
          const int s = q % a.stages;
          const uint32_t ph = (q / a.stages) & 1;
          if (!tc::mbar_wait(&full_bar[s], ph, a.err, abort_p)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t st = tc::smem_u32(ring + (size_t)s * kStageBytes);
          const uint64_t dW = tc::sdesc_sw128(st);
          const uint64_t dH = tc::sdesc_sw128(st + kWBytes);
          const uint64_t dL = tc::sdesc_sw128(st + kWBytes + kABytes);
#pragma unroll
          for (int k = 0; k < kTcBK / 16; ++k) {
            // advance 16 bf16 = 32 bytes along K inside the swizzled row
            tc::mma_bf16(tmem, dW + 2 * k, dH + 2 * k, kIdesc, (kb > kb0 || k > 0) ? 1u : 0u);
            tc::mma_bf16(tmem, dW + 2 * k, dL + 2 * k, kIdesc, 1u);
          }
          tc::mma_commit(&empty_bar[s]);
        }
        if (!ok) break;
        tc::mma_commit(&accum_full);
        ++seg;
        it += kb1 - kb0;
      }
      // every MMA this thread issued completes before TMEM is released
      tc::mma_commit(&mma_done);
      int no_abort = 0;
      tc::mbar_wait(&mma_done, 0, a.err, &no_abort);
    }
  } else {
    // ------------------------------------------------ epilogue warps 2..5
    const int lg = warp & 3;                    // TMEM lane group
    const int m_loc = lg * 32 + lane;           // feature within the tile
    const uint32_t taddr = tmem + ((uint32_t)(lg * 32) << 16);
    long long it = begin;
    uint32_t seg = 0;
    while (it < end) {
      const int u = (int)(it / a.KB);
      const int kb0 = (int)(it - (long long)u * a.KB);
      const int kb1 = tc_seg_end(a.KB, kb0, end - it);
      const int t = u % a.T, nt = u / a.T;
      const int m = t * kTcBM + m_loc;
      tc::mbar_wait(&accum_full, seg & 1, a.err, abort_p);
      // one uniform decision for all 128 epilogue threads, so no warp is
      // ever left alone in a named barrier
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (threadIdx.x == 64) last_flag = *abort_p;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (last_flag) break;
      asm volatile("bar.sync 1, 128;" ::: "memory");
      tc::tc_fence_after();
      const bool whole = kb0 == 0 && kb1 == a.KB;
      const long long first_it = (long long)u * a.KB;
      const int c_first = tc_cta_of(first_it, total, G);
      const int c_last = tc_cta_of(first_it + a.KB - 1, total, G);
      const int my_slot = 2 * (int)blockIdx.x + (begin >= first_it ? 0 : 1);
      float* mypart = a.part + (size_t)my_slot * NT * kTcBM;
#pragma unroll 1
      for (int c0 = 0; c0 < NT; c0 += 16) {
        float v[16];
        tc::tmem_ld16(taddr + c0, v);
        if (whole) {
          epi_rows<16>(ep, m, lane, nt * NT + c0, a.n, v);
        } else {
          float4* dst = reinterpret_cast<float4*>(mypart + (size_t)m_loc * NT + c0);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&tmem_empty);
      if (!whole) {
        __threadfence();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (threadIdx.x == 64) {
          const int nseg = c_last - c_first + 1;
          const int prev = atomicAdd(&a.counters[u], 1);
          last_flag = prev == nseg - 1;
          if (last_flag) a.counters[u] = 0;     // ready for the next launch
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (last_flag) {
          __threadfence();
          // the tile's partial slots in k order, computed once in parallel
          const int nseg = c_last - c_first + 1;
          for (int i = threadIdx.x - 64; i < nseg && i < kTcMaxSegs; i += 128) {
            const int c = c_first + i;
            seg_slot[i] = 2 * c + (tc_begin(c, total, G) >= first_it ? 0 : 1);
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
          // sum in k order (fixed), 8 columns at a time, with the loads of up
          // to kTcSegBatch segments in flight together
#pragma unroll 1
          for (int c0 = 0; c0 < NT; c0 += 8) {
            float acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll 1
            for (int sb = 0; sb < nseg; sb += kTcSegBatch) {
              float4 t4[kTcSegBatch][2];
#pragma unroll
              for (int i = 0; i < kTcSegBatch; ++i) {
                if (sb + i < nseg) {
                  const int c = c_first + sb + i;
                  const int slot = sb + i < kTcMaxSegs ? seg_slot[sb + i]
                                                        : 2 * c + (tc_begin(c, total, G) >= first_it ? 0 : 1);
                  const float4* src = reinterpret_cast<const float4*>(a.part + (size_t)slot * NT * kTcBM +
                                                                       (size_t)m_loc * NT + c0);
                  t4[i][0] = __ldcg(src);
                  t4[i][1] = __ldcg(src + 1);
                }
              }
#pragma unroll
              for (int i = 0; i < kTcSegBatch; ++i) {
                if (sb + i < nseg) {
                  acc[0] += t4[i][0].x; acc[1] += t4[i][0].y; acc[2] += t4[i][0].z; acc[3] += t4[i][0].w;
                  acc[4] += t4[i][1].x; acc[5] += t4[i][1].y; acc[6] += t4[i][1].z; acc[7] += t4[i][1].w;
                }
              }
            }
            epi_rows<8>(ep, m, lane, nt * NT + c0, a.n, acc);
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
      ++seg;
      it += kb1 - kb0;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
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

template <int NT>
static cudaError_t launch_tc_t(const TcGemm& g, int n, const EpiArgs& ep, const TcWork& w, int sm_count,
                               cudaStream_t s) {
  constexpr int stage_bytes = kTcBM * kTcBK * 2 + 2 * NT * kTcBK * 2;
  const int stages = std::min(kTcMaxStages, kTcSmemBudget / stage_bytes);
  const size_t smem = (size_t)stages * stage_bytes + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t ce = cudaFuncSetAttribute(gemm_tc_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (ce != cudaSuccess) return ce;
    attr_set = true;
  }
  TcArgs a{};
  a.M = g.M; a.K = g.K; a.n = n;
  a.T = g.M / kTcBM; a.NTILES = (n + NT - 1) / NT; a.KB = g.K / kTcBK;
  a.total = (long long)a.T * a.NTILES * a.KB;
  a.G = (int)std::min<long long>(sm_count, a.total);
  a.stages = stages;
  a.part = w.part; a.counters = w.counters; a.err = ep.err;
  if ((long long)a.T * a.NTILES > w.max_units) return cudaErrorInvalidValue;
  return launch_pdl(gemm_tc_kernel<NT>, dim3(a.G), dim3(kTcThreads), smem, s, *g.w, *g.hi, *g.lo, a, ep);
}

cudaError_t launch_gemm_tc(const TcGemm& g, int n, const EpiArgs& ep, const TcWork& w, int sm_count,
                           cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (g.M % kTcBM || g.K % kTcBK) return cudaErrorInvalidValue;
  if (n <= 16) return launch_tc_t<16>(g, n, ep, w, sm_count, s);
  if (n <= 32) return launch_tc_t<32>(g, n, ep, w, sm_count, s);
  if (n <= 64) return launch_tc_t<64>(g, n, ep, w, sm_count, s);
  return launch_tc_t<128>(g, n, ep, w, sm_count, s);
}

}  // namespace cbd
