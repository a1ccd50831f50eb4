// Fused per-row sampler: penalty from the slot's decayed occurrence
// counters, temperature, top-k, top-p, a Philox-4x32-10 uniform and an
// inverse-CDF draw, then the counter update.  Parameters and defaults are
// those of the Albatross backend article (discosf.com/news/5420690),
// sections "适配器" (temperature 1.0, top_p 0.3, top_k 0, frequency penalty 1,
// decay 0.996) and "Worker 主循环" (penalties, then batched sampling of every
// row).  The order of operations is this library's reading:
//   l' = (l - presence*[cnt>0]) - frequency*cnt   (fp32, separately rounded)
//   greedy argmax (ties -> lowest id) if T == 0 or top_k == 1, else
//   z = l'/T; keep the top_k by (z desc, id asc); the nucleus is the
//   shortest prefix in that order whose probability mass reaches top_p;
//   the token is the first id, ascending, whose cumulative kept mass
//   exceeds u times the kept total.  Then cnt *= decay; cnt[tok] += 1.
//
// One CTA of 1024 threads per sampled row; thread t owns a contiguous id
// range, so id-ordered prefix sums are block scans.  Probability masses are
// fixed-point integers (exp(z - zmax) * 2^40), so every sum, threshold and
// scan is exact and independent of thread timing; the k-th largest key and
// the top-p cutoff are found by 8-bit radix selection over order-preserving
// 32-bit keys of z.
#include "common.cuh"

namespace cbd {

constexpr int kST = 1024;            // threads per sampler CTA
constexpr double kFix = 1099511627776.0;   // 2^40

// Philox-4x32-10 (Salmon et al., SC'11): 10 rounds of the 4x32 bijection
// with multipliers 0xD2511F53, 0xCD9E8D57 and Weyl key increments
// 0x9E3779B9, 0xBB67AE85.
__device__ __forceinline__ uint32_t philox_x(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                             uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return c0;
}

__device__ __forceinline__ uint32_t ord_key(float f) {
  if (f == 0.0f) f = 0.0f;                       // -0 and +0 compare equal
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Radix histograms: every warp owns a private [256] count and mass
// histogram in dynamic shared memory (no atomics contend across warps);
// the block then sums them bin by bin in warp order.
constexpr int kHistBins = 256;
constexpr size_t kSampDynSmem = (size_t)(kST / 32) * kHistBins * (sizeof(uint32_t) + sizeof(unsigned long long));

struct SampShared {
  unsigned long long wsum[32];
  uint32_t wkey[32];
  int32_t widx[32];
  unsigned long long hm[256];
  uint32_t hc[256];
  uint32_t sel_prefix, sel_mask;
  unsigned long long sel_above, sel_rem;
  int32_t tok;
  int32_t cut_id;
};

// Exclusive scan of one u64 per thread over the block; returns the prefix
// and writes the block total to *total.
__device__ unsigned long long block_exscan(unsigned long long v, SampShared& sh, unsigned long long* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  __syncthreads();
  if (lane == 31) sh.wsum[w] = inc;
  __syncthreads();
  if (w == 0) {
    unsigned long long s = sh.wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long t = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += t;
    }
    sh.wsum[lane] = s;     // inclusive warp-prefix totals
  }
  __syncthreads();
  const unsigned long long before = (w ? sh.wsum[w - 1] : 0ull) + inc - v;
  *total = sh.wsum[31];
  return before;
}

__global__ void __launch_bounds__(kST) sampler_kernel(const float* __restrict__ logits, int V,
                                                      float* __restrict__ counters,
                                                      const int32_t* __restrict__ slots,
                                                      const SampDev* __restrict__ samp,
                                                      float* __restrict__ scratch,
                                                      int32_t* __restrict__ out, int32_t* err) {
  __shared__ SampShared sh;
  extern __shared__ __align__(16) uint8_t samp_dyn[];
  unsigned long long* whm = reinterpret_cast<unsigned long long*>(samp_dyn);             // [32][256]
  uint32_t* whc = reinterpret_cast<uint32_t*>(samp_dyn + (kST / 32) * kHistBins * 8);  // [32][256]
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const SampDev sp = samp[row];
  const float* lg = logits + (size_t)row * V;
  float* cnt = counters + (size_t)slots[row] * V;
  float* z = scratch + (size_t)row * V;
  const int per = (V + kST - 1) / kST;
  const int i0 = min(V, tid * per), i1 = min(V, i0 + per);
  const bool greedy = sp.temperature == 0.0f || sp.top_k == 1;

  // 1. penalty (and temperature); best key, lowest id on ties
  uint32_t bk = 0;
  int32_t bi = 0x7fffffff;
  for (int v = i0; v < i1; ++v) {
    const float c = cnt[v];
    const float l1 = __fsub_rn(lg[v], c > 0.0f ? sp.presence : 0.0f);
    const float l2 = __fsub_rn(l1, __fmul_rn(sp.frequency, c));
    const float val = greedy ? l2 : __fdiv_rn(l2, sp.temperature);
    z[v] = val;
    const uint32_t k = ord_key(val);
    if (bi == 0x7fffffff || k > bk) { bk = k; bi = v; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
    const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (oi != 0x7fffffff && (bi == 0x7fffffff || ok > bk || (ok == bk && oi < bi))) { bk = ok; bi = oi; }
  }
  if (lane == 0) { sh.wkey[w] = bk; sh.widx[w] = bi; }
  __syncthreads();
  if (w == 0) {
    bk = sh.wkey[lane];
    bi = sh.widx[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint32_t ok = __shfl_xor_sync(0xffffffffu, bk, o);
      const int32_t oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ok > bk || (ok == bk && oi < bi))) { bk = ok; bi = oi; }
    }
    if (lane == 0) sh.tok = bi;
  }
  __syncthreads();

  if (!greedy) {
    const float zmax = z[sh.tok];
    // 2. top-k: radix-select the k-th largest key; keep key > tk, and the
    //    lowest-id `need` elements with key == tk.
    uint32_t tk = 0;
    long long need_eq = 0x7fffffffffffffffLL;
    const bool do_topk = sp.top_k > 0 && sp.top_k < V;
    if (do_topk) {
      uint32_t prefix = 0, mask = 0;
      unsigned long long rem = (unsigned long long)sp.top_k;
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < (kST / 32) * kHistBins; i += kST) whc[i] = 0;
        __syncthreads();
        for (int v = i0; v < i1; ++v) {
          const uint32_t k = ord_key(z[v]);
          if ((k & mask) == prefix) atomicAdd(&whc[w * kHistBins + ((k >> shift) & 255u)], 1u);
        }
        __syncthreads();
        for (int b = tid; b < kHistBins; b += kST) {
          uint32_t c = 0;
          for (int ww = 0; ww < kST / 32; ++ww) c += whc[ww * kHistBins + b];
          sh.hc[b] = c;
        }
        __syncthreads();
        if (tid == 0) {
          unsigned long long cum = 0;
          int d = 255;
          for (; d > 0; --d) {
            if (cum + sh.hc[d] >= rem) break;
            cum += sh.hc[d];
          }
          sh.sel_rem = rem - cum;
          sh.sel_prefix = prefix | ((uint32_t)d << shift);
          sh.sel_mask = mask | (255u << shift);
        }
        __syncthreads();
        prefix = sh.sel_prefix;
        mask = sh.sel_mask;
        rem = sh.sel_rem;
        __syncthreads();
      }
      tk = prefix;
      need_eq = (long long)rem;
      // rank of equal keys by id: keep the first need_eq of them
      unsigned long long mine = 0;
      for (int v = i0; v < i1; ++v) mine += ord_key(z[v]) == tk;
      unsigned long long tot;
      unsigned long long rank = block_exscan(mine, sh, &tot);
      for (int v = i0; v < i1; ++v) {
        const uint32_t k = ord_key(z[v]);
        if (k < tk) z[v] = -INFINITY;
        else if (k == tk) {
          if ((long long)rank >= need_eq) z[v] = -INFINITY;
          ++rank;
        }
      }
      __syncthreads();
    }
    // 3. fixed-point masses of the kept set
    auto mass = [&](float zv) -> unsigned long long {
      if (zv == -INFINITY) return 0ull;
      return __double2ull_rn((double)expf(zv - zmax) * kFix);
    };
    // 4. top-p cutoff: shortest prefix by (key desc, id asc) with mass >= top_p * S
    bool use_cut = false;
    uint32_t tp = 0;
    int32_t cut_id = 0x7fffffff;
    if (sp.top_p < 1.0f) {
      unsigned long long mine = 0;
      for (int v = i0; v < i1; ++v) mine += mass(z[v]);
      unsigned long long S;
      (void)block_exscan(mine, sh, &S);
      const double target = (double)sp.top_p * (double)S;
      if ((double)S >= target) {
        use_cut = true;
        uint32_t prefix = 0, mask = 0;
        unsigned long long above = 0;
        for (int shift = 24; shift >= 0; shift -= 8) {
          for (int i = tid; i < (kST / 32) * kHistBins; i += kST) { whc[i] = 0; whm[i] = 0; }
          __syncthreads();
          for (int v = i0; v < i1; ++v) {
            const float zv = z[v];
            if (zv == -INFINITY) continue;
            const uint32_t k = ord_key(zv);
            if ((k & mask) == prefix) {
              const uint32_t dg = (k >> shift) & 255u;
              atomicAdd(&whc[w * kHistBins + dg], 1u);
              atomicAdd(&whm[w * kHistBins + dg], mass(zv));
            }
          }
          __syncthreads();
          for (int b = tid; b < kHistBins; b += kST) {
            uint32_t c = 0;
            unsigned long long mm = 0;
            for (int ww = 0; ww < kST / 32; ++ww) {
              c += whc[ww * kHistBins + b];
              mm += whm[ww * kHistBins + b];
            }
            sh.hc[b] = c;
            sh.hm[b] = mm;
          }
          __syncthreads();
          if (tid == 0) {
            int d = 255, last = -1;
            for (; d >= 0; --d) {
              if (sh.hc[d] == 0) continue;
              last = d;
              if ((double)(above + sh.hm[d]) >= target) break;
              above += sh.hm[d];
            }
            if (d < 0) d = last;        // rounding: take the lowest non-empty digit
            sh.sel_above = above;
            sh.sel_prefix = prefix | ((uint32_t)d << shift);
            sh.sel_mask = mask | (255u << shift);
          }
          __syncthreads();
          prefix = sh.sel_prefix;
          mask = sh.sel_mask;
          above = sh.sel_above;
          __syncthreads();
        }
        tp = prefix;
        // among key == tp, ascending id: first id where above + cum >= target
        unsigned long long eqm = 0;
        for (int v = i0; v < i1; ++v)
          if (z[v] != -INFINITY && ord_key(z[v]) == tp) eqm += mass(z[v]);
        unsigned long long tot;
        unsigned long long before = block_exscan(eqm, sh, &tot);
        if (tid == 0) sh.cut_id = 0x7fffffff;
        __syncthreads();
        unsigned long long run = above + before;
        for (int v = i0; v < i1; ++v) {
          if (z[v] == -INFINITY || ord_key(z[v]) != tp) continue;
          run += mass(z[v]);
          if ((double)run >= target) { atomicMin(&sh.cut_id, v); break; }
        }
        __syncthreads();
        cut_id = sh.cut_id;
        if (cut_id == 0x7fffffff) {      // rounding: keep every element of the tie group
          cut_id = V;
        }
      }
    }
    auto kept_mass = [&](int v) -> unsigned long long {
      const float zv = z[v];
      if (zv == -INFINITY) return 0ull;
      if (use_cut) {
        const uint32_t k = ord_key(zv);
        if (k < tp || (k == tp && v > cut_id)) return 0ull;
      }
      return mass(zv);
    };
    // 5. inverse CDF in ascending id order
    float u = sp.uniform;
    if (u < 0.0f) {
      const uint32_t x = philox_x(sp.token_index, sp.req_lo, sp.req_hi, 0u, sp.seed_lo, sp.seed_hi);
      u = (float)(x >> 8) * (1.0f / 16777216.0f);
    }
    unsigned long long mine = 0;
    for (int v = i0; v < i1; ++v) mine += kept_mass(v);
    unsigned long long Sk;
    const unsigned long long before = block_exscan(mine, sh, &Sk);
    const unsigned long long T = (unsigned long long)floor((double)u * (double)Sk);
    if (tid == 0) sh.tok = 0x7fffffff;
    __syncthreads();
    if (before <= T && before + mine > T) {
      unsigned long long run = before;
      for (int v = i0; v < i1; ++v) {
        run += kept_mass(v);
        if (run > T) { sh.tok = v; break; }
      }
    }
    __syncthreads();
    if (sh.tok == 0x7fffffff) {
      if (tid == 0) { set_err(err, kDevSampler); sh.tok = 0; }
      __syncthreads();
    }
  }
  // 6. counters: decay everything, then count the drawn token
  const int tok = sh.tok;
  for (int v = i0; v < i1; ++v) cnt[v] = __fmul_rn(cnt[v], sp.decay);
  __syncthreads();
  if (tid == 0) {
    cnt[tok] = __fadd_rn(cnt[tok], 1.0f);
    out[row] = tok;
  }
}

// One launch of the sampler over m rows (shared by cbd_step, cbd_sample and
// cbd_sample_static).
cudaError_t sampler_launch(const float* logits, int m, int V, float* counters, const int32_t* slots,
                           const SampDev* samp, float* scratch, int32_t* out_tokens, int32_t* err, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  static bool attr = false;
  if (!attr) {
    cudaError_t ce = cudaFuncSetAttribute(sampler_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSampDynSmem);
    if (ce != cudaSuccess) return ce;
    attr = true;
  }
  sampler_kernel<<<m, kST, kSampDynSmem, s>>>(logits, V, counters, slots, samp, scratch, out_tokens, err);
  return cudaGetLastError();
}

cudaError_t launch_sampler(const cbd_engine* e, const float* logits, int m, const int32_t* slots,
                           const SampDev* samp, int32_t* out_tokens, cudaStream_t s) {
  return sampler_launch(logits, m, e->dm.V, e->counters, slots, samp, e->samp_scratch, out_tokens, e->err, s);
}

}  // namespace cbd
