// Fused per-row sampler: penalty from the slot's decayed occurrence
// counters, temperature, top-k, top-p, a Philox-4x32-10 uniform and an
// inverse-CDF draw, then the counter update.  Parameters and defaults are
// those of "RWKV Runner Albatross 后端",
// sections "适配器" (temperature 1.0, top_p 0.3, top_k 0, frequency penalty 1,
// decay 0.996) and "Worker 主循环" (penalties, then batched sampling of every
// row).  The order of operations is this library's reading:
//   forbidden ids (the engine's mask, Worker 主循环: "forbidden token 屏蔽"
//   before the penalties) take l = -inf: never chosen, zero mass
//   l' = (l - presence*[cnt>0]) - frequency*cnt   (fp32, separately rounded)
//   greedy argmax (ties -> lowest id) if T == 0 or top_k == 1, else
//   z = l'/T; keep the top_k by (z desc, id asc); the nucleus is the
//   shortest prefix in that order whose probability mass reaches top_p;
//   the token is the first id, ascending, whose cumulative kept mass
//   exceeds u times the kept total.  Then cnt *= decay; cnt[tok] += 1.
//
// A cluster of kSC CTAs (1024 threads each) per sampled row: CTA rank r
// owns ids [r*V/kSC, (r+1)*V/kSC) and its warp w a contiguous part of that,
// walked in coalesced 32-id rounds, so id-ordered prefix sums are a prefix
// over the cluster's CTAs (read over distributed shared memory, rank order)
// plus one over warps plus per-round warp scans.  A CTA keeps its ids' z in
// shared memory (up to kZCache ids; beyond that they live in the scratch
// row).  Probability masses are fixed-point integers (exp(z - zmax) * 2^40),
// so every sum, threshold and scan is exact and independent of thread
// timing.  The k-th largest key is found by 8-bit radix selection over
// order-preserving 32-bit keys of z.  The top-p cutoff: 8-bit radix passes
// over the same keys build the cluster's histograms of counts and masses
// (the first pass also gives the total mass S) and narrow down the bucket
// where the cumulative mass in descending key order reaches ceil(top_p * S);
// as soon as that bucket holds at most kCandCap elements, they are gathered
// from the cluster, sorted by (key desc, id asc) and scanned exactly.
#include "common.cuh"

namespace cbd {

constexpr int kST = 1024;            // threads per sampler CTA
constexpr int kSC = 4;               // CTAs (one cluster) per sampled row
constexpr float kFix = 1099511627776.0f;   // 2^40 (exact in fp32)

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
// The float whose key ord_key gives (+0 for a zero).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// Shared memory.  Radix histograms: every warp owns a private [256] count
// and mass histogram; the block then sums them bin by bin in warp order (and
// the cluster over its CTAs in rank order) -- no atomics, so no contention on
// the few buckets most keys share.  Then the cutoff bucket's candidates.
constexpr int kHistBins = 256;
constexpr int kCandCap = 1024;        // candidates gathered and sorted exactly
constexpr int kZCache = 16384;        // ids per CTA whose z stay in shared memory
struct Cand {
  uint32_t key;
  int32_t id;
  unsigned long long mass;
};
// dynamic layout: z [kZCache] f32 | counts [32][256] u32 | masses [32][256]
// u64 | own candidates [kCandCap] | gathered candidates [kCandCap]
constexpr size_t kSmZ = 0;
constexpr size_t kSmHc = kSmZ + (size_t)kZCache * 4;
constexpr size_t kSmHm = kSmHc + (size_t)(kST / 32) * kHistBins * 4;
constexpr size_t kSmOwn = kSmHm + (size_t)(kST / 32) * kHistBins * 8;
constexpr size_t kSmAll = kSmOwn + (size_t)kCandCap * sizeof(Cand);
constexpr size_t kSampDynSmem = kSmAll + (size_t)kCandCap * sizeof(Cand);
static_assert(kSampDynSmem + sizeof(unsigned long long) * 1024 <= 227 * 1024, "shared memory");

// Add the participating lanes' (digit, mass) to this warp's histogram: the
// lanes holding the same digit are one match group; its count is a popcount
// and its mass a reduction over the group's own mask, and only the group's
// leader lane writes (groups have distinct digits, and every warp owns its
// histogram) -- no atomics, one round of instructions however many digits
// the 32 lanes hold.
__device__ __forceinline__ void warp_hist_add(bool part, uint32_t dg, unsigned long long mv, uint32_t* hc,
                                              unsigned long long* hm, int lane) {
  const unsigned act = __ballot_sync(0xffffffffu, part);
  if (!part) return;
  const unsigned grp = __match_any_sync(act, dg);
  const bool leader = lane == __ffs(grp) - 1;
  if (hm) {
    // masses < 2^41: sum the low 20 bits and the rest separately (each sum
    // of at most 32 lanes fits 32 bits)
    const uint32_t slo = __reduce_add_sync(grp, (uint32_t)(mv & 0xFFFFFull));
    const uint32_t shi = __reduce_add_sync(grp, (uint32_t)(mv >> 20));
    if (leader) hm[dg] += ((unsigned long long)shi << 20) + slo;
  }
  if (leader) hc[dg] += __popc(grp);
}
struct SampShared {
  unsigned long long wsum[32];
  uint32_t wkey[32];
  int32_t widx[32];
  unsigned long long hm[256];        // this CTA's histogram
  uint32_t hc[256];
  unsigned long long chm[256];       // the cluster's histogram (rank order sum)
  uint32_t chc[256];
  uint32_t sel_prefix, sel_mask, sel_cnt, ncand;
  int32_t sel_found;
  unsigned long long sel_above, sel_rem, sel_target;
  int32_t tok;
  int32_t cut_id;
  unsigned long long cx;             // a value this CTA shares with its cluster
  uint32_t ckey;
  int32_t cidx;
};

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ void csync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t crank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cmap(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ unsigned long long cld_u64(const unsigned long long* p, uint32_t rank) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(cmap(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t cld_u32(const void* p, uint32_t rank) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cmap(p, rank)) : "memory");
  return v;
}
// Every CTA of the cluster contributes x (thread 0's value counts); all
// threads get the sum over lower ranks and the cluster total (rank order).
__device__ __forceinline__ void cluster_scan(unsigned long long x, SampShared& sh, uint32_t my,
                                             unsigned long long* before, unsigned long long* total) {
  if (threadIdx.x == 0) sh.cx = x;
  csync();
  unsigned long long v[kSC], b = 0, t = 0;
#pragma unroll
  for (uint32_t r = 0; r < (uint32_t)kSC; ++r) v[r] = cld_u64(&sh.cx, r);   // all loads in flight
#pragma unroll
  for (uint32_t r = 0; r < (uint32_t)kSC; ++r) {
    if (r < my) b += v[r];
    t += v[r];
  }
  csync();      // every peer has read sh.cx before it is written again
  *before = b;
  *total = t;
}
// The cluster's histogram: each CTA's sh.hc (and sh.hm when `masses`) summed
// bin by bin in rank order into sh.chc / sh.chm (every CTA the same).
__device__ __forceinline__ void cluster_hist(SampShared& sh, bool masses) {
  csync();
  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) {
    uint32_t cv[kSC], c = 0;
    unsigned long long mv[kSC], mm = 0;
#pragma unroll
    for (uint32_t r = 0; r < (uint32_t)kSC; ++r) {     // all loads in flight, then the sums in rank order
      cv[r] = cld_u32(&sh.hc[b], r);
      mv[r] = masses ? cld_u64(&sh.hm[b], r) : 0ull;
    }
#pragma unroll
    for (uint32_t r = 0; r < (uint32_t)kSC; ++r) {
      c += cv[r];
      mm += mv[r];
    }
    sh.chc[b] = c;
    sh.chm[b] = mm;
  }
  csync();
}
// Smallest of one int per CTA (e.g. a token id found by one of them).
__device__ __forceinline__ int32_t cluster_min_i32(int32_t x, SampShared& sh) {
  if (threadIdx.x == 0) sh.cidx = x;
  csync();
  int32_t v[kSC], m = 0x7fffffff;
#pragma unroll
  for (uint32_t r = 0; r < (uint32_t)kSC; ++r) v[r] = (int32_t)cld_u32(&sh.cidx, r);
#pragma unroll
  for (uint32_t r = 0; r < (uint32_t)kSC; ++r) m = min(m, v[r]);
  csync();
  return m;
}

// Warp w owns the contiguous ids [w*PW, (w+1)*PW) and walks them in
// rounds of 32 consecutive ids (lane = offset), so every load is coalesced
// and id-ordered prefix sums are a warp scan per round plus a carry.
__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Visit this warp's ids in coalesced 32-id rounds, loading kRoundsAhead
// rounds of `src` before running the rounds' bodies in order: a pass costs a
// few memory round trips instead of one per round.  f(v, valid, value) runs
// on every lane for every round (so it may use ballots and shuffles).
// Id v is read at src[v - off].
constexpr int kRoundsAhead = 16;
template <class F>
__device__ __forceinline__ void for_each_id(const float* src, int off, int v0, int v1, int lane, F&& f) {
  for (int base = v0; base < v1; base += 32 * kRoundsAhead) {
    float val[kRoundsAhead];
#pragma unroll
    for (int u = 0; u < kRoundsAhead; ++u) {
      const int v = base + u * 32 + lane;
      val[u] = v < v1 ? src[v - off] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kRoundsAhead; ++u) {
      const int v = base + u * 32 + lane;
      f(v, v < v1, val[u]);
    }
  }
}

// One warp over the 256 bins of a cluster histogram in descending digit
// order (lane L holds digits 255 - 8L .. 248 - 8L): the first digit whose
// running total, starting from `base`, reaches `need` (>= 1, so an empty
// bin is never chosen), and the running total before it.  -1 (and the
// grand total) if no digit reaches it.  v64 (masses) or v32 (counts).
__device__ __forceinline__ int warp_first_reach(const unsigned long long* v64, const uint32_t* v32,
                                                unsigned long long base, unsigned long long need, int lane,
                                                unsigned long long* before) {
  unsigned long long vals[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int d = 255 - 8 * lane - j;
    vals[j] = v64 ? v64[d] : (unsigned long long)v32[d];
    sum += vals[j];
  }
  const unsigned long long incl = warp_incl_scan_u64(sum, lane);
  const unsigned bal = __ballot_sync(0xffffffffu, base + incl >= need);
  if (!bal) {
    *before = base + __shfl_sync(0xffffffffu, incl, 31);
    return -1;
  }
  const int L = __ffs(bal) - 1;
  int d = -1;
  unsigned long long run = base + incl - sum;
  if (lane == L) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (d < 0) {
        if (run + vals[j] >= need) d = 255 - 8 * lane - j;
        else run += vals[j];
      }
    }
  }
  *before = __shfl_sync(0xffffffffu, run, L);
  return __shfl_sync(0xffffffffu, d, L);
}

// Exclusive prefix over the 32 warps of one value per warp (lane 0's value
// counts); returns this warp's prefix and the block total.
__device__ unsigned long long warp_prefix(unsigned long long mine, SampShared& sh, unsigned long long* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) sh.wsum[w] = mine;
  __syncthreads();
  if (w == 0) {
    const unsigned long long x = sh.wsum[lane];
    const unsigned long long inc = warp_incl_scan_u64(x, lane);
    sh.wsum[lane] = inc - x;
    if (lane == 31) sh.sel_above = inc;
  }
  __syncthreads();
  *total = sh.sel_above;
  const unsigned long long r = sh.wsum[w];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kST) sampler_kernel(const float* __restrict__ logits, int V,
                                                      float* __restrict__ counters,
                                                      const int32_t* __restrict__ slots,
                                                      const SampDev* __restrict__ samp,
                                                      float* __restrict__ scratch,
                                                      const uint32_t* __restrict__ forbid,
                                                      int32_t* __restrict__ out, int32_t* err,
                                                      int32_t* __restrict__ last_tok) {
  __shared__ SampShared sh;
  extern __shared__ __align__(16) uint8_t samp_dyn[];
  float* zc = reinterpret_cast<float*>(samp_dyn + kSmZ);
  uint32_t* whc = reinterpret_cast<uint32_t*>(samp_dyn + kSmHc);                       // [32][256] counts
  unsigned long long* whm = reinterpret_cast<unsigned long long*>(samp_dyn + kSmHm);   // [32][256] masses
  Cand* own = reinterpret_cast<Cand*>(samp_dyn + kSmOwn);
  Cand* all = reinterpret_cast<Cand*>(samp_dyn + kSmAll);
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x / kSC, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t my = crank();
  const SampDev sp = samp[row];
  const float* lg = logits + (size_t)row * V;
  float* cnt = counters + (size_t)slots[row] * V;
  // this CTA's ids [c0, c1); warp w's part of them [v0, v1)
  const int c0 = (int)((long long)V * my / kSC), c1 = (int)((long long)V * (my + 1) / kSC);
  const int PW = ((c1 - c0 + 32 * 32 - 1) / (32 * 32)) * 32;   // ids per warp, a multiple of 32
  const int v0 = min(c1, c0 + w * PW);
  const int v1 = min(c1, v0 + PW);
  const bool greedy = sp.temperature == 0.0f || sp.top_k == 1;
  const unsigned lt_mask = (1u << lane) - 1u;
  // z of id v at zs[v - zoff]: shared memory, or the scratch row
  const bool cached = c1 - c0 <= kZCache;
  float* zs = cached ? zc : scratch + (size_t)row * V;
  const int zoff = cached ? c0 : 0;

  // 1. penalty (and temperature); best key, lowest id on ties
  uint32_t bk = 0;
  int32_t bi = 0x7fffffff;
  for (int base = v0; base < v1; base += 32 * kRoundsAhead) {
    float cv[kRoundsAhead], lv[kRoundsAhead];
#pragma unroll
    for (int u = 0; u < kRoundsAhead; ++u) {
      const int v = base + u * 32 + lane;
      cv[u] = v < v1 ? cnt[v] : 0.f;
      lv[u] = v < v1 ? lg[v] : 0.f;
      if (forbid && v < v1 && ((forbid[v >> 5] >> (v & 31)) & 1u)) lv[u] = -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < kRoundsAhead; ++u) {
      const int v = base + u * 32 + lane;
      if (v >= v1) continue;
      const float c = cv[u];
      const float l1 = __fsub_rn(lv[u], c > 0.0f ? sp.presence : 0.0f);
      const float l2 = __fsub_rn(l1, __fmul_rn(sp.frequency, c));
      const float val = greedy ? l2 : __fdiv_rn(l2, sp.temperature);
      zs[v - zoff] = val;
      const uint32_t k = ord_key(val);
      if (bi == 0x7fffffff || k > bk) { bk = k; bi = v; }
    }
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
    if (lane == 0) { sh.ckey = bk; sh.cidx = bi; }
  }
  // the cluster's best: key desc, then lowest id (rank order)
  csync();
  if (tid == 0) {
    uint32_t k = 0;
    int32_t idx = 0x7fffffff;
    for (uint32_t r = 0; r < (uint32_t)kSC; ++r) {
      const uint32_t ok = cld_u32(&sh.ckey, r);
      const int32_t oi = (int32_t)cld_u32(&sh.cidx, r);
      if (oi != 0x7fffffff && (idx == 0x7fffffff || ok > k || (ok == k && oi < idx))) { k = ok; idx = oi; }
    }
    sh.tok = idx;
    sh.sel_mask = k;         // the best key (z of the best id)
  }
  csync();

  if (!greedy) {
    const float zmax = key_float(sh.sel_mask);
    // 2. top-k: radix-select the k-th largest key; keep key > tk, and the
    //    lowest-id `need` elements with key == tk.
    if (sp.top_k > 0 && sp.top_k < V) {
      uint32_t prefix = 0, mask = 0;
      unsigned long long rem = (unsigned long long)sp.top_k;
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < (kST / 32) * kHistBins; i += kST) whc[i] = 0;
        __syncthreads();
        for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) {
          const uint32_t k = ord_key(zv);
          warp_hist_add(valid && (k & mask) == prefix, (k >> shift) & 255u, 0ull, whc + w * kHistBins, nullptr,
                        lane);
        });
        __syncthreads();
        for (int b = tid; b < kHistBins; b += kST) {
          uint32_t c = 0;
          for (int ww = 0; ww < kST / 32; ++ww) c += whc[ww * kHistBins + b];
          sh.hc[b] = c;
        }
        cluster_hist(sh, false);
        if (w == 0) {
          // the digit holding the rem-th largest key (descending digits)
          unsigned long long cum;
          int d = warp_first_reach(nullptr, sh.chc, 0ull, rem, lane, &cum);
          if (d < 0) {       // cannot happen: rem <= the keys left; take digit 0
            d = 0;
            cum -= sh.chc[0];
          }
          if (lane == 0) {
            sh.sel_rem = rem - cum;
            sh.sel_prefix = prefix | ((uint32_t)d << shift);
            sh.sel_mask = mask | (255u << shift);
          }
        }
        __syncthreads();
        prefix = sh.sel_prefix;
        mask = sh.sel_mask;
        rem = sh.sel_rem;
      }
      const uint32_t tk = prefix;
      const unsigned long long need_eq = rem;
      // rank among equal keys in id order
      unsigned long long eq = 0;
      for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) { eq += valid && ord_key(zv) == tk; });
      unsigned long long tot, cbefore, ctot;
      unsigned long long base = warp_prefix(warp_sum_u64(eq), sh, &tot);
      cluster_scan(tot, sh, my, &cbefore, &ctot);
      base += cbefore;
      for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) {
        const uint32_t k = valid ? ord_key(zv) : 0u;
        const unsigned bal = __ballot_sync(0xffffffffu, valid && k == tk);
        if (valid) {
          if (k < tk) zs[v - zoff] = -INFINITY;
          else if (k == tk && base + __popc(bal & lt_mask) >= need_eq) zs[v - zoff] = -INFINITY;
        }
        base += __popc(bal);
      });
      __syncthreads();
    }
    // 3. fixed-point masses of the kept set
    // exp(z - zmax) * 2^40 is exact in fp32 (a power-of-two scale of an fp32
    // value), so rounding it to an integer needs no fp64 arithmetic
    auto mass = [&](float zv) -> unsigned long long {
      if (zv == -INFINITY) return 0ull;
      return __float2ull_rn(expf(zv - zmax) * kFix);
    };
    // 4. top-p cutoff: shortest prefix by (key desc, id asc) with mass >=
    //    top_p * S; the first element past it is (tp, cut_id)
    bool use_cut = false;
    uint32_t tp = 0;
    int32_t cut_id = 0x7fffffff;
    if (sp.top_p < 1.0f) {
      uint32_t prefix = 0, mask = 0, cnt_b = 0;
      unsigned long long above = 0, target = 0;
      // 4a. the bucket where the cumulative mass (descending keys) reaches
      //     the target, 8 bits at a time while it holds more than kCandCap
      //     elements; the first pass also gives the total mass S
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < (kST / 32) * kHistBins; i += kST) { whc[i] = 0; whm[i] = 0; }
        __syncthreads();
        for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) {
          const uint32_t k = ord_key(zv);
          const bool part = valid && zv != -INFINITY && (k & mask) == prefix;
          warp_hist_add(part, (k >> shift) & 255u, part ? mass(zv) : 0ull, whc + w * kHistBins, whm + w * kHistBins,
                        lane);
        });
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
        cluster_hist(sh, true);
        if (w == 0) {
          if (shift == 24) {
            // cumulative mass >= top_p * S  <=>  cumulative >= ceil(top_p * S)
            unsigned long long S = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) S += sh.chm[8 * lane + j];
            S = warp_sum_u64(S);
            const unsigned long long tg = (unsigned long long)ceil((double)sp.top_p * (double)S);
            if (lane == 0) {
              sh.sel_target = tg;
              sh.sel_found = S >= tg;
            }
            __syncwarp();
          }
          if (sh.sel_found) {
            // need >= 1: with a zero target the highest non-empty digit (it
            // holds zmax, mass 2^40) is the one the cumulative reaches first
            const unsigned long long tg = sh.sel_target;
            const unsigned long long need = tg > above ? tg : above + 1;
            unsigned long long bef;
            int d = warp_first_reach(sh.chm, nullptr, above, need, lane, &bef);
            if (d < 0) {      // cannot happen with exact sums: the lowest non-empty digit
              d = 0;
              while (d < 255 && sh.chc[d] == 0) ++d;
              bef = above;
            }
            if (lane == 0) {
              sh.sel_rem = bef;
              sh.sel_prefix = prefix | ((uint32_t)d << shift);
              sh.sel_cnt = sh.chc[d];
            }
          }
        }
        __syncthreads();
        if (!sh.sel_found) break;      // S < target: no cutoff
        use_cut = true;
        target = sh.sel_target;
        prefix = sh.sel_prefix;
        mask |= 255u << shift;
        above = sh.sel_rem;
        cnt_b = sh.sel_cnt;
        __syncthreads();
        if (cnt_b <= (uint32_t)kCandCap) break;
      }
      if (use_cut && cnt_b <= (uint32_t)kCandCap) {
        // 4b. the bucket's elements from the whole cluster, sorted by (key
        //     desc, id asc); the first whose cumulative mass reaches the
        //     target is the cutoff
        if (tid == 0) sh.ncand = 0;
        __syncthreads();
        for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) {
          const uint32_t k = ord_key(zv);
          const bool part = valid && zv != -INFINITY && (k & mask) == prefix;
          const unsigned bal = __ballot_sync(0xffffffffu, part);
          uint32_t slot0 = 0;
          if (lane == 0 && bal) slot0 = atomicAdd(&sh.ncand, (uint32_t)__popc(bal));
          slot0 = __shfl_sync(0xffffffffu, slot0, 0);
          if (part) {
            const uint32_t slot = slot0 + __popc(bal & lt_mask);
            if (slot < (uint32_t)kCandCap) own[slot] = Cand{k, v, mass(zv)};
          }
        });
        __syncthreads();
        csync();
        uint32_t nr[kSC], n = 0;
#pragma unroll
        for (uint32_t r = 0; r < (uint32_t)kSC; ++r) {
          nr[r] = min(cld_u32(&sh.ncand, r), (uint32_t)kCandCap);
          n += nr[r];
        }
        n = min(n, (uint32_t)kCandCap);
        uint32_t n2 = 1;
        while (n2 < n) n2 <<= 1;
        for (uint32_t i = tid; i < n2; i += kST) {
          Cand c{0u, 0x7fffffff, 0ull};      // padding: after every real key
          if (i < n) {
            uint32_t r = 0, j = i;
            while (r + 1 < (uint32_t)kSC && j >= nr[r]) { j -= nr[r]; ++r; }
            const uint32_t a = cmap(&own[j], r);
            uint32_t k, id, mlo, mhi;
            asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(k), "=r"(id), "=r"(mlo), "=r"(mhi)
                         : "r"(a)
                         : "memory");
            c = Cand{k, (int32_t)id, ((unsigned long long)mhi << 32) | mlo};
          }
          all[i] = c;
        }
        csync();      // every peer has read this CTA's candidates
        // bitonic sort of [0, n2) into (key desc, id asc) order
        for (uint32_t k2 = 2; k2 <= n2; k2 <<= 1) {
          for (uint32_t j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
            for (uint32_t i = tid; i < n2; i += kST) {
              const uint32_t l = i ^ j2;
              if (l > i) {
                const Cand a = all[i], b = all[l];
                const bool b_first = b.key > a.key || (b.key == a.key && b.id < a.id);
                if (((i & k2) == 0) == b_first) {
                  all[i] = b;
                  all[l] = a;
                }
              }
            }
            __syncthreads();
          }
        }
        // cumulative masses in that order; the first that reaches the target
        const unsigned long long q0 = 2 * tid < n ? all[2 * tid].mass : 0ull;
        const unsigned long long q1 = 2 * tid + 1 < n ? all[2 * tid + 1].mass : 0ull;
        const unsigned long long y = q0 + q1;
        const unsigned long long yi = warp_incl_scan_u64(y, lane);
        unsigned long long ytot;
        const unsigned long long yincl = warp_prefix(__shfl_sync(0xffffffffu, yi, 31), sh, &ytot) + yi;
        const unsigned long long yex = yincl - y;
        if (tid == 0) sh.sel_found = 0;
        __syncthreads();
        const unsigned long long need = target > above ? target - above : 1ull;
        int hit = -1;
        if (2 * tid < n && yex < need && yex + q0 >= need) hit = 0;
        else if (2 * tid + 1 < n && yex + q0 < need && yex + q0 + q1 >= need) hit = 1;
        if (hit >= 0) {
          sh.ckey = all[2 * tid + hit].key;
          sh.cut_id = all[2 * tid + hit].id;
          sh.sel_found = 1;
        }
        __syncthreads();
        if (sh.sel_found) {
          tp = sh.ckey;
          cut_id = sh.cut_id;
        } else {      // cannot happen with exact sums: keep the bucket's tie group
          tp = n ? all[n - 1].key : prefix;
          cut_id = V;
        }
      } else if (use_cut) {
        // 4c. more than kCandCap elements share one key: among them, in
        //     ascending id order, the first where the cumulative mass reaches
        //     the target
        tp = prefix;
        unsigned long long eqm = 0;
        for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) {
          if (valid && zv != -INFINITY && ord_key(zv) == tp) eqm += mass(zv);
        });
        unsigned long long tot, cbefore, ctot;
        const unsigned long long wbase0 = warp_prefix(warp_sum_u64(eqm), sh, &tot);
        cluster_scan(tot, sh, my, &cbefore, &ctot);
        const unsigned long long wbase = wbase0 + cbefore;
        const unsigned long long wtot = warp_sum_u64(eqm);
        if (tid == 0) sh.cut_id = 0x7fffffff;
        __syncthreads();
        if (above + wbase + wtot >= target) {   // the crossing may lie in this warp
          unsigned long long run = above + wbase;
          bool found = false;
          for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) {
            if (found) return;
            const bool eqk = valid && zv != -INFINITY && ord_key(zv) == tp;
            const unsigned long long mv = eqk ? mass(zv) : 0ull;
            const unsigned long long inc = warp_incl_scan_u64(mv, lane);
            const unsigned bal = __ballot_sync(0xffffffffu, eqk && run + inc >= target);
            if (bal) {
              if (lane == __ffs(bal) - 1) atomicMin(&sh.cut_id, v);
              found = true;
              return;
            }
            run += __shfl_sync(0xffffffffu, inc, 31);
          });
        }
        __syncthreads();
        cut_id = cluster_min_i32(sh.cut_id, sh);
        if (cut_id == 0x7fffffff) cut_id = V;   // rounding: keep every element of the tie group
      }
    }
    // 5. inverse CDF in ascending id order
    float u = sp.uniform;
    if (u < 0.0f) {
      const uint32_t x = philox_x(sp.token_index, sp.req_lo, sp.req_hi, 0u, sp.seed_lo, sp.seed_hi);
      u = (float)(x >> 8) * (1.0f / 16777216.0f);
    }
    auto kept_mass_z = [&](int v, float zv) -> unsigned long long {
      if (zv == -INFINITY) return 0ull;
      if (use_cut) {
        const uint32_t k = ord_key(zv);
        if (k < tp || (k == tp && v > cut_id)) return 0ull;
      }
      return mass(zv);
    };
    unsigned long long mine = 0;
    for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) { if (valid) mine += kept_mass_z(v, zv); });
    const unsigned long long wtot = warp_sum_u64(mine);
    unsigned long long Sk, cbefore;
    const unsigned long long wbase0 = warp_prefix(wtot, sh, &Sk);
    cluster_scan(Sk, sh, my, &cbefore, &Sk);
    const unsigned long long wbase = wbase0 + cbefore;
    const unsigned long long T = (unsigned long long)floor((double)u * (double)Sk);
    if (tid == 0) sh.tok = 0x7fffffff;
    __syncthreads();
    if (wbase <= T && wbase + wtot > T) {
      unsigned long long run = wbase;
      bool found = false;
      for_each_id(zs, zoff, v0, v1, lane, [&](int v, bool valid, float zv) {
        if (found) return;
        const unsigned long long mv = valid ? kept_mass_z(v, zv) : 0ull;
        const unsigned long long inc = warp_incl_scan_u64(mv, lane);
        const unsigned bal = __ballot_sync(0xffffffffu, run + inc > T && mv > 0);
        if (bal) {
          if (lane == __ffs(bal) - 1) sh.tok = v;
          found = true;
          return;
        }
        run += __shfl_sync(0xffffffffu, inc, 31);
      });
    }
    __syncthreads();
    const int32_t found = cluster_min_i32(sh.tok, sh);
    if (tid == 0) {
      sh.tok = found;
      if (found == 0x7fffffff) {
        if (my == 0) set_err(err, kDevSampler);
        sh.tok = 0;
      }
    }
    __syncthreads();
  }
  // 6. counters: every CTA decays its ids, then the drawn token's owner
  //    counts it
  const int tok = sh.tok;
  for_each_id(cnt, 0, v0, v1, lane, [&](int v, bool valid, float c) { if (valid) cnt[v] = __fmul_rn(c, sp.decay); });
  __syncthreads();
  if (tid == 0) {
    if (tok >= c0 && tok < c1) cnt[tok] = __fadd_rn(cnt[tok], 1.0f);
    if (my == 0) {
      out[row] = tok;
      if (last_tok) last_tok[slots[row]] = tok;     // the slot's last token (CBD_TOKEN_LAST)
    }
  }
}

// One launch of the sampler over m rows (cbd_step and cbd_sample record
// each drawn token as its slot's last token in last_tok; cbd_sample_static
// passes none).
static cudaError_t sampler_launch_ex(const float* logits, int m, int V, float* counters, const int32_t* slots,
                                     const SampDev* samp, float* scratch, const uint32_t* forbid,
                                     int32_t* out_tokens, int32_t* err, int32_t* last_tok, cudaStream_t s) {
  if (m <= 0) return cudaSuccess;
  static DeviceOnce attr;
  {
    const cudaError_t ce = set_smem_once(attr, sampler_kernel, (int)kSampDynSmem);
    if (ce != cudaSuccess) return ce;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(m * kSC);
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = kSampDynSmem;
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = kSC;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, sampler_kernel, logits, V, counters, slots, samp, scratch, forbid, out_tokens, err,
                            last_tok);
}

cudaError_t sampler_launch(const float* logits, int m, int V, float* counters, const int32_t* slots,
                           const SampDev* samp, float* scratch, const uint32_t* forbid, int32_t* out_tokens,
                           int32_t* err, cudaStream_t s) {
  return sampler_launch_ex(logits, m, V, counters, slots, samp, scratch, forbid, out_tokens, err, nullptr, s);
}

cudaError_t launch_sampler(const cbd_engine* e, const float* logits, int m, const int32_t* slots,
                           const SampDev* samp, int32_t* out_tokens, cudaStream_t s) {
  return sampler_launch_ex(logits, m, e->dm.V, e->counters, slots, samp, e->samp_scratch,
                           e->n_forbidden > 0 ? e->forbid : nullptr, out_tokens, e->err, e->last_tok, s);
}

}  // namespace cbd
