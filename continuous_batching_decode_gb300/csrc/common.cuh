// Device helpers shared by the kernels: bf16 <-> fp32, the hi/lo split,
// warp reductions and the GEMM epilogues (one definition used by every
// GEMM variant, so all variants store identical results).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "cbd_internal.h"

namespace cbd {

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
__device__ __forceinline__ float bf16lo_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}
// x = hi + lo with hi = bf16(x), lo = bf16(x - hi): 16 significant bits.
__device__ __forceinline__ void split_bf16(float x, uint16_t& hi, uint16_t& lo) {
  hi = f32_to_bf16(x);
  lo = f32_to_bf16(x - bf16_to_f32(hi));
}

// SwiGLU's gate: silu(a) * b = a / (1 + e^-a) * b, with the hardware
// exponential and divide (a few ulp; the result is rounded to hi + lo bf16
// right after).  For a very negative, e^-a overflows to +inf and the
// quotient is 0, the limit of silu.
__device__ __forceinline__ float silu_mul(float a, float b) { return __fdividef(a, 1.0f + __expf(-a)) * b; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Programmatic dependent launch: every kernel of the step lets the next one
// launch as soon as all of its CTAs have started, and waits for the
// previous kernel to complete (and its writes to be visible) before it
// touches anything that kernel wrote.  Without the launch attribute both
// are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Timeline tracing, compiled in only with -DCBD_TRACE (a separate debug
// build of the library): thread 0 of every CTA records %globaltimer at the
// CTA's start, after its dependency wait (TR_MARK1), at one kernel-specific
// milestone (TR_MARK2) and at its end, with the kernel kind and the SM.
// Each translation unit has its own trace pointer, bound from the host by
// its exported cbd_trace_bind_<unit>(buffer) (5 x u64 per record, at most
// 2^20 records; buffer = null turns tracing off).
#ifdef CBD_TRACE
static __device__ unsigned long long* g_trace = nullptr;
static __device__ unsigned int g_trace_n = 0;
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void trace_put(unsigned kind, unsigned long long t0, unsigned long long t1,
                                          unsigned long long t2, unsigned long long t3) {
  if (!g_trace) return;
  const unsigned i = atomicAdd(&g_trace_n, 1u);
  if (i >= (1u << 20)) return;
  unsigned sm;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
  unsigned long long* p = g_trace + (size_t)i * 5;
  p[0] = ((unsigned long long)kind << 32) | ((unsigned long long)sm << 24) | (blockIdx.x + blockIdx.y * gridDim.x);
  p[1] = t0; p[2] = t1; p[3] = t2; p[4] = t3;
}
#define TR_DECL unsigned long long _tr0 = gtimer(), _tr1 = 0, _tr2 = 0
#define TR_MARK1 (_tr1 = gtimer())
#define TR_MARK2 (_tr2 = gtimer())
#define TR_END(kind) do { if (threadIdx.x == 0) trace_put((kind), _tr0, _tr1, _tr2, gtimer()); } while (0)
#define CBD_TRACE_BIND(unit)                                                             \
  extern "C" int cbd_trace_bind_##unit(void* buf) {                                      \
    unsigned long long* p = static_cast<unsigned long long*>(buf);                       \
    unsigned int z = 0;                                                                  \
    if (cudaMemcpyToSymbol(g_trace, &p, sizeof p) != cudaSuccess) return -1;             \
    return cudaMemcpyToSymbol(g_trace_n, &z, sizeof z) == cudaSuccess ? 0 : -1;          \
  }
#else
#define TR_DECL
#define TR_MARK1
#define TR_MARK2
#define TR_END(kind)
#define CBD_TRACE_BIND(unit)
#endif
// kinds: 1 embed, 2 rmsnorm, 3 attention stream, 4 attention merge,
// 5 sampler, 6 GEMV, (16 << 12) | M/256 tcgen05 GEMM

__device__ __forceinline__ void set_err(int32_t* err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// KV pool layout: [L][n_blocks][H_kv][K|V][tile], one tile = 32 positions x
// hd dims of bf16 stored in the order a 128-byte-swizzled shared-memory copy
// of it has: dims in 64-wide halves, each half 32 rows of 128 bytes, and
// the 16-byte chunk c of row r at chunk position c ^ (r & 7).  So K and V of
// one (layer, block, KV head) are one contiguous 2 * 32 * hd * 2-byte run
// that a single bulk copy lands in shared memory ready for ldmatrix.
__host__ __device__ __forceinline__ int tile_elem(int r, int d) {
  return (d >> 6) * 2048 + r * 64 + ((((d & 63) >> 3) ^ (r & 7)) << 3) + (d & 7);
}
__host__ __device__ __forceinline__ size_t pool_tile(int layer, int nblocks, int blk, int hkv, int kvh, int kv, int hd) {
  return ((((size_t)layer * nblocks + blk) * hkv + kvh) * 2 + kv) * (size_t)(kBlock * hd);
}
__device__ __forceinline__ size_t pool_off(int layer, int kv, int nblocks, int blk, int hkv, int kvh, int hd, int p,
                                           int dim) {
  return pool_tile(layer, nblocks, blk, hkv, kvh, kv, hd) + tile_elem(p, dim);
}

// FP8 (E4M3) pool: the same [L][n_blocks][H_kv][K|V][tile] order with one
// byte per element, tiles of 32 * hd bytes.  K tile: rows = positions of hd
// bytes; V tile transposed: rows = head dims of 32 bytes (positions).  In
// both the 16-byte chunk c of row r sits at c ^ swizzle(r), so that the 8
// rows an ldmatrix reads hit 8 different bank groups: K rows of 128 bytes
// use r & 7, of 64 bytes (r >> 1) & 3; V rows of 32 bytes use (r >> 2) & 1.
template <int HD>
__host__ __device__ __forceinline__ uint32_t k8_off(int r, int c) {
  static_assert(HD == 64 || HD == 128, "head dim");
  return HD == 128 ? (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)) : (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}
__host__ __device__ __forceinline__ uint32_t v8_off(int r, int c) { return (uint32_t)(r * 32 + ((c ^ ((r >> 2) & 1)) << 4)); }
// byte of (position p, dim d) in a K or V FP8 tile
__host__ __device__ __forceinline__ uint32_t k8_elem(int hd, int p, int d) {
  return (hd == 128 ? k8_off<128>(p, d >> 4) : k8_off<64>(p, d >> 4)) + (d & 15);
}
__host__ __device__ __forceinline__ uint32_t v8_elem(int p, int d) { return v8_off(d, p >> 4) + (p & 15); }
// two floats -> two E4M3 bytes (round to nearest even, finite values
// saturate to +-448): `lo` in byte 0, `hi` in byte 1
__device__ __forceinline__ uint16_t f32x2_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Epilogue for a pair of adjacent output features (f, f+1), f even, of
// one row.  QKV: f, f+1 are RoPE partners (dims i, i + hd/2 of one q or k
// head, rows interleaved by the engine's repack) or two consecutive v dims.
// SwiGLU: f = 2i is gate_i and f+1 is up_i.
__device__ __forceinline__ void epi_pair(const EpiArgs& ep, int f, int row, float a, float b) {
  if (ep.kind == kEpiSwiGLU) {
    float y = silu_mul(a, b);
    uint16_t hi, lo;
    split_bf16(y, hi, lo);
    size_t o = (size_t)row * ep.ld_act + (f >> 1);
    ep.out_hi[o] = hi;
    ep.out_lo[o] = lo;
    return;
  }
  // QKV
  const RowDev rw = ep.rows[row];
  const int hd = ep.hd, half = hd >> 1;
  const int nq = ep.hq * hd, nk = ep.hkv * hd;
  if (f < nq + nk) {
    const int head = (f < nq ? f : f - nq) / hd;
    const int i = ((f < nq ? f : f - nq) % hd) >> 1;
    const float2 cs = reinterpret_cast<const float2*>(ep.rope_cs)[(size_t)rw.pos * half + i];
    const float ra = a * cs.x - b * cs.y;
    const float rb = b * cs.x + a * cs.y;
    if (f < nq) {
      float* qrow = ep.out_f32 + (size_t)row * nq + head * hd;
      qrow[i] = ra;
      qrow[i + half] = rb;
    } else {
      const int blk = ep.tables[(size_t)rw.slot * ep.max_blocks_per_seq + (rw.pos >> 5)];
      if (blk < 0 || blk >= ep.n_blocks) { set_err(ep.err, kDevBadBlock); return; }
      const size_t t0 = pool_tile(ep.layer, ep.n_blocks, blk, ep.hkv, head, 0, hd);
      if (ep.kv_fp8) {
        uint8_t* t8 = reinterpret_cast<uint8_t*>(ep.pool) + t0;
        const uint16_t e = f32x2_e4m3x2(ra, rb);
        t8[k8_elem(hd, rw.pos & 31, i)] = (uint8_t)(e & 0xff);
        t8[k8_elem(hd, rw.pos & 31, i + half)] = (uint8_t)(e >> 8);
        return;
      }
      ep.pool[t0 + tile_elem(rw.pos & 31, i)] = f32_to_bf16(ra);
      ep.pool[t0 + tile_elem(rw.pos & 31, i + half)] = f32_to_bf16(rb);
    }
  } else {
    const int fv = f - nq - nk;
    const int head = fv / hd, j = fv % hd;
    const int blk = ep.tables[(size_t)rw.slot * ep.max_blocks_per_seq + (rw.pos >> 5)];
    if (blk < 0 || blk >= ep.n_blocks) { set_err(ep.err, kDevBadBlock); return; }
    if (ep.kv_fp8) {
      uint8_t* t8 = reinterpret_cast<uint8_t*>(ep.pool) + pool_tile(ep.layer, ep.n_blocks, blk, ep.hkv, head, 1, hd);
      const uint16_t e = f32x2_e4m3x2(a, b);
      t8[v8_elem(rw.pos & 31, j)] = (uint8_t)(e & 0xff);
      t8[v8_elem(rw.pos & 31, j + 1)] = (uint8_t)(e >> 8);
      return;
    }
    size_t o = pool_off(ep.layer, 1, ep.n_blocks, blk, ep.hkv, head, hd, rw.pos & 31, j);
    ep.pool[o] = f32_to_bf16(a);
    ep.pool[o + 1] = f32_to_bf16(b);
  }
}

// Epilogue for one output feature of one row: residual add or logits store.
__device__ __forceinline__ void epi_single(const EpiArgs& ep, int f, int row, float v) {
  float* p = ep.out_f32 + (size_t)row * ep.ld + f;
  if (ep.kind == kEpiResid) *p += v;
  else *p = v;
}

__device__ __forceinline__ bool epi_is_pair(int kind) { return kind == kEpiQKV || kind == kEpiSwiGLU; }

// Epilogue for NB consecutive rows row0..row0+NB-1 of output feature m held
// by this lane (all 32 lanes of the warp call it; lanes hold consecutive
// features).  Same arithmetic as epi_pair / epi_single, but every global
// read a group of rows needs (residual x, row records, block table, RoPE
// table) is issued before any is used, so a group costs one memory round
// trip instead of one per row.
template <int NB>
__device__ __forceinline__ void epi_rows(const EpiArgs& ep, int m, int lane, int row0, int n, const float (&v)[NB]) {
  float pv[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) pv[j] = __shfl_xor_sync(0xffffffffu, v[j], 1);
  if (ep.kind == kEpiLogits) {
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (row0 + j < n) ep.out_f32[(size_t)(row0 + j) * ep.ld + m] = v[j];
    return;
  }
  if (ep.kind == kEpiResid) {
    float x[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (row0 + j < n) x[j] = ep.out_f32[(size_t)(row0 + j) * ep.ld + m];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (row0 + j < n) ep.out_f32[(size_t)(row0 + j) * ep.ld + m] = x[j] + v[j];
    return;
  }
  if (lane & 1) return;                       // pair kinds: even lane owns (m, m+1)
  if (ep.kind == kEpiSwiGLU) {
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (row0 + j < n) epi_pair(ep, m, row0 + j, v[j], pv[j]);
    return;
  }
  // QKV: row records, then RoPE factors and block ids, then compute + store
  const int hd = ep.hd, half = hd >> 1, nq = ep.hq * hd, nk = ep.hkv * hd;
  RowDev rw[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j)
    if (row0 + j < n) rw[j] = ep.rows[row0 + j];
  if (m < nq) {
    const int head = m / hd, i = (m % hd) >> 1;
    float2 cs[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (row0 + j < n) cs[j] = reinterpret_cast<const float2*>(ep.rope_cs)[(size_t)rw[j].pos * half + i];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (row0 + j < n) {
        float* qrow = ep.out_f32 + (size_t)(row0 + j) * nq + head * hd;
        qrow[i] = v[j] * cs[j].x - pv[j] * cs[j].y;
        qrow[i + half] = pv[j] * cs[j].x + v[j] * cs[j].y;
      }
    return;
  }
  int blk[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j)
    if (row0 + j < n) blk[j] = ep.tables[(size_t)rw[j].slot * ep.max_blocks_per_seq + (rw[j].pos >> 5)];
  if (m < nq + nk) {
    const int head = (m - nq) / hd, i = ((m - nq) % hd) >> 1;
    float2 cs[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (row0 + j < n) cs[j] = reinterpret_cast<const float2*>(ep.rope_cs)[(size_t)rw[j].pos * half + i];
#pragma unroll
    for (int j = 0; j < NB; ++j)
      if (row0 + j < n) {
        if (blk[j] < 0 || blk[j] >= ep.n_blocks) { set_err(ep.err, kDevBadBlock); continue; }
        const size_t t0 = pool_tile(ep.layer, ep.n_blocks, blk[j], ep.hkv, head, 0, hd);
        const float ra = v[j] * cs[j].x - pv[j] * cs[j].y, rb = pv[j] * cs[j].x + v[j] * cs[j].y;
        if (ep.kv_fp8) {
          uint8_t* t8 = reinterpret_cast<uint8_t*>(ep.pool) + t0;
          const uint16_t e = f32x2_e4m3x2(ra, rb);
          t8[k8_elem(hd, rw[j].pos & 31, i)] = (uint8_t)(e & 0xff);
          t8[k8_elem(hd, rw[j].pos & 31, i + half)] = (uint8_t)(e >> 8);
        } else {
          ep.pool[t0 + tile_elem(rw[j].pos & 31, i)] = f32_to_bf16(ra);
          ep.pool[t0 + tile_elem(rw[j].pos & 31, i + half)] = f32_to_bf16(rb);
        }
      }
    return;
  }
  const int fv = m - nq - nk, head = fv / hd, jd = fv % hd;
#pragma unroll
  for (int j = 0; j < NB; ++j)
    if (row0 + j < n) {
      if (blk[j] < 0 || blk[j] >= ep.n_blocks) { set_err(ep.err, kDevBadBlock); continue; }
      if (ep.kv_fp8) {
        uint8_t* t8 = reinterpret_cast<uint8_t*>(ep.pool) + pool_tile(ep.layer, ep.n_blocks, blk[j], ep.hkv, head, 1, hd);
        const uint16_t e = f32x2_e4m3x2(v[j], pv[j]);
        t8[v8_elem(rw[j].pos & 31, jd)] = (uint8_t)(e & 0xff);
        t8[v8_elem(rw[j].pos & 31, jd + 1)] = (uint8_t)(e >> 8);
        continue;
      }
      const size_t o = pool_off(ep.layer, 1, ep.n_blocks, blk[j], ep.hkv, head, hd, rw[j].pos & 31, jd);
      ep.pool[o] = f32_to_bf16(v[j]);
      ep.pool[o + 1] = f32_to_bf16(pv[j]);
    }
}

}  // namespace cbd
