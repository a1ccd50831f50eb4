// Vectorised GEMM epilogues shared by the tensor-core GEMM kernels: four
// consecutive output features of one row at a time, with the one global
// operand a quad needs (the residual x, or the RoPE factors of its two
// rotation pairs) loaded separately by the caller, so that a caller can
// issue the loads of several quads before it uses any of them.  Per element
// the arithmetic is that of epi_pair / epi_single in common.cuh.
#pragma once

#include "tc.cuh"

namespace cbd {

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  return (uint32_t)f32_to_bf16(a) | ((uint32_t)f32_to_bf16(b) << 16);
}

// Address of the epilogue operand that comes from global memory: the
// residual x (residual epilogue) or the RoPE factors (cos, sin) of the
// quad's two rotation pairs (QKV q / k features); null if none.
template <int KIND>
__device__ __forceinline__ const float* epi_pre_addr(const EpiArgs& ep, int row, int fg, const int2* rinfo, int ri) {
  if constexpr (KIND == kEpiResid || KIND == kEpiResidNorm) return ep.out_f32 + (size_t)row * ep.ld + fg;
  if constexpr (KIND == kEpiQKV) {
    const int hd = ep.hd, nq = ep.hq * hd, nk = ep.hkv * hd;
    if (fg < nq + nk) {
      const int i = ((fg < nq ? fg : fg - nq) % hd) >> 1;
      return ep.rope_cs + ((size_t)rinfo[ri].x * (hd >> 1) + i) * 2;
    }
  }
  return nullptr;
}
template <int KIND>
__device__ __forceinline__ float4 epi_preload(const EpiArgs& ep, int row, int fg, const int2* rinfo, int ri) {
  if constexpr (KIND == kEpiResid || KIND == kEpiResidNorm || KIND == kEpiQKV) {
    const float* p = epi_pre_addr<KIND>(ep, row, fg, rinfo, ri);
    if (p) return *reinterpret_cast<const float4*>(p);
  }
  return make_float4(0.f, 0.f, 0.f, 0.f);
}

// Epilogue for one (row, feature quad): features fg..fg+3 (fg % 4 == 0) of
// row `row` with values v.  Per element the arithmetic is that of
// epi_pair / epi_single (the GEMV path's epilogue); stores are 8-16 bytes.
//   QKV: (fg, fg+1) and (fg+2, fg+3) are RoPE partners (dims i, i + hd/2
//        and i+1, i+1 + hd/2 of one q or k head) or four v dims.
//   SwiGLU: (fg, fg+1) = (gate, up) of output fg/2, (fg+2, fg+3) of fg/2+1.
//   ResidNorm: x += v, then split(x * g) of the next norm; returns the
//        quad's sum of x^2 (every other kind returns 0).
template <int KIND>
__device__ __forceinline__ float epi_quad(const EpiArgs& ep, int row, int fg, float4 v, float4 pre,
                                          const int2* rinfo, int ri) {
  if constexpr (KIND == kEpiResidNorm) {
    const float4 x = make_float4(pre.x + v.x, pre.y + v.y, pre.z + v.z, pre.w + v.w);
    *reinterpret_cast<float4*>(ep.out_f32 + (size_t)row * ep.ld + fg) = x;
    const float4 g = *reinterpret_cast<const float4*>(ep.norm_g + fg);
    uint16_t h[4], l[4];
    split_bf16(x.x * g.x, h[0], l[0]);
    split_bf16(x.y * g.y, h[1], l[1]);
    split_bf16(x.z * g.z, h[2], l[2]);
    split_bf16(x.w * g.w, h[3], l[3]);
    const size_t o = (size_t)row * ep.ld + fg;
    *reinterpret_cast<uint2*>(ep.norm_hi + o) =
        make_uint2((uint32_t)h[0] | ((uint32_t)h[1] << 16), (uint32_t)h[2] | ((uint32_t)h[3] << 16));
    *reinterpret_cast<uint2*>(ep.norm_lo + o) =
        make_uint2((uint32_t)l[0] | ((uint32_t)l[1] << 16), (uint32_t)l[2] | ((uint32_t)l[3] << 16));
    return x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
  } else if constexpr (KIND == kEpiLogits) {
    *reinterpret_cast<float4*>(ep.out_f32 + (size_t)row * ep.ld + fg) = v;
  } else if constexpr (KIND == kEpiResid) {
    *reinterpret_cast<float4*>(ep.out_f32 + (size_t)row * ep.ld + fg) =
        make_float4(pre.x + v.x, pre.y + v.y, pre.z + v.z, pre.w + v.w);
  } else if constexpr (KIND == kEpiSwiGLU) {
    const float y0 = silu_mul(v.x, v.y);
    const float y1 = silu_mul(v.z, v.w);
    uint16_t h0, l0, h1, l1;
    split_bf16(y0, h0, l0);
    split_bf16(y1, h1, l1);
    const size_t o = (size_t)row * ep.ld_act + (fg >> 1);
    *reinterpret_cast<uint32_t*>(ep.out_hi + o) = (uint32_t)h0 | ((uint32_t)h1 << 16);
    *reinterpret_cast<uint32_t*>(ep.out_lo + o) = (uint32_t)l0 | ((uint32_t)l1 << 16);
  } else {
    const int hd = ep.hd, half = hd >> 1, nq = ep.hq * hd, nk = ep.hkv * hd;
    const int pos = rinfo[ri].x;
    if (fg < nq + nk) {
      const float r0 = v.x * pre.x - v.y * pre.y, r1 = v.y * pre.x + v.x * pre.y;   // dims i, i + half
      const float r2 = v.z * pre.z - v.w * pre.w, r3 = v.w * pre.z + v.z * pre.w;   // dims i + 1, i + 1 + half
      const int fh = fg < nq ? fg : fg - nq;
      const int head = fh / hd, i = (fh % hd) >> 1;
      if (fg < nq) {
        float* qrow = ep.out_f32 + (size_t)row * nq + head * hd;
        *reinterpret_cast<float2*>(qrow + i) = make_float2(r0, r2);
        *reinterpret_cast<float2*>(qrow + i + half) = make_float2(r1, r3);
        return 0.f;
      }
      const int blk = rinfo[ri].y;
      if (blk < 0 || blk >= ep.n_blocks) { set_err(ep.err, kDevBadBlock); return 0.f; }
      const size_t t0 = pool_tile(ep.layer, ep.n_blocks, blk, ep.hkv, head, 0, hd);
      if (ep.kv_fp8) {          // dims (i, i + 1) and (i + half, i + half + 1): two adjacent bytes each
        uint8_t* t8 = reinterpret_cast<uint8_t*>(ep.pool) + t0;
        *reinterpret_cast<uint16_t*>(t8 + k8_elem(hd, pos & 31, i)) = f32x2_e4m3x2(r0, r2);
        *reinterpret_cast<uint16_t*>(t8 + k8_elem(hd, pos & 31, i + half)) = f32x2_e4m3x2(r1, r3);
        return 0.f;
      }
      *reinterpret_cast<uint32_t*>(ep.pool + t0 + tile_elem(pos & 31, i)) = pack_bf16x2(r0, r2);
      *reinterpret_cast<uint32_t*>(ep.pool + t0 + tile_elem(pos & 31, i + half)) = pack_bf16x2(r1, r3);
      return 0.f;
    }
    const int blk = rinfo[ri].y;
    if (blk < 0 || blk >= ep.n_blocks) { set_err(ep.err, kDevBadBlock); return 0.f; }
    const int fv = fg - nq - nk, head = fv / hd, jd = fv % hd;
    if (ep.kv_fp8) {            // V is stored transposed: the 4 dims are 4 rows of the tile
      uint8_t* t8 = reinterpret_cast<uint8_t*>(ep.pool) + pool_tile(ep.layer, ep.n_blocks, blk, ep.hkv, head, 1, hd);
      const uint16_t e01 = f32x2_e4m3x2(v.x, v.y), e23 = f32x2_e4m3x2(v.z, v.w);
      t8[v8_elem(pos & 31, jd)] = (uint8_t)(e01 & 0xff);
      t8[v8_elem(pos & 31, jd + 1)] = (uint8_t)(e01 >> 8);
      t8[v8_elem(pos & 31, jd + 2)] = (uint8_t)(e23 & 0xff);
      t8[v8_elem(pos & 31, jd + 3)] = (uint8_t)(e23 >> 8);
      return 0.f;
    }
    const size_t o = pool_off(ep.layer, 1, ep.n_blocks, blk, ep.hkv, head, hd, pos & 31, jd);
    *reinterpret_cast<uint2*>(ep.pool + o) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
  return 0.f;
}

}  // namespace cbd
