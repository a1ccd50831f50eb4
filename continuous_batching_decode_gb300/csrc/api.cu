// libcbd C ABI: engine, KV pool, batch (validated step inputs) and the step
// launch sequence.  The Scheduler (sched.cpp) decides what runs; a Batch
// runs it -- the split "20.3 服务、批处理与流式" section 20.3.2 describes for
// Forma, which keeps admission bugs and batching bugs apart.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <memory>
#include <string>
#include <vector>

#include "common.cuh"

namespace cbd {

static thread_local std::string g_err;

cbd_status fail(cbd_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}
void clear_error() { g_err.clear(); }

static cbd_status cuda_fail(cudaError_t err, const char* what) {
  return fail(err == cudaErrorMemoryAllocation ? CBD_ENOMEM : CBD_ECUDA, "%s: %s", what, cudaGetErrorString(err));
}

// Entry points that enqueue work, synchronise or allocate for an engine run
// on the engine's device, whichever device is current in the calling thread.
#define CBD_ON_DEVICE(dev_)                                                   \
  DeviceGuard _dg(dev_);                                                      \
  if (!_dg.ok()) return fail(CBD_ECUDA, "cannot make device %d current", (int)(dev_))

#define CBD_CUDA(call)                                   \
  do {                                                   \
    cudaError_t _e = (call);                             \
    if (_e != cudaSuccess) return cuda_fail(_e, #call);  \
  } while (0)

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Kernel classes for cbd_engine_profile.
static const char* kKernelClass[] = {"embed", "rmsnorm", "gemm_qkv", "attention", "gemm_o",
                                     "gemm_gate_up", "gemm_down", "final_norm", "gemm_lm_head", "sampler",
                                     "gemm_chain"};
enum KClass { kcEmbed, kcNorm, kcQKV, kcAttn, kcO, kcGU, kcDown, kcFinal, kcLM, kcSamp, kcChain, kcCount };


// ---------------------------------------------------------------- repack
// Weight layout for the kernels: row r of the (row-permuted) matrix, column
// k, lives at [r / 256][k / 64][r % 256][k % 64] -- 32 KB tiles of 256 rows
// by 64 columns, each one contiguous.  perm (nullable) gives the source row
// of each destination row.
__global__ void permute_tile_kernel(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src,
                                    const int32_t* __restrict__ perm, int K, int N) {
  const int r = blockIdx.x;
  const int sr = perm ? perm[r] : r;
  const int KB = K / 64;
  const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)sr * K);
  for (int c = threadIdx.x; c < K / 8; c += blockDim.x) {
    const int k = c * 8;
    *reinterpret_cast<uint4*>(dst + tiled_off(r, k, N, KB)) = s[c];
  }
}
// Per-row int8 quantisation (cbd_config.weights_int8) of a row-major bf16
// matrix [.][K] into the tiled layout (byte (r, k) at tiled_off(r, k, N,
// K / 64)): destination row r takes source row perm[r] (or r).  Per row:
// s = fp32(max|w| / 127) (IEEE single division), q = w / s in fp64 rounded
// to the nearest integer, ties to even, clamped to [-127, 127]; s = 0 gives
// q = 0.  One CTA per row.
__global__ void quantize_tile_kernel(uint8_t* __restrict__ dst, float* __restrict__ scale,
                                     const uint16_t* __restrict__ src, const int32_t* __restrict__ perm, int K,
                                     int N) {
  __shared__ float red[32];
  const int r = blockIdx.x;
  const int sr = perm ? perm[r] : r;
  const uint16_t* row = src + (size_t)sr * K;
  float m = 0.f;
  for (int k = threadIdx.x; k < K; k += blockDim.x) m = fmaxf(m, fabsf(bf16_to_f32(row[k])));
  m = warp_max(m);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) red[w] = m;
  __syncthreads();
  if (w == 0) {
    m = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
    m = warp_max(m);
    if (lane == 0) red[0] = m;
  }
  __syncthreads();
  const float s = __fdiv_rn(red[0], 127.0f);
  if (threadIdx.x == 0) scale[r] = s;
  const int KB = K / 64;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    int q = 0;
    if (s > 0.f) {
      const double v = rint((double)bf16_to_f32(row[k]) / (double)s);
      q = (int)fmin(fmax(v, -127.0), 127.0);
    }
    dst[tiled_off(r, k, N, KB)] = (uint8_t)(int8_t)q;
  }
}
// Tiled matrix (elements of `eb` bytes, N rows per tile) -> row-major [M][K].
__global__ void untile_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src, int K, int N, int eb) {
  const int r = blockIdx.x;
  const int KB = K / 64;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    const size_t o = tiled_off(r, k, N, KB) * (size_t)eb;
    for (int b = 0; b < eb; ++b) dst[((size_t)r * K + k) * eb + b] = src[o + b];
  }
}
__global__ void bf16_to_f32_kernel(float* __restrict__ dst, const uint16_t* __restrict__ src, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = bf16_to_f32(src[i]);
}

struct Arena {
  size_t off = 0;
  size_t take(size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  }
};

}  // namespace cbd

using namespace cbd;

extern "C" {

const char* cbd_last_error(void) { return g_err.c_str(); }
const char* cbd_version(void) { return "cbd 0.1 sm_103a"; }

}  // extern "C"

namespace {

cbd_status check_config(const cbd_config* c) {
  if (!c) return fail(CBD_EINVAL, "cfg is NULL");
  if (c->n_layers < 1 || c->d_model < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 1 ||
      c->ffn_dim < 1 || c->vocab < 1)
    return fail(CBD_EINVAL, "model dimensions must be positive");
  if (c->n_heads % c->n_kv_heads) return fail(CBD_EINVAL, "n_kv_heads must divide n_heads");
  if (c->block_size != kBlock) return fail(CBD_EINVAL, "block_size must be 32");
  if (c->max_rows < 1 || c->max_rows > 4096) return fail(CBD_EINVAL, "max_rows must be in [1, 4096]");
  if (c->max_slots < 1 || c->max_slots > 65536) return fail(CBD_EINVAL, "max_slots out of range");
  if (c->max_blocks_per_seq < 1 || c->max_blocks_per_seq > 65536)
    return fail(CBD_EINVAL, "max_blocks_per_seq out of range");
  if (!(c->rope_base > 0.f) || !(c->rms_eps >= 0.f)) return fail(CBD_EINVAL, "rope_base/rms_eps invalid");
  if (c->head_dim != 64 && c->head_dim != 128) return fail(CBD_EUNSUPPORTED, "head_dim must be 64 or 128");
  if (c->kv_fp8 != 0 && c->kv_fp8 != 1) return fail(CBD_EINVAL, "kv_fp8 must be 0 or 1");
  if (c->weights_int8 != 0 && c->weights_int8 != 1) return fail(CBD_EINVAL, "weights_int8 must be 0 or 1");
  const int g = c->n_heads / c->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return fail(CBD_EUNSUPPORTED, "n_heads/n_kv_heads must be 1, 2, 4 or 8");
  if (c->d_model % 256 || c->ffn_dim % 256 || (c->n_heads * c->head_dim) % 256)
    return fail(CBD_EUNSUPPORTED, "d_model, ffn_dim and n_heads*head_dim must be multiples of 256");
  if (c->vocab > kMaxVocab || c->vocab % 256) return fail(CBD_EUNSUPPORTED, "vocab must be a multiple of 256, <= 65536");
  if (((c->n_heads + 2 * c->n_kv_heads) * c->head_dim) % 256)
    return fail(CBD_EUNSUPPORTED, "(n_heads + 2 n_kv_heads) * head_dim must be a multiple of 256");
  return CBD_OK;
}

// Copy `bytes` from a host or device source into device memory.
cbd_status upload(void* dst, const void* src, size_t bytes, bool on_device) {
  if (!src) return fail(CBD_EINVAL, "a weight pointer is NULL");
  CBD_CUDA(cudaMemcpy(dst, src, bytes, on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice));
  return CBD_OK;
}

}  // namespace

extern "C" cbd_status cbd_engine_create(const cbd_config* cfg, const cbd_weights* w, cbd_engine** out) {
  clear_error();
  if (!out) return fail(CBD_EINVAL, "out is NULL");
  *out = nullptr;
  cbd_status st = check_config(cfg);
  if (st) return st;
  if (!w || !w->layers) return fail(CBD_EINVAL, "weights are NULL");
  int dev = 0;
  CBD_CUDA(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  CBD_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3)
    return fail(CBD_EUNSUPPORTED, "libcbd is built for sm_103a; device %d is sm_%d%d", dev, prop.major, prop.minor);

  auto e = std::make_unique<cbd_engine>();
  e->cfg = *cfg;
  e->device = dev;
  e->sm_count = prop.multiProcessorCount;
  Dims& dm = e->dm;
  dm.L = cfg->n_layers; dm.d = cfg->d_model; dm.hq = cfg->n_heads; dm.hkv = cfg->n_kv_heads;
  dm.hd = cfg->head_dim; dm.F = cfg->ffn_dim; dm.V = cfg->vocab;
  dm.qkv_out = (dm.hq + 2 * dm.hkv) * dm.hd;
  dm.max_rows = cfg->max_rows; dm.max_slots = cfg->max_slots; dm.max_blocks_per_seq = cfg->max_blocks_per_seq;
  dm.rope_base = cfg->rope_base; dm.eps = cfg->rms_eps;
  e->kv_fp8 = cfg->kv_fp8 != 0;
  e->w_int8 = cfg->weights_int8 != 0;
  e->max_pos = dm.max_blocks_per_seq * kBlock;
  const bool ondev = w->on_device != 0;
  CBD_CUDA(cudaDeviceSynchronize());   // weights produced on any stream are complete
  const size_t d = dm.d, V = dm.V, F = dm.F, qo = dm.qkv_out, hqd = (size_t)dm.hq * dm.hd;

  // ---- weight arena (streamed matrices: bf16, or int8 plus per-row fp32 scales)
  const bool i8 = e->w_int8;
  const size_t eb = i8 ? 1 : 2;
  auto sc = [&](Arena& a, size_t rows) { return i8 ? a.take(rows * 4) : (size_t)0; };
  Arena A;
  const size_t o_embed = A.take(V * d * 2), o_lm = A.take(V * d * eb), s_lm = sc(A, V), o_fn = A.take(d * 4);
  std::vector<size_t> o_an(dm.L), o_fnn(dm.L), o_qkv(dm.L), o_o(dm.L), o_gu(dm.L), o_dn(dm.L);
  std::vector<size_t> s_qkv(dm.L), s_o(dm.L), s_gu(dm.L), s_dn(dm.L);
  for (int l = 0; l < dm.L; ++l) {
    o_an[l] = A.take(d * 4); o_fnn[l] = A.take(d * 4);
    o_qkv[l] = A.take(qo * d * eb); s_qkv[l] = sc(A, qo);
    o_o[l] = A.take(d * hqd * eb); s_o[l] = sc(A, d);
    o_gu[l] = A.take(2 * F * d * eb); s_gu[l] = sc(A, 2 * F);
    o_dn[l] = A.take(d * F * eb); s_dn[l] = sc(A, d);
  }
  const size_t o_rope = A.take((size_t)e->max_pos * (dm.hd / 2) * 2 * 4);
  e->arena_bytes = A.off;
  CBD_CUDA(cudaMalloc(&e->arena, e->arena_bytes));
  auto cleanup = [&]() {
    if (e->arena) cudaFree(e->arena);
    e->arena = nullptr;
  };
  uint8_t* base = static_cast<uint8_t*>(e->arena);
  e->embed = reinterpret_cast<uint16_t*>(base + o_embed);
  if (i8) {
    e->lm_q = base + o_lm;
    e->lm_scale = reinterpret_cast<float*>(base + s_lm);
  } else {
    e->lm_head = reinterpret_cast<uint16_t*>(base + o_lm);
  }
  e->final_norm = reinterpret_cast<float*>(base + o_fn);
  e->rope_cs = reinterpret_cast<float*>(base + o_rope);

  // temporary device buffers: the largest source matrix, a permutation, a gain
  const size_t tmp_elems = std::max({qo * d, 2 * F * d, d * F, d * hqd, V * d});
  void* tmp = nullptr;
  int32_t* perm_d = nullptr;
  cudaError_t ce = cudaMalloc(&tmp, tmp_elems * 2);
  if (ce == cudaSuccess) ce = cudaMalloc(&perm_d, std::max(qo, 2 * F) * sizeof(int32_t));
  if (ce != cudaSuccess) {
    if (tmp) cudaFree(tmp);
    cleanup();
    return cuda_fail(ce, "cudaMalloc(repack temporaries)");
  }
  auto free_tmp = [&]() { cudaFree(tmp); cudaFree(perm_d); };
  auto gain = [&](size_t off, const void* src) -> cbd_status {
    cbd_status s2 = upload(tmp, src, d * 2, ondev);
    if (s2) return s2;
    bf16_to_f32_kernel<<<(int)((d + 255) / 256), 256>>>(reinterpret_cast<float*>(base + off),
                                                          static_cast<uint16_t*>(tmp), (int)d);
    CBD_CUDA(cudaGetLastError());
    return CBD_OK;
  };
  // tile widths (weight rows per tile) per matrix shape, for this GPU
  e->tile_qkv = gemm_tc_pick_tile((int)qo, (int)d);
  e->tile_o = gemm_tc_pick_tile((int)d, (int)hqd);
  e->tile_gu = gemm_tc_pick_tile((int)(2 * F), (int)d);
  e->tile_dn = gemm_tc_pick_tile((int)d, (int)F);
  e->tile_lm = gemm_tc_pick_tile((int)V, (int)d);
  // tmp (row-major [M][K]) -> arena (tiled, N rows per tile), rows permuted
  // when perm is given; int8 engines quantise each row on the way (scales
  // at soff, in the same row order)
  auto tiled = [&](size_t off, size_t soff, const std::vector<int32_t>* perm, int M, int K, int N) -> cbd_status {
    if (perm) CBD_CUDA(cudaMemcpy(perm_d, perm->data(), perm->size() * 4, cudaMemcpyHostToDevice));
    if (i8)
      quantize_tile_kernel<<<M, 256>>>(base + off, reinterpret_cast<float*>(base + soff), static_cast<uint16_t*>(tmp),
                                       perm ? perm_d : nullptr, K, N);
    else
      permute_tile_kernel<<<M, 256>>>(reinterpret_cast<uint16_t*>(base + off), static_cast<uint16_t*>(tmp),
                                      perm ? perm_d : nullptr, K, N);
    CBD_CUDA(cudaGetLastError());
    CBD_CUDA(cudaDeviceSynchronize());
    return CBD_OK;
  };
  // Row orders (then tiled, see permute_tile_kernel): q and k rows within each head become (i, i + hd/2) pairs so
  // the RoPE partners are adjacent outputs; gate/up rows interleave so
  // SwiGLU partners are adjacent.  v, o, down, embed, lm_head keep their order.
  std::vector<int32_t> perm_qkv(qo), perm_gu(2 * F);
  {
    const int hd = dm.hd, half = hd / 2;
    for (int h = 0; h < dm.hq + dm.hkv; ++h)
      for (int i = 0; i < half; ++i) {
        perm_qkv[(size_t)h * hd + 2 * i] = h * hd + i;
        perm_qkv[(size_t)h * hd + 2 * i + 1] = h * hd + i + half;
      }
    for (size_t r = (size_t)(dm.hq + dm.hkv) * hd; r < qo; ++r) perm_qkv[r] = (int32_t)r;
    for (int i = 0; i < dm.F; ++i) { perm_gu[2 * i] = i; perm_gu[2 * i + 1] = dm.F + i; }
  }
  cbd_status s2 = CBD_OK;
#define TRY(x) do { s2 = (x); if (s2) { free_tmp(); cleanup(); return s2; } } while (0)
  TRY(upload(base + o_embed, w->embed, V * d * 2, ondev));
  TRY(upload(tmp, w->lm_head, V * d * 2, ondev));
  TRY(tiled(o_lm, s_lm, nullptr, (int)V, (int)d, e->tile_lm));
  TRY(gain(o_fn, w->final_norm));
  e->layers.resize(dm.L);
  for (int l = 0; l < dm.L; ++l) {
    const cbd_layer_weights& lw = w->layers[l];
    TRY(gain(o_an[l], lw.attn_norm));
    TRY(gain(o_fnn[l], lw.ffn_norm));
    uint8_t* t = static_cast<uint8_t*>(tmp);
    TRY(upload(t, lw.wq, hqd * d * 2, ondev));
    TRY(upload(t + hqd * d * 2, lw.wk, (size_t)dm.hkv * dm.hd * d * 2, ondev));
    TRY(upload(t + (hqd + (size_t)dm.hkv * dm.hd) * d * 2, lw.wv, (size_t)dm.hkv * dm.hd * d * 2, ondev));
    TRY(tiled(o_qkv[l], s_qkv[l], &perm_qkv, (int)qo, (int)d, e->tile_qkv));
    TRY(upload(t, lw.wo, d * hqd * 2, ondev));
    TRY(tiled(o_o[l], s_o[l], nullptr, (int)d, (int)hqd, e->tile_o));
    TRY(upload(t, lw.w_gate, F * d * 2, ondev));
    TRY(upload(t + F * d * 2, lw.w_up, F * d * 2, ondev));
    TRY(tiled(o_gu[l], s_gu[l], &perm_gu, (int)(2 * F), (int)d, e->tile_gu));
    TRY(upload(t, lw.w_down, d * F * 2, ondev));
    TRY(tiled(o_dn[l], s_dn[l], nullptr, (int)d, (int)F, e->tile_dn));
    LayerDev& L = e->layers[l];
    L = LayerDev{};
    L.attn_norm = reinterpret_cast<float*>(base + o_an[l]);
    L.ffn_norm = reinterpret_cast<float*>(base + o_fnn[l]);
    if (i8) {
      L.q_qkv = base + o_qkv[l]; L.s_qkv = reinterpret_cast<float*>(base + s_qkv[l]);
      L.q_o = base + o_o[l]; L.s_o = reinterpret_cast<float*>(base + s_o[l]);
      L.q_gu = base + o_gu[l]; L.s_gu = reinterpret_cast<float*>(base + s_gu[l]);
      L.q_down = base + o_dn[l]; L.s_down = reinterpret_cast<float*>(base + s_dn[l]);
    } else {
      L.w_qkv = reinterpret_cast<uint16_t*>(base + o_qkv[l]);
      L.w_o = reinterpret_cast<uint16_t*>(base + o_o[l]);
      L.w_gu = reinterpret_cast<uint16_t*>(base + o_gu[l]);
      L.w_down = reinterpret_cast<uint16_t*>(base + o_dn[l]);
    }
  }
#undef TRY
  free_tmp();
  {  // RoPE table: fp64 angles rounded to fp32, [pos][i] = (cos, sin)
    const int half = dm.hd / 2;
    std::vector<float> cs((size_t)e->max_pos * half * 2);
    for (int p = 0; p < e->max_pos; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = (double)p * std::pow((double)dm.rope_base, -2.0 * i / dm.hd);
        cs[((size_t)p * half + i) * 2] = (float)std::cos(ang);
        cs[((size_t)p * half + i) * 2 + 1] = (float)std::sin(ang);
      }
    cudaError_t e2 = cudaMemcpy(base + o_rope, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice);
    if (e2 != cudaSuccess) { cleanup(); return cuda_fail(e2, "upload RoPE table"); }
  }

  // ---- workspaces
  const size_t R = dm.max_rows, S = dm.max_slots;
  const size_t act_w = std::max(d, hqd);
  const size_t chunks_per_seq = ((size_t)e->max_pos + kAttnChunk - 1) / kAttnChunk;
  e->max_work = (int)std::min<size_t>(R * chunks_per_seq, (size_t)1 << 16);
  Arena W;
  // GEMM inputs: rows padded to whole activation boxes
  const size_t RA = (R + kActBoxRows - 1) / kActBoxRows * kActBoxRows;
  const size_t o_x = W.take(R * d * 4), o_ah = W.take(RA * act_w * 2), o_al = W.take(RA * act_w * 2);
  const size_t o_fh = W.take(RA * F * 2), o_fl = W.take(RA * F * 2), o_q = W.take(R * hqd * 4);
  const size_t o_nh = W.take(RA * d * 2), o_nl = W.take(RA * d * 2), o_ssq = W.take(R * kMaxSsqParts * 4);
  const size_t o_ao = W.take((size_t)e->max_work * hqd * 4), o_aml = W.take((size_t)e->max_work * dm.hq * 2 * 4);
  const size_t o_lg = W.take(S * V * 4), o_sc = W.take(S * V * 4), o_cn = W.take(S * V * 4), o_err = W.take(16);
  const size_t o_fb = W.take((V + 31) / 32 * 4);
  const size_t o_last = W.take(S * 4);
  // per layer: the attention task counter, then the GEMM chain's barriers
  const size_t o_anext = W.take((size_t)dm.L * (1 + kChainMaxPhases) * 4);

  e->work_bytes = W.off;
  cudaError_t e3 = cudaMalloc(&e->work, e->work_bytes);
  if (e3 != cudaSuccess) { cleanup(); return cuda_fail(e3, "cudaMalloc(workspaces)"); }
  uint8_t* wb = static_cast<uint8_t*>(e->work);
  e->x = reinterpret_cast<float*>(wb + o_x);
  e->act_hi = reinterpret_cast<uint16_t*>(wb + o_ah);
  e->act_lo = reinterpret_cast<uint16_t*>(wb + o_al);
  e->norm_hi = reinterpret_cast<uint16_t*>(wb + o_nh);
  e->norm_lo = reinterpret_cast<uint16_t*>(wb + o_nl);
  e->ssq = reinterpret_cast<float*>(wb + o_ssq);
  e->ffn_hi = reinterpret_cast<uint16_t*>(wb + o_fh);
  e->ffn_lo = reinterpret_cast<uint16_t*>(wb + o_fl);
  e->q = reinterpret_cast<float*>(wb + o_q);
  e->attn_o = reinterpret_cast<float*>(wb + o_ao);
  e->attn_ml = reinterpret_cast<float*>(wb + o_aml);
  e->logits = reinterpret_cast<float*>(wb + o_lg);
  e->samp_scratch = reinterpret_cast<float*>(wb + o_sc);
  e->counters = reinterpret_cast<float*>(wb + o_cn);
  e->forbid = reinterpret_cast<uint32_t*>(wb + o_fb);
  e->last_tok = reinterpret_cast<int32_t*>(wb + o_last);
  e->err = reinterpret_cast<int32_t*>(wb + o_err);
  e->attn_next = reinterpret_cast<int32_t*>(wb + o_anext);
  e->chain_sync = reinterpret_cast<uint32_t*>(wb + o_anext + (size_t)dm.L * 4);

  e3 = cudaMemset(e->work, 0, e->work_bytes);
  // ---- staging for cbd_step / cbd_sample
  const size_t stage_bytes = align_up(R * sizeof(RowDev), 16) + 2 * align_up(S * 4, 16) +
                             align_up(S * sizeof(SampDev), 16) + align_up(S * dm.max_blocks_per_seq * 4, 16) +
                             align_up((size_t)e->max_work * sizeof(AttnWork), 16) + align_up((R + 1) * 4, 16) +
                             align_up(R * sizeof(PfBlock), 16) + 2 * align_up(R * 4, 16) + 256;
  for (auto& sg : e->stage) {
    if (e3 == cudaSuccess) e3 = cudaMallocHost(&sg.host, stage_bytes);
    if (e3 == cudaSuccess) e3 = cudaMalloc(&sg.dev, stage_bytes);
    if (e3 == cudaSuccess) e3 = cudaEventCreateWithFlags(&sg.done, cudaEventDisableTiming);
    sg.bytes = stage_bytes;
  }
  if (e3 == cudaSuccess) e3 = cudaDeviceSynchronize();
  if (e3 != cudaSuccess) {
    cbd_engine* raw = e.release();
    cbd_engine_destroy(raw);
    return cuda_fail(e3, "engine workspaces");
  }
  // tensor maps for the tcgen05 GEMM: weights (one tile per box) and the
  // activation matrices in each layout the step uses (box 64 rows)
  {
    const int L = dm.L;
    e->tmaps.resize((size_t)4 * L + 1 + 8);
    bool ok = true;
    for (int l = 0; l < L && ok; ++l) {
      const LayerDev& Ld = e->layers[l];
      // tiled weights: a [M*K/64][64] matrix, one N-row box per tile (int8: 64 bytes per row)
      if (i8) {
        ok = ok && make_tmap_i8(&e->tmaps[4 * l + 0], Ld.q_qkv, qo * d / 64, e->tile_qkv);
        ok = ok && make_tmap_i8(&e->tmaps[4 * l + 1], Ld.q_o, d * hqd / 64, e->tile_o);
        ok = ok && make_tmap_i8(&e->tmaps[4 * l + 2], Ld.q_gu, 2 * F * d / 64, e->tile_gu);
        ok = ok && make_tmap_i8(&e->tmaps[4 * l + 3], Ld.q_down, d * F / 64, e->tile_dn);
      } else {
        ok = ok && make_tmap_bf16(&e->tmaps[4 * l + 0], Ld.w_qkv, 64, qo * d / 64, 64, e->tile_qkv);
        ok = ok && make_tmap_bf16(&e->tmaps[4 * l + 1], Ld.w_o, 64, d * hqd / 64, 64, e->tile_o);
        ok = ok && make_tmap_bf16(&e->tmaps[4 * l + 2], Ld.w_gu, 64, 2 * F * d / 64, 64, e->tile_gu);
        ok = ok && make_tmap_bf16(&e->tmaps[4 * l + 3], Ld.w_down, 64, d * F / 64, 64, e->tile_dn);
      }
    }
    const size_t a0 = (size_t)4 * L + 1;
    ok = ok && (i8 ? make_tmap_i8(&e->tmaps[4 * L], e->lm_q, V * d / 64, e->tile_lm)
                   : make_tmap_bf16(&e->tmaps[4 * L], e->lm_head, 64, V * d / 64, 64, e->tile_lm));
    ok = ok && make_tmap_bf16(&e->tmaps[a0 + 0], e->act_hi, d, RA, d, kActBoxRows);
    ok = ok && make_tmap_bf16(&e->tmaps[a0 + 1], e->act_lo, d, RA, d, kActBoxRows);
    ok = ok && make_tmap_bf16(&e->tmaps[a0 + 2], e->act_hi, hqd, RA, hqd, kActBoxRows);
    ok = ok && make_tmap_bf16(&e->tmaps[a0 + 3], e->act_lo, hqd, RA, hqd, kActBoxRows);
    ok = ok && make_tmap_bf16(&e->tmaps[a0 + 4], e->ffn_hi, F, RA, F, kActBoxRows);
    ok = ok && make_tmap_bf16(&e->tmaps[a0 + 5], e->ffn_lo, F, RA, F, kActBoxRows);
    ok = ok && make_tmap_bf16(&e->tmaps[a0 + 6], e->norm_hi, d, RA, d, kActBoxRows);
    ok = ok && make_tmap_bf16(&e->tmaps[a0 + 7], e->norm_lo, d, RA, d, kActBoxRows);
    if (!ok) {
      cbd_engine* raw = e.release();
      cbd_engine_destroy(raw);
      return fail(CBD_ECUDA, "cuTensorMapEncodeTiled failed (driver entry point missing or bad layout)");
    }
  }
  e->step_batch = new cbd_batch();
  e->step_batch->owns_dev = false;
  e->step_batch->device = e->device;
  *out = e.release();
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_destroy(cbd_engine* e) {
  if (!e) return CBD_OK;
  DeviceGuard dg(e->device);
  cudaDeviceSynchronize();
  for (auto& sg : e->stage) {
    if (sg.host) cudaFreeHost(sg.host);
    if (sg.dev) cudaFree(sg.dev);
    if (sg.done) cudaEventDestroy(sg.done);
  }
  if (e->work) cudaFree(e->work);
  if (e->arena) cudaFree(e->arena);
  for (auto& r : e->prof_recs) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
  for (auto ev : e->prof_free) cudaEventDestroy(ev);
  for (auto& cache : e->step_graphs)
    for (auto& g : cache) cudaGraphExecDestroy(g.exec);
  if (e->cap_stream) cudaStreamDestroy(e->cap_stream);
  delete e->step_batch;
  delete e;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_check(cbd_engine* e) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  CBD_ON_DEVICE(e->device);
  CBD_CUDA(cudaDeviceSynchronize());
  int32_t v = 0;
  CBD_CUDA(cudaMemcpy(&v, e->err, 4, cudaMemcpyDeviceToHost));
  if (v) {
    CBD_CUDA(cudaMemset(e->err, 0, 4));
    return fail(CBD_EDEVICE, "device error code %d", v);
  }
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_test_wait_timeout(cbd_engine* e, int64_t limit_cycles, void* stream) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  if (limit_cycles < 1 || limit_cycles > ((int64_t)1 << 31))
    return fail(CBD_EINVAL, "limit_cycles %lld not in [1, 2^31]", (long long)limit_cycles);
  CBD_ON_DEVICE(e->device);
  CBD_CUDA(launch_wait_probe((long long)limit_cycles, e->err, static_cast<cudaStream_t>(stream)));
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_profile(cbd_engine* e, int32_t enable) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  CBD_ON_DEVICE(e->device);
  CBD_CUDA(cudaDeviceSynchronize());
  for (auto& r : e->prof_recs) { e->prof_free.push_back(r.a); e->prof_free.push_back(r.b); }
  e->prof_recs.clear();
  e->prof = enable != 0;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_profile_read(cbd_engine* e, cbd_kernel_stat* out, int32_t cap, int32_t* n) {
  clear_error();
  if (!e || !n) return fail(CBD_EINVAL, "NULL argument");
  CBD_ON_DEVICE(e->device);
  CBD_CUDA(cudaDeviceSynchronize());
  std::vector<double> ms(kcCount, 0.0);
  std::vector<int64_t> cnt(kcCount, 0);
  for (auto& r : e->prof_recs) {
    float t = 0.f;
    CBD_CUDA(cudaEventElapsedTime(&t, r.a, r.b));
    ms[r.cls] += t;
    cnt[r.cls]++;
  }
  int32_t k = 0;
  for (int c = 0; c < kcCount; ++c) {
    if (!cnt[c]) continue;
    if (out && k < cap) {
      std::memset(&out[k], 0, sizeof(out[k]));
      std::strncpy(out[k].name, kKernelClass[c], sizeof(out[k].name) - 1);
      out[k].launches = cnt[c];
      out[k].total_ms = ms[c];
    }
    ++k;
  }
  *n = std::min(k, cap);
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_gemm_path(cbd_engine* e, int32_t path, int32_t gemv_max_rows) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  if (path < 0 || path > 2) return fail(CBD_EINVAL, "gemm path must be 0, 1 or 2");
  if (e->w_int8 && path == 1) return fail(CBD_EUNSUPPORTED, "an int8-weight engine has no CUDA-core GEMV path");
  if (gemv_max_rows < 0) return fail(CBD_EINVAL, "gemv_max_rows must be >= 0");
  e->gemm_path = path;
  ++e->epoch;
  e->gemv_max_rows = gemv_max_rows;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_prefill_attention(cbd_engine* e, int32_t enable) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  e->prefill_attn = enable != 0;
  ++e->epoch;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_rows_gemm(cbd_engine* e, int32_t min_rows, int32_t force) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  if (min_rows < 0) return fail(CBD_EINVAL, "min_rows must be >= 0");
  e->rows_gemm_min = min_rows;
  e->rows_gemm_force = force != 0;
  ++e->epoch;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_attention_path(cbd_engine* e, int32_t path) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  if (path < 0 || path > 2) return fail(CBD_EINVAL, "attention path must be 0, 1 or 2");
  if (e->kv_fp8 && path != 0) return fail(CBD_EUNSUPPORTED, "an FP8 KV engine has attention path 0 only");
  e->attn_path = path;
  ++e->epoch;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_fused_norm(cbd_engine* e, int32_t enable) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  e->fuse_norm = enable != 0;
  ++e->epoch;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_gemm_chain(cbd_engine* e, int32_t enable) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  e->gemm_chain = enable != 0;
  ++e->epoch;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_forbidden(cbd_engine* e, const int32_t* ids, int32_t n) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  CBD_ON_DEVICE(e->device);
  const int64_t V = e->dm.V;
  if (n < 0 || n >= V) return fail(CBD_EINVAL, "%d forbidden ids: must be 0..vocab-1", (int)n);
  if (n > 0 && !ids) return fail(CBD_EINVAL, "ids is NULL");
  std::vector<uint32_t> bits((size_t)(V + 31) / 32, 0u);
  int32_t distinct = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= V) return fail(CBD_EINVAL, "forbidden id %d outside the vocabulary", (int)ids[i]);
    uint32_t& w = bits[(size_t)ids[i] >> 5];
    const uint32_t b = 1u << (ids[i] & 31);
    if (!(w & b)) ++distinct;
    w |= b;
  }
  if (distinct >= V) return fail(CBD_EINVAL, "every token id is forbidden");
  cudaError_t ce = cudaDeviceSynchronize();      // no step in flight reads the old mask
  if (ce == cudaSuccess) ce = cudaMemcpy(e->forbid, bits.data(), bits.size() * 4, cudaMemcpyHostToDevice);
  if (ce != cudaSuccess) return cuda_fail(ce, "forbidden-token mask");
  e->n_forbidden = distinct;
  ++e->epoch;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_l2_prefetch(cbd_engine* e, uint64_t bytes) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  if (bytes > ((uint64_t)1 << 30)) return fail(CBD_EINVAL, "prefetch of %llu bytes is more than 1 GiB",
                                              (unsigned long long)bytes);
  e->l2_prefetch = (size_t)bytes;
  ++e->epoch;
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_read_weight(cbd_engine* e, int32_t which, int32_t layer, void* dst, float* scales) {
  clear_error();
  if (!e || !dst) return fail(CBD_EINVAL, "NULL argument");
  if (which < 0 || which > 4) return fail(CBD_EINVAL, "matrix %d: must be 0..4", which);
  if (which < 4 && (layer < 0 || layer >= e->dm.L)) return fail(CBD_EINVAL, "layer %d out of range", layer);
  CBD_ON_DEVICE(e->device);
  const Dims& dm = e->dm;
  const int hqd = dm.hq * dm.hd;
  const void* src = nullptr;
  const float* sc = nullptr;
  int M = 0, K = 0, N = 0;
  if (which == 4) {
    src = e->w_int8 ? (const void*)e->lm_q : (const void*)e->lm_head;
    sc = e->lm_scale; M = dm.V; K = dm.d; N = e->tile_lm;
  } else {
    const LayerDev& L = e->layers[layer];
    const bool q = e->w_int8;
    switch (which) {
      case 0: src = q ? (const void*)L.q_qkv : L.w_qkv; sc = L.s_qkv; M = dm.qkv_out; K = dm.d; N = e->tile_qkv; break;
      case 1: src = q ? (const void*)L.q_o : L.w_o; sc = L.s_o; M = dm.d; K = hqd; N = e->tile_o; break;
      case 2: src = q ? (const void*)L.q_gu : L.w_gu; sc = L.s_gu; M = 2 * dm.F; K = dm.d; N = e->tile_gu; break;
      default: src = q ? (const void*)L.q_down : L.w_down; sc = L.s_down; M = dm.d; K = dm.F; N = e->tile_dn; break;
    }
  }
  const int eb = e->w_int8 ? 1 : 2;
  const size_t bytes = (size_t)M * K * eb;
  void* tmp = nullptr;
  CBD_CUDA(cudaMalloc(&tmp, bytes));
  untile_kernel<<<M, 256>>>(static_cast<uint8_t*>(tmp), static_cast<const uint8_t*>(src), K, N, eb);
  cudaError_t ce = cudaGetLastError();
  if (ce == cudaSuccess) ce = cudaMemcpy(dst, tmp, bytes, cudaMemcpyDeviceToHost);
  if (ce == cudaSuccess && scales && sc) ce = cudaMemcpy(scales, sc, (size_t)M * 4, cudaMemcpyDeviceToHost);
  cudaFree(tmp);
  if (ce != cudaSuccess) return cuda_fail(ce, "read weight");
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_counters(cbd_engine* e, float** counters) {
  if (!e || !counters) return fail(CBD_EINVAL, "NULL argument");
  *counters = e->counters;
  return CBD_OK;
}

extern "C" cbd_status cbd_slot_reset(cbd_engine* e, int32_t slot, void* stream) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  CBD_ON_DEVICE(e->device);
  if (slot < 0 || slot >= e->dm.max_slots) return fail(CBD_EINVAL, "slot %d out of range", slot);
  CBD_CUDA(cudaMemsetAsync(e->counters + (size_t)slot * e->dm.V, 0, (size_t)e->dm.V * 4,
                           static_cast<cudaStream_t>(stream)));
  CBD_CUDA(cudaMemsetAsync(e->last_tok + slot, 0, 4, static_cast<cudaStream_t>(stream)));
  return CBD_OK;
}

// ---------------------------------------------------------------- KV pool
extern "C" cbd_status cbd_kv_pool_create(cbd_engine* e, int32_t n_blocks, cbd_kv_pool** out) {
  clear_error();
  if (!e || !out) return fail(CBD_EINVAL, "NULL argument");
  CBD_ON_DEVICE(e->device);
  *out = nullptr;
  if (n_blocks < 1) return fail(CBD_EINVAL, "n_blocks must be >= 1");
  const size_t bytes = (size_t)e->dm.L * 2 * (size_t)n_blocks * e->dm.hkv * kBlock * e->dm.hd * (e->kv_fp8 ? 1 : 2);
  auto p = std::make_unique<cbd_kv_pool>();
  p->e = e;
  p->device = e->device;
  p->n_blocks = n_blocks;
  p->bytes = bytes;
  void* b = nullptr;
  CBD_CUDA(cudaMalloc(&b, bytes));
  if (e->kv_fp8) {
    // unwritten positions must not hold NaN codes: P = 0 times V there
    const cudaError_t ce = cudaMemset(b, 0, bytes);
    if (ce != cudaSuccess) {
      cudaFree(b);
      return cuda_fail(ce, "FP8 pool clear");
    }
  }
  p->base = static_cast<uint16_t*>(b);
  *out = p.release();
  return CBD_OK;
}

extern "C" cbd_status cbd_kv_pool_destroy(cbd_kv_pool* p) {
  if (!p) return CBD_OK;
  DeviceGuard dg(p->device);
  cudaDeviceSynchronize();
  cudaFree(p->base);
  delete p;
  return CBD_OK;
}

extern "C" cbd_status cbd_kv_pool_data(cbd_kv_pool* p, void** base, uint64_t* bytes, int32_t* n_blocks) {
  if (!p) return fail(CBD_EINVAL, "pool is NULL");
  if (base) *base = p->base;
  if (bytes) *bytes = p->bytes;
  if (n_blocks) *n_blocks = p->n_blocks;
  return CBD_OK;
}

// ---------------------------------------------------------------- batch
namespace cbd {

cbd_status build_batch_image(const cbd_engine* e, const cbd_kv_pool* pool, const cbd_row* rows, int32_t n_rows,
                             const int32_t* tables, int32_t table_slots, const int32_t* nbps,
                             const cbd_sampling* sp, const float* uniforms, BatchImage* img) {
  if (!e || !pool) return fail(CBD_EINVAL, "engine or pool is NULL");
  if (pool->e != e) return fail(CBD_EINVAL, "pool belongs to another engine");
  const Dims& dm = e->dm;
  if (n_rows < 1 || n_rows > dm.max_rows) return fail(CBD_EINVAL, "n_rows %d not in [1, %d]", n_rows, dm.max_rows);
  if (!rows || !tables || !nbps) return fail(CBD_EINVAL, "rows, block_tables or n_blocks_per_slot is NULL");
  if (table_slots < 1 || table_slots > dm.max_slots)
    return fail(CBD_EINVAL, "table_slots %d not in [1, %d]", table_slots, dm.max_slots);
  const int mbps = dm.max_blocks_per_seq;
  // per-slot summaries
  std::vector<int32_t> cnt(table_slots, 0), pmin(table_slots, INT32_MAX), pmax(table_slots, -1), smp(table_slots, 0);
  int32_t m = 0;
  for (int32_t r = 0; r < n_rows; ++r) {
    const cbd_row& w = rows[r];
    if (w.slot < 0 || w.slot >= table_slots) return fail(CBD_EINVAL, "row %d: slot %d out of range", r, w.slot);
    if (w.token == CBD_TOKEN_LAST) {
      if (w.is_prefill) return fail(CBD_EINVAL, "row %d: CBD_TOKEN_LAST on a prefill row", r);
    } else if (w.token < 0 || w.token >= dm.V) {
      return fail(CBD_EINVAL, "row %d: token %d out of range", r, w.token);
    }
    const int32_t nb = nbps[w.slot];
    if (nb < 1 || nb > mbps) return fail(CBD_EINVAL, "slot %d: n_blocks %d not in [1, %d]", w.slot, nb, mbps);
    if (w.pos < 0 || w.pos >= nb * kBlock)
      return fail(CBD_EINVAL, "row %d: pos %d outside the slot's %d blocks", r, w.pos, nb);
    cnt[w.slot]++;
    pmin[w.slot] = std::min(pmin[w.slot], w.pos);
    pmax[w.slot] = std::max(pmax[w.slot], w.pos);
    if (w.sample) {
      if (++smp[w.slot] > 1) return fail(CBD_EINVAL, "slot %d has more than one sampled row", w.slot);
      ++m;
    }
  }
  // positions of a slot: one contiguous run with no repeats
  {
    for (int32_t s = 0; s < table_slots; ++s)
      if (cnt[s] && pmax[s] - pmin[s] + 1 != cnt[s])
        return fail(CBD_EINVAL, "slot %d: positions not one contiguous run", s);
    std::vector<std::vector<uint8_t>> seen(table_slots);
    for (int32_t r = 0; r < n_rows; ++r) {
      const int32_t s = rows[r].slot;
      if (cnt[s] < 2) continue;
      auto& b = seen[s];
      if (b.empty()) b.assign(cnt[s], 0);
      const int32_t k = rows[r].pos - pmin[s];
      if (b[k]) return fail(CBD_EINVAL, "slot %d: position %d appears twice", s, rows[r].pos);
      b[k] = 1;
    }
  }
  // blocks: in range and owned by one slot only
  {
    std::vector<int32_t> owner(pool->n_blocks, -1);
    for (int32_t s = 0; s < table_slots; ++s) {
      if (!cnt[s]) continue;
      for (int32_t b = 0; b < nbps[s]; ++b) {
        const int32_t id = tables[(size_t)s * mbps + b];
        if (id < 0 || id >= pool->n_blocks)
          return fail(CBD_EINVAL, "slot %d block %d: physical id %d outside the pool", s, b, id);
        if (owner[id] >= 0 && owner[id] != s)
          return fail(CBD_EINVAL, "physical block %d shared by slots %d and %d", id, owner[id], s);
        if (owner[id] == s) return fail(CBD_EINVAL, "physical block %d used twice by slot %d", id, s);
        owner[id] = s;
      }
    }
  }
  if (m > 0 && !sp) return fail(CBD_EINVAL, "sampling is NULL but %d rows are sampled", m);
  if (m > dm.max_slots) return fail(CBD_EINVAL, "too many sampled rows");
  for (int32_t j = 0; j < m; ++j) {
    const cbd_sampling& s = sp[j];
    if (!std::isfinite(s.temperature) || s.temperature < 0.f) return fail(CBD_EINVAL, "sampling %d: temperature", j);
    if (!std::isfinite(s.top_p) || s.top_p < 0.f || s.top_p > 1.f) return fail(CBD_EINVAL, "sampling %d: top_p", j);
    if (s.top_k < 0 || s.top_k > dm.V) return fail(CBD_EINVAL, "sampling %d: top_k", j);
    if (!std::isfinite(s.presence_penalty) || !std::isfinite(s.frequency_penalty) || !std::isfinite(s.penalty_decay))
      return fail(CBD_EINVAL, "sampling %d: penalty not finite", j);
    if (s.reserved) return fail(CBD_EINVAL, "sampling %d: reserved field must be 0", j);
    if (uniforms && !(uniforms[j] >= 0.f && uniforms[j] < 1.f)) return fail(CBD_EINVAL, "uniform %d not in [0,1)", j);
  }
  // prefill runs: maximal runs of consecutive positions of one slot (in
  // any row order), at least kPfMinRun long, cut into blocks from the run's
  // first position for the prefill attention kernel -- so which rows form
  // runs, and the blocks, do not depend on the order of the rows
  std::vector<uint8_t> in_run(n_rows, 0);
  std::vector<PfBlock> pfb;
  std::vector<int32_t> pf_rows;
  {
    const int BQ = prefill_block_positions(dm.hq / dm.hkv);
    std::vector<int32_t> ord(n_rows);
    for (int32_t r = 0; r < n_rows; ++r) ord[r] = r;
    std::sort(ord.begin(), ord.end(), [&](int32_t x, int32_t y) {
      return rows[x].slot != rows[y].slot ? rows[x].slot < rows[y].slot : rows[x].pos < rows[y].pos;
    });
    for (int32_t a = 0; a < n_rows;) {
      int32_t b1 = a + 1;
      while (b1 < n_rows && rows[ord[b1]].slot == rows[ord[a]].slot &&
             rows[ord[b1]].pos == rows[ord[b1 - 1]].pos + 1)
        ++b1;
      if (b1 - a >= kPfMinRun) {
        const int32_t base = (int32_t)pf_rows.size();
        for (int32_t i = a; i < b1; ++i) {
          in_run[ord[i]] = 1;
          pf_rows.push_back(ord[i]);
        }
        for (int32_t k = 0; k < b1 - a; k += BQ)
          pfb.push_back(PfBlock{base + k, std::min<int32_t>(BQ, b1 - a - k), rows[ord[a + k]].pos, rows[ord[a]].slot});
      }
      a = b1;
    }
    // longest context first, so the last CTAs to start are the short ones
    std::stable_sort(pfb.begin(), pfb.end(),
                     [](const PfBlock& x, const PfBlock& y) { return x.pos0 + x.npos > y.pos0 + y.npos; });
  }
  // work list: fixed 128-position chunks of every row
  int64_t n_work = 0;
  for (int32_t r = 0; r < n_rows; ++r) n_work += rows[r].pos / kAttnChunk + 1;
  if (n_work > e->max_work)
    return fail(CBD_EUNSUPPORTED, "step needs %lld attention chunks, more than the %d the workspace holds",
                (long long)n_work, e->max_work);
  // layout
  BatchImage& I = *img;
  I.n_rows = n_rows; I.m = m; I.n_work = (int32_t)n_work; I.table_slots = table_slots;
  I.n_pfb = (int32_t)pfb.size();
  size_t off = 0;
  auto take = [&](size_t b) { size_t o = off; off = align_up(off + b, 16); return o; };
  I.off_rows = take(n_rows * sizeof(RowDev));
  I.off_sr = take(std::max(m, 1) * 4);
  I.off_ss = take(std::max(m, 1) * 4);
  I.off_samp = take(std::max(m, 1) * sizeof(SampDev));
  I.off_tables = take((size_t)table_slots * mbps * 4);
  I.off_work = take(n_work * sizeof(AttnWork));
  I.off_row_work = take((n_rows + 1) * 4);
  I.off_pfb = take(pfb.size() * sizeof(PfBlock));
  I.off_pf_rows = take(pf_rows.size() * 4);
  I.off_comb = take((size_t)n_rows * 4);
  I.bytes.assign(off, 0);
  uint8_t* B = I.bytes.data();
  RowDev* rd = reinterpret_cast<RowDev*>(B + I.off_rows);
  int32_t* sr = reinterpret_cast<int32_t*>(B + I.off_sr);
  int32_t* ss = reinterpret_cast<int32_t*>(B + I.off_ss);
  SampDev* sd = reinterpret_cast<SampDev*>(B + I.off_samp);
  AttnWork* wk = reinterpret_cast<AttnWork*>(B + I.off_work);
  int32_t* rw = reinterpret_cast<int32_t*>(B + I.off_row_work);
  int32_t j = 0, wi = 0;
  int32_t max_chunks = 0;
  for (int32_t r = 0; r < n_rows; ++r) {
    const cbd_row& w = rows[r];
    rd[r] = RowDev{w.slot, w.token, w.pos, (w.is_prefill ? 1 : 0) | (w.sample ? 2 : 0) | (in_run[r] ? 4 : 0)};
    if (w.sample) {
      const cbd_sampling& s = sp[j];
      sr[j] = r;
      ss[j] = w.slot;
      sd[j] = SampDev{s.temperature, s.top_p, s.presence_penalty, s.frequency_penalty, s.penalty_decay, s.top_k,
                      (uint32_t)(s.seed & 0xffffffffu), (uint32_t)(s.seed >> 32),
                      (uint32_t)(s.request_id & 0xffffffffu), (uint32_t)(s.request_id >> 32), s.token_index,
                      uniforms ? uniforms[j] : -1.0f};
      ++j;
    }
  }
  // work items: rows outside prefill runs first, then the runs' rows (which
  // the prefill kernel covers when it runs); a row's items are consecutive
  int32_t n_dec = 0;
  for (int pass = 0; pass < 2; ++pass) {
    for (int32_t r = 0; r < n_rows; ++r) {
      if (in_run[r] != pass) continue;
      const cbd_row& w = rows[r];
      rw[r] = wi;
      const int32_t nch = w.pos / kAttnChunk + 1;
      max_chunks = std::max(max_chunks, nch);
      for (int32_t c = 0; c < nch; ++c) {
        AttnWork a{};
        a.row = r;
        a.start = c * kAttnChunk;
        a.end = std::min(a.start + kAttnChunk, w.pos + 1);
        a.wn = (wi << 16) | nch;
        for (int32_t k = 0; k < kAttnChunk / kBlock; ++k) {
          const int32_t p0 = a.start + k * kBlock;
          a.blk[k] = p0 < a.end ? tables[(size_t)w.slot * mbps + p0 / kBlock] : -1;
        }
        wk[wi++] = a;
      }
    }
    if (pass == 0) n_dec = wi;
  }
  rw[n_rows] = wi;
  I.max_chunks = max_chunks;
  I.n_dec = n_dec;
  // within each part, largest chunks first (ties in chunk order): dynamic
  // scheduling then ends on the short last chunks of rows
  auto by_size = [](const AttnWork& x, const AttnWork& y) { return (x.end - x.start) > (y.end - y.start); };
  std::stable_sort(wk, wk + n_dec, by_size);
  std::stable_sort(wk + n_dec, wk + wi, by_size);
  if (!pfb.empty()) std::memcpy(B + I.off_pfb, pfb.data(), pfb.size() * sizeof(PfBlock));
  if (!pf_rows.empty()) std::memcpy(B + I.off_pf_rows, pf_rows.data(), pf_rows.size() * 4);
  {
    int32_t* cr = reinterpret_cast<int32_t*>(B + I.off_comb);
    int32_t k = 0;
    for (int pass = 0; pass < 2; ++pass) {
      for (int32_t r = 0; r < n_rows; ++r)
        if (in_run[r] == pass && rows[r].pos >= kAttnChunk) cr[k++] = r;
      if (pass == 0) I.n_comb_dec = k;
    }
    I.n_comb_all = k;
  }
  std::memcpy(B + I.off_tables, tables, (size_t)table_slots * mbps * 4);
  return CBD_OK;
}

void bind_batch(cbd_batch* b, const BatchImage& I, void* dev) {
  uint8_t* D = static_cast<uint8_t*>(dev);
  b->dev = dev;
  b->dev_bytes = I.bytes.size();
  b->n_rows = I.n_rows; b->m = I.m; b->n_work = I.n_work; b->table_slots = I.table_slots;
  b->max_chunks = I.max_chunks;
  b->rows = reinterpret_cast<RowDev*>(D + I.off_rows);
  b->sampled_rows = reinterpret_cast<int32_t*>(D + I.off_sr);
  b->sampled_slots = reinterpret_cast<int32_t*>(D + I.off_ss);
  b->samp = reinterpret_cast<SampDev*>(D + I.off_samp);
  b->tables = reinterpret_cast<int32_t*>(D + I.off_tables);
  b->work = reinterpret_cast<AttnWork*>(D + I.off_work);
  b->row_work = reinterpret_cast<int32_t*>(D + I.off_row_work);
  b->pfb = reinterpret_cast<PfBlock*>(D + I.off_pfb);
  b->pf_rows = reinterpret_cast<int32_t*>(D + I.off_pf_rows);
  b->comb_rows = reinterpret_cast<int32_t*>(D + I.off_comb);
  b->n_comb_dec = I.n_comb_dec;
  b->n_comb_all = I.n_comb_all;
  b->n_dec = I.n_dec;
  b->n_pfb = I.n_pfb;
}

static cudaEvent_t prof_event(cbd_engine* e) {
  if (!e->prof_free.empty()) {
    cudaEvent_t ev = e->prof_free.back();
    e->prof_free.pop_back();
    return ev;
  }
  cudaEvent_t ev{};
  cudaEventCreate(&ev);
  return ev;
}

// Launch `fn` bracketed by events when profiling is on.
template <class Fn>
static cudaError_t timed(cbd_engine* e, int cls, cudaStream_t s, Fn&& fn) {
  if (!e->prof) return fn();
  cudaEvent_t a = prof_event(e), b = prof_event(e);
  cudaEventRecord(a, s);
  cudaError_t ce = fn();
  cudaEventRecord(b, s);
  e->prof_recs.push_back({cls, a, b});
  return ce;
}

// The step: embed; per layer norm -> QKV(+RoPE, KV append) -> attention ->
// O(+residual) -> norm -> gate/up(+SwiGLU) -> down(+residual); final norm of
// the sampled rows -> LM head -> sampler.
static cbd_status run_batch(cbd_engine* e, cbd_kv_pool* p, cbd_batch* b, int32_t* out_tokens, float* out_logits,
                            cudaStream_t s) {
  const Dims& dm = e->dm;
  const int n = b->n_rows;
  const int hqd = dm.hq * dm.hd;
  int launches = 0;
  auto chk = [&](cudaError_t ce, const char* what) -> cbd_status {
    if (ce != cudaSuccess) return cuda_fail(ce, what);
    return CBD_OK;
  };
  if (out_logits && (reinterpret_cast<uintptr_t>(out_logits) & 15))
    return fail(CBD_EINVAL, "out_logits must be 16-byte aligned");
  if (b->m > 0 && !out_tokens) return fail(CBD_EINVAL, "out_tokens is NULL but rows are sampled");
  // Fused RMSNorm on the tensor-core path: the embedding and the residual
  // epilogues write split(x * g) and per-row partial sums of x^2, and the
  // QKV / gate-up GEMMs apply 1/rms in their epilogues (no norm launches).
  const int o_parts = gemm_tc_units(dm.d, hqd, e->tile_o, n, e->w_int8),
            dn_parts = gemm_tc_units(dm.d, dm.F, e->tile_dn, n, e->w_int8);
  const bool fused = e->fuse_norm && gemm_uses_tc(e, n) && !gemm_uses_rows(e, n) && o_parts <= kMaxSsqParts && dn_parts <= kMaxSsqParts;
  cbd_status st;
  if ((st = chk(timed(e, kcEmbed, s, [&] { return launch_embed(e, b, fused ? e->layers[0].attn_norm : nullptr, s); }),
                "embed")))
    return st;
  ++launches;
  EpiArgs qkv{};
  qkv.kind = kEpiQKV; qkv.out_f32 = e->q; qkv.ld = hqd;
  qkv.pool = p->base; qkv.kv_fp8 = e->kv_fp8 ? 1 : 0; qkv.n_blocks = p->n_blocks; qkv.hq = dm.hq; qkv.hkv = dm.hkv; qkv.hd = dm.hd;
  qkv.max_blocks_per_seq = dm.max_blocks_per_seq; qkv.max_pos = e->max_pos; qkv.rope_cs = e->rope_cs;
  qkv.rows = b->rows; qkv.tables = b->tables; qkv.err = e->err;
  EpiArgs res{};
  res.kind = kEpiResid; res.out_f32 = e->x; res.ld = dm.d; res.err = e->err;
  EpiArgs resn = res;
  resn.kind = kEpiResidNorm; resn.norm_hi = e->norm_hi; resn.norm_lo = e->norm_lo; resn.ssq_out = e->ssq;
  EpiArgs glu{};
  glu.kind = kEpiSwiGLU; glu.out_hi = e->ffn_hi; glu.out_lo = e->ffn_lo; glu.ld_act = dm.F; glu.err = e->err;
  if (fused) {
    qkv.ssq_in = e->ssq; qkv.d_norm = dm.d; qkv.eps = dm.eps;
    glu.ssq_in = e->ssq; glu.d_norm = dm.d; glu.eps = dm.eps; glu.n_parts_in = o_parts;
  }
  const size_t a0 = (size_t)4 * dm.L + 1;
  const CUtensorMap* tm = e->tmaps.data();
  // normalised-input activations: the rmsnorm kernel's act_hi / act_lo, or
  // the fused epilogues' norm_hi / norm_lo
  const uint16_t* in_hi = fused ? e->norm_hi : e->act_hi;
  const uint16_t* in_lo = fused ? e->norm_lo : e->act_lo;
  const CUtensorMap* tm_in_hi = fused ? &tm[a0 + 6] : &tm[a0 + 0];
  const CUtensorMap* tm_in_lo = fused ? &tm[a0 + 7] : &tm[a0 + 1];
  // The step's GEMMs in order; each kernel prefetches (into L2) the first
  // k-blocks of the GEMM after it, so HBM keeps streaming across launches.
  auto g_qkv_of = [&](int l) {
    return GemmOp{e->layers[l].w_qkv, dm.qkv_out, dm.d, in_hi, in_lo, dm.d,
                  {&tm[4 * l + 0], tm_in_hi, tm_in_lo, dm.qkv_out, dm.d, e->tile_qkv, e->layers[l].s_qkv,
                   e->layers[l].q_qkv}};
  };
  const GemmOp g_lm{e->lm_head, dm.V, dm.d, e->act_hi, e->act_lo, dm.d,
                    {&tm[4 * dm.L], &tm[a0 + 0], &tm[a0 + 1], dm.V, dm.d, e->tile_lm, e->lm_scale, e->lm_q}};
  const PfSpec pf_none{};
  // Decode steps (one activation tile of rows) on the fused tcgen05 path
  // run each layer's O, gate/up and down contractions and the next layer's
  // QKV as one persistent launch with the same sums (k_gemm_chain.cu).
  const bool chain = e->gemm_chain && fused && !e->w_int8 && n <= 64;
  bool qkv_done = false;              // this layer's QKV ran inside the previous layer's chain
  for (int l = 0; l < dm.L; ++l) {
    const LayerDev& L = e->layers[l];
    qkv.layer = l;
    qkv.n_parts_in = l == 0 ? 1 : dn_parts;
    const GemmOp g_qkv = g_qkv_of(l);
    const GemmOp g_o{L.w_o, dm.d, hqd, e->act_hi, e->act_lo, hqd,
                     {&tm[4 * l + 1], &tm[a0 + 2], &tm[a0 + 3], dm.d, hqd, e->tile_o, L.s_o, L.q_o}};
    const GemmOp g_gu{L.w_gu, 2 * dm.F, dm.d, in_hi, in_lo, dm.d,
                      {&tm[4 * l + 2], tm_in_hi, tm_in_lo, 2 * dm.F, dm.d, e->tile_gu, L.s_gu, L.q_gu}};
    const GemmOp g_dn{L.w_down, dm.d, dm.F, e->ffn_hi, e->ffn_lo, dm.F,
                      {&tm[4 * l + 3], &tm[a0 + 4], &tm[a0 + 5], dm.d, dm.F, e->tile_dn, L.s_down, L.q_down}};
    const PfSpec pf_o = next_prefetch(e, g_o, n), pf_gu = next_prefetch(e, g_gu, n),
                 pf_dn = next_prefetch(e, g_dn, n);
    const PfSpec pf_after_dn = l + 1 < dm.L ? next_prefetch(e, g_qkv_of(l + 1), n)
                                            : (b->m > 0 ? next_prefetch(e, g_lm, b->m) : pf_none);
    EpiArgs res_o = res, res_dn = res;
    if (fused) {
      res_o = resn;
      res_o.norm_g = L.ffn_norm;
      if (l + 1 < dm.L) {
        res_dn = resn;
        res_dn.norm_g = e->layers[l + 1].attn_norm;
      }
    }
    if (!fused) {
      if ((st = chk(timed(e, kcNorm, s, [&] { return launch_rmsnorm(e, e->x, L.attn_norm, n, nullptr, e->act_hi, e->act_lo, s); }),
                    "rmsnorm")))
        return st;
      ++launches;
    }
    if (!qkv_done) {
      if ((st = chk(timed(e, kcQKV, s, [&] { return launch_gemm(e, g_qkv, n, qkv, pf_none, s); }),
                    "qkv")))
        return st;
      ++launches;
    }
    if ((st = chk(timed(e, kcAttn, s, [&] { return launch_attention(e, p, b, l, pf_o, s); }), "attention"))) return st;
    launches += attention_launches(e, b);
    qkv_done = false;
    if (chain) {
      TcGemm cg[kChainMaxPhases] = {g_o.tc, g_gu.tc, g_dn.tc};
      EpiArgs ce[kChainMaxPhases] = {res_o, glu, res_dn};
      int np = 3;
      if (l + 1 < dm.L) {
        cg[3] = g_qkv_of(l + 1).tc;
        ce[3] = qkv;
        ce[3].layer = l + 1;
        ce[3].n_parts_in = dn_parts;
        np = 4;
      }
      // the next layer's QKV joins the chain only if its K split fits the
      // chain's clusters; otherwise it runs on its own at the next layer
      if (np == 4 && !gemm_chain_possible(cg, np, n)) np = 3;
      if (gemm_chain_possible(cg, np, n)) {
        uint32_t* sync = e->chain_sync + (size_t)l * kChainMaxPhases;
        if ((st = chk(timed(e, kcChain, s, [&] { return launch_gemm_chain(cg, ce, np, n, sync, e->l2_prefetch, s); }),
                      "gemm_chain")))
          return st;
        ++launches;
        qkv_done = np == 4;
        continue;
      }
    }
    if ((st = chk(timed(e, kcO, s, [&] { return launch_gemm(e, g_o, n, res_o, pf_gu, s); }),
                  "o_proj")))
      return st;
    if (!fused) {
      if ((st = chk(timed(e, kcNorm, s, [&] { return launch_rmsnorm(e, e->x, L.ffn_norm, n, nullptr, e->act_hi, e->act_lo, s); }),
                    "rmsnorm")))
        return st;
      ++launches;
    }
    if ((st = chk(timed(e, kcGU, s, [&] { return launch_gemm(e, g_gu, n, glu, pf_dn, s); }),
                  "gate_up")))
      return st;
    if ((st = chk(timed(e, kcDown, s, [&] { return launch_gemm(e, g_dn, n, res_dn, pf_after_dn, s); }),
                  "down")))
      return st;
    launches += 3;
  }
  if (b->m > 0) {
    float* lg = out_logits ? out_logits : e->logits;
    if (!out_tokens) return fail(CBD_EINVAL, "out_tokens is NULL but rows are sampled");
    if ((st = chk(timed(e, kcFinal, s, [&] { return launch_rmsnorm(e, e->x, e->final_norm, b->m, b->sampled_rows, e->act_hi, e->act_lo, s); }),
                  "final_norm")))
      return st;
    EpiArgs lo{};
    lo.kind = kEpiLogits; lo.out_f32 = lg; lo.ld = dm.V; lo.err = e->err;
    if ((st = chk(timed(e, kcLM, s, [&] { return launch_gemm(e, g_lm, b->m, lo, pf_none, s); }),
                  "lm_head")))
      return st;
    if ((st = chk(timed(e, kcSamp, s, [&] { return launch_sampler(e, lg, b->m, b->sampled_slots, b->samp, out_tokens, s); }),
                  "sampler")))
      return st;
    launches += 3;
  }
  b->launches = launches;
  return CBD_OK;
}

}  // namespace cbd

extern "C" cbd_status cbd_step(cbd_engine* e, cbd_kv_pool* pool, const cbd_row* rows, int32_t n_rows,
                               const int32_t* block_tables, int32_t table_slots, const int32_t* n_blocks_per_slot,
                               const cbd_sampling* sampling, const float* uniforms, int32_t* out_tokens,
                               float* out_logits, void* stream) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  CBD_ON_DEVICE(e->device);
  BatchImage img;
  cbd_status st = build_batch_image(e, pool, rows, n_rows, block_tables, table_slots, n_blocks_per_slot, sampling,
                                    uniforms, &img);
  if (st) return st;
  if (img.m > 0 && !out_tokens) return fail(CBD_EINVAL, "out_tokens is NULL but rows are sampled");
  if (out_logits && (reinterpret_cast<uintptr_t>(out_logits) & 15))
    return fail(CBD_EINVAL, "out_logits must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cbd_engine::Stage& sg = e->stage[e->stage_idx];
  e->stage_idx ^= 1;
  if (img.bytes.size() > sg.bytes) return fail(CBD_EUNSUPPORTED, "step image larger than the staging buffer");
  CBD_CUDA(cudaEventSynchronize(sg.done));  // the step that last used this buffer has finished
  std::memcpy(sg.host, img.bytes.data(), img.bytes.size());
  if (e->step_graph && !e->prof) {
    // the upload and the launches as one graph: its kernels' arguments
    // depend only on the image layout, this staging buffer, the pool, the
    // outputs and the engine settings, which together make the key
    const uint64_t key[cbd_engine::kStepGraphKey] = {
        (uint64_t)img.n_rows, (uint64_t)img.m, (uint64_t)img.n_work, (uint64_t)img.table_slots,
        (uint64_t)img.max_chunks, (uint64_t)img.bytes.size(), reinterpret_cast<uint64_t>(pool),
        reinterpret_cast<uint64_t>(out_tokens), reinterpret_cast<uint64_t>(out_logits), e->epoch,
        (uint64_t)img.n_dec, (uint64_t)img.n_pfb, (uint64_t)img.n_comb_dec, (uint64_t)img.n_comb_all};
    auto& cache = e->step_graphs[&sg - e->stage];
    cbd_engine::StepGraph* hit = nullptr;
    for (auto& g : cache)
      if (std::memcmp(g.key, key, sizeof(key)) == 0) hit = &g;
    if (!hit) {
      bind_batch(e->step_batch, img, sg.dev);
      if (!e->cap_stream) CBD_CUDA(cudaStreamCreateWithFlags(&e->cap_stream, cudaStreamNonBlocking));
      CBD_CUDA(cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeRelaxed));
      cudaError_t cc = cudaMemcpyAsync(sg.dev, sg.host, img.bytes.size(), cudaMemcpyHostToDevice, e->cap_stream);
      cbd_status cs = cc == cudaSuccess ? run_batch(e, pool, e->step_batch, out_tokens, out_logits, e->cap_stream)
                                        : cuda_fail(cc, "staging upload");
      cudaGraph_t g = nullptr;
      const cudaError_t ce = cudaStreamEndCapture(e->cap_stream, &g);
      if (cs) {
        if (g) cudaGraphDestroy(g);
        return cs;
      }
      if (ce != cudaSuccess) return cuda_fail(ce, "graph capture");
      cudaGraphExec_t exec = nullptr;
      const cudaError_t ci = cudaGraphInstantiate(&exec, g, 0);
      cudaGraphDestroy(g);
      if (ci != cudaSuccess) return cuda_fail(ci, "graph instantiation");
      if (cache.size() >= cbd_engine::kStepGraphCache) {     // drop the least recently used
        size_t lru = 0;
        for (size_t i = 1; i < cache.size(); ++i)
          if (cache[i].last_use < cache[lru].last_use) lru = i;
        cudaGraphExecDestroy(cache[lru].exec);
        cache.erase(cache.begin() + (ptrdiff_t)lru);
      }
      cbd_engine::StepGraph ng{};
      std::memcpy(ng.key, key, sizeof(key));
      ng.exec = exec;
      cache.push_back(ng);
      hit = &cache.back();
      ++e->step_graph_captures;
    }
    hit->last_use = ++e->step_graph_clock;
    CBD_CUDA(cudaGraphLaunch(hit->exec, s));
    CBD_CUDA(cudaEventRecord(sg.done, s));
    return CBD_OK;
  }
  CBD_CUDA(cudaMemcpyAsync(sg.dev, sg.host, img.bytes.size(), cudaMemcpyHostToDevice, s));
  bind_batch(e->step_batch, img, sg.dev);
  st = run_batch(e, pool, e->step_batch, out_tokens, out_logits, s);
  cudaError_t ce = cudaEventRecord(sg.done, s);
  if (st) return st;
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaEventRecord");
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_set_step_graph(cbd_engine* e, int32_t enable) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  CBD_ON_DEVICE(e->device);
  e->step_graph = enable != 0;
  if (!e->step_graph) {
    CBD_CUDA(cudaDeviceSynchronize());
    for (auto& cache : e->step_graphs) {
      for (auto& g : cache) cudaGraphExecDestroy(g.exec);
      cache.clear();
    }
  }
  return CBD_OK;
}

extern "C" cbd_status cbd_engine_step_graph_captures(cbd_engine* e, int32_t* n) {
  clear_error();
  if (!e || !n) return fail(CBD_EINVAL, "NULL argument");
  *n = e->step_graph_captures;
  return CBD_OK;
}

extern "C" cbd_status cbd_batch_create(cbd_engine* e, cbd_kv_pool* pool, const cbd_row* rows, int32_t n_rows,
                                       const int32_t* block_tables, int32_t table_slots,
                                       const int32_t* n_blocks_per_slot, const cbd_sampling* sampling,
                                       const float* uniforms, cbd_batch** out, void* stream) {
  clear_error();
  if (!out) return fail(CBD_EINVAL, "out is NULL");
  *out = nullptr;
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  CBD_ON_DEVICE(e->device);
  BatchImage img;
  cbd_status st = build_batch_image(e, pool, rows, n_rows, block_tables, table_slots, n_blocks_per_slot, sampling,
                                    uniforms, &img);
  if (st) return st;
  auto b = std::make_unique<cbd_batch>();
  b->device = e->device;
  void* dev = nullptr;
  CBD_CUDA(cudaMalloc(&dev, img.bytes.size()));
  cudaError_t ce = cudaMemcpyAsync(dev, img.bytes.data(), img.bytes.size(), cudaMemcpyHostToDevice,
                                   static_cast<cudaStream_t>(stream));
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) {
    cudaFree(dev);
    return cuda_fail(ce, "batch upload");
  }
  bind_batch(b.get(), img, dev);
  b->owns_dev = true;
  // launch count of one run
  b->launches = 1 + e->dm.L * (4 + attention_launches(e, b.get()) + (e->fuse_norm ? 0 : 2)) + (img.m > 0 ? 3 : 0);
  *out = b.release();
  return CBD_OK;
}

static void drop_graph(cbd_batch* b) {
  if (b->exec) cudaGraphExecDestroy(b->exec);
  b->exec = nullptr;
}

extern "C" cbd_status cbd_batch_run(cbd_engine* e, cbd_kv_pool* pool, cbd_batch* b, int32_t* out_tokens,
                                    float* out_logits, void* stream) {
  clear_error();
  if (!e || !pool || !b) return fail(CBD_EINVAL, "NULL argument");
  if (pool->e != e) return fail(CBD_EINVAL, "pool belongs to another engine");
  CBD_ON_DEVICE(e->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!b->graph_on || e->prof) return run_batch(e, pool, b, out_tokens, out_logits, s);
  if (!b->exec || b->g_epoch != e->epoch || b->g_pool != pool || b->g_tok != out_tokens || b->g_lg != out_logits) {
    // capture the launch sequence on a private stream (nothing executes),
    // then instantiate it; the graph is replayed into the caller's stream
    drop_graph(b);
    if (!e->cap_stream) CBD_CUDA(cudaStreamCreateWithFlags(&e->cap_stream, cudaStreamNonBlocking));
    CBD_CUDA(cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeRelaxed));
    const cbd_status st = run_batch(e, pool, b, out_tokens, out_logits, e->cap_stream);
    cudaGraph_t g = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(e->cap_stream, &g);
    if (st) {
      if (g) cudaGraphDestroy(g);
      return st;
    }
    if (ce != cudaSuccess) return cuda_fail(ce, "graph capture");
    const cudaError_t ci = cudaGraphInstantiate(&b->exec, g, 0);
    cudaGraphDestroy(g);
    if (ci != cudaSuccess) {
      b->exec = nullptr;
      return cuda_fail(ci, "graph instantiation");
    }
    b->g_epoch = e->epoch;
    b->g_pool = pool;
    b->g_tok = out_tokens;
    b->g_lg = out_logits;
    ++b->captures;
  }
  CBD_CUDA(cudaGraphLaunch(b->exec, s));
  return CBD_OK;
}

extern "C" cbd_status cbd_batch_set_graph(cbd_batch* b, int32_t enable) {
  clear_error();
  if (!b) return fail(CBD_EINVAL, "batch is NULL");
  b->graph_on = enable != 0;
  if (!b->graph_on) drop_graph(b);
  return CBD_OK;
}

extern "C" cbd_status cbd_batch_captures(cbd_batch* b, int32_t* n) {
  clear_error();
  if (!b || !n) return fail(CBD_EINVAL, "NULL argument");
  *n = b->captures;
  return CBD_OK;
}

extern "C" cbd_status cbd_batch_destroy(cbd_batch* b) {
  if (!b) return CBD_OK;
  DeviceGuard dg(b->device);
  if (b->owns_dev && b->dev) {
    cudaDeviceSynchronize();
    cudaFree(b->dev);
  }
  drop_graph(b);
  delete b;
  return CBD_OK;
}

extern "C" cbd_status cbd_batch_launches(cbd_batch* b, int32_t* n) {
  if (!b || !n) return fail(CBD_EINVAL, "NULL argument");
  *n = b->launches;
  return CBD_OK;
}

extern "C" cbd_status cbd_sample(cbd_engine* e, const float* logits, int32_t m, const int32_t* slots,
                                 const cbd_sampling* sampling, const float* uniforms, int32_t* out_tokens,
                                 void* stream) {
  clear_error();
  if (!e) return fail(CBD_EINVAL, "engine is NULL");
  CBD_ON_DEVICE(e->device);
  if (m < 1 || m > e->dm.max_slots) return fail(CBD_EINVAL, "m %d not in [1, %d]", m, e->dm.max_slots);
  if (!logits || !slots || !sampling || !out_tokens) return fail(CBD_EINVAL, "NULL argument");
  std::vector<uint8_t> seen(e->dm.max_slots, 0);
  std::vector<SampDev> sd(m);
  for (int32_t j = 0; j < m; ++j) {
    if (slots[j] < 0 || slots[j] >= e->dm.max_slots) return fail(CBD_EINVAL, "slot %d out of range", slots[j]);
    if (seen[slots[j]]++) return fail(CBD_EINVAL, "slot %d appears twice", slots[j]);
    const cbd_sampling& s = sampling[j];
    if (!std::isfinite(s.temperature) || s.temperature < 0.f || !std::isfinite(s.top_p) || s.top_p < 0.f ||
        s.top_p > 1.f || s.top_k < 0 || s.top_k > e->dm.V || s.reserved)
      return fail(CBD_EINVAL, "sampling %d invalid", j);
    if (uniforms && !(uniforms[j] >= 0.f && uniforms[j] < 1.f)) return fail(CBD_EINVAL, "uniform %d not in [0,1)", j);
    sd[j] = SampDev{s.temperature, s.top_p, s.presence_penalty, s.frequency_penalty, s.penalty_decay, s.top_k,
                    (uint32_t)(s.seed & 0xffffffffu), (uint32_t)(s.seed >> 32), (uint32_t)(s.request_id & 0xffffffffu),
                    (uint32_t)(s.request_id >> 32), s.token_index, uniforms ? uniforms[j] : -1.0f};
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cbd_engine::Stage& sg = e->stage[e->stage_idx];
  e->stage_idx ^= 1;
  CBD_CUDA(cudaEventSynchronize(sg.done));
  uint8_t* H = static_cast<uint8_t*>(sg.host);
  const size_t o_samp = align_up((size_t)m * 4, 16);
  std::memcpy(H, slots, (size_t)m * 4);
  std::memcpy(H + o_samp, sd.data(), (size_t)m * sizeof(SampDev));
  CBD_CUDA(cudaMemcpyAsync(sg.dev, sg.host, o_samp + (size_t)m * sizeof(SampDev), cudaMemcpyHostToDevice, s));
  uint8_t* D = static_cast<uint8_t*>(sg.dev);
  cudaError_t ce = launch_sampler(e, logits, m, reinterpret_cast<int32_t*>(D),
                                  reinterpret_cast<SampDev*>(D + o_samp), out_tokens, s);
  cudaError_t ce2 = cudaEventRecord(sg.done, s);
  if (ce != cudaSuccess) return cuda_fail(ce, "sampler");
  if (ce2 != cudaSuccess) return cuda_fail(ce2, "cudaEventRecord");
  return CBD_OK;
}
