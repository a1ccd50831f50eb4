// The streaming attention kernel over an FP8 (E4M3) KV pool ("大模型推理为什么
// 需要 Continuous Batching", section 6: FP8 KV quantisation fits more
// sequences in the same memory).  Same tasks, chunks, online softmax and
// merge as the bf16 kernel in k_attn.cu; the K/V tiles are half the bytes,
// converted exactly to f16 in registers, and the products run as f16 MMAs
// with q and P split into f16 hi + lo (attn_stream.cuh).  Its own
// translation unit so the two sets of instantiations compile in parallel.
#include <algorithm>

#include "attn_stream.cuh"

namespace cbd {

template <int HD, int G>
static cudaError_t launch_fp8_t(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                                int n_items, const PfSpec& pf, cudaStream_t s) {
  const Dims& dm = e->dm;
  constexpr int smem = stream_smem<HD, true>();
  constexpr int NW = stream_warps<HD, true>();
  static DeviceOnce attr;
  {
    const cudaError_t ce = set_smem_once(attr, attn_stream_kernel<HD, G, true>, smem);
    if (ce != cudaSuccess) return ce;
  }
  const int n_tasks = n_items * dm.hkv;
  if (n_tasks <= 0) return cudaSuccess;
  const int grid = std::min(e->sm_count, (n_tasks + NW - 1) / NW);
  return launch_pdl(attn_stream_kernel<HD, G, true>, dim3(grid), dim3(NW * 32), smem, s,
                    (const uint16_t*)p->base, (const float*)e->q, (const RowDev*)b->rows, (const int32_t*)b->tables,
                    (const AttnWork*)b->work, (const int32_t*)b->row_work, n_tasks, layer, p->n_blocks, dm.hkv,
                    dm.max_blocks_per_seq, e->attn_o, e->attn_ml, e->act_hi, e->act_lo, e->attn_next + layer, pf,
                    e->err);
}

cudaError_t launch_attn_stream_fp8(const cbd_engine* e, const cbd_kv_pool* p, const cbd_batch* b, int layer,
                                   int n_items, const PfSpec& pf, cudaStream_t s) {
  const int G = e->dm.hq / e->dm.hkv;
  const int HD = e->dm.hd;
  if (HD == 64 && G == 1) return launch_fp8_t<64, 1>(e, p, b, layer, n_items, pf, s);
  if (HD == 64 && G == 2) return launch_fp8_t<64, 2>(e, p, b, layer, n_items, pf, s);
  if (HD == 64 && G == 4) return launch_fp8_t<64, 4>(e, p, b, layer, n_items, pf, s);
  if (HD == 64 && G == 8) return launch_fp8_t<64, 8>(e, p, b, layer, n_items, pf, s);
  if (HD == 128 && G == 1) return launch_fp8_t<128, 1>(e, p, b, layer, n_items, pf, s);
  if (HD == 128 && G == 2) return launch_fp8_t<128, 2>(e, p, b, layer, n_items, pf, s);
  if (HD == 128 && G == 4) return launch_fp8_t<128, 4>(e, p, b, layer, n_items, pf, s);
  if (HD == 128 && G == 8) return launch_fp8_t<128, 8>(e, p, b, layer, n_items, pf, s);
  return cudaErrorInvalidValue;
}

CBD_TRACE_BIND(attn8)

}  // namespace cbd
