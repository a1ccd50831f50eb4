// cbd_sample_static: the step's sampler for callers that cannot allocate
// device memory.
//
// Some embedders cannot call cudaMalloc: a host framework whose caching
// allocator has already reserved the device's memory budget (a raw
// cudaMalloc there either fails or fragments the pool the framework
// manages), or a latency-critical serving loop that forbids allocation after
// warm-up because an allocation can synchronise the device and stall every
// other stream.  Those callers still own their inputs and outputs; what the
// sampler needs beyond them -- a scratch row of temperature-scaled logits
// per sampled row, plus the rows' slots and parameters on the device -- lives
// here in one file-scope device array of fixed size, so this entry point
// allocates nothing.
//
// The array is part of the library image: every GPU that loads libcbd holds
// it until the process exits.  It is shared by every call on a device and
// keeps the last call's contents; everything a call reads from it is written
// earlier by the same call, except the error word, which starts at zero when
// the library loads, is set by the first row that finds no token, and is
// cleared only by cbd_sample_static_check.  Calls whose work overlaps on the
// GPU (different streams, no ordering between them) race on the array.
//
// The rows' parameters reach the device as the arguments of a small kernel
// that writes them into the array, so a call copies nothing from host
// memory.
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace cbd {

// The sampler launch of k_sampler.cu (same kernel as cbd_sample).
cudaError_t sampler_launch(const float* logits, int m, int V, float* counters, const int32_t* slots,
                           const SampDev* samp, float* scratch, const uint32_t* forbid, int32_t* out_tokens,
                           int32_t* err, cudaStream_t s);

namespace {

constexpr int kStaticRows = CBD_SAMPLE_STATIC_MAX_ROWS;
constexpr int kStaticVocab = CBD_SAMPLE_STATIC_MAX_VOCAB;
constexpr size_t kZBytes = (size_t)kStaticRows * kStaticVocab * sizeof(float);
constexpr size_t kSampOff = kZBytes;
constexpr size_t kSlotOff = kSampOff + ((kStaticRows * sizeof(SampDev) + 255) / 256) * 256;
constexpr size_t kErrOff = kSlotOff + ((kStaticRows * sizeof(int32_t) + 255) / 256) * 256;
constexpr size_t kAreaBytes = kErrOff + 256;

// [rows][vocab] fp32 scratch, then [rows] SampDev, then [rows] int32 slots,
// then the int32 error word.
static __device__ __align__(256) unsigned char g_sample_area[kAreaBytes];

// The rows' parameters, passed by value to the kernel that stores them.
struct StaticParams {
  SampDev sd[kStaticRows];
  int32_t slots[kStaticRows];
  int32_t m;
};

__global__ void store_params_kernel(const StaticParams p) {
  SampDev* sd = reinterpret_cast<SampDev*>(g_sample_area + kSampOff);
  int32_t* sl = reinterpret_cast<int32_t*>(g_sample_area + kSlotOff);
  for (int j = threadIdx.x; j < p.m; j += blockDim.x) {
    sd[j] = p.sd[j];
    sl[j] = p.slots[j];
  }
}

std::mutex g_mu;
unsigned char* g_area_ptr[kMaxDevices] = {};

// Device address of g_sample_area on the current device (looked up once per
// device; host code cannot use the symbol's name as a device address).
cbd_status area_on_current_device(unsigned char** out) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(CBD_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(ce));
  if (dev < 0 || dev >= kMaxDevices) return fail(CBD_EUNSUPPORTED, "device ordinal %d too large", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_area_ptr[dev]) {
    void* p = nullptr;
    ce = cudaGetSymbolAddress(&p, g_sample_area);
    if (ce != cudaSuccess || !p)
      return fail(CBD_ECUDA, "cudaGetSymbolAddress(sampler scratch): %s", cudaGetErrorString(ce));
    g_area_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_area_ptr[dev];
  return CBD_OK;
}

}  // namespace
}  // namespace cbd

using namespace cbd;

extern "C" cbd_status cbd_sample_static(const float* logits, int32_t m, int32_t vocab, float* counters,
                                        int32_t counter_rows, const int32_t* slots, const cbd_sampling* sampling,
                                        const float* uniforms, int32_t* out_tokens, void* stream) {
  clear_error();
  if (m < 1 || m > kStaticRows)
    return fail(CBD_EINVAL, "cbd_sample_static: m = %d rows, the static scratch holds 1..%d", m, kStaticRows);
  if (vocab < 1 || vocab > kStaticVocab)
    return fail(CBD_EINVAL, "cbd_sample_static: vocab = %d, the static scratch holds 1..%d", vocab, kStaticVocab);
  if (!logits || !counters || !slots || !sampling || !out_tokens)
    return fail(CBD_EINVAL, "cbd_sample_static: NULL argument");
  if (counter_rows < 1) return fail(CBD_EINVAL, "cbd_sample_static: counter_rows must be >= 1");
  StaticParams prm{};
  prm.m = m;
  for (int32_t j = 0; j < m; ++j) {
    if (slots[j] < 0 || slots[j] >= counter_rows)
      return fail(CBD_EINVAL, "cbd_sample_static: slot %d outside the %d counter rows", slots[j], counter_rows);
    for (int32_t i = 0; i < j; ++i)
      if (slots[i] == slots[j]) return fail(CBD_EINVAL, "cbd_sample_static: slot %d appears twice", slots[j]);
    const cbd_sampling& s = sampling[j];
    if (!std::isfinite(s.temperature) || s.temperature < 0.f || !std::isfinite(s.top_p) || s.top_p < 0.f ||
        s.top_p > 1.f || s.top_k < 0 || s.top_k > vocab || s.reserved || !std::isfinite(s.presence_penalty) ||
        !std::isfinite(s.frequency_penalty) || !std::isfinite(s.penalty_decay))
      return fail(CBD_EINVAL, "cbd_sample_static: sampling %d invalid", j);
    if (uniforms && !(uniforms[j] >= 0.f && uniforms[j] < 1.f))
      return fail(CBD_EINVAL, "cbd_sample_static: uniform %d not in [0,1)", j);
    prm.sd[j] = SampDev{s.temperature, s.top_p, s.presence_penalty, s.frequency_penalty, s.penalty_decay, s.top_k,
                        (uint32_t)(s.seed & 0xffffffffu), (uint32_t)(s.seed >> 32),
                        (uint32_t)(s.request_id & 0xffffffffu), (uint32_t)(s.request_id >> 32), s.token_index,
                        uniforms ? uniforms[j] : -1.0f};
    prm.slots[j] = slots[j];
  }
  unsigned char* area = nullptr;
  cbd_status st = area_on_current_device(&area);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  store_params_kernel<<<1, 32, 0, s>>>(prm);
  cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) return fail(CBD_ECUDA, "cbd_sample_static: parameter store: %s", cudaGetErrorString(ce));
  ce = sampler_launch(logits, m, vocab, counters, reinterpret_cast<const int32_t*>(area + kSlotOff),
                      reinterpret_cast<const SampDev*>(area + kSampOff), reinterpret_cast<float*>(area), nullptr,
                      out_tokens, reinterpret_cast<int32_t*>(area + kErrOff), s);
  if (ce != cudaSuccess) return fail(CBD_ECUDA, "cbd_sample_static: launch: %s", cudaGetErrorString(ce));
  return CBD_OK;
}

extern "C" cbd_status cbd_sample_static_check(void* stream) {
  clear_error();
  unsigned char* area = nullptr;
  cbd_status st = area_on_current_device(&area);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t ce = cudaMemcpyAsync(&v, area + kErrOff, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
  if (ce != cudaSuccess) return fail(CBD_ECUDA, "cbd_sample_static_check: %s", cudaGetErrorString(ce));
  if (v) {
    ce = cudaMemsetAsync(area + kErrOff, 0, sizeof(v), s);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
    if (ce != cudaSuccess) return fail(CBD_ECUDA, "cbd_sample_static_check: clear: %s", cudaGetErrorString(ce));
    return fail(CBD_EDEVICE, "cbd_sample_static: device error code %d%s", v,
                v == kDevSampler ? " (a row had no token to draw: every logit -inf or NaN)" : "");
  }
  return CBD_OK;
}
