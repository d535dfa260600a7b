// sink_attn_decode_noalloc: split-KV decode and merge in one call that
// allocates nothing.
//
// Who needs it: code that must not call cudaMalloc (or any allocator) when it
// enqueues work -- for example a plugin inside another runtime that only hands
// it input and output buffers, or a serving loop that forbids allocation on its
// hot path because an allocation can synchronise the device or fail under
// memory pressure.  Such callers cannot provide the fp32 split partials that
// sink_attn_decode + sink_attn_merge exchange, so this entry point keeps them in
// a fixed, file-scope device array instead.
//
// The array (kScratchFloats floats, 8 MiB) belongs to the library's device code:
// under CUDA's lazy module loading (the default) it is created on a device when
// the library's code is first used there (at the latest by this entry point's
// first call on that device, which also looks up its address), and the device
// then holds it until the process exits.  That first call loads code and must
// not happen while the stream is being captured into a graph, so make it once
// before any capture.  All calls on a device share the array and it keeps the
// previous call's contents; every
// element a call reads is written earlier in the same call (each split writes
// its whole partial, empty splits included), so nothing needs clearing.  Two
// calls that overlap on the GPU (different streams, no ordering) race on it.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/sink_attn.h"

namespace {

constexpr size_t kScratchFloats = size_t(1) << 21;  // 2,097,152 floats = 8 MiB
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
float* g_scratch_dev[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device.  The symbol's name
// in host code is only a host-side stand-in, never a device address, so the
// address is looked up once per device (with that device current) and cached.
sa_status scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return SA_ERR_CUDA;
    g_scratch_dev[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_dev[dev];
  return SA_OK;
}

}  // namespace

extern "C" sa_status sink_attn_decode_noalloc(const void* q, const void* paged_k,
                                              const void* paged_v, const int32_t* page_table,
                                              const int32_t* kv_lens, const float* sinks,
                                              int batch, int num_qo_heads, int num_kv_heads,
                                              int head_dim, int page_size, int max_pages,
                                              int num_pages, float sm_scale, int num_splits,
                                              void* out, float* lse, cudaStream_t stream) {
  if (num_splits <= 1)  // nothing to exchange between splits: the plain decode writes `out`
    return sink_attn_decode(q, paged_k, paged_v, page_table, kv_lens, sinks, batch, num_qo_heads,
                            num_kv_heads, head_dim, page_size, max_pages, num_pages, sm_scale,
                            num_splits, out, lse, stream);
  if (!out) return SA_ERR_NULL;
  if (batch < 0 || num_qo_heads <= 0 || head_dim <= 0 || num_splits > 256) return SA_ERR_SHAPE;
  const unsigned long long rows =
      static_cast<unsigned long long>(batch) * num_splits * num_qo_heads;
  const unsigned long long need = rows * static_cast<unsigned long long>(head_dim) + rows;
  if (need > kScratchFloats) return SA_ERR_CAPACITY;
  if (batch == 0) return SA_OK;
  float* scratch = nullptr;
  if (sa_status s = scratch_for_current_device(&scratch)) return s;
  float* partial_o = scratch;                             // [batch, splits, heads, head_dim]
  float* partial_lse = scratch + rows * head_dim;         // [batch, splits, heads]
  if (sa_status s = sink_attn_decode(q, paged_k, paged_v, page_table, kv_lens, sinks, batch,
                                     num_qo_heads, num_kv_heads, head_dim, page_size, max_pages,
                                     num_pages, sm_scale, num_splits, partial_o, partial_lse,
                                     stream))
    return s;
  return sink_attn_merge(partial_o, partial_lse, batch, num_splits, num_qo_heads, head_dim, out,
                         lse, stream);
}
