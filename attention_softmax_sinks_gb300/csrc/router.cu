// Top-K-then-softmax MoE router (page "GPT-OSS on day 0", section "Kernels for
// GPT-OSS / MoE": the softmax runs over the K selected experts only, and the
// expert weights are computed in bf16).
//
// One warp per token row (a warp walks rows grid-stride and loads the next
// row's logits before ranking the current one).  The bf16 logits are turned into 32-bit keys that
// sort like the values (high 16 bits: the bf16 pattern mapped to an unsigned
// order, -0 folded onto +0; low 16 bits: 0xFFFF - expert, so that among equal
// logits the lower expert index is the larger key).  K rounds of a warp-wide
// unsigned max (one redux.sync each) pick the experts, largest first.  The
// softmax over the K selected logits runs in fp32 in every lane and lane r
// stores pick r: its expert index, its weight rounded to bf16, and one count
// into a shared-memory histogram that is added to the global counts at the end.
#include <cstdint>

#include "ops_internal.h"
#include "ptx.cuh"

namespace sa {
namespace {

constexpr int kRouterWarps = 32;
constexpr int kMaxTopK = 8;

__device__ __forceinline__ uint32_t order16(uint32_t bits) {
  if (bits == 0x8000u) bits = 0;  // -0 == +0
  return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
}

__device__ __forceinline__ float value_of(uint32_t key) {
  const uint32_t o = key >> 16;
  const uint32_t bits = (o & 0x8000u) ? (o & 0x7FFFu) : (~o & 0xFFFFu);
  return __uint_as_float(bits << 16);
}

template <int kPerLane>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_topk_kernel(const RouterArgs a) {
  __shared__ int hist[256];
  const int E = a.num_experts;
  const int K = a.top_k;
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const long long stride = static_cast<long long>(gridDim.x) * kRouterWarps;
  auto load_keys = [&](long long t, uint32_t (&key)[kPerLane]) {
    const uint16_t* row = a.logits + t * E;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      const int e = lane + 32 * j;
      key[j] = (t < a.num_tokens && e < E) ? ((order16(__ldg(row + e)) << 16) | (0xFFFFu - e)) : 0u;
    }
  };
  long long t = static_cast<long long>(blockIdx.x) * kRouterWarps + (threadIdx.x >> 5);
  uint32_t key[kPerLane];
  load_keys(t, key);
  for (; t < a.num_tokens; t += stride) {
    uint32_t next[kPerLane];
    load_keys(t + stride, next);  // the next row's logits are in flight while this row is ranked
    uint32_t pick[kMaxTopK];
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
      pick[r] = 0;
      if (r < K) {
        uint32_t best = key[0];
#pragma unroll
        for (int j = 1; j < kPerLane; ++j) best = key[j] > best ? key[j] : best;
        const uint32_t w = __reduce_max_sync(0xffffffffu, best);
        pick[r] = w;
#pragma unroll
        for (int j = 0; j < kPerLane; ++j) key[j] = key[j] == w ? 0u : key[j];
      }
    }
    const float m = value_of(pick[0]);
    float ex[kMaxTopK];
    float sum = 0.0f;
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
      ex[r] = 0.0f;
      if (r < K) {
        ex[r] = expf(value_of(pick[r]) - m);
        sum += ex[r];
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxTopK; ++r) {
      if (r < K && lane == r) {
        const int e = static_cast<int>(0xFFFFu - (pick[r] & 0xFFFFu));
        a.topk_idx[t * K + r] = e;
        a.topk_w[t * K + r] = static_cast<uint16_t>(pack_bf16x2(ex[r] / sum, 0.0f) & 0xFFFFu);
        if (a.counts) atomicAdd(&hist[e], 1);
      }
    }
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) key[j] = next[j];
  }
  if (a.counts) {
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x)
      if (hist[i]) atomicAdd(a.counts + i, hist[i]);
  }
}

template <int kPerLane>
cudaError_t launch_router_t(const RouterArgs& a, cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // one 1024-thread block per SM at most: few blocks keep the global count
  // atomics (one per expert per block) off the critical path
  const long long need = (a.num_tokens + kRouterWarps - 1) / kRouterWarps;
  const long long cap = static_cast<long long>(sms);
  const int blocks = static_cast<int>(need < cap ? need : cap);
  router_topk_kernel<kPerLane><<<blocks, kRouterWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream) {
  const int per_lane = (a.num_experts + 31) / 32;
  switch (per_lane) {
    case 1: return launch_router_t<1>(a, stream);
    case 2: return launch_router_t<2>(a, stream);
    case 3: return launch_router_t<3>(a, stream);
    case 4: return launch_router_t<4>(a, stream);
    case 5: return launch_router_t<5>(a, stream);
    case 6: return launch_router_t<6>(a, stream);
    case 7: return launch_router_t<7>(a, stream);
    default: return launch_router_t<8>(a, stream);
  }
}

}  // namespace sa
