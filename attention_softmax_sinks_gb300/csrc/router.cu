// Top-K-then-softmax MoE router (page "GPT-OSS on day 0", section "Kernels for
// GPT-OSS / MoE": the softmax runs over the K selected experts only, and the
// expert weights are computed in bf16).
//
// Four threads per token row.  The bf16 logits become 32-bit keys that sort like
// the values (high 16 bits: 0x8000 + magnitude for a non-negative logit, 0x8000 -
// magnitude for a negative one, so -0 and +0 share a code; low 16 bits: 0xFFFF -
// expert, so that among equal logits the lower expert index is the larger key).
// The codes of the two logits of a 32-bit word are made together.  Thread j of a
// row streams every fourth 8-expert chunk of it in 16-byte vectors and keeps its K
// largest keys in a sorted register list: each key bubbles through the list with K
// unsigned max/min pairs, no branches.  Two shuffle rounds (partners j ^ 1, then
// j ^ 2) merge the four lists (for K = 1, 2, 4, 8 by a bitonic merge: the
// elementwise max of one list and the other reversed, then a half-cleaner sort);
// every key is unique, so the merged list is the row's Top-K.  The softmax over the
// K selected logits runs in fp32; thread 0 of the row stores the K expert indices,
// the K weights rounded to bf16, and adds K counts to a shared-memory histogram
// that is added to the global counts at the end.  At most one block per SM walks
// the rows (an equal share each), so each global count receives at most one add
// per SM.
#include <cstdint>

#include "router_args.h"
#include "ptx.cuh"

namespace sa {
namespace {

constexpr int kRouterThreads = 1024;
constexpr int kSplit = 4;  // threads per token row
constexpr int kMaxChunks = 256 / 8 / kSplit;  // 16-byte chunks per thread at 256 experts

template <int K>
__device__ __forceinline__ void offer(uint32_t (&best)[K], uint32_t key) {
#pragma unroll
  for (int r = 0; r < K; ++r) {  // best[] stays sorted, largest first
    const uint32_t hi = max(best[r], key);
    key = min(best[r], key);
    best[r] = hi;
  }
}

// 16-bit order code of one bf16 pattern: 0x8000 + magnitude, or 0x8000 - magnitude
// for a negative value (so -0 and +0 meet at 0x8000).
__device__ __forceinline__ uint32_t order16(uint32_t bits) {
  return (bits & 0x8000u) ? 0x8000u - (bits & 0x7FFFu) : bits | 0x8000u;
}

// The order codes of both bf16 halves of w at once: in a negative half
// (b ^ 0xFFFF) + 1 = 0x8000 - magnitude, in a non-negative one b ^ 0x8000; the +1
// cannot carry out of a half, whose value is then at most 0x7FFF.
__device__ __forceinline__ uint32_t order16x2(uint32_t w) {
  const uint32_t s = (w >> 15) & 0x00010001u;  // 1 in each negative half
  return (w ^ (s * 0x7FFFu) ^ 0x80008000u) + s;
}

__device__ __forceinline__ float value_of(uint32_t key) {
  const uint32_t o = key >> 16;
  const uint32_t bits = (o >= 0x8000u) ? o - 0x8000u : 0x8000u | (0x8000u - o);
  return __uint_as_float(bits << 16);
}

// best[] (sorted, largest first) becomes the K largest of best[] and other[] (both
// sorted, all keys distinct).
template <int K>
__device__ __forceinline__ void merge_lists(uint32_t (&best)[K], const uint32_t (&other)[K]) {
  if constexpr ((K & (K - 1)) == 0) {
    // elementwise max against the reversed other list: a bitonic sequence holding
    // the K largest; then a half-cleaner network sorts it
#pragma unroll
    for (int r = 0; r < K; ++r) best[r] = max(best[r], other[K - 1 - r]);
#pragma unroll
    for (int stride = K / 2; stride > 0; stride >>= 1) {
#pragma unroll
      for (int r = 0; r < K; ++r) {
        if ((r & stride) == 0) {
          const uint32_t hi = max(best[r], best[r + stride]);
          best[r + stride] = min(best[r], best[r + stride]);
          best[r] = hi;
        }
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < K; ++r) offer<K>(best, other[r]);
  }
}

template <int K>
__global__ void __launch_bounds__(kRouterThreads) router_topk_kernel(const RouterArgs a) {
  __shared__ int hist[256];
  const int E = a.num_experts;
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int j = threadIdx.x % kSplit;
  constexpr int kRowsPerPass = kRouterThreads / kSplit;
  // an equal share of consecutive rows per block, walked 256 rows per pass
  const long long share = (a.num_tokens + gridDim.x - 1) / gridDim.x;
  const long long r0 = static_cast<long long>(blockIdx.x) * share;
  const long long r1 = min(r0 + share, a.num_tokens);
  const long long passes = (share + kRowsPerPass - 1) / kRowsPerPass;  // same for every thread
  for (long long pass = 0; pass < passes; ++pass) {
    const long long t = r0 + pass * kRowsPerPass + threadIdx.x / kSplit;
    const bool live = t < r1;  // the four threads of a row agree
    uint32_t best[K];
#pragma unroll
    for (int r = 0; r < K; ++r) best[r] = 0;  // below every real key
    if (live) {
      const uint16_t* row = a.logits + t * E;
      if (a.vec16) {
        // every load of the row is issued before any key is ranked
        const uint4* v = reinterpret_cast<const uint4*>(row);
        uint4 buf[kMaxChunks];
#pragma unroll
        for (int q = 0; q < kMaxChunks; ++q) {
          const int c = j + q * kSplit;
          buf[q] = c < E / 8 ? __ldg(v + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < kMaxChunks; ++q) {
          const int c = j + q * kSplit;
          if (c < E / 8) {
            const uint32_t ws[4] = {buf[q].x, buf[q].y, buf[q].z, buf[q].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t e = 8 * c + 2 * i;
              const uint32_t x = order16x2(ws[i]);
              offer<K>(best, __byte_perm(x, 0xFFFFu - e, 0x1054));      // code of expert e, low half
              offer<K>(best, __byte_perm(x, 0xFFFFu - e - 1, 0x3254));  // expert e + 1, high half
            }
          }
        }
      } else {
        for (int e = j; e < E; e += kSplit) offer<K>(best, (order16(__ldg(row + e)) << 16) | (0xFFFFu - e));
      }
    }
    // merge the four lists of the row (all 32 lanes take part in the shuffles)
#pragma unroll
    for (int o = 1; o < kSplit; o <<= 1) {
      uint32_t other[K];
#pragma unroll
      for (int r = 0; r < K; ++r) other[r] = __shfl_xor_sync(0xffffffffu, best[r], o);
      merge_lists<K>(best, other);
    }
    if (live && j == 0) {
      const float m = value_of(best[0]);
      float ex[K];
      float sum = 0.0f;
#pragma unroll
      for (int r = 0; r < K; ++r) {
        ex[r] = expf(value_of(best[r]) - m);
        sum += ex[r];
      }
      const float inv = 1.0f / sum;
#pragma unroll
      for (int r = 0; r < K; ++r) {
        const int e = static_cast<int>(0xFFFFu - (best[r] & 0xFFFFu));
        a.topk_idx[t * K + r] = e;
        a.topk_w[t * K + r] = static_cast<uint16_t>(pack_bf16x2(ex[r] * inv, 0.0f) & 0xFFFFu);
        if (a.counts) atomicAdd(&hist[e], 1);
      }
    }
  }
  if (a.counts) {
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x)
      if (hist[i]) atomicAdd(a.counts + i, hist[i]);
  }
}

template <int K>
cudaError_t launch_router_t(const RouterArgs& a, cudaStream_t stream) {
  // At most one block per SM: every block adds its histogram to the global
  // counts once, and same-address atomics serialise in L2, so the block count
  // (not the token count) sets the cost of the counts.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long need = (a.num_tokens + 63) / 64;  // at least 64 rows per block
  const int blocks = static_cast<int>(need < sms ? need : sms);
  router_topk_kernel<K><<<blocks, kRouterThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream) {
  switch (a.top_k) {
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
