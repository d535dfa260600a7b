// Merge of split-KV partials: lse = ln sum_s e^(lse_s), out = sum_s e^(lse_s - lse) o_s.
//
// The split rule comes from the page "GPT-OSS on day 0", section "Kernels for
// GPT-OSS / Sink Attention" (the sink-seeded max belongs to the first block
// only); this is the log-sum-exp combine that undoes the split.  One warp per
// (sequence, head): lanes read the split lse values, a shuffle max, each lane
// turns one split's lse into its weight, and every lane accumulates two of the
// 64 output dims over the splits with coalesced float2 loads (256 contiguous
// bytes per split per warp), the weights broadcast by shuffle.  Up to 32 splits,
// every split's lse and output is requested before the max is reduced (one L2
// round trip per row; one sequence of 131072 tokens in 32 splits, graph step
// 44.84 -> 44.57 us against loading the outputs after the max).
#include "internal.h"
#include "ptx.cuh"

namespace sa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kPosInf = __builtin_huge_valf();
constexpr int kMergeWarps = 4;

__device__ __forceinline__ float split_weight(float lse_s, float M) {
  // e^(lse_s - M); the max term gets exactly 1, -inf terms exactly 0
  if (lse_s == M) return 1.0f;
  if (lse_s == kNegInf || M == kPosInf) return 0.0f;
  return ex2((lse_s - M) * kLog2e);
}

// Up to N splits: every split's weight and partial output is requested at once, so the
// row costs one round trip to L2 for the lse values and one for the outputs; the sum runs
// over the splits in order, like the general loop.
template <int N>
__device__ __forceinline__ void load_partials(const float* o_p, int heads, int S, float2 (&v)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i)
    v[i] = i < S ? *reinterpret_cast<const float2*>(o_p + static_cast<size_t>(i) * heads * kHeadDim)
                 : make_float2(0.0f, 0.0f);
}

template <int N>
__device__ __forceinline__ void merge_loaded(const float2 (&v)[N], float lse_mine, int S, float M, int lane,
                                             float& z, float2& acc) {
  const float w_mine = lane < S ? split_weight(lse_mine, M) : 0.0f;
  z = w_mine;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float w = __shfl_sync(0xffffffffu, w_mine, i);
    acc.x = fmaf(w, v[i].x, acc.x);
    acc.y = fmaf(w, v[i].y, acc.y);
  }
}

__global__ void __launch_bounds__(kMergeWarps * 32) sink_merge_kernel(const MergeArgs a) {
  // the next decode grid may start its set-up now (it waits for this grid
  // before reading anything)
  pdl_launch_dependents();
  // launched with programmatic stream serialisation: the partials come from the
  // preceding decode grid, so wait for it before reading them
  pdl_wait_primary();
  const int row = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.batch * a.heads) return;
  const int b = row / a.heads, h = row % a.heads;
  const int S = a.num_splits;
  const float* lse_p = a.partial_lse + static_cast<size_t>(b) * S * a.heads + h;

  const float* o_p = a.partial_o + (static_cast<size_t>(b) * S * a.heads + h) * kHeadDim + 2 * lane;
  float z = 0.0f;
  float2 acc = make_float2(0.0f, 0.0f);
  float M = kNegInf;
  // Up to 32 splits every split's partial output and lse is requested before the max is
  // reduced, so the row costs one round trip to L2.  Lane i turns split i's lse into its
  // weight and hands it to the warp by shuffle.  A split with weight 0 (lse -inf, or below a
  // +inf one) holds o = 0 (decode writes empty splits as zeros), so it adds nothing.
  if (S <= 32) {
    const float lse_mine = lane < S ? lse_p[static_cast<size_t>(lane) * a.heads] : kNegInf;
    if (S <= 8) {
      float2 v[8];
      load_partials<8>(o_p, a.heads, S, v);
      M = lse_mine;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      if (M != kNegInf) merge_loaded<8>(v, lse_mine, S, M, lane, z, acc);
    } else if (S <= 16) {
      float2 v[16];
      load_partials<16>(o_p, a.heads, S, v);
      M = lse_mine;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      if (M != kNegInf) merge_loaded<16>(v, lse_mine, S, M, lane, z, acc);
    } else {
      float2 v[32];
      load_partials<32>(o_p, a.heads, S, v);
      M = lse_mine;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      if (M != kNegInf) merge_loaded<32>(v, lse_mine, S, M, lane, z, acc);
    }
  } else {
    for (int s = lane; s < S; s += 32) M = fmaxf(M, lse_p[static_cast<size_t>(s) * a.heads]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (M != kNegInf) {
      for (int s0 = 0; s0 < S; s0 += 32) {
        const int n = min(32, S - s0);
        const float w_mine = lane < n ? split_weight(lse_p[static_cast<size_t>(s0 + lane) * a.heads], M) : 0.0f;
        z += w_mine;
#pragma unroll 8
        for (int i = 0; i < n; ++i) {
          const float w = __shfl_sync(0xffffffffu, w_mine, i);
          const float2 v =
              *reinterpret_cast<const float2*>(o_p + static_cast<size_t>(s0 + i) * a.heads * kHeadDim);
          acc.x = fmaf(w, v.x, acc.x);
          acc.y = fmaf(w, v.y, acc.y);
        }
      }
    }
  }
  // every lane's share of the denominator (all zero when every split is empty)
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  const float inv = z > 0.0f ? 1.0f / z : 0.0f;
  uint16_t* out = static_cast<uint16_t*>(a.out) + static_cast<size_t>(row) * kHeadDim + 2 * lane;
  *reinterpret_cast<uint32_t*>(out) = pack_bf16x2(acc.x * inv, acc.y * inv);
  if (a.lse && lane == 0) {
    float l = kNegInf;
    if (M == kPosInf) l = kPosInf;
    else if (z > 0.0f) l = M + lg2(z) * kLn2;
    a.lse[row] = l;
  }
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int rows = a.batch * a.heads;
  const int blocks = (rows + kMergeWarps - 1) / kMergeWarps;
  // Programmatic dependent launch: the grid may be scheduled while the decode
  // kernel before it drains, hiding the launch latency of this short kernel.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, sink_merge_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sa
