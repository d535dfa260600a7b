// QKV bias + YaRN rotary encoding + K/V write, the step that feeds sink
// attention (page "GPT-OSS on day 0", model overview list: QKV projections
// with biases; YaRN positional encoding).  The frequencies and the attention
// temperature (YaRN paper, section 3) arrive precomputed from the host.
//
// Rotating K when it is written costs one pass over the new tokens; rotating it
// inside the attention kernels would redo the work for every query block
// (prefill) or every decode step, so the rotation lives here and the attention
// kernels read K as stored.
//
// One CTA handles kRopeTokens tokens.  First 32 threads per token compute, for
// the token's position p and each of the 32 frequency pairs, the angle p * theta
// in fp64, reduce it to [-pi, pi] in fp64 and take sincosf of the reduced fp32
// angle; the (cos, sin) table, scaled by the temperature, goes to shared
// memory with the token's page slot.  Then the CTA streams the token rows
// (Hq + 2 Hkv head rows of 64 bf16) in 16-byte chunks: a head row is 8 chunks
// held by 8 consecutive lanes, and a lane pairs feature i with feature i + 32
// by exchanging its 8 biased values with lane ^ 4.
#include <cmath>
#include <cstdint>

#include "ops_internal.h"
#include "ptx.cuh"

namespace sa {
namespace {

constexpr int kRopeTokens = 4;
constexpr int kRopeThreads = 256;
constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr double kInvTwoPi = 0.15915494309189533576888376337251;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kRopeThreads) qkv_rope_kernel(const RopeArgs a) {
  __shared__ float2 cs[kRopeTokens][kMaxRopePairs];
  __shared__ long long dst_row[kRopeTokens];  // paged: (page * Hkv) * 16 + slot row; contiguous: token
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kRopeTokens;
  const int rows = a.hq + 2 * a.hkv;

  if (tid < kRopeTokens * kMaxRopePairs) {
    const int tok = tid / kMaxRopePairs;
    const int pair = tid % kMaxRopePairs;
    const int t = t0 + tok;
    if (t < a.total_tokens) {
      // sequence of token t: the last b with cu_q[b] <= t (empty sequences skipped)
      int lo = 0, hi = a.batch;  // invariant: cu_q[lo] <= t < cu_q[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(a.cu_q + mid) <= t) lo = mid; else hi = mid;
      }
      const int b = lo;
      const int q_start = __ldg(a.cu_q + b);
      const int q_len = __ldg(a.cu_q + b + 1) - q_start;
      const int kv = a.kv_lens ? __ldg(a.kv_lens + b) : q_len;
      const long long pos = static_cast<long long>(kv) - q_len + (t - q_start);
      const double ang = static_cast<double>(pos) * a.inv_freq[pair];
      const double red = ang - kTwoPi * rint(ang * kInvTwoPi);
      float s, c;
      sincosf(static_cast<float>(red), &s, &c);
      cs[tok][pair] = make_float2(c * a.mscale, s * a.mscale);
      if (pair == 0) {
        long long dst = t;
        if (a.paged) {
          dst = -1;
          const long long pidx = pos >> 4;
          if (pos < 0 || pidx >= a.max_pages || kv < q_len) {
            raise_status(a.status, kStatusBadLen);
          } else {
            const int page = __ldg(a.page_table + static_cast<long long>(b) * a.max_pages + pidx);
            if (page < 0 || page >= a.num_pages) raise_status(a.status, kStatusBadPage);
            else dst = static_cast<long long>(page) * a.hkv * kPageSize + (pos & 15);
          }
        }
        dst_row[tok] = dst;
      }
    }
  }
  __syncthreads();

  const int chunks = kRopeTokens * rows * 8;
  for (int base = 0; base < chunks; base += kRopeThreads) {
    const int c = base + tid;
    const int tok = c / (rows * 8);
    const int t = t0 + tok;
    const bool live = c < chunks && t < a.total_tokens;
    const int row = (c >> 3) % rows;
    const int part = c & 7;
    float y[8];
    if (live) {
      const long long off = (static_cast<long long>(t) * rows + row) * kHeadDim + part * 8;
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(a.qkv + off));
      uint4 bb = make_uint4(0, 0, 0, 0);
      if (a.bias) bb = __ldg(reinterpret_cast<const uint4*>(a.bias + row * kHeadDim + part * 8));
      const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
      const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        y[2 * i] = bf16_lo(xw[i]) + bf16_lo(bw[i]);
        y[2 * i + 1] = bf16_hi(xw[i]) + bf16_hi(bw[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) y[i] = 0.0f;
    }
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = __shfl_xor_sync(0xffffffffu, y[i], 4);
    if (!live) continue;
    const bool second = part >= 4;
    if (row < a.hq + a.hkv) {
      const int p0 = (part & 3) * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 r = cs[tok][p0 + i];
        // first half: a cos - b sin ; second half: b cos + a sin
        o[i] = second ? fmaf(y[i], r.x, o[i] * r.y) : fmaf(y[i], r.x, -o[i] * r.y);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = y[i];
    }
    const uint4 out = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                                 pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
    if (row < a.hq) {
      *reinterpret_cast<uint4*>(a.q_out + (static_cast<long long>(t) * a.hq + row) * kHeadDim +
                                part * 8) = out;
    } else {
      const bool is_k = row < a.hq + a.hkv;
      const int kvh = is_k ? row - a.hq : row - a.hq - a.hkv;
      uint16_t* dst = is_k ? a.k_out : a.v_out;
      const long long r = dst_row[tok];
      if (dst == nullptr || r < 0) continue;
      long long off;
      if (a.paged) {
        // r = page * Hkv * 16 + slot: head kvh of that page starts kvh * 16 rows later
        off = (r + static_cast<long long>(kvh) * kPageSize) * kHeadDim + part * 8;
      } else {
        off = (r * a.hkv + kvh) * kHeadDim + part * 8;
      }
      *reinterpret_cast<uint4*>(dst + off) = out;
    }
  }
}

}  // namespace

cudaError_t launch_rope(const RopeArgs& a, cudaStream_t stream) {
  const int blocks = (a.total_tokens + kRopeTokens - 1) / kRopeTokens;
  qkv_rope_kernel<<<blocks, kRopeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace sa
