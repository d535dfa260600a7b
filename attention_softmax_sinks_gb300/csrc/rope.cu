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
// A CTA handles as many consecutive tokens as fit in a 64 KB tile (6 with 64
// query and 8 KV heads).  Their qkv rows are contiguous, so thread 0 copies
// them into shared memory with one bulk copy per token on an mbarrier; the
// CTA's whole input is in flight at once, without holding registers (streaming
// each thread's next token through registers kept about 60 KB per SM in flight
// and reached 83% of the copy bandwidth, against 92% this way).  While the copy
// runs, the CTA computes, for each token position p and frequency pair i, the
// angle p * theta'_i in fp64, reduces it to [-pi, pi] in fp64 and takes sincosf
// of the reduced fp32 angle; the (cos, sin) table, scaled by the temperature,
// and each token's page slot go to shared memory.  Thread u of a token owns one
// head row and one quarter j of its features: features [8j, 8j + 8) and their
// rotation partners [8j + 32, 8j + 40), read from the tile as two 16-byte
// vectors, so no lane exchange is needed; its bias values are loaded once.
//
// K/V-only mode (for the attention calls that rotate Q themselves): only the
// K and V rows of each token are copied and written, and the (cos, sin) table
// of every token goes to `table_out`, where those calls read it.
#include <cmath>
#include <cstdint>

#include "rope_args.h"
#include "rope_math.cuh"
#include "ptx.cuh"

namespace sa {
namespace {

constexpr int kMaxRopeTokens = 16;     // tokens per CTA at most (small head counts)
constexpr int kRopeTileBytes = 65536;  // input tile of a CTA: as many whole tokens as fit
constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr double kInvTwoPi = 0.15915494309189533576888376337251;
constexpr unsigned long long kDrainTimeoutNs = 2000000000ull;

// Untiled bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Tokens per CTA for `rows` = Hq + 2 Hkv head rows of 128 bytes each.
__host__ __device__ constexpr int rope_tokens_per_cta(int rows) {
  const int t = kRopeTileBytes / (rows * 128);
  return t < 1 ? 1 : (t > kMaxRopeTokens ? kMaxRopeTokens : t);
}

// blockDim.x = units * tpar: units = 4 (Hq + 2 Hkv) threads per token, tpar
// tokens processed side by side.  Dynamic shared memory: the CTA's input tile.
__global__ void __launch_bounds__(512) qkv_rope_kernel(const RopeArgs a, int tpar) {
  extern __shared__ __align__(128) uint8_t tile[];
  __shared__ float4 cs4[kMaxRopeTokens][kMaxRopePairs / 2];  // (cos, sin) of pairs 2i, 2i + 1
  __shared__ long long dst_row[kMaxRopeTokens];  // paged: page * Hkv * 16 + slot; contiguous: token
  __shared__ uint64_t full;
  const int all_rows = a.hq + 2 * a.hkv;
  const int first_row = a.kv_only ? a.hq : 0;  // head rows of a token this kernel handles
  const int rows = all_rows - first_row;
  const int units = rows * 4;
  const int tid = threadIdx.x;
  const int unit = tid % units;
  const int lane_tok = tid / units;  // < tpar
  const int row = first_row + (unit >> 2);  // head row within the token's qkv row
  const int j = unit & 3;
  const int per_cta = rope_tokens_per_cta(rows);
  const int t0 = blockIdx.x * per_cta;
  const int ntok = min(per_cta, a.total_tokens - t0);
  const uint32_t token_bytes = static_cast<uint32_t>(rows) * 128u;      // copied per token
  const uint32_t src_token_bytes = static_cast<uint32_t>(all_rows) * 128u;
  const uint32_t bar = smem_u32(&full);

  // The CTA's tokens are contiguous in qkv: one bulk copy per token into shared
  // memory, in flight while the angle table is computed.
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, token_bytes * ntok);
    const uint64_t policy = l2_policy_evict_first();  // read once
    const uint8_t* src = reinterpret_cast<const uint8_t*>(a.qkv) + static_cast<size_t>(t0) * src_token_bytes +
                         static_cast<size_t>(first_row) * 128u;
    for (int tok = 0; tok < ntok; ++tok)
      bulk_load(smem_u32(tile + tok * token_bytes), src + static_cast<size_t>(tok) * src_token_bytes,
                token_bytes, bar, policy);
  }
  float b1[8], b2[8];
  const long long col = static_cast<long long>(row) * kHeadDim + 8 * j;
  if (a.bias) {
    widen8(__ldg(reinterpret_cast<const uint4*>(a.bias + col)), b1);
    widen8(__ldg(reinterpret_cast<const uint4*>(a.bias + col + 32)), b2);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) b1[i] = b2[i] = 0.0f;
  }
  float* cs = reinterpret_cast<float*>(cs4);
  for (int e = tid; e < ntok * kMaxRopePairs; e += blockDim.x) {
    const int tok = e / kMaxRopePairs;
    const int pair = e % kMaxRopePairs;
    const int t = t0 + tok;
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
    float sn, cn;
    sincosf(static_cast<float>(red), &sn, &cn);
    cs[(tok * kMaxRopePairs + pair) * 2] = cn * a.mscale;
    cs[(tok * kMaxRopePairs + pair) * 2 + 1] = sn * a.mscale;
    if (a.table_out)
      reinterpret_cast<float2*>(a.table_out)[static_cast<long long>(t) * kMaxRopePairs + pair] =
          make_float2(cn * a.mscale, sn * a.mscale);
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
  __syncthreads();  // table and page slots ready

  const bool rotate = row < a.hq + a.hkv;
  const bool is_q = row < a.hq;
  const bool is_k = !is_q && rotate;
  const int kvh = is_q ? 0 : (is_k ? row - a.hq : row - a.hq - a.hkv);
  uint16_t* kv_dst = is_k ? a.k_out : a.v_out;
  if (!mbar_wait(bar, 0, a.timeout_ns)) {
    raise_status(a.status, kStatusTimeout);
    mbar_wait(bar, 0, kDrainTimeoutNs);  // the copy lands in this CTA's shared memory before it exits
    return;
  }
  for (int tok = lane_tok; tok < ntok; tok += tpar) {
    // Odd rows read their second half first: the two rows of a quarter-warp then
    // fall in different banks (bytes [0, 64) and [64, 128) of a row) at each load.
    const uint8_t* src = tile + tok * token_bytes + (row - first_row) * 128 + 16 * j;
    const int first = (row & 1) * 64;
    const uint4 u_first = *reinterpret_cast<const uint4*>(src + first);
    const uint4 u_second = *reinterpret_cast<const uint4*>(src + (64 - first));
    float y1[8], y2[8];
    widen8((row & 1) ? u_second : u_first, y1);
    widen8((row & 1) ? u_first : u_second, y2);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y1[i] += b1[i];
      y2[i] += b2[i];
    }
    if (rotate) {
#pragma unroll
      for (int i = 0; i < 4; ++i) rotate2(y1, y2, i, cs4[tok][4 * j + i]);  // pairs 8j + 2i, 8j + 2i + 1
    }
    const int t = t0 + tok;
    uint16_t* dst = nullptr;
    if (is_q) {
      dst = a.q_out + (static_cast<long long>(t) * a.hq + row) * kHeadDim + 8 * j;
    } else if (kv_dst != nullptr && dst_row[tok] >= 0) {
      const long long r = dst_row[tok];
      // paged: r = page * Hkv * 16 + slot, head kvh of that page starts kvh * 16 rows later
      const long long off = a.paged ? (r + static_cast<long long>(kvh) * kPageSize) * kHeadDim
                                    : (r * a.hkv + kvh) * kHeadDim;
      dst = kv_dst + off + 8 * j;
    }
    if (dst) {
      *reinterpret_cast<uint4*>(dst) = pack8(y1);
      *reinterpret_cast<uint4*>(dst + 32) = pack8(y2);
    }
  }
}

}  // namespace

cudaError_t launch_rope(const RopeArgs& a, cudaStream_t stream) {
  const int rows = a.kv_only ? 2 * a.hkv : a.hq + 2 * a.hkv;
  const int units = 4 * rows;
  const int per_cta = rope_tokens_per_cta(rows);
  int tpar = 256 / units;
  tpar = tpar < 1 ? 1 : (tpar > per_cta ? per_cta : tpar);
  const int blocks = (a.total_tokens + per_cta - 1) / per_cta;
  const size_t smem = static_cast<size_t>(per_cta) * rows * 128;
  cudaError_t e = cudaFuncSetAttribute(qkv_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  qkv_rope_kernel<<<blocks, units * tpar, smem, stream>>>(a, tpar);
  return cudaGetLastError();
}

}  // namespace sa
