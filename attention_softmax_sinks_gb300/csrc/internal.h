// Internal interface between the C-ABI layer (abi.cu) and the kernel
// translation units.  Arguments arrive here already validated.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sa {

constexpr int kHeadDim = 64;
constexpr int kPageSize = 16;

struct DecodeArgs {
  const void* q;
  const int32_t* page_table;
  const int32_t* kv_lens;
  const float* sinks;
  void* out;
  float* lse;
  int batch, hq, hkv, group, max_pages, num_pages, num_splits;
  int cluster;       // > 1 (num_splits == 1 only): KV range split across a CTA cluster, merged on chip
  float scale_log2;  // sm_scale * log2(e)
  unsigned* status;
  unsigned long long timeout_ns;
};

// Decode with q taken from the projection output [B, (Hq + 2 Hkv) * 64] (one new token per
// sequence): the kernel adds q_bias ([Hq * 64] bf16, or nullptr) and rotates by row b of
// table ([B, 32] (cos, sin) x temperature).  table == nullptr: q [B, Hq, 64] as given.
struct DecodeRopeArgs {
  const uint16_t* q_bias;
  const float2* table;
};

struct MergeArgs {
  const float* partial_o;
  const float* partial_lse;
  void* out;
  float* lse;
  int batch, num_splits, heads;
};

struct PrefillArgs {
  const void* q;           // [T, Hq, 64], or the projection output (see PrefillRopeArgs)
  const int32_t* cu_q;     // [B + 1]
  const int32_t* kv_lens;  // [B] (paged) or nullptr (contiguous: kv_len == q_len)
  const int32_t* page_table;
  const float* sinks;
  void* out;
  float* lse;
  int batch, total_q, max_q, hq, hkv, group, max_pages, num_pages, causal, paged;
  float scale_log2;
  unsigned* status;
  unsigned long long timeout_ns;
};

// Prefill with q taken from the projection output [T, (Hq + 2 Hkv) * 64]: the kernel adds
// q_bias ([Hq * 64] bf16, or nullptr) and rotates the rows by rope_table ([T, 32] (cos, sin)
// x temperature) on chip.  table == nullptr: q is used as given.
struct PrefillRopeArgs {
  const uint16_t* q_bias;
  const float2* table;
};

// Tensor maps (TMA descriptors) built on the host by abi.cu.
cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeArgs& a,
                          const DecodeRopeArgs& rope, cudaStream_t stream);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);
// qpmap: Q in boxes of (128 / group tokens, group heads), used for packed short sequences.
// omap: the output [T, Hq, 64] mapped like qmap (boxes of 128 tokens x 1 head); full query
// blocks are written through it with TMA stores.
cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& qpmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, const CUtensorMap& omap, const PrefillArgs& a,
                           const PrefillRopeArgs& rope, cudaStream_t stream);

}  // namespace sa
