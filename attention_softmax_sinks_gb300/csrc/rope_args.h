// Launcher interface of the QKV bias + rotary + K/V write kernel (rope.cu).
// Arguments arrive already validated by abi.cu.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"

namespace sa {

constexpr int kMaxRopePairs = kHeadDim / 2;

struct RopeArgs {
  const uint16_t* qkv;         // bf16 [T, (Hq + 2 Hkv) * 64]
  const uint16_t* bias;        // bf16 [(Hq + 2 Hkv) * 64] or nullptr
  const int32_t* cu_q;         // [B + 1]
  const int32_t* kv_lens;      // [B] or nullptr (kv_len == q_len)
  uint16_t* q_out;             // bf16 [T, Hq, 64]; unused when kv_only
  float* table_out;            // fp32 [T, 32, 2] (cos, sin) x temperature per token and pair, or nullptr
  uint16_t* k_out;             // contiguous: bf16 [T, Hkv, 64]; paged: [num_pages, Hkv, 16, 64]
  uint16_t* v_out;
  const int32_t* page_table;   // paged only: [B, max_pages]
  int paged;
  int kv_only;                 // rotate and write K and V only: Q is neither read nor written
  int batch, total_tokens, hq, hkv, max_pages, num_pages;
  float mscale;
  double inv_freq[kMaxRopePairs];
  unsigned* status;
  unsigned long long timeout_ns;  // bound on the kernel's wait for its input copy
};

cudaError_t launch_rope(const RopeArgs& a, cudaStream_t stream);

}  // namespace sa
