// Launcher interface of the standalone Top-K-then-softmax router (router.cu).
// Arguments arrive already validated by abi.cu.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sa {

struct RouterArgs {
  const uint16_t* logits;  // bf16 [T, E]
  int32_t* topk_idx;       // [T, k]
  uint16_t* topk_w;        // bf16 [T, k]
  int32_t* counts;         // [E] (already zeroed) or nullptr
  long long num_tokens;
  int num_experts, top_k;
  int vec16;               // rows read as 16-byte vectors (E % 8 == 0, 16-byte aligned base)
};

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream);

}  // namespace sa
