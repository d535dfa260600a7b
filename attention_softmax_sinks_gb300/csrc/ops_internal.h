// Internal interface of the kernels around attention (router, QKV bias +
// rotary + K/V write) between abi.cu and their translation units.  Arguments
// arrive here already validated.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

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

constexpr int kMaxRopePairs = kHeadDim / 2;

struct RopeArgs {
  const uint16_t* qkv;         // bf16 [T, (Hq + 2 Hkv) * 64]
  const uint16_t* bias;        // bf16 [(Hq + 2 Hkv) * 64] or nullptr
  const int32_t* cu_q;         // [B + 1]
  const int32_t* kv_lens;      // [B] or nullptr (kv_len == q_len)
  uint16_t* q_out;             // bf16 [T, Hq, 64]
  uint16_t* k_out;             // contiguous: bf16 [T, Hkv, 64]; paged: [num_pages, Hkv, 16, 64]
  uint16_t* v_out;
  const int32_t* page_table;   // paged only: [B, max_pages]
  int paged;
  int batch, total_tokens, hq, hkv, max_pages, num_pages;
  float mscale;
  double inv_freq[kMaxRopePairs];
  unsigned* status;
};

struct LinearArgs {
  const uint16_t* bias;  // bf16 [N] or nullptr
  uint16_t* out;         // bf16 [M, N] (plain linear layer)
  int M, N, K;
  int block_n, tiles_m, tiles_n;
  unsigned* status;
  unsigned long long timeout_ns;
  // fused router (N = experts <= block_n, one column tile): per row, the Top-K of
  // the bf16-rounded logits, softmax weights and per-expert counts
  int32_t* topk_idx;     // [M, top_k]
  uint16_t* topk_w;      // bf16 [M, top_k]
  int32_t* counts;       // [N] (zeroed by the caller) or nullptr
  int top_k;
};

// Output tile width (128, 192, 240 or 256) for N output features.
int linear_tile_n(int n);
// amap: x [M, K] in boxes of 128 rows x 64; bmap: W [N, K] in boxes of block_n rows x 64.
cudaError_t launch_linear(const CUtensorMap& amap, const CUtensorMap& bmap, const LinearArgs& a,
                          int sms, cudaStream_t stream);
// Router projection + Top-K softmax in the epilogue; a.block_n must be 32, 64, 128 or 256.
cudaError_t launch_linear_router(const CUtensorMap& amap, const CUtensorMap& bmap, const LinearArgs& a,
                                 int sms, cudaStream_t stream);
cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream);
cudaError_t launch_rope(const RopeArgs& a, cudaStream_t stream);

}  // namespace sa
