// Launcher interface of the bias-seeded linear layer and its router form
// (linear.cu).  Arguments arrive already validated by abi.cu.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sa {

struct LinearArgs {
  const uint16_t* bias;  // bf16 [N] or nullptr
  uint16_t* out;         // bf16 [M, N] (plain linear layer)
  int M, N, K;
  int block_n, tiles_m, tiles_n;
  int m_sub;  // 128-row sub-tiles per output tile (1 or 2; 2 only with block_n <= 128)
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
// 128-row sub-tiles per output tile (1 or 2) for an M x N output in block_n-wide column
// tiles on `sms` SMs: 2 when the output is one column tile no wider than 128 and 128-row
// tiles would take more than one wave (the two sub-tiles share every W stage).
int linear_m_sub(long long m, int n, int block_n, int sms);
// amap: x [M, K] in boxes of 128 rows x 64; bmap: W [N, K] in boxes of block_n rows x 64.
cudaError_t launch_linear(const CUtensorMap& amap, const CUtensorMap& bmap, const LinearArgs& a,
                          int sms, cudaStream_t stream);
// Router projection + Top-K softmax in the epilogue; a.block_n must be 32, 64, 128 or 256.
cudaError_t launch_linear_router(const CUtensorMap& amap, const CUtensorMap& bmap, const LinearArgs& a,
                                 int sms, cudaStream_t stream);

}  // namespace sa
