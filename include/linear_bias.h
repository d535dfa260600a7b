/*
 * linear_bias.h -- bias-seeded linear layer of libsinkattn.so (sm_103a), the
 * GEMM shape that follows sink attention (the output projection) and runs the
 * experts.
 *
 * The page "GPT-OSS on day 0" (Perplexity, 2025) states in its model overview
 * that the output projection and the experts carry bias terms, and in section
 * "Kernels for GPT-OSS / MoE" that bias support was added to the GEMM kernels
 * by initialising the accumulator from the bias values, once per output tile.
 * This call computes
 *
 *     out[m, n] = sum_k x[m, k] * w[n, k] + bias[n]
 *
 * on the tcgen05 tensor cores: bf16 inputs, fp32 accumulation in tensor
 * memory that starts from the bias (no separate bias add), bf16 output
 * (round to nearest even).
 *
 *  x    bf16 [m, k] row-major;   w bf16 [n, k] row-major (one row per output
 *       feature, the layout of a PyTorch Linear weight);  bias bf16 [n] or NULL
 *  out  bf16 [m, n] row-major
 *  n and k must be multiples of 8 (16-byte rows for the tensor-memory copies);
 *  any m >= 0.  x, w, out 16-byte aligned.
 *
 * Conventions of sink_attn.h apply (device pointers, asynchronous on
 * `stream`, no allocation).  Status: SA_ERR_SHAPE (m < 0, n or k <= 0 or > 2^30,
 * more than 2^31 - 1 output tiles),
 * SA_ERR_UNSUPPORTED (n or k not a multiple of 8), SA_ERR_NULL,
 * SA_ERR_ALIGNMENT, SA_ERR_CUDA / SA_ERR_LAUNCH; m == 0 launches nothing.
 * A device wait that runs out of time (sink_attn_set_wait_timeout_ns) stops
 * the kernel cleanly and sets SA_ERR_TIMEOUT in the device status word.
 */
#ifndef LINEAR_BIAS_H
#define LINEAR_BIAS_H

#include "sink_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

sa_status linear_bias(const void* x, const void* w, const void* bias, int m, int n, int k,
                      void* out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LINEAR_BIAS_H */
