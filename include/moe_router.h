/*
 * moe_router.h -- Top-K-then-softmax MoE router of libsinkattn.so (sm_103a).
 *
 * The page "GPT-OSS on day 0" (Perplexity, 2025) lists, in its model overview,
 * "softmax after Top-K for the expert weights", and its section "Kernels for
 * GPT-OSS / MoE" states that for GPT-OSS the softmax runs over the K selected
 * experts only (not over all experts as in DeepSeek-style routers) and that
 * the expert weights must be computed in bfloat16 for accuracy.  Per token t:
 *
 *     S_t = the K experts with the largest logits x[t, e], largest first;
 *           equal logits keep the lower expert index first (-0 equals +0)
 *     w[t, r] = exp(x[t, S_t[r]] - x[t, S_t[0]]) / sum_r' exp(x[t, S_t[r']] - x[t, S_t[0]])
 *
 * The decision is taken on the bf16 logits as given; the weights are computed
 * in fp32 and stored as bf16 (round to nearest even).
 *
 * Shares sa_status and the conventions of sink_attn.h: device pointers owned
 * by the caller, asynchronous on `stream`, no allocation.
 */
#ifndef MOE_ROUTER_H
#define MOE_ROUTER_H

#include "sink_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 *  logits        bf16 [num_tokens, num_experts], row-major (NaN not allowed)
 *  topk_idx      int32 [num_tokens, top_k]: expert ids, largest logit first
 *  topk_weight   bf16 [num_tokens, top_k]: softmax over the selected logits
 *  expert_counts int32 [num_experts] or NULL: overwritten with the number of
 *                (token, selected expert) pairs per expert (the library
 *                clears it with an asynchronous memset on `stream`)
 *  1 <= num_experts <= 256, 1 <= top_k <= min(8, num_experts).
 *  SA_ERR_NULL for a missing required pointer (pointers may be NULL when
 *  num_tokens == 0), SA_ERR_SHAPE for sizes out of
 *  range, SA_ERR_LAUNCH if the launch fails; num_tokens == 0 launches nothing
 *  (the counts are still cleared).
 */
sa_status moe_router_topk_softmax(const void* logits, long long num_tokens, int num_experts,
                                  int top_k, int32_t* topk_idx, void* topk_weight,
                                  int32_t* expert_counts, cudaStream_t stream);

/*
 * The whole router in one tcgen05 kernel: logits = x W_router^T + bias (the
 * accumulator seeded with the bias, as in linear_bias.h), each logit rounded to
 * bf16, then the Top-K softmax above, in the epilogue of the kernel that owns
 * the token's row; no logits are written.  The results are bit-identical to
 * linear_bias followed by moe_router_topk_softmax.
 *
 *  x         bf16 [num_tokens, hidden], 16-byte aligned
 *  w_router  bf16 [num_experts, hidden] (one row per expert), 16-byte aligned
 *  bias      bf16 [num_experts] or NULL
 *  outputs as for moe_router_topk_softmax (expert_counts cleared by the call).
 *  1 <= num_experts <= 256, 1 <= top_k <= min(8, num_experts), hidden a
 *  multiple of 8 (<= 2^30).  Status codes as above; num_tokens == 0 launches
 *  nothing.  A device wait that runs out (sink_attn_set_wait_timeout_ns) ends
 *  the kernel cleanly and sets SA_ERR_TIMEOUT in the device status word.
 */
sa_status moe_router(const void* x, const void* w_router, const void* bias, int num_tokens,
                     int hidden, int num_experts, int top_k, int32_t* topk_idx, void* topk_weight,
                     int32_t* expert_counts, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTER_H */
