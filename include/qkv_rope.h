/*
 * qkv_rope.h -- QKV bias + YaRN rotary encoding + K/V write of libsinkattn.so
 * (sm_103a): the step that produces the q, k, v read by sink attention.
 *
 * The page "GPT-OSS on day 0" (Perplexity, 2025), model overview list, states
 * that the QKV projections carry biases (as in Qwen 2) and that positions use
 * YaRN (as in DeepSeek-V3); it gives no constants.  The rotation follows the
 * YaRN paper (Peng et al., 2023, section 3):
 *
 *   theta_i  = rope_base^(-2 i / 64), i < 32 (feature pairs (i, i + 32))
 *   c(n)     = 32 ln(orig_len / (2 pi n)) / ln(rope_base)
 *   rho_i    = clamp((i - c(beta_fast)) / (c(beta_slow) - c(beta_fast)), 0, 1)
 *   theta'_i = theta_i (1 - rho_i) + (theta_i / factor) rho_i     (factor > 1)
 *   mscale   = 0.1 ln(factor) + 1                                 (factor > 1)
 *   (a, b) = (x_i, x_{i+32})  ->  mscale (a cos - b sin, b cos + a sin),
 *   angle = p theta'_i; factor == 1 gives plain rotary encoding (theta' = theta,
 *   mscale = 1).
 *
 * Token t of sequence b (q_len new tokens, kv_len cached tokens including the
 * new ones) has position p = kv_len - q_len + (t - cu_seqlens_q[b]).
 *
 * Input qkv is the projection output without bias, bf16 [T, (Hq + 2 Hkv) * 64]
 * (all query heads, then key heads, then value heads); bias bf16
 * [(Hq + 2 Hkv) * 64] or NULL is added first (in fp32).  q and k are rotated,
 * v is not; results are rounded once to bf16.  head_dim is 64 and
 * Hq + 2 Hkv <= 128 (SA_ERR_UNSUPPORTED otherwise).
 *
 * Conventions of sink_attn.h apply (device pointers, 16-byte alignment,
 * asynchronous on `stream`, no allocation, status codes).
 */
#ifndef QKV_ROPE_H
#define QKV_ROPE_H

#include "sink_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Contiguous outputs: q_out bf16 [T, Hq, 64], k_out and v_out bf16
 * [T, Hkv, 64] (either may be NULL to skip it).  kv_lens int32 [batch] or
 * NULL (then kv_len == q_len, positions start at 0).
 * SA_ERR_SHAPE: sizes out of range, rope_base <= 1, factor < 1,
 * orig_len < 1 or beta_fast <= beta_slow <= 0 (when factor > 1).
 */
sa_status qkv_bias_rope(const void* qkv, const void* bias, const int32_t* cu_seqlens_q,
                        const int32_t* kv_lens, int batch, int total_tokens, int num_qo_heads,
                        int num_kv_heads, int head_dim, double rope_base, double factor,
                        int orig_len, double beta_fast, double beta_slow, void* q_out,
                        void* k_out, void* v_out, cudaStream_t stream);

/*
 * Same, but k and v are written into the paged cache [num_pages, Hkv, 16, 64]
 * at each new token's position: page page_table[b, p / 16], row p % 16.  No
 * other slot is touched.  kv_lens is required.  A position outside the page
 * table or a page id outside [0, num_pages) is skipped and recorded in the
 * device status word (sink_attn_device_status), never faulted.
 */
sa_status qkv_bias_rope_append_paged(const void* qkv, const void* bias,
                                     const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                     int batch, int total_tokens, int num_qo_heads,
                                     int num_kv_heads, int head_dim, double rope_base,
                                     double factor, int orig_len, double beta_fast,
                                     double beta_slow, void* q_out, void* paged_k, void* paged_v,
                                     const int32_t* page_table, int page_size, int max_pages,
                                     int num_pages, cudaStream_t stream);

/*
 * K/V half of the step, for the attention calls that take q straight from the
 * projection output and rotate it on chip (sink_attn_prefill_qkv,
 * sink_attn_prefill_paged_qkv, sink_attn_decode_qkv in sink_attn.h).  Only
 * the key and value rows of qkv are read; k and v are biased, k rotated, both
 * written as by qkv_bias_rope (contiguous k_out, v_out bf16 [T, Hkv, 64]) or
 * qkv_bias_rope_append_paged (into the paged cache); q is neither read nor
 * written.  Also writes rope_table, fp32 [T, 32, 2]: for every new token t and
 * feature pair i the rotation (mscale cos(p theta'_i), mscale sin(p theta'_i))
 * applied to its k, which the attention call applies to its q.  Every
 * pointer but bias (and kv_lens for the contiguous form) is required.
 */
sa_status qkv_bias_rope_kv(const void* qkv, const void* bias, const int32_t* cu_seqlens_q,
                           const int32_t* kv_lens, int batch, int total_tokens, int num_qo_heads,
                           int num_kv_heads, int head_dim, double rope_base, double factor,
                           int orig_len, double beta_fast, double beta_slow, void* k_out,
                           void* v_out, float* rope_table, cudaStream_t stream);

sa_status qkv_bias_rope_append_paged_kv(const void* qkv, const void* bias,
                                        const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                        int batch, int total_tokens, int num_qo_heads,
                                        int num_kv_heads, int head_dim, double rope_base,
                                        double factor, int orig_len, double beta_fast,
                                        double beta_slow, void* paged_k, void* paged_v,
                                        const int32_t* page_table, int page_size, int max_pages,
                                        int num_pages, float* rope_table, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* QKV_ROPE_H */
