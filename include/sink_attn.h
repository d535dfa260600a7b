/*
 * sink_attn.h -- C ABI of libsinkattn.so: GQA attention with per-head softmax
 * sinks on NVIDIA GB300 (sm_103a).
 *
 * The operation is the one stated on the page "GPT-OSS on day 0" (Perplexity,
 * 2025), section "Kernels for GPT-OSS / Sink Attention":
 *
 *     attn = softmax(q k^T * sm_scale  (+)  sink_h) V
 *
 * where each query head h owns one pretrained sink logit sink_h that joins
 * the softmax denominator as one extra column and contributes no row of V.
 * For one query row over its visible keys J (s_j = sm_scale * q.k_j):
 *
 *     M = max(max_j s_j, sink_h),  Z = sum_j e^(s_j - M) + e^(sink_h - M)
 *     out = sum_j e^(s_j - M) v_j / Z,   lse = M + ln Z   (natural log)
 *
 * The same section's online algorithm seeds the running max with the sink
 * (and the running denominator with 1) and, when the KV range is split into
 * blocks, does so for the first block only; sink_attn_decode follows that rule
 * across its splits and sink_attn_merge recombines the split results.
 *
 * Conventions shared by every entry point
 *  - All tensors are DEVICE pointers owned by the caller; the library never
 *    allocates, frees or synchronises.  Every call is asynchronous on `stream`.
 *  - q/k/v/out are bf16 (passed as void*), row-major, dense, 16-byte aligned.
 *    sinks are fp32 [num_qo_heads]; lse outputs are fp32.
 *  - Grouped-query attention: query head h reads KV head h / (Hq / Hkv).
 *  - head_dim must be 64 and page_size 16; Hq % Hkv == 0 and Hq / Hkv <= 16.
 *  - sm_scale must be finite and > 0; it multiplies q.k only, never the sink.
 *  - Invalid arguments are rejected before any launch with a status code.
 *    Device-side problems (a page id outside [0, num_pages), a length larger
 *    than the declared bound, a bounded wait that ran out) never fault: the
 *    kernel skips the access, ORs a bit into a per-device status word and
 *    carries on; sink_attn_device_status() reports and clears it.
 *  - Empty work (batch == 0 or no tokens) returns SA_OK without launching.
 */
#ifndef SINK_ATTN_H
#define SINK_ATTN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sa_status {
  SA_OK = 0,
  SA_ERR_NULL = 1,        /* a required pointer is NULL                        */
  SA_ERR_SHAPE = 2,       /* inconsistent or out-of-range sizes / sm_scale      */
  SA_ERR_UNSUPPORTED = 3, /* head_dim != 64, page_size != 16, group size > 16   */
  SA_ERR_LAUNCH = 4,      /* the kernel launch itself failed                   */
  SA_ERR_BOUNDS = 5,      /* device saw a bad page id or length (status word)  */
  SA_ERR_TIMEOUT = 6,     /* device wait ran out of time (status word)         */
  SA_ERR_ALIGNMENT = 7,   /* a tensor pointer is not 16-byte aligned           */
  SA_ERR_CUDA = 8,        /* a CUDA runtime call made by the library failed    */
  SA_ERR_CAPACITY = 9     /* request larger than sink_attn_decode_noalloc's
                             fixed device scratch                              */
} sa_status;

/*
 * Causal or full attention over a ragged batch of contiguous sequences whose
 * queries are their keys (q_len == kv_len for every sequence): prefill.
 * Section "Kernels for GPT-OSS / Sink Attention" (formula, and the note that
 * the page's FlashInfer-based template serves prefill).
 *
 *  q          bf16 [total_tokens, num_qo_heads, head_dim]
 *  k, v       bf16 [total_tokens, num_kv_heads, head_dim]
 *  sinks      fp32 [num_qo_heads]  (may hold -inf: no sink; +inf: all weight)
 *  cu_seqlens int32 [batch + 1], device; sequence b is rows
 *             [cu_seqlens[b], cu_seqlens[b+1]); must be non-decreasing,
 *             cu_seqlens[0] == 0, cu_seqlens[batch] == total_tokens and every
 *             length <= max_seqlen (violations set SA_ERR_BOUNDS, rows skipped)
 *  causal     nonzero: key j visible to query i iff j <= i
 *  out        bf16 [total_tokens, num_qo_heads, head_dim]
 *  lse        fp32 [total_tokens, num_qo_heads] or NULL
 */
sa_status sink_attn_prefill(const void* q, const void* k, const void* v, const float* sinks,
                            const int32_t* cu_seqlens, int batch, int total_tokens,
                            int max_seqlen, int num_qo_heads, int num_kv_heads, int head_dim,
                            float sm_scale, int causal, void* out, float* lse,
                            cudaStream_t stream);

/*
 * Attention of a mixed batch of new tokens over a paged KV cache: sequence b
 * has q_len_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] new query tokens which are
 * the last q_len_b of its kv_lens[b] cached tokens (q_len_b <= kv_lens[b]).
 * Decode rows (q_len 1) and prefill chunks may be mixed in one call.
 * Causal masking is bottom-right aligned: query i sees key j iff
 * j <= i + kv_len - q_len.
 *
 *  q            bf16 [total_q_tokens, num_qo_heads, head_dim]
 *  paged_k/v    bf16 [num_pages, num_kv_heads, page_size, head_dim]
 *  page_table   int32 [batch, max_pages]; entry (b, j) is the physical page of
 *               logical tokens [j*page_size, (j+1)*page_size) of sequence b
 *  cu_seqlens_q int32 [batch + 1];  kv_lens int32 [batch]
 *  max_q_len    upper bound on every q_len_b
 *  out, lse     as for sink_attn_prefill, indexed by query token
 */
sa_status sink_attn_prefill_paged(const void* q, const void* paged_k, const void* paged_v,
                                  const int32_t* page_table, const int32_t* cu_seqlens_q,
                                  const int32_t* kv_lens, const float* sinks, int batch,
                                  int total_q_tokens, int max_q_len, int num_qo_heads,
                                  int num_kv_heads, int head_dim, int page_size, int max_pages,
                                  int num_pages, float sm_scale, int causal, void* out,
                                  float* lse, cudaStream_t stream);

/*
 * Decode: one new query token per sequence against its paged KV cache, with
 * the KV range optionally split across CTAs.  Section "Kernels for GPT-OSS /
 * Sink Attention": parallel over heads and along the KV length; the sink seeds
 * the running max of the first block only.  Split s of a sequence with
 * n = ceil(kv_len / page_size) pages covers pages [s*c, min((s+1)*c, n)),
 * c = ceil(n / num_splits); only split 0 carries the sink.
 *
 *  q          bf16 [batch, num_qo_heads, head_dim]
 *  paged_k/v, page_table, kv_lens: as for sink_attn_prefill_paged
 *  num_splits 1..256.
 *    == 1: out bf16 [batch, num_qo_heads, head_dim], lse fp32
 *          [batch, num_qo_heads] or NULL -- the final result.  The library
 *          may still divide each sequence's KV range among up to 16 CTAs of a
 *          thread-block cluster (split 0 carries the sink) and combine their
 *          states on chip through distributed shared memory, in one launch.
 *    >  1: out fp32 [batch, num_splits, num_qo_heads, head_dim] holds each
 *          split's normalised partial output and lse fp32
 *          [batch, num_splits, num_qo_heads] (required) its log-sum-exp
 *          (-inf for an empty split without sink); combine with
 *          sink_attn_merge.
 */
sa_status sink_attn_decode(const void* q, const void* paged_k, const void* paged_v,
                           const int32_t* page_table, const int32_t* kv_lens, const float* sinks,
                           int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                           int page_size, int max_pages, int num_pages, float sm_scale,
                           int num_splits, void* out, float* lse, cudaStream_t stream);

/*
 * The same three calls with q taken straight from the QKV projection output,
 * the query bias added and the YaRN rotation applied on chip (page "GPT-OSS on
 * day 0", model overview list: QKV projections with biases, YaRN positions;
 * the rotation itself is specified in qkv_rope.h).  The keys must already be
 * biased and rotated in k / the paged cache, and the (cos, sin) table of the
 * new tokens computed, by qkv_bias_rope_kv or qkv_bias_rope_append_paged_kv
 * (qkv_rope.h); each query row then goes through the same arithmetic as in
 * qkv_bias_rope, so the result equals qkv_bias_rope followed by the plain call.
 *
 *  qkv        bf16 [tokens, (num_qo_heads + 2 num_kv_heads) * head_dim], the
 *             projection output without bias (query heads first); only the
 *             query heads are read.  tokens = total_tokens / total_q_tokens /
 *             batch (decode: one new token per sequence)
 *  qkv_bias   bf16 [(num_qo_heads + 2 num_kv_heads) * head_dim] or NULL; only
 *             the query part is read
 *  rope_table fp32 [tokens, head_dim / 2, 2], as written by the _kv calls
 *  other arguments as for the plain call; num_qo_heads + 2 num_kv_heads <= 128
 *  (SA_ERR_UNSUPPORTED otherwise).  The prefills use the same schedules as
 *  the plain calls; once a query tile has landed in shared memory, each
 *  softmax thread biases and rotates its own row there before the tile's
 *  first score product.
 */
sa_status sink_attn_prefill_qkv(const void* qkv, const void* qkv_bias, const float* rope_table,
                                const void* k, const void* v, const float* sinks,
                                const int32_t* cu_seqlens, int batch, int total_tokens,
                                int max_seqlen, int num_qo_heads, int num_kv_heads, int head_dim,
                                float sm_scale, int causal, void* out, float* lse,
                                cudaStream_t stream);
sa_status sink_attn_prefill_paged_qkv(const void* qkv, const void* qkv_bias, const float* rope_table,
                                      const void* paged_k, const void* paged_v,
                                      const int32_t* page_table, const int32_t* cu_seqlens_q,
                                      const int32_t* kv_lens, const float* sinks, int batch,
                                      int total_q_tokens, int max_q_len, int num_qo_heads,
                                      int num_kv_heads, int head_dim, int page_size, int max_pages,
                                      int num_pages, float sm_scale, int causal, void* out,
                                      float* lse, cudaStream_t stream);
sa_status sink_attn_decode_qkv(const void* qkv, const void* qkv_bias, const float* rope_table,
                               const void* paged_k, const void* paged_v, const int32_t* page_table,
                               const int32_t* kv_lens, const float* sinks, int batch,
                               int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                               int max_pages, int num_pages, float sm_scale, int num_splits,
                               void* out, float* lse, cudaStream_t stream);

/*
 * Merge split partials into the final result:
 *   lse = ln sum_s e^(lse_s),  out = sum_s e^(lse_s - lse) o_s  (bf16).
 * Implied by the split rule of section "Kernels for GPT-OSS / Sink Attention";
 * the combine itself is the standard log-sum-exp merge.
 *
 *  partial_o   fp32 [batch, num_splits, num_heads, head_dim]
 *  partial_lse fp32 [batch, num_splits, num_heads]
 *  out         bf16 [batch, num_heads, head_dim];  lse_out fp32 [batch, num_heads] or NULL
 * A row whose partials are all -inf yields out = 0, lse = -inf.
 */
sa_status sink_attn_merge(const float* partial_o, const float* partial_lse, int batch,
                          int num_splits, int num_heads, int head_dim, void* out, float* lse_out,
                          cudaStream_t stream);

/*
 * Split-KV decode followed by the merge, in one call that allocates nothing.
 * The page has no counterpart for this entry point; it exists for callers that
 * cannot allocate device memory when they enqueue work (a plugin that is only
 * handed its input and output buffers, a serving loop that bans allocation on
 * its hot path because cudaMalloc may synchronise or fail).  Those callers
 * cannot supply the fp32 partials that sink_attn_decode and sink_attn_merge
 * exchange, so this call keeps them in a fixed device array inside the library
 * (8 MiB, 2,097,152 floats).  Under CUDA's lazy module loading (the default)
 * the array is created on a device when the library's device code is first
 * used there, at the latest by this call's first use on that device, and is
 * then held until the process exits.
 *
 *  Arguments are those of sink_attn_decode, but `out` is always the final
 *  bf16 [batch, num_qo_heads, head_dim] and `lse` the final fp32
 *  [batch, num_qo_heads] (or NULL), whatever num_splits is.
 *  Limit: batch * num_splits * num_qo_heads * (head_dim + 1) <= 2,097,152,
 *  otherwise SA_ERR_CAPACITY and nothing is launched.  num_splits == 1 needs
 *  no scratch and behaves exactly like sink_attn_decode.
 *  No cudaMalloc, cudaFree or other allocation happens in this call.  The first
 *  call on each device may load the library's device code there and looks up
 *  the array's device address (a runtime query, not an allocation); because of
 *  that module load, make that first call before any stream capture.
 *  Every call shares the array, which keeps the previous call's contents; a
 *  call writes every element it later reads, so nothing needs clearing, but
 *  two calls that overlap on the GPU race on it: order them on one stream.
 */
sa_status sink_attn_decode_noalloc(const void* q, const void* paged_k, const void* paged_v,
                                   const int32_t* page_table, const int32_t* kv_lens,
                                   const float* sinks, int batch, int num_qo_heads,
                                   int num_kv_heads, int head_dim, int page_size, int max_pages,
                                   int num_pages, float sm_scale, int num_splits, void* out,
                                   float* lse, cudaStream_t stream);

/*
 * Host-only helper: a split count for sink_attn_decode (fp32 partials, then
 * sink_attn_merge).  With fewer than 64 (sequence, KV head) units it aims at
 * about 5/3 CTAs per SM in all, otherwise at about four waves of resident
 * CTAs, keeping every split at least 32 pages long.  Returns a value in
 * [1, 256].  1 means: call sink_attn_decode with num_splits == 1 (no merge
 * call); it is returned when the clusters that call would use, one per
 * (sequence, KV head), fit one wave of resident CTAs (3 per SM) and each of
 * their CTAs keeps at most 96 pages: the on-chip cluster merge then beats
 * explicit splits.  No CUDA call.
 */
int sink_attn_decode_splits(int batch, int num_kv_heads, int max_kv_len, int page_size,
                            int num_sms);

/*
 * Read (and, if `clear` is nonzero, reset) the current device's status word.
 * SYNCHRONISES the device.  Returns SA_OK, SA_ERR_BOUNDS or SA_ERR_TIMEOUT
 * (timeout wins if both bits are set), or SA_ERR_CUDA.
 */
sa_status sink_attn_device_status(int clear);

/* Upper bound, in nanoseconds, on every device-side wait of later launches
 * (default 2e9).  A wait that runs out stops its CTA cleanly and sets
 * SA_ERR_TIMEOUT in the status word.  Host-only, not thread-safe. */
void sink_attn_set_wait_timeout_ns(unsigned long long ns);

/* Diagnostic: launch one warp that waits on a device barrier nothing will
 * ever release, using the same bounded wait as the attention kernels.  After
 * timeout_ns (capped at 1e9) the wait gives up and SA_ERR_TIMEOUT is recorded
 * in the status word; read it with sink_attn_device_status().  Lets a caller
 * confirm, without faulting the GPU, that device waits end and are reported.
 * Not part of the page's method. */
sa_status sink_attn_selftest_wait_timeout(unsigned long long timeout_ns, cudaStream_t stream);

/* Static string for a status code (never NULL). */
const char* sink_attn_status_string(sa_status status);

/* Version of this ABI (incremented on incompatible change). */
int sink_attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SINK_ATTN_H */
