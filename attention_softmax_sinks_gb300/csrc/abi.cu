// C-ABI entry points of libsinkattn.so (declared in include/sink_attn.h):
// argument validation, the per-device status word, TMA descriptor encoding
// and the launches.  No allocation, no synchronisation (except the explicit
// status read-back).
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/linear_bias.h"
#include "../../include/moe_router.h"
#include "../../include/qkv_rope.h"
#include "../../include/sink_attn.h"
#include "internal.h"
#include "ops_internal.h"
#include "ptx.cuh"

namespace {

// Bits set by the kernels (see ptx.cuh); one word per device.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
unsigned* g_status_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
unsigned long long g_timeout_ns = 2000000000ull;

sa_status cuda_fail() { return SA_ERR_CUDA; }

// Device address of this device's status word (host code must not use the
// symbol directly).  Looked up once per device.
sa_status status_ptr(unsigned** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cuda_fail();
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return cuda_fail();
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  *out = g_status_ptr[dev];
  return SA_OK;
}

sa_status encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return cuda_fail();
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *fn = g_encode;
  return SA_OK;
}

// [rows, heads, 64] bf16 tensor read in boxes of (box_rows tokens, box_heads heads, 64 dims);
// consecutive tokens are row_heads head rows apart (heads when 0: a dense tensor; more for
// the query heads inside a [T, (Hq + 2 Hkv) * 64] projection output).
sa_status map_tokens_heads(CUtensorMap* m, const void* base, long long rows, int heads,
                           int box_rows, int box_heads = 1, int row_heads = 0) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  if (sa_status s = encoder(&enc)) return s;
  if (row_heads <= 0) row_heads = heads;
  cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {64 * 2, static_cast<cuuint64_t>(row_heads) * 64 * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_heads), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SA_OK : SA_ERR_CUDA;
}

// Row-major bf16 matrix [rows, cols] read in boxes of (box_rows rows, 64 columns).
sa_status map_matrix(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  if (sa_status s = encoder(&enc)) return s;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SA_OK : SA_ERR_CUDA;
}

// Paged cache [num_pages, hkv, 16, 64] viewed as [num_pages*hkv*16, 64] rows,
// one box = one (page, kv head) = 16 rows.
sa_status map_pages(CUtensorMap* m, const void* base, int num_pages, int hkv) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  if (sa_status s = encoder(&enc)) return s;
  cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(num_pages) * hkv * sa::kPageSize};
  cuuint64_t strides[1] = {64 * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(sa::kPageSize)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SA_OK : SA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool good_scale(float s) { return std::isfinite(s) && s > 0.0f; }

sa_status check_heads(int hq, int hkv, int head_dim) {
  if (hq <= 0 || hkv <= 0) return SA_ERR_SHAPE;
  if (head_dim != sa::kHeadDim) return SA_ERR_UNSUPPORTED;
  if (hq % hkv != 0) return SA_ERR_SHAPE;
  if (hq / hkv > 16) return SA_ERR_UNSUPPORTED;
  return SA_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

std::atomic<int> g_sm_count[kMaxDevices];  // 0 until asked (host threads may race)

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
  if (!g_sm_count[dev].load(std::memory_order_relaxed)) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return g_sm_count[dev].load(std::memory_order_relaxed);
}

// Cluster size for an unsplit decode: CTAs of one (sequence, KV head) share its
// KV range and merge on chip.  Grow (powers of two) to 4 while the grid is below
// about four waves of resident CTAs, and on to 8 or 16 only while it still fits
// one wave (beyond one wave large clusters schedule poorly), every CTA keeping
// >= 16 pages.  One sequence of 4096 tokens with 8 KV heads: 16-CTA clusters,
// 7.3 us per captured step against 9.0 us for 16 explicit splits + merge.
// `slots`: resident decode CTAs on the device (3 per SM).
int cluster_split_for(long long units, long long max_pages, long long slots) {
  int c = 1;
  while (c < 4 && units * c < 4 * slots && max_pages / (2 * c) >= 16) c *= 2;
  // a grid that fits one wave of resident CTAs even split 8 or 16 ways: larger clusters
  // (16 is the non-portable size; the launcher uses 8 when the clusters of 16 would not
  // all be resident at once)
  while (c < 16 && units * 2 * c <= slots && max_pages / (2 * c) >= 16) c *= 2;
  return c;
}

int cluster_split(int units, int max_pages) { return cluster_split_for(units, max_pages, 3LL * sm_count()); }

// One warp waits on a barrier that nothing will ever complete, with the same
// bounded wait the attention kernels use, and reports the timeout.
__global__ void selftest_wait_kernel(unsigned* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    sa::mbar_init(sa::smem_u32(&bar), 1);
    sa::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !sa::mbar_wait(sa::smem_u32(&bar), 0, timeout_ns))
    sa::raise_status(status, sa::kStatusTimeout);
}

// YaRN frequencies and temperature (YaRN paper, section 3, "NTK-by-parts"):
// pairs whose frequency turns at least beta_fast times over the original
// context keep theta_i, pairs that turn at most beta_slow times use
// theta_i / factor, with a ramp linear in the pair index between the two
// (fractional) indices where the number of turns equals beta_fast and beta_slow.
sa_status yarn_tables(double base, double factor, int orig_len, double beta_fast,
                      double beta_slow, double* inv_freq, float* mscale) {
  if (!(base > 1.0) || !std::isfinite(base) || !(factor >= 1.0) || !std::isfinite(factor))
    return SA_ERR_SHAPE;
  const int pairs = sa::kMaxRopePairs;
  for (int i = 0; i < pairs; ++i) inv_freq[i] = std::pow(base, -2.0 * i / sa::kHeadDim);
  *mscale = 1.0f;
  if (factor == 1.0) return SA_OK;
  if (orig_len < 1 || !(beta_slow > 0.0) || !(beta_fast > beta_slow) || !std::isfinite(beta_fast))
    return SA_ERR_SHAPE;
  const double kPi = 3.14159265358979323846;
  auto index_of_turns = [&](double turns) {
    return (sa::kHeadDim / 2.0) * std::log(orig_len / (2.0 * kPi * turns)) / std::log(base);
  };
  const double lo = index_of_turns(beta_fast);
  const double hi = index_of_turns(beta_slow);
  for (int i = 0; i < pairs; ++i) {
    double rho = (i - lo) / (hi - lo);
    rho = rho < 0.0 ? 0.0 : (rho > 1.0 ? 1.0 : rho);
    inv_freq[i] = inv_freq[i] * (1.0 - rho) + inv_freq[i] / factor * rho;
  }
  *mscale = static_cast<float>(0.1 * std::log(factor) + 1.0);
  return SA_OK;
}

sa_status rope_common(const void* qkv, const void* bias, const int32_t* cu_q, const int32_t* kv_lens,
                      int batch, int total_tokens, int hq, int hkv, int head_dim, double base,
                      double factor, int orig_len, double beta_fast, double beta_slow, void* q_out,
                      void* k_out, void* v_out, const int32_t* page_table, int max_pages,
                      int num_pages, bool paged, cudaStream_t stream, bool kv_only = false,
                      float* table_out = nullptr) {
  if (batch < 0 || total_tokens < 0) return SA_ERR_SHAPE;
  const bool work = batch > 0 && total_tokens > 0;  // empty tensors may carry NULL pointers
  if (work && (!qkv || !cu_q || (!kv_only && !q_out))) return SA_ERR_NULL;
  if (work && kv_only && (!k_out || !v_out || !table_out)) return SA_ERR_NULL;
  if (work && paged && (!kv_lens || !page_table || !k_out || !v_out)) return SA_ERR_NULL;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return SA_ERR_SHAPE;
  if (head_dim != sa::kHeadDim) return SA_ERR_UNSUPPORTED;
  if (hq + 2 * hkv > 128) return SA_ERR_UNSUPPORTED;  // one thread per (head row, quarter) per token
  if (paged && (max_pages <= 0 || num_pages <= 0)) return SA_ERR_SHAPE;
  if (static_cast<long long>(total_tokens) * (hq + 2 * hkv) * sa::kHeadDim >= (1LL << 40))
    return SA_ERR_SHAPE;
  const void* ptrs[] = {qkv, bias, kv_only ? nullptr : q_out, k_out, v_out, table_out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return SA_ERR_ALIGNMENT;
  sa::RopeArgs a{};
  if (sa_status s = yarn_tables(base, factor, orig_len, beta_fast, beta_slow, a.inv_freq, &a.mscale))
    return s;
  if (batch == 0 || total_tokens == 0) return SA_OK;
  unsigned* status = nullptr;
  if (sa_status s = status_ptr(&status)) return s;
  a.qkv = static_cast<const uint16_t*>(qkv);
  a.bias = static_cast<const uint16_t*>(bias);
  a.cu_q = cu_q;
  a.kv_lens = kv_lens;
  a.q_out = kv_only ? nullptr : static_cast<uint16_t*>(q_out);
  a.table_out = table_out;
  a.kv_only = kv_only ? 1 : 0;
  a.k_out = static_cast<uint16_t*>(k_out);
  a.v_out = static_cast<uint16_t*>(v_out);
  a.page_table = page_table;
  a.paged = paged ? 1 : 0;
  a.batch = batch;
  a.total_tokens = total_tokens;
  a.hq = hq;
  a.hkv = hkv;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.status = status;
  a.timeout_ns = g_timeout_ns;
  return sa::launch_rope(a, stream) == cudaSuccess ? SA_OK : SA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int sink_attn_abi_version(void) { return 1; }

const char* sink_attn_status_string(sa_status s) {
  switch (s) {
    case SA_OK: return "ok";
    case SA_ERR_NULL: return "a required pointer is NULL";
    case SA_ERR_SHAPE: return "inconsistent or out-of-range sizes or sm_scale";
    case SA_ERR_UNSUPPORTED: return "unsupported configuration (head_dim 64, page_size 16, group <= 16)";
    case SA_ERR_LAUNCH: return "kernel launch failed";
    case SA_ERR_BOUNDS: return "device saw an out-of-range page id or length";
    case SA_ERR_TIMEOUT: return "a device-side wait ran out of time";
    case SA_ERR_ALIGNMENT: return "a tensor pointer is not 16-byte aligned";
    case SA_ERR_CUDA: return "a CUDA runtime call failed";
    case SA_ERR_CAPACITY: return "request exceeds the fixed device scratch of sink_attn_decode_noalloc";
  }
  return "unknown status";
}

void sink_attn_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns = ns; }

sa_status sink_attn_selftest_wait_timeout(unsigned long long timeout_ns, cudaStream_t stream) {
  if (timeout_ns > 1000000000ull) timeout_ns = 1000000000ull;
  unsigned* st = nullptr;
  if (sa_status s = status_ptr(&st)) return s;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(st, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_LAUNCH;
}

sa_status sink_attn_device_status(int clear) {
  unsigned* p = nullptr;
  if (sa_status s = status_ptr(&p)) return s;
  unsigned word = 0;
  if (cudaMemcpy(&word, p, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_fail();
  if (clear && word) {
    const unsigned zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return cuda_fail();
  }
  if (word & sa::kStatusTimeout) return SA_ERR_TIMEOUT;
  if (word & (sa::kStatusBadPage | sa::kStatusBadLen)) return SA_ERR_BOUNDS;
  return SA_OK;
}

int sink_attn_decode_splits(int batch, int num_kv_heads, int max_kv_len, int page_size,
                            int num_sms) {
  if (batch <= 0 || num_kv_heads <= 0 || max_kv_len <= 0 || page_size <= 0) return 1;
  if (num_sms <= 0) num_sms = 152;
  const long long units = static_cast<long long>(batch) * num_kv_heads;
  const long long pages = (max_kv_len + page_size - 1) / page_size;
  const long long slots = 3LL * num_sms;  // resident decode CTAs per GPU
  // num_splits = 1 whenever its clusters (one per (sequence, KV head), merged on chip) fit
  // one wave of resident CTAs and each CTA keeps at most 96 pages: then the on-chip merge
  // beats explicit splits and a merge launch (64/8 heads, 4096 tokens: batch 1-8 run
  // 7.8-15.4 us per step this way against 8.1-20.3 us with the split count below; one
  // sequence of 16384 tokens, 64 pages per CTA: 14.7 against 15.1 us).  With more pages
  // per CTA a warp's page walk is too long (one sequence of 32768 / 65536 tokens: 24.1 /
  // 42.6 us with clusters of 16 against 20.0 / 29.9 us with 32 splits).
  const int c = cluster_split_for(units, pages, slots);
  if (units * c <= slots && pages <= 96LL * c) return 1;
  // Few units: about 5/3 CTAs per SM in all (batch 1 / 2 / 4 at 65536-131072 tokens: 32 /
  // 16 / 8 splits were best or within 3% of it; one 131072-token sequence took 50.5 us so,
  // 84 us with four waves of CTAs).  Otherwise about four waves of CTAs (8 x 131072:
  // 312 us with 32 splits against 332 us with clusters of 4).
  const long long few = 5LL * num_sms / 3;
  long long s = units < 64 ? (few + units - 1) / units : (4 * slots + units - 1) / units;
  // >= 32 pages per split (batch 16 x 4096 tokens: 8 splits 28.1 us, 16 splits 31.6 us)
  const long long max_by_pages = pages / 32 > 0 ? pages / 32 : 1;
  if (s > max_by_pages) s = max_by_pages;
  if (s < 1) s = 1;
  if (s > 256) s = 256;
  return static_cast<int>(s);
}

}  // extern "C"

// rope.table != nullptr: q is the projection output [B, (Hq + 2 Hkv) * 64] and the kernel
// adds rope.q_bias (nullable) and rotates each sequence's query rows by its table row.
static sa_status decode_common(const void* q, const void* paged_k, const void* paged_v,
                               const int32_t* page_table, const int32_t* kv_lens, const float* sinks,
                               int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                               int page_size, int max_pages, int num_pages, float sm_scale,
                               int num_splits, void* out, float* lse, cudaStream_t stream,
                               const sa::DecodeRopeArgs& rope) {
  if (!q || !paged_k || !paged_v || !page_table || !kv_lens || !sinks || !out) return SA_ERR_NULL;
  if (rope.table && (!aligned16(rope.table) || (rope.q_bias && !aligned16(rope.q_bias))))
    return SA_ERR_ALIGNMENT;
  if (num_splits > 1 && !lse) return SA_ERR_NULL;
  if (batch < 0 || max_pages <= 0 || num_pages <= 0) return SA_ERR_SHAPE;
  if (num_splits < 1 || num_splits > 256) return SA_ERR_SHAPE;
  if (sa_status s = check_heads(num_qo_heads, num_kv_heads, head_dim)) return s;
  if (page_size != sa::kPageSize) return SA_ERR_UNSUPPORTED;
  if (!good_scale(sm_scale)) return SA_ERR_SHAPE;
  if (static_cast<long long>(num_pages) * num_kv_heads * page_size >= (1LL << 31)) return SA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(paged_k) || !aligned16(paged_v) || !aligned16(out))
    return SA_ERR_ALIGNMENT;
  if (batch > 65535) return SA_ERR_SHAPE;
  if (batch == 0) return SA_OK;
  sa::DecodeArgs a{};
  a.q = q;
  a.page_table = page_table;
  a.kv_lens = kv_lens;
  a.sinks = sinks;
  a.out = out;
  a.lse = lse;
  a.batch = batch;
  a.hq = num_qo_heads;
  a.hkv = num_kv_heads;
  a.group = num_qo_heads / num_kv_heads;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.num_splits = num_splits;
  a.cluster = num_splits == 1 ? cluster_split(batch * num_kv_heads, max_pages) : 1;
  a.scale_log2 = sm_scale * kLog2e;
  a.timeout_ns = g_timeout_ns;
  if (sa_status s = status_ptr(&a.status)) return s;
  CUtensorMap km, vm;
  if (sa_status s = map_pages(&km, paged_k, num_pages, num_kv_heads)) return s;
  if (sa_status s = map_pages(&vm, paged_v, num_pages, num_kv_heads)) return s;
  return sa::launch_decode(km, vm, a, rope, stream) == cudaSuccess ? SA_OK : SA_ERR_LAUNCH;
}

extern "C" {

sa_status sink_attn_decode(const void* q, const void* paged_k, const void* paged_v,
                           const int32_t* page_table, const int32_t* kv_lens, const float* sinks,
                           int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                           int page_size, int max_pages, int num_pages, float sm_scale,
                           int num_splits, void* out, float* lse, cudaStream_t stream) {
  return decode_common(q, paged_k, paged_v, page_table, kv_lens, sinks, batch, num_qo_heads,
                       num_kv_heads, head_dim, page_size, max_pages, num_pages, sm_scale, num_splits,
                       out, lse, stream, sa::DecodeRopeArgs{});
}

sa_status sink_attn_decode_qkv(const void* qkv, const void* qkv_bias, const float* rope_table,
                               const void* paged_k, const void* paged_v, const int32_t* page_table,
                               const int32_t* kv_lens, const float* sinks, int batch,
                               int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                               int max_pages, int num_pages, float sm_scale, int num_splits,
                               void* out, float* lse, cudaStream_t stream) {
  if (!rope_table) return SA_ERR_NULL;
  if (num_qo_heads > 0 && num_kv_heads > 0 && num_qo_heads + 2 * num_kv_heads > 128)
    return SA_ERR_UNSUPPORTED;
  sa::DecodeRopeArgs rope{static_cast<const uint16_t*>(qkv_bias), reinterpret_cast<const float2*>(rope_table)};
  return decode_common(qkv, paged_k, paged_v, page_table, kv_lens, sinks, batch, num_qo_heads,
                       num_kv_heads, head_dim, page_size, max_pages, num_pages, sm_scale, num_splits,
                       out, lse, stream, rope);
}

sa_status sink_attn_merge(const float* partial_o, const float* partial_lse, int batch,
                          int num_splits, int num_heads, int head_dim, void* out, float* lse_out,
                          cudaStream_t stream) {
  if (!partial_o || !partial_lse || !out) return SA_ERR_NULL;
  if (batch < 0 || num_heads <= 0 || num_splits < 1) return SA_ERR_SHAPE;
  if (head_dim != sa::kHeadDim) return SA_ERR_UNSUPPORTED;
  if (!aligned16(partial_o) || !aligned16(out)) return SA_ERR_ALIGNMENT;
  if (static_cast<long long>(batch) * num_heads >= (1LL << 31)) return SA_ERR_SHAPE;
  if (batch == 0) return SA_OK;
  sa::MergeArgs a{partial_o, partial_lse, out, lse_out, batch, num_splits, num_heads};
  return sa::launch_merge(a, stream) == cudaSuccess ? SA_OK : SA_ERR_LAUNCH;
}

// rope_table != nullptr: q is the projection output [T, (Hq + 2 Hkv) * 64] and the kernel
// adds q_bias (nullable) and rotates the query rows on chip.
static sa_status prefill_common(const void* q, const void* k, const void* v,
                                const int32_t* page_table, const int32_t* cu_q,
                                const int32_t* kv_lens, const float* sinks, int batch,
                                int total_q, int max_q, int hq, int hkv, int head_dim,
                                int max_pages, int num_pages, float sm_scale, int causal,
                                void* out, float* lse, cudaStream_t stream, bool paged,
                                const void* q_bias = nullptr, const float* rope_table = nullptr) {
  if (!q || !k || !v || !cu_q || !sinks || !out) return SA_ERR_NULL;
  const bool rope = rope_table != nullptr;
  if (rope && (!aligned16(rope_table) || (q_bias && !aligned16(q_bias)))) return SA_ERR_ALIGNMENT;
  if (paged && (!page_table || !kv_lens)) return SA_ERR_NULL;
  if (batch < 0 || total_q < 0 || max_q < 0) return SA_ERR_SHAPE;
  if (sa_status s = check_heads(hq, hkv, head_dim)) return s;
  if (!good_scale(sm_scale)) return SA_ERR_SHAPE;
  if (paged && (max_pages <= 0 || num_pages <= 0)) return SA_ERR_SHAPE;
  if (paged && static_cast<long long>(num_pages) * hkv * sa::kPageSize >= (1LL << 31)) return SA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return SA_ERR_ALIGNMENT;
  if (batch == 0 || total_q == 0 || max_q == 0) return SA_OK;
  if (static_cast<long long>(total_q) >= (1LL << 31) - 256) return SA_ERR_SHAPE;
  sa::PrefillArgs a{};
  a.q = q;
  a.cu_q = cu_q;
  a.kv_lens = paged ? kv_lens : nullptr;
  a.page_table = paged ? page_table : nullptr;
  a.sinks = sinks;
  a.out = out;
  a.lse = lse;
  a.batch = batch;
  a.total_q = total_q;
  a.max_q = max_q;
  a.hq = hq;
  a.hkv = hkv;
  a.group = hq / hkv;
  a.max_pages = paged ? max_pages : 0;
  a.num_pages = paged ? num_pages : 0;
  a.causal = causal ? 1 : 0;
  a.paged = paged ? 1 : 0;
  a.scale_log2 = sm_scale * kLog2e;
  a.timeout_ns = g_timeout_ns;
  sa::PrefillRopeArgs ra{};
  ra.q_bias = rope ? static_cast<const uint16_t*>(q_bias) : nullptr;
  ra.table = rope ? reinterpret_cast<const float2*>(rope_table) : nullptr;
  if (sa_status s = status_ptr(&a.status)) return s;
  const int q_row_heads = rope ? hq + 2 * hkv : hq;  // head rows between consecutive tokens of q
  CUtensorMap qm, qpm, km, vm, om;
  if (sa_status s = map_tokens_heads(&qm, q, total_q, hq, 128, 1, q_row_heads)) return s;
  if (sa_status s = map_tokens_heads(&om, out, total_q, hq, 128)) return s;
  // packed short sequences (G = 4, 8, 16): boxes of 128 / G tokens x the G heads of a group
  const int group = hq / hkv;
  if (group >= 4 && 128 % group == 0) {
    if (sa_status s = map_tokens_heads(&qpm, q, total_q, hq, 128 / group, group, q_row_heads)) return s;
  } else {
    qpm = qm;
  }
  if (paged) {
    if (sa_status s = map_pages(&km, k, num_pages, hkv)) return s;
    if (sa_status s = map_pages(&vm, v, num_pages, hkv)) return s;
  } else {
    if (sa_status s = map_tokens_heads(&km, k, total_q, hkv, 128)) return s;
    if (sa_status s = map_tokens_heads(&vm, v, total_q, hkv, 128)) return s;
  }
  return sa::launch_prefill(qm, qpm, km, vm, om, a, ra, stream) == cudaSuccess ? SA_OK : SA_ERR_LAUNCH;
}

sa_status sink_attn_prefill(const void* q, const void* k, const void* v, const float* sinks,
                            const int32_t* cu_seqlens, int batch, int total_tokens,
                            int max_seqlen, int num_qo_heads, int num_kv_heads, int head_dim,
                            float sm_scale, int causal, void* out, float* lse,
                            cudaStream_t stream) {
  return prefill_common(q, k, v, nullptr, cu_seqlens, nullptr, sinks, batch, total_tokens,
                        max_seqlen, num_qo_heads, num_kv_heads, head_dim, 0, 0, sm_scale, causal,
                        out, lse, stream, false);
}

sa_status sink_attn_prefill_paged(const void* q, const void* paged_k, const void* paged_v,
                                  const int32_t* page_table, const int32_t* cu_seqlens_q,
                                  const int32_t* kv_lens, const float* sinks, int batch,
                                  int total_q_tokens, int max_q_len, int num_qo_heads,
                                  int num_kv_heads, int head_dim, int page_size, int max_pages,
                                  int num_pages, float sm_scale, int causal, void* out,
                                  float* lse, cudaStream_t stream) {
  if (page_size != sa::kPageSize && page_size > 0) return SA_ERR_UNSUPPORTED;
  if (page_size <= 0) return SA_ERR_SHAPE;
  return prefill_common(q, paged_k, paged_v, page_table, cu_seqlens_q, kv_lens, sinks, batch,
                        total_q_tokens, max_q_len, num_qo_heads, num_kv_heads, head_dim,
                        max_pages, num_pages, sm_scale, causal, out, lse, stream, true);
}

sa_status sink_attn_prefill_qkv(const void* qkv, const void* qkv_bias, const float* rope_table,
                                const void* k, const void* v, const float* sinks,
                                const int32_t* cu_seqlens, int batch, int total_tokens,
                                int max_seqlen, int num_qo_heads, int num_kv_heads, int head_dim,
                                float sm_scale, int causal, void* out, float* lse,
                                cudaStream_t stream) {
  if (!rope_table) return SA_ERR_NULL;
  if (num_qo_heads > 0 && num_kv_heads > 0 && num_qo_heads + 2 * num_kv_heads > 128)
    return SA_ERR_UNSUPPORTED;
  return prefill_common(qkv, k, v, nullptr, cu_seqlens, nullptr, sinks, batch, total_tokens,
                        max_seqlen, num_qo_heads, num_kv_heads, head_dim, 0, 0, sm_scale, causal,
                        out, lse, stream, false, qkv_bias, rope_table);
}

sa_status sink_attn_prefill_paged_qkv(const void* qkv, const void* qkv_bias, const float* rope_table,
                                      const void* paged_k, const void* paged_v,
                                      const int32_t* page_table, const int32_t* cu_seqlens_q,
                                      const int32_t* kv_lens, const float* sinks, int batch,
                                      int total_q_tokens, int max_q_len, int num_qo_heads,
                                      int num_kv_heads, int head_dim, int page_size, int max_pages,
                                      int num_pages, float sm_scale, int causal, void* out,
                                      float* lse, cudaStream_t stream) {
  if (!rope_table) return SA_ERR_NULL;
  if (page_size != sa::kPageSize && page_size > 0) return SA_ERR_UNSUPPORTED;
  if (page_size <= 0) return SA_ERR_SHAPE;
  if (num_qo_heads > 0 && num_kv_heads > 0 && num_qo_heads + 2 * num_kv_heads > 128)
    return SA_ERR_UNSUPPORTED;
  return prefill_common(qkv, paged_k, paged_v, page_table, cu_seqlens_q, kv_lens, sinks, batch,
                        total_q_tokens, max_q_len, num_qo_heads, num_kv_heads, head_dim,
                        max_pages, num_pages, sm_scale, causal, out, lse, stream, true, qkv_bias,
                        rope_table);
}

sa_status linear_bias(const void* x, const void* w, const void* bias, int m, int n, int k,
                      void* out, cudaStream_t stream) {
  if (m < 0 || n <= 0 || k <= 0 || n > (1 << 30) || k > (1 << 30)) return SA_ERR_SHAPE;
  if (n % 8 != 0 || k % 8 != 0) return SA_ERR_UNSUPPORTED;
  if (m == 0) return SA_OK;
  if (!x || !w || !out) return SA_ERR_NULL;
  if (!aligned16(x) || !aligned16(w) || !aligned16(out) ||
      (bias && (reinterpret_cast<uintptr_t>(bias) & 1u)))
    return SA_ERR_ALIGNMENT;
  sa::LinearArgs a{};
  a.bias = static_cast<const uint16_t*>(bias);
  a.out = static_cast<uint16_t*>(out);
  a.M = m;
  a.N = n;
  a.K = k;
  a.block_n = sa::linear_tile_n(n);
  const long long tiles_m = (static_cast<long long>(m) + 127) / 128;
  const long long tiles_n = (static_cast<long long>(n) + a.block_n - 1) / a.block_n;
  if (tiles_m * tiles_n >= (1LL << 31)) return SA_ERR_SHAPE;
  a.tiles_n = static_cast<int>(tiles_n);
  unsigned* status = nullptr;
  if (sa_status s = status_ptr(&status)) return s;
  a.status = status;
  a.timeout_ns = g_timeout_ns;
  const int sms = sm_count();
  a.m_sub = sa::linear_m_sub(m, n, a.block_n, sms);  // tiles_m above bounds the count for m_sub = 2
  a.tiles_m = static_cast<int>((tiles_m + a.m_sub - 1) / a.m_sub);
  CUtensorMap am, bm;
  if (sa_status s = map_matrix(&am, x, m, k, 128)) return s;
  if (sa_status s = map_matrix(&bm, w, n, k, a.block_n)) return s;
  return sa::launch_linear(am, bm, a, sms, stream) == cudaSuccess ? SA_OK : SA_ERR_LAUNCH;
}

sa_status moe_router(const void* x, const void* w_router, const void* bias, int num_tokens,
                     int hidden, int num_experts, int top_k, int32_t* topk_idx, void* topk_weight,
                     int32_t* expert_counts, cudaStream_t stream) {
  if (num_tokens < 0 || hidden <= 0 || hidden > (1 << 30)) return SA_ERR_SHAPE;
  if (num_experts < 1 || num_experts > 256) return SA_ERR_SHAPE;
  if (top_k < 1 || top_k > 8 || top_k > num_experts) return SA_ERR_SHAPE;
  if (hidden % 8 != 0) return SA_ERR_UNSUPPORTED;
  if (num_tokens > 0 && (!x || !w_router || !topk_idx || !topk_weight)) return SA_ERR_NULL;
  if (num_tokens > 0 && (!aligned16(x) || !aligned16(w_router) ||
                         (bias && (reinterpret_cast<uintptr_t>(bias) & 1u))))
    return SA_ERR_ALIGNMENT;
  if (expert_counts &&
      cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * num_experts, stream) != cudaSuccess)
    return SA_ERR_CUDA;
  if (num_tokens == 0) return SA_OK;
  unsigned* status = nullptr;
  if (sa_status s = status_ptr(&status)) return s;
  sa::LinearArgs a{};
  a.bias = static_cast<const uint16_t*>(bias);
  a.M = num_tokens;
  a.N = num_experts;
  a.K = hidden;
  a.block_n = num_experts <= 32 ? 32 : num_experts <= 64 ? 64 : num_experts <= 128 ? 128 : 256;
  const int sms = sm_count();
  a.m_sub = sa::linear_m_sub(num_tokens, num_experts, a.block_n, sms);
  a.tiles_m = (num_tokens + 128 * a.m_sub - 1) / (128 * a.m_sub);
  a.tiles_n = 1;
  a.status = status;
  a.timeout_ns = g_timeout_ns;
  a.topk_idx = topk_idx;
  a.topk_w = static_cast<uint16_t*>(topk_weight);
  a.counts = expert_counts;
  a.top_k = top_k;
  CUtensorMap am, bm;
  if (sa_status s = map_matrix(&am, x, num_tokens, hidden, 128)) return s;
  if (sa_status s = map_matrix(&bm, w_router, num_experts, hidden, a.block_n)) return s;
  return sa::launch_linear_router(am, bm, a, sms, stream) == cudaSuccess ? SA_OK : SA_ERR_LAUNCH;
}

sa_status moe_router_topk_softmax(const void* logits, long long num_tokens, int num_experts,
                                  int top_k, int32_t* topk_idx, void* topk_weight,
                                  int32_t* expert_counts, cudaStream_t stream) {
  if (num_tokens < 0 || num_experts < 1 || num_experts > 256) return SA_ERR_SHAPE;
  if (top_k < 1 || top_k > 8 || top_k > num_experts) return SA_ERR_SHAPE;
  if (num_tokens > (1LL << 40) / num_experts) return SA_ERR_SHAPE;
  if (num_tokens > 0 && (!logits || !topk_idx || !topk_weight)) return SA_ERR_NULL;
  if (expert_counts &&
      cudaMemsetAsync(expert_counts, 0, sizeof(int32_t) * num_experts, stream) != cudaSuccess)
    return SA_ERR_CUDA;
  if (num_tokens == 0) return SA_OK;
  sa::RouterArgs a{static_cast<const uint16_t*>(logits), topk_idx,
                   static_cast<uint16_t*>(topk_weight), expert_counts, num_tokens, num_experts,
                   top_k, (num_experts % 8 == 0 && aligned16(logits)) ? 1 : 0};
  return sa::launch_router(a, stream) == cudaSuccess ? SA_OK : SA_ERR_LAUNCH;
}

sa_status qkv_bias_rope(const void* qkv, const void* bias, const int32_t* cu_seqlens_q,
                        const int32_t* kv_lens, int batch, int total_tokens, int num_qo_heads,
                        int num_kv_heads, int head_dim, double rope_base, double factor,
                        int orig_len, double beta_fast, double beta_slow, void* q_out,
                        void* k_out, void* v_out, cudaStream_t stream) {
  return rope_common(qkv, bias, cu_seqlens_q, kv_lens, batch, total_tokens, num_qo_heads,
                     num_kv_heads, head_dim, rope_base, factor, orig_len, beta_fast, beta_slow,
                     q_out, k_out, v_out, nullptr, 0, 0, false, stream);
}

sa_status qkv_bias_rope_append_paged(const void* qkv, const void* bias,
                                     const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                     int batch, int total_tokens, int num_qo_heads,
                                     int num_kv_heads, int head_dim, double rope_base,
                                     double factor, int orig_len, double beta_fast,
                                     double beta_slow, void* q_out, void* paged_k, void* paged_v,
                                     const int32_t* page_table, int page_size, int max_pages,
                                     int num_pages, cudaStream_t stream) {
  if (page_size != sa::kPageSize && page_size > 0) return SA_ERR_UNSUPPORTED;
  if (page_size <= 0) return SA_ERR_SHAPE;
  return rope_common(qkv, bias, cu_seqlens_q, kv_lens, batch, total_tokens, num_qo_heads,
                     num_kv_heads, head_dim, rope_base, factor, orig_len, beta_fast, beta_slow,
                     q_out, paged_k, paged_v, page_table, max_pages, num_pages, true, stream);
}

sa_status qkv_bias_rope_kv(const void* qkv, const void* bias, const int32_t* cu_seqlens_q,
                           const int32_t* kv_lens, int batch, int total_tokens, int num_qo_heads,
                           int num_kv_heads, int head_dim, double rope_base, double factor,
                           int orig_len, double beta_fast, double beta_slow, void* k_out,
                           void* v_out, float* rope_table, cudaStream_t stream) {
  return rope_common(qkv, bias, cu_seqlens_q, kv_lens, batch, total_tokens, num_qo_heads,
                     num_kv_heads, head_dim, rope_base, factor, orig_len, beta_fast, beta_slow,
                     nullptr, k_out, v_out, nullptr, 0, 0, false, stream, true, rope_table);
}

sa_status qkv_bias_rope_append_paged_kv(const void* qkv, const void* bias,
                                        const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                                        int batch, int total_tokens, int num_qo_heads,
                                        int num_kv_heads, int head_dim, double rope_base,
                                        double factor, int orig_len, double beta_fast,
                                        double beta_slow, void* paged_k, void* paged_v,
                                        const int32_t* page_table, int page_size, int max_pages,
                                        int num_pages, float* rope_table, cudaStream_t stream) {
  if (page_size != sa::kPageSize && page_size > 0) return SA_ERR_UNSUPPORTED;
  if (page_size <= 0) return SA_ERR_SHAPE;
  return rope_common(qkv, bias, cu_seqlens_q, kv_lens, batch, total_tokens, num_qo_heads,
                     num_kv_heads, head_dim, rope_base, factor, orig_len, beta_fast, beta_slow,
                     nullptr, paged_k, paged_v, page_table, max_pages, num_pages, true, stream, true,
                     rope_table);
}

}  // extern "C"
