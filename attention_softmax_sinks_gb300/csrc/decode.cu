// Paged split-KV decode with softmax sinks (one new query token per sequence).
//
// Page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention":
// attention is parallel over heads and along the KV length; the online
// softmax keeps a running max m and denominator d, seeded with the head's
// sink (m = sink, d = 1) in the first KV block only.
//
// GB300 design (memory bound, ~8 flop per KV byte at a group of 8):
//  * one CTA per (split, kv head, sequence); its 4 warps walk the split's
//    pages interleaved, each with a private 4-deep ring of TMA page loads
//    (one 2 KiB K box + one 2 KiB V box per page, 128-byte swizzle, L2
//    evict-first), so no CTA-wide barrier sits in the streaming loop; a warp
//    consumes two pages per step (one max reduction and one rescale for both)
//    and keeps the page ids of its next 32 pages in registers;
//  * the whole GQA group of a KV head is one 8-wide MMA "N" tile: scores are
//    computed transposed, S^T[16 tok x 8 heads] = K_page . Q^T, and the PV
//    product as O^T[64 x 8] += V^T . P^T, so mma.sync m16n8k16 runs with no
//    padding; P^T is formed from the score fragments with movmatrix;
//  * per-lane partial denominators, warp-shuffle row max, one smem merge of
//    the 4 warp states at the end; split 0's warp 0 starts from the sink;
//  * an unsplit call may divide a sequence's range among the CTAs of a
//    cluster (up to 16): each CTA pushes its state for every (head, 4-dim
//    chunk) output into the shared memory of the rank that combines it, one
//    cluster barrier later each rank combines from its own shared memory and
//    no rank waits for another before it exits (4096-token graph step 6.66 ->
//    6.22 us, against reading the other ranks' states between two barriers);
//  * launched with programmatic dependent launch, so a CTA is resident while
//    the kernel before it (the previous step's merge) still runs: in that time
//    it asks L2 for the first four pages of each warp's ring, which hides the
//    page-table -> page latency of its start (headline step 85.8 -> 80.8 us);
//    after the wait, the warp's first page ids are read in the same round trip
//    as the sequence length, for the length seen before the wait, and read
//    again only if the length changed (64 x 4096 step 78.3 -> 78.0 us).
#include <mutex>
#include "internal.h"
#include "ptx.cuh"
#include "rope_math.cuh"

namespace sa {
namespace {

constexpr int kWarps = 4;
constexpr int kStages = 4;
constexpr int kPageBytes = kPageSize * kHeadDim * 2;  // 2 KiB per (page, kv head)
constexpr int kSlotBytes = 2 * kPageBytes;            // K + V
constexpr int kRingBytes = kWarps * kStages * kSlotBytes;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

template <int NT>
struct MergeArea {  // aliases the ring once streaming is over
  float m[kWarps][NT * 8];
  float d[kWarps][NT * 8];
  float o[kWarps][NT * 8][kHeadDim];
};

// Ask L2 for one tensor-map box (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}

// Cluster merge: every CTA pushes the partial state of each (head, 4-dim chunk) output to
// the rank that combines it, into that rank's receive area (outside the ring, which a slower
// rank may still be streaming through): 8 floats (o[4], m, d, pad) per (source, item).
constexpr int kRecvEntries = 16 * 8 + 16;  // csz * ceil(16 G / csz) <= 16 G + csz - 1
constexpr int kRecvBytes = 2 * kRecvEntries * 32;  // up to two query tiles (G <= 16)
constexpr size_t decode_smem_bytes() {
  return 1024 /*alignment slack*/ + kRingBytes + kWarps * kStages * sizeof(uint64_t) + kRecvBytes;
}

// Rank r combines items [r * per_rank, (r + 1) * per_rank) of the G * 16 (head, 4-dim chunk)
// outputs from the csz states pushed into its receive area (the merge kernel's arithmetic;
// the sums over the csz sources are taken in a butterfly's order).  Kept out of line: inlined,
// the cluster merge changed the streaming loop's code and slowed unclustered launches.
__device__ __noinline__ void cluster_combine(uint32_t recv, int csz, void* out_bf16, float* lse_out, int hq, int b,
                                             int kvh, int G) {
  const int n_out = G * 16;
  const int per_rank = (n_out + csz - 1) / csz;
  const int rank = static_cast<int>(cluster_ctarank());
  for (int j = threadIdx.x; j < per_rank; j += kWarps * 32) {
    const int i = rank * per_rank + j;
    if (i >= n_out) break;
    float ms[16], dn[16], o0[16], o1[16], o2[16], o3[16];
    float M = kNegInf;
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s < csz) {
        const uint32_t e = recv + static_cast<uint32_t>((s * per_rank + j) * 32);
        float4 o;
        float2 md;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(o.x), "=f"(o.y), "=f"(o.z), "=f"(o.w) : "r"(e));
        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(md.x), "=f"(md.y) : "r"(e + 16));
        ms[s] = md.x;
        M = fmaxf(M, md.x);
        dn[s] = md.y;
        o0[s] = o.x;
        o1[s] = o.y;
        o2[s] = o.z;
        o3[s] = o.w;
      }
    }
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s < csz) {
        const float c = (M == kNegInf || ms[s] == M) ? 1.0f : ex2(ms[s] - M);
        dn[s] *= c;
        o0[s] *= c;
        o1[s] *= c;
        o2[s] *= c;
        o3[s] *= c;
      }
    }
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) {
      if (off < csz) {
#pragma unroll
        for (int s = 0; s < 16; s += 2 * off) {
          if (s + off < csz) {
            dn[s] = dn[s] + dn[s + off];
            o0[s] = o0[s] + o0[s + off];
            o1[s] = o1[s] + o1[s + off];
            o2[s] = o2[s] + o2[s + off];
            o3[s] = o3[s] + o3[s + off];
          }
        }
      }
    }
    const float den = dn[0];
    const float inv = den > 0.0f ? 1.0f / den : 0.0f;
    const int hh = i >> 4, d0 = (i & 15) * 4;
    const int head = kvh * G + hh;
    uint16_t* out = static_cast<uint16_t*>(out_bf16) + (static_cast<size_t>(b) * hq + head) * kHeadDim + d0;
    uint2 pk;
    pk.x = pack_bf16x2(o0[0] * inv, o1[0] * inv);
    pk.y = pack_bf16x2(o2[0] * inv, o3[0] * inv);
    *reinterpret_cast<uint2*>(out) = pk;
    if (lse_out && d0 == 0)
      lse_out[static_cast<size_t>(b) * hq + head] = den > 0.0f ? (M + lg2(den)) * kLn2 : kNegInf;
  }
}

template <int NT, bool kRope>
__global__ void __launch_bounds__(kWarps * 32)
    sink_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const DecodeArgs a,
                       const DecodeRopeArgs rope) {
  static_assert(sizeof(MergeArea<NT>) <= kRingBytes, "the merge area must fit in the ring");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kRingBytes);
  const uint32_t recv_u32 = smem_u32(ring + kRingBytes + kWarps * kStages * sizeof(uint64_t));

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // clustered launch: announce that this CTA runs (waited for before the first remote store)
  if (a.cluster > 1) cluster_arrive_relaxed();
  const int G = a.group;
  const uint32_t ring_w = smem_u32(ring + warp * kStages * kSlotBytes);
  const uint32_t full_w = smem_u32(full + warp * kStages);

  // kv_lens and the page table may still be being written by the kernel before this one:
  // what is read before the wait below only chooses what to prefetch and which page-table
  // entries to read early (both are read again after the wait and checked).
  const int kvl = a.kv_lens[blockIdx.z];
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(full_w + 8 * s, 1);
    fence_barrier_init();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    // While the kernel before this one finishes, ask L2 for this warp's first pages.
    if (kvl > 0 && kvl <= a.max_pages * kPageSize) {
      const int np = (kvl + kPageSize - 1) / kPageSize;
      const int ns = a.cluster > 1 ? a.cluster : a.num_splits;
      const int per = (np + ns - 1) / ns;
      const int pb = min(static_cast<int>(blockIdx.x) * per, np);
      const int pe = min(pb + per, np);
      const int32_t* pt = a.page_table + static_cast<size_t>(blockIdx.z) * a.max_pages;
      for (int j = 0; j < kStages; ++j) {
        const int pg = pb + warp + j * kWarps;
        if (pg >= pe) break;
        const int phys = pt[pg];
        if (phys < 0 || phys >= a.num_pages) continue;
        const int row = (phys * a.hkv + static_cast<int>(blockIdx.y)) * kPageSize;
        tma_prefetch_l2_2d(&kmap, 0, row);
        tma_prefetch_l2_2d(&vmap, 0, row);
      }
    }
  }
  __syncwarp();
  // Launched with programmatic stream serialisation: the set-up above may overlap
  // the kernel before this one; apart from the prefetch hints above, every read of
  // an input comes after this wait.
  pdl_wait_primary();

  const int cap = a.max_pages * kPageSize;
  const bool clustered = a.cluster > 1;  // splits of one (sequence, KV head) form a cluster
  const int n_split = clustered ? a.cluster : a.num_splits;
  const int32_t* ptab = a.page_table + static_cast<size_t>(b) * a.max_pages;
  // this warp's pages for a sequence of kv tokens: p_begin + warp + j * kWarps, j < count
  auto warp_pages = [&](int kv, int& first, int& count) {
    const int np = (kv + kPageSize - 1) / kPageSize;
    const int per = (np + n_split - 1) / n_split;
    const int pb = min(split * per, np);
    const int pe = min(pb + per, np);
    first = pb + warp;
    count = first < pe ? (pe - first + kWarps - 1) / kWarps : 0;
  };
  // Page ids, 32 of this warp's pages at a time: lane l of ids_cur holds the id of the
  // warp's page 32 w + l (window w holds the page being consumed) and ids_next those of
  // window w + 1, read a whole window ahead, so no page-table read sits in the loop.
  int my_first, my_count;
  auto load_ids = [&](int w) {
    const int jj = w * 32 + lane;
    return jj < my_count ? ptab[my_first + jj * kWarps] : -1;
  };
  // The first window is read together with kv_lens, for the length read before the wait;
  // if the length read now differs, it is read again.
  const int kv_early = (kvl < 0 || kvl > cap) ? 0 : kvl;
  warp_pages(kv_early, my_first, my_count);
  int ids_cur = load_ids(0);
  int kv_len = a.kv_lens[b];
  if (kv_len < 0 || kv_len > cap) {
    if (threadIdx.x == 0) raise_status(a.status, kStatusBadLen);
    kv_len = kv_len < 0 ? 0 : cap;
  }
  if (kv_len != kv_early) {
    warp_pages(kv_len, my_first, my_count);
    ids_cur = load_ids(0);
  }
  int ids_next = load_ids(1);
  auto id_of = [&](int k, int w) {  // all lanes; page k lies in window w or w + 1
    const int in_cur = __shfl_sync(0xffffffffu, ids_cur, k & 31);
    const int in_next = __shfl_sync(0xffffffffu, ids_next, k & 31);
    return (k >> 5) == w ? in_cur : in_next;
  };

  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int j, int phys) {  // lane 0 only
    const uint32_t bar = full_w + 8 * (j % kStages);
    if (phys < 0 || phys >= a.num_pages) {
      raise_status(a.status, kStatusBadPage);
      mbar_arrive(bar);  // completes the phase with nothing copied; page is skipped
      return;
    }
    const uint32_t dst = ring_w + (j % kStages) * kSlotBytes;
    const int row = (phys * a.hkv + kvh) * kPageSize;
    mbar_arrive_expect_tx(bar, kSlotBytes);
    tma_load_2d(dst, &kmap, 0, row, bar, policy);
    tma_load_2d(dst + kPageBytes, &vmap, 0, row, bar, policy);
  };
  int issued = min(kStages, my_count);  // meaningful on lane 0
  {
    int first_ids[kStages];
#pragma unroll
    for (int jj = 0; jj < kStages; ++jj) first_ids[jj] = id_of(jj, 0);
    if (lane == 0)
      for (int jj = 0; jj < issued; ++jj) issue(jj, first_ids[jj]);
  }

  // Q^T fragments (B operand of S^T = K Q^T): lane holds head (lane/4) of each
  // 8-wide tile, dims kk*16 + 2*(lane%4) + {0,1} and +8.
  // With q taken from the projection output (kRope), the lane adds the bias and rotates
  // its pairs in registers (it holds dims d and d + 32 of its heads: fragments kk and
  // kk + 2), with the arithmetic of the kernel that writes rotated q.
  uint32_t qf[NT][4][2];
  const int q_row_heads = kRope ? a.hq + 2 * a.hkv : a.hq;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 8 + (lane >> 2);
    const bool ok = hh < G;
    const int head = kvh * G + (ok ? hh : 0);
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const uint16_t*>(a.q) + (static_cast<size_t>(b) * q_row_heads + head) * kHeadDim);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      qf[nt][kk][0] = ok ? qrow[kk * 8 + (lane & 3)] : 0u;
      qf[nt][kk][1] = ok ? qrow[kk * 8 + 4 + (lane & 3)] : 0u;
    }
    if (kRope && ok) {
      const uint32_t* brow = rope.q_bias ? reinterpret_cast<const uint32_t*>(rope.q_bias + head * kHeadDim) : nullptr;
      const float4* cs = reinterpret_cast<const float4*>(rope.table + static_cast<size_t>(b) * (kHeadDim / 2));
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int w = kk * 8 + 4 * c + (lane & 3);  // 32-bit word: dims 2w, 2w + 1 (pair index)
          float a0 = bf16_lo(qf[nt][kk][c]), a1 = bf16_hi(qf[nt][kk][c]);
          float b0 = bf16_lo(qf[nt][kk + 2][c]), b1 = bf16_hi(qf[nt][kk + 2][c]);
          if (brow) {
            const uint32_t ba = brow[w], bb = brow[w + 16];
            a0 += bf16_lo(ba);
            a1 += bf16_hi(ba);
            b0 += bf16_lo(bb);
            b1 += bf16_hi(bb);
          }
          const float4 r = cs[w];  // (cos, sin) of pairs 2w and 2w + 1
          rotate_pair(a0, b0, r.x, r.y);
          rotate_pair(a1, b1, r.z, r.w);
          qf[nt][kk][c] = pack_bf16x2(a0, a1);
          qf[nt][kk + 2][c] = pack_bf16x2(b0, b1);
        }
      }
    }
  }

  // Running state for heads nt*8 + 2*(lane%4) + {0,1}; m in log2 units.
  float m[NT][2], dsum[NT][2], o[NT][4][4];
  const bool seed = (split == 0 && warp == 0);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hh = nt * 8 + 2 * (lane & 3) + e;
      float sink = kNegInf;
      if (seed && hh < G) sink = a.sinks[kvh * G + hh] * kLog2e;
      m[nt][e] = sink;
      // d starts at exp(sink - sink) = 1, counted once (lane/4 == 0); 0 for -inf
      dsum[nt][e] = (sink != kNegInf && (lane >> 2) == 0) ? 1.0f : 0.0f;
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) o[nt][mt][r] = 0.0f;
  }

  // S^T = K Q^T of the page in ring slot `slot` (16 tokens x 8 heads per tile)
  auto scores = [&](int slot, float (&sc)[NT][4]) {
    const uint32_t kb = ring_w + slot * kSlotBytes;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) sc[nt][r] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int chunk = kk * 2 + (lane >> 4);
      uint32_t a0, a1, a2, a3;
      ldsm_x4(kb + row * 128 + ((chunk ^ (row & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sc[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
    }
  };
  // O^T += V^T P^T for the page in ring slot `slot` (64 dims x 8 heads per tile)
  auto accumulate = [&](int slot, const uint32_t (&pt)[NT][2]) {
    const uint32_t vb = ring_w + slot * kSlotBytes + kPageBytes;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int tok = (lane & 7) + (lane >> 4) * 8;
      const int chunk = mt * 2 + ((lane >> 3) & 1);
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(vb + tok * 128 + ((chunk ^ (tok & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[nt][mt], a0, a1, a2, a3, pt[nt][0], pt[nt][1]);
    }
  };

  // Two pages per step: their score products are independent, and one max reduction and
  // one rescale serve both, so a warp's serial chain per page is about halved.
  bool timed_out = false;
  int j = 0;
  for (; j < my_count; j += 2) {
    const int win = j >> 5;  // j is even: page j + 1 lies in the same window
    if ((j & 31) == 0 && j > 0) {  // entering window win: its ids are loaded, fetch the next
      ids_cur = ids_next;
      ids_next = load_ids(win + 1);
    }
    const bool two = j + 1 < my_count;
    if (!mbar_wait(full_w + 8 * (j % kStages), (j / kStages) & 1, a.timeout_ns) ||
        (two && !mbar_wait(full_w + 8 * ((j + 1) % kStages), ((j + 1) / kStages) & 1, a.timeout_ns))) {
      timed_out = true;
      break;
    }
    const int phys_a = id_of(j, win), phys_b = id_of(j + 1, win);
    const bool use_a = phys_a >= 0 && phys_a < a.num_pages;
    const bool use_b = two && phys_b >= 0 && phys_b < a.num_pages;
    if (use_a || use_b) {
      float sa[NT][4], sb[NT][4];
      if (use_a) scores(j % kStages, sa);
      if (use_b) scores((j + 1) % kStages, sb);
      // ---- scale, mask the ragged tail (and a skipped page), online softmax update
      const int tok_a = (my_first + j * kWarps) * kPageSize + (lane >> 2);
      const int tok_b = tok_a + kWarps * kPageSize;
      const bool a0v = use_a && tok_a < kv_len, a1v = use_a && tok_a + 8 < kv_len;
      const bool b0v = use_b && tok_b < kv_len, b1v = use_b && tok_b + 8 < kv_len;
      uint32_t pta[NT][2], ptb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float xa0 = a0v ? sa[nt][0] * a.scale_log2 : kNegInf;
        const float xa1 = a0v ? sa[nt][1] * a.scale_log2 : kNegInf;
        const float xa2 = a1v ? sa[nt][2] * a.scale_log2 : kNegInf;
        const float xa3 = a1v ? sa[nt][3] * a.scale_log2 : kNegInf;
        const float xb0 = b0v ? sb[nt][0] * a.scale_log2 : kNegInf;
        const float xb1 = b0v ? sb[nt][1] * a.scale_log2 : kNegInf;
        const float xb2 = b1v ? sb[nt][2] * a.scale_log2 : kNegInf;
        const float xb3 = b1v ? sb[nt][3] * a.scale_log2 : kNegInf;
        float mx0 = fmaxf(fmaxf(xa0, xa2), fmaxf(xb0, xb2));
        float mx1 = fmaxf(fmaxf(xa1, xa3), fmaxf(xb1, xb3));
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
        const float mu0 = mn0 == kNegInf ? 0.0f : mn0;
        const float mu1 = mn1 == kNegInf ? 0.0f : mn1;
        const float c0 = m[nt][0] == mn0 ? 1.0f : ex2(m[nt][0] - mu0);
        const float c1 = m[nt][1] == mn1 ? 1.0f : ex2(m[nt][1] - mu1);
        m[nt][0] = mn0;
        m[nt][1] = mn1;
        const float pa0 = ex2(xa0 - mu0), pa1 = ex2(xa1 - mu1);
        const float pa2 = ex2(xa2 - mu0), pa3 = ex2(xa3 - mu1);
        const float pb0 = ex2(xb0 - mu0), pb1 = ex2(xb1 - mu1);
        const float pb2 = ex2(xb2 - mu0), pb3 = ex2(xb3 - mu1);
        dsum[nt][0] = dsum[nt][0] * c0 + ((pa0 + pa2) + (pb0 + pb2));
        dsum[nt][1] = dsum[nt][1] * c1 + ((pa1 + pa3) + (pb1 + pb3));
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          o[nt][mt][0] *= c0;
          o[nt][mt][1] *= c1;
          o[nt][mt][2] *= c0;
          o[nt][mt][3] *= c1;
        }
        // P^T as the B operand of O^T += V^T P^T: transpose the two 8x8 blocks
        pta[nt][0] = movmatrix_trans(pack_bf16x2(pa0, pa1));
        pta[nt][1] = movmatrix_trans(pack_bf16x2(pa2, pa3));
        ptb[nt][0] = movmatrix_trans(pack_bf16x2(pb0, pb1));
        ptb[nt][1] = movmatrix_trans(pack_bf16x2(pb2, pb3));
      }
      if (use_a) accumulate(j % kStages, pta);
      if (use_b) accumulate((j + 1) % kStages, ptb);
    }
    __syncwarp();
    const int next_a = id_of(j + kStages, win), next_b = id_of(j + kStages + 1, win);
    if (lane == 0) {
      if (j + kStages < my_count) {
        issue(j + kStages, next_a);
        ++issued;
      }
      if (j + kStages + 1 < my_count) {
        issue(j + kStages + 1, next_b);
        ++issued;
      }
    }
  }

  if (timed_out) {
    if (lane == 0) {
      raise_status(a.status, kStatusTimeout);
      // let copies still in flight land before the CTA's shared memory goes away
      // (bounded again; default limit even if the caller asked for a tiny one)
      for (int jj = j; jj < issued; ++jj)
        mbar_wait(full_w + 8 * (jj % kStages), (jj / kStages) & 1, 2000000000ull);
    }
    __syncwarp();
  }

  // the merge kernel that follows may start launching; it waits for this grid's results
  pdl_launch_dependents();

  // ---- combine the lanes' partial denominators
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        dsum[nt][e] += __shfl_xor_sync(0xffffffffu, dsum[nt][e], off);

  __syncthreads();  // every warp is done with its ring; reuse it for the merge
  MergeArea<NT>* mg = reinterpret_cast<MergeArea<NT>*>(ring);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hh = nt * 8 + 2 * (lane & 3) + e;
      if ((lane >> 2) == 0) {
        mg->m[warp][hh] = m[nt][e];
        mg->d[warp][hh] = dsum[nt][e];
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        mg->o[warp][hh][mt * 16 + (lane >> 2)] = o[nt][mt][e];
        mg->o[warp][hh][mt * 16 + (lane >> 2) + 8] = o[nt][mt][2 + e];
      }
    }
  }
  __syncthreads();

  if (clustered) cluster_wait();  // every CTA of the cluster has started: its shared memory may be written
  for (int i = threadIdx.x; i < G * 16; i += kWarps * 32) {
    const int hh = i >> 4, d0 = (i & 15) * 4;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mg->m[w][hh]);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float den = 0.0f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = mg->m[w][hh];
        const float c = mw == M ? 1.0f : ex2(mw - M);
        den += mg->d[w][hh] * c;
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[r] += mg->o[w][hh][d0 + r] * c;
      }
    }
    if (clustered) {  // push the CTA's state for item i to the rank that combines it
      const int csz = a.cluster;
      const int per_rank = (G * 16 + csz - 1) / csz;
      const int owner = i / per_rank, slot = i - owner * per_rank;
      const uint32_t entry = recv_u32 + static_cast<uint32_t>((cluster_ctarank() * per_rank + slot) * 32);
      const uint32_t remote = dsmem_addr(entry, static_cast<uint32_t>(owner));
      dsmem_st4(remote, acc[0], acc[1], acc[2], acc[3]);
      dsmem_st2(remote + 16, M, den);
      continue;
    }
    const float inv = den > 0.0f ? 1.0f / den : 0.0f;
    const float lse = den > 0.0f ? (M + lg2(den)) * kLn2 : kNegInf;
    const int head = kvh * G + hh;
    if (a.num_splits == 1) {
      uint16_t* out = static_cast<uint16_t*>(a.out) +
                      (static_cast<size_t>(b) * a.hq + head) * kHeadDim + d0;
      uint2 pk;
      pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(out) = pk;
      if (a.lse && d0 == 0) a.lse[static_cast<size_t>(b) * a.hq + head] = lse;
    } else {
      const size_t row = (static_cast<size_t>(b) * a.num_splits + split) * a.hq + head;
      float* out = static_cast<float*>(a.out) + row * kHeadDim + d0;
      *reinterpret_cast<float4*>(out) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv,
                                                    acc[3] * inv);
      if (d0 == 0) a.lse[row] = lse;
    }
  }
  if (!clustered) return;

  // ---- on-chip merge of the cluster's splits (same log-sum-exp combine as the merge kernel):
  // every push has landed after one cluster barrier, and each rank then reads only its own
  // shared memory, so no rank waits for the others before it exits
  cluster_sync();
  cluster_combine(recv_u32, a.cluster, a.out, a.lse, a.hq, b, kvh, G);
}

}  // namespace

// How many clusters of 16 CTAs of `kern` can be resident at once on this device
// (16 is above the portable cluster size of 8); asked once per device and kernel,
// never while `stream` is being captured into a graph (the answer is then 0 for
// that launch, which runs with clusters of 8).  Host threads may race on the
// first call: the cache is filled under a mutex.
template <typename Kern>
int cluster16_capacity(Kern kern, int nt_index, cudaStream_t stream) {
  static int known[64][4] = {};  // 0 unknown, else 1 + the number of resident clusters
  static std::mutex known_mutex;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(known_mutex);
  int& k = known[dev][nt_index];
  if (k == 0) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return 0;
    k = 1;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16, 1, 1);
      cfg.blockDim = dim3(kWarps * 32, 1, 1);
      cfg.dynamicSmemBytes = decode_smem_bytes();
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 16;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) k = 1 + n;
    }
    cudaGetLastError();  // a refused query leaves no error behind
  }
  return k - 1;
}

cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeArgs& args,
                          const DecodeRopeArgs& rope, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes();
  auto kern = rope.table ? (args.group <= 8 ? sink_decode_kernel<1, true> : sink_decode_kernel<2, true>)
                         : (args.group <= 8 ? sink_decode_kernel<1, false> : sink_decode_kernel<2, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  DecodeArgs a = args;
  // clusters of 16 only while all of them can be resident at once (one per (sequence,
  // KV head)); beyond that, waiting clusters cost more than the larger split saves
  if (a.cluster > 8 &&
      static_cast<long long>(a.batch) * a.hkv >
          cluster16_capacity(kern, (args.group <= 8 ? 0 : 1) + (rope.table ? 2 : 0), stream))
    a.cluster = 8;
  const bool clustered = a.cluster > 1;
  const dim3 grid(clustered ? a.cluster : a.num_splits, a.hkv, a.batch);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // programmatic dependent launch: the grid may start while the previous kernel
  // on the stream finishes; the kernel waits for it before reading any input
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = clustered ? a.cluster : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = clustered ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, a, rope);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sa
