// Causal / ragged prefill with softmax sinks on tcgen05 tensor cores.
//
// Page "GPT-OSS on day 0", section "Kernels for GPT-OSS / Sink Attention":
// attn = softmax(q k^T * sm_scale + sink) V with the head's sink seeding the
// online softmax (running max m = sink, running denominator d = 1).  Each
// work item is one 128-token query block of a whole sequence, so the sink
// seeds its single KV walk.
//
// GB300 design: 12 warps, warp-specialised, one CTA per SM at a time.
//  * Schedule.  Work items are (sequence, 128-token query block, pair of
//    query heads of one KV group).  Every CTA sorts the (sequence, query
//    block) pairs by their number of KV tiles in shared memory (heaviest
//    first; all CTAs compute the same order) and deals the items out in
//    alternating (snake) order, so long rows of a ragged batch start first, the
//    CTAs end up with nearly equal work and no scratch memory is needed.  The
//    grid is persistent (one CTA per SM): a CTA loads the next item's Q while
//    the current item drains, which a fresh CTA per item cannot.  Only a
//    uniform contiguous batch (every sequence the same length) with no more
//    items than SMs launches one CTA per item, heaviest first, which skips the
//    sort.
//  * GQA packing (persistent schedule, group G = 4, 8 or 16).  A sequence with at most
//    2 * 128 / G new tokens (a decode row, a short chunk) would fill one row of
//    each 128-row tile per head; instead it becomes one item per KV head whose
//    two tiles hold 128 / G tokens x all G query heads of the group (row r:
//    token r / G, head r % G), which share the K/V tiles.  Q arrives through a
//    second tensor map with (64, G, 128 / G) boxes.  Items per pair then vary,
//    so the CTA keeps an exclusive prefix sum of the sorted pairs' item counts.
//  * warp 0 -- TMA producer: Q for two query heads (two 128x64 tiles,
//    double-buffered across items), then K and V tiles of 128 keys into a
//    4-stage ring shared by consecutive items (128-byte swizzle; contiguous
//    tensors by one 3-D box from lane 0, paged caches by eight 16-row page
//    boxes through the page table, one page per lane).
//  * warps 1 and 2, lane 0 -- one tcgen05 issuer per query tile t:
//    S_t = Q_t K^T (M=128, N=128, K=64) into TMEM and O_t += P_t V with P_t
//    read from TMEM (M=128, N=64, K=128); completion through tcgen05.commit.
//    Per KV tile the issuer puts PV(j-1) ahead of S(j+1).
//  * warps 4-7 and 8-11 -- one softmax warpgroup per query tile; thread r
//    owns row r (TMEM lane r): reads its 128 scores with the reducing TMEM load
//    (tcgen05.ld.red, sm_103a), which also returns each 32-column slice's max, so
//    a full tile's row max costs three max instructions; masks and takes the max
//    itself on diagonal and tail tiles only; updates the running max lazily
//    (O and d are rescaled only when the max grows by more than 2^8, which
//    leaves O/d unchanged), writes P as bf16
//    into TMEM and finally stores out = O/d and lse = m + ln d.
//  TMEM columns: S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384)
//                P0 [384,448) P1 [448,512).
#include <atomic>
#include <cstddef>

#include "internal.h"
#include "ptx.cuh"
#include "rope_math.cuh"

namespace sa {
namespace {

constexpr int kBlockQ = 128;
constexpr int kBlockK = 128;
constexpr int kStages = 4;
constexpr int kThreads = 384;
constexpr int kTileBytes = kBlockQ * kHeadDim * 2;  // 16 KiB
constexpr int kMaxPairs = 1024;                     // (sequence, query block) pairs sorted on chip
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384, kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct __align__(1024) PrefillSmem {
  uint8_t q0[2][kTileBytes];    // Q of even items [query tile]
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint64_t q_full[2];           // Q of the item landed                         (TMA tx)
  uint64_t q_ready[2][2];       // fused q: [buffer][tile] the tile's Q rows biased and rotated (128 arrivals)
  uint64_t q_empty[2];          // the item's Q buffers are free again: its MMAs are done and the
                                //   output staged there has been read by the TMA (1 arrival per tile)
  uint64_t kv_full[kStages];    // K_j and V_j landed                           (TMA tx)
  uint64_t kv_empty[kStages];   // every query tile's MMAs on the stage finished (1 commit per tile)
  uint64_t s_full[2];           // S_t(j) is in TMEM                             (tcgen05.commit)
  uint64_t s_free[2];           // softmax warpgroup t has read S_t(j)           (128 arrivals)
  uint64_t p_full[2];           // P_t(j) written and O_t rescaled               (128 arrivals)
  uint64_t pv_done[2];          // O_t += P_t(j) V_j completed                   (tcgen05.commit)
  uint64_t o_free[2];           // softmax warpgroup t has read O_t of its item  (128 arrivals)
  uint64_t drain[2];
  uint64_t stage_full[2];       // every row of tile t's output box is staged   (128 arrivals)
  int n_pairs;                  // pairs with work (a prefix of sortkey)
  int sorted;                   // 0 when the items are in reverse query-block order
  uint32_t tmem_base;
  int abort_flag;
  int issued_kv;                // producer bookkeeping for the drain
  int issued_q;
  // Only the persistent schedule uses what follows; a one-item-per-CTA launch
  // allocates shared memory up to here (a smaller carve-out leaves more L1).
  alignas(1024) uint8_t q1[2][kTileBytes];  // Q of odd items [query tile]
  unsigned long long sortkey[kMaxPairs];    // (KV tiles << 32) | packed << 31 | (2^31 - 1 - pair)
  int item_prefix[kMaxPairs + 1];           // items before sorted pair rank r
  int warp_sum[kThreads / 32];
};
constexpr size_t kSmemOnePerCta = offsetof(PrefillSmem, q1);

__device__ __forceinline__ uint8_t* q_tile(PrefillSmem& sm, int parity, int t) {
  return parity ? sm.q1[t] : sm.q0[t];
}

// Shared-memory matrix descriptor, 128-byte swizzle, 8-row atoms 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1024 >> 4) << 16;  // leading byte offset (unused for N <= 64 / K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset: next 8-row group
  d |= 1ull << 46;                               // descriptor version for tcgen05
  d |= 2ull << 61;                               // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A/B, fp32 D, M x N, optional MN-major B.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
constexpr uint32_t kIdescS = idesc_bf16(128, 128, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, true);

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                         volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      return false;
    }
  }
}

// TMA store of one box of the 3D tensor map `map` from this CTA's shared memory
// (128-byte swizzled rows), tracked by the issuing thread's bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(map),
               "r"(c0), "r"(c1), "r"(c2), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared memory of every committed store has been read (may be overwritten)
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
struct WorkItem {
  int b, h0, q0, q_start, q_len, kv_len, n_kv;
  int kvh;     // KV head of the item
  int packed;  // rows are (token r / G, head r % G) of a short sequence
};

struct Schedule {
  int n_qb, n_hg, tiles;
};

__device__ __forceinline__ Schedule make_schedule(const PrefillArgs& a) {
  Schedule s;
  s.tiles = (a.group % 2 == 0) ? 2 : 1;
  s.n_hg = a.hq / s.tiles;
  s.n_qb = (a.max_q + kBlockQ - 1) / kBlockQ;
  return s;
}

// Lengths of sequence b; false when they break the declared bounds.
__device__ __forceinline__ bool seq_lengths(const PrefillArgs& a, int b, int& qs, int& q_len,
                                            int& kv_len) {
  qs = a.cu_q[b];
  const int qe = a.cu_q[b + 1];
  q_len = qe - qs;
  kv_len = a.paged ? a.kv_lens[b] : q_len;
  const bool bad = qs < 0 || q_len < 0 || q_len > a.max_q || qe > a.total_q || kv_len < q_len ||
                   (a.paged && kv_len > a.max_pages * kPageSize);
  return !bad;
}

// KV tiles a query block visits (0 when the block is empty): the keys visible to
// its last row under bottom-right causal alignment, or all keys.
__device__ __forceinline__ int block_tiles(const PrefillArgs& a, int q0, int q_len, int kv_len) {
  if (q0 >= q_len) return 0;
  const int last_row = min(q0 + kBlockQ, q_len) - 1;
  const int kv_end = a.causal ? min(kv_len, last_row + kv_len - q_len + 1) : kv_len;
  return (kv_end + kBlockK - 1) / kBlockK;
}

// A sequence of q_len new tokens is packed (see the schedule notes) when the
// group has at least 4 query heads and divides the 128 tile rows (G = 4, 8, 16),
// and its tokens fit the two tiles of one item.
__device__ __forceinline__ bool packs(const PrefillArgs& a, int q_len) {
  return a.group >= 4 && kBlockQ % a.group == 0 && q_len <= 2 * (kBlockQ / a.group);
}

__device__ __forceinline__ unsigned long long pair_key(int tiles, bool packed, int pair) {
  return (static_cast<unsigned long long>(tiles) << 32) | (packed ? 0x80000000ull : 0ull) |
         static_cast<unsigned long long>(0x7fffffffu - static_cast<uint32_t>(pair));
}

// Work item k of the schedule.  n_kv == 0 marks an item with nothing to do
// (only possible in the unsorted fallback order).
__device__ __forceinline__ WorkItem item_at(const PrefillArgs& a, const PrefillSmem& sm,
                                            const Schedule& sc, int k) {
  int b, qb, slot;
  bool packed = false;
  if (sm.sorted) {
    // sorted pair rank: the last rank whose prefix is <= k
    int lo = 0, hi = sm.n_pairs;  // item_prefix[lo] <= k < item_prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sm.item_prefix[mid] <= k) lo = mid; else hi = mid;
    }
    const unsigned long long key = sm.sortkey[lo];
    const int pair = static_cast<int>(0x7fffffffu - static_cast<uint32_t>(key & 0x7fffffffu));
    packed = (key & 0x80000000ull) != 0;
    slot = k - sm.item_prefix[lo];
    b = pair / sc.n_qb;
    qb = pair % sc.n_qb;
  } else {  // reverse query-block order
    const int rank = k / sc.n_hg;
    slot = k % sc.n_hg;
    qb = sc.n_qb - 1 - rank / a.batch;
    b = rank % a.batch;
  }
  WorkItem w;
  w.b = b;
  w.packed = packed ? 1 : 0;
  w.kvh = packed ? slot : (slot * sc.tiles) / a.group;
  w.h0 = packed ? slot * a.group : slot * sc.tiles;
  w.q0 = qb * kBlockQ;
  int qs, q_len, kv_len;
  const bool good = seq_lengths(a, b, qs, q_len, kv_len);
  w.q_start = qs;
  w.q_len = q_len;
  w.kv_len = kv_len;
  w.n_kv = good ? block_tiles(a, w.q0, q_len, kv_len) : 0;
  return w;
}

// The r-th item of CTA c in "snake" order: rounds of gridDim.x items are
// dealt alternately left-to-right and right-to-left, which balances the sorted
// (heaviest first) list across CTAs.  Returns -1 past the end.
__device__ __forceinline__ int snake_item(int r, int n_items) {
  const int g = gridDim.x, c = blockIdx.x;
  const int base = r * g;
  if (base >= n_items) return -1;
  const int k = base + ((r & 1) ? g - 1 - c : c);
  return k < n_items ? k : -2;  // -2: this CTA sits out the last, partial round
}

// Exclusive prefix of the items per sorted pair (Hkv for a packed pair, n_hg otherwise):
// each thread sums up to ceil(n / 384) consecutive ranks, then a shuffle scan within the
// warp and a scan of the warp totals.  The thread's ranks are read twice instead of being
// kept in a per-thread array (which would live in local memory), and the scan is out of
// line: it runs once per CTA, and inlined it changed the step loop's code (about 1% on
// uniform batches).
__device__ __noinline__ void item_prefix_scan(PrefillSmem& sm, int hkv, int n_hg) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = sm.n_pairs;
  const int per = (n + kThreads - 1) / kThreads;  // <= 3
  const int r0 = threadIdx.x * per;
  auto count = [&](int r) { return r < n ? ((sm.sortkey[r] & 0x80000000ull) ? hkv : n_hg) : 0; };
  int sum = 0;
  for (int e = 0; e < per; ++e) sum += count(r0 + e);
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) sm.warp_sum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w2 = 0; w2 < warp; ++w2) base += sm.warp_sum[w2];
  int run = base + incl - sum;  // items before rank r0
  for (int e = 0; e < per; ++e) {  // second pass over the same keys
    if (r0 + e < n) sm.item_prefix[r0 + e] = run;
    run += count(r0 + e);
  }
  if (threadIdx.x == kThreads - 1) sm.item_prefix[n] = base + incl;
}

template <bool kPaged, bool kPersistent>
__global__ void __launch_bounds__(kThreads, 1)
    sink_prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                        const __grid_constant__ CUtensorMap qpmap,
                        const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap omap, const PrefillArgs a,
                        const PrefillRopeArgs rope) {
  extern __shared__ uint8_t smem_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Schedule sc = make_schedule(a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Launched with programmatic stream serialisation: this CTA may be resident
  // while the kernel before it on the stream finishes.  The tensor-map
  // descriptors are kernel parameters, so they are fetched now; every read of an
  // input comes after the wait.  Dependents may be scheduled at once: they wait
  // for this whole grid before reading anything, and they can only start when
  // every CTA of this grid has started.
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&qmap);
    if (kPersistent) tma_prefetch_desc(&qpmap);
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&omap);
  }
  pdl_launch_dependents();
  pdl_wait_primary();

  // ---------------------------------------------------------------- schedule
  const int pairs = a.batch * sc.n_qb;
  int n_items;
  if constexpr (kPersistent) {
    // Sort the (sequence, query block) pairs by KV tiles, heaviest first.
    // Every CTA computes the same order; a pair with no work sorts last (key 0).
    if (pairs <= kMaxPairs) {
      int cap = 1;
      while (cap < pairs) cap <<= 1;
      for (int p = threadIdx.x; p < cap; p += kThreads) {
        unsigned long long key = 0;
        if (p < pairs) {
          const int b = p / sc.n_qb, qb = p % sc.n_qb;
          int qs, q_len, kv_len;
          int tiles = 0;
          bool packed = false;
          if (seq_lengths(a, b, qs, q_len, kv_len)) {
            tiles = block_tiles(a, qb * kBlockQ, q_len, kv_len);
            packed = packs(a, q_len);
          } else if (qb == 0 && blockIdx.x == 0) {
            raise_status(a.status, kStatusBadLen);
          }
          key = tiles > 0 ? pair_key(tiles, packed, p) : 0ull;
        }
        sm.sortkey[p] = key;
      }
      __syncthreads();
      for (int size = 2; size <= cap; size <<= 1) {  // bitonic sort, descending
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int i = threadIdx.x; i < cap; i += kThreads) {
            const int jx = i ^ stride;
            if (jx > i) {
              const bool desc = (i & size) == 0;
              const unsigned long long x = sm.sortkey[i], y = sm.sortkey[jx];
              if (desc ? (x < y) : (x > y)) {
                sm.sortkey[i] = y;
                sm.sortkey[jx] = x;
              }
            }
          }
          __syncthreads();
        }
      }
      // pairs with work: the non-zero keys (they sort first), counted by the whole block
      int n = 0;
      for (int p0 = 0; p0 < pairs; p0 += kThreads) {
        const int p = p0 + static_cast<int>(threadIdx.x);
        n += __syncthreads_count(p < pairs && sm.sortkey[p] != 0ull);
      }
      if (threadIdx.x == 0) {
        sm.n_pairs = n;
        sm.sorted = 1;
      }
      __syncthreads();
      item_prefix_scan(sm, a.hkv, sc.n_hg);
    } else if (threadIdx.x == 0) {
      // too many pairs to sort on chip: reverse query-block order (empty items skipped)
      sm.n_pairs = pairs;
      sm.sorted = 0;
      if (blockIdx.x == 0)
        for (int b = 0; b < a.batch; ++b) {
          int qs, q_len, kv_len;
          if (!seq_lengths(a, b, qs, q_len, kv_len)) raise_status(a.status, kStatusBadLen);
        }
    }
    __syncthreads();
    n_items = sm.sorted ? sm.item_prefix[sm.n_pairs] : sm.n_pairs * sc.n_hg;
    if (static_cast<int>(blockIdx.x) >= n_items) return;  // uniform; before any barrier or TMEM use
  } else {
    // one item per CTA, reverse query-block order (heaviest first for causal blocks)
    if (threadIdx.x == 0) sm.sorted = 0;
    __syncthreads();
    n_items = pairs * sc.n_hg;
  }
  // the one item of a non-persistent CTA: leave at once when it has no work
  if constexpr (!kPersistent) {
    const WorkItem w0 = item_at(a, sm, sc, blockIdx.x);
    if (w0.n_kv == 0) {
      if (threadIdx.x == 0 && w0.q0 == 0 && w0.h0 == 0) {
        int qs, q_len, kv_len;
        if (!seq_lengths(a, w0.b, qs, q_len, kv_len)) raise_status(a.status, kStatusBadLen);
      }
      return;  // uniform across the CTA
    }
  }

  volatile int* abort_flag = &sm.abort_flag;
  const int ntiles = sc.tiles;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.q_full[i]), 1);
      mbar_init(smem_u32(&sm.q_ready[i][0]), 128);
      mbar_init(smem_u32(&sm.q_ready[i][1]), 128);
      mbar_init(smem_u32(&sm.q_empty[i]), ntiles);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.kv_full[s]), 1);
      mbar_init(smem_u32(&sm.kv_empty[s]), ntiles);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&sm.s_full[t]), 1);
      mbar_init(smem_u32(&sm.s_free[t]), 128);
      mbar_init(smem_u32(&sm.p_full[t]), 128);
      mbar_init(smem_u32(&sm.pv_done[t]), 1);
      mbar_init(smem_u32(&sm.o_free[t]), 128);
      mbar_init(smem_u32(&sm.drain[t]), 1);
      mbar_init(smem_u32(&sm.stage_full[t]), 128);
    }
    sm.abort_flag = 0;
    sm.issued_kv = 0;
    sm.issued_q = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The TMEM base is read from shared memory inside each role that needs it: kept in a
  // register across the register split, the one-item form spilled it.
  auto tmem_base = [&]() { return *reinterpret_cast<volatile const uint32_t*>(&sm.tmem_base); };

  // Runs `body(item, item_index_of_this_cta, first_global_kv_tile)` for every
  // item of this CTA: the single item of a non-persistent CTA, or the snake
  // sequence of the persistent schedule.  Stops when body returns false.
  auto for_items = [&](auto&& body) {
    if constexpr (!kPersistent) {
      // recomputed in each role rather than kept live across the register split
      body(item_at(a, sm, sc, blockIdx.x), 0, 0);
    } else {
      int it = 0, g = 0;
      for (int rr = 0;; ++rr) {
        const int k = snake_item(rr, n_items);
        if (k == -1) break;
        if (k < 0) continue;
        const WorkItem w = item_at(a, sm, sc, k);
        if (w.n_kv == 0) continue;
        if (!body(w, it, g)) break;
        ++it;
        g += w.n_kv;
      }
    }
  };

  // Producer / MMA warpgroup needs few registers; the softmax warpgroups hold a
  // whole 128-wide score row each.  128*56 + 256*224 = 384*168 (launch total).
  // Each setmaxnreg sits inside its own role branch so the compiler can give
  // every region its own budget.
  if (warp < 4) {
    regs_dec<56>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      // The whole warp walks the items in step; lane 0 waits on barriers (and
      // shares the outcome), arms them and loads Q.  A paged K/V tile is eight
      // 16-row page boxes: lane i < 8 holds the page id of box i (one coalesced
      // load, a tile ahead) and issues that page's K and V copies.
      if (lane == 0) {
        tma_prefetch_desc(&qmap);
        if (kPersistent) tma_prefetch_desc(&qpmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
      }
      const uint64_t keep = l2_policy_evict_last();  // K/V are re-read by the group's other heads
      const uint64_t once = l2_policy_evict_first();
      auto warp_wait = [&](uint32_t bar, uint32_t parity) {
        int r = 1;
        if (lane == 0) r = wait_bar(bar, parity, a.timeout_ns, abort_flag) ? 1 : 0;
        return __shfl_sync(0xffffffffu, r, 0) != 0;
      };
      bool ok = true;
      for_items([&](const WorkItem& w, int it, int g) {
        const int kvh = w.kvh;
        const int qb = it & 1;
        if (it >= 2 && !warp_wait(smem_u32(&sm.q_empty[qb]), ((it >> 1) - 1) & 1)) return ok = false;
        if (lane == 0) {
          const uint32_t qbar = smem_u32(&sm.q_full[qb]);
          mbar_arrive_expect_tx(qbar, ntiles * kTileBytes);
          for (int t = 0; t < ntiles; ++t) {
            if (kPersistent && w.packed)  // 128 / G tokens x the G heads of the group
              tma_load_3d(smem_u32(q_tile(sm, qb, t)), &qpmap, 0, w.h0, w.q_start + t * (kBlockQ / a.group),
                          qbar, once);
            else
              tma_load_3d(smem_u32(q_tile(sm, qb, t)), &qmap, 0, w.h0 + t, w.q_start + w.q0, qbar, once);
          }
          sm.issued_q = it + 1;
        }
        const int32_t* ptab = kPaged ? a.page_table + static_cast<size_t>(w.b) * a.max_pages : nullptr;
        const int seq_pages = (w.kv_len + kPageSize - 1) / kPageSize;
        constexpr int kPagesPerTile = kBlockK / kPageSize;
        auto load_id = [&](int j) {  // page id of box `lane` of tile j (lanes < 8)
          if (lane >= kPagesPerTile) return 0;
          const int lp = min(j * kPagesPerTile + lane, seq_pages - 1);  // ragged tail: any valid page
          return ptab[lp];
        };
        int id = 0;
        if constexpr (kPaged) id = load_id(0);
        for (int j = 0; j < w.n_kv; ++j) {
          const int gg = g + j, st = gg % kStages;
          int next = 0;
          if constexpr (kPaged) {
            if (j + 1 < w.n_kv) next = load_id(j + 1);  // in flight while tile j is issued
          }
          if (gg >= kStages && !warp_wait(smem_u32(&sm.kv_empty[st]), ((gg / kStages) - 1) & 1))
            return ok = false;
          const uint32_t bar = smem_u32(&sm.kv_full[st]);
          if (lane == 0) mbar_arrive_expect_tx(bar, 2 * kTileBytes);
          if constexpr (kPaged) {
            if (lane < kPagesPerTile) {
              int phys = id;
              if (phys < 0 || phys >= a.num_pages) {
                raise_status(a.status, kStatusBadPage);
                phys = 0;
              }
              const int row = (phys * a.hkv + kvh) * kPageSize;
              tma_load_2d(smem_u32(sm.k[st]) + lane * kPageSize * 128, &kmap, 0, row, bar, keep);
              tma_load_2d(smem_u32(sm.v[st]) + lane * kPageSize * 128, &vmap, 0, row, bar, keep);
            }
            id = next;
          } else if (lane == 0) {
            tma_load_3d(smem_u32(sm.k[st]), &kmap, 0, kvh, w.q_start + j * kBlockK, bar, keep);
            tma_load_3d(smem_u32(sm.v[st]), &vmap, 0, kvh, w.q_start + j * kBlockK, bar, keep);
          }
          if (lane == 0) sm.issued_kv = gg + 1;
        }
        return true;
      });
      if (!ok && lane == 0) raise_status(a.status, kStatusTimeout);
    } else if (warp == 1 || warp == 2) {
      // ---------------------------------------------------------- MMA issuers
      // Warp 1 issues query tile 0's MMAs, warp 2 tile 1's: the two tiles run
      // as independent pipelines that only share Q buffers and K/V stages.
      const int t = warp - 1;
      if (lane == 0 && t < ntiles) {
        bool ok = true;
        const uint32_t tmem = tmem_base();
        const uint32_t d_s = tmem + kColS + t * 128, d_o = tmem + kColO + t * 64;
        const uint32_t a_p = tmem + kColP + t * 64;
        for_items([&](const WorkItem& w, int it, int g) {
          const int qb = it & 1;
          // fused q: the rows are ready once the softmax threads have biased and rotated them
          ok = wait_bar(smem_u32(rope.table ? &sm.q_ready[qb][t] : &sm.q_full[qb]), (it >> 1) & 1,
                        a.timeout_ns, abort_flag);
          if (!ok) return false;
          const uint32_t q_addr = smem_u32(q_tile(sm, qb, t));
          auto s_step = [&](int jj) {  // S_t(jj) = Q_t K_jj^T
            const int gg = g + jj;
            ok = wait_bar(smem_u32(&sm.kv_full[gg % kStages]), (gg / kStages) & 1, a.timeout_ns,
                          abort_flag);
            if (!ok) return;
            tc_fence_after();
            const uint32_t k_addr = smem_u32(sm.k[gg % kStages]);
#pragma unroll
            for (int kk = 0; kk < kHeadDim / 16; ++kk)
              tc_mma_ss(d_s, sw128_desc(q_addr + kk * 32), sw128_desc(k_addr + kk * 32), kIdescS, kk > 0);
            tc_commit(smem_u32(&sm.s_full[t]));
          };
          auto pv_step = [&](int jj) {  // O_t += P_t(jj) V_jj
            const int gg = g + jj;
            if (jj == 0 && it > 0)  // O_t still holds the previous item until its epilogue read it
              ok = wait_bar(smem_u32(&sm.o_free[t]), (it - 1) & 1, a.timeout_ns, abort_flag);
            if (ok) ok = wait_bar(smem_u32(&sm.p_full[t]), gg & 1, a.timeout_ns, abort_flag);
            if (!ok) return;
            tc_fence_after();
            const uint32_t v_addr = smem_u32(sm.v[gg % kStages]);
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk)
              tc_mma_ts(d_o, a_p + kk * 8, sw128_desc(v_addr + kk * 16 * 128), kIdescPV,
                        (jj > 0 || kk > 0) ? 1u : 0u);
            tc_commit(smem_u32(&sm.pv_done[t]));
            tc_commit(smem_u32(&sm.kv_empty[gg % kStages]));
          };
          // The very first tile of tile 1 starts one softmax phase behind tile 0,
          // so one warpgroup runs exp2 while the other loads and stores.  A parity wait on
          // p_full[0] is only sound if it begins before tile 0 completes its second step
          // (parity 0 again).  With q as given both issuers pass the same q_full wait and
          // tile 1's comes straight here, so it does.  With fused q, tile 1's rows are
          // released after tile 0's have been rotated and then its own, which already puts
          // it a phase behind, and the wait could begin too late: it is skipped there.
          if (it == 0 && t == 1 && !rope.table)
            ok = wait_bar(smem_u32(&sm.p_full[0]), 0, a.timeout_ns, abort_flag);
          if (ok) s_step(0);
          // Step j: PV_t(j-1) (P_t(j-1) is ready before softmax(j) starts), then
          // S_t(j+1) once softmax t has read S_t(j).
          for (int j = 0; j < w.n_kv && ok; ++j) {
            if (j >= 1) pv_step(j - 1);
            if (ok && j + 1 < w.n_kv) {
              ok = wait_bar(smem_u32(&sm.s_free[t]), (g + j) & 1, a.timeout_ns, abort_flag);
              if (ok) s_step(j + 1);
            }
          }
          if (ok) pv_step(w.n_kv - 1);
          // Q_t of the item is released by the softmax warpgroup once its epilogue is done
          // with the buffer (it stages the output there)
          return ok;
        });
        if (!ok) raise_status(a.status, kStatusTimeout);
        // whatever happened, wait for every MMA this thread issued before TMEM is released
        tc_commit(smem_u32(&sm.drain[t]));
        mbar_wait(smem_u32(&sm.drain[t]), 0, 2000000000ull);
      }
    }
  } else {
    regs_inc<224>();
    // ------------------------------------------------------------ softmax + epilogue
    const int t = (warp - 4) >> 2;      // query tile of this warpgroup
    const int qw = warp & 3;            // TMEM lane quarter
    const int r = qw * 32 + lane;       // row within the block
    if (t < ntiles) {
      const uint32_t lane_base = tmem_base() + (static_cast<uint32_t>(qw * 32) << 16);
      const uint32_t s_col = lane_base + kColS + t * 128;
      const uint32_t o_col = lane_base + kColO + t * 64;
      const uint32_t p_col = lane_base + kColP + t * 64;
      const uint64_t scale2 = f2(a.scale_log2, a.scale_log2);
      bool ok = true;
      int n_staged = 0;  // output boxes this warpgroup has staged (stage_full phase)
      for_items([&](const WorkItem& w, int it, int g) {
        // head and query index (within the sequence) of TMEM lane r
        const int h = w.packed ? w.h0 + r % a.group : w.h0 + t;
        const int i = w.packed ? t * (kBlockQ / a.group) + r / a.group : w.q0 + r;
        const int limit = a.causal ? min(i + w.kv_len - w.q_len, w.kv_len - 1) : w.kv_len - 1;
        if (rope.table) {
          // Fused q: this thread's query row is the projection output as loaded; add the
          // head's bias, rotate each feature pair (i, i + 32) by the token's (cos, sin) row of
          // the table and round back to bf16 in place, before the tile's first S MMA (the
          // arithmetic of the kernel that writes rotated q).  The table row and the bias are
          // requested before the wait for Q, so they arrive while the Q copy lands.
          const int qb = it & 1;
          const bool live = i < w.q_len;
          float4 cs[16];
          uint4 bias[8];
          const uint4* brow = reinterpret_cast<const uint4*>(rope.q_bias + h * kHeadDim);
#pragma unroll
          for (int e = 0; e < 8; ++e) bias[e] = (live && rope.q_bias) ? __ldg(brow + e) : make_uint4(0, 0, 0, 0);
          const float4* crow = reinterpret_cast<const float4*>(
              rope.table + (static_cast<long long>(w.q_start) + (live ? i : 0)) * (kHeadDim / 2));
#pragma unroll
          for (int e = 0; e < 16; ++e) cs[e] = live ? __ldg(crow + e) : make_float4(0.f, 0.f, 0.f, 0.f);
          if (!wait_bar(smem_u32(&sm.q_full[qb]), (it >> 1) & 1, a.timeout_ns, abort_flag)) return ok = false;
          // tile 1 waits for tile 0's rows, so tile 0 (whose first S MMA comes first) is not
          // slowed by tile 1's transform; tile 1 starts a softmax phase later anyway
          if (t == 1 && !wait_bar(smem_u32(&sm.q_ready[qb][0]), (it >> 1) & 1, a.timeout_ns, abort_flag))
            return ok = false;
          if (live) {
            uint8_t* row = q_tile(sm, qb, t) + r * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // features [8j, 8j + 8) and their partners [8j + 32, 8j + 40)
              uint4* p1 = reinterpret_cast<uint4*>(row + ((j ^ (r & 7)) << 4));
              uint4* p2 = reinterpret_cast<uint4*>(row + (((j + 4) ^ (r & 7)) << 4));
              float y1[8], y2[8];
              widen8(*p1, y1);
              widen8(*p2, y2);
              if (rope.q_bias) {
                add_bias8(y1, bias[j]);
                add_bias8(y2, bias[j + 4]);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) rotate2(y1, y2, e, cs[4 * j + e]);
              *p1 = pack8(y1);
              *p2 = pack8(y2);
            }
          }
          fence_proxy_async_smem();  // the rows are read by the tensor core (async proxy)
          mbar_arrive(smem_u32(&sm.q_ready[qb][t]));
        }
        const float sink = a.sinks[h] * kLog2e;
        float m = sink;                                 // running max (log2 units)
        float d = (sink == kNegInf) ? 0.0f : 1.0f;      // running denominator
        for (int j = 0; j < w.n_kv; ++j) {
          const int gg = g + j;
          if (!wait_bar(smem_u32(&sm.s_full[t]), gg & 1, a.timeout_ns, abort_flag)) return ok = false;
          tc_fence_after();
          // S_t row r with the maxima of its four 32-column slices (reducing loads)
          uint32_t sr[128];
          float pm0, pm1, pm2, pm3;
          tmem_ld32_max_at<0>(s_col + 0, sr, pm0);
          tmem_ld32_max_at<32>(s_col + 32, sr, pm1);
          tmem_ld32_max_at<64>(s_col + 64, sr, pm2);
          tmem_ld32_max_at<96>(s_col + 96, sr, pm3);
          tc_wait_ld();
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.s_free[t]));  // the MMA may now overwrite S_t
          float s[128];
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
          // Row max over the visible keys: on a full tile, the loads' own maxima; on a
          // diagonal or tail tile the masked scores are dropped first, then four independent
          // 3-input max chains take the max of what is left.
          const int key0 = j * kBlockK;
          float mraw = fmax3(pm0, pm1, fmaxf(pm2, pm3));
          if (key0 + kBlockK - 1 > limit) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (key0 + c > limit) s[c] = kNegInf;
            float m0 = s[0], m1 = s[1], m2 = s[2], m3 = s[3];
#pragma unroll
            for (int c = 4; c < 124; c += 8) {
              m0 = fmax3(m0, s[c], s[c + 1]);
              m1 = fmax3(m1, s[c + 2], s[c + 3]);
              m2 = fmax3(m2, s[c + 4], s[c + 5]);
              m3 = fmax3(m3, s[c + 6], s[c + 7]);
            }
            m0 = fmax3(m0, s[124], s[125]);
            m1 = fmax3(m1, s[126], s[127]);
            mraw = fmax3(m0, m1, fmaxf(m2, m3));
          }
          const float mx = mraw * a.scale_log2;
          const bool grow = mx > m + kRescaleThreshold;
          float factor = 1.0f;
          if (grow) {
            factor = (m == kNegInf) ? 0.0f : ex2(m - mx);
            m = mx;
            d *= factor;
          }
          const float mu = (m == kNegInf) ? 0.0f : m;
          const uint64_t negm2 = f2(-mu, -mu);
          // p = 2^(s * scale - m), packed two per instruction; four partial row sums
          uint32_t pk[64];
          uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            float x0, x1;
            f2_split(f2_fma(f2(s[2 * c], s[2 * c + 1]), scale2, negm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            const uint64_t pp = f2(p0, p1);
            if ((c & 3) == 0) acc0 = f2_add(acc0, pp);
            if ((c & 3) == 1) acc1 = f2_add(acc1, pp);
            if ((c & 3) == 2) acc2 = f2_add(acc2, pp);
            if ((c & 3) == 3) acc3 = f2_add(acc3, pp);
            pk[c] = pack_bf16x2(p0, p1);
          }
          float r0, r1;
          f2_split(f2_add(f2_add(acc0, acc1), f2_add(acc2, acc3)), r0, r1);
          d += r0 + r1;
          // P_t and O_t are still in use by the previous PV until it completes
          if (j > 0 && !wait_bar(smem_u32(&sm.pv_done[t]), (gg - 1) & 1, a.timeout_ns, abort_flag))
            return ok = false;
          tc_fence_after();
          if (j > 0 && __any_sync(0xffffffffu, grow)) {  // O holds earlier tiles: rescale it
            const uint64_t f22 = f2(factor, factor);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t u[32];
              tmem_ld32(o_col + c * 32, u);
              tc_wait_ld();
              uint32_t lo[16], hi[16];
#pragma unroll
              for (int e = 0; e < 16; e += 2) {
                float a0, a1;
                f2_split(f2_mul(f2(__uint_as_float(u[e]), __uint_as_float(u[e + 1])), f22), a0, a1);
                lo[e] = __float_as_uint(a0);
                lo[e + 1] = __float_as_uint(a1);
                f2_split(f2_mul(f2(__uint_as_float(u[16 + e]), __uint_as_float(u[17 + e])), f22), a0, a1);
                hi[e] = __float_as_uint(a0);
                hi[e + 1] = __float_as_uint(a1);
              }
              tmem_st16(o_col + c * 32, lo);
              tmem_st16(o_col + c * 32 + 16, hi);
            }
          }
          tmem_st16_at<0>(p_col + 0, pk);
          tmem_st16_at<16>(p_col + 16, pk);
          tmem_st16_at<32>(p_col + 32, pk);
          tmem_st16_at<48>(p_col + 48, pk);
          tc_wait_st();
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.p_full[t]));
        }
        if (!wait_bar(smem_u32(&sm.pv_done[t]), (g + w.n_kv - 1) & 1, a.timeout_ns, abort_flag))
          return ok = false;
        // ---- epilogue: out = O / d (bf16), lse = m + ln d; then O_t is free again
        tc_fence_after();
        const bool row_ok = i < w.q_len;
        const float inv = d > 0.0f ? 1.0f / d : 0.0f;
        uint32_t ou[2][32];
        tmem_ld32(o_col, ou[0]);
        tmem_ld32(o_col + 32, ou[1]);
        tc_wait_ld();
        if (kPersistent) {
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.o_free[t]));  // the next item's first PV may overwrite O_t
        }
        auto chunk = [&](int c) {  // output columns [8c, 8c + 8) of this row as bf16
          const uint32_t* u = ou[c >> 2] + 8 * (c & 3);
          return make_uint4(pack_bf16x2(__uint_as_float(u[0]) * inv, __uint_as_float(u[1]) * inv),
                            pack_bf16x2(__uint_as_float(u[2]) * inv, __uint_as_float(u[3]) * inv),
                            pack_bf16x2(__uint_as_float(u[4]) * inv, __uint_as_float(u[5]) * inv),
                            pack_bf16x2(__uint_as_float(u[6]) * inv, __uint_as_float(u[7]) * inv));
        };
        // In the persistent kernel a full query block of one head leaves through a TMA store:
        // the rows are staged in this item's Q_t buffer (every MMA that read it has completed)
        // with the 128-byte swizzle of the output map, then one thread stores the 128 x 64 box
        // while the warpgroup moves on to the next item.  Row by row the output of one head is
        // 8 KB apart, so direct stores touch 32 lines per warp instruction and hold up the
        // next item's softmax.  Partial and packed blocks, whose boxes would reach other rows,
        // store directly, and so does the one-item CTA, whose posted stores retire while the
        // next CTA starts (staging would keep it resident until the copy has read the tile).
        const bool staged = kPersistent && !w.packed && w.q0 + kBlockQ <= w.q_len;  // warpgroup-uniform
        if (staged) {
          uint8_t* stage = q_tile(sm, it & 1, t) + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(stage + ((c ^ (r & 7)) << 4)) = chunk(c);
          fence_proxy_async_smem();  // visible to the TMA (async proxy)
          mbar_arrive(smem_u32(&sm.stage_full[t]));
          if (qw == 0 && lane == 0) {  // bounded wait for the warpgroup's 128 rows
            if (!wait_bar(smem_u32(&sm.stage_full[t]), n_staged & 1, a.timeout_ns, abort_flag)) return ok = false;
            tma_store_3d(&omap, smem_u32(q_tile(sm, it & 1, t)), 0, h, w.q_start + w.q0);
            bulk_commit();
            bulk_wait_read();  // the buffer may be reused (or released) once the TMA has read it;
                               // the writes themselves complete by the end of the grid
          }
          ++n_staged;
        } else if (row_ok) {
          uint16_t* out = static_cast<uint16_t*>(a.out) +
                          (static_cast<size_t>(w.q_start + i) * a.hq + h) * kHeadDim;
#pragma unroll
          for (int c = 0; c < 8; ++c) reinterpret_cast<uint4*>(out)[c] = chunk(c);
        }
        if (row_ok && a.lse)
          a.lse[static_cast<size_t>(w.q_start + i) * a.hq + h] = d > 0.0f ? (m + lg2(d)) * kLn2 : kNegInf;
        if (kPersistent && qw == 0 && lane == 0) mbar_arrive(smem_u32(&sm.q_empty[it & 1]));
        return true;
      });
      if (!ok) raise_status(a.status, kStatusTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag && warp == 0 && lane == 0) {
    // some role gave up: copies it never consumed may still be in flight; let
    // the last tile of every stage and the last Q loads land before shared
    // memory is released
    const int issued = sm.issued_kv, issued_q = sm.issued_q;
    for (int gg = max(0, issued - kStages); gg < issued; ++gg)
      mbar_wait(smem_u32(&sm.kv_full[gg % kStages]), (gg / kStages) & 1, 2000000000ull);
    for (int it = max(0, issued_q - 2); it < issued_q; ++it)
      mbar_wait(smem_u32(&sm.q_full[it & 1]), (it >> 1) & 1, 2000000000ull);
  }
  if (warp == 1) tmem_dealloc(tmem_base(), kTmemCols);
}

std::atomic<int> g_prefill_sms[64];  // SM count per device, 0 until asked (host threads may race)

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& qmap, const CUtensorMap& qpmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, const CUtensorMap& omap, const PrefillArgs& a,
                           const PrefillRopeArgs& rope, cudaStream_t stream) {
  const int tiles = (a.group % 2 == 0) ? 2 : 1;
  const int n_qb = (a.max_q + kBlockQ - 1) / kBlockQ;
  const long long items = static_cast<long long>(n_qb) * (a.hq / tiles) * a.batch;
  if (items <= 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = g_prefill_sms[dev].load(std::memory_order_relaxed);
  if (!sms) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (sms <= 0) sms = 1;
    g_prefill_sms[dev].store(sms, std::memory_order_relaxed);
  }
  // Contiguous KV with every sequence at max_q tokens (their sum is then
  // batch * max_q) and one wave of items at most: one CTA per item in
  // heaviest-first order, no sort.  Otherwise a persistent grid with the sorted
  // schedule, which overlaps each item's Q load with the previous item's tail
  // (4 x 8192 causal: 1057 against 1029 TFLOP/s as one CTA per item).
  const bool uniform = !a.paged && static_cast<long long>(a.total_q) == static_cast<long long>(a.batch) * a.max_q;
  const bool persistent = !uniform || items > sms;
  const int blocks = static_cast<int>(persistent ? (items < sms ? items : sms) : items);
  const size_t smem = (persistent ? sizeof(PrefillSmem) : kSmemOnePerCta) + 1024;
  auto kern = a.paged ? (persistent ? sink_prefill_kernel<true, true> : sink_prefill_kernel<true, false>)
                      : (persistent ? sink_prefill_kernel<false, true> : sink_prefill_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, qmap, qpmap, kmap, vmap, omap, a, rope);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sa
