// Linear layer with bias, out = x W^T + b, on the 5th-generation tensor cores
// (page "GPT-OSS on day 0": the output projection and the experts carry bias
// terms; section "Kernels for GPT-OSS / MoE": bias support was added to the
// expert GEMMs by starting the accumulator registers from the bias values, a
// one-time step per output (MN) tile).
//
// The Blackwell form of that idea: the accumulator lives in tensor memory, so
// the epilogue warps write the bias row into the TMEM accumulator of the next
// tile (tcgen05.st) and every MMA of the tile accumulates onto it; there is no
// zero-initialising first MMA and no bias add in the epilogue.
//
// Persistent kernel, one CTA per SM; an output tile is MT x 128 rows by BN
// columns (MT = 1 or 2 sub-tiles of 128 rows), 128 + 128 MT threads:
//   warp 0        TMA producer: MT A boxes (x, 128 x 64 each) and one B box
//                 (W, BN x 64), 128-byte swizzle, into a kStages-deep ring
//   warp 1        TMEM owner and MMA issuer (one elected thread): per 64-wide
//                 K step and sub-tile four tcgen05.mma M=128 N=BN K=16,
//                 accumulate always on; the MT sub-tiles read the same B stage
//   warps 4..     epilogue, four warps per sub-tile: warp w reads TMEM lanes
//                 [32 (w % 4), +32) of its sub-tile's accumulator (one output
//                 row per thread), converts to bf16, stores, then seeds the
//                 buffer with the bias of the tile that will use it next
// Two TMEM accumulators (each MT sub-tiles) alternate, so the epilogue of tile
// i overlaps the MMAs of tile i + 1.  Tiles are numbered with the N index
// fastest: the CTAs working at the same time share one row block of x through
// L2.  MT = 2 serves skinny outputs (one column tile, N <= 128: the router
// projection): the layer streams x once while every row block re-reads all of
// W, so two sub-tiles per W stage halve the W bytes per x byte and leave more
// of the ring to x.
//
// Router form (SLOTS > 0): the MoE router projection (N = experts <= 256, one
// column tile) whose epilogue takes the page's Top-K-then-softmax router
// instead of storing logits: the thread that owns a token row rounds each
// logit to bf16, ranks it in a sorted register list of SLOTS packed keys (4
// for top_k <= 4, else 8; bf16 order in the high half, 0xFFFF - expert in the
// low half, so equal logits keep the lower expert first), and writes the K
// selected experts, their softmax weights (fp32, stored as bf16) and
// per-expert counts (shared histogram, added to the global counts once per
// CTA).  With four slots each group of eight keys is sorted as two quads (five
// compare-exchanges each), reduced to its top four by a bitonic merge and
// merged into the list the same way, instead of eight insertions (the epilogue
// runs after the CTA's last MMA, so its instruction count is exposed).  The
// arithmetic is that of the plain layer followed by the standalone router, bit
// for bit.
#include <atomic>
#include <cstdint>

#include "linear_args.h"
#include "ptx.cuh"

namespace sa {
namespace {

constexpr int kBM = 128;  // rows of one sub-tile (one tcgen05.mma M)
constexpr int kBK = 64;
constexpr int kEpiWarp0 = 4;
// Drains (MMAs before TMEM is freed, copies before shared memory is released)
// always wait up to this long, even when the caller set a shorter wait budget.
constexpr unsigned long long kDrainTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint64_t sw128_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1024 >> 4) << 16;  // leading byte offset (unused, K-major SW128)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;  // stride byte offset: next 8-row group
  d |= 1ull << 46;                               // tcgen05 descriptor version
  d |= 2ull << 61;                               // 128-byte swizzle
  return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16_kk(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

template <int BN, int MT>
struct LinCfg {
  static_assert(MT == 1 || (MT == 2 && BN <= 128), "two sub-tiles need BN <= 128 (TMEM)");
  static constexpr int kThreads = 128 + 128 * MT;  // 4 control warps + 4 epilogue warps per sub-tile
  static constexpr int kSubABytes = kBM * kBK * 2;
  static constexpr int kABytes = MT * kSubABytes;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (200 * 1024) / kStageBytes > 6 ? 6 : (200 * 1024) / kStageBytes;
  static constexpr int kAccStride = BN <= 128 ? 128 : 256;  // TMEM columns between sub-tile accumulators
  static constexpr int kTmemCols = 2 * MT * kAccStride;     // two buffers of MT sub-tiles
  static_assert(kTmemCols <= 512, "TMEM holds 512 columns");
  static constexpr size_t kSmem = 1024 /*alignment slack*/ + static_cast<size_t>(kStages) * kStageBytes + 2048;
};

struct LinBarriers {
  uint64_t full[8], empty[8], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort_flag;
  int issued;
  int hist[256];  // router form: expert counts of this CTA
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                              volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t order16(uint32_t bits) {  // bf16 bits -> unsigned order
  if (bits == 0x8000u) bits = 0;                               // -0 == +0
  return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  const uint32_t o = key >> 16;
  const uint32_t bits = (o & 0x8000u) ? (o & 0x7FFFu) : (~o & 0xFFFFu);
  return __uint_as_float(bits << 16);
}

// Compare-exchange: afterwards a >= b.
__device__ __forceinline__ void cmpx(uint32_t& a, uint32_t& b) {
  const uint32_t hi = max(a, b);
  b = min(a, b);
  a = hi;
}

// Four keys sorted largest first (five compare-exchanges).
__device__ __forceinline__ void sort4(uint32_t (&x)[4]) {
  cmpx(x[0], x[1]);
  cmpx(x[2], x[3]);
  cmpx(x[0], x[2]);
  cmpx(x[1], x[3]);
  cmpx(x[1], x[2]);
}

// a <- the four largest of a and b, both sorted largest first: max(a[i], b[3 - i]) holds
// those four as a bitonic sequence, which two rounds of compare-exchanges sort.
__device__ __forceinline__ void merge4(uint32_t (&a)[4], const uint32_t (&b)[4]) {
  uint32_t c[4] = {max(a[0], b[3]), max(a[1], b[2]), max(a[2], b[1]), max(a[3], b[0])};
  cmpx(c[0], c[2]);
  cmpx(c[1], c[3]);
  cmpx(c[0], c[1]);
  cmpx(c[2], c[3]);
#pragma unroll
  for (int r = 0; r < 4; ++r) a[r] = c[r];
}

// Router form: S slots hold the S largest keys (S = 4 serves top_k <= 4, 8 up to 8).
template <int S>
__device__ __forceinline__ void offer(uint32_t (&best)[S], uint32_t key) {
#pragma unroll
  for (int r = 0; r < S; ++r) {  // best[] stays sorted, largest first
    const uint32_t hi = max(best[r], key);
    key = min(best[r], key);
    best[r] = hi;
  }
}

// Write bias[n0 + c] (c < BN, zero past N) into every lane of the accumulator
// columns [col, col + BN) owned by this warp's TMEM lane quarter.
template <int BN>
__device__ __forceinline__ void seed_bias(uint32_t taddr, const uint16_t* bias, int n0, int N) {
#pragma unroll 1
  for (int c = 0; c < BN; c += 16) {
    uint32_t r[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int n = n0 + c + i;
      const uint32_t bits = (bias != nullptr && n < N) ? static_cast<uint32_t>(__ldg(bias + n)) : 0u;
      r[i] = bits << 16;  // bf16 -> fp32 bit pattern
    }
    tmem_st16(taddr + c, r);
  }
}

// SLOTS = 0: plain layer (bf16 output); SLOTS = 4 or 8: router form keeping that
// many candidates per token row.
template <int BN, int MT, int SLOTS>
__global__ void __launch_bounds__(LinCfg<BN, MT>::kThreads, 1)
linear_bias_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                   const LinearArgs a) {
  using C = LinCfg<BN, MT>;
  constexpr bool kRouter = SLOTS > 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  LinBarriers& sb = *reinterpret_cast<LinBarriers*>(tiles + static_cast<size_t>(C::kStages) * C::kStageBytes);
  volatile int* abort_flag = &sb.abort_flag;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_total = a.tiles_m * a.tiles_n;
  constexpr uint32_t kIdesc = idesc_bf16_kk(kBM, BN);
  const int k_steps = (a.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&sb.full[s]), 1);
      mbar_init(smem_u32(&sb.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sb.acc_full[b]), 1);
      mbar_init(smem_u32(&sb.acc_empty[b]), 4 * MT);  // lane 0 of every epilogue warp
    }
    mbar_init(smem_u32(&sb.drain), 1);
    sb.abort_flag = 0;
    sb.issued = 0;
    fence_barrier_init();
  }
  if constexpr (kRouter)
    for (int e = threadIdx.x; e < 256; e += C::kThreads) sb.hist[e] = 0;
  if (warp == 1) {
    tmem_alloc(smem_u32(&sb.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sb.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&amap);
      tma_prefetch_desc(&bmap);
      const uint64_t pol_a = l2_policy_evict_first();  // x: read by the tiles_n CTAs of one row block
      const uint64_t pol_b = l2_policy_evict_last();   // W: re-read by every row block
      int g = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles_total && ok; t += gridDim.x) {
        const int m0 = (t / a.tiles_n) * (kBM * MT);
        const int n0 = (t % a.tiles_n) * BN;
        for (int kb = 0; kb < k_steps; ++kb, ++g) {
          const int s = g % C::kStages;
          if (g >= C::kStages &&
              !wait_or_abort(smem_u32(&sb.empty[s]), ((g / C::kStages) - 1) & 1, a.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t bar = smem_u32(&sb.full[s]);
          const uint32_t dst = smem_u32(tiles + static_cast<size_t>(s) * C::kStageBytes);
          mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
          for (int sub = 0; sub < MT; ++sub)  // rows past M are zero-filled
            tma_load_2d(dst + sub * C::kSubABytes, &amap, kb * kBK, m0 + sub * kBM, bar, pol_a);
          tma_load_2d(dst + C::kABytes, &bmap, kb * kBK, n0, bar, pol_b);
          sb.issued = g + 1;
        }
      }
      if (!ok) raise_status(a.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int g = 0, i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles_total && ok; t += gridDim.x, ++i) {
        const int b = i & 1;
        ok = wait_or_abort(smem_u32(&sb.acc_empty[b]), (i >> 1) & 1, a.timeout_ns, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + b * MT * C::kAccStride;
        for (int kb = 0; kb < k_steps; ++kb, ++g) {
          const int s = g % C::kStages;
          ok = wait_or_abort(smem_u32(&sb.full[s]), (g / C::kStages) & 1, a.timeout_ns, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + static_cast<size_t>(s) * C::kStageBytes);
          const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
            for (int sub = 0; sub < MT; ++sub)
              tc_mma_ss(d + sub * C::kAccStride, sw128_kmajor(a_addr + sub * C::kSubABytes + kk * 32),
                        sw128_kmajor(b_addr + kk * 32), kIdesc, 1u);
          tc_commit(smem_u32(&sb.empty[s]));
        }
        if (ok) tc_commit(smem_u32(&sb.acc_full[b]));
      }
      if (!ok) raise_status(a.status, kStatusTimeout);
      // every MMA issued by this thread has finished before TMEM is released
      tc_commit(smem_u32(&sb.drain));
      if (!mbar_wait(smem_u32(&sb.drain), 0, kDrainTimeoutNs)) raise_status(a.status, kStatusTimeout);
    }
  } else if (warp >= kEpiWarp0) {
    const int sub = (warp - kEpiWarp0) >> 2;           // sub-tile of this warp
    const int q = warp & 3;                            // TMEM lane quarter (a warp reaches lanes 32 (warp % 4) ..)
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // TMEM column of this warp's accumulator in buffer j
    auto acc_col = [&](int j) { return static_cast<uint32_t>((j * MT + sub) * C::kAccStride); };
    // seed both accumulators for this CTA's first two tiles
    for (int j = 0; j < 2; ++j) {
      const int t = blockIdx.x + j * gridDim.x;
      if (t < tiles_total) seed_bias<BN>(tmem + lane_base + acc_col(j), a.bias, (t % a.tiles_n) * BN, a.N);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sb.acc_empty[j]));
    }
    int i = 0;
    for (int t = blockIdx.x; t < tiles_total; t += gridDim.x, ++i) {
      const int b = i & 1;
      bool ok = true;
      if (lane == 0) ok = wait_or_abort(smem_u32(&sb.acc_full[b]), (i >> 1) & 1, a.timeout_ns, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const int m0 = (t / a.tiles_n) * (kBM * MT) + sub * kBM;
      const int n0 = (t % a.tiles_n) * BN;
      const int row = m0 + 32 * q + lane;
      uint16_t* orow = a.out + static_cast<long long>(row) * a.N;
      const uint32_t acc = tmem + lane_base + acc_col(b);
      if constexpr (kRouter) {
        // logits of token `row`: bf16-rounded, ranked into the SLOTS largest keys
        uint32_t best[SLOTS];
#pragma unroll
        for (int r = 0; r < SLOTS; ++r) best[r] = 0;  // below every real key
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r32[32];
          tmem_ld32(acc + c, r32);
          tc_wait_ld();
          bool whole = c + 32 <= a.N;
          if constexpr (SLOTS != 4) whole = false;
          if (whole) {
            if constexpr (SLOTS == 4) {
              // 32 keys as four groups of eight: two sorted quads, their top four by a
              // bitonic merge, merged into the list the same way
#pragma unroll
              for (int g8 = 0; g8 < 4; ++g8) {
                uint32_t q[2][4];
#pragma unroll
                for (int v = 0; v < 8; v += 2) {
                  const uint32_t w = pack_bf16x2(__uint_as_float(r32[8 * g8 + v]), __uint_as_float(r32[8 * g8 + v + 1]));
                  const uint32_t e = static_cast<uint32_t>(c + 8 * g8 + v);
                  q[v >> 2][v & 3] = (order16(w & 0xFFFFu) << 16) | (0xFFFFu - e);
                  q[v >> 2][(v & 3) + 1] = (order16(w >> 16) << 16) | (0xFFFFu - e - 1);
                }
                sort4(q[0]);
                sort4(q[1]);
                merge4(q[0], q[1]);
                merge4(best, q[0]);
              }
            }
          } else {
#pragma unroll
            for (int v = 0; v < 32; ++v) {
              const int e = c + v;
              if (e < a.N) {
                const uint32_t bits = pack_bf16x2(__uint_as_float(r32[v]), 0.0f) & 0xFFFFu;
                offer<SLOTS>(best, (order16(bits) << 16) | (0xFFFFu - static_cast<uint32_t>(e)));
              }
            }
          }
        }
        if (row < a.M) {
          const int K = a.top_k;
          const float mx = key_value(best[0]);
          float ex[SLOTS];
          float sum = 0.0f;
#pragma unroll
          for (int r = 0; r < SLOTS; ++r) {
            ex[r] = 0.0f;
            if (r < K) {
              ex[r] = expf(key_value(best[r]) - mx);
              sum += ex[r];
            }
          }
          const float inv = 1.0f / sum;
#pragma unroll
          for (int r = 0; r < SLOTS; ++r) {
            if (r < K) {
              const int e = static_cast<int>(0xFFFFu - (best[r] & 0xFFFFu));
              a.topk_idx[static_cast<long long>(row) * K + r] = e;
              a.topk_w[static_cast<long long>(row) * K + r] =
                  static_cast<uint16_t>(pack_bf16x2(ex[r] * inv, 0.0f) & 0xFFFFu);
              if (a.counts) atomicAdd(&sb.hist[e], 1);
            }
          }
        }
      } else {
      auto store8 = [&](const uint32_t* r, int n) {  // 8 fp32 accumulators -> 8 bf16 at column n
        if (row < a.M && n < a.N) {
          const uint4 w = make_uint4(pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1])),
                                     pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3])),
                                     pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5])),
                                     pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7])));
          *reinterpret_cast<uint4*>(orow + n) = w;
        }
      };
#pragma unroll 1
      for (int c = 0; c + 32 <= BN; c += 32) {
        uint32_t r[32];
        tmem_ld32(acc + c, r);
        tc_wait_ld();
#pragma unroll
        for (int v = 0; v < 4; ++v) store8(r + 8 * v, n0 + c + 8 * v);
      }
      if constexpr (BN % 32 == 16) {  // last 16 columns
        uint32_t r[16];
        tmem_ld16(acc + BN - 16, r);
        tc_wait_ld();
        store8(r, n0 + BN - 16);
        store8(r + 8, n0 + BN - 8);
      }
      }
      // this buffer's next tile starts from its bias
      const int t2 = t + 2 * gridDim.x;
      if (t2 < tiles_total) seed_bias<BN>(tmem + lane_base + acc_col(b), a.bias, (t2 % a.tiles_n) * BN, a.N);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sb.acc_empty[b]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    // copies still in flight land before the shared memory is released
    const int issued = sb.issued;
    for (int s = 0; s < C::kStages && s < issued; ++s) {
      const int last = issued - 1 - ((issued - 1 - s) % C::kStages);
      if (!mbar_wait(smem_u32(&sb.full[s]), (last / C::kStages) & 1, kDrainTimeoutNs))
        raise_status(a.status, kStatusTimeout);
    }
  }
  __syncthreads();
  if constexpr (kRouter) {
    if (a.counts)
      for (int e = threadIdx.x; e < a.N; e += C::kThreads)
        if (sb.hist[e]) atomicAdd(a.counts + e, sb.hist[e]);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, int MT, int SLOTS = 0>
cudaError_t launch_linear_t(const CUtensorMap& amap, const CUtensorMap& bmap, const LinearArgs& a,
                            int sms, cudaStream_t stream) {
  using C = LinCfg<BN, MT>;
  // the shared-memory opt-in, once per device (host threads may race here: atomic flags,
  // and setting the attribute twice is harmless)
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(linear_bias_kernel<BN, MT, SLOTS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::kSmem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
  }
  const int tiles = a.tiles_m * a.tiles_n;
  const int grid = tiles < sms ? tiles : sms;
  linear_bias_kernel<BN, MT, SLOTS><<<grid, C::kThreads, C::kSmem, stream>>>(amap, bmap, a);
  return cudaGetLastError();
}

}  // namespace

int linear_m_sub(long long m, int n, int block_n, int sms) {
  return (block_n <= 128 && n <= block_n && (m + kBM - 1) / kBM > sms) ? 2 : 1;
}

template <int S>
cudaError_t launch_router_s(const CUtensorMap& amap, const CUtensorMap& bmap, const LinearArgs& a, int sms,
                            cudaStream_t stream) {
  const bool two = a.m_sub == 2;
  switch (a.block_n) {
    case 32: return two ? launch_linear_t<32, 2, S>(amap, bmap, a, sms, stream)
                        : launch_linear_t<32, 1, S>(amap, bmap, a, sms, stream);
    case 64: return two ? launch_linear_t<64, 2, S>(amap, bmap, a, sms, stream)
                        : launch_linear_t<64, 1, S>(amap, bmap, a, sms, stream);
    case 128: return two ? launch_linear_t<128, 2, S>(amap, bmap, a, sms, stream)
                         : launch_linear_t<128, 1, S>(amap, bmap, a, sms, stream);
    default: return launch_linear_t<256, 1, S>(amap, bmap, a, sms, stream);
  }
}

cudaError_t launch_linear_router(const CUtensorMap& amap, const CUtensorMap& bmap, const LinearArgs& a,
                                 int sms, cudaStream_t stream) {
  return a.top_k <= 4 ? launch_router_s<4>(amap, bmap, a, sms, stream)
                      : launch_router_s<8>(amap, bmap, a, sms, stream);
}

int linear_tile_n(int n) {
  // fewest estimated cycles per row block: ceil(N / BN) tiles of (BN + 32) each
  int best = 256;
  long long best_cost = -1;
  for (int bn : {256, 240, 192, 128}) {
    const long long cost = static_cast<long long>((n + bn - 1) / bn) * (bn + 32);
    if (best_cost < 0 || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

cudaError_t launch_linear(const CUtensorMap& amap, const CUtensorMap& bmap, const LinearArgs& a,
                          int sms, cudaStream_t stream) {
  switch (a.block_n) {
    case 128: return a.m_sub == 2 ? launch_linear_t<128, 2>(amap, bmap, a, sms, stream)
                                  : launch_linear_t<128, 1>(amap, bmap, a, sms, stream);
    case 192: return launch_linear_t<192, 1>(amap, bmap, a, sms, stream);
    case 240: return launch_linear_t<240, 1>(amap, bmap, a, sms, stream);
    default: return launch_linear_t<256, 1>(amap, bmap, a, sms, stream);
  }
}

}  // namespace sa
