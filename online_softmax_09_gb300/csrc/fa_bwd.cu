// fa_bwd.cu -- backward pass of exact softmax attention on sm_103a.
//
// The forward pass kept only O and the per-row log-sum-exp; the probabilities are recomputed
// tile by tile from Q, K, V and LSE instead of being stored ("LLM Architecture Refresh [3]:
// Flash Attention Is Exact", section 8, its paragraph on the backward pass). Gradients are
// the textbook ones for O = softmax(scale Q K^T) V:
//   P = exp(scale S - LSE), dV = P^T dO, dP = dO V^T, delta = rowsum(dO * O),
//   dS = P * (dP - delta), dQ = scale dS K, dK = scale dS^T Q.
//
// Three kernels on the caller's stream:
//   1. preprocess: -delta and -LSE*log2(e) per query row (padded rows: 0 and -inf), and
//      zeroes the fp32 dQ accumulator and the main kernel's work counter.     (HBM-bound)
//   2. main: persistent, one CTA per SM walking work items, one item per (batch, kv head,
//      128-key tile). For an item it keeps K_n and V_n in shared memory and the dK, dV
//      accumulators in TMEM, and loops over the G query heads of its group and their query
//      tiles (causal: from the diagonal tile on). Per query tile i:
//        softmax warps (thread = key row): P_i^T = 2^(S_i^T scale log2e - LSE2), bf16 -> TMEM
//        MMA  dV += P_i^T dO_i ;  dP_i^T = V_n dO_i^T ;  S_{i+1}^T = K_n Q_{i+1}^T
//        softmax warps: dS_i^T = P_i^T (dP_i^T - delta), bf16 -> shared memory
//        MMA  dQ_i = dS_i K_n  (into the dP^T columns, now free) ;  dK += dS_i^T Q_i
//        drain warps (thread = query row): dQ_i TMEM -> shared memory -> bulk tensor
//        reduction (add) into the fp32 workspace accumulator.
//      The next tile's S^T is computed while the softmax warps work on dS_i, and its P while
//      the dQ and dK MMAs run, so the tensor core does not wait for the softmax warps. The one
//      shared-memory copy of dS serves both of its MMAs (MN-major A of dQ, K-major A of dK),
//      and dQ goes first so that its drain overlaps the dK MMA. Items are numbered in bands of
//      (batch, kv head) pairs, key tile by key tile within a band, so that the Q, dO and dQ
//      accumulator rows that a band's items share stay in L2 (see bwd_band), and handed out
//      in that order from a counter as CTAs finish their previous item. An item's end overlaps
//      the next one's start: its V tile loads once its last dP^T MMA has read V, the next
//      item's first dP^T and the softmax warps' next P phase run while the drain warps write
//      dK and dV out.
//   3. dQ conversion: dq = bf16(scale * accumulator).
//
// Warp roles of the main kernel: 0-3 and 10-13 softmax/dS (thread = key row; warps 0-3 take
// query columns [0, 64) of every row, warps 10-13 columns [64, 128), so each row's elementwise
// work is split between two warps of the same TMEM lane quarter); 4 TMA producer and work
// fetcher, 5 MMA issuer (the whole warp runs the loop, one elected lane issues) and TMEM owner,
// 6-9 dQ drain and, at the end of each item, the dV and dK epilogue.
// TMEM columns: S^T/P^T [0,128), dP^T/dQ [128,256), dV [256,256+D), dK [256+D,256+2D).
// P^T is packed bf16 (two queries per column): queries [0, 64) in columns [0, 32), queries
// [64, 128) in [64, 96), i.e. each half over score columns its own warps have already read.
// For D = 128 the dS operand of the dQ MMA is written into the dO slot of the current stage
// once the dV and dP MMAs (the readers of dO) have completed; for D = 64 it has its own buffer.
#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------------------------------
// 1. Preprocess: delta = rowsum(dO * O), LSE2 = LSE * log2(e), dQ accumulator = 0.
// ------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dout,
                                                         const float* __restrict__ lse, float* __restrict__ dq_acc,
                                                         float* __restrict__ delta, float* __restrict__ lse2,
                                                         uint32_t* __restrict__ next_item, int N, int Npad,
                                                         long long rows) {
  constexpr int TPR = D / 8;  // threads per row, 8 elements (16 bytes) each
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long r = gt / TPR;  // row of the padded [B*Hq][Npad] grid
  const int part = (int)(gt % TPR);
  if (gt == 0) next_item[0] = next_item[1] = 0u;  // the main kernel's work-item counters
  if (r >= rows) return;  // rows are whole TPR-lane groups, so groups exit together
  const long long bh = r / Npad;
  const int n = (int)(r - bh * Npad);
  float4* acc = reinterpret_cast<float4*>(dq_acc + r * D + part * 8);
  acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
  acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  float s = 0.f;
  if (n < N) {
    const size_t off = ((size_t)bh * N + n) * D + part * 8;
    const uint4 ov = *reinterpret_cast<const uint4*>(o + off);
    const uint4 dv = *reinterpret_cast<const uint4*>(dout + off);
    const __nv_bfloat162* op = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* dp = reinterpret_cast<const __nv_bfloat162*>(&dv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = __bfloat1622float2(op[i]);
      const float2 b = __bfloat1622float2(dp[i]);
      s = fmaf(a.x, b.x, s);
      s = fmaf(a.y, b.y, s);
    }
  }
  const int lane = threadIdx.x & 31;
  const unsigned group = ((TPR == 32) ? 0xffffffffu : ((1u << TPR) - 1u)) << (lane & ~(TPR - 1));
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(group, s, off);
  if (part == 0) {  // stored negated: the main kernel adds them with packed f32x2 arithmetic
    delta[r] = (n < N) ? -s : 0.f;
    lse2[r] = (n < N) ? -(lse[(size_t)bh * N + n] * kLog2e) : -INFINITY;
  }
}

// ------------------------------------------------------------------------------------------
// 3. dq = bf16(scale * dq_acc) on the unpadded rows.
// ------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ dq_acc,
                                                        __nv_bfloat16* __restrict__ dq, int N, int Npad,
                                                        long long n_vec4, float scale) {
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec4;
       v += (long long)gridDim.x * blockDim.x) {
    const long long e = v * 4;
    const long long row = e / D;  // over [B*Hq][N]
    const int col = (int)(e - row * D);
    const long long bh = row / N;
    const long long n = row - bh * N;
    const float4 a = *reinterpret_cast<const float4*>(dq_acc + (bh * Npad + n) * D + col);
    uint2 w;
    w.x = pack_bf16(a.x * scale, a.y * scale);
    w.y = pack_bf16(a.z * scale, a.w * scale);
    *reinterpret_cast<uint2*>(dq + e) = w;
  }
}

// ------------------------------------------------------------------------------------------
// 2. Main kernel.
// ------------------------------------------------------------------------------------------
struct BwdParams {
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* delta;
  const float* lse2;
  uint32_t* status;
  int B, Hq, Hkv, N, Npad, causal, num_tiles;
  int window;  // > 0: causal sliding window of this many keys
  float scale, scale_log2;
  int band;       // (b, kv head) pairs per band of work items; B * Hkv for a single band
  int num_items;  // B * Hkv * num_tiles work items (key tiles)
  uint32_t* next_item;  // workspace: [0] items handed out beyond the first gridDim.x,
                        // [1] CTAs that found no more items
};

// Work item `idx`: key tile n of kv head (b, hkv). Items are numbered band by band (p.band
// consecutive (b, kv head) pairs, the last band possibly narrower) and key tile by key tile
// within a band, so a band's causal tiles with the most query tiles come first and its Q, dO
// and dQ accumulator rows stay in L2 while its items run. The item visits the G query heads of
// its group and, per head, query tiles [i0, i0 + n_i): from the diagonal (causal) to, with a
// sliding window, the tile of the last query within `window` of the tile's last key.
struct BwdItem {
  int b, hkv, n, i0, n_i, n_iter;
};
template <bool kWin>
__device__ __forceinline__ BwdItem bwd_item(int idx, const BwdParams& p) {
  BwdItem w;
  const int BHk = p.B * p.Hkv;
  const int per_band = p.band * p.num_tiles;
  const int band_i = idx / per_band;
  const int first = band_i * p.band;
  const int width = min(p.band, BHk - first);
  const int local = idx - band_i * per_band;
  w.n = local / width;
  const int bhk = first + (local - w.n * width);
  w.b = bhk / p.Hkv;
  w.hkv = bhk - w.b * p.Hkv;
  w.i0 = p.causal ? w.n : 0;
  const int i_end =
      kWin ? min(p.num_tiles, (w.n * kTile + kTile - 1 + p.window - 1) / kTile + 1) : p.num_tiles;
  w.n_i = i_end - w.i0;
  w.n_iter = (p.Hq / p.Hkv) * w.n_i;
  return w;
}

template <int D>
struct BwdSmem {
  static constexpr bool kAliasDS = (D == 128);
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kStage0 = kV + kTileBytes;
  // Stage layout: Q tile, dO tile, LSE2 (128 fp32), delta (128 fp32).
  static constexpr int kStQ = 0;
  static constexpr int kStDO = kTileBytes;
  static constexpr int kStL = 2 * kTileBytes;
  static constexpr int kStD = 2 * kTileBytes + 512;
  static constexpr int kStageBytes = 2 * kTileBytes + 1024;
  static constexpr int kDS = kStage0 + 2 * kStageBytes;
  // dQ staging for the bulk reductions (and, at an item's end, the dK / dV bulk stores):
  // 4 drain warps x 2 buffers x 32 rows x 128 bytes.
  static constexpr int kDQ = kDS + (kAliasDS ? 0 : kTile * kTile * 2);
  static constexpr int kBar = kDQ + 4 * 2 * 32 * 128;
  enum {
    bK = 0,
    bV,
    bQFull,           // 2
    bDOFull = 4,      // 2
    bStageEmpty = 6,  // 2
    bSFull = 8,
    bDPFull,
    bPReady,
    bSmemDS,
    bDVDone,  // dV_i has finished reading dO_i (whose slot then takes dS_i)
    bDQFull,
    bDQFree,
    bFinal,   // every MMA of the item has completed: dK, dV final in TMEM
    bKFree,   // the item's last dQ MMA has read K
    bVFree,   // the item's last dP^T MMA has read V
    bAccFree, // the epilogue has read dK and dV out of TMEM
    bItemFull = 19,   // 2
    bItemEmpty = 21,  // 2
    bDrain = 23,
    kNumBars
  };
  static_assert(bDOFull == bQFull + 2 && bStageEmpty == bDOFull + 2 && bSFull == bStageEmpty + 2 &&
                    bItemEmpty == bItemFull + 2 && bDrain == bItemEmpty + 2,
                "two-slot barriers overlap");
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kItem = kAbort + 4;  // 2 slots: work item index, -1 past the end
  static constexpr int kBytes = kItem + 8;
  // No alignment slack: the kernel uses no static shared memory, so the dynamic window starts
  // on a 1024-byte boundary; the kernel checks this and stops (status 2) if it ever does not.
  static constexpr int kAlloc = kBytes;
  static_assert(kStageBytes % 1024 == 0 && kStage0 % 1024 == 0 && kDS % 1024 == 0 && kDQ % 1024 == 0,
                "1024-byte alignment");
};

constexpr int kBwdThreads = 448;
// Arrivals that release an item slot: the MMA warp, eight softmax warps and four drain warps.
constexpr int kItemConsumers = 13;
// TMEM column of the packed bf16 P^T operand for the 16 queries of MMA step kk.
__device__ __forceinline__ uint32_t packed_col(int kk) { return (uint32_t)(kk * 8 + (kk >= 4 ? 32 : 0)); }

template <int D, bool kWin>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                       const __grid_constant__ CUtensorMap tm_dv, const BwdParams p) {
  using L = BwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  if (raw & 1023u) {  // uniform over the CTA, before any barrier or tensor memory is touched
    if (threadIdx.x == 0) atomicCAS(p.status, kStatusOk, kStatusSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + L::kK;
  const uint32_t sV = sbase + L::kV;
  auto stage = [&](int s) -> uint32_t { return sbase + L::kStage0 + (uint32_t)s * L::kStageBytes; };
  auto stage_ptr = [&](int s) -> uint8_t* { return smem + L::kStage0 + s * L::kStageBytes; };
  auto sDS = [&](int s) -> uint32_t { return L::kAliasDS ? stage(s) + L::kStDO : sbase + L::kDS; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const Ctl ctl{abort_flag, p.status};
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int G = p.Hq / p.Hkv;
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + L::kItem);

  if (threadIdx.x == 0) {
    mbar_init(bar(L::bK), 1);
    mbar_init(bar(L::bV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::bQFull + s), 1);
      mbar_init(bar(L::bDOFull + s), 1);
      mbar_init(bar(L::bStageEmpty + s), 1);
      mbar_init(bar(L::bItemFull + s), 1);
      mbar_init(bar(L::bItemEmpty + s), kItemConsumers);
    }
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bDPFull), 1);
    mbar_init(bar(L::bPReady), 256);
    mbar_init(bar(L::bSmemDS), 256);
    mbar_init(bar(L::bDQFull), 1);
    mbar_init(bar(L::bDVDone), 1);
    mbar_init(bar(L::bDQFree), 128);
    mbar_init(bar(L::bFinal), 1);
    mbar_init(bar(L::bKFree), 1);
    mbar_init(bar(L::bVFree), 1);
    mbar_init(bar(L::bAccFree), 128);
    mbar_init(bar(L::bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);

  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;         // S^T, then P^T (bf16)
  const uint32_t tdP = tmem + 128;  // dP^T, then dQ
  const uint32_t tdV = tmem + 256;
  const uint32_t tdK = tmem + 256 + D;

  // Item r of this CTA, consumer side: waits until the producer has published it, reads it and
  // releases the slot (one arrival per consumer warp). -1: no more items, or an abort.
  auto take_item = [&](int r) -> int {
    if (!mbar_wait_warp(bar(L::bItemFull + (r & 1)), (r >> 1) & 1, ctl)) return -1;
    const int idx = item_slot[r & 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::bItemEmpty + (r & 1)));
    return idx;
  };

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    // Persistent: the CTA's first item is blockIdx.x, later ones come from a workspace counter
    // in launch order, so items still start in the order a one-CTA-per-item launch would start
    // them (and the band order holds). Each item is published to the other roles through a
    // two-slot ring. V of the next item is loaded once the previous item's last dP^T MMA has
    // read V, K once its last dQ MMA has read K (both are prefetched into L2 when the item is
    // fetched); Q, dO, LSE2 and delta go through the two stages.
    if (lane == 0) {
      constexpr uint32_t kTB = L::kTileBytes;
      int g = 0;        // query tiles loaded so far (all items)
      int issued = 0;   // tiles whose loads were issued
      int r = 0;        // items published
      int v_loads = 0, k_loads = 0;  // items whose V / K loads were issued
      bool ok = true;
      for (;; ++r) {
        int idx = (r == 0) ? (int)blockIdx.x : (int)gridDim.x + (int)atomicAdd(p.next_item, 1u);
        if (idx >= p.num_items) {
          idx = -1;
          // The last CTA to run out of items puts the counters back to zero (no CTA fetches
          // again), so that the kernel can run again without a new prepare pass.
          if (r > 0 && atomicAdd(p.next_item + 1, 1u) == gridDim.x - 1) {
            atomicExch(p.next_item, 0u);
            atomicExch(p.next_item + 1, 0u);
          }
        }
        if (r >= 2 && !(ok = mbar_wait(bar(L::bItemEmpty + (r & 1)), ((r >> 1) - 1) & 1, ctl))) break;
        item_slot[r & 1] = idx;
        mbar_arrive(bar(L::bItemFull + (r & 1)));
        if (idx < 0) break;
        const BwdItem w = bwd_item<kWin>(idx, p);
        const int kv_z = w.b * p.Hkv + w.hkv;
        if (r > 0) {  // K and V into L2 now; into shared memory once the previous item frees them
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tma_prefetch_l2_3d(&tm_k, c * 64, w.n * kTile, kv_z);
            tma_prefetch_l2_3d(&tm_v, c * 64, w.n * kTile, kv_z);
          }
        }
        auto load_tile = [&](int it) -> bool {
          const int s = g & 1;
          if (!mbar_wait(bar(L::bStageEmpty + s), ((g >> 1) & 1) ^ 1, ctl)) return false;
          const int gi = it / w.n_i;
          const int hq = w.hkv * G + gi;
          const int i = w.i0 + (it - gi * w.n_i);
          const int qz = w.b * p.Hq + hq;
          const size_t srow = (size_t)qz * p.Npad + (size_t)i * kTile;
          const uint32_t st = stage(s);
          mbar_expect_tx(bar(L::bQFull + s), kTB + 512);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(st + L::kStQ + c * 16384, &tm_q, bar(L::bQFull + s), c * 64, i * kTile, qz);
          bulk_load(st + L::kStL, p.lse2 + srow, 512, bar(L::bQFull + s));
          mbar_expect_tx(bar(L::bDOFull + s), kTB + 512);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(st + L::kStDO + c * 16384, &tm_do, bar(L::bDOFull + s), c * 64, i * kTile, qz);
          bulk_load(st + L::kStD, p.delta + srow, 512, bar(L::bDOFull + s));
          ++g;
          issued = g;
          return true;
        };
        // V (its slot frees first), the first query tile, then K.
        if (r > 0 && !(ok = mbar_wait(bar(L::bVFree), (r - 1) & 1, ctl))) break;
        mbar_expect_tx(bar(L::bV), kTB);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sV + c * 16384, &tm_v, bar(L::bV), c * 64, w.n * kTile, kv_z);
        v_loads = r + 1;
        if (w.n_iter > 0 && !(ok = load_tile(0))) break;
        if (r > 0 && !(ok = mbar_wait(bar(L::bKFree), (r - 1) & 1, ctl))) break;
        mbar_expect_tx(bar(L::bK), kTB);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sK + c * 16384, &tm_k, bar(L::bK), c * 64, w.n * kTile, kv_z);
        k_loads = r + 1;
        for (int it = 1; ok && it < w.n_iter; ++it) ok = load_tile(it);
        if (!ok) break;
      }
      if (!ok || *abort_flag) {
        // Let the copies in flight land before the CTA releases its shared memory.
        if (k_loads > 0) drain_wait(bar(L::bK), (k_loads - 1) & 1);
        if (v_loads > 0) drain_wait(bar(L::bV), (v_loads - 1) & 1);
        for (int t = issued > 2 ? issued - 2 : 0; t < issued; ++t) {
          drain_wait(bar(L::bQFull + (t & 1)), (t >> 1) & 1);
          drain_wait(bar(L::bDOFull + (t & 1)), (t >> 1) & 1);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    // Per query tile i: dV += P_i^T dO_i, S_{i+1}^T = K Q_{i+1}^T, dQ_i = dS_i K,
    // dK += dS_i^T Q_i, then dP_{i+1}^T = V dO_{i+1}^T. dP does not depend on P, so it is issued
    // as soon as its TMEM columns are free (dQ_i drained), ahead of the P phase it will meet:
    // the softmax warps then go from P_{i+1} straight to dS_{i+1}. The dQ drain overlaps dK.
    // The whole warp runs the loop (warp-uniform counters, phases and descriptors); one elected
    // lane issues each group of MMAs and each commit.
    constexpr uint32_t idSS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
    constexpr uint32_t idTS = idesc_bf16_f32(128, D, false, true);     // dV, dK
    constexpr uint32_t idDQ = idesc_bf16_f32(128, D, true, true);      // dQ
    // Descriptor bases (K-major with 16-byte leading offset; MN-major with 16 KB); an operand
    // or MMA step adds its byte offset / 16 to the start-address field.
    const uint64_t dK_k = sdesc_sw128(sK, 16, 1024), dV_k = sdesc_sw128(sV, 16, 1024);
    const uint64_t dK_mn = sdesc_sw128(sK, 16384, 1024);
    const uint64_t dSt_k = sdesc_sw128(stage(0), 16, 1024), dSt_mn = sdesc_sw128(stage(0), 16384, 1024);
    const uint64_t dDS_k = sdesc_sw128(sDS(0), 16, 1024), dDS_mn = sdesc_sw128(sDS(0), 16384, 1024);
    constexpr uint32_t kStage16 = L::kStageBytes >> 4;
    auto kmajor = [](int kk) -> uint32_t { return (uint32_t)(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); };
    // Tiles are counted over all items of the CTA (t), which sets every barrier phase.
    auto issue_s = [&](int t) {  // S^T = K_n Q_t^T into tS
      const uint64_t q = dSt_k + (uint32_t)((t & 1) * kStage16 + (L::kStQ >> 4));
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tS, dK_k + kmajor(kk), q + kmajor(kk), idSS, kk > 0);
        mma_commit(bar(L::bSFull));
      }
      __syncwarp();
    };
    // dP^T_t = V_n dO_t^T into tdP, once dO_t has landed and dQ_{t-1} has been drained out of
    // these columns.
    auto issue_dp = [&](int t) -> bool {
      if (!mbar_wait_warp(bar(L::bDOFull + (t & 1)), (t >> 1) & 1, ctl)) return false;
      if (t > 0 && !mbar_wait_warp(bar(L::bDQFree), (t - 1) & 1, ctl)) return false;
      tc_fence_after();
      const uint64_t dO = dSt_k + (uint32_t)((t & 1) * kStage16 + (L::kStDO >> 4));
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tdP, dV_k + kmajor(kk), dO + kmajor(kk), idSS, kk > 0);
        mma_commit(bar(L::bDPFull));
      }
      __syncwarp();
      return true;
    };
    auto commit = [&](int b_) {
      if (elect_one()) mma_commit(bar(b_));
      __syncwarp();
    };
    bool ok = true;
    int g = 0;  // query tiles of earlier items
    for (int r = 0; ok; ++r) {
      const int idx = take_item(r);
      if (idx < 0) break;
      const int n_iter = bwd_item<kWin>(idx, p).n_iter;  // >= 1: the diagonal tile always sees its keys
      // The item's first dP^T needs V only (loaded as soon as the previous item's last dP^T read
      // V); its first S^T waits for K, which follows the previous item's last MMAs.
      ok = mbar_wait_warp(bar(L::bV), r & 1, ctl) && issue_dp(g);
      if (ok && n_iter == 1) commit(L::bVFree);
      ok = ok && mbar_wait_warp(bar(L::bK), r & 1, ctl) && mbar_wait_warp(bar(L::bQFull + (g & 1)), (g >> 1) & 1, ctl);
      if (!ok) break;
      tc_fence_after();
      issue_s(g);
      for (int it = 0; it < n_iter; ++it) {
        const int t = g + it;
        const int s = t & 1;
        const uint32_t st16 = (uint32_t)s * kStage16;
        // dV += P^T dO_t (P^T from TMEM; dO as the MN-major B operand; dO_t waited for dP_t).
        // The item's first dV (and dK) overwrite the accumulators: the previous item's epilogue
        // must have read them out.
        if (!(ok = mbar_wait_warp(bar(L::bPReady), t & 1, ctl))) break;
        if (it == 0 && r > 0 && !(ok = mbar_wait_warp(bar(L::bAccFree), (r - 1) & 1, ctl))) break;
        tc_fence_after();
        {
          const uint64_t dO = dSt_mn + st16 + (L::kStDO >> 4);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ts(tdV, tS + packed_col(kk), dO + (uint32_t)(kk * (2048 >> 4)), idTS, (it > 0 || kk > 0));
            mma_commit(bar(L::bDVDone));
          }
          __syncwarp();
        }
        // S^T of the next query tile (P_t^T in these columns was read by the dV MMA above).
        if (it + 1 < n_iter) {
          if (!(ok = mbar_wait_warp(bar(L::bQFull + (s ^ 1)), ((t + 1) >> 1) & 1, ctl))) break;
          tc_fence_after();
          issue_s(t + 1);
        }
        // dQ_t = dS K_n (dS and K both MN-major in shared memory) into the dP^T columns, first,
        // so the drain starts as early as possible; then dK += dS^T Q_t with the same
        // shared-memory dS as the K-major A operand.
        if (!(ok = mbar_wait_warp(bar(L::bSmemDS), t & 1, ctl))) break;
        tc_fence_after();
        {
          const uint32_t ds16 = L::kAliasDS ? st16 + (L::kStDO >> 4) : 0u;
          const uint64_t ds_mn = (L::kAliasDS ? dSt_mn : dDS_mn) + ds16;
          const uint64_t ds_k = (L::kAliasDS ? dSt_k : dDS_k) + ds16;
          const uint64_t q_mn = dSt_mn + st16 + (L::kStQ >> 4);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ss(tdP, ds_mn + (uint32_t)(kk * (2048 >> 4)), dK_mn + (uint32_t)(kk * (2048 >> 4)), idDQ,
                     kk > 0);
            mma_commit(bar(L::bDQFull));
            if (it + 1 == n_iter) mma_commit(bar(L::bKFree));  // the item's last reader of K
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_ss(tdK, ds_k + kmajor(kk), q_mn + (uint32_t)(kk * (2048 >> 4)), idTS, (it > 0 || kk > 0));
            mma_commit(bar(L::bStageEmpty + s));
          }
          __syncwarp();
        }
        if (it + 1 < n_iter) {
          if (!(ok = issue_dp(t + 1))) break;
          if (it + 2 == n_iter) commit(L::bVFree);  // the item's last reader of V
        }
      }
      if (!ok) break;
      commit(L::bFinal);
      g += n_iter;
    }
    if (*abort_flag) {
      if (elect_one()) {
        mma_commit(bar(L::bDrain));
        drain_wait(bar(L::bDrain), 0);
      }
      __syncwarp();
    }
  } else if (warp < 4 || warp >= 10) {
    // ------------------------------------------------------------------ softmax / dS warps
    const int grp = warp >= 10;  // query columns [64 grp, 64 grp + 64) of each key row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int kr = (warp & 3) * 32 + lane;  // key row within the tile
    const float sl2 = p.scale_log2;
    bool ok = true;
    uint32_t pk[2][16];  // this warp's half of P_t^T as packed bf16, kept for the dS phase
    int g = 0;           // query tiles of earlier items
    for (int r = 0; ok; ++r) {
    const int idx = take_item(r);
    if (idx < 0) break;
    const BwdItem w = bwd_item<kWin>(idx, p);
    const int n = w.n, n_iter = w.n_iter;
    const int key = n * kTile + kr;
    const bool key_ok = key < p.N;
    // P phase of the item's query tile `it` (tile t = g + it of the CTA):
    // P^T = 2^(S^T scale log2e - LSE2), bf16 into TMEM and pk.
    auto p_phase = [&](int it) -> bool {
      const int t = g + it;
      const int s = t & 1;
      const int i = w.i0 + it % w.n_i;
      const bool diag = p.causal && i == n;
      // Window: query q sees key j only if q - j < window; (i - n) * 128 + q - kr is q - j.
      const bool wmask = kWin && (i - n) * kTile + kTile - 1 >= p.window;
      const float* sl = reinterpret_cast<const float*>(stage_ptr(s) + L::kStL);
      // Queries of this tile that see this key row: [q_lo, q_hi] (none for a key past N).
      const int q_lo = !key_ok ? kTile : (diag ? kr : 0);
      const int q_hi = wmask ? kr + p.window - 1 - (i - n) * kTile : kTile - 1;
      const bool masked = __any_sync(0xffffffffu, q_lo > 0 || q_hi < kTile - 1);  // warp-uniform
      if (!mbar_wait_warp(bar(L::bQFull + s), (t >> 1) & 1, ctl)) return false;
      if (!mbar_wait_warp(bar(L::bSFull), t & 1, ctl)) return false;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * grp + cc;  // 32-query chunk
        uint32_t sr[32];
        tmem_ld32(tS + lane_off + c * 32, sr);
        tmem_ld_wait(sr);
        if (masked) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(sl + c * 32 + j);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
            float pv[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int q = c * 32 + j + t;
              pv[t] = (q < q_lo || q > q_hi) ? 0.f : ex2(fmaf(__uint_as_float(sr[j + t]), sl2, lv[t]));
            }
            pk[cc][j / 2] = pack_bf16(pv[0], pv[1]);
            pk[cc][j / 2 + 1] = pack_bf16(pv[2], pv[3]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(sl + c * 32 + j);  // -LSE2
            const float2 x01 = fma2(make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])),
                                    make_float2(sl2, sl2), make_float2(l4.x, l4.y));
            const float2 x23 = fma2(make_float2(__uint_as_float(sr[j + 2]), __uint_as_float(sr[j + 3])),
                                    make_float2(sl2, sl2), make_float2(l4.z, l4.w));
            pk[cc][j / 2] = pack_bf16(ex2(x01.x), ex2(x01.y));
            pk[cc][j / 2 + 1] = pack_bf16(ex2(x23.x), ex2(x23.y));
          }
        }
        // P^T (bf16) of chunk c into columns [64 grp + 16 cc, +16): score columns this warp
        // has already read.
        tmem_st16(tS + lane_off + 64 * grp + 16 * cc, pk[cc]);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(L::bPReady));
      return true;
    };
    ok = p_phase(0);
    for (int it = 0; ok && it < n_iter; ++it) {
      const int t = g + it;
      const int s = t & 1;
      const float* sd = reinterpret_cast<const float*>(stage_ptr(s) + L::kStD);
      if (!(ok = mbar_wait_warp(bar(L::bDOFull + s), (t >> 1) & 1, ctl))) break;
      if (!(ok = mbar_wait_warp(bar(L::bDPFull), t & 1, ctl))) break;
      tc_fence_after();
      // dS^T = P^T (dP^T - delta) with the bf16 P the dV MMA used. dS goes to shared memory
      // only after dV_it (issued after dP_it) has read the dO slot it reuses (d = 128), and
      // after dK_{it-2}, dQ_{it-2} -- the previous readers of this stage -- which the stage's
      // reload for dO_it already implies.
      const uint32_t row_base = sDS(s) + (uint32_t)kr * 128;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * grp + cc;
        uint32_t dr[32];
        tmem_ld32(tdP + lane_off + c * 32, dr);
        tmem_ld_wait(dr);
        uint32_t ds[16];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(sd + c * 32 + j);  // -delta
          const float2 p01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[cc][j / 2]));
          const float2 p23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&pk[cc][j / 2 + 1]));
          const float2 s01 = mul2(add2(make_float2(__uint_as_float(dr[j]), __uint_as_float(dr[j + 1])),
                                       make_float2(d4.x, d4.y)), p01);
          const float2 s23 = mul2(add2(make_float2(__uint_as_float(dr[j + 2]), __uint_as_float(dr[j + 3])),
                                       make_float2(d4.z, d4.w)), p23);
          ds[j / 2] = pack_bf16(s01.x, s01.y);
          ds[j / 2 + 1] = pack_bf16(s23.x, s23.y);
        }
        // dS takes dO_it's slot (d = 128): dV_it, issued after dP_it, must have read it.
        if (cc == 0 && !(ok = mbar_wait_warp(bar(L::bDVDone), t & 1, ctl))) break;
        // Shared-memory copy of dS: row = key, 64-query chunks 16 KB apart, 16-byte granules
        // (8 queries) XOR-swizzled by (key mod 8): the MN-major A operand of the dQ MMA.
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          const int g = cc * 4 + g4;
          st_shared_v4(row_base + grp * 16384 + ((g ^ (kr & 7)) << 4), ds[4 * g4], ds[4 * g4 + 1],
                       ds[4 * g4 + 2], ds[4 * g4 + 3]);
        }
      }
      if (!ok) break;
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar(L::bSmemDS));
      if (it + 1 < n_iter && !(ok = p_phase(it + 1))) break;
    }
    g += n_iter;
    }  // items
  } else {
    // ------------------------------------------------------------------ dQ drain warps 6-9
    // Each warp owns 32 query rows (its TMEM lane quarter). 32 columns at a time, the warp
    // stages its 32 x 32 fp32 block of dQ_i in shared memory (128-byte swizzled: 16-byte granule
    // g of row r at g ^ (r mod 8)) and one lane adds it into the workspace accumulator with a
    // bulk tensor reduction. Warps never wait for one another.
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t stage_buf = sbase + L::kDQ + (uint32_t)(warp & 3) * 8192;
    bool ok = true;
    int t = 0;  // query tiles drained (all items)
    for (int r = 0; ok; ++r) {
    const int idx = take_item(r);
    if (idx < 0) break;
    const BwdItem w = bwd_item<kWin>(idx, p);
    for (int it = 0; it < w.n_iter; ++it, ++t) {
      const int gi = it / w.n_i;
      const int hq = w.hkv * G + gi;
      const int i = w.i0 + (it - gi * w.n_i);
      if (!(ok = mbar_wait_warp(bar(L::bDQFull), t & 1, ctl))) break;
      tc_fence_after();
      const int row0 = (w.b * p.Hq + hq) * p.Npad + i * kTile + (warp & 3) * 32;
      // Two halves of 64 columns (the register budget of 14 warps), each chunk staged through
      // buffer (chunk mod 2): a buffer is rewritten only after the reduction issued from it
      // two chunks earlier has read it, so the first half never waits for a reduction and the
      // columns are released right after the second half is loaded.
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        uint32_t a[2][32];
        tmem_ld32(tdP + lane_off + (2 * h) * 32, a[0]);
        tmem_ld32(tdP + lane_off + (2 * h + 1) * 32, a[1]);
        tmem_ld_wait(a[0]);
        tmem_ld_wait(a[1]);
        if (h == D / 64 - 1) {
          tc_fence_before();
          mbar_arrive(bar(L::bDQFree));
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * h + cc;
          const uint32_t buf = stage_buf + (uint32_t)cc * 4096;
          if (lane == 0) bulk_wait_read_but1();  // the reduction from this buffer has read it
          __syncwarp();
#pragma unroll
          for (int g = 0; g < 8; ++g)
            st_shared_v4(buf + (uint32_t)lane * 128 + ((g ^ (lane & 7)) << 4), a[cc][4 * g], a[cc][4 * g + 1],
                         a[cc][4 * g + 2], a[cc][4 * g + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_2d(&tm_dq, buf, c * 32, row0);
            bulk_commit_group();
          }
        }
      }
    }
    if (!ok) break;
    // ---------------------------------------------------------------- dV / dK epilogue
    // Once every MMA of the item has completed, the drain warp moves its 32 key rows of dV,
    // then dK, out of TMEM 64 columns at a time, releases the accumulator columns after the last
    // read (the next item's first dV / dK MMA may then start), and writes each chunk as bf16
    // through its staging buffers with a bulk tensor store (whole lines; rows past N are not
    // written). The softmax warps meanwhile start on the next item.
    if (!(ok = mbar_wait_warp(bar(L::bFinal), r & 1, ctl))) break;
    tc_fence_after();
    {
      const int y0 = w.n * kTile + (warp & 3) * 32;
      const int kv_z = w.b * p.Hkv + w.hkv;
#pragma unroll
      for (int grp = 0; grp < 2; ++grp) {
        const uint32_t src = grp ? tdK : tdV;
        const float mul = grp ? p.scale : 1.f;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t a[2][32];
          tmem_ld32(src + lane_off + (2 * c) * 32, a[0]);
          tmem_ld32(src + lane_off + (2 * c + 1) * 32, a[1]);
          tmem_ld_wait(a[0]);
          tmem_ld_wait(a[1]);
          if (grp == 1 && c == D / 64 - 1) {
            tc_fence_before();
            mbar_arrive(bar(L::bAccFree));
          }
          // Chunks alternate between the two buffers (dV then dK at d = 64).
          const uint32_t buf = stage_buf + (uint32_t)((grp * (D / 64) + c) & 1) * 4096;
          if (lane == 0) bulk_wait_read_but1();  // the copy issued from this buffer has read it
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t* v = a[q >> 2] + 8 * (q & 3);
            st_shared_v4(buf + (uint32_t)lane * 128 + ((q ^ (lane & 7)) << 4),
                         pack_bf16(__uint_as_float(v[0]) * mul, __uint_as_float(v[1]) * mul),
                         pack_bf16(__uint_as_float(v[2]) * mul, __uint_as_float(v[3]) * mul),
                         pack_bf16(__uint_as_float(v[4]) * mul, __uint_as_float(v[5]) * mul),
                         pack_bf16(__uint_as_float(v[6]) * mul, __uint_as_float(v[7]) * mul));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (y0 < p.N) tma_store_3d(grp ? &tm_dk : &tm_dv, buf, c * 64, y0, kv_z);
            bulk_commit_group();
          }
        }
      }
    }
    }  // items
    if (lane == 0) bulk_wait_all();  // every reduction has landed before the CTA exits
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// (b, kv head) pairs per band of work items. Bands shrink the set of heads whose Q, dO and fp32
// dQ accumulator rows the items in flight share: as many bands as keep each band's work per SM
// at least 1.4 times its longest item (whose G * T query tiles would otherwise end alone; a
// measured margin: 1.28 lost 3 %, 1.41 and above gained), but no more than it takes to fit a
// band's working set (its G query heads' Q and dO, bf16, and dQ accumulator, fp32, plus K and
// V) in about 80 MiB of the 129 MB L2. One band (plain key-tile-major order) where the margin
// allows no split, and for the sliding window.
static int bwd_band(int B, int Hq, int Hkv, int N, int d, int causal, int window, int num_sms) {
  const int BHk = B * Hkv;
  const int T = (N + kTile - 1) / kTile;
  const int G = Hq / Hkv;
  if (window > 0 || num_sms < 1) return BHk;
  const double ws = (double)N * d * (8.0 * G + 4.0);
  const int kb_l2 = std::max(1, (int)(80.0 * 1024.0 * 1024.0 / ws));
  // Work of one (b, kv head) in query-tile iterations, over its longest item's: (T + 1) / 2
  // causal, T non-causal.
  const double ratio = causal ? (T + 1) / 2.0 : (double)T;
  const int kb_tail = (int)std::ceil(1.4 * num_sms / ratio);
  if (kb_tail >= BHk) return BHk;
  // As many bands as the tail margin allows, but no more than it takes to fit the L2 budget;
  // fewer if the last (narrower) band would miss the margin.
  const int nb_l2 = (BHk + kb_l2 - 1) / kb_l2;
  for (int nb = std::min(nb_l2, BHk / kb_tail); nb > 1; --nb) {
    const int kb = (BHk + nb - 1) / nb;
    if (kb >= kb_tail && BHk - (nb - 1) * kb >= kb_tail) return kb;
  }
  return BHk;
}

template <int D>
static cudaError_t launch_bwd_t(const BwdLaunch& a, int stages) {
  const int T = (a.N + kTile - 1) / kTile;
  const int Npad = T * kTile;
  const long long rows = (long long)a.B * a.Hq * Npad;
  if (stages & kBwdPrepare) {
    const long long threads = rows * (D / 8);
    const unsigned blocks = (unsigned)((threads + 255) / 256);
    fa_bwd_pre_kernel<D><<<blocks, 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(a.o), static_cast<const __nv_bfloat16*>(a.dout), a.lse, a.dq_acc,
        a.delta, a.lse2, a.next_item, a.N, Npad, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdCompute) {
    constexpr int smem = BwdSmem<D>::kAlloc;
    static_assert(smem <= 232448, "backward shared memory exceeds the 227 KB per-CTA limit");
    auto kern = a.window > 0 ? fa_bwd_main_kernel<D, true> : fa_bwd_main_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    BwdParams p;
    p.dk = static_cast<__nv_bfloat16*>(a.dk);
    p.dv = static_cast<__nv_bfloat16*>(a.dv);
    p.delta = a.delta;
    p.lse2 = a.lse2;
    p.status = a.status;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.N = a.N;
    p.Npad = Npad;
    p.causal = a.causal;
    p.num_tiles = T;
    p.window = a.window;
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;
    p.band = bwd_band(a.B, a.Hq, a.Hkv, a.N, D, a.causal, a.window, a.num_sms);
    p.num_items = a.B * a.Hkv * T;
    p.next_item = a.next_item;
    // Persistent: one CTA per SM (fewer if there are fewer items).
    const long long grid = std::min<long long>(p.num_items, a.num_sms);
    kern<<<(unsigned)grid, kBwdThreads, smem, a.stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, *a.tm_dq, *a.tm_dk,
                                                          *a.tm_dv, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (stages & kBwdFinalize) {
    const long long n_vec4 = (long long)a.B * a.Hq * a.N * D / 4;
    const long long want = (n_vec4 + 255) / 256;
    const unsigned blocks = (unsigned)(want < 152 * 32 ? want : 152 * 32);
    fa_bwd_dq_kernel<D><<<blocks, 256, 0, a.stream>>>(a.dq_acc, static_cast<__nv_bfloat16*>(a.dq), a.N, Npad,
                                                      n_vec4, a.scale);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

cudaError_t launch_bwd(const BwdLaunch& a, int stages) {
  if (a.d == 128) return launch_bwd_t<128>(a, stages);
  return launch_bwd_t<64>(a, stages);
}

}  // namespace fa
