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
//      zeroes the fp32 dQ accumulator.                                         (HBM-bound)
//   2. main: one CTA per (batch, kv head, 128-key tile). It keeps K_n and V_n in shared
//      memory and the dK, dV accumulators in TMEM, and loops over the G query heads of its
//      group and their query tiles (causal: from the diagonal tile on). Per query tile i:
//        softmax warps (thread = key row): P_i^T = 2^(S_i^T scale log2e - LSE2), bf16 -> TMEM
//        MMA  dV += P_i^T dO_i ;  dP_i^T = V_n dO_i^T ;  S_{i+1}^T = K_n Q_{i+1}^T
//        softmax warps: dS_i^T = P_i^T (dP_i^T - delta), bf16 -> shared memory
//        MMA  dQ_i = dS_i K_n  (into the dP^T columns, now free) ;  dK += dS_i^T Q_i
//        drain warps (thread = query row): dQ_i TMEM -> shared memory -> bulk tensor
//        reduction (add) into the fp32 workspace accumulator.
//      The next tile's S^T is computed while the softmax warps work on dS_i, and its P while
//      the dQ and dK MMAs run, so the tensor core does not wait for the softmax warps. The one
//      shared-memory copy of dS serves both of its MMAs (MN-major A of dQ, K-major A of dK),
//      and dQ goes first so that its drain overlaps the dK MMA. CTAs are launched in bands of
//      (batch, kv head) pairs, key tile by key tile within a band, so that the Q, dO and dQ
//      accumulator rows that a band's CTAs share stay in L2 (see bwd_band).
//   3. dQ conversion: dq = bf16(scale * accumulator).
//
// Warp roles of the main kernel: 0-3 and 10-13 softmax/dS (thread = key row; warps 0-3 take
// query columns [0, 64) of every row, warps 10-13 columns [64, 128), so each row's elementwise
// work is split between two warps of the same TMEM lane quarter), then the final dV (0-3) and
// dK (10-13) epilogue; 4 TMA producer, 5 MMA issuer (the whole warp runs the loop, one elected
// lane issues) and TMEM owner, 6-9 dQ drain.
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
                                                         int N, int Npad, long long rows) {
  constexpr int TPR = D / 8;  // threads per row, 8 elements (16 bytes) each
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long r = gt / TPR;  // row of the padded [B*Hq][Npad] grid
  const int part = (int)(gt % TPR);
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
  float* dq_acc;
  const float* delta;
  const float* lse2;
  uint32_t* status;
  int B, Hq, Hkv, N, Npad, causal, num_tiles;
  int window;  // > 0: causal sliding window of this many keys
  float scale, scale_log2;
  int band;  // (b, kv head) pairs per launch band; B * Hkv for a single band
};

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
  // dQ staging for the bulk reductions: 4 drain warps x 2 buffers x 32 rows x 128 bytes.
  static constexpr int kDQ = kDS + (kAliasDS ? 0 : kTile * kTile * 2);
  static constexpr int kBar = kDQ + 4 * 2 * 32 * 128;
  enum {
    bKV = 0,
    bQFull = 1,       // 2
    bDOFull = 3,      // 2
    bStageEmpty = 5,  // 2
    bSFull = 7,
    bDPFull,
    bPReady,
    bSmemDS,
    bDVDone,  // dV_i has finished reading dO_i (whose slot then takes dS_i)
    bDQFull,
    bDQFree,
    bFinal,
    bDrain,
    kNumBars
  };
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  // No alignment slack: the kernel uses no static shared memory, so the dynamic window starts
  // on a 1024-byte boundary; the kernel checks this and stops (status 2) if it ever does not.
  static constexpr int kAlloc = kBytes;
  static_assert(kStageBytes % 1024 == 0 && kStage0 % 1024 == 0 && kDS % 1024 == 0 && kDQ % 1024 == 0,
                "1024-byte alignment");
};

constexpr int kBwdThreads = 448;
// CTAs of at most this many query tiles store dK and dV with bulk tensor stores (see the epilogue).
constexpr int kBwdStoreViaTmaMaxIter = 32;
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

  // Work item: key tile n of kv head (b, hkv). CTAs are numbered band by band (p.band
  // consecutive (b, kv head) pairs, the last band possibly narrower) and key tile by key tile
  // within a band, so a band's causal tiles with the most query tiles start first and its
  // Q, dO and dQ accumulator rows stay in L2 while its CTAs run.
  const int BHk = p.B * p.Hkv;
  const int per_band = p.band * p.num_tiles;
  const int band_i = blockIdx.x / per_band;
  const int first = band_i * p.band;
  const int width = min(p.band, BHk - first);
  const int local = blockIdx.x - band_i * per_band;
  const int n = local / width;
  const int bhk = first + (local - n * width);
  const int b = bhk / p.Hkv;
  const int hkv = bhk - b * p.Hkv;
  const int G = p.Hq / p.Hkv;
  // Query tiles that see key tile n: from the diagonal (causal) to, with a sliding window, the
  // tile of the last query within `window` of the tile's last key.
  const int i0 = p.causal ? n : 0;
  const int i_end = kWin ? min(p.num_tiles, (n * kTile + kTile - 1 + p.window - 1) / kTile + 1) : p.num_tiles;
  const int n_i = i_end - i0;
  const int n_iter = G * n_i;
  auto item = [&](int it, int& hq, int& i) {
    const int g = it / n_i;
    hq = hkv * G + g;
    i = i0 + (it - g * n_i);
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::bKV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(L::bQFull + s), 1);
      mbar_init(bar(L::bDOFull + s), 1);
      mbar_init(bar(L::bStageEmpty + s), 1);
    }
    mbar_init(bar(L::bSFull), 1);
    mbar_init(bar(L::bDPFull), 1);
    mbar_init(bar(L::bPReady), 256);
    mbar_init(bar(L::bSmemDS), 256);
    mbar_init(bar(L::bDQFull), 1);
    mbar_init(bar(L::bDVDone), 1);
    mbar_init(bar(L::bDQFree), 128);
    mbar_init(bar(L::bFinal), 1);
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

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      constexpr uint32_t kTB = L::kTileBytes;
      const int kv_z = b * p.Hkv + hkv;
      mbar_expect_tx(bar(L::bKV), 2 * kTB);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d(sK + c * 16384, &tm_k, bar(L::bKV), c * 64, n * kTile, kv_z);
        tma_load_3d(sV + c * 16384, &tm_v, bar(L::bKV), c * 64, n * kTile, kv_z);
      }
      int issued = 0;
      for (int it = 0; it < n_iter; ++it) {
        const int s = it & 1;
        if (!mbar_wait(bar(L::bStageEmpty + s), ((it >> 1) & 1) ^ 1, ctl)) break;
        int hq, i;
        item(it, hq, i);
        const int qz = b * p.Hq + hq;
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
        issued = it + 1;
      }
      if (*abort_flag) {
        drain_wait(bar(L::bKV), 0);
        for (int it = issued > 2 ? issued - 2 : 0; it < issued; ++it) {
          drain_wait(bar(L::bQFull + (it & 1)), (it >> 1) & 1);
          drain_wait(bar(L::bDOFull + (it & 1)), (it >> 1) & 1);
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
    auto issue_s = [&](int it) {  // S^T = K_n Q_it^T into tS
      const uint64_t q = dSt_k + (uint32_t)((it & 1) * kStage16 + (L::kStQ >> 4));
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tS, dK_k + kmajor(kk), q + kmajor(kk), idSS, kk > 0);
        mma_commit(bar(L::bSFull));
      }
      __syncwarp();
    };
    // dP^T_it = V_n dO_it^T into tdP, once dO_it has landed and dQ_{it-1} has been drained
    // out of these columns.
    auto issue_dp = [&](int it) -> bool {
      if (!mbar_wait_warp(bar(L::bDOFull + (it & 1)), (it >> 1) & 1, ctl)) return false;
      if (it > 0 && !mbar_wait_warp(bar(L::bDQFree), (it - 1) & 1, ctl)) return false;
      tc_fence_after();
      const uint64_t dO = dSt_k + (uint32_t)((it & 1) * kStage16 + (L::kStDO >> 4));
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ss(tdP, dV_k + kmajor(kk), dO + kmajor(kk), idSS, kk > 0);
        mma_commit(bar(L::bDPFull));
      }
      __syncwarp();
      return true;
    };
    bool ok = mbar_wait_warp(bar(L::bKV), 0, ctl) && mbar_wait_warp(bar(L::bQFull), 0, ctl);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      ok = n_iter > 0 && issue_dp(0);
    }
    for (int it = 0; ok && it < n_iter; ++it) {
      const int s = it & 1;
      const uint32_t st16 = (uint32_t)s * kStage16;
      // dV += P^T dO_i  (P^T from TMEM; dO as the MN-major B operand; dO_i waited for dP_i)
      if (!(ok = mbar_wait_warp(bar(L::bPReady), it & 1, ctl))) break;
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
      // S^T of the next query tile (P_i^T in these columns was read by the dV MMA above).
      if (it + 1 < n_iter) {
        if (!(ok = mbar_wait_warp(bar(L::bQFull + (s ^ 1)), ((it + 1) >> 1) & 1, ctl))) break;
        tc_fence_after();
        issue_s(it + 1);
      }
      // dQ_i = dS K_n (dS and K both MN-major in shared memory) into the dP^T columns, first,
      // so the drain starts as early as possible; then dK += dS^T Q_i with the same
      // shared-memory dS as the K-major A operand.
      if (!(ok = mbar_wait_warp(bar(L::bSmemDS), it & 1, ctl))) break;
      tc_fence_after();
      {
        const uint32_t ds16 = L::kAliasDS ? st16 + (L::kStDO >> 4) : 0u;
        const uint64_t ds_mn = (L::kAliasDS ? dSt_mn : dDS_mn) + ds16;
        const uint64_t ds_k = (L::kAliasDS ? dSt_k : dDS_k) + ds16;
        const uint64_t q_mn = dSt_mn + st16 + (L::kStQ >> 4);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ss(tdP, ds_mn + (uint32_t)(kk * (2048 >> 4)), dK_mn + (uint32_t)(kk * (2048 >> 4)), idDQ, kk > 0);
          mma_commit(bar(L::bDQFull));
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_ss(tdK, ds_k + kmajor(kk), q_mn + (uint32_t)(kk * (2048 >> 4)), idTS, (it > 0 || kk > 0));
          mma_commit(bar(L::bStageEmpty + s));
        }
        __syncwarp();
      }
      if (it + 1 < n_iter && !(ok = issue_dp(it + 1))) break;
    }
    if (ok) {
      if (elect_one()) mma_commit(bar(L::bFinal));
      __syncwarp();
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
    const int key = n * kTile + kr;
    const bool key_ok = key < p.N;
    const float sl2 = p.scale_log2;
    bool ok = true;
    uint32_t pk[2][16];  // this warp's half of P_it^T as packed bf16, kept for the dS phase
    // P phase of query tile `it`: P^T = 2^(S^T scale log2e - LSE2), bf16 into TMEM and pk.
    auto p_phase = [&](int it) -> bool {
      const int s = it & 1;
      int hq, i;
      item(it, hq, i);
      const bool diag = p.causal && i == n;
      // Window: query q sees key j only if q - j < window; (i - n) * 128 + q - kr is q - j.
      const bool wmask = kWin && (i - n) * kTile + kTile - 1 >= p.window;
      const float* sl = reinterpret_cast<const float*>(stage_ptr(s) + L::kStL);
      // Queries of this tile that see this key row: [q_lo, q_hi] (none for a key past N).
      const int q_lo = !key_ok ? kTile : (diag ? kr : 0);
      const int q_hi = wmask ? kr + p.window - 1 - (i - n) * kTile : kTile - 1;
      const bool masked = __any_sync(0xffffffffu, q_lo > 0 || q_hi < kTile - 1);  // warp-uniform
      if (!mbar_wait_warp(bar(L::bQFull + s), (it >> 1) & 1, ctl)) return false;
      if (!mbar_wait_warp(bar(L::bSFull), it & 1, ctl)) return false;
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
    ok = n_iter > 0 && p_phase(0);
    for (int it = 0; ok && it < n_iter; ++it) {
      const int s = it & 1;
      const float* sd = reinterpret_cast<const float*>(stage_ptr(s) + L::kStD);
      if (!(ok = mbar_wait_warp(bar(L::bDOFull + s), (it >> 1) & 1, ctl))) break;
      if (!(ok = mbar_wait_warp(bar(L::bDPFull), it & 1, ctl))) break;
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
        if (cc == 0 && !(ok = mbar_wait_warp(bar(L::bDVDone), it & 1, ctl))) break;
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
    // ---------------------------------------------------------------- dV (0-3) / dK (10-13) epilogue
    if (ok) ok = mbar_wait_warp(bar(L::bFinal), 0, ctl);
    if (ok) {
      tc_fence_after();
      const uint32_t src = grp ? tdK : tdV;
      const float mul = grp ? p.scale : 1.f;
      if (n_iter <= kBwdStoreViaTmaMaxIter) {
        // A short CTA's epilogue is a noticeable part of its time: every MMA has completed, so the
        // Q/dO stages are idle, and warp w of the dV (dK) warps writes its 32 key rows, one
        // 64-column chunk at a time, into an 8 KB region of stage 0 (1) in the 128-byte swizzled
        // order; one lane stores each chunk with a bulk tensor store (whole lines; rows past N are
        // not written). Measured +9 % on the backward at N = 512 and +3.6 % at B=4 H=16 N=4096
        // causal. A long CTA stores its rows directly and leaves the TMA unit to its dQ
        // reductions (the same speed on CTAs of 128 query tiles; this build, with both paths,
        // also ran ~2 % faster there than one with the bulk path alone).
        const uint32_t buf = stage(grp) + (uint32_t)(warp & 3) * 8192;
        const int y0 = n * kTile + (warp & 3) * 32;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t a[2][32];
          tmem_ld32(src + lane_off + (2 * c) * 32, a[0]);
          tmem_ld32(src + lane_off + (2 * c + 1) * 32, a[1]);
          tmem_ld_wait(a[0]);
          tmem_ld_wait(a[1]);
          const uint32_t cb = buf + (uint32_t)c * 4096;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t* v = a[g >> 2] + 8 * (g & 3);
            st_shared_v4(cb + (uint32_t)lane * 128 + ((g ^ (lane & 7)) << 4),
                         pack_bf16(__uint_as_float(v[0]) * mul, __uint_as_float(v[1]) * mul),
                         pack_bf16(__uint_as_float(v[2]) * mul, __uint_as_float(v[3]) * mul),
                         pack_bf16(__uint_as_float(v[4]) * mul, __uint_as_float(v[5]) * mul),
                         pack_bf16(__uint_as_float(v[6]) * mul, __uint_as_float(v[7]) * mul));
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && y0 < p.N) {
            tma_store_3d(grp ? &tm_dk : &tm_dv, cb, c * 64, y0, b * p.Hkv + hkv);
            bulk_commit_group();
          }
        }
        if (lane == 0) bulk_wait_read_all();  // the stores have read their shared memory
      } else {
        const size_t row_off = ((size_t)(b * p.Hkv + hkv) * p.N + key) * D;
        __nv_bfloat16* dst_base = grp ? p.dk : p.dv;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t a[32];
          tmem_ld32(src + lane_off + c * 32, a);
          tmem_ld_wait(a);
          uint4 w[4];
          uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            wp[j] = pack_bf16(__uint_as_float(a[2 * j]) * mul, __uint_as_float(a[2 * j + 1]) * mul);
          if (key_ok) {
            uint4* dst = reinterpret_cast<uint4*>(dst_base + row_off + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = w[j];
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ dQ drain warps 6-9
    // Each warp owns 32 query rows (its TMEM lane quarter). 32 columns at a time, the warp
    // stages its 32 x 32 fp32 block of dQ_i in shared memory (128-byte swizzled: 16-byte granule
    // g of row r at g ^ (r mod 8)) and one lane adds it into the workspace accumulator with a
    // bulk tensor reduction. Warps never wait for one another.
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t stage_buf = sbase + L::kDQ + (uint32_t)(warp & 3) * 8192;
    for (int it = 0; it < n_iter; ++it) {
      int hq, i;
      item(it, hq, i);
      if (!mbar_wait_warp(bar(L::bDQFull), it & 1, ctl)) break;
      tc_fence_after();
      const int row0 = (b * p.Hq + hq) * p.Npad + i * kTile + (warp & 3) * 32;
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

// (b, kv head) pairs per launch band. Bands shrink the set of heads whose Q, dO and fp32 dQ
// accumulator rows the resident CTAs share: as many bands as keep each band's work per SM at
// least 1.4 times its longest CTA (whose G * T query tiles would otherwise end alone; a
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
  // Work of one (b, kv head) in query-tile iterations, over its longest CTA's: (T + 1) / 2
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
        a.delta, a.lse2, a.N, Npad, rows);
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
    p.dq_acc = a.dq_acc;
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
    const long long grid = (long long)a.B * a.Hkv * T;
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
