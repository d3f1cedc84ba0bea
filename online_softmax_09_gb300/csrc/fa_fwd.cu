// fa_fwd.cu -- forward pass of exact softmax attention on sm_103a.
//
// Persistent kernel: one CTA per SM walks a list of work items (longest first for causal).
// An item is two 128-row query tiles (256 consecutive rows) of one (batch, query head); both
// tiles share every K/V tile loaded. The next item's Q loads and score MMAs start while the
// previous item's epilogue is still writing O. Roles:
//   warp 8      TMA producer: Q0, Q1 once, then K_j into an NK-stage ring and V_j into an
//               NV-stage ring.
//   warp 9      MMA issuer and TMEM owner: the whole warp runs the issue loop (warp-uniform
//               indices and descriptors) and one elected lane issues. Issue order per key tile j:
//                 O0 += P0_j V_j, S0_{j+1} = Q0 K_{j+1}^T, O1 += P1_j V_j, S1_{j+1} = Q1 K_{j+1}^T
//               so that while one softmax warpgroup turns S into P, the tensor core works on
//               the other tile (separate-P mode below: both S_{j+1} first, then both P.V).
//   warps 0-3   softmax warpgroup of tile 0, warps 4-7 of tile 1: one thread per query row,
//               running max m and sum l ("FlashAttention Implementation > How FlashAttention
//               Uses Tiling", "The Running Statistics"), correction exp(m_old - m_new) applied
//               to l and to the output accumulator in TMEM ("Why the Correction Factor
//               Works"), P = exp(S - m) written back to TMEM as bf16 over the S columns, and
//               the epilogue O = acc / l, LSE = m + ln l ("LLM Architecture Refresh [3]",
//               section 4), O leaving through a per-warp shared buffer and bulk tensor stores.
// Causal: key tiles after a query tile are never loaded or computed (same post, section 7);
// the diagonal tile and a ragged last tile are masked element-wise.
//
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O0 [256,256+D), O1 [384,384+D).
// Separate-P mode (D = 64, where each O region leaves 64 columns free): P_t lives in
// [320,384) / [448,512) instead of over S_t. The next score MMA of a tile then needs only that
// its softmax warps have read S_t into registers (bSFree), not that P.V has consumed P, so it
// leaves the tile's critical loop, which becomes the softmax alone; bPFree (a commit after each
// P.V) tells the softmax warps when P_t may be rewritten and O_t rescaled.
// The running max is kept in base-2 units (scores scaled by scale*log2 e) so P uses the
// hardware exp2. P is taken against a reference max m_ref that follows the true running max
// lazily: a warp rescales l and O (and moves m_ref of its rows to their true max) only when one
// of its rows' max has risen more than kRescaleLog2 above m_ref; otherwise weights up to
// 2^kRescaleLog2 are used as they are. Any reference gives the same softmax (the correction
// factors cancel between O and l), so this only skips the O pass on most tiles. A weight above 1
// is generally not a bf16 number, and the P.V MMA consumes it rounded while l holds it exact: for
// a row dominated by one key that mismatch would show in O at bf16's relative precision. So each
// tile's largest weight is recomputed exactly as pass 2 computes it, its bf16 rounding error is
// accumulated in e (rescaled like l), and O is divided by l + e; LSE keeps the fp32 l.
// Each row's S is read from TMEM once into registers (128 values per thread).
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  float* o_part;    // split-KV partial outputs [num_splits][B*Hq][N][D] fp32 (split mode only)
  float* lse_part;  // split-KV partial LSE (natural log) [num_splits][B*Hq][N] (split mode only)
  unsigned long long* counters;
  uint32_t* status;
  int B, Hq, Hkv, N, causal;
  int window;        // > 0: key j visible to query i only if i - window < j (causal as well)
  int num_tiles;     // ceil(N / 128): query tiles per head == key tiles per head
  int num_pairs;     // ceil(num_tiles / 2): query-tile pairs per head
  int num_splits;    // key-tile ranges per pair (1 = no split)
  int split_len;     // key tiles per split
  int num_items;     // num_pairs * B * Hq * num_splits
  float scale_log2;  // scale * log2(e)
};

// One work item: query tiles 2*pair and 2*pair+1 of head bh over one range of key tiles. Query
// tile t visits key tiles [j0 + a[t], j0 + b[t]) (none when a[t] == b[t]): causal tiles stop at
// the diagonal, a sliding window starts at the first key tile any row of the tile can see, and
// a split keeps one of num_splits consecutive ranges of split_len key tiles. Items are
// numbered so that, for causal attention, the longest pairs come first.
struct FwdItem {
  int bh, kv_z, qt0, j0, n_max, split;
  int a[2], b[2];
  bool exists[2];  // the query tile has rows (qt < num_tiles)
};

// Item of this CTA in round r: items are dealt in rounds of gridDim.x, snake order (CTA c gets
// item r*G + c in even rounds and r*G + G-1-c in odd rounds), which balances the linearly
// decreasing causal item lengths across CTAs. Returns -1 past the end.
__device__ __forceinline__ int fwd_item_index(int r, int num_items) {
  const int G = gridDim.x;
  const int k = r * G + ((r & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
  return k < num_items ? k : -1;
}

// Splits that hold key tiles for query tile qt: the first ceil(hi / split_len) of them, hi being
// the tile's end of visible keys (the diagonal when causal). Split mode has no window.
__host__ __device__ __forceinline__ int split_count(int qt, const FwdParams& p) {
  const int hi = p.causal ? qt + 1 : p.num_tiles;
  return min(p.num_splits, (hi + p.split_len - 1) / p.split_len);
}

template <bool kWin, bool kSplit>
__device__ __forceinline__ FwdItem fwd_item(int k, const FwdParams& p) {
  FwdItem it;
  const int BH = p.B * p.Hq;
  it.split = kSplit ? k % p.num_splits : 0;
  const int kk = kSplit ? k / p.num_splits : k;
  const int rank = kk / BH;
  it.bh = kk - rank * BH;
  const int pair = p.causal ? (p.num_pairs - 1 - rank) : rank;
  const int b = it.bh / p.Hq;
  const int hq = it.bh - b * p.Hq;
  it.kv_z = b * p.Hkv + hq / (p.Hq / p.Hkv);
  it.qt0 = 2 * pair;
  int lo[2], hi[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = it.qt0 + t;
    it.exists[t] = qt < p.num_tiles;
    lo[t] = hi[t] = 0;
    if (!it.exists[t]) continue;
    hi[t] = p.causal ? qt + 1 : p.num_tiles;
    lo[t] = kWin ? max(0, qt * kTile - p.window + 1) / kTile : 0;
    if (kSplit) {
      lo[t] = max(lo[t], it.split * p.split_len);
      hi[t] = min(hi[t], (it.split + 1) * p.split_len);
    }
    if (hi[t] < lo[t]) hi[t] = lo[t];
  }
  it.j0 = 0;
  bool any = false;
#pragma unroll
  for (int t = 0; t < 2; ++t)
    if (hi[t] > lo[t]) {
      it.j0 = any ? min(it.j0, lo[t]) : lo[t];
      any = true;
    }
  it.n_max = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    it.a[t] = (hi[t] > lo[t]) ? lo[t] - it.j0 : 0;
    it.b[t] = (hi[t] > lo[t]) ? hi[t] - it.j0 : 0;
    it.n_max = max(it.n_max, it.b[t]);
  }
  return it;
}

template <int D, int NK, int NV>
struct FwdSmem {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQ = 0;  // Q0, Q1
  static constexpr int kK = kQ + 2 * kTileBytes;
  static constexpr int kV = kK + NK * kTileBytes;
  // O staging for the epilogue's bulk tensor stores: one 4 KB buffer (32 rows x 64 columns,
  // 128-byte swizzled) per softmax warp.
  static constexpr int kOStage = kV + NV * kTileBytes;
  static constexpr int kBar = kOStage + 8 * 4096;
  // mbarrier indices
  static constexpr int bQ = 0;                // 2
  static constexpr int bKFull = bQ + 2;       // NK
  static constexpr int bKEmpty = bKFull + NK; // NK
  static constexpr int bVFull = bKEmpty + NK; // NV
  static constexpr int bVEmpty = bVFull + NV; // NV
  static constexpr int bSFull = bVEmpty + NV; // 2 (per tile)
  static constexpr int bPFull = bSFull + 2;   // 2
  static constexpr int bOFull = bPFull + 2;   // 2
  static constexpr int bQEmpty = bOFull + 2;  // 2: Q buffer t no longer read by MMAs
  static constexpr int bOFree = bQEmpty + 2;  // 2: O_t read out by the epilogue
  static constexpr int bSFree = bOFree + 2;   // 2: S_t read into registers (separate-P mode)
  static constexpr int bPFree = bSFree + 2;   // 2: P_t consumed by its P.V (separate-P mode)
  static constexpr int bDrain = bPFree + 2;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
};

constexpr int kFwdThreads = 320;
// A warp rescales when a row's max exceeds its reference by more than this (base 2): weights
// stay below 2^8, far inside fp32 and bf16 range.
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kNegInf = 0xff800000u;

// Maximum of 64 values held in two 32-register chunks (three-input max, 8 partial maxima).
__device__ __forceinline__ float max64(const uint32_t (&a)[32], const uint32_t (&b)[32], float init) {
  float m[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    m[k] = max3f(__uint_as_float(a[k]), __uint_as_float(a[k + 8]), __uint_as_float(a[k + 16]));
    m[k] = max3f(m[k], __uint_as_float(a[k + 24]), __uint_as_float(b[k]));
    m[k] = max3f(m[k], __uint_as_float(b[k + 8]), __uint_as_float(b[k + 16]));
    m[k] = fmaxf(m[k], __uint_as_float(b[k + 24]));
  }
  return max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), max3f(m[6], m[7], init));
}

// Columns outside [lo, lim] (the visible keys of this row within the tile) become -inf.
__device__ __forceinline__ void mask32(uint32_t (&s)[32], int col0, int lo, int lim) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (col0 + i > lim || col0 + i < lo) s[i] = kNegInf;
}

template <int D, int NK, int NV, bool kWin, bool kSplit>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const __grid_constant__ CUtensorMap tm_opart, const FwdParams p) {
  using L = FwdSmem<D, NK, NV>;
  // Separate-P mode (see the TMEM plan above) and the first TMEM column of P_0.
  constexpr bool kSepP = (D == 64);
  constexpr uint32_t kPCol = kSepP ? 256 + 64 : 0;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + L::kQ;
  const uint32_t sK = sbase + L::kK;
  const uint32_t sV = sbase + L::kV;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const Ctl ctl{abort_flag, p.status};
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::bQ + t), 1);
      mbar_init(bar(L::bSFull + t), 1);
      mbar_init(bar(L::bPFull + t), 128);
      mbar_init(bar(L::bOFull + t), 1);
      mbar_init(bar(L::bQEmpty + t), 1);
      mbar_init(bar(L::bOFree + t), 128);
      mbar_init(bar(L::bSFree + t), 128);
      mbar_init(bar(L::bPFree + t), 1);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(bar(L::bKFull + s), 1);
      mbar_init(bar(L::bKEmpty + s), 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(bar(L::bVFull + s), 1);
      mbar_init(bar(L::bVEmpty + s), 1);
    }
    mbar_init(bar(L::bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Persistent CTAs: every role walks the same item sequence (fwd_item_index) and keeps running
  // counts, from which all barrier phases follow.
  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      constexpr uint32_t kBytes = L::kTileBytes;
      uint32_t gk = 0, gv = 0;  // K and V tiles loaded so far
      uint32_t qn[2] = {0, 0};  // Q loads into each buffer so far
      bool ok = true;
      for (int r = 0; ok && r * (int)gridDim.x < p.num_items; ++r) {
        const int k = fwd_item_index(r, p.num_items);
        if (k < 0) continue;
        const FwdItem it = fwd_item<kWin, kSplit>(k, p);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (it.b[t] == it.a[t]) continue;
          if (!(ok = mbar_wait(bar(L::bQEmpty + t), (qn[t] & 1) ^ 1, ctl))) break;
          mbar_expect_tx(bar(L::bQ + t), kBytes);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sQ + t * kBytes + c * 16384, &tm_q, bar(L::bQ + t), c * 64, (it.qt0 + t) * kTile, it.bh);
          ++qn[t];
        }
        for (int j = 0; ok && j < it.n_max; ++j) {
          const uint32_t sk = gk % NK, sv = gv % NV;
          const int jy = (it.j0 + j) * kTile;
          if (!(ok = mbar_wait(bar(L::bKEmpty + sk), ((gk / NK) & 1) ^ 1, ctl))) break;
          mbar_expect_tx(bar(L::bKFull + sk), kBytes);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sK + sk * kBytes + c * 16384, &tm_k, bar(L::bKFull + sk), c * 64, jy, it.kv_z);
          ++gk;
          if (!(ok = mbar_wait(bar(L::bVEmpty + sv), ((gv / NV) & 1) ^ 1, ctl))) break;
          mbar_expect_tx(bar(L::bVFull + sv), kBytes);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sV + sv * kBytes + c * 16384, &tm_v, bar(L::bVFull + sv), c * 64, jy, it.kv_z);
          ++gv;
        }
      }
      if (*abort_flag) {  // let every copy still in flight land before shared memory is freed
        for (int t = 0; t < 2; ++t)
          if (qn[t] > 0) drain_wait(bar(L::bQ + t), (qn[t] - 1) & 1);
        for (uint32_t g = gk > NK ? gk - NK : 0; g < gk; ++g) drain_wait(bar(L::bKFull + g % NK), (g / NK) & 1);
        for (uint32_t g = gv > NV ? gv - NV : 0; g < gv; ++g) drain_wait(bar(L::bVFull + g % NV), (g / NV) & 1);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, so its counters, barrier phases and descriptors are
    // warp-uniform; one elected lane issues each group of MMAs and each commit. (A single-lane
    // loop paced the tensor core: its issue of one MMA took ~85 cycles against the 64 the MMA
    // runs, and each satisfied wait and the loop bookkeeping another ~100.)
    constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
    // Descriptor bases of the Q tiles and the K and V rings; a tile or an MMA step adds its byte
    // offset / 16 to the start-address field (every shared address fits that 14-bit field).
    const uint64_t dQ = sdesc_sw128(sQ, 16, 1024);
    const uint64_t dK = sdesc_sw128(sK, 16, 1024);
    const uint64_t dV = sdesc_sw128(sV, 16384, 1024);
    uint32_t gk = 0, gv = 0;  // K and V tiles consumed so far
    uint32_t qn[2] = {0, 0};  // items in which query tile t was active
    uint32_t pc[2] = {0, 0};  // P.V MMAs issued for tile t
    auto commit = [&](uint32_t b) {
      if (elect_one()) mma_commit(b);
      __syncwarp();
    };
    // S_t = Q_t K^T with K tile number g; `ready`: K tile g's full barrier was already waited
    // on for the other query tile.
    auto issue_s = [&](int t, uint32_t g, bool ready) -> bool {
      const uint32_t sk = g % NK;
      if (!ready && !mbar_wait_warp(bar(L::bKFull + sk), (g / NK) & 1, ctl)) return false;
      tc_fence_after();
      const uint64_t a = dQ + (uint32_t)(t * (L::kTileBytes >> 4));
      const uint64_t bk = dK + sk * (uint32_t)(L::kTileBytes >> 4);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major, 128B swizzle: 64-element column blocks 16 KB apart, 16 elements = 32 B.
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(tmem + 128 * t, a + off, bk + off, idS, kk > 0);
        }
        mma_commit(bar(L::bSFull + t));
      }
      __syncwarp();
      return true;
    };
    // O_t += P_t V with V tile number g. O_t's completion is signalled only after an item's last
    // P.V (for the epilogue): each earlier one is followed by S_t's next score MMA, whose
    // completion (which the softmax warps wait for) implies it.
    auto issue_pv = [&](int t, uint32_t g, bool first, bool last, bool ready) -> bool {
      const uint32_t sv = g % NV;
      if (!mbar_wait_warp(bar(L::bPFull + t), pc[t] & 1, ctl)) return false;
      if (!ready && !mbar_wait_warp(bar(L::bVFull + sv), (g / NV) & 1, ctl)) return false;
      // The first P.V of an item overwrites O_t: the previous item's epilogue must be done.
      if (first && qn[t] > 1 && !mbar_wait_warp(bar(L::bOFree + t), (qn[t] - 2) & 1, ctl)) return false;
      tc_fence_after();
      const uint64_t bv = dV + sv * (uint32_t)(L::kTileBytes >> 4);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          // V as the MN-major B operand: 16 keys = 2 swizzle atoms of 8 rows x 128 B.
          mma_ts(tmem + 256 + 128 * t, tmem + kPCol + 128 * t + kk * 8, bv + (uint32_t)(kk * (2048 >> 4)), idO,
                 (!first || kk > 0));
        }
        if (last) mma_commit(bar(L::bOFull + t));
      }
      __syncwarp();
      ++pc[t];
      return true;
    };
    bool ok = true;
    if constexpr (kSepP) {
      uint32_t sn[2] = {0, 0};  // score MMAs issued for tile t (all items)
      // S_t of K tile g once the softmax warps have read the previous S_t out of its columns.
      auto issue_s_sep = [&](int t, uint32_t g, bool ready) -> bool {
        if (sn[t] > 0 && !mbar_wait_warp(bar(L::bSFree + t), (sn[t] - 1) & 1, ctl)) return false;
        ++sn[t];
        return issue_s(t, g, ready);
      };
      for (int r = 0; ok && r * (int)gridDim.x < p.num_items; ++r) {
        const int k = fwd_item_index(r, p.num_items);
        if (k < 0) continue;
        const FwdItem it = fwd_item<kWin, kSplit>(k, p);
        if (it.n_max == 0) continue;
        bool k_ready = false;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          if (it.b[t] == it.a[t]) continue;
          if (!(ok = mbar_wait_warp(bar(L::bQ + t), qn[t] & 1, ctl))) break;
          ++qn[t];
          tc_fence_after();
          if (it.a[t] == 0) {  // score MMA of the item's first key tile
            if (!(ok = issue_s_sep(t, gk, k_ready))) break;
            k_ready = true;
            if (it.b[t] == 1) commit(bar(L::bQEmpty + t));  // Q_t's last score MMA
          }
        }
        if (!ok) break;
        commit(bar(L::bKEmpty + gk % NK));  // key tile 0 of the item: its score MMAs are issued
        for (int j = 0; ok && j < it.n_max; ++j) {
          // Next scores first (they wait only for S_t to be read), then this step's P.V.
          bool k_next_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (it.a[t] <= j + 1 && j + 1 < it.b[t]) {
              if (!(ok = issue_s_sep(t, gk + j + 1, k_next_ready))) break;
              k_next_ready = true;
              if (j + 2 == it.b[t]) commit(bar(L::bQEmpty + t));
            }
          }
          if (!ok) break;
          if (j + 1 < it.n_max) commit(bar(L::bKEmpty + (gk + j + 1) % NK));
          bool v_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (it.a[t] <= j && j < it.b[t]) {
              if (!(ok = issue_pv(t, gv + j, j == it.a[t], j + 1 == it.b[t], v_ready))) break;
              v_ready = true;
              commit(bar(L::bPFree + t));
            }
          }
          if (!ok) break;
          commit(bar(L::bVEmpty + (gv + j) % NV));
        }
        gk += it.n_max;
        gv += it.n_max;
      }
    } else {
      for (int r = 0; ok && r * (int)gridDim.x < p.num_items; ++r) {
        const int k = fwd_item_index(r, p.num_items);
        if (k < 0) continue;
        const FwdItem it = fwd_item<kWin, kSplit>(k, p);
        if (it.n_max == 0) continue;
        bool k_ready = false;
  #pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!ok) break;
          if (it.b[t] == it.a[t]) continue;
          if (!(ok = mbar_wait_warp(bar(L::bQ + t), qn[t] & 1, ctl))) break;
          ++qn[t];
          tc_fence_after();
          if (it.a[t] == 0) {  // score MMA of the item's first key tile
            if (!(ok = issue_s(t, gk, k_ready))) break;
            k_ready = true;
            if (it.b[t] == 1) commit(bar(L::bQEmpty + t));  // Q_t's last score MMA
          }
        }
        if (!ok) break;
        commit(bar(L::bKEmpty + gk % NK));  // key tile 0 of the item: its score MMAs are issued
        for (int j = 0; ok && j < it.n_max; ++j) {
          bool v_ready = false, k_next_ready = false;
  #pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (it.a[t] <= j && j < it.b[t]) {
              if (!(ok = issue_pv(t, gv + j, j == it.a[t], j + 1 == it.b[t], v_ready))) break;
              v_ready = true;
            }
            if (it.a[t] <= j + 1 && j + 1 < it.b[t]) {
              if (!(ok = issue_s(t, gk + j + 1, k_next_ready))) break;
              k_next_ready = true;
              if (j + 2 == it.b[t]) commit(bar(L::bQEmpty + t));
            }
          }
          if (!ok) break;
          commit(bar(L::bVEmpty + (gv + j) % NV));
          if (j + 1 < it.n_max) commit(bar(L::bKEmpty + (gk + j + 1) % NK));
        }
        gk += it.n_max;
        gv += it.n_max;
      }
    }
    if (*abort_flag) {  // wait for issued MMAs before tensor memory is released
      if (elect_one()) {
        mma_commit(bar(L::bDrain));
        drain_wait(bar(L::bDrain), 0);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;  // query tile of this warpgroup within an item
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 128 * t + lane_off;
    const uint32_t tO = tmem + 256 + 128 * t + lane_off;
    const uint32_t tP = kSepP ? tmem + kPCol + 128 * t + lane_off : tS;  // where P_t is written
    const float sl2 = p.scale_log2;
    const uint32_t o_stage = sbase + L::kOStage + (uint32_t)warp * 4096;  // this warp's O buffer
    uint32_t sc = 0;  // score tiles of this query tile processed so far (all items)
    uint32_t on = 0;  // items of this query tile whose output was completed
    bool ok = true;
    for (int r = 0; ok && r * (int)gridDim.x < p.num_items; ++r) {
      const int k = fwd_item_index(r, p.num_items);
      if (k < 0) continue;
      const FwdItem itm = fwd_item<kWin, kSplit>(k, p);
      if (!(t ? itm.exists[1] : itm.exists[0])) continue;
      const int qt = itm.qt0 + t;
      const int row = qt * kTile + (threadIdx.x & 127);
      const int a_t = t ? itm.a[1] : itm.a[0];
      const int n_kv = (t ? itm.b[1] : itm.b[0]) - a_t;
      const size_t part_row = ((size_t)itm.split * p.B * p.Hq + itm.bh) * p.N + row;
      // This split has no key tile for this query tile: nothing to write, since the merge reads
      // only the splits that hold keys for the tile.
      if (n_kv == 0) continue;
      const int jbase = itm.j0 + a_t;  // absolute index of the first key tile
      float m_run = -INFINITY;  // reference max (base 2) of P, l and O
      float m_hi = -INFINITY;   // true running max (base 2)
      float l_run = 0.f;
      float e_run = 0.f;        // bf16 rounding error of the tile maxima's weights (see above)
      uint32_t n_raised = 0;
      for (int j = 0; j < n_kv; ++j) {
        if (!mbar_wait_warp(bar(L::bSFull + t), (sc + j) & 1, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kv0 = (jbase + j) * kTile;
        // Visible columns of this row within the tile: [lo, lim].
        const bool need_mask = (p.causal && jbase + j == qt) || kv0 + kTile > p.N ||
                               (kWin && kv0 < qt * kTile + kTile - p.window);
        const int lim = min(p.N - 1, p.causal ? row : p.N - 1) - kv0;
        const int lo = kWin ? row - p.window + 1 - kv0 : -kTile;
        // The row's 128 scores, read from TMEM once: four 32-column loads in flight together.
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
        if constexpr (kSepP) {  // S_t's columns may now take the next score MMA
          tc_fence_before();
          mbar_arrive(bar(L::bSFree + t));
        }
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 4; ++c) mask32(sr[c], c * 32, lo, lim);
        }
        const float mx = max64(sr[2], sr[3], max64(sr[0], sr[1], -INFINITY));
        // Reference max in base-2 units, moved to the true max only when some row of the warp
        // has outgrown it by more than kRescaleLog2 (always on the first tile, where
        // m_run = -inf); correction exp(m_old - m_new) (0 on the first tile).
        const float mt = mx * sl2;
        if (j > 0 && mt > m_hi && row < p.N) ++n_raised;  // the true running max rose
        m_hi = fmaxf(m_hi, mt);
        const bool resc = __any_sync(0xffffffffu, m_hi > m_run + kRescaleLog2);
        const float m_new = resc ? m_hi : m_run;
        const float corr = (m_new > m_run) ? ex2(m_run - m_new) : 1.f;
        m_run = m_new;
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        {
          // This tile's largest weight, bit-identical to its value below (same correctly
          // rounded fma and exp2), and the error its bf16 rounding makes in the P.V MMA.
          const float pmx = ex2(fmaf(mx, sl2, -m_use));
          e_run = e_run * corr + (__uint_as_float(pack_bf16(pmx, 0.f) << 16) - pmx);
        }
        if constexpr (kSepP) {
          // The previous P.V of this tile has consumed P_t and updated O_t (before the first
          // tile of an item that is the previous item's last P.V, already complete).
          if (sc + j > 0 && !mbar_wait_warp(bar(L::bPFree + t), (sc + j - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        // P = 2^(S*scale*log2e - m) as bf16 over the S columns (all already in registers), or
        // into P_t's own columns in separate-P mode, and the row sum.
        float2 sum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        const float2 sl2x2 = make_float2(sl2, sl2);
        const float2 negm = make_float2(-m_use, -m_use);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x = fma2(make_float2(__uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1])), sl2x2, negm);
            const float2 pp = make_float2(ex2(x.x), ex2(x.y));
            sum[(i >> 1) & 1] = add2(sum[(i >> 1) & 1], pp);
            pk[i >> 1] = pack_bf16(pp.x, pp.y);
          }
          // P chunk c covers columns [16c, 16c+16) of tP.
          tmem_st16(tP + c * 16, pk);
        }
        // O += P_{j-1} V has completed (it was issued before S_j, whose completion implies it,
        // or, in separate-P mode, bPFree said so); a rescale of O must land before this tile's
        // P.V, which waits for the arrival below.
        if (j > 0 && resc) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 r = mul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                    make_float2(corr, corr));
              o[i] = __float_as_uint(r.x);
              o[i + 1] = __float_as_uint(r.y);
            }
            tmem_st32(tO + c * 32, o);
          }
        }
        l_run = l_run * corr + ((sum[0].x + sum[1].x) + (sum[0].y + sum[1].y));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(L::bPFull + t));
      }
      if (!ok) break;
      // ---------------------------------------------------------------- epilogue
      if (!(ok = mbar_wait_warp(bar(L::bOFull + t), on & 1, ctl))) break;  // the item's last P.V
      ++on;
      sc += n_kv;
      tc_fence_after();
      const float inv_l = 1.f / (l_run + e_run);
      if (kSplit && split_count(qt, p) > 1) {
        // Split mode: the partial output acc / l (fp32) and its LSE, merged later. (A tile whose
        // keys all fall in one split gets its final O and LSE below, as without splits.)
        // The partial rows go out like O below, 32 fp32 columns (a 4 KB box) at a time.
        if (row < p.N) p.lse_part[part_row] = (m_run + lg2(l_run)) * 0.6931471805599453f;
        const int y0 = qt * kTile + (warp & 3) * 32;
        const int zp = itm.split * p.B * p.Hq + itm.bh;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
          if (y0 < p.N) {
            if (lane == 0) bulk_wait_read_all();  // the previous store from this buffer has read it
            __syncwarp();
#pragma unroll
            for (int g = 0; g < 8; ++g)
              st_shared_v4(o_stage + (uint32_t)lane * 128 + ((g ^ (lane & 7)) << 4),
                           __float_as_uint(__uint_as_float(o[4 * g]) * inv_l),
                           __float_as_uint(__uint_as_float(o[4 * g + 1]) * inv_l),
                           __float_as_uint(__uint_as_float(o[4 * g + 2]) * inv_l),
                           __float_as_uint(__uint_as_float(o[4 * g + 3]) * inv_l));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tm_opart, o_stage, c * 32, y0, zp);
              bulk_commit_group();
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bar(L::bOFree + t));
        continue;
      }
      uint4 w[D / 32][4];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait(o);
        uint32_t* wp = reinterpret_cast<uint32_t*>(w[c]);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 r = mul2(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])),
                                make_float2(inv_l, inv_l));
          wp[i] = pack_bf16(r.x, r.y);
        }
      }
      // O_t has been read: the next item's first P.V may overwrite it.
      tc_fence_before();
      mbar_arrive(bar(L::bOFree + t));
      // O leaves through shared memory: the warp writes its 32 rows of one 64-column chunk into
      // its buffer (16-byte granule g of row r at g ^ (r mod 8), the 128-byte swizzle, so the
      // writes are free of bank conflicts) and one lane stores the box with a bulk tensor store,
      // which writes whole lines and leaves out rows past N. Storing each row from its own
      // thread wrote 16 bytes into each of 32 rows per instruction.
      const int y0 = qt * kTile + (warp & 3) * 32;  // this warp's first row
#pragma unroll
      for (int c = 0; c < D / 64 && y0 < p.N; ++c) {  // (a warp whose rows all lie past N stores nothing)
        if (lane == 0) bulk_wait_read_all();  // the previous store from this buffer has read it
        __syncwarp();
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 v4 = w[2 * c + (g >> 2)][g & 3];
          st_shared_v4(o_stage + (uint32_t)lane * 128 + ((g ^ (lane & 7)) << 4), v4.x, v4.y, v4.z, v4.w);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tm_o, o_stage, c * 64, y0, itm.bh);
          bulk_commit_group();
        }
      }
      if (row < p.N) p.lse[(size_t)itm.bh * p.N + row] = (m_run + lg2(l_run)) * 0.6931471805599453f;
      if (!kSplit && p.counters != nullptr) {
        unsigned int r = n_raised;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
        if (lane == 0 && r) atomicAdd(&p.counters[2], (unsigned long long)r);
        if ((threadIdx.x & 127) == 0) {
          atomicAdd(&p.counters[0], (unsigned long long)n_kv);
          atomicAdd(&p.counters[1], (unsigned long long)(p.num_tiles - n_kv));
        }
      }
    }
  }

  // Every O store has read its shared memory before the CTA releases it (the stores' writes to
  // global memory complete by the end of the kernel).
  if (warp < 8 && lane == 0) bulk_wait_read_all();

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int NK, int NV, bool kWin, bool kSplit>
static cudaError_t launch_fwd_mode(const FwdLaunch& a, const FwdParams& p) {
  constexpr int smem = FwdSmem<D, NK, NV>::kAlloc;
  static_assert(smem <= 232448, "forward shared memory exceeds the 227 KB per-CTA limit");
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, NK, NV, kWin, kSplit>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = p.num_items < a.num_sms ? p.num_items : a.num_sms;
  fa_fwd_kernel<D, NK, NV, kWin, kSplit><<<grid, kFwdThreads, smem, a.stream>>>(*a.tm_q, *a.tm_k, *a.tm_v,
                                                                                  *a.tm_o, *a.tm_opart, p);
  return cudaGetLastError();
}

// Plain, sliding-window and split-KV forwards are separate instantiations, so the plain kernel
// carries none of the other modes' index arithmetic.
template <int D, int NK, int NV>
static cudaError_t launch_fwd_t(const FwdLaunch& a, const FwdParams& p) {
  if (p.num_splits > 1) return launch_fwd_mode<D, NK, NV, false, true>(a, p);
  if (p.window > 0) return launch_fwd_mode<D, NK, NV, true, false>(a, p);
  return launch_fwd_mode<D, NK, NV, false, false>(a, p);
}

// Split-KV merge ("LLM Architecture Refresh [3]", section 3, "Partial softmaxes compose"): per
// row, O = sum_s w_s O_s / sum_s w_s and LSE = m + ln(sum_s w_s) with w_s = exp(LSE_s - m),
// m = max_s LSE_s, over the splits that hold keys for the row's tile. Rows whose keys all fall in
// one split were written in full by the attention kernel. One thread per 4 columns of a row.
template <int D>
__global__ void __launch_bounds__(256) fa_split_merge_kernel(const float* __restrict__ o_part,
                                                            const float* __restrict__ lse_part,
                                                            __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                            long long rows, const FwdParams p) {
  const long long gt = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = gt / (D / 4);
  const int col = (int)(gt - row * (D / 4)) * 4;
  if (row >= rows) return;
  const int ns = split_count((int)(row % p.N) / kTile, p);
  if (ns <= 1) return;
  float m = -INFINITY;
  for (int s = 0; s < ns; ++s) m = fmaxf(m, lse_part[(size_t)s * rows + row]);
  float wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < ns; ++s) {
    const float w = __expf(lse_part[(size_t)s * rows + row] - m);
    const float4 v = *reinterpret_cast<const float4*>(o_part + ((size_t)s * rows + row) * D + col);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
    wsum += w;
  }
  const float inv = 1.f / wsum;
  uint2 packed;
  packed.x = pack_bf16(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(o + row * D + col) = packed;
  if (col == 0) lse[row] = m + __logf(wsum);
}

cudaError_t launch_fwd(const FwdLaunch& a) {
  FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.window = a.window;
  p.counters = a.counters;
  p.status = a.status;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.N = a.N;
  p.causal = a.causal;
  p.num_tiles = (a.N + kTile - 1) / kTile;
  p.num_pairs = (p.num_tiles + 1) / 2;
  p.num_splits = a.num_splits > 1 ? a.num_splits : 1;
  p.split_len = (p.num_tiles + p.num_splits - 1) / p.num_splits;
  p.num_items = p.num_pairs * a.B * a.Hq * p.num_splits;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  // K and V rings: two stages each at d = 128 (a third K stage measured no faster, and its 32 KB
  // now hold the O staging buffers), four each at d = 64.
  cudaError_t e = (a.d == 128) ? launch_fwd_t<128, 2, 2>(a, p) : launch_fwd_t<64, 4, 4>(a, p);
  if (e != cudaSuccess || p.num_splits == 1) return e;
  const long long rows = (long long)a.B * a.Hq * a.N;
  const long long threads = rows * (a.d / 4);
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (a.d == 128)
    fa_split_merge_kernel<128><<<blocks, 256, 0, a.stream>>>(a.o_part, a.lse_part, p.o, a.lse, rows, p);
  else
    fa_split_merge_kernel<64><<<blocks, 256, 0, a.stream>>>(a.o_part, a.lse_part, p.o, a.lse, rows, p);
  return cudaGetLastError();
}

}  // namespace fa
