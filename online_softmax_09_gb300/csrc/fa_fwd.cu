// fa_fwd.cu -- forward pass of exact softmax attention on sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, query head):
//   warp 4      TMA producer: Q once, then K_j / V_j tiles into an NS-stage ring.
//   warp 5      MMA issuer (one thread) and TMEM owner: S_j = Q K_j^T (smem x smem -> TMEM),
//               O += P_j V_j (P from TMEM, V from smem -> TMEM).
//   warps 0-3   softmax warpgroup, one thread per query row: running max m and sum l
//               ("FlashAttention Implementation > How FlashAttention Uses Tiling", "The Running
//               Statistics"), correction exp(m_old - m_new) applied to l and to the output
//               accumulator in TMEM ("Why the Correction Factor Works"), P = exp(S - m) written
//               back to TMEM as bf16, and the epilogue O = acc / l, LSE = m + ln l
//               ("LLM Architecture Refresh [3]", section 4).
// Causal: key tiles after the query tile are never loaded or computed (same post, section
// 7); the diagonal tile and a ragged last tile are masked element-wise.
//
// TMEM columns: S/P double buffer at [0,128) and [128,256); O accumulator at [256, 256+D).
// The running max is kept in base-2 units (scores scaled by scale*log2 e) so P uses the
// hardware exp2. The max is the true running max: l and O are rescaled whenever a tile raises
// it, so the largest weight of each row is exactly 1 and loses nothing to bf16 rounding.
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  unsigned long long* counters;
  uint32_t* status;
  int B, Hq, Hkv, N, causal;
  int num_tiles;     // ceil(N / 128): query tiles per head == key tiles per head
  float scale_log2;  // scale * log2(e)
};

template <int D, int NS>
struct FwdSmem {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + NS * kTileBytes;
  static constexpr int kBar = kV + NS * kTileBytes;
  // mbarrier indices
  static constexpr int bQ = 0;
  static constexpr int bKFull = 1;
  static constexpr int bVFull = bKFull + NS;
  static constexpr int bKVEmpty = bVFull + NS;
  static constexpr int bSFull = bKVEmpty + NS;  // 2
  static constexpr int bPFull = bSFull + 2;     // 2
  static constexpr int bOFull = bPFull + 2;
  static constexpr int bDrain = bOFull + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
};

constexpr int kFwdThreads = 192;
constexpr uint32_t kTmemCols = 512;

template <int D, int NS>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdSmem<D, NS>;
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

  // Work item. Causal tiles are issued longest first: blockIdx 0.. take the last query tile.
  const int BH = p.B * p.Hq;
  const int rank = blockIdx.x / BH;
  const int bh = blockIdx.x - rank * BH;
  const int q_tile = p.causal ? (p.num_tiles - 1 - rank) : rank;
  const int b = bh / p.Hq;
  const int hq = bh - b * p.Hq;
  const int kv_z = b * p.Hkv + hq / (p.Hq / p.Hkv);
  const int q0 = q_tile * kTile;
  const int n_kv = p.causal ? (q_tile + 1) : p.num_tiles;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::bQ), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(L::bKFull + s), 1);
      mbar_init(bar(L::bVFull + s), 1);
      mbar_init(bar(L::bKVEmpty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(L::bSFull + i), 1);
      mbar_init(bar(L::bPFull + i), 128);
    }
    mbar_init(bar(L::bOFull), 1);
    mbar_init(bar(L::bDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO = tmem + 256;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      constexpr uint32_t kBytes = L::kTileBytes;
      mbar_expect_tx(bar(L::bQ), kBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tma_load_3d(sQ + c * 16384, &tm_q, bar(L::bQ), c * 64, q0, bh);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % NS;
        if (!mbar_wait(bar(L::bKVEmpty + s), ((j / NS) & 1) ^ 1, ctl)) break;
        const uint32_t k_dst = sK + s * L::kTileBytes;
        const uint32_t v_dst = sV + s * L::kTileBytes;
        mbar_expect_tx(bar(L::bKFull + s), kBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(k_dst + c * 16384, &tm_k, bar(L::bKFull + s), c * 64, j * kTile, kv_z);
        mbar_expect_tx(bar(L::bVFull + s), kBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(v_dst + c * 16384, &tm_v, bar(L::bVFull + s), c * 64, j * kTile, kv_z);
        issued = j + 1;
      }
      if (*abort_flag) {  // let every copy still in flight land before shared memory is freed
        drain_wait(bar(L::bQ), 0);
        for (int j = issued > NS ? issued - NS : 0; j < issued; ++j) {
          drain_wait(bar(L::bKFull + j % NS), (j / NS) & 1);
          drain_wait(bar(L::bVFull + j % NS), (j / NS) & 1);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      auto issue_s = [&](int t) -> bool {
        const int s = t % NS;
        if (!mbar_wait(bar(L::bKFull + s), (t / NS) & 1, ctl)) return false;
        tc_fence_after();
        const uint32_t k_base = sK + s * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // K-major, 128B swizzle: 64-element column blocks 16 KB apart, 16 elements = 32 B.
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tS[t & 1], sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(k_base + off, 16, 1024),
                 idS, kk > 0);
        }
        mma_commit(bar(L::bSFull + (t & 1)));
        return true;
      };
      bool ok = mbar_wait(bar(L::bQ), 0, ctl);
      if (ok) {
        tc_fence_after();
        ok = issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv && !issue_s(j + 1)) break;
        const int s = j % NS;
        if (!mbar_wait(bar(L::bPFull + (j & 1)), (j >> 1) & 1, ctl)) break;
        if (!mbar_wait(bar(L::bVFull + s), (j / NS) & 1, ctl)) break;
        tc_fence_after();
        const uint32_t v_base = sV + s * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          // V as the MN-major B operand: 16 keys = 2 swizzle atoms of 8 rows x 128 B.
          mma_ts(tO, tS[j & 1] + kk * 8, sdesc_sw128(v_base + kk * 2048, 16384, 1024), idO,
                 (j > 0 || kk > 0));
        }
        mma_commit(bar(L::bKVEmpty + s));
        mma_commit(bar(L::bOFull));
      }
      if (*abort_flag) {  // wait for issued MMAs before tensor memory is released
        mma_commit(bar(L::bDrain));
        drain_wait(bar(L::bDrain), 0);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroup
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int row = q0 + threadIdx.x;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY;
    float l_run = 0.f;
    uint32_t n_rescaled = 0;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      if (!mbar_wait_warp(bar(L::bSFull + sb), (j >> 1) & 1, ctl)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tS[sb] + lane_off;
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(t_row + c * 32, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(sr[c]);
      const int kv0 = j * kTile;
      if ((p.causal && j == q_tile) || kv0 + kTile > p.N) {
        const int lim = min(p.N - 1, p.causal ? row : p.N - 1) - kv0;  // last visible column
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i > lim) sr[c][i] = 0xff800000u;  // -inf
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sr[c][i]));
      // Running max in base-2 units; correction exp(m_old - m_new) (0 on the first tile).
      const float m_new = fmaxf(m_run, mx * sl2);
      const float corr = (m_new > m_run) ? ex2(m_run - m_new) : 1.f;
      if (j > 0 && m_new > m_run && row < p.N) ++n_rescaled;
      m_run = m_new;
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      float sum = 0.f;
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[c][i]), sl2, -m_use));
          const float p1 = ex2(fmaf(__uint_as_float(sr[c][i + 1]), sl2, -m_use));
          sum += p0 + p1;
          pk[c >> 1][(c & 1) * 16 + (i >> 1)] = pack_bf16(p0, p1);
        }
      l_run = l_run * corr + sum;
      tmem_st32(t_row, pk[0]);
      tmem_st32(t_row + 32, pk[1]);
      if (j > 0) {
        // Wait for O += P_{j-1} V_{j-1}. Waiting at every tile keeps this warp's view of the
        // barrier's phase exact; the wait overlaps the tail of that MMA only.
        if (!mbar_wait_warp(bar(L::bOFull), (j - 1) & 1, ctl)) {
          ok = false;
          break;
        }
        if (__any_sync(0xffffffffu, corr != 1.f)) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tmem_st32(tO + lane_off + c * 32, o);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(L::bPFull + sb));
    }
    // ---------------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait_warp(bar(L::bOFull), (n_kv - 1) & 1, ctl);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l_run;
      const size_t row_off = ((size_t)bh * p.N + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_ld_wait(o);
        uint4 w[4];
        uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          wp[i] = pack_bf16(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
        if (row < p.N) {
          uint4* dst = reinterpret_cast<uint4*>(p.o + row_off + c * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = w[i];
        }
      }
      if (row < p.N) p.lse[(size_t)bh * p.N + row] = (m_run + lg2(l_run)) * 0.6931471805599453f;
    }
    if (p.counters != nullptr) {
      unsigned int r = n_rescaled;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
      if (lane == 0 && r) atomicAdd(&p.counters[2], (unsigned long long)r);
      if (threadIdx.x == 0) {
        atomicAdd(&p.counters[0], (unsigned long long)n_kv);
        atomicAdd(&p.counters[1], (unsigned long long)(p.num_tiles - n_kv));
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int NS>
static cudaError_t launch_fwd_t(const FwdLaunch& a, const FwdParams& p) {
  constexpr int smem = FwdSmem<D, NS>::kAlloc;
  static_assert(smem <= 232448, "forward shared memory exceeds the 227 KB per-CTA limit");
  cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, NS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.num_tiles * p.B * p.Hq;
  fa_fwd_kernel<D, NS><<<(unsigned)grid, kFwdThreads, smem, a.stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdLaunch& a) {
  FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.counters = a.counters;
  p.status = a.status;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.N = a.N;
  p.causal = a.causal;
  p.num_tiles = (a.N + kTile - 1) / kTile;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  if (a.d == 128) return launch_fwd_t<128, 2>(a, p);
  return launch_fwd_t<64, 4>(a, p);
}

}  // namespace fa
