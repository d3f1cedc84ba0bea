// fa_softmax.cu -- row-wise softmax by the online normaliser, on sm_103a.
//
// For each row x of length n: a running max m and running sum l are carried over the elements
// ("LLM Architecture Refresh [3]: Flash Attention Is Exact", section 2, "Online softmax: the one
// idea": m_new = max(m_old, x), l_new = l_old * exp(m_old - m_new) + exp(x - m_new)), partial
// (m, l) pairs of different threads are merged by the same rebasing (section 3, "Partial
// softmaxes compose"), and then p = exp(x - m) / l, LSE = m + ln l.
//
// Rows of up to 2048 elements (n a multiple of 4): one warp per row, values in registers (see
// fa_softmax_warp_rows_kernel). Otherwise one CTA of 256 threads per row; thread t owns the
// float4 groups t, t+256, ... . Rows of up to kCached = 8192 elements stay in registers between
// the two phases (one HBM read and one write per element); longer rows are streamed twice
// (normaliser pass, then output pass). HBM-bound: 8 bytes per element at best.
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

constexpr int kSmThreads = 256;
constexpr int kSmCachedVec = 8;  // float4 groups per thread kept in registers
constexpr int kSmCached = kSmThreads * 4 * kSmCachedVec;

// Online update of (m, l) by one value; -inf (a masked logit) contributes nothing.
__device__ __forceinline__ void online_push(float& m, float& l, float x) {
  if (x > m) {
    l = l * __expf(m - x) + 1.f;  // exp(-inf) = 0 on the first finite value
    m = x;
  } else if (x != -INFINITY) {
    l += __expf(x - m);
  }
}

// Merge of two partial normalisers: both rebased to the larger max.
__device__ __forceinline__ void online_merge(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  l = l * __expf(m - mn) + l2 * __expf(m2 - mn);
  m = mn;
}

__device__ __forceinline__ void block_merge(float& m, float& l, float* sm_m, float* sm_l) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    online_merge(m, l, m2, l2);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  __syncthreads();
  m = sm_m[0];
  l = sm_l[0];
#pragma unroll
  for (int w = 1; w < kSmThreads / 32; ++w) online_merge(m, l, sm_m[w], sm_l[w]);
}

template <bool kCached>
__global__ void __launch_bounds__(kSmThreads) fa_softmax_rows_kernel(const float* __restrict__ x,
                                                                     float* __restrict__ p,
                                                                     float* __restrict__ lse, int n) {
  __shared__ float sm_m[kSmThreads / 32], sm_l[kSmThreads / 32];
  const size_t row = blockIdx.x;
  const float* xr = x + row * (size_t)n;
  float* pr = p + row * (size_t)n;
  const int nvec = n >> 2;  // whole float4 groups (row base is 16-byte aligned when n % 4 == 0)
  const bool vec_ok = (n & 3) == 0;
  // Four running (m, l) pairs per thread, one per float4 lane, keep each fp32 sum chain short;
  // they are merged (rebased to the larger max) before the block-wide merge.
  float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY}, lq[4] = {0.f, 0.f, 0.f, 0.f};
  float4 cache[kCached ? kSmCachedVec : 1];
  if (vec_ok) {
    const float4* xv = reinterpret_cast<const float4*>(xr);
#pragma unroll
    for (int k = 0; k < (kCached ? kSmCachedVec : 1); ++k) {
      if (!kCached) break;
      const int g = threadIdx.x + k * kSmThreads;
      cache[k] = g < nvec ? xv[g] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      online_push(mq[0], lq[0], cache[k].x);
      online_push(mq[1], lq[1], cache[k].y);
      online_push(mq[2], lq[2], cache[k].z);
      online_push(mq[3], lq[3], cache[k].w);
    }
    if (!kCached) {
      for (int g = threadIdx.x; g < nvec; g += kSmThreads) {
        const float4 v = xv[g];
        online_push(mq[0], lq[0], v.x);
        online_push(mq[1], lq[1], v.y);
        online_push(mq[2], lq[2], v.z);
        online_push(mq[3], lq[3], v.w);
      }
    }
  } else {
    int q = 0;
    for (int i = threadIdx.x; i < n; i += kSmThreads, q = (q + 1) & 3) online_push(mq[q], lq[q], xr[i]);
  }
  float m = mq[0], l = lq[0];
  online_merge(m, l, mq[1], lq[1]);
  online_merge(m, l, mq[2], lq[2]);
  online_merge(m, l, mq[3], lq[3]);
  block_merge(m, l, sm_m, sm_l);
  const float inv_l = 1.f / l;
  if (vec_ok) {
    float4* pv = reinterpret_cast<float4*>(pr);
    if (kCached) {
#pragma unroll
      for (int k = 0; k < kSmCachedVec; ++k) {
        const int g = threadIdx.x + k * kSmThreads;
        if (g < nvec) {
          const float4 v = cache[k];
          pv[g] = make_float4(__expf(v.x - m) * inv_l, __expf(v.y - m) * inv_l, __expf(v.z - m) * inv_l,
                              __expf(v.w - m) * inv_l);
        }
      }
    } else {
      const float4* xv = reinterpret_cast<const float4*>(xr);
      for (int g = threadIdx.x; g < nvec; g += kSmThreads) {
        const float4 v = xv[g];
        pv[g] = make_float4(__expf(v.x - m) * inv_l, __expf(v.y - m) * inv_l, __expf(v.z - m) * inv_l,
                            __expf(v.w - m) * inv_l);
      }
    }
  } else {
    for (int i = threadIdx.x; i < n; i += kSmThreads) pr[i] = __expf(xr[i] - m) * inv_l;
  }
  if (lse != nullptr && threadIdx.x == 0) lse[row] = m + __logf(l);
}

// Short rows (n <= 128 * VEC <= 2048, n % 4 == 0): one warp per row, 8 rows per CTA. Each lane keeps
// its VEC float4 groups in registers, forms its own partial (m_lane, l_lane) with
// e = exp(x - m_lane) stored in place, the lanes merge their partials by rebasing to the larger
// max (warp shuffles), and p = e * exp(m_lane - m) / l: one exp per element, one HBM read and
// one write.
template <int VEC>
__global__ void __launch_bounds__(256) fa_softmax_warp_rows_kernel(const float* __restrict__ x,
                                                                   float* __restrict__ p,
                                                                   float* __restrict__ lse, long long rows,
                                                                   int n) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;  // whole warps exit together
  const int lane = threadIdx.x & 31;
  const int nvec = n >> 2;
  const float4* xv = reinterpret_cast<const float4*>(x + row * (size_t)n);
  float4 e[VEC];
  float mt = -INFINITY;
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int g = lane + 32 * k;
    e[k] = g < nvec ? xv[g] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    mt = fmaxf(mt, fmaxf(fmaxf(e[k].x, e[k].y), fmaxf(e[k].z, e[k].w)));
  }
  float ls[4] = {0.f, 0.f, 0.f, 0.f};
  const float mref = (mt == -INFINITY) ? 0.f : mt;  // a lane with no finite value keeps l = 0
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    e[k] = make_float4(__expf(e[k].x - mref), __expf(e[k].y - mref), __expf(e[k].z - mref), __expf(e[k].w - mref));
    ls[0] += e[k].x;
    ls[1] += e[k].y;
    ls[2] += e[k].z;
    ls[3] += e[k].w;
  }
  float m = mt, l = (ls[0] + ls[1]) + (ls[2] + ls[3]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    online_merge(m, l, m2, l2);
  }
  const float f = (mt == -INFINITY) ? 0.f : expf(mt - m) / l;  // rebases this lane's terms
  float4* pv = reinterpret_cast<float4*>(p + row * (size_t)n);
#pragma unroll
  for (int k = 0; k < VEC; ++k) {
    const int g = lane + 32 * k;
    if (g < nvec) pv[g] = make_float4(e[k].x * f, e[k].y * f, e[k].z * f, e[k].w * f);
  }
  if (lse != nullptr && lane == 0) lse[row] = m + __logf(l);
}

template <int VEC>
static cudaError_t launch_warp_rows(const float* x, float* p, float* lse, long long rows, int n, cudaStream_t st) {
  fa_softmax_warp_rows_kernel<VEC><<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(x, p, lse, rows, n);
  return cudaGetLastError();
}

cudaError_t launch_softmax_rows(const float* x, float* p, float* lse, long long rows, int n, cudaStream_t st) {
  if (n % 4 == 0 && n <= 2048) {
    if (n <= 128) return launch_warp_rows<1>(x, p, lse, rows, n, st);
    if (n <= 256) return launch_warp_rows<2>(x, p, lse, rows, n, st);
    if (n <= 512) return launch_warp_rows<4>(x, p, lse, rows, n, st);
    if (n <= 1024) return launch_warp_rows<8>(x, p, lse, rows, n, st);
    return launch_warp_rows<16>(x, p, lse, rows, n, st);
  }
  const bool cached = (n % 4 == 0) && n <= kSmCached;
  if (cached)
    fa_softmax_rows_kernel<true><<<(unsigned)rows, kSmThreads, 0, st>>>(x, p, lse, n);
  else
    fa_softmax_rows_kernel<false><<<(unsigned)rows, kSmThreads, 0, st>>>(x, p, lse, n);
  return cudaGetLastError();
}

}  // namespace fa
