// fa_naive.cu -- standard (naive) attention with the score matrix in HBM, as a baseline.
//
// "LLM Architecture Refresh [3]: Flash Attention Is Exact", section 1: compute S = QK^T and
// write it out; read it back, compute P = softmax(S) and write it out; read it back and compute
// O = PV. Here: S (fp32) and O = P V (bf16 P, fp32 accumulation) are cuBLAS batched GEMMs, and
// the masked row softmax (fp32 S -> bf16 P, LSE) is a kernel of this library. The N x N
// intermediates live in a caller-provided workspace. cuBLAS is opened with dlopen on first use,
// so the library has no link-time dependency on it; cuBLAS manages its own handle memory.
#include <cublas_v2.h>
#include <dlfcn.h>
#include <math.h>

#include <mutex>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

// Masked row softmax over S [rows][N] fp32 (row r of head h is query r % N): P bf16, LSE fp32.
// One CTA of 256 threads per row, online (m, l) per thread, block merge, then the output pass.
__global__ void __launch_bounds__(256) fa_naive_softmax_kernel(const float* __restrict__ S,
                                                               __nv_bfloat16* __restrict__ P,
                                                               float* __restrict__ lse, int N, int causal) {
  __shared__ float sm_m[8], sm_l[8];
  const size_t row = blockIdx.x;
  const int q = (int)(row % (size_t)N);
  const int n_vis = causal ? q + 1 : N;
  const float* s = S + row * (size_t)N;
  float m = -INFINITY, l = 0.f;
  for (int j = threadIdx.x; j < n_vis; j += 256) {
    const float x = s[j];
    if (x > m) {
      l = l * __expf(m - x) + 1.f;
      m = x;
    } else {
      l += __expf(x - m);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    const float mn = fmaxf(m, m2);
    if (mn != -INFINITY) {
      l = l * __expf(m - mn) + l2 * __expf(m2 - mn);
      m = mn;
    }
  }
  if ((threadIdx.x & 31) == 0) {
    sm_m[threadIdx.x >> 5] = m;
    sm_l[threadIdx.x >> 5] = l;
  }
  __syncthreads();
  m = sm_m[0];
  l = sm_l[0];
  for (int w = 1; w < 8; ++w) {
    const float mn = fmaxf(m, sm_m[w]);
    if (mn == -INFINITY) continue;
    l = l * __expf(m - mn) + sm_l[w] * __expf(sm_m[w] - mn);
    m = mn;
  }
  const float inv = 1.f / l;
  __nv_bfloat16* pr = P + row * (size_t)N;
  for (int j = threadIdx.x; j < N; j += 256) pr[j] = __float2bfloat16(j < n_vis ? __expf(s[j] - m) * inv : 0.f);
  if (threadIdx.x == 0) lse[row] = m + __logf(l);
}

namespace {

// The C entry point of cuBLAS's strided batched GEMM with separate compute type.
typedef cublasStatus_t (*GemmStridedBatchedEx)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int,
                                               const void*, const void*, cudaDataType, int, long long, const void*,
                                               cudaDataType, int, long long, const void*, void*, cudaDataType, int,
                                               long long, int, cublasComputeType_t, cublasGemmAlgo_t);

struct Cublas {
  bool tried = false, ok = false;
  decltype(&cublasCreate_v2) create = nullptr;
  decltype(&cublasSetStream_v2) set_stream = nullptr;
  GemmStridedBatchedEx gemm = nullptr;
  cublasHandle_t handles[64] = {};
};
Cublas g_cublas;
std::mutex g_cublas_mutex;

bool load_cublas() {
  if (g_cublas.tried) return g_cublas.ok;
  g_cublas.tried = true;
  const char* names[] = {"libcublas.so.13", "/usr/local/cuda/lib64/libcublas.so.13", "libcublas.so"};
  void* h = nullptr;
  for (const char* n : names)
    if ((h = dlopen(n, RTLD_NOW | RTLD_GLOBAL)) != nullptr) break;
  if (h == nullptr) return false;
  g_cublas.create = reinterpret_cast<decltype(&cublasCreate_v2)>(dlsym(h, "cublasCreate_v2"));
  g_cublas.set_stream = reinterpret_cast<decltype(&cublasSetStream_v2)>(dlsym(h, "cublasSetStream_v2"));
  g_cublas.gemm = reinterpret_cast<GemmStridedBatchedEx>(dlsym(h, "cublasGemmStridedBatchedEx"));
  g_cublas.ok = g_cublas.create && g_cublas.set_stream && g_cublas.gemm;
  return g_cublas.ok;
}

}  // namespace

size_t naive_workspace_bytes(int B, int Hq, int N) {
  const size_t nn = (size_t)B * Hq * N * N;
  return (nn * 4 + 255) / 256 * 256 + (nn * 2 + 255) / 256 * 256;
}

// Returns 0, or 1 when cuBLAS cannot be loaded, or 2 on a cuBLAS / launch error.
int launch_naive_fwd(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace, int B,
                     int Hq, int Hkv, int N, int d, int causal, float scale, cudaStream_t st) {
  // One cuBLAS handle per device, shared by all callers: the lock covers setting its stream and
  // every GEMM enqueued with it, so concurrent calls on other streams cannot redirect them.
  std::lock_guard<std::mutex> lock(g_cublas_mutex);
  if (!load_cublas()) return 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 2;
  if (g_cublas.handles[dev] == nullptr && g_cublas.create(&g_cublas.handles[dev]) != CUBLAS_STATUS_SUCCESS)
    return 2;
  cublasHandle_t handle = g_cublas.handles[dev];
  if (g_cublas.set_stream(handle, st) != CUBLAS_STATUS_SUCCESS) return 2;
  const size_t nn = (size_t)N * N;
  float* S = static_cast<float*>(workspace);
  __nv_bfloat16* P = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) +
                                                       ((size_t)B * Hq * nn * 4 + 255) / 256 * 256);
  const int G = Hq / Hkv;
  const float alpha_s = scale, one = 1.f, zero = 0.f;
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k);
  const auto* vb = static_cast<const __nv_bfloat16*>(v);
  auto* ob = static_cast<__nv_bfloat16*>(o);
  // S (row-major, N x N per query head) = scale * Q K^T, i.e. column-major S^T = K Q^T; the G
  // query heads of a kv group share K (stride 0).
  for (int b = 0; b < B; ++b)
    for (int hk = 0; hk < Hkv; ++hk) {
      const size_t qh0 = (size_t)b * Hq + (size_t)hk * G;
      if (g_cublas.gemm(handle, CUBLAS_OP_T, CUBLAS_OP_N, N, N, d, &alpha_s, kb + ((size_t)b * Hkv + hk) * N * d,
                        CUDA_R_16BF, d, 0, qb + qh0 * N * d, CUDA_R_16BF, d, (long long)N * d, &zero, S + qh0 * nn,
                        CUDA_R_32F, N, (long long)nn, G, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) !=
          CUBLAS_STATUS_SUCCESS)
        return 2;
    }
  fa_naive_softmax_kernel<<<(unsigned)((size_t)B * Hq * N), 256, 0, st>>>(S, P, lse, N, causal);
  if (cudaGetLastError() != cudaSuccess) return 2;
  // O (row-major N x d) = P V, i.e. column-major O^T = V^T P^T.
  for (int b = 0; b < B; ++b)
    for (int hk = 0; hk < Hkv; ++hk) {
      const size_t qh0 = (size_t)b * Hq + (size_t)hk * G;
      if (g_cublas.gemm(handle, CUBLAS_OP_N, CUBLAS_OP_N, d, N, N, &one, vb + ((size_t)b * Hkv + hk) * N * d,
                        CUDA_R_16BF, d, 0, P + qh0 * nn, CUDA_R_16BF, N, (long long)nn, &zero, ob + qh0 * N * d,
                        CUDA_R_16BF, d, (long long)N * d, G, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) !=
          CUBLAS_STATUS_SUCCESS)
        return 2;
    }
  return 0;
}

}  // namespace fa
