// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA descriptors, launch.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

// One warp waits, with the kernels' own bounded wait, on an mbarrier that nothing arrives at:
// the wait gives up after its time limit, raises the CTA abort flag and records the timeout
// in the device status word, and the kernel returns.
__global__ void __launch_bounds__(32) fa_selftest_wait_kernel(uint32_t* status, int* result) {
  __shared__ __align__(8) uint64_t bar_storage;
  __shared__ int abort_flag;
  const uint32_t bar = smem_u32(&bar_storage);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  const Ctl ctl{&abort_flag, status};
  const bool ok = mbar_wait_warp(bar, 0, ctl);
  if (threadIdx.x == 0) *result = ok ? 1 : (abort_flag ? 2 : 3);
}

}  // namespace fa

namespace {

// Per-device status word written by kernels whose pipeline waits time out.
__device__ uint32_t g_fa_status;

constexpr int kMaxDevices = 64;
struct DeviceState {
  bool init = false;
  bool supported = false;
  int num_sms = 0;
  uint32_t* status = nullptr;  // device address of g_fa_status in the context below
  unsigned long long ctx = 0;  // id of the context `status` was looked up in (0: none yet)
};
DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;
std::once_flag g_ctx_once;

// Looks up whether the current device is an sm_103 part (once per device) and the device
// address of its status word (again whenever the current context is not the one the address
// was taken in: a context re-created after cudaDeviceReset loads the module afresh).
int current_device(uint32_t** status, int* num_sms = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_devices[dev];
  if (!s.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_LAUNCH;
    s.supported = (major == 10 && minor == 3);
    if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FA_ERR_LAUNCH;
    s.init = true;
  }
  if (!s.supported) return FA_ERR_DEVICE;
  if (status) {
    const unsigned long long ctx = fa::current_context_id();
    if (s.status == nullptr || ctx == 0 || ctx != s.ctx) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_fa_status) != cudaSuccess) return FA_ERR_LAUNCH;
      s.status = static_cast<uint32_t*>(addr);
      s.ctx = fa::current_context_id();  // the lookup made the primary context current if it was not
    }
    *status = s.status;
  }
  if (num_sms) *num_sms = s.num_sms;
  return FA_OK;
}

}  // namespace

unsigned long long fa::current_context_id() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (g_ctx_current == nullptr || g_ctx_get_id == nullptr) return 0;
  CUcontext c = nullptr;
  if (g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  return g_ctx_get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

int fa::check_current_device() { return current_device(nullptr); }

namespace {

bool load_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 3-D map over a [planes][N][d] bf16 tensor; box = 64 columns (128 B, one swizzle span) x
// box_rows rows (128 unless given) x 1 plane, 128-byte swizzle. Rows past N read as zero (loads)
// or are not written (stores).
int make_map(CUtensorMap* m, const void* base, int d, int N, long long planes, int box_rows = fa::kTile) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_INVALID;
}

// 3-D map over split-KV partial outputs [planes][N][d] fp32; box = 32 columns (128 B) x 32 rows
// x 1 plane, 128-byte swizzle (the staging layout of the forward's epilogue stores).
int make_map_part(CUtensorMap* m, void* base, int d, int N, long long planes) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)N * (cuuint64_t)d * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_INVALID;
}

// 2-D map over the fp32 dQ accumulator [rows][d]; box = 32 columns (128 B) x 32 rows,
// 128-byte swizzle (the staging layout the backward's dQ drain writes).
int make_map_dq(CUtensorMap* m, void* base, int d, long long rows) {
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_INVALID;
}

int check_sizes(int B, int Hq, int Hkv, int N, int d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || N < 1) return FA_ERR_INVALID;
  if (Hq % Hkv != 0) return FA_ERR_INVALID;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long tiles = (long long)B * Hq * ((N + fa::kTile - 1) / fa::kTile);
  if (tiles > 0x7fffffffLL) return FA_ERR_INVALID;
  if ((long long)B * Hq > 0x7fffffffLL) return FA_ERR_INVALID;
  return FA_OK;
}

int check_ptr(const void* p) {
  if (p == nullptr) return FA_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(p) & 15u) return FA_ERR_ALIGN;
  return FA_OK;
}

float resolve_scale(float scale, int d) { return (scale > 0.f) ? scale : 1.0f / std::sqrt((float)d); }

struct WorkspaceLayout {
  size_t dq_acc, delta, lse2, next_item, total;
};
WorkspaceLayout workspace_layout(int B, int Hq, int N, int d) {
  const size_t rows = (size_t)B * Hq * fa::round_up_tile(N);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  WorkspaceLayout w;
  w.dq_acc = 0;
  w.delta = up(rows * d * 4);
  w.lse2 = w.delta + up(rows * 4);
  w.next_item = w.lse2 + up(rows * 4);
  w.total = w.next_item + 256;
  return w;
}

#define FA_TRY(x)               \
  do {                          \
    int _r = (x);               \
    if (_r != FA_OK) return _r; \
  } while (0)

// Split-KV workspace: fp32 partial outputs [splits][B*Hq][N][d], then partial LSE [splits][B*Hq][N].
size_t splitkv_bytes(int B, int Hq, int N, int d, int splits, size_t* lse_off) {
  const size_t rows = (size_t)splits * B * Hq * N;
  const size_t o_bytes = (rows * d * 4 + 255) / 256 * 256;
  if (lse_off) *lse_off = o_bytes;
  return o_bytes + (rows * 4 + 255) / 256 * 256;
}

// Split count for automatic selection: the s in {1, 2, 4, 8, 16} with the least predicted time,
// taken only for a predicted gain of 10 % or more over no split. The persistent forward takes the
// longer of its longest work item and its work per SM, counted in key-tile steps of a two-tile
// item (about 1.9 us at d = 128 and 1.6 us at d = 64, measured on GB300); a split adds the merge
// kernel (about 5 us) and the fp32 partial outputs of every query tile that has more than one
// non-empty split, written and read back (about 5 TB/s). Fitted to measured times of 1 to 16
// splits on small-batch shapes, which it predicts within about 10 %.
int auto_splits(int B, int Hq, int N, int d, int causal, int num_sms) {
  const int T = (N + fa::kTile - 1) / fa::kTile;
  const int pairs = (T + 1) / 2;
  const double step_us = d == 128 ? 1.9 : 1.6;
  const double heads = (double)B * Hq;
  const double sms = num_sms > 0 ? num_sms : 1;
  double t_plain = 0.0, t_best = 0.0;
  int best = 1;
  for (int s = 1; s <= 16 && s <= T; s *= 2) {
    const int len = (T + s - 1) / s;
    double longest = 0.0, work = 0.0;
    for (int pr = 0; pr < pairs; ++pr) {
      const int hi = causal ? std::min(2 * pr + 2, T) : T;  // key tiles of the pair's upper query tile
      for (int sp = 0; sp * len < hi; ++sp) {
        const int steps = std::min(hi, (sp + 1) * len) - sp * len;
        longest = std::max(longest, (double)steps);
        work += steps;
      }
    }
    double t = std::max(longest, work * heads / sms) * step_us;
    if (s > 1) {
      double part_bytes = 0.0;  // per head
      for (int qt = 0; qt < T; ++qt) {
        const int hi = causal ? qt + 1 : T;
        const int ns = std::min(s, (hi + len - 1) / len);
        if (ns > 1) part_bytes += (double)ns * fa::kTile * d * 4;
      }
      t += 5.0 + 2.0 * part_bytes * heads / 5.0e6;
    }
    if (s == 1) {
      t_plain = t_best = t;
    } else if (t < 0.9 * t_plain && t < t_best) {
      best = s;
      t_best = t;
    }
  }
  return best;
}

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
             int d, int causal, float scale, unsigned long long* counters, fa_stream_t stream, int window = 0,
             int num_splits = 1, float* o_part = nullptr, float* lse_part = nullptr) {
  FA_TRY(check_sizes(B, Hq, Hkv, N, d));
  FA_TRY(check_ptr(q));
  FA_TRY(check_ptr(k));
  FA_TRY(check_ptr(v));
  FA_TRY(check_ptr(o));
  FA_TRY(check_ptr(lse));
  if (counters != nullptr && (reinterpret_cast<uintptr_t>(counters) & 7u)) return FA_ERR_ALIGN;
  uint32_t* status = nullptr;
  int num_sms = 0;
  FA_TRY(current_device(&status, &num_sms));
  if (!load_encoder()) return FA_ERR_LAUNCH;
  CUtensorMap tq, tk, tv, to;
  FA_TRY(make_map(&tq, q, d, N, (long long)B * Hq));
  FA_TRY(make_map(&tk, k, d, N, (long long)B * Hkv));
  FA_TRY(make_map(&tv, v, d, N, (long long)B * Hkv));
  FA_TRY(make_map(&to, o, d, N, (long long)B * Hq, 32));  // O stores: 32 rows (one warp) per box
  CUtensorMap tp = to;  // split-KV partial outputs (fp32); unused without splits
  if (num_splits > 1) FA_TRY(make_map_part(&tp, o_part, d, N, (long long)num_splits * B * Hq));
  fa::FwdLaunch a;
  a.tm_q = &tq;
  a.tm_k = &tk;
  a.tm_v = &tv;
  a.tm_o = &to;
  a.tm_opart = &tp;
  a.o = o;
  a.lse = lse;
  a.counters = counters;
  a.status = status;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.d = d;
  a.causal = causal ? 1 : 0;
  a.window = window;
  a.num_splits = num_splits;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.num_sms = num_sms;
  a.scale = resolve_scale(scale, d);
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return fa::launch_fwd(a) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

int fa::check_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* dout, const void* lse,
                       const void* dq, const void* dk, const void* dv, int B, int Hq, int Hkv, int N, int d) {
  FA_TRY(check_sizes(B, Hq, Hkv, N, d));
  for (const void* p : {q, k, v, o, dout, lse, dq, dk, dv}) FA_TRY(check_ptr(p));
  return FA_OK;
}

namespace {

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N,
             int d, int causal, float scale, fa_stream_t stream, int stages, int window = 0) {
  FA_TRY(check_sizes(B, Hq, Hkv, N, d));
  // Pointers each stage reads or writes.
  if (stages & fa::kBwdPrepare) {
    for (const void* p : {o, dout, static_cast<const void*>(lse)}) FA_TRY(check_ptr(p));
  }
  if (stages & fa::kBwdCompute) {
    for (const void* p : {q, k, v, dout, static_cast<const void*>(dk), static_cast<const void*>(dv)})
      FA_TRY(check_ptr(p));
  }
  if (stages & fa::kBwdFinalize) FA_TRY(check_ptr(dq));
  const WorkspaceLayout w = workspace_layout(B, Hq, N, d);
  if (workspace == nullptr || workspace_bytes < w.total) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_ALIGN;
  uint32_t* status = nullptr;
  int num_sms = 0;
  FA_TRY(current_device(&status, &num_sms));
  char* ws = static_cast<char*>(workspace);
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if (stages & fa::kBwdCompute) {
    if (!load_encoder()) return FA_ERR_LAUNCH;
    FA_TRY(make_map(&tq, q, d, N, (long long)B * Hq));
    FA_TRY(make_map(&tk, k, d, N, (long long)B * Hkv));
    FA_TRY(make_map(&tv, v, d, N, (long long)B * Hkv));
    FA_TRY(make_map(&tdo, dout, d, N, (long long)B * Hq));
    FA_TRY(make_map_dq(&tdq, ws + w.dq_acc, d, (long long)B * Hq * fa::round_up_tile(N)));
    FA_TRY(make_map(&tdk, dk, d, N, (long long)B * Hkv, 32));  // dK, dV stores: 32 rows per box
    FA_TRY(make_map(&tdv, dv, d, N, (long long)B * Hkv, 32));
  }
  fa::BwdLaunch a;
  a.tm_dk = &tdk;
  a.tm_dv = &tdv;
  a.tm_q = &tq;
  a.tm_k = &tk;
  a.tm_v = &tv;
  a.tm_do = &tdo;
  a.tm_dq = &tdq;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc);
  a.delta = reinterpret_cast<float*>(ws + w.delta);
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2);
  a.next_item = reinterpret_cast<uint32_t*>(ws + w.next_item);
  a.status = status;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.d = d;
  a.causal = (causal || window > 0) ? 1 : 0;
  a.window = window;
  a.num_sms = num_sms;
  a.scale = resolve_scale(scale, d);
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return fa::launch_bwd(a, stages) == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
           int d, int causal, float scale, fa_stream_t stream) {
  fa::TraceRange trace("fa_fwd");
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, nullptr, stream);
}

int fa_fwd_stats(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                 int N, int d, int causal, float scale, unsigned long long* counters, fa_stream_t stream) {
  fa::TraceRange trace("fa_fwd_stats");
  if (counters == nullptr) return FA_ERR_INVALID;
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, counters, stream);
}

int fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                  int d, int window, float scale, fa_stream_t stream) {
  fa::TraceRange trace("fa_fwd_window");
  if (window < 1) return FA_ERR_INVALID;
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, 1, scale, nullptr, stream, window);
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int num_splits) {
  if (check_sizes(B, Hq, Hkv, N, d) != FA_OK || num_splits < 1 || num_splits > 64) return 0;
  return splitkv_bytes(B, Hq, N, d, num_splits, nullptr);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int N,
                   int d, int causal, float scale, int num_splits, void* workspace, size_t workspace_bytes,
                   fa_stream_t stream) {
  fa::TraceRange trace("fa_fwd_splitkv");
  FA_TRY(check_sizes(B, Hq, Hkv, N, d));
  if (num_splits > 64) return FA_ERR_INVALID;
  if (num_splits <= 0) {
    int sms = 0;
    FA_TRY(current_device(nullptr, &sms));
    num_splits = auto_splits(B, Hq, N, d, causal, sms);
  }
  size_t lse_off = 0;
  const size_t need = splitkv_bytes(B, Hq, N, d, num_splits, &lse_off);
  if (num_splits > 1) {
    if (workspace == nullptr || workspace_bytes < need) return FA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_ALIGN;
  }
  char* ws = static_cast<char*>(workspace);
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, scale, nullptr, stream, 0, num_splits,
                  num_splits > 1 ? reinterpret_cast<float*>(ws) : nullptr,
                  num_splits > 1 ? reinterpret_cast<float*>(ws + lse_off) : nullptr);
}

int fa_fwd_splitkv_auto(int B, int Hq, int Hkv, int N, int d, int causal, int num_sms) {
  FA_TRY(check_sizes(B, Hq, Hkv, N, d));
  if (num_sms < 1) return FA_ERR_INVALID;
  return auto_splits(B, Hq, N, d, causal, num_sms);
}

size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  if (check_sizes(B, Hq, Hkv, N, d) != FA_OK) return 0;
  return workspace_layout(B, Hq, N, d).total;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
           void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
           int N, int d, int causal, float scale, fa_stream_t stream) {
  fa::TraceRange trace("fa_bwd");
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d, causal, scale,
                  stream, fa::kBwdAll);
}

int fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv,
                  int N, int d, int window, float scale, fa_stream_t stream) {
  fa::TraceRange trace("fa_bwd_window");
  if (window < 1) return FA_ERR_INVALID;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d, 1, scale,
                  stream, fa::kBwdAll, window);
}

int fa_bwd_prepare(const void* o, const void* dout, const float* lse, void* workspace, size_t workspace_bytes,
                   int B, int Hq, int Hkv, int N, int d, fa_stream_t stream) {
  fa::TraceRange trace("fa_bwd_prepare");
  return bwd_impl(nullptr, nullptr, nullptr, o, dout, lse, nullptr, nullptr, nullptr, workspace, workspace_bytes,
                  B, Hq, Hkv, N, d, 0, 0.f, stream, fa::kBwdPrepare);
}

int fa_bwd_compute(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                   void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d, int causal,
                   float scale, fa_stream_t stream) {
  fa::TraceRange trace("fa_bwd_compute");
  return bwd_impl(q, k, v, nullptr, dout, nullptr, nullptr, dk, dv, workspace, workspace_bytes, B, Hq, Hkv, N, d,
                  causal, scale, stream, fa::kBwdCompute);
}

int fa_bwd_finalize(void* dq, void* workspace, size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d,
                    float scale, fa_stream_t stream) {
  fa::TraceRange trace("fa_bwd_finalize");
  return bwd_impl(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, dq, nullptr, nullptr, workspace,
                  workspace_bytes, B, Hq, Hkv, N, d, 0, scale, stream, fa::kBwdFinalize);
}

size_t fa_naive_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  if (check_sizes(B, Hq, Hkv, N, d) != FA_OK) return 0;
  return fa::naive_workspace_bytes(B, Hq, N);
}

int fa_naive_fwd(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                 size_t workspace_bytes, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                 fa_stream_t stream) {
  fa::TraceRange trace("fa_naive_fwd");
  FA_TRY(check_sizes(B, Hq, Hkv, N, d));
  for (const void* p : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)}) FA_TRY(check_ptr(p));
  if (workspace == nullptr || workspace_bytes < fa::naive_workspace_bytes(B, Hq, N)) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return FA_ERR_ALIGN;
  FA_TRY(current_device(nullptr));
  const int r = fa::launch_naive_fwd(q, k, v, o, lse, workspace, B, Hq, Hkv, N, d, causal ? 1 : 0,
                                     resolve_scale(scale, d), reinterpret_cast<cudaStream_t>(stream));
  return r == 0 ? FA_OK : (r == 1 ? FA_ERR_UNSUPPORTED : FA_ERR_LAUNCH);
}

int fa_softmax_rows(const float* x, float* p, float* lse, long long rows, int n, fa_stream_t stream) {
  fa::TraceRange trace("fa_softmax_rows");
  if (rows < 1 || rows > 0x7fffffffLL || n < 1) return FA_ERR_INVALID;
  FA_TRY(check_ptr(x));
  FA_TRY(check_ptr(p));
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_ALIGN;
  FA_TRY(current_device(nullptr));
  return fa::launch_softmax_rows(x, p, lse, rows, n, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA_OK
             : FA_ERR_LAUNCH;
}

int fa_selftest_wait_timeout(int* result, fa_stream_t stream) {
  if (result == nullptr) return FA_ERR_INVALID;
  uint32_t* status = nullptr;
  int r = current_device(&status);
  if (r != FA_OK) return r;
  fa::fa_selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, result);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_check(fa_stream_t stream) {
  uint32_t* status = nullptr;
  int r = current_device(&status);
  if (r != FA_OK) return r;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_LAUNCH;
  uint32_t h = 0;
  if (cudaMemcpy(&h, status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_LAUNCH;
  if (h != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_LAUNCH;
    return h == 1 ? FA_ERR_TIMEOUT : FA_ERR_LAUNCH;  // 2: a kernel found its shared memory misaligned
  }
  return FA_OK;
}

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID: return "invalid argument (null pointer, size < 1, Hq % Hkv != 0 or size overflow)";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension (d must be 64 or 128)";
    case FA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FA_ERR_LAUNCH: return "CUDA launch or runtime error";
    case FA_ERR_TIMEOUT: return "a device pipeline wait exceeded its time limit; outputs are undefined";
    case FA_ERR_WORKSPACE: return "backward workspace missing or smaller than fa_bwd_workspace_bytes()";
    case FA_ERR_DEVICE: return "current device is not an sm_103 (GB300) GPU";
    default: return "unknown status";
  }
}

int fa_version(void) { return (1 << 16) | 0; }

}  // extern "C"
