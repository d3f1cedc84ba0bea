// fa_bwd_noalloc.cu -- the backward pass for callers that cannot allocate device memory.
//
// fa_bwd needs a workspace (fp32 dQ accumulator plus two per-row statistics) that the caller
// allocates. Some callers must not call cudaMalloc at all: a plugin running inside a host
// runtime that owns and budgets every byte of device memory, or a latency-critical loop in
// which cudaMalloc's implicit device synchronisation is not allowed. fa_bwd_noalloc gives them
// the same backward pass with the workspace taken from a fixed device array that is part of
// this library's module: it exists from the moment the module is loaded on a device until the
// process exits, and no call allocates or frees anything.
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

// The backward workspace as fixed device memory. In host code this name is only a host-side
// stand-in for the symbol, never a device address: its device address comes from
// cudaGetSymbolAddress below, once per device context.
static __device__ __align__(256) unsigned char g_fa_bwd_scratch[FA_BWD_NOALLOC_MAX_BYTES];

namespace {

constexpr int kMaxScratchDevices = 64;
void* g_scratch_addr[kMaxScratchDevices];
unsigned long long g_scratch_ctx[kMaxScratchDevices];  // context the address was taken in
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device. The first call on a device
// looks it up (with that device current) and caches it with the id of the current context;
// later calls in the same context only read the cache. A different context (one re-created
// after cudaDeviceReset, or another context the caller made current) has the module loaded
// anew, so the address is looked up again there.
int scratch_on_current_device(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxScratchDevices) return FA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  const unsigned long long ctx = fa::current_context_id();
  if (g_scratch_addr[dev] == nullptr || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_bwd_scratch) != cudaSuccess || p == nullptr) return FA_ERR_LAUNCH;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = fa::current_context_id();
  }
  *addr = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                              const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                              int d, int causal, float scale, fa_stream_t stream) {
  fa::TraceRange trace("fa_bwd_noalloc");
  // Checks in the order every other entry point takes them: arguments (no CUDA call), then the
  // size limit of the fixed scratch, then the device, and only then the scratch lookup.
  int r = fa::check_bwd_args(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d);
  if (r != FA_OK) return r;
  const size_t need = fa_bwd_workspace_bytes(B, Hq, Hkv, N, d);
  if (need > FA_BWD_NOALLOC_MAX_BYTES) return FA_ERR_WORKSPACE;  // too large for the fixed scratch
  if ((r = fa::check_current_device()) != FA_OK) return r;
  void* scratch = nullptr;
  if ((r = scratch_on_current_device(&scratch)) != FA_OK) return r;
  // The prepare stage of fa_bwd rewrites every byte of the workspace it reads (the dQ
  // accumulator is zeroed, delta and LSE2 are overwritten), so the previous call's contents
  // never leak into this one.
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, scratch, FA_BWD_NOALLOC_MAX_BYTES, B, Hq, Hkv, N, d, causal,
                scale, stream);
}
