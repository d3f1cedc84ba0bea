// fa_host_step.cu -- forward and backward of one attention layer on host buffers, with the
// host<->device copies overlapped with the computation.
//
// The computation is fa_fwd followed by fa_bwd ("LLM Architecture Refresh [3]: Flash Attention
// Is Exact", sections 4 and 8), run once per batch element on that element's slices of the
// [B][H][N][d] tensors (contiguous in this layout). Three streams carry a software pipeline:
//   input stream    copies q, k, v, then dO of each element to the device,
//   compute streams run the forward and backward kernels of even elements on the caller's
//                   stream and of odd elements on a second stream, each with its own backward
//                   workspace, so one element's kernels fill the SMs that the previous
//                   element's longest key tiles leave idle at the end of its backward,
//   output stream   copies o, lse of an element once its forward is done, then dq, dk, dv once
//                   its backward is,
// ordered by events (each element's forward waits only for q, k, v; its backward for dO). GB300's copy engines move host data at about
// 200 GB/s per direction and both directions at once, so for large steps the copies hide behind
// the kernels except for the first element's inputs and the last element's outputs.
// The input and output streams and the events are created once per device and reused; device
// memory comes from the caller's workspace only.
#include <stdint.h>

#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_internal.h"

namespace {

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr, comp = nullptr;
  std::vector<cudaEvent_t> ev;  // [0] start, [1] done, then 4 per batch element
};
HostPipe g_pipe[64];
std::mutex g_pipe_mutex;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct StepLayout {
  size_t q, kv, lse, bwd;  // bytes of one batch element's q/dO/o/dq, k/v/dk/dv, lse; bwd workspace
  size_t total;
};

bool step_layout(int B, int Hq, int Hkv, int N, int d, StepLayout* L) {
  // Both return 0 for invalid sizes (including products that overflow at batch B).
  const size_t bwd = fa_bwd_workspace_bytes(1, Hq, Hkv, N, d);
  if (bwd == 0 || B < 1 || fa_bwd_workspace_bytes(B, Hq, Hkv, N, d) == 0) return false;
  L->q = (size_t)Hq * N * d * 2;
  L->kv = (size_t)Hkv * N * d * 2;
  L->lse = (size_t)Hq * N * 4;
  L->bwd = bwd;
  // q, dO, o, dq: B * q each; k, v, dk, dv: B * kv each; lse: B * lse; a backward workspace
  // per compute stream.
  L->total = 4 * align256(B * L->q) + 4 * align256(B * L->kv) + align256(B * L->lse) +
             (B > 1 ? 2 : 1) * align256(bwd);
  return true;
}

cudaEvent_t* pipe_events(int dev, int B) {
  HostPipe& P = g_pipe[dev];
  if (!P.ready) {
    if (cudaStreamCreateWithFlags(&P.in, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithFlags(&P.out, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaStreamCreateWithFlags(&P.comp, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    P.ready = true;
  }
  while ((int)P.ev.size() < 2 + 4 * B) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    P.ev.push_back(e);
  }
  return P.ev.data();
}

}  // namespace

extern "C" {

size_t fa_fwd_bwd_host_workspace_bytes(int B, int Hq, int Hkv, int N, int d) {
  StepLayout L;
  return step_layout(B, Hq, Hkv, N, d, &L) ? L.total : 0;
}

int fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dout, void* o, float* lse, void* dq,
                    void* dk, void* dv, int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                    void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  StepLayout L;
  if (!step_layout(B, Hq, Hkv, N, d, &L)) return FA_ERR_INVALID;
  if (!q || !k || !v || !dout || !o || !lse || !dq || !dk || !dv) return FA_ERR_INVALID;
  if (!workspace || workspace_bytes < L.total) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return FA_ERR_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_LAUNCH;

  // Device copies of every tensor, then the backward workspace.
  char* w = static_cast<char*>(workspace);
  auto take = [&](size_t bytes) {
    char* p = w;
    w += align256(bytes);
    return p;
  };
  char* d_q = take(B * L.q);
  char* d_k = take(B * L.kv);
  char* d_v = take(B * L.kv);
  char* d_do = take(B * L.q);
  char* d_o = take(B * L.q);
  char* d_lse = take(B * L.lse);
  char* d_dq = take(B * L.q);
  char* d_dk = take(B * L.kv);
  char* d_dv = take(B * L.kv);
  char* d_ws[2];
  d_ws[0] = take(L.bwd);
  d_ws[1] = B > 1 ? take(L.bwd) : d_ws[0];

  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  cudaEvent_t* ev = pipe_events(dev, B);
  if (ev == nullptr) return FA_ERR_LAUNCH;
  HostPipe& P = g_pipe[dev];
  cudaEvent_t ev_start = ev[0], ev_done = ev[1];
  cudaEvent_t* ev_qkv = ev + 2;          // q, k, v of element b on the device
  cudaEvent_t* ev_do = ev + 2 + B;       // dO of element b on the device
  cudaEvent_t* ev_fwd = ev + 2 + 2 * B;  // o, lse of element b computed
  cudaEvent_t* ev_bwd = ev + 2 + 3 * B;  // dq, dk, dv of element b computed
  const auto H2D = cudaMemcpyHostToDevice;
  const auto D2H = cudaMemcpyDeviceToHost;
#define FA_CU(x) \
  if ((x) != cudaSuccess) return FA_ERR_LAUNCH
  // Everything the caller enqueued before (including a previous call's use of this workspace)
  // happens first.
  FA_CU(cudaEventRecord(ev_start, st));
  FA_CU(cudaStreamWaitEvent(P.in, ev_start, 0));
  FA_CU(cudaStreamWaitEvent(P.out, ev_start, 0));
  FA_CU(cudaStreamWaitEvent(P.comp, ev_start, 0));
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  const char* hdo = static_cast<const char*>(dout);
  for (int b = 0; b < B; ++b) {
    FA_CU(cudaMemcpyAsync(d_q + b * L.q, hq + b * L.q, L.q, H2D, P.in));
    FA_CU(cudaMemcpyAsync(d_k + b * L.kv, hk + b * L.kv, L.kv, H2D, P.in));
    FA_CU(cudaMemcpyAsync(d_v + b * L.kv, hv + b * L.kv, L.kv, H2D, P.in));
    FA_CU(cudaEventRecord(ev_qkv[b], P.in));
    FA_CU(cudaMemcpyAsync(d_do + b * L.q, hdo + b * L.q, L.q, H2D, P.in));
    FA_CU(cudaEventRecord(ev_do[b], P.in));
  }
  for (int b = 0; b < B; ++b) {
    const cudaStream_t cs = (b & 1) ? P.comp : st;
    const fa_stream_t cs_h = reinterpret_cast<fa_stream_t>(cs);
    FA_CU(cudaStreamWaitEvent(cs, ev_qkv[b], 0));
    int r = fa_fwd(d_q + b * L.q, d_k + b * L.kv, d_v + b * L.kv, d_o + b * L.q,
                   reinterpret_cast<float*>(d_lse + b * L.lse), 1, Hq, Hkv, N, d, causal, scale, cs_h);
    if (r != FA_OK) return r;
    FA_CU(cudaEventRecord(ev_fwd[b], cs));
    FA_CU(cudaStreamWaitEvent(cs, ev_do[b], 0));
    r = fa_bwd(d_q + b * L.q, d_k + b * L.kv, d_v + b * L.kv, d_o + b * L.q, d_do + b * L.q,
               reinterpret_cast<const float*>(d_lse + b * L.lse), d_dq + b * L.q, d_dk + b * L.kv, d_dv + b * L.kv,
               d_ws[b & 1], L.bwd, 1, Hq, Hkv, N, d, causal, scale, cs_h);
    if (r != FA_OK) return r;
    FA_CU(cudaEventRecord(ev_bwd[b], cs));
  }
  char* ho = static_cast<char*>(o);
  char* hl = reinterpret_cast<char*>(lse);
  char* hdq = static_cast<char*>(dq);
  char* hdk = static_cast<char*>(dk);
  char* hdv = static_cast<char*>(dv);
  for (int b = 0; b < B; ++b) {
    FA_CU(cudaStreamWaitEvent(P.out, ev_fwd[b], 0));
    FA_CU(cudaMemcpyAsync(ho + b * L.q, d_o + b * L.q, L.q, D2H, P.out));
    FA_CU(cudaMemcpyAsync(hl + b * L.lse, d_lse + b * L.lse, L.lse, D2H, P.out));
    FA_CU(cudaStreamWaitEvent(P.out, ev_bwd[b], 0));
    FA_CU(cudaMemcpyAsync(hdq + b * L.q, d_dq + b * L.q, L.q, D2H, P.out));
    FA_CU(cudaMemcpyAsync(hdk + b * L.kv, d_dk + b * L.kv, L.kv, D2H, P.out));
    FA_CU(cudaMemcpyAsync(hdv + b * L.kv, d_dv + b * L.kv, L.kv, D2H, P.out));
  }
  FA_CU(cudaEventRecord(ev_done, P.out));
  FA_CU(cudaStreamWaitEvent(st, ev_done, 0));
#undef FA_CU
  return FA_OK;
}

}  // extern "C"
