// fa_host_step.cu -- forward and backward of one attention layer on host buffers, with the
// host<->device copies overlapped with the computation.
//
// The computation is fa_fwd followed by fa_bwd ("LLM Architecture Refresh [3]: Flash Attention
// Is Exact", sections 4 and 8), run chunk by chunk. A chunk is one batch element's slice of
// whole KV-head groups (kv heads [g0, g0 + hk) and the hk * Hq/Hkv query heads that read them),
// contiguous in every [B][H][N][d] tensor, and self-contained: its forward and backward need
// no other chunk's data. Streams carry a software pipeline:
//   input stream     copies q, k, v, then dO of each chunk to the device,
//   compute streams  run the forward and backward kernels of chunk c on stream c mod S (the
//                    caller's stream is stream 0), each with its own backward workspace, so that
//                    several chunks' kernels share the SMs (one chunk's grid is too small to fill
//                    them, and the longest key tiles of a chunk's backward end alone),
//   output streams   copy o, lse of a chunk once its forward is done (one stream), and dq, dk, dv
//                    once its backward is (another, so that forward outputs never queue behind a
//                    backward that is still running),
// ordered by events. GB300's copy engines move host data at about 200 GB/s in one direction
// and 150-170 GB/s each way with both busy, so a large step is bound by the copies: the inputs
// arrive over most of the step, and after the last chunk's dO there remain that chunk's backward
// (as long as its longest key tile's pass over all its query tiles, whatever the chunk's size)
// and the copy of its gradients. About 8 chunks per call measured best: fewer leave the output
// link idle longer at the start and put more bytes behind the last backward; more make copies
// and grids small enough to slow both.
// The streams and events are created once per device and reused; device memory comes from the
// caller's workspace only.
#include <stdint.h>

#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kTargetChunks = 8;    // chunks per call the split aims for (at least)
constexpr int kComputeStreams = 4;  // the caller's stream and three library streams

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out_fwd = nullptr, out_bwd = nullptr, comp[kComputeStreams - 1] = {};
  std::vector<cudaEvent_t> ev;  // [0] start, [1], [2] output streams done, then 4 per chunk
};
HostPipe g_pipe[64];
std::mutex g_pipe_mutex;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Each batch element is split into `split` chunks of Hkv/split kv heads: split is the smallest
// divisor of Hkv with B * split >= kTargetChunks, or Hkv.
struct StepLayout {
  int Hkv, G;
  int split;                // a divisor of Hkv
  int chunks;               // B * split
  int streams;              // compute streams in use
  int nkv;                  // kv heads of a chunk
  size_t head_q, head_lse;  // bytes of one head's [N][d] bf16 slice and [N] fp32 slice
  size_t lse_chunk;         // device lse of a chunk: its slice rounded up to 256 bytes
  size_t bwd;               // backward workspace of a chunk
  size_t total;
};

bool step_layout(int B, int Hq, int Hkv, int N, int d, StepLayout* L) {
  // fa_bwd_workspace_bytes returns 0 for invalid sizes (including products that overflow at B).
  if (B < 1 || Hkv < 1 || fa_bwd_workspace_bytes(B, Hq, Hkv, N, d) == 0) return false;
  const int want = (kTargetChunks + B - 1) / B;
  int split = Hkv;
  for (int s = 1; s <= Hkv; ++s)
    if (Hkv % s == 0 && s >= want) {
      split = s;
      break;
    }
  L->Hkv = Hkv;
  L->G = Hq / Hkv;
  L->split = split;
  L->chunks = B * split;
  L->streams = L->chunks < kComputeStreams ? L->chunks : kComputeStreams;
  L->nkv = Hkv / split;
  L->head_q = (size_t)N * d * 2;
  L->head_lse = (size_t)N * 4;
  // The kernels want lse 16-byte aligned, which a chunk's slice of [B][Hq][N] is not for odd
  // N, so each chunk's device lse starts on a 256-byte boundary.
  L->lse_chunk = align256((size_t)L->nkv * L->G * L->head_lse);
  L->bwd = fa_bwd_workspace_bytes(1, L->nkv * L->G, L->nkv, N, d);
  if (L->bwd == 0) return false;
  // Device copies of q, dO, o, dq ([B][Hq][N][d]), k, v, dk, dv ([B][Hkv][N][d]) and lse, then
  // one backward workspace per compute stream.
  const size_t q = (size_t)B * Hq * L->head_q, kv = (size_t)B * Hkv * L->head_q;
  L->total = 4 * align256(q) + 4 * align256(kv) + (size_t)L->chunks * L->lse_chunk + L->streams * align256(L->bwd);
  return true;
}

cudaEvent_t* pipe_events(int dev, int chunks) {
  HostPipe& P = g_pipe[dev];
  if (!P.ready) {
    cudaStream_t* all[] = {&P.in, &P.out_fwd, &P.out_bwd, &P.comp[0], &P.comp[1], &P.comp[2]};
    for (cudaStream_t* sp : all)
      if (cudaStreamCreateWithFlags(sp, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    P.ready = true;
  }
  while ((int)P.ev.size() < 3 + 4 * chunks) {
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
  fa::TraceRange trace("fa_fwd_bwd_host");
  StepLayout L;
  if (!step_layout(B, Hq, Hkv, N, d, &L)) return FA_ERR_INVALID;
  if (!q || !k || !v || !dout || !o || !lse || !dq || !dk || !dv) return FA_ERR_INVALID;
  if (!workspace || workspace_bytes < L.total) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return FA_ERR_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA_ERR_LAUNCH;

  // Device copies of every tensor (same layouts as the host buffers), then the backward
  // workspaces.
  char* w = static_cast<char*>(workspace);
  auto take = [&](size_t bytes) {
    char* p = w;
    w += align256(bytes);
    return p;
  };
  const size_t q_bytes = (size_t)B * Hq * L.head_q, kv_bytes = (size_t)B * Hkv * L.head_q;
  char* d_q = take(q_bytes);
  char* d_k = take(kv_bytes);
  char* d_v = take(kv_bytes);
  char* d_do = take(q_bytes);
  char* d_o = take(q_bytes);
  char* d_lse = take((size_t)L.chunks * L.lse_chunk);
  char* d_dq = take(q_bytes);
  char* d_dk = take(kv_bytes);
  char* d_dv = take(kv_bytes);
  char* d_ws[kComputeStreams];
  for (int s = 0; s < L.streams; ++s) d_ws[s] = take(L.bwd);

  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  cudaEvent_t* ev = pipe_events(dev, L.chunks);
  if (ev == nullptr) return FA_ERR_LAUNCH;
  HostPipe& P = g_pipe[dev];
  const cudaStream_t comp[kComputeStreams] = {st, P.comp[0], P.comp[1], P.comp[2]};
  cudaEvent_t ev_start = ev[0], ev_done_fwd = ev[1], ev_done_bwd = ev[2];
  cudaEvent_t* ev_qkv = ev + 3;                 // q, k, v of chunk c on the device
  cudaEvent_t* ev_do = ev + 3 + L.chunks;       // dO of chunk c on the device
  cudaEvent_t* ev_fwd = ev + 3 + 2 * L.chunks;  // o, lse of chunk c computed
  cudaEvent_t* ev_bwd = ev + 3 + 3 * L.chunks;  // dq, dk, dv of chunk c computed
  const auto H2D = cudaMemcpyHostToDevice;
  const auto D2H = cudaMemcpyDeviceToHost;
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  const char* hdo = static_cast<const char*>(dout);
  char* ho = static_cast<char*>(o);
  char* hl = reinterpret_cast<char*>(lse);
  char* hdq = static_cast<char*>(dq);
  char* hdk = static_cast<char*>(dk);
  char* hdv = static_cast<char*>(dv);
#define FA_CU(x) \
  if ((x) != cudaSuccess) return FA_ERR_LAUNCH
  // Everything the caller enqueued before (including a previous call's use of this workspace)
  // happens first.
  FA_CU(cudaEventRecord(ev_start, st));
  FA_CU(cudaStreamWaitEvent(P.in, ev_start, 0));
  FA_CU(cudaStreamWaitEvent(P.out_fwd, ev_start, 0));
  FA_CU(cudaStreamWaitEvent(P.out_bwd, ev_start, 0));
  for (int s = 1; s < L.streams; ++s) FA_CU(cudaStreamWaitEvent(comp[s], ev_start, 0));
  // Chunk by chunk, so that the first chunks' kernels start while later ones are still being
  // enqueued.
  for (int c = 0; c < L.chunks; ++c) {
    const int b = c / L.split, kv0 = (c % L.split) * L.nkv, hq_c = L.nkv * L.G;
    const size_t oq = ((size_t)b * Hq + (size_t)kv0 * L.G) * L.head_q;
    const size_t okv = ((size_t)b * Hkv + kv0) * L.head_q;
    const size_t ol = ((size_t)b * Hq + (size_t)kv0 * L.G) * L.head_lse;
    const size_t nq = hq_c * L.head_q, nkv = L.nkv * L.head_q, nl = hq_c * L.head_lse;
    float* lse_c = reinterpret_cast<float*>(d_lse + c * L.lse_chunk);
    FA_CU(cudaMemcpyAsync(d_q + oq, hq + oq, nq, H2D, P.in));
    FA_CU(cudaMemcpyAsync(d_k + okv, hk + okv, nkv, H2D, P.in));
    FA_CU(cudaMemcpyAsync(d_v + okv, hv + okv, nkv, H2D, P.in));
    FA_CU(cudaEventRecord(ev_qkv[c], P.in));
    FA_CU(cudaMemcpyAsync(d_do + oq, hdo + oq, nq, H2D, P.in));
    FA_CU(cudaEventRecord(ev_do[c], P.in));

    const int s = c % L.streams;
    const cudaStream_t cs = comp[s];
    const fa_stream_t cs_h = reinterpret_cast<fa_stream_t>(cs);
    FA_CU(cudaStreamWaitEvent(cs, ev_qkv[c], 0));
    int r = fa_fwd(d_q + oq, d_k + okv, d_v + okv, d_o + oq, lse_c, 1, hq_c, L.nkv, N,
                   d, causal, scale, cs_h);
    if (r != FA_OK) return r;
    FA_CU(cudaEventRecord(ev_fwd[c], cs));
    FA_CU(cudaStreamWaitEvent(cs, ev_do[c], 0));
    r = fa_bwd(d_q + oq, d_k + okv, d_v + okv, d_o + oq, d_do + oq, lse_c,
               d_dq + oq, d_dk + okv, d_dv + okv, d_ws[s], L.bwd, 1, hq_c, L.nkv, N, d, causal, scale, cs_h);
    if (r != FA_OK) return r;
    FA_CU(cudaEventRecord(ev_bwd[c], cs));

    FA_CU(cudaStreamWaitEvent(P.out_fwd, ev_fwd[c], 0));
    FA_CU(cudaMemcpyAsync(ho + oq, d_o + oq, nq, D2H, P.out_fwd));
    FA_CU(cudaMemcpyAsync(hl + ol, lse_c, nl, D2H, P.out_fwd));
    FA_CU(cudaStreamWaitEvent(P.out_bwd, ev_bwd[c], 0));
    FA_CU(cudaMemcpyAsync(hdq + oq, d_dq + oq, nq, D2H, P.out_bwd));
    FA_CU(cudaMemcpyAsync(hdk + okv, d_dk + okv, nkv, D2H, P.out_bwd));
    FA_CU(cudaMemcpyAsync(hdv + okv, d_dv + okv, nkv, D2H, P.out_bwd));
  }
  // Every chunk's backward precedes its gradient copies, so the two output streams' ends cover
  // all the work of the call.
  FA_CU(cudaEventRecord(ev_done_fwd, P.out_fwd));
  FA_CU(cudaEventRecord(ev_done_bwd, P.out_bwd));
  FA_CU(cudaStreamWaitEvent(st, ev_done_fwd, 0));
  FA_CU(cudaStreamWaitEvent(st, ev_done_bwd, 0));
#undef FA_CU
  return FA_OK;
}

}  // extern "C"
