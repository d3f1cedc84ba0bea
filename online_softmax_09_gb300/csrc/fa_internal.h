// fa_internal.h -- host-side interface between the C ABI (fa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

namespace fa {

constexpr int kTile = 128;  // query rows and key rows per tile (B_r = B_c = 128)

// A named range on the host timeline around one library call (NVTX), for Nsight tools when one
// is attached; without a tool each push and pop is a call that returns at once.
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

struct FwdLaunch {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_o;  // O as [B*Hq][N][d], box 64 columns x 32 rows (epilogue stores)
  const CUtensorMap* tm_opart;  // split-KV partials as [splits*B*Hq][N][d] fp32, box 32 x 32
  void* o;
  float* lse;
  unsigned long long* counters;  // nullable
  uint32_t* status;
  int B, Hq, Hkv, N, d, causal;
  int window;      // 0: none; > 0: causal sliding window of this many keys
  int num_splits;  // 1: plain; > 1: split-KV into o_part / lse_part, then merged into o / lse
  float* o_part;   // [num_splits][B*Hq][N][d] fp32 (split mode)
  float* lse_part; // [num_splits][B*Hq][N] fp32 (split mode)
  int num_sms;     // persistent grid size
  float scale;
  cudaStream_t stream;
};
cudaError_t launch_fwd(const FwdLaunch& a);

struct BwdLaunch {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_do;
  const CUtensorMap* tm_dq;  // fp32 dQ accumulator viewed as [B*Hq*Npad][d], box 32 x 32
  const CUtensorMap* tm_dk;  // dK, dV as [B*Hkv][N][d], box 64 columns x 32 rows (epilogue stores)
  const CUtensorMap* tm_dv;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  float* dq_acc;   // workspace: [B*Hq][Npad][d] fp32
  float* delta;    // workspace: [B*Hq][Npad] fp32
  float* lse2;     // workspace: [B*Hq][Npad] fp32 (LSE * log2 e; +inf on padded rows)
  uint32_t* next_item;  // workspace: work-item counter of the main kernel (zeroed by prepare)
  uint32_t* status;
  int B, Hq, Hkv, N, d, causal;
  int window;  // 0: none; > 0: causal sliding window
  int num_sms;
  float scale;
  cudaStream_t stream;
};
// Backward stages (bit mask): 1 = prepare (delta, LSE2, zero dQ accumulator), 2 = compute
// (main kernel: dK, dV, dQ accumulation), 4 = finalize (dQ accumulator -> bf16 dq).
enum : int { kBwdPrepare = 1, kBwdCompute = 2, kBwdFinalize = 4, kBwdAll = 7 };
cudaError_t launch_bwd(const BwdLaunch& a, int stages);

// Row-wise online softmax: x, p [rows][n] fp32, lse [rows] (nullable).
cudaError_t launch_softmax_rows(const float* x, float* p, float* lse, long long rows, int n, cudaStream_t st);

// Naive attention baseline (S and P in HBM): workspace bytes and launch (0 ok, 1 no cuBLAS,
// 2 error).
size_t naive_workspace_bytes(int B, int Hq, int N);
int launch_naive_fwd(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace, int B,
                     int Hq, int Hkv, int N, int d, int causal, float scale, cudaStream_t st);

inline int round_up_tile(int n) { return (n + kTile - 1) / kTile * kTile; }

// Unique id of the calling thread's current CUDA context, 0 if there is none (or it cannot be
// read). Context ids are never reused, so a context re-created after cudaDeviceReset has a new
// one: device addresses of module variables cached under an id stay valid while it matches.
unsigned long long current_context_id();

// FA_OK if the current device is an sm_103 GPU; FA_ERR_DEVICE (or FA_ERR_LAUNCH) otherwise.
int check_current_device();

// The argument checks of fa_bwd that need no CUDA call (sizes, pointers): FA_OK or the status
// fa_bwd would return for them.
int check_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* dout, const void* lse,
                   const void* dq, const void* dk, const void* dv, int B, int Hq, int Hkv, int N, int d);

}  // namespace fa
