/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact softmax attention library (libfa.so).
 *
 * Operation. For every batch b and query head hq, with kv head hkv = hq / (Hq/Hkv):
 *     S = scale * Q K^T            (N x N, never stored)
 *     S[i][j] = -inf for j > i     (only when causal != 0)
 *     O = softmax_rows(S) V,  LSE_i = log(sum_j exp(S_ij))   (natural log)
 * computed tile by tile with a running max m, running sum l and a rescaled output
 * accumulator ("FlashAttention Implementation > How FlashAttention Uses Tiling",
 * sections "The Running Statistics" and "Why the Correction Factor Works";
 * "LLM Architecture Refresh [3]: Flash Attention Is Exact", sections 2 and 4).
 * Key/value tiles lying wholly in a query tile's causal future are skipped, not masked
 * (same post, section 7). The backward pass recomputes P from Q, K, V and LSE instead
 * of storing it (same post, section 8, its paragraph on the backward pass).
 *
 * Layout. All tensors are dense, row-major and contiguous:
 *     q, o, dout, dq : [B][Hq ][N][d]   bfloat16 (2 bytes, IEEE bfloat16 bit pattern)
 *     k, v, dk, dv   : [B][Hkv][N][d]   bfloat16
 *     lse            : [B][Hq ][N]      float32
 * Supported: d in {64, 128}; N >= 1 (any value, not only multiples of 128); B, Hq, Hkv >= 1;
 * Hq % Hkv == 0. Every pointer is a DEVICE pointer on the current CUDA device and must be
 * 16-byte aligned.
 *
 * Ownership. The caller allocates and owns every buffer, including the backward
 * workspace; the library never allocates device memory (except inside cuBLAS, which only the
 * fa_naive_fwd baseline uses).
 *
 * Streams and errors. `stream` is a cudaStream_t (NULL = legacy default stream). Every call
 * is asynchronous on that stream. The return value reports argument errors (nothing is
 * launched) and launch errors synchronously. A device-side failure (a pipeline wait that
 * exceeded its time limit; the kernel then stops early and its outputs are undefined) is
 * recorded in a per-device status word and reported by fa_check(), which synchronises the
 * stream. No call traps, asserts or spins without bound on the device.
 *
 * scale <= 0 (or NaN) selects the default 1/sqrt(d) ("LLM Architecture Refresh [3]",
 * section 5, sliding_window_attention's scale).
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID = -1,     /* null pointer, non-positive size, Hq % Hkv != 0, size overflow */
  FA_ERR_UNSUPPORTED = -2, /* head dimension d not in {64, 128} */
  FA_ERR_ALIGN = -3,       /* a pointer is not 16-byte aligned */
  FA_ERR_LAUNCH = -4,      /* CUDA launch or runtime error (see cudaGetLastError) */
  FA_ERR_TIMEOUT = -5,     /* a device pipeline wait exceeded its limit; outputs undefined */
  FA_ERR_WORKSPACE = -6,   /* workspace pointer null or smaller than fa_bwd_workspace_bytes() */
  FA_ERR_DEVICE = -7       /* current device is not an sm_103 GPU (this library is sm_103a only) */
} fa_status;

/*
 * Forward pass. Writes o (bf16) and lse (fp32, natural log).
 * Source: "LLM Architecture Refresh [3]", section 4 (tiled loop, O = acc / l after the
 * inner loop) and section 7 (causal tile skipping); LSE = m + ln(l) is the saved statistic
 * that the backward pass needs (section 8).
 * Extra device memory: none.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int Hq, int Hkv, int N, int d, int causal, float scale,
           fa_stream_t stream);

/*
 * Forward pass with a causal sliding window of `window` keys: query i sees keys
 * i - window < j <= i ("LLM Architecture Refresh [3]", section 5, sliding_window_attention:
 * keys older than i - window + 1 or in the future are masked). Key tiles wholly outside every
 * row's window are skipped on both sides. window >= 1 (window >= N is plain causal).
 * Same arguments, layouts and errors as fa_fwd otherwise. Extra device memory: none.
 */
int fa_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int Hq, int Hkv, int N, int d, int window, float scale,
                  fa_stream_t stream);

/*
 * Split-KV forward: the key tiles of every pair of query tiles are divided into num_splits
 * ranges processed by different CTAs, each writing a partial output and its LSE; a merge
 * kernel combines them by the rule that partial softmaxes compose ("LLM Architecture
 * Refresh [3]", section 3): with w_s = exp(LSE_s - max_s LSE_s),
 * O = sum_s w_s O_s / sum_s w_s and LSE = max_s LSE_s + ln(sum_s w_s). Fills the GPU when
 * B * Hq * ceil(N / 256) is below the SM count.
 *   num_splits : 1..64, or <= 0 to let the library choose: fa_fwd_splitkv_auto's count for the
 *                current device (1 unless splitting is predicted to save 10 % or more).
 *   workspace  : device, 16-byte aligned, >= fa_fwd_splitkv_workspace_bytes() bytes for the
 *                splits used (unused when 1 split is used); contents on entry do not matter.
 * Same outputs and errors as fa_fwd; FA_ERR_WORKSPACE if the workspace is too small.
 */
size_t fa_fwd_splitkv_workspace_bytes(int B, int Hq, int Hkv, int N, int d, int num_splits);
/*
 * The split count fa_fwd_splitkv uses for num_splits <= 0 on a GPU with num_sms SMs: the count
 * in {1, 2, 4, 8, 16} with the least time predicted by a cost model of the persistent forward
 * (its longest work item against its work per SM, in key-tile steps) plus the merge and the
 * partial outputs' traffic, chosen only for a predicted gain of 10 % or more. Host-only, needs no
 * GPU. Returns FA_ERR_INVALID (< 0) for invalid sizes or num_sms < 1.
 */
int fa_fwd_splitkv_auto(int B, int Hq, int Hkv, int N, int d, int causal, int num_sms);
int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int Hq, int Hkv, int N, int d, int causal, float scale, int num_splits,
                   void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Same as fa_fwd, and additionally adds to counters[0..2] (device pointer to three
 * unsigned 64-bit integers, which the caller zeroes): [0] key/value tiles computed,
 * [1] key/value tiles skipped by the causal rule, [2] query rows whose running max was
 * raised by a later tile (a rescale of l and O; "LLM Architecture Refresh [3]",
 * section 2, "How often does it fire?"). Tiles are 128 x 128.
 */
int fa_fwd_stats(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                 unsigned long long *counters, fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs: an fp32 dQ accumulator, the per-row
 * delta = rowsum(dO * O) and the base-2 LSE, each over rows padded to a multiple of 128,
 * and 256 bytes for the compute stage's work-item counter.
 * Grows as O(B * Hq * N * d): never with N^2. Returns 0 for invalid sizes.
 */
size_t fa_bwd_workspace_bytes(int B, int Hq, int Hkv, int N, int d);

/*
 * Backward pass: given q, k, v, the forward output o, its gradient dout and lse from
 * fa_fwd (same causal and scale), writes dq, dk, dv (bf16). dk and dv are summed over the
 * Hq/Hkv query heads that share a kv head. P is recomputed tile by tile as
 * exp(scale * q k^T - lse) ("LLM Architecture Refresh [3]", section 8), then
 *     dV = P^T dO,  dP = dO V^T,  delta = rowsum(dO * O),  dS = P * (dP - delta),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 * workspace: device buffer of at least fa_bwd_workspace_bytes() bytes, 16-byte aligned;
 * its contents on entry do not matter. dq is not deterministic bit for bit: the fp32 dQ
 * contributions of different key tiles are added by bulk tensor reductions in whichever order
 * the CTAs reach them.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
           const float *lse, void *dq, void *dk, void *dv,
           void *workspace, size_t workspace_bytes,
           int B, int Hq, int Hkv, int N, int d, int causal, float scale,
           fa_stream_t stream);

/*
 * Backward of fa_fwd_window: the same as fa_bwd for the causal sliding window of `window`
 * keys (query i sees keys i - window < j <= i); query tiles wholly outside a key tile's reach
 * are skipped. window >= 1; workspace as for fa_bwd.
 */
int fa_bwd_window(const void *q, const void *k, const void *v, const void *o, const void *dout,
                  const float *lse, void *dq, void *dk, void *dv,
                  void *workspace, size_t workspace_bytes,
                  int B, int Hq, int Hkv, int N, int d, int window, float scale,
                  fa_stream_t stream);

/*
 * The three stages fa_bwd runs, exposed so that a caller can schedule or time them apart.
 * They must be called in this order on one stream with the same sizes and workspace;
 * fa_bwd(...) is exactly prepare, compute, finalize.
 *   fa_bwd_prepare : -delta = -rowsum(dout * o) and -lse * log2(e) per query row into the
 *                    workspace (negated for the compute kernel's packed arithmetic), and
 *                    zeroes the workspace's fp32 dQ accumulator and work-item counter
 *                    (memory-bound: reads o, dout, lse).
 *   fa_bwd_compute : the recompute kernel: writes dk, dv and adds dQ contributions (before
 *                    the final scale) into the workspace accumulator (reads q, k, v, dout).
 *                    It leaves the counter at zero, so it may be run again (to time it
 *                    alone, say); dq is right only for one compute after each prepare.
 *   fa_bwd_finalize: dq = bf16(scale * accumulator).
 * Same argument meanings, layouts and errors as fa_bwd.
 */
int fa_bwd_prepare(const void *o, const void *dout, const float *lse,
                   void *workspace, size_t workspace_bytes,
                   int B, int Hq, int Hkv, int N, int d, fa_stream_t stream);
int fa_bwd_compute(const void *q, const void *k, const void *v, const void *dout,
                   void *dk, void *dv, void *workspace, size_t workspace_bytes,
                   int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                   fa_stream_t stream);
int fa_bwd_finalize(void *dq, void *workspace, size_t workspace_bytes,
                    int B, int Hq, int Hkv, int N, int d, float scale, fa_stream_t stream);

/*
 * Backward pass for callers that cannot allocate device memory. The pages this library
 * follows have no counterpart to this entry point; it exists for callers that must not call
 * cudaMalloc, such as a plugin inside a host runtime that owns and budgets all device memory,
 * or a latency-critical loop where cudaMalloc's implicit device synchronisation is not
 * allowed. It computes exactly what fa_bwd computes (same arguments, minus the workspace) and
 * takes the workspace from a fixed device array of FA_BWD_NOALLOC_MAX_BYTES bytes inside the
 * library, which every GPU that loads the library holds until the process exits.
 *   - Returns FA_ERR_WORKSPACE, launching nothing, when fa_bwd_workspace_bytes(B, Hq, Hkv, N, d)
 *     exceeds FA_BWD_NOALLOC_MAX_BYTES (64 MiB: e.g. B*Hq*N up to about 129,000 query rows
 *     at d = 128, or 254,000 at d = 64; rows are counted after rounding N up to a multiple of 128).
 *   - The first call on a device (and the first after the device context is re-created, e.g.
 *     by cudaDeviceReset) looks up the array's device address (with that device
 *     current) and caches it; make that first call before any stream capture.
 *   - All calls on a device share the one array. Calls whose kernels overlap on the GPU (on
 *     different streams, or from different threads) race on it and give wrong results;
 *     serialise them. Calls in sequence are safe: each call clears what must start at zero.
 *   - Nothing is allocated or freed.
 */
#define FA_BWD_NOALLOC_MAX_BYTES ((size_t)64 << 20)
int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const void *dout,
                   const float *lse, void *dq, void *dk, void *dv,
                   int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                   fa_stream_t stream);

/*
 * Forward and backward pass of one attention layer on HOST buffers: the computations of
 * fa_fwd then fa_bwd ("LLM Architecture Refresh [3]", sections 4 and 8) with the
 * host<->device copies done by the library and overlapped with the kernels. The pages have no
 * counterpart for the data movement.
 *   q, k, v, dout: host inputs, same layouts and types as fa_fwd / fa_bwd.
 *   o (bf16), lse (fp32), dq, dk, dv (bf16): host outputs, same layouts as there.
 *   workspace: device memory of at least fa_fwd_bwd_host_workspace_bytes(...) bytes, 256-byte
 *     aligned; it holds device copies of all nine tensors and one backward workspace (sized
 *     for one chunk) per compute stream.
 * The work runs in chunks: each chunk is one batch element's slice of Hkv/s whole kv heads and
 * the query heads that read them, s the smallest divisor of Hkv with B*s >= 8 (or Hkv). While
 * the kernels of some chunks run, the inputs of later chunks are copied in and the outputs of
 * earlier ones out. Chunk c computes on compute stream c mod min(B*s, 4), stream 0 being
 * `stream`, so that several chunks' kernels share the GPU.
 * The library creates its six streams once per device. Host buffers must be page-locked (pinned)
 * for the copies to overlap; pageable buffers give correct results without the overlap. The
 * call is asynchronous like the others: the outputs are complete once `stream` has passed this
 * call (e.g. after fa_check(stream)), and the call starts after everything enqueued on `stream`
 * before it. Calls on one device are serialised by the library on the host. Errors as for
 * fa_fwd and fa_bwd, plus FA_ERR_WORKSPACE (workspace missing or too small) and FA_ERR_ALIGN
 * (workspace not 256-byte aligned); after an error some copies or kernels may already have
 * been enqueued and the outputs are undefined.
 */
size_t fa_fwd_bwd_host_workspace_bytes(int B, int Hq, int Hkv, int N, int d);
int fa_fwd_bwd_host(const void *q, const void *k, const void *v, const void *dout,
                    void *o, float *lse, void *dq, void *dk, void *dv,
                    int B, int Hq, int Hkv, int N, int d, int causal, float scale,
                    void *workspace, size_t workspace_bytes, fa_stream_t stream);

/*
 * Baseline: standard attention with the N x N score matrix in HBM ("LLM Architecture
 * Refresh [3]", section 1: S = QK^T written out, read back for P = softmax(S), written, read
 * back for O = PV). S (fp32) and P (bf16) live in the workspace; the two products are cuBLAS
 * batched GEMMs (fp32 accumulation), the masked softmax a kernel of this library. Same
 * outputs as fa_fwd. Exists to measure what tiling saves; it needs O(B * Hq * N^2) bytes.
 *   workspace: >= fa_naive_workspace_bytes() bytes, 16-byte aligned.
 * cuBLAS is loaded at the first call (FA_ERR_UNSUPPORTED if it cannot be found) and keeps a
 * handle, with its own device memory, per device.
 */
size_t fa_naive_workspace_bytes(int B, int Hq, int Hkv, int N, int d);
int fa_naive_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                 void *workspace, size_t workspace_bytes,
                 int B, int Hq, int Hkv, int N, int d, int causal, float scale, fa_stream_t stream);

/*
 * Row-wise softmax by the online normaliser ("LLM Architecture Refresh [3]", section 2, "Online
 * softmax: the one idea", and section 3, "Partial softmaxes compose"): for each row of x,
 * a running max m and sum l = sum exp(x - m) are carried in one pass, partial (m, l) pairs are
 * merged by rebasing to the larger max, then p = exp(x - m) / l and lse = m + ln l.
 *   x, p : [rows][n] fp32, device, 16-byte aligned, not overlapping.
 *   lse  : [rows] fp32, device, or NULL.
 * Entries equal to -inf get p = 0 (masked logits); a row with no finite entry is undefined.
 * Rows of up to 8192 elements (n a multiple of 4) are read once; longer rows twice.
 */
int fa_softmax_rows(const float *x, float *p, float *lse, long long rows, int n, fa_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status word:
 * FA_OK, FA_ERR_TIMEOUT (a kernel gave up waiting) or FA_ERR_LAUNCH (the stream reported
 * a CUDA error).
 */
int fa_check(fa_stream_t stream);

/*
 * Self-test of the device failure path (the pages have no counterpart). Launches one warp
 * that waits, with the same bounded wait every pipeline wait of the kernels uses, on a
 * barrier that nothing completes. After the wait's time limit (2 s) the warp records the
 * timeout in the device status word, as a stuck kernel would, and the kernel returns, so the
 * context stays usable. *result (a device int) receives 2 when the wait gave up and raised
 * its abort flag (1 if it had completed, 3 otherwise). The following fa_check(stream) returns
 * FA_ERR_TIMEOUT and clears the status. Argument errors: FA_ERR_INVALID for a null result.
 */
int fa_selftest_wait_timeout(int *result, fa_stream_t stream);

/* Static, human-readable description of a status code. */
const char *fa_strerror(int status);

/* ABI version: (major << 16) | minor. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
