/*
 * lik.h -- C ABI of liblik, a GB300 (sm_103a) implementation of the
 * late-interaction MaxSim operator.
 *
 * The operator (Late Interaction Kernels README, "What does it compute?"):
 *
 *     score(q, d) = sum over valid query tokens i of
 *                   max over valid document tokens j of  Q[q,i,:] . D[d,j,:]
 *
 * Semantics shared by every entry point (README, "Scoring interface" and
 * "Precision and compatibility"):
 *   - Q and D share one dtype (fp32, fp16 or bf16) and one embedding size
 *     `dim`; the library never normalises them (raw dot products).
 *   - Masks are 1 byte per token (C `bool`, torch.bool): nonzero = valid,
 *     0 = padding.  A NULL mask means every token is valid.  A query mask
 *     removes token i from the sum; a document mask removes token j from the
 *     max.
 *   - A document with no valid token scores exactly -1e9, whatever the query.
 *     A non-empty document scored against a query with no valid token
 *     scores 0.
 *   - Scores are fp32.  Similarities accumulate in fp32: fp16/bf16 inputs on
 *     the tensor cores (tcgen05, fp32 accumulators), fp32 inputs with fp32
 *     FMA (never TF32).
 *   - argmax[..., i] is the document-token index j (0 <= j < Ld, counted
 *     within its own document) whose similarity is the max for query token
 *     i; the lowest such j on exact ties.  It is -1 for a masked query token
 *     and for every token of an empty document.
 *
 * Backward (README, "What does it compute?": gradients flow into query and
 * document embeddings; LIK announcement thread, post 5/N: the backward is
 * fused).  The score is piecewise linear; with upstream gradient g per score
 *     grad_Q[q,i,:] = sum over pairs (q,d) of g[q,d] * D[d, argmax[q,d,i], :]
 *     grad_D[d,j,:] = sum over (q,i) with argmax[q,d,i] == j of g[q,d] * Q[q,i,:]
 * Entries with argmax -1 contribute nothing, so grad_out of an empty
 * document is ignored.  The backward reads the masks only through the
 * argmax that the forward saved.  grad_Q is summed in a fixed order.  An
 * fp32 grad_D is zero-filled and then receives every hit as an fp32 atomic
 * addition, so its last bits can change from run to run.  With both fp32
 * gradients requested, dim % 8 == 0 and dim <= 256, a single launch writes
 * both; otherwise each gradient takes its own launch.
 *
 * Memory, ownership, streams:
 *   - Every pointer is a device pointer (cudaMalloc or managed memory) of
 *     the current device, row-major and contiguous.  Q, D, grad_Q and grad_D
 *     must be 16-byte aligned; scores, argmax and grad_out 4-byte aligned.
 *     Host pointers are rejected with LIK_ERR_INVALID_ARG.
 *   - The caller allocates every buffer, outputs included.  The one device
 *     allocation the library makes is the workspace of the fp16/bf16 pairwise
 *     and kd forward (the streaming kernel's schedule: with a document mask,
 *     4 bytes per pair and 16 bytes per 128-token document tile; always
 *     about 0.5 KB per SM) when the caller does not pass one: the
 *     lik_maxsim_{pairwise,kd}_fwd_ws entry points take it from the caller
 *     (its size from lik_maxsim_{pairwise,kd}_fwd_workspace_bytes) and
 *     allocate nothing; the plain _fwd entry points take it with
 *     cudaMallocFromPoolAsync from a library-owned memory pool of the device
 *     and release it with cudaFreeAsync on `stream` after the kernel.  The
 *     pool keeps the memory it has mapped for later calls.  The library keeps
 *     no other per-call state.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream).
 *     Outputs are complete when the stream reaches the call.  Gradients are
 *     overwritten, not accumulated into.
 *   - Functions are thread-safe.
 *   - Per device, the library looks up the device addresses of its own
 *     status word (and of the no-allocation entry point's array, below) on
 *     its first call with that device current and keeps them for the
 *     process's life.  Resetting the device (cudaDeviceReset) after that
 *     invalidates them: a process that resets a device must not call the
 *     library on it again.
 *
 * Errors:
 *   - LIK_ERR_INVALID_ARG: a negative size, a NULL required pointer, a host
 *     pointer, a misaligned Q/D, an unknown dtype.  Nothing is launched.
 *   - LIK_ERR_UNSUPPORTED: the current device is not sm_103 (GB300), or a
 *     size is beyond the documented limits.  Nothing is launched.  There is
 *     no fallback to another backend.
 *   - LIK_ERR_CUDA: a CUDA call or launch failed; the CUDA error is
 *     propagated, never swallowed (colpali PR "Add support for
 *     late-interaction-kernels (LIK)", Design section: real kernel errors
 *     always propagate).  lik_last_error_message() names it.
 *   - LIK_ERR_TIMEOUT: reported by lik_check_device_error() when a kernel's
 *     bounded pipeline wait expired; the kernel stopped and its outputs are
 *     not valid.
 *
 * Sizes: 0 <= Nq, Nd, B, N; 0 <= Lq, Ld; 1 <= dim <= 1024.  Zero pairs is a
 * no-op.  Ld == 0 makes every document empty (-1e9).  Lq == 0 gives 0 for
 * every non-empty document.
 */
#ifndef LIK_H
#define LIK_H

#include <stdbool.h>
#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LIK_F32 = 0,
    LIK_F16 = 1,
    LIK_BF16 = 2
} lik_dtype;

typedef enum {
    LIK_OK = 0,
    LIK_ERR_INVALID_ARG = 1,
    LIK_ERR_UNSUPPORTED = 2,
    LIK_ERR_CUDA = 3,
    LIK_ERR_TIMEOUT = 4
} lik_status;

/* Static, never-NULL description of a status code. */
const char* lik_status_string(lik_status status);

/* Human-readable detail of the last non-OK status returned on the calling
 * host thread ("" if none).  Valid until the next call on that thread. */
const char* lik_last_error_message(void);

/* Library version string, e.g. "0.1.0". */
const char* lik_version(void);

/*
 * Synchronises `stream`, then reads and clears the device-side error word
 * that kernels set when a bounded wait expires.  Returns LIK_ERR_TIMEOUT if
 * it was set, LIK_ERR_CUDA if the stream reported a CUDA error, LIK_OK
 * otherwise.  This is the only entry point that blocks the host.
 */
lik_status lik_check_device_error(cudaStream_t stream);

/*
 * Self-test of the failure path of the kernels' bounded waits.  Launches on
 * `stream` one thread that waits, with the same bounded mbarrier wait the
 * tensor-core pipelines use and a limit of `timeout_us` microseconds, on an
 * mbarrier that nothing ever arrives at; when the limit passes it sets the
 * device error word and returns.  A following lik_check_device_error(stream)
 * must then return LIK_ERR_TIMEOUT (and clear the word), and the context
 * stays usable.  No copy, MMA or tensor memory is involved.  The pages have
 * no counterpart to this entry point; it exists to test that a wait that
 * runs out reaches the caller as a status (colpali PR "Add support for
 * late-interaction-kernels (LIK)", Design section: kernel failures are
 * reported, never hidden).
 *   timeout_us  1 .. 1000000, else LIK_ERR_INVALID_ARG (nothing launched)
 */
lik_status lik_selftest_bounded_wait(int64_t timeout_us, cudaStream_t stream);

/* ------------------------------------------------------------ all-pairs --
 * README "Scoring interface" table, layer MaxSim: every query against every
 * document, the layout of in-batch contrastive training.
 *   Q      [Nq, Lq, dim]   dtype
 *   D      [Nd, Ld, dim]   dtype
 *   qmask  [Nq, Lq]        or NULL
 *   dmask  [Nd, Ld]        or NULL
 *   scores [Nq, Nd]        fp32, written
 *   argmax [Nq, Nd, Lq]    int32, written; NULL for inference (no backward)
 */
lik_status lik_maxsim_allpairs_fwd(const void* Q, const void* D, lik_dtype dtype,
                                   int64_t Nq, int64_t Nd, int64_t Lq, int64_t Ld,
                                   int64_t dim, const bool* qmask, const bool* dmask,
                                   float* scores, int32_t* argmax, cudaStream_t stream);

/*
 *   grad_out [Nq, Nd]        fp32
 *   argmax   [Nq, Nd, Lq]    int32, as written by lik_maxsim_allpairs_fwd
 *   grad_Q   [Nq, Lq, dim]   fp32, overwritten; NULL to skip
 *   grad_D   [Nd, Ld, dim]   fp32, overwritten; NULL to skip
 */
lik_status lik_maxsim_allpairs_bwd(const void* Q, const void* D, lik_dtype dtype,
                                   int64_t Nq, int64_t Nd, int64_t Lq, int64_t Ld,
                                   int64_t dim, const float* grad_out,
                                   const int32_t* argmax, float* grad_Q, float* grad_D,
                                   cudaStream_t stream);

/* ------------------------------------------------------------- pairwise --
 * README "Scoring interface" table, layer MaxSimPairwise: query b against
 * document b only, the reranking layout, with no query-by-document cross
 * product computed.
 *   Q [B, Lq, dim], D [B, Ld, dim], qmask [B, Lq], dmask [B, Ld],
 *   scores [B], argmax [B, Lq] (or NULL)
 * fp16/bf16 with dim % 16 == 0, dim <= 256 and Lq <= 32 take the streaming
 * tensor-core kernel: a plan kernel over the document mask, then the forward,
 * both on `stream`, with the pooled workspace described above.
 */
lik_status lik_maxsim_pairwise_fwd(const void* Q, const void* D, lik_dtype dtype,
                                   int64_t B, int64_t Lq, int64_t Ld, int64_t dim,
                                   const bool* qmask, const bool* dmask,
                                   float* scores, int32_t* argmax, cudaStream_t stream);

/*   grad_out [B], argmax [B, Lq], grad_Q [B, Lq, dim], grad_D [B, Ld, dim] */
lik_status lik_maxsim_pairwise_bwd(const void* Q, const void* D, lik_dtype dtype,
                                   int64_t B, int64_t Lq, int64_t Ld, int64_t dim,
                                   const float* grad_out, const int32_t* argmax,
                                   float* grad_Q, float* grad_D, cudaStream_t stream);

/* ------------------------------------- caller-provided forward workspace --
 * The pairwise and kd forward with its schedule workspace supplied by the
 * caller, so that the library allocates no device memory at all: for a
 * caller that manages every byte of device memory itself.  The pages have
 * no counterpart; their layers (README, "Scoring interface") take only the
 * operator's own tensors.
 *
 * lik_maxsim_{pairwise,kd}_fwd_workspace_bytes writes to *bytes the size of
 * the workspace the matching _fwd_ws call needs for these sizes, dtype and
 * whether a document mask is passed (has_dmask != 0), on the current device
 * (it depends on the device's SM count); 0 when the call takes a kernel
 * that needs none (fp32 inputs, shapes outside the streaming kernel's
 * limits).  It launches nothing.
 *
 * lik_maxsim_{pairwise,kd}_fwd_ws: the _fwd entry point with
 *   workspace        device memory of the current device, 16-byte aligned,
 *                    at least the queried size (may be NULL when that is 0);
 *                    overwritten; no contents need to survive between calls
 *   workspace_bytes  its size
 * A workspace that is NULL, too small, misaligned or not device memory gives
 * LIK_ERR_INVALID_ARG and nothing is launched.  Calls that overlap on the
 * GPU must not share a workspace (order them, or give each its own).  The
 * results are bit-identical to the _fwd entry point's.
 */
lik_status lik_maxsim_pairwise_fwd_workspace_bytes(lik_dtype dtype, int64_t B, int64_t Lq, int64_t Ld,
                                                  int64_t dim, int has_dmask, size_t* bytes);

lik_status lik_maxsim_pairwise_fwd_ws(const void* Q, const void* D, lik_dtype dtype, int64_t B,
                                      int64_t Lq, int64_t Ld, int64_t dim, const bool* qmask,
                                      const bool* dmask, float* scores, int32_t* argmax,
                                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------- per-query candidates --
 * colpali PR "Add support for late-interaction-kernels (LIK)", Design
 * section (maxsim_kd, the per-query candidate layout used by the
 * negative-document losses): query b against its own N candidates.
 *   Q [B, Lq, dim], D [B, N, Ld, dim], qmask [B, Lq], dmask [B, N, Ld],
 *   scores [B, N], argmax [B, N, Lq] (or NULL)
 * The same streaming kernel (and workspace) as the pairwise layout.
 */
lik_status lik_maxsim_kd_fwd(const void* Q, const void* D, lik_dtype dtype,
                             int64_t B, int64_t N, int64_t Lq, int64_t Ld, int64_t dim,
                             const bool* qmask, const bool* dmask,
                             float* scores, int32_t* argmax, cudaStream_t stream);

/* The kd forward with a caller-provided workspace: see the pairwise
 * _fwd_workspace_bytes / _fwd_ws entry points above. */
lik_status lik_maxsim_kd_fwd_workspace_bytes(lik_dtype dtype, int64_t B, int64_t N, int64_t Lq,
                                            int64_t Ld, int64_t dim, int has_dmask, size_t* bytes);

lik_status lik_maxsim_kd_fwd_ws(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t N,
                                int64_t Lq, int64_t Ld, int64_t dim, const bool* qmask,
                                const bool* dmask, float* scores, int32_t* argmax, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*   grad_out [B, N], argmax [B, N, Lq], grad_Q [B, Lq, dim], grad_D [B, N, Ld, dim] */
lik_status lik_maxsim_kd_bwd(const void* Q, const void* D, lik_dtype dtype,
                             int64_t B, int64_t N, int64_t Lq, int64_t Ld, int64_t dim,
                             const float* grad_out, const int32_t* argmax,
                             float* grad_Q, float* grad_D, cudaStream_t stream);

/* ------------------------------------------- gradients in the inputs' dtype --
 * The same backward with grad_Q and grad_D in the dtype of Q and D instead of
 * fp32, so a bf16/fp16 training step keeps no fp32 gradient buffers and writes
 * half the bytes (colpali PR "Add support for late-interaction-kernels
 * (LIK)", Results: the fused backward's memory is the two input gradients,
 * and writing grad_D is most of its cost).  Every element is summed in
 * fp32 and rounded to the output type once (round to nearest even); each
 * row of grad_D is written exactly once, zeros included.
 *   - fp32 inputs: identical to the fp32 entry points.
 *   - fp16/bf16 inputs: need dim % 8 == 0 and dim <= 256, else
 *     LIK_ERR_UNSUPPORTED (the fp32-gradient entry points take any dim).
 *   - grad_Q, grad_D: same shapes as Q and D, dtype of Q and D, 16-byte
 *     aligned, overwritten; NULL to skip.  Other arguments and errors as in
 *     the fp32-gradient entry points above.
 */
lik_status lik_maxsim_allpairs_bwd_same_dtype(const void* Q, const void* D, lik_dtype dtype,
                                              int64_t Nq, int64_t Nd, int64_t Lq, int64_t Ld,
                                              int64_t dim, const float* grad_out,
                                              const int32_t* argmax, void* grad_Q, void* grad_D,
                                              cudaStream_t stream);

lik_status lik_maxsim_pairwise_bwd_same_dtype(const void* Q, const void* D, lik_dtype dtype,
                                              int64_t B, int64_t Lq, int64_t Ld, int64_t dim,
                                              const float* grad_out, const int32_t* argmax,
                                              void* grad_Q, void* grad_D, cudaStream_t stream);

lik_status lik_maxsim_kd_bwd_same_dtype(const void* Q, const void* D, lik_dtype dtype, int64_t B,
                                        int64_t N, int64_t Lq, int64_t Ld, int64_t dim,
                                        const float* grad_out, const int32_t* argmax,
                                        void* grad_Q, void* grad_D, cudaStream_t stream);

/* ------------------------------------------- backward that recomputes argmax --
 * For an argmax-free training forward (call the _fwd entry point with argmax
 * = NULL, which saves only the scores; the LIK announcement thread, post
 * 5/N, and the colpali PR's Results describe the fused path as holding only
 * the score output between forward and backward): the backward re-runs the
 * forward into `argmax_workspace` and then runs the _bwd entry point on it.
 * So the int32 argmax [pairs, Lq] exists only for the duration of this call
 * (the caller may share one workspace between calls on one stream).
 *   qmask, dmask            as passed to the forward (the argmax depends on them)
 *   argmax_workspace        int32 [pairs, Lq], device, 4-byte aligned, required;
 *                           overwritten, its contents after the call are the argmax
 *   grad_out, grad_Q, grad_D as in the _bwd entry points (fp32 gradients)
 * Cost: one forward (with argmax) plus one backward.  Errors as in _fwd and
 * _bwd.
 */
lik_status lik_maxsim_allpairs_bwd_recompute(const void* Q, const void* D, lik_dtype dtype,
                                             int64_t Nq, int64_t Nd, int64_t Lq, int64_t Ld,
                                             int64_t dim, const bool* qmask, const bool* dmask,
                                             const float* grad_out, int32_t* argmax_workspace,
                                             float* grad_Q, float* grad_D, cudaStream_t stream);

lik_status lik_maxsim_pairwise_bwd_recompute(const void* Q, const void* D, lik_dtype dtype,
                                             int64_t B, int64_t Lq, int64_t Ld, int64_t dim,
                                             const bool* qmask, const bool* dmask,
                                             const float* grad_out, int32_t* argmax_workspace,
                                             float* grad_Q, float* grad_D, cudaStream_t stream);

lik_status lik_maxsim_kd_bwd_recompute(const void* Q, const void* D, lik_dtype dtype, int64_t B,
                                       int64_t N, int64_t Lq, int64_t Ld, int64_t dim,
                                       const bool* qmask, const bool* dmask,
                                       const float* grad_out, int32_t* argmax_workspace,
                                       float* grad_Q, float* grad_D, cudaStream_t stream);

/*
 * The same all-pairs recompute backward for callers that cannot allocate
 * device memory (for example a memory manager that owns the whole device,
 * or a loop that cannot pay for cudaMalloc): the argmax workspace is an
 * array built into the library, 2^21 int32 entries (8 MiB), held on every
 * GPU that loads the library until the process exits.  The pages have no
 * counterpart to this entry point.
 *   - Nq * Nd * Lq <= 2097152, else LIK_ERR_UNSUPPORTED (nothing launched).
 *   - Nothing is allocated.  The first call on a device, with that device
 *     current, looks up the array's device address (cudaGetSymbolAddress);
 *     make that first call before any stream capture, and do not reset the
 *     device afterwards (the address is kept for the process's life).
 *   - Every call shares the array; calls whose work overlaps on the GPU
 *     race on it, so order them (one stream, or events).  Its contents need
 *     no clearing: the forward writes every entry the backward reads.
 *   - Other arguments, outputs and errors as in
 *     lik_maxsim_allpairs_bwd_recompute.
 */
lik_status lik_maxsim_allpairs_bwd_recompute_noalloc(const void* Q, const void* D,
                                                     lik_dtype dtype, int64_t Nq, int64_t Nd,
                                                     int64_t Lq, int64_t Ld, int64_t dim,
                                                     const bool* qmask, const bool* dmask,
                                                     const float* grad_out, float* grad_Q,
                                                     float* grad_D, cudaStream_t stream);

/* --------------------------------------------------- cross-entropy head --
 * colpali PR "Add support for late-interaction-kernels (LIK)": "What this PR
 * adds" routes the in-batch ColBERT losses (a query against the batch's
 * documents, its own document the target) and the negative-document losses
 * (a query against its own candidates, the positive first, via the kd
 * layout) through the kernel; "Results" time that loss head forward and
 * backward.
 *
 * lik_ce_rows: softmax cross-entropy over the rows of scores[rows, cols]
 * with logits z = scale * scores[r, :] and target[r]:
 *     row_loss[r]       = log(sum_c exp(z_c)) - z_target         (fp32, written)
 *     *loss             = mean over rows of row_loss             (fp32, written)
 *     grad_scores[r, c] = scale * (softmax(z)_c - [c == target]) / rows
 *                         (the gradient of *loss; written unless NULL)
 * A target outside [0, cols) leaves its row out (row_loss 0, zero gradient);
 * the mean still divides by rows.  Rows of -1e9 (empty documents) add
 * nothing to the softmax.  The mean is summed in a fixed order.
 *   scores [rows, cols], target [rows] int32, loss [1], row_loss [rows]:
 *   device pointers, 4-byte aligned; all but grad_scores required.
 */
lik_status lik_ce_rows(const float* scores, int64_t rows, int64_t cols, const int32_t* target,
                       float scale, float* loss, float* row_loss, float* grad_scores,
                       cudaStream_t stream);

/*
 * One loss-head training step on `stream`, with no host synchronisation:
 * the forward (scores and argmax), lik_ce_rows over the score rows
 * (all-pairs: rows = Nq, cols = Nd; kd: rows = B, cols = N), then the
 * backward with grad_out = grad_scores.  Gradients are fp32 (grad_Q, grad_D
 * as float*) or, with grads_in_input_dtype != 0, in the inputs' dtype as in
 * the _bwd_same_dtype entry points.  Arguments, shapes and errors as in the
 * entry points it calls; scores, argmax, loss, row_loss and grad_scores are
 * caller-allocated outputs.  It returns the first non-OK status.
 *
 * The results are those of the three calls in that order; the launches
 * differ.  When grad_Q and grad_D are both given, dim % 8 == 0, dim <= 256
 * and rows * cols <= 2^20, the loss head runs inside the backward.  With fp32
 * gradients and at most 4096 rows the backward is one launch: its blocks
 * compute their row's log-sum-exp and grad_scores before they use them, and
 * one more block writes row_loss and *loss (the same fixed-order mean).
 * Otherwise the grad_Q launch computes the log-sum-exp, row_loss and
 * grad_scores, and the grad_D launch's first block writes *loss.  With fp32
 * gradients and the fp16/bf16 all-pairs forward, the forward also zero-fills
 * grad_D (16-byte aligned, element count a multiple of 4) on its producer
 * warp instead of a separate memset.
 */
lik_status lik_maxsim_allpairs_ce_step(const void* Q, const void* D, lik_dtype dtype, int64_t Nq,
                                       int64_t Nd, int64_t Lq, int64_t Ld, int64_t dim,
                                       const bool* qmask, const bool* dmask,
                                       const int32_t* target, float scale, float* scores,
                                       int32_t* argmax, float* loss, float* row_loss,
                                       float* grad_scores, void* grad_Q, void* grad_D,
                                       int grads_in_input_dtype, cudaStream_t stream);

lik_status lik_maxsim_kd_ce_step(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t N,
                                 int64_t Lq, int64_t Ld, int64_t dim, const bool* qmask,
                                 const bool* dmask, const int32_t* target, float scale,
                                 float* scores, int32_t* argmax, float* loss, float* row_loss,
                                 float* grad_scores, void* grad_Q, void* grad_D,
                                 int grads_in_input_dtype, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LIK_H */
