// lik_internal.h -- declarations shared by the translation units of liblik.
//
// Not part of the public ABI (include/lik.h is).  Every layout of the
// operator is described by one Problem: a list of (query, document) pairs
// in which pair p joins query p / pairs_per_query with
//   all-pairs:  document p % Nd          (pairs_per_query = Nd)
//   pairwise:   document p               (pairs_per_query = 1)
//   kd:         document p  (= b*N + n)  (pairs_per_query = N)
// and writes scores[p] and argmax[p*Lq .. p*Lq+Lq-1].
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace lik {

enum Layout : int { kAllPairs = 0, kPairwise = 1, kKd = 2 };
enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

// Score of a document with no valid token (Late Interaction Kernels README,
// "Scoring interface").  -1e9 = 15625000 * 2^6 is exact in fp32.
constexpr float kEmptyDocScore = -1e9f;

struct Problem {
    int layout;
    int dtype;
    const void* Q;            // [n_query, Lq, dim]
    const void* D;            // [n_doc, Ld, dim]
    const uint8_t* qmask;     // [n_query, Lq] or nullptr
    const uint8_t* dmask;     // [n_doc, Ld] or nullptr
    int64_t n_query;          // Nq | B | B
    int64_t n_doc;            // Nd | B | B*N
    int64_t pairs_per_query;  // Nd | 1 | N
    int64_t n_pairs;          // Nq*Nd | B | B*N
    int64_t Lq, Ld, dim;
    // Set only for the backward of a one-call loss-head step: the grad_D launch
    // also writes *ce_loss = the mean of ce_row_loss[0, n_query), summed in a
    // fixed order (the row losses come from the grad_Q launch before it).
    float* ce_loss = nullptr;
    const float* ce_row_loss = nullptr;
    // Set only inside a one-call step whose backward follows on the stream:
    // the tensor-core all-pairs forward zero-fills fwd_zero (fwd_zero_bytes, a
    // multiple of 16, 16-byte aligned) on the side, and the fp32 grad_D launch
    // of that backward then skips its own zero-fill (grad_d_zeroed).
    void* fwd_zero = nullptr;
    int64_t fwd_zero_bytes = 0;
    bool grad_d_zeroed = false;

    __host__ __device__ int64_t query_of(int64_t p) const { return p / pairs_per_query; }
    __host__ __device__ int64_t doc_of(int64_t p) const {
        return layout == kAllPairs ? p % pairs_per_query : p;
    }
    // Document of the t-th pair of query q (pair q*pairs_per_query + t), without a division.
    __host__ __device__ int64_t doc_of_query_pair(int64_t q, int64_t t) const {
        return layout == kAllPairs ? t : q * pairs_per_query + t;
    }
};

// Device properties the launchers need, cached per device.
struct DeviceInfo {
    int device;
    int sm_count;
    int major, minor;
    int max_smem_optin;
};
const DeviceInfo& device_info(int device);

// Device address of the library's error word (set by a kernel whose bounded
// wait expired), for the current device.
unsigned int* device_error_word();

// Error word codes (bit flags).
constexpr unsigned int kErrTimeout = 1u;    // a bounded pipeline wait expired
constexpr unsigned int kErrBadIndex = 2u;   // a saved argmax was >= Ld (skipped)

// ---- launchers (return cudaSuccess or the launch error) ----------------

// Portable FFMA forward for every dtype, layout and size in range.
cudaError_t launch_fwd_simt(const Problem& P, float* scores, int32_t* argmax,
                            cudaStream_t stream);

// Tensor-core (tcgen05) all-pairs forward for fp16/bf16: dim % 16 == 0,
// dim <= 256, 1 <= Lq <= 128, Ld >= 1.
bool tc_allpairs_eligible(const Problem& P);
cudaError_t launch_fwd_tc_allpairs(const Problem& P, float* scores, int32_t* argmax,
                                   cudaStream_t stream);

// Tensor-core (tcgen05) streaming forward for the pairwise and kd layouts,
// fp16/bf16: dim % 16 == 0, dim <= 256, 1 <= Lq <= 32, Ld >= 1.  It needs a
// device workspace of stream_workspace_bytes(P, P.dmask != nullptr) bytes
// (16-byte aligned): the caller's, or, with workspace == nullptr, one from
// the library's pool.
bool tc_stream_eligible(const Problem& P);
size_t stream_workspace_bytes(const Problem& P, bool has_dmask);
cudaError_t launch_fwd_tc_stream(const Problem& P, float* scores, int32_t* argmax, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

// Tensor-core (tcgen05 kind::tf32, three-product hi/lo split) forward for
// fp32 inputs, every layout: dim % 8 == 0, dim <= 128, 1 <= Lq <= 128, Ld >= 1.
bool tc_f32_eligible(const Problem& P);
cudaError_t launch_fwd_tc_f32(const Problem& P, float* scores, int32_t* argmax, cudaStream_t stream);

// Backward: grad_Q gather and grad_D scatter (grad_D zero-filled first).
cudaError_t launch_bwd_grad_q(const Problem& P, const float* grad_out,
                              const int32_t* argmax, float* grad_Q, cudaStream_t stream);
cudaError_t launch_bwd_grad_d(const Problem& P, const float* grad_out,
                              const int32_t* argmax, float* grad_D, cudaStream_t stream);

// Both fp32 gradients in one launch (grad_D zero-filled first unless
// Problem::grad_d_zeroed): the grad_Q gather also scatters each hit into
// grad_D.  With scores != nullptr the cross-entropy head over the score rows
// runs inside it (g is then not read: grad_scores is written, with row_loss
// and *Problem::ce_loss).  Needs Lq >= 1, pairs_per_query >= 1, dim % 8 == 0,
// dim <= 256; with the head also grad_q_ce_fusable, at most 4096 rows and
// Problem::ce_loss set.
bool bwd_qd_fusable(const Problem& P, bool ce);
cudaError_t launch_bwd_qd(const Problem& P, const float* grad_out, const int32_t* argmax, float* grad_Q,
                          float* grad_D, const float* scores, const int32_t* target, float scale, float* row_loss,
                          float* grad_scores, cudaStream_t stream);

// Backward with gradients in the inputs' 16-bit dtype: fp32 sums, one rounded
// write per element, no zero-fill.  fp16/bf16, dim % 8 == 0, dim <= 256.
bool bwd_same_dtype_supported(const Problem& P);
cudaError_t launch_bwd_grad_q_same(const Problem& P, const float* grad_out, const int32_t* argmax,
                                   void* grad_Q, cudaStream_t stream);
cudaError_t launch_bwd_grad_d_same(const Problem& P, const float* grad_out, const int32_t* argmax,
                                   void* grad_D, cudaStream_t stream);

// The grad_Q gather with the cross-entropy head over the score rows (row =
// query, cols = its pairs) computed inside it: it writes the row losses and
// the score gradient, which the grad_D launch then reads (with
// Problem::ce_loss set, that launch also writes the losses' mean).  Needs
// Lq >= 1, dim % 8 == 0, dim <= 256, rows * cols <= 2^20.
bool grad_q_ce_fusable(const Problem& P);
cudaError_t launch_bwd_grad_q_ce(const Problem& P, const float* scores, const int32_t* target, float scale,
                                 float* row_loss, float* grad_scores, const int32_t* am, void* gQ, bool same_dtype,
                                 cudaStream_t stream);

// Softmax cross-entropy over score rows: per-row losses, their mean and the
// gradient with respect to the scores (grad may be NULL).
cudaError_t launch_ce_rows(const float* scores, int64_t rows, int64_t cols, const int32_t* target, float scale,
                           float* loss, float* row_loss, float* grad, cudaStream_t stream);

}  // namespace lik
