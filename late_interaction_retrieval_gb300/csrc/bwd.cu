// bwd.cu -- MaxSim backward: grad_Q gather and grad_D scatter.
//
// The score is piecewise linear in Q and D; for every valid query token i of
// a non-empty document only the term Q[q,i].D[d,a] with a = argmax is active
// (Late Interaction Kernels README, "What does it compute?": gradients flow
// into query and document embeddings).  With upstream gradient g per score:
//
//   grad_Q[q,i,:] = sum over the pairs p of query q of g[p] * D[doc(p), a[p,i], :]
//   grad_D[d,j,:] = sum over the pairs p of document d and tokens i with
//                   a[p,i] == j of g[p] * Q[query(p), i, :]
//
// argmax -1 (masked query token, empty document) contributes nothing.  The
// backward allocates nothing: it writes the two input gradients only (colpali
// PR "Add support for late-interaction-kernels (LIK)", Results: the fused
// backward allocates only the input gradients).
#include "dtype_load.cuh"
#include "lik_internal.h"

namespace lik {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// One warp per (query, token) row of grad_Q; lanes stride over dim.  The
// pairs of a query are visited in ascending order, so the fp32 sum order is
// fixed.
template <typename T>
__global__ void __launch_bounds__(kThreads)
grad_q_gather_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                     float* __restrict__ gQ, unsigned int* err) {
    const T* D = static_cast<const T*>(P.D);
    const int lane = threadIdx.x & 31;
    const int64_t rows = P.n_query * P.Lq;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); row < rows;
         row += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int64_t q = row / P.Lq, i = row - q * P.Lq;
        for (int64_t k0 = 0; k0 < P.dim; k0 += 128) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int64_t t = 0; t < P.pairs_per_query; ++t) {
                const int64_t p = q * P.pairs_per_query + t;
                const int32_t a = am[p * P.Lq + i];
                if (a < 0) continue;  // warp-uniform
                if (a >= P.Ld) {      // not an index the forward writes: flag, never touch memory
                    if (lane == 0) atomicOr(err, kErrBadIndex);
                    continue;
                }
                const float gv = g[p];
                const T* drow = D + (P.doc_of(p) * P.Ld + a) * P.dim;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int64_t k = k0 + lane + 32 * m;
                    if (k < P.dim) acc[m] = fmaf(gv, load_f32(drow + k), acc[m]);
                }
            }
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int64_t k = k0 + lane + 32 * m;
                if (k < P.dim) gQ[row * P.dim + k] = acc[m];
            }
        }
    }
}

// One warp per (pair, token) hit; adds g * Q[q,i,:] into grad_D[d, a, :]
// with fp32 atomics.  grad_D is zero-filled on the stream first.
template <typename T>
__global__ void __launch_bounds__(kThreads)
grad_d_scatter_atomic_kernel(Problem P, const float* __restrict__ g,
                             const int32_t* __restrict__ am, float* __restrict__ gD,
                             unsigned int* err) {
    const T* Q = static_cast<const T*>(P.Q);
    const int lane = threadIdx.x & 31;
    const int64_t hits = P.n_pairs * P.Lq;
    for (int64_t h = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); h < hits;
         h += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int32_t a = am[h];
        if (a < 0) continue;  // warp-uniform
        if (a >= P.Ld) {
            if (lane == 0) atomicOr(err, kErrBadIndex);
            continue;
        }
        const int64_t p = h / P.Lq, i = h - p * P.Lq;
        const float gv = g[p];
        const T* qrow = Q + (P.query_of(p) * P.Lq + i) * P.dim;
        float* out = gD + (P.doc_of(p) * P.Ld + a) * P.dim;
        for (int64_t k = lane; k < P.dim; k += 32) atomicAdd(out + k, gv * load_f32(qrow + k));
    }
}

unsigned grid_for(int64_t warps_of_work) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t cap = static_cast<int64_t>(device_info(dev).sm_count) * 16;
    int64_t blocks = (warps_of_work + kWarps - 1) / kWarps;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_bwd_grad_q(const Problem& P, const float* g, const int32_t* am, float* gQ,
                              cudaStream_t stream) {
    const int64_t rows = P.n_query * P.Lq;
    if (rows == 0) return cudaSuccess;
    const unsigned blocks = grid_for(rows);
    unsigned int* err = device_error_word();
    switch (P.dtype) {
    case kF32: grad_q_gather_kernel<float><<<blocks, kThreads, 0, stream>>>(P, g, am, gQ, err); break;
    case kF16: grad_q_gather_kernel<__half><<<blocks, kThreads, 0, stream>>>(P, g, am, gQ, err); break;
    default: grad_q_gather_kernel<__nv_bfloat16><<<blocks, kThreads, 0, stream>>>(P, g, am, gQ, err);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_grad_d(const Problem& P, const float* g, const int32_t* am, float* gD,
                              cudaStream_t stream) {
    const int64_t elems = P.n_doc * P.Ld * P.dim;
    if (elems == 0) return cudaSuccess;
    const cudaError_t e = cudaMemsetAsync(gD, 0, sizeof(float) * elems, stream);
    if (e != cudaSuccess) return e;
    const int64_t hits = P.n_pairs * P.Lq;
    if (hits == 0) return cudaSuccess;
    const unsigned blocks = grid_for(hits);
    unsigned int* err = device_error_word();
    switch (P.dtype) {
    case kF32: grad_d_scatter_atomic_kernel<float><<<blocks, kThreads, 0, stream>>>(P, g, am, gD, err); break;
    case kF16: grad_d_scatter_atomic_kernel<__half><<<blocks, kThreads, 0, stream>>>(P, g, am, gD, err); break;
    default: grad_d_scatter_atomic_kernel<__nv_bfloat16><<<blocks, kThreads, 0, stream>>>(P, g, am, gD, err);
    }
    return cudaGetLastError();
}

}  // namespace lik
