// fwd_simt.cu -- FFMA MaxSim forward for every dtype, layout and size.
//
// This is the fp32 path (fp32 inputs are computed with fp32 FMA, never TF32,
// so fp32 scores keep fp32 accuracy; Late Interaction Kernels README,
// "Precision and compatibility") and the path for shapes the tensor-core
// kernels do not take.  It computes the same thing as those kernels
// (README, "What does it compute?" and "Scoring interface"):
//
//   for every pair p = (q, d):
//     empty document            -> score -1e9, argmax -1
//     for every valid i:  m_i = max over valid j of Q[q,i].D[d,j]
//                         (first j reaching it), score = sum of m_i
//
// One CTA owns one pair at a time (grid-stride over pairs).  Document tokens
// stream through shared memory in tiles of 32 (one per lane); each warp owns
// a subset of query tokens, computes the 32 similarities of its token with
// one lane per document token, and folds them into a running max/argmax kept
// in shared memory.  The similarity grid never leaves the SM.
#include <cfloat>
#include <climits>

#include "dtype_load.cuh"
#include "lik_internal.h"

namespace lik {
namespace {

constexpr int kThreads = 256;
constexpr int kTileJ = 32;

__device__ __forceinline__ int64_t smem_stride(int64_t dim) {
    // odd row stride: lane j reading row j, column k hits bank (j*stride+k)%32,
    // distinct across the 32 lanes
    return (dim & 1) ? dim : dim + 1;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(Problem P, float* __restrict__ scores, int32_t* __restrict__ argmax) {
    extern __shared__ float smem[];
    const int64_t stride = smem_stride(P.dim);
    float* Ds = smem;                                   // [kTileJ][stride]
    float* best = Ds + kTileJ * stride;                 // [Lq]
    int* best_j = reinterpret_cast<int*>(best + P.Lq);  // [Lq]

    const T* Q = static_cast<const T*>(P.Q);
    const T* D = static_cast<const T*>(P.D);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = kThreads / 32;

    for (int64_t p = blockIdx.x; p < P.n_pairs; p += gridDim.x) {
        const int64_t q = P.query_of(p), d = P.doc_of(p);
        const uint8_t* dm = P.dmask ? P.dmask + d * P.Ld : nullptr;
        const uint8_t* qm = P.qmask ? P.qmask + q * P.Lq : nullptr;

        int any = 0;
        for (int64_t j = tid; j < P.Ld; j += kThreads) any |= (!dm || dm[j]) ? 1 : 0;
        any = __syncthreads_or(any);

        if (!any) {
            if (tid == 0 && scores) scores[p] = kEmptyDocScore;
            if (argmax)
                for (int64_t i = tid; i < P.Lq; i += kThreads) argmax[p * P.Lq + i] = -1;
            __syncthreads();
            continue;
        }

        for (int64_t i = tid; i < P.Lq; i += kThreads) {
            best[i] = -INFINITY;
            best_j[i] = -1;
        }

        for (int64_t j0 = 0; j0 < P.Ld; j0 += kTileJ) {
            __syncthreads();  // previous tile fully consumed
            const int64_t tile_elems = kTileJ * P.dim;
            const T* src = D + (d * P.Ld + j0) * P.dim;
            const int64_t avail = (P.Ld - j0) * P.dim;  // elements left in this document
            for (int64_t e = tid; e < tile_elems; e += kThreads) {
                const int64_t jj = e / P.dim, k = e - jj * P.dim;
                Ds[jj * stride + k] = e < avail ? load_f32(src + e) : 0.0f;
            }
            __syncthreads();

            const int64_t j = j0 + lane;
            const bool valid = j < P.Ld && (!dm || dm[j]);
            const float* drow = Ds + lane * stride;
            for (int64_t i = warp; i < P.Lq; i += nwarps) {
                if (qm && !qm[i]) continue;  // warp-uniform
                const T* qrow = Q + (q * P.Lq + i) * P.dim;
                float s = 0.0f;
                for (int64_t k = 0; k < P.dim; ++k) s = fmaf(load_f32(qrow + k), drow[k], s);
                float v = valid ? s : -INFINITY;
                int vj = valid ? static_cast<int>(j) : INT_MAX;
                // warp max; equal values resolve to the lower token index
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
                    const int oj = __shfl_xor_sync(0xffffffffu, vj, off);
                    if (ov > v || (ov == v && oj < vj)) {
                        v = ov;
                        vj = oj;
                    }
                }
                // tiles arrive in ascending j: only a strictly larger value moves the argmax
                if (lane == 0 && vj != INT_MAX && v > best[i]) {
                    best[i] = v;
                    best_j[i] = vj;
                }
            }
        }
        __syncthreads();

        if (tid == 0) {
            float sum = 0.0f;
            for (int64_t i = 0; i < P.Lq; ++i)
                if (!qm || qm[i]) sum += best[i];
            if (scores) scores[p] = sum;
        }
        if (argmax)
            for (int64_t i = tid; i < P.Lq; i += kThreads)
                argmax[p * P.Lq + i] = (!qm || qm[i]) ? best_j[i] : -1;
        __syncthreads();
    }
}

template <typename T>
cudaError_t launch_typed(const Problem& P, float* scores, int32_t* argmax, cudaStream_t stream) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const DeviceInfo& info = device_info(dev);
    const int64_t stride = (P.dim & 1) ? P.dim : P.dim + 1;
    const size_t smem = sizeof(float) * (kTileJ * stride) + (sizeof(float) + sizeof(int)) * P.Lq;
    if (smem > 48 * 1024) {
        err = cudaFuncSetAttribute(fwd_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(smem));
        if (err != cudaSuccess) return err;
    }
    int64_t blocks = P.n_pairs;
    const int64_t cap = static_cast<int64_t>(info.sm_count) * 8;
    if (blocks > cap) blocks = cap;
    fwd_simt_kernel<T><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(P, scores, argmax);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const Problem& P, float* scores, int32_t* argmax, cudaStream_t stream) {
    switch (P.dtype) {
    case kF32: return launch_typed<float>(P, scores, argmax, stream);
    case kF16: return launch_typed<__half>(P, scores, argmax, stream);
    default: return launch_typed<__nv_bfloat16>(P, scores, argmax, stream);
    }
}

}  // namespace lik
