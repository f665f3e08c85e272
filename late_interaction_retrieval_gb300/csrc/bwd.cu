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
// backward allocates only the input gradients).  Every saved argmax is
// checked: an index >= Ld is skipped (never dereferenced) and flagged in the
// library's error word.
#include "dtype_load.cuh"
#include "lik_internal.h"

namespace lik {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// ------------------------------------------------------------- grad_Q --
//
// Vector path (dim % 8 == 0, dim <= 256): one CTA per (query, group of 16
// query tokens), 2 x 128 threads.  Eight threads own one token row, each a
// set of 8-element vectors (16 B of fp16/bf16); the two 128-thread halves
// take alternate pairs of the query.  The pairs are visited in chunks whose
// argmax slice and upstream gradients (both contiguous in memory) are staged
// in shared memory; every thread then gathers its document rows with
// independent 16-byte loads, eight pairs at a time.  The halves' partial sums
// are added in a fixed order at the end, so the result is deterministic.

constexpr int kRowsPerCta = 16;
constexpr int kThreadsPerRow = 8;
constexpr int kPairGroups = 2;
constexpr int kVecThreads = kRowsPerCta * kThreadsPerRow * kPairGroups;  // 256
constexpr int kVec = 8;                                                  // elements per vector
constexpr int kPairChunk = 64;

// Eight consecutive elements kept in their storage type until the FMA, so
// that many rows can be in flight per thread: 16 bytes for fp16/bf16.
template <typename T>
struct Raw8 {
    uint4 v;
    __device__ __forceinline__ void load(const T* p) { v = *reinterpret_cast<const uint4*>(p); }
    __device__ __forceinline__ float get(int e) const {
        const T* h = reinterpret_cast<const T*>(&v);
        return to_f32(h[e]);
    }
};
template <>
struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = *reinterpret_cast<const float4*>(p);
        b = *reinterpret_cast<const float4*>(p + 4);
    }
    __device__ __forceinline__ float get(int e) const {
        const float* f = e < 4 ? reinterpret_cast<const float*>(&a) : reinterpret_cast<const float*>(&b);
        return f[e & 3];
    }
};

// VECS vectors of 8 elements per thread: dim <= VECS * 64.
template <typename T, int VECS, int kUnroll>
__global__ void __launch_bounds__(kVecThreads)
grad_q_vec_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                  float* __restrict__ gQ, unsigned int* err) {
    __shared__ int s_am[kPairChunk][kRowsPerCta];
    __shared__ float s_g[kPairChunk];
    __shared__ float s_part[kRowsPerCta][VECS * kThreadsPerRow * kVec];
    const T* D = static_cast<const T*>(P.D);
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t q = blockIdx.x / groups;
    const int64_t i0 = (blockIdx.x - q * groups) * kRowsPerCta;
    const int pg = threadIdx.x / (kRowsPerCta * kThreadsPerRow);  // pair group
    const int tl = threadIdx.x % (kRowsPerCta * kThreadsPerRow);
    const int r = tl / kThreadsPerRow, sub = tl % kThreadsPerRow;
    const int rows_here = static_cast<int>(P.Lq - i0 < kRowsPerCta ? P.Lq - i0 : kRowsPerCta);

    float acc[VECS][kVec];
#pragma unroll
    for (int m = 0; m < VECS; ++m)
#pragma unroll
        for (int t = 0; t < kVec; ++t) acc[m][t] = 0.f;

    const int64_t p0 = q * P.pairs_per_query;
    bool bad = false;
    for (int64_t c0 = 0; c0 < P.pairs_per_query; c0 += kPairChunk) {
        const int nc = static_cast<int>(P.pairs_per_query - c0 < kPairChunk ? P.pairs_per_query - c0 : kPairChunk);
        __syncthreads();
        for (int e = threadIdx.x; e < nc * kRowsPerCta; e += kVecThreads) {
            const int t = e / kRowsPerCta, rr = e % kRowsPerCta;
            s_am[t][rr] = rr < rows_here ? am[(p0 + c0 + t) * P.Lq + i0 + rr] : -1;
        }
        for (int t = threadIdx.x; t < nc; t += kVecThreads) s_g[t] = g[p0 + c0 + t];
        __syncthreads();
        if (r >= rows_here) continue;
        // this half takes pairs t = pg, pg + 2, pg + 4, ... of the chunk
        for (int t = pg; t < nc; t += kUnroll * kPairGroups) {
            const T* rows[kUnroll];
            float gv[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int tt = t + u * kPairGroups;
                int a = tt < nc ? s_am[tt][r] : -1;
                if (a >= P.Ld) {
                    bad = true;
                    a = -1;
                }
                gv[u] = a >= 0 ? s_g[tt] : 0.f;
                rows[u] = a >= 0 ? D + (P.doc_of_query_pair(q, c0 + tt) * P.Ld + a) * P.dim : nullptr;
            }
#pragma unroll
            for (int m = 0; m < VECS; ++m) {
                const int64_t k = static_cast<int64_t>(m * kThreadsPerRow + sub) * kVec;
                if (k >= P.dim) break;
                Raw8<T> x[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    if (rows[u]) x[u].load(rows[u] + k);
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    if (rows[u])
#pragma unroll
                        for (int e = 0; e < kVec; ++e) acc[m][e] = fmaf(gv[u], x[u].get(e), acc[m][e]);
            }
        }
    }
    if (bad) atomicOr(err, kErrBadIndex);
    __syncthreads();
    if (pg == 1 && r < rows_here) {
#pragma unroll
        for (int m = 0; m < VECS; ++m)
#pragma unroll
            for (int e = 0; e < kVec; ++e) s_part[r][(m * kThreadsPerRow + sub) * kVec + e] = acc[m][e];
    }
    __syncthreads();
    if (pg == 1 || r >= rows_here) return;
    float* out = gQ + (q * P.Lq + i0 + r) * P.dim;
#pragma unroll
    for (int m = 0; m < VECS; ++m) {
        const int64_t k = static_cast<int64_t>(m * kThreadsPerRow + sub) * kVec;
        if (k >= P.dim) break;
        float o[kVec];
#pragma unroll
        for (int e = 0; e < kVec; ++e) o[e] = acc[m][e] + s_part[r][k + e];
        *reinterpret_cast<float4*>(out + k) = make_float4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<float4*>(out + k + 4) = make_float4(o[4], o[5], o[6], o[7]);
    }
}

// Any-dim path: one warp per (query, token) row; lanes stride over dim.
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

// ------------------------------------------------------------- grad_D --
//
// grad_D is zero-filled on the stream, then every (pair, token) hit adds
// g * Q[q,i,:] into grad_D[d, a, :].  Vector path (dim % 4 == 0): one warp
// per pair loads 32 of the pair's saved argmax at once; each lane adds 4
// consecutive fp32 with one 16-byte reduction (red.global.add.v4.f32), a
// warp covers 128 dims of one hit, and two hits are in flight per step.

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

__device__ __forceinline__ void load4(const float* p, float (&o)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x;
    o[1] = v.y;
    o[2] = v.z;
    o[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&o)[4]) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
    const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
    o[0] = a.x;
    o[1] = a.y;
    o[2] = b.x;
    o[3] = b.y;
}
__device__ __forceinline__ void load4(const __half* p, float (&o)[4]) {
    const uint2 r = *reinterpret_cast<const uint2*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&r);
    const float2 a = __half22float2(h[0]), b = __half22float2(h[1]);
    o[0] = a.x;
    o[1] = a.y;
    o[2] = b.x;
    o[3] = b.y;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
grad_d_scatter_vec_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                          float* __restrict__ gD, unsigned int* err) {
    const T* Q = static_cast<const T*>(P.Q);
    const int lane = threadIdx.x & 31;
    // one warp per pair; its query tokens' argmax are loaded 32 at a time
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); p < P.n_pairs;
         p += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int64_t q = P.query_of(p), d = P.doc_of(p);
        const float gv = g[p];
        const T* qbase = Q + q * P.Lq * P.dim;
        float* dbase = gD + d * P.Ld * P.dim;
        for (int64_t i0 = 0; i0 < P.Lq; i0 += 32) {
            const int64_t i = i0 + lane;
            int32_t a = i < P.Lq ? am[p * P.Lq + i] : -1;
            if (a >= P.Ld) {
                atomicOr(err, kErrBadIndex);
                a = -1;
            }
            uint32_t live = __ballot_sync(0xffffffffu, a >= 0);
            // two hits in flight per step
            while (live) {
                const int s0 = __ffs(live) - 1;
                live &= live - 1;
                const int s1 = live ? __ffs(live) - 1 : -1;
                if (s1 >= 0) live &= live - 1;
                const int a0 = __shfl_sync(0xffffffffu, a, s0);
                const int a1 = __shfl_sync(0xffffffffu, a, s1 >= 0 ? s1 : s0);
                const T* q0 = qbase + (i0 + s0) * P.dim;
                const T* q1 = qbase + (i0 + (s1 >= 0 ? s1 : s0)) * P.dim;
                for (int64_t k = lane * 4; k < P.dim; k += 128) {
                    float x0[4], x1[4];
                    load4(q0 + k, x0);
                    if (s1 >= 0) load4(q1 + k, x1);
                    red_add_v4(dbase + a0 * P.dim + k, gv * x0[0], gv * x0[1], gv * x0[2], gv * x0[3]);
                    if (s1 >= 0)
                        red_add_v4(dbase + a1 * P.dim + k, gv * x1[0], gv * x1[1], gv * x1[2], gv * x1[3]);
                }
            }
        }
    }
}

// Any-dim path: one warp per hit, scalar fp32 atomics.
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

unsigned grid_for(int64_t warps_of_work, int per_sm) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t cap = static_cast<int64_t>(device_info(dev).sm_count) * per_sm;
    int64_t blocks = (warps_of_work + kWarps - 1) / kWarps;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return static_cast<unsigned>(blocks);
}

template <typename T>
cudaError_t grad_q_typed(const Problem& P, const float* g, const int32_t* am, float* gQ,
                         cudaStream_t stream, unsigned int* err) {
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t blocks = P.n_query * groups;
    if (P.dim % kVec == 0 && P.dim <= 256 && blocks < (int64_t(1) << 31)) {
        // 8 (dim <= 128) or 4 (dim <= 256) independent row loads in flight per thread
        if (P.dim <= 128)
            grad_q_vec_kernel<T, 2, 8><<<static_cast<unsigned>(blocks), kVecThreads, 0, stream>>>(P, g, am, gQ, err);
        else
            grad_q_vec_kernel<T, 4, 4><<<static_cast<unsigned>(blocks), kVecThreads, 0, stream>>>(P, g, am, gQ, err);
        return cudaGetLastError();
    }
    grad_q_gather_kernel<T><<<grid_for(P.n_query * P.Lq, 16), kThreads, 0, stream>>>(P, g, am, gQ, err);
    return cudaGetLastError();
}

template <typename T>
cudaError_t grad_d_typed(const Problem& P, const float* g, const int32_t* am, float* gD,
                         cudaStream_t stream, unsigned int* err) {
    const int64_t hits = P.n_pairs * P.Lq;
    if (P.dim % 4 == 0)
        grad_d_scatter_vec_kernel<T><<<grid_for(P.n_pairs, 16), kThreads, 0, stream>>>(P, g, am, gD, err);
    else
        grad_d_scatter_atomic_kernel<T><<<grid_for(hits, 16), kThreads, 0, stream>>>(P, g, am, gD, err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_grad_q(const Problem& P, const float* g, const int32_t* am, float* gQ,
                              cudaStream_t stream) {
    if (P.n_query * P.Lq == 0) return cudaSuccess;
    unsigned int* err = device_error_word();
    switch (P.dtype) {
    case kF32: return grad_q_typed<float>(P, g, am, gQ, stream, err);
    case kF16: return grad_q_typed<__half>(P, g, am, gQ, stream, err);
    default: return grad_q_typed<__nv_bfloat16>(P, g, am, gQ, stream, err);
    }
}

cudaError_t launch_bwd_grad_d(const Problem& P, const float* g, const int32_t* am, float* gD,
                              cudaStream_t stream) {
    const int64_t elems = P.n_doc * P.Ld * P.dim;
    if (elems == 0) return cudaSuccess;
    const cudaError_t e = cudaMemsetAsync(gD, 0, sizeof(float) * elems, stream);
    if (e != cudaSuccess) return e;
    if (P.n_pairs * P.Lq == 0) return cudaSuccess;
    unsigned int* err = device_error_word();
    switch (P.dtype) {
    case kF32: return grad_d_typed<float>(P, g, am, gD, stream, err);
    case kF16: return grad_d_typed<__half>(P, g, am, gD, stream, err);
    default: return grad_d_typed<__nv_bfloat16>(P, g, am, gD, stream, err);
    }
}

}  // namespace lik
