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
// backward's memory is the two input gradients and nothing else).  Every saved argmax is
// checked: an index >= Ld is skipped (never dereferenced) and flagged in the
// library's error word.
//
// Kernels: with both gradients in fp32 one launch writes the two
// (grad_qd_vec_kernel); a gradient requested alone, or gradients in the
// inputs' 16-bit dtype, take a launch each.  All of them are bound by L2:
// the gathers read document rows resident there, and the fp32 grad_D
// reductions are 16-byte read-modify-writes of L2 lines.
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

// Gradient outputs: fp32, or the inputs' 16-bit type (rounded to nearest
// even once, from the fp32 sum).
__device__ __forceinline__ void store8(float* out, const float (&o)[8]) {
    *reinterpret_cast<float4*>(out) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4*>(out + 4) = make_float4(o[4], o[5], o[6], o[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* out, const float (&o)[8]) {
    __nv_bfloat162 h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(o[2 * e], o[2 * e + 1]);
    *reinterpret_cast<uint4*>(out) = *reinterpret_cast<const uint4*>(h);
}
__device__ __forceinline__ void store8(__half* out, const float (&o)[8]) {
    __half2 h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(o[2 * e], o[2 * e + 1]);
    *reinterpret_cast<uint4*>(out) = *reinterpret_cast<const uint4*>(h);
}
__device__ __forceinline__ void store1(float* out, float v) { *out = v; }
__device__ __forceinline__ void store1(__nv_bfloat16* out, float v) { *out = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store1(__half* out, float v) { *out = __float2half_rn(v); }

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The loss mean of a one-call loss-head step (Problem::ce_loss), written by
// warp 0 of block 0 of the grad_D launch: lane l sums rows l, l + 32, ... in
// order, then a fixed butterfly.
__device__ __forceinline__ void ce_loss_mean(const Problem& P) {
    if (P.ce_loss == nullptr || blockIdx.x != 0 || threadIdx.x >= 32) return;
    float acc = 0.0f;
    for (int64_t r = threadIdx.x; r < P.n_query; r += 32) acc += P.ce_row_loss[r];
    acc = warp_sum_f(acc);
    if (threadIdx.x == 0) *P.ce_loss = acc / static_cast<float>(P.n_query);
}

// Log-sum-exp of the logits scale * s[row, 0:cols) for R rows at once (one
// warp; every lane gets them), each row reduced in the same fixed order: lane
// l takes columns l, l + 32, ..., then a butterfly.  The rows' loads are
// independent, so R rows cost about one row's latency.
template <int R>
__device__ __forceinline__ void ce_rows_lse(const float* s, const int64_t (&row)[R], int64_t cols, float scale,
                                            int lane, float (&lse)[R]) {
    float m[R], sum[R];
#pragma unroll
    for (int k = 0; k < R; ++k) m[k] = -INFINITY;
    for (int64_t c = lane; c < cols; c += 32)
#pragma unroll
        for (int k = 0; k < R; ++k) m[k] = fmaxf(m[k], scale * s[row[k] * cols + c]);
#pragma unroll
    for (int k = 0; k < R; ++k) {
        m[k] = warp_max_f(m[k]);
        sum[k] = 0.0f;
    }
    for (int64_t c = lane; c < cols; c += 32)
#pragma unroll
        for (int k = 0; k < R; ++k) sum[k] += expf(scale * s[row[k] * cols + c] - m[k]);
#pragma unroll
    for (int k = 0; k < R; ++k) lse[k] = m[k] + logf(warp_sum_f(sum[k]));
}

__device__ __forceinline__ float ce_row_lse(const float* s, int64_t cols, float scale, int lane) {
    const int64_t row[1] = {0};
    float lse[1];
    ce_rows_lse<1>(s, row, cols, scale, lane, lse);
    return lse[0];
}

// Softmax cross-entropy over the score rows, computed by the grad_Q gather
// (the loss head of lik_maxsim_*_ce_step): row r = query r, cols = its pairs.
struct CeHead {
    const float* scores;   // [rows, cols]
    const int32_t* target; // [rows]; outside [0, cols): the row is left out
    float scale;
    float* row_loss;       // [rows]
    float* grad;           // [rows, cols]: d loss / d scores, the backward's upstream gradient
};

// VECS vectors of 8 elements per thread: dim <= VECS * 64.  With kCE the
// upstream gradient is not read but computed from the scores (CeHead): the
// CTA's warp 0 takes its query row's log-sum-exp, the first CTA of each query
// writes the row's loss and gradient (which grad_D then reads; the grad_D
// launch also takes the mean of the row losses).
template <typename T, int VECS, int kUnroll, typename TO, bool kCE = false>
__global__ void __launch_bounds__(kVecThreads)
grad_q_vec_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                  TO* __restrict__ gQ, unsigned int* err, CeHead ce = CeHead()) {
    __shared__ int s_am[kPairChunk][kRowsPerCta];
    __shared__ float s_g[kPairChunk];
    __shared__ float s_part[kRowsPerCta][VECS * kThreadsPerRow * kVec];
    __shared__ float s_lse;
    __shared__ int s_t;
    const T* D = static_cast<const T*>(P.D);
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t q = blockIdx.x / groups;
    const int64_t i0 = (blockIdx.x - q * groups) * kRowsPerCta;
    const int64_t cols = P.pairs_per_query;
    const float inv_rows = 1.0f / static_cast<float>(P.n_query);
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
        // with the loss head, warp 0 first takes the row's log-sum-exp while the
        // other warps stage the first chunk's argmax
        const int stage_lo = (kCE && c0 == 0) ? 32 : 0;
        if (static_cast<int>(threadIdx.x) >= stage_lo) {
            for (int e = threadIdx.x - stage_lo; e < nc * kRowsPerCta; e += kVecThreads - stage_lo) {
                const int t = e / kRowsPerCta, rr = e % kRowsPerCta;
                s_am[t][rr] = rr < rows_here ? am[(p0 + c0 + t) * P.Lq + i0 + rr] : -1;
            }
        } else if constexpr (kCE) {
            const int lane = threadIdx.x & 31;
            const int32_t t = ce.target[q];
            const float* srow = ce.scores + q * cols;
            const float lse = ce_row_lse(srow, cols, ce.scale, lane);
            if (lane == 0) {
                s_lse = lse;
                s_t = t;
                if (i0 == 0) ce.row_loss[q] = (t >= 0 && t < cols) ? lse - ce.scale * srow[t] : 0.0f;
            }
        }
        if constexpr (kCE) {
            if (c0 == 0) __syncthreads();  // s_lse, s_t
            const float lse = s_lse;
            const int32_t tq = s_t;
            const bool row_in = tq >= 0 && tq < cols;
            for (int t = threadIdx.x; t < nc; t += kVecThreads) {
                const int64_t c = c0 + t;
                const float gv = row_in ? ce.scale * (expf(ce.scale * ce.scores[q * cols + c] - lse) -
                                                      (c == tq ? 1.0f : 0.0f)) * inv_rows
                                        : 0.0f;
                s_g[t] = gv;
                if (i0 == 0) ce.grad[q * cols + c] = gv;
            }
        } else {
            for (int t = threadIdx.x; t < nc; t += kVecThreads) s_g[t] = g[p0 + c0 + t];
        }
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
    TO* out = gQ + (q * P.Lq + i0 + r) * P.dim;
#pragma unroll
    for (int m = 0; m < VECS; ++m) {
        const int64_t k = static_cast<int64_t>(m * kThreadsPerRow + sub) * kVec;
        if (k >= P.dim) break;
        float o[kVec];
#pragma unroll
        for (int e = 0; e < kVec; ++e) o[e] = acc[m][e] + s_part[r][k + e];
        store8(out + k, o);
    }
}

// Any-dim path: one warp per (query, token) row; lanes stride over dim.
template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads)
grad_q_gather_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                     TO* __restrict__ gQ, unsigned int* err) {
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
                if (k < P.dim) store1(gQ + row * P.dim + k, acc[m]);
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
    ce_loss_mean(P);
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
    ce_loss_mean(P);
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

// ------------------------------------------- grad_Q and grad_D in one pass --
//
// Both gradients in fp32, dim % 8 == 0, dim <= 256: one launch does the two.
// Its CTAs are those of grad_q_vec_kernel (one per query and 16 of its
// tokens, the query's pairs visited in the same order), so grad_Q is the same
// fixed-order sum.  The thread that gathers its share of the row D[d, a] for
// a hit (pair, token i, a = argmax) also adds its share of g * Q[q, i, :]
// into grad_D[d, a, :] with 16-byte reductions.  That share of Q[q, i, :]
// (4 consecutive elements in every 32, so that the 8 threads of a row cover
// 128 contiguous bytes per reduction) is loaded once into registers: the
// scatter reads nothing per hit, and its reductions are issued while the
// gathers are in flight.  grad_D must be zero on entry.
//
// With the loss head (kCE) every work CTA takes its query row's log-sum-exp
// for the score gradient, as grad_q_vec_kernel does, and one more CTA, the
// last, writes every row's loss and their mean (summed as in ce_loss_mean).

constexpr int kLossRows = 4;       // score rows per warp and step in the loss CTA
constexpr int64_t kFusedLossMaxRows = 4096;

// The rows' losses and their mean (one CTA of kVecThreads threads).
__device__ __forceinline__ void ce_losses_and_mean(const Problem& P, const CeHead& ce) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t rows = P.n_query, cols = P.pairs_per_query;
    for (int64_t r0 = static_cast<int64_t>(warp) * kLossRows; r0 < rows; r0 += (kVecThreads / 32) * kLossRows) {
        int64_t row[kLossRows];
        float lse[kLossRows];
#pragma unroll
        for (int k = 0; k < kLossRows; ++k) row[k] = r0 + k < rows ? r0 + k : rows - 1;
        ce_rows_lse<kLossRows>(ce.scores, row, cols, ce.scale, lane, lse);
        if (lane < kLossRows && r0 + lane < rows) {
            float l = 0.0f;
#pragma unroll
            for (int k = 0; k < kLossRows; ++k) if (k == lane) l = lse[k];
            const int64_t r = r0 + lane;
            const int32_t t = ce.target[r];
            ce.row_loss[r] = (t >= 0 && t < cols) ? l - ce.scale * ce.scores[r * cols + t] : 0.0f;
        }
    }
    __syncthreads();  // the row losses written above are visible to the whole CTA
    if (warp != 0) return;
    float acc = 0.0f;
    for (int64_t r = lane; r < rows; r += 32) acc += ce.row_loss[r];
    acc = warp_sum_f(acc);
    if (lane == 0) *P.ce_loss = acc / static_cast<float>(rows);
}

// A 16-byte reduction with no compiler memory barrier: the kernel below never
// reads grad_D, so its loads need no ordering against these adds.
__device__ __forceinline__ void red_add_v4_unordered(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d));
}

template <typename T, int VECS, int kUnroll, bool kCE>
__global__ void __launch_bounds__(kVecThreads, 2)
grad_qd_vec_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                   float* __restrict__ gQ, float* __restrict__ gD, unsigned int* err, CeHead ce) {
    constexpr int kRedVecs = VECS * 2;  // 4-element pieces of Q per thread: dim <= kRedVecs * 32
    __shared__ int s_am[kPairChunk][kRowsPerCta];
    __shared__ float s_g[kPairChunk];
    __shared__ float s_part[kRowsPerCta][VECS * kThreadsPerRow * kVec];
    __shared__ float s_lse;
    __shared__ int s_t;
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    if constexpr (kCE) {
        if (blockIdx.x == P.n_query * groups) {
            ce_losses_and_mean(P, ce);
            return;
        }
    }
    const T* D = static_cast<const T*>(P.D);
    const T* Q = static_cast<const T*>(P.Q);
    const int64_t q = blockIdx.x / groups;
    const int64_t i0 = (blockIdx.x - q * groups) * kRowsPerCta;
    const int64_t cols = P.pairs_per_query;
    const float inv_rows = 1.0f / static_cast<float>(P.n_query);
    const int pg = threadIdx.x / (kRowsPerCta * kThreadsPerRow);  // pair group
    const int tl = threadIdx.x % (kRowsPerCta * kThreadsPerRow);
    const int r = tl / kThreadsPerRow, sub = tl % kThreadsPerRow;
    const int rows_here = static_cast<int>(P.Lq - i0 < kRowsPerCta ? P.Lq - i0 : kRowsPerCta);

    float acc[VECS][kVec];
#pragma unroll
    for (int m = 0; m < VECS; ++m)
#pragma unroll
        for (int t = 0; t < kVec; ++t) acc[m][t] = 0.f;
    // this thread's share of Q[q, i0 + r, :] for the scatter
    float qv[kRedVecs][4];
#pragma unroll
    for (int j = 0; j < kRedVecs; ++j) {
        const int64_t k = static_cast<int64_t>(j) * 32 + sub * 4;
        if (r < rows_here && k < P.dim)
            load4(Q + (q * P.Lq + i0 + r) * P.dim + k, qv[j]);
        else
            qv[j][0] = qv[j][1] = qv[j][2] = qv[j][3] = 0.f;
    }

    const int64_t p0 = q * P.pairs_per_query;
    bool bad = false;
    for (int64_t c0 = 0; c0 < P.pairs_per_query; c0 += kPairChunk) {
        const int nc = static_cast<int>(P.pairs_per_query - c0 < kPairChunk ? P.pairs_per_query - c0 : kPairChunk);
        __syncthreads();
        const int stage_lo = (kCE && c0 == 0) ? 32 : 0;
        if (static_cast<int>(threadIdx.x) >= stage_lo) {
            for (int e = threadIdx.x - stage_lo; e < nc * kRowsPerCta; e += kVecThreads - stage_lo) {
                const int t = e / kRowsPerCta, rr = e % kRowsPerCta;
                s_am[t][rr] = rr < rows_here ? am[(p0 + c0 + t) * P.Lq + i0 + rr] : -1;
            }
        } else if constexpr (kCE) {
            const int lane = threadIdx.x & 31;
            const float lse = ce_row_lse(ce.scores + q * cols, cols, ce.scale, lane);
            if (lane == 0) {
                s_lse = lse;
                s_t = ce.target[q];
            }
        }
        if constexpr (kCE) {
            if (c0 == 0) __syncthreads();  // s_lse, s_t
            const float lse = s_lse;
            const int32_t tq = s_t;
            const bool row_in = tq >= 0 && tq < cols;
            for (int t = threadIdx.x; t < nc; t += kVecThreads) {
                const int64_t c = c0 + t;
                const float gv = row_in ? ce.scale * (expf(ce.scale * ce.scores[q * cols + c] - lse) -
                                                      (c == tq ? 1.0f : 0.0f)) * inv_rows
                                        : 0.0f;
                s_g[t] = gv;
                if (i0 == 0) ce.grad[q * cols + c] = gv;
            }
        } else {
            for (int t = threadIdx.x; t < nc; t += kVecThreads) s_g[t] = g[p0 + c0 + t];
        }
        __syncthreads();
        if (r >= rows_here) continue;
        for (int t = pg; t < nc; t += kUnroll * kPairGroups) {
            int64_t off[kUnroll];  // element offset of row (d, a) in D and grad_D; -1: no hit
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
                off[u] = a >= 0 ? (P.doc_of_query_pair(q, c0 + tt) * P.Ld + a) * P.dim : -1;
            }
#pragma unroll
            for (int m = 0; m < VECS; ++m) {
                const int64_t k = static_cast<int64_t>(m * kThreadsPerRow + sub) * kVec;
                const bool k_in = k < P.dim;
                Raw8<T> x[kUnroll];
                if (k_in)
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u)
                        if (off[u] >= 0) x[u].load(D + off[u] + k);
                // a share of the scatter (its own range of elements), while the loads are in flight
#pragma unroll
                for (int jj = 0; jj < kRedVecs / VECS; ++jj) {
                    const int j = m * (kRedVecs / VECS) + jj;
                    const int64_t kr = static_cast<int64_t>(j) * 32 + sub * 4;
                    if (kr < P.dim) {
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u)
                            if (off[u] >= 0)
                                red_add_v4_unordered(gD + off[u] + kr, gv[u] * qv[j][0], gv[u] * qv[j][1],
                                                     gv[u] * qv[j][2], gv[u] * qv[j][3]);
                    }
                }
                if (k_in)
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u)
                        if (off[u] >= 0)
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
        store8(out + k, o);
    }
}

// ------------------------------------------- grad_D in the inputs' dtype --
//
// A 16-bit grad_D cannot be accumulated with global atomics without rounding
// at every addition, so these kernels sum each row's hits in fp32 (registers
// or shared memory) and write every row exactly once (zeros included: no
// zero-fill).  dim % 8 == 0, dim <= 256.

constexpr int kOwnRowThreads = 16;                        // threads sharing one grad_D row
constexpr int kOwnSlots = kThreads / kOwnRowThreads;      // rows handled at once by a CTA

// Pairwise and kd (one pair per document, Lq <= 32): one CTA per document.
// Warp 0 ranks the pair's hits by (row, token) into shared memory; the CTA
// then walks the document's rows in order, each row-slot keeping a cursor
// into the sorted hits, and writes every row.
template <typename T, int VECS, typename TO>
__global__ void __launch_bounds__(kThreads)
grad_d_doc_stream_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                         TO* __restrict__ gD, unsigned int* err) {
    ce_loss_mean(P);
    __shared__ int s_row[32], s_qrow[32], s_nh;
    __shared__ float s_g;
    const T* Q = static_cast<const T*>(P.Q);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = threadIdx.x / kOwnRowThreads, sub = threadIdx.x % kOwnRowThreads;
    const int Lq = static_cast<int>(P.Lq);
    for (int64_t dd = blockIdx.x; dd < P.n_doc; dd += gridDim.x) {
        if (warp == 0) {
            int32_t a = lane < Lq ? am[dd * Lq + lane] : -1;
            if (a >= P.Ld) {
                atomicOr(err, kErrBadIndex);
                a = -1;
            }
            const unsigned valid = __ballot_sync(0xffffffffu, a >= 0);
            int rank = 0;
            for (int o = 0; o < 32; ++o) {
                const int32_t ao = __shfl_sync(0xffffffffu, a, o);
                rank += ((valid >> o) & 1u) && (ao < a || (ao == a && o < lane)) ? 1 : 0;
            }
            if (a >= 0) {
                s_row[rank] = a;
                s_qrow[rank] = static_cast<int>(P.query_of(dd) * Lq + lane);
            }
            if (lane == 0) {
                s_nh = __popc(valid);
                s_g = valid ? g[dd] : 0.f;
            }
        }
        __syncthreads();
        const int nh = s_nh;
        const float gv = s_g;
        TO* base = gD + dd * P.Ld * P.dim;
        int ptr = 0;
        for (int64_t j = slot; j < P.Ld; j += kOwnSlots) {
            while (ptr < nh && s_row[ptr] < j) ++ptr;
            float acc[VECS][kVec];
#pragma unroll
            for (int m = 0; m < VECS; ++m)
#pragma unroll
                for (int e = 0; e < kVec; ++e) acc[m][e] = 0.f;
            for (int h = ptr; h < nh && s_row[h] == j; ++h) {
                const T* src = Q + static_cast<int64_t>(s_qrow[h]) * P.dim;
#pragma unroll
                for (int m = 0; m < VECS; ++m) {
                    const int64_t kk = static_cast<int64_t>(m * kOwnRowThreads + sub) * kVec;
                    if (kk >= P.dim) break;
                    Raw8<T> x;
                    x.load(src + kk);
#pragma unroll
                    for (int e = 0; e < kVec; ++e) acc[m][e] = fmaf(gv, x.get(e), acc[m][e]);
                }
            }
#pragma unroll
            for (int m = 0; m < VECS; ++m) {
                const int64_t kk = static_cast<int64_t>(m * kOwnRowThreads + sub) * kVec;
                if (kk >= P.dim) break;
                store8(base + j * P.dim + kk, acc[m]);
            }
        }
        __syncthreads();  // s_row, s_qrow, s_nh and s_g are rewritten for the next document
    }
}

// All-pairs (and pairwise/kd with Lq > 32): one CTA owns a block of rows of
// one document and keeps their fp32 sums in shared memory (64 KB: 16384 /
// dim rows).  Per round of kChunkRound hits (the (pair, token) entries that
// use the document), the CTA stages each hit's row within the block (or -1)
// in shared memory; warp w then adds the Q rows of the hits on the block's
// rows r with r % 8 == w, four hits' rows loaded at once, with plain float4
// read-modify-writes: no two warps touch one row, and one lane's updates of a
// row are in program order, so no atomics are needed.  Every row of the block
// is written once at the end.
constexpr int kChunkFloats = 16384;                        // 64 KB of fp32 sums per CTA
constexpr int kChunkRound = 4096;                          // hits staged per round

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads)
grad_d_chunk_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                    TO* __restrict__ gD, int64_t rows_per_cta, int64_t chunks, unsigned int* err) {
    ce_loss_mean(P);
    extern __shared__ float s_acc[];                              // rows x dim
    int* s_row = reinterpret_cast<int*>(s_acc + kChunkFloats);  // [kChunkRound]
    const T* Q = static_cast<const T*>(P.Q);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t dd = blockIdx.x / chunks;
    const int64_t j0 = (static_cast<int64_t>(blockIdx.x) - dd * chunks) * rows_per_cta;
    const int rows = static_cast<int>(P.Ld - j0 < rows_per_cta ? P.Ld - j0 : rows_per_cta);
    const int dim = static_cast<int>(P.dim);
    const bool all = P.layout == kAllPairs;
    const int64_t K = all ? P.n_query : 1;            // pairs that use document dd
    const int64_t q_one = all ? 0 : P.query_of(dd);  // their query when there is one pair
    const int Lq = static_cast<int>(P.Lq);
    const int total = static_cast<int>(K * Lq);       // hits e = k * Lq + i (host: K * Lq < 2^31)
    bool bad = false;

    for (int x = threadIdx.x * 4; x < rows * dim; x += kThreads * 4)
        *reinterpret_cast<float4*>(s_acc + x) = make_float4(0.f, 0.f, 0.f, 0.f);

    for (int e0 = 0; e0 < total; e0 += kChunkRound) {
        __syncthreads();  // the previous round's rows are consumed (and the zero-fill is done)
#pragma unroll 4
        for (int t = threadIdx.x; t < kChunkRound; t += kThreads) {
            const int e = e0 + t;
            int32_t a = -1;
            if (e < total) {
                const int k = e / Lq, i = e - k * Lq;
                a = am[((all ? k * P.pairs_per_query : 0) + dd) * Lq + i];
            }
            if (a >= P.Ld) bad = true;
            const int64_t r = static_cast<int64_t>(a) - j0;
            s_row[t] = (a >= 0 && a < P.Ld && r >= 0 && r < rows) ? static_cast<int>(r) : -1;
        }
        __syncthreads();
        for (int t0 = 0; t0 < kChunkRound; t0 += 32) {
            const int my_row = s_row[t0 + lane];
            unsigned live = __ballot_sync(0xffffffffu, my_row >= 0 && (my_row & (kWarps - 1)) == warp);
            while (live) {
                int src[4], rr[4];
                float gv[4];
                const T* qr[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    src[u] = live ? __ffs(live) - 1 : -1;
                    if (src[u] >= 0) live &= live - 1;
                    const int sl = src[u] >= 0 ? src[u] : 0;
                    rr[u] = __shfl_sync(0xffffffffu, my_row, sl);
                    const int e = e0 + t0 + sl;
                    const int k = e / Lq, i = e - k * Lq;
                    const int64_t pair = all ? k * P.pairs_per_query + dd : dd;
                    gv[u] = src[u] >= 0 ? g[pair] : 0.f;
                    qr[u] = Q + ((all ? k : q_one) * Lq + i) * static_cast<int64_t>(dim);
                }
                for (int k0 = lane * 4; k0 < dim; k0 += 128) {
                    float x[4][4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (src[u] >= 0) load4(qr[u] + k0, x[u]);
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (src[u] >= 0) {
                            float4* dst = reinterpret_cast<float4*>(s_acc + rr[u] * dim + k0);
                            float4 v = *dst;
                            v.x = fmaf(gv[u], x[u][0], v.x);
                            v.y = fmaf(gv[u], x[u][1], v.y);
                            v.z = fmaf(gv[u], x[u][2], v.z);
                            v.w = fmaf(gv[u], x[u][3], v.w);
                            *dst = v;
                        }
                }
            }
        }
    }
    __syncthreads();
    TO* out = gD + (dd * P.Ld + j0) * P.dim;
    for (int x = threadIdx.x * kVec; x < rows * dim; x += kThreads * kVec) {
        float o[kVec];
#pragma unroll
        for (int c = 0; c < kVec; ++c) o[c] = s_acc[x + c];
        store8(out + x, o);
    }
    if (bad) atomicOr(err, kErrBadIndex);
}

// All-pairs with at most kOwnWindow hits per document (Nq * Lq <= 4096):
// document-owner gather.  One CTA owns kOwnRows rows of one document.  Each
// thread reads 16 of the document's argmax entries into registers (all loads
// in flight together); the hits that land in the CTA's rows are bucketed by a
// stable counting sort in shared memory (per-warp counts, a block-wide scan,
// ranks among equal rows from __match_any_sync); then 16 threads per row sum
// the row's hits in fp32 registers, four row loads in flight, and write the
// row once.  The bucket order depends only on the data: bit-reproducible.
constexpr int kOwnRows = 128;                              // rows of grad_D per CTA
constexpr int kOwnHitsPerThread = 16;
constexpr int kOwnWindow = kOwnHitsPerThread * kThreads;   // 4096 hits

template <typename T, int VECS, typename TO>
__global__ void __launch_bounds__(kThreads, 3)
grad_d_owner_kernel(Problem P, const float* __restrict__ g, const int32_t* __restrict__ am,
                    TO* __restrict__ gD, int64_t chunks, unsigned int* err) {
    ce_loss_mean(P);
    __shared__ int2 s_hit[kOwnWindow];             // (Q row, pair) in bucket order
    __shared__ int s_cnt[kOwnRows * kWarps];       // per (row, warp), row-major; then offsets
    __shared__ int s_start[kOwnRows + 1];          // first hit of each row in s_hit
    __shared__ int s_wsum[kWarps];
    static_assert(kWarps == 8 && kOwnRows * kWarps == 4 * kThreads, "scan layout");
    const T* Q = static_cast<const T*>(P.Q);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t dd = blockIdx.x / chunks;
    const int64_t j0 = (static_cast<int64_t>(blockIdx.x) - dd * chunks) * kOwnRows;
    const int rows = static_cast<int>(P.Ld - j0 < kOwnRows ? P.Ld - j0 : kOwnRows);
    const int Lq = static_cast<int>(P.Lq);
    const int total = static_cast<int>(P.n_query * Lq);  // hits e = q * Lq + i (host: <= kOwnWindow)
    const int slot = threadIdx.x / kOwnRowThreads, sub = threadIdx.x % kOwnRowThreads;
    bool bad = false;

    // ---- this thread's hits, all loads in flight together
    int row[kOwnHitsPerThread];  // row within the block, or -1
#pragma unroll
    for (int m = 0; m < kOwnHitsPerThread; ++m) {
        const int e = m * kThreads + static_cast<int>(threadIdx.x);
        int32_t a = -1;
        if (e < total) {
            const int q = e / Lq, i = e - q * Lq;
            a = am[(q * P.pairs_per_query + dd) * Lq + i];
        }
        row[m] = a;
    }
    for (int e = threadIdx.x; e < kOwnRows * kWarps; e += kThreads) s_cnt[e] = 0;
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kOwnHitsPerThread; ++m) {
        const int32_t a = row[m];
        if (a >= P.Ld) bad = true;
        const int64_t r = static_cast<int64_t>(a) - j0;
        row[m] = (a >= 0 && a < P.Ld && r >= 0 && r < rows) ? static_cast<int>(r) : -1;
        if (row[m] >= 0) atomicAdd(&s_cnt[row[m] * kWarps + warp], 1);
    }
    __syncthreads();

    // ---- exclusive scan over (row, warp) in row-major order, 4 entries per thread
    {
        const int t = threadIdx.x;
        const int v0 = s_cnt[4 * t], v1 = s_cnt[4 * t + 1], v2 = s_cnt[4 * t + 2], v3 = s_cnt[4 * t + 3];
        const int tsum = v0 + v1 + v2 + v3;
        int x = tsum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        int base = 0;
        for (int w = 0; w < warp; ++w) base += s_wsum[w];
        const int excl = base + x - tsum;
        s_cnt[4 * t] = excl;
        s_cnt[4 * t + 1] = excl + v0;
        s_cnt[4 * t + 2] = excl + v0 + v1;
        s_cnt[4 * t + 3] = excl + v0 + v1 + v2;
        if ((t & 1) == 0) s_start[t >> 1] = excl;  // entry (row t/2, warp 0)
        if (t == kThreads - 1) s_start[kOwnRows] = excl + tsum;
    }
    __syncthreads();

    // ---- place, batch by batch in a fixed order; equal rows ranked by lane
#pragma unroll
    for (int m = 0; m < kOwnHitsPerThread; ++m) {
        const bool in = row[m] >= 0;
        const int key = in ? row[m] : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        if (in) {
            const int pos = s_cnt[key * kWarps + warp] + __popc(peers & ((1u << lane) - 1u));
            const int e = m * kThreads + static_cast<int>(threadIdx.x);
            const int q = e / Lq;
            s_hit[pos] = make_int2(e, static_cast<int>(q * P.pairs_per_query + dd));
        }
        __syncwarp();
        if (in && lane == __ffs(peers) - 1) s_cnt[key * kWarps + warp] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();

    // ---- sum each row's hits in bucket order and write the row (zeros included)
    for (int r = slot; r < rows; r += kOwnSlots) {
        const int hs = s_start[r], he = s_start[r + 1];
        float acc[VECS][kVec];
#pragma unroll
        for (int m = 0; m < VECS; ++m)
#pragma unroll
            for (int c = 0; c < kVec; ++c) acc[m][c] = 0.f;
        for (int h = hs; h < he; h += 4) {
            const T* src[4];
            float gu[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool live = h + u < he;
                const int2 hv = live ? s_hit[h + u] : make_int2(0, 0);
                src[u] = live ? Q + static_cast<int64_t>(hv.x) * P.dim : nullptr;  // Q row q*Lq+i = e
                gu[u] = live ? g[hv.y] : 0.f;
            }
#pragma unroll
            for (int m = 0; m < VECS; ++m) {
                const int64_t kk = static_cast<int64_t>(m * kOwnRowThreads + sub) * kVec;
                if (kk >= P.dim) break;
                Raw8<T> x[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (src[u]) x[u].load(src[u] + kk);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (src[u])
#pragma unroll
                        for (int c = 0; c < kVec; ++c) acc[m][c] = fmaf(gu[u], x[u].get(c), acc[m][c]);
            }
        }
        TO* out = gD + ((dd * P.Ld) + j0 + r) * P.dim;
#pragma unroll
        for (int m = 0; m < VECS; ++m) {
            const int64_t kk = static_cast<int64_t>(m * kOwnRowThreads + sub) * kVec;
            if (kk >= P.dim) break;
            store8(out + kk, acc[m]);
        }
    }
    if (bad) atomicOr(err, kErrBadIndex);
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

template <typename T, typename TO>
cudaError_t grad_q_typed(const Problem& P, const float* g, const int32_t* am, TO* gQ,
                         cudaStream_t stream, unsigned int* err) {
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t blocks = P.n_query * groups;
    if (P.dim % kVec == 0 && P.dim <= 256 && blocks < (int64_t(1) << 31)) {
        // 8 (dim <= 128) or 4 (dim <= 256) independent row loads in flight per thread
        if (P.dim <= 128)
            grad_q_vec_kernel<T, 2, 8, TO><<<static_cast<unsigned>(blocks), kVecThreads, 0, stream>>>(P, g, am, gQ, err);
        else
            grad_q_vec_kernel<T, 4, 4, TO><<<static_cast<unsigned>(blocks), kVecThreads, 0, stream>>>(P, g, am, gQ, err);
        return cudaGetLastError();
    }
    grad_q_gather_kernel<T, TO><<<grid_for(P.n_query * P.Lq, 16), kThreads, 0, stream>>>(P, g, am, gQ, err);
    return cudaGetLastError();
}

template <typename T, typename TO>
cudaError_t grad_q_ce_typed(const Problem& P, const CeHead& ce, const int32_t* am, TO* gQ, cudaStream_t stream,
                            unsigned int* err) {
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    const int64_t blocks = P.n_query * groups;
    if (P.dim <= 128)
        grad_q_vec_kernel<T, 2, 8, TO, true><<<static_cast<unsigned>(blocks), kVecThreads, 0, stream>>>(
            P, nullptr, am, gQ, err, ce);
    else
        grad_q_vec_kernel<T, 4, 4, TO, true><<<static_cast<unsigned>(blocks), kVecThreads, 0, stream>>>(
            P, nullptr, am, gQ, err, ce);
    return cudaGetLastError();
}

template <typename T>
cudaError_t grad_qd_typed(const Problem& P, const float* g, const int32_t* am, float* gQ, float* gD,
                          const CeHead* ce, cudaStream_t stream, unsigned int* err) {
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    const unsigned blocks = static_cast<unsigned>(P.n_query * groups + (ce ? 1 : 0));
    // rows in flight per thread: as many as 128 registers hold (fp32 rows take twice the registers)
    constexpr int kU = sizeof(T) == 4 ? 4 : 8;
    if (ce) {
        if (P.dim <= 128)
            grad_qd_vec_kernel<T, 2, kU, true><<<blocks, kVecThreads, 0, stream>>>(P, nullptr, am, gQ, gD, err, *ce);
        else
            grad_qd_vec_kernel<T, 4, kU / 2, true><<<blocks, kVecThreads, 0, stream>>>(P, nullptr, am, gQ, gD, err,
                                                                                    *ce);
    } else {
        if (P.dim <= 128)
            grad_qd_vec_kernel<T, 2, kU, false><<<blocks, kVecThreads, 0, stream>>>(P, g, am, gQ, gD, err, CeHead());
        else
            grad_qd_vec_kernel<T, 4, kU / 2, false><<<blocks, kVecThreads, 0, stream>>>(P, g, am, gQ, gD, err,
                                                                                     CeHead());
    }
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
    case kF32: return grad_q_typed<float, float>(P, g, am, gQ, stream, err);
    case kF16: return grad_q_typed<__half, float>(P, g, am, gQ, stream, err);
    default: return grad_q_typed<__nv_bfloat16, float>(P, g, am, gQ, stream, err);
    }
}

bool bwd_qd_fusable(const Problem& P, bool ce) {
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    if (!(P.Lq >= 1 && P.n_query >= 1 && P.pairs_per_query >= 1 && P.n_doc * P.Ld * P.dim > 0 &&
          P.dim % kVec == 0 && P.dim <= 256 && P.n_query * groups < (int64_t(1) << 31) - 1))
        return false;
    return !ce || (grad_q_ce_fusable(P) && P.n_query <= kFusedLossMaxRows && P.ce_loss != nullptr);
}

cudaError_t launch_bwd_qd(const Problem& P, const float* g, const int32_t* am, float* gQ, float* gD,
                          const float* scores, const int32_t* target, float scale, float* row_loss,
                          float* grad_scores, cudaStream_t stream) {
    if (!P.grad_d_zeroed) {  // else the forward of the same step has zero-filled it
        const cudaError_t e = cudaMemsetAsync(gD, 0, sizeof(float) * P.n_doc * P.Ld * P.dim, stream);
        if (e != cudaSuccess) return e;
    }
    unsigned int* err = device_error_word();
    const CeHead head{scores, target, scale, row_loss, grad_scores};
    const CeHead* ce = scores ? &head : nullptr;
    switch (P.dtype) {
    case kF32: return grad_qd_typed<float>(P, g, am, gQ, gD, ce, stream, err);
    case kF16: return grad_qd_typed<__half>(P, g, am, gQ, gD, ce, stream, err);
    default: return grad_qd_typed<__nv_bfloat16>(P, g, am, gQ, gD, ce, stream, err);
    }
}

cudaError_t launch_bwd_grad_d(const Problem& P, const float* g, const int32_t* am, float* gD,
                              cudaStream_t stream) {
    const int64_t elems = P.n_doc * P.Ld * P.dim;
    if (elems == 0) return cudaSuccess;
    if (!P.grad_d_zeroed) {  // else the forward of the same step has zero-filled it
        const cudaError_t e = cudaMemsetAsync(gD, 0, sizeof(float) * elems, stream);
        if (e != cudaSuccess) return e;
    }
    if (P.n_pairs * P.Lq == 0) return cudaSuccess;
    unsigned int* err = device_error_word();
    switch (P.dtype) {
    case kF32: return grad_d_typed<float>(P, g, am, gD, stream, err);
    case kF16: return grad_d_typed<__half>(P, g, am, gD, stream, err);
    default: return grad_d_typed<__nv_bfloat16>(P, g, am, gD, stream, err);
    }
}


namespace {

template <typename T, typename TO>
cudaError_t grad_d_same_typed(const Problem& P, const float* g, const int32_t* am, TO* gD, cudaStream_t stream,
                              unsigned int* err) {
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t sms = device_info(dev).sm_count;
    if (P.layout != kAllPairs && P.Lq <= 32) {
        const int64_t grid = P.n_doc < sms * 8 ? P.n_doc : sms * 8;
        if (P.dim <= kOwnRowThreads * kVec)
            grad_d_doc_stream_kernel<T, 1, TO><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(P, g, am, gD, err);
        else
            grad_d_doc_stream_kernel<T, 2, TO><<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(P, g, am, gD, err);
        return cudaGetLastError();
    }
    if (P.layout == kAllPairs && P.n_query * P.Lq <= kOwnWindow) {
        const int64_t chunks = (P.Ld + kOwnRows - 1) / kOwnRows;
        const int64_t blocks = P.n_doc * chunks;
        if (P.dim <= kOwnRowThreads * kVec)
            grad_d_owner_kernel<T, 1, TO><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(P, g, am, gD, chunks, err);
        else
            grad_d_owner_kernel<T, 2, TO><<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(P, g, am, gD, chunks, err);
        return cudaGetLastError();
    }
    const int64_t rows_per_cta = kChunkFloats / P.dim;
    const int64_t chunks = (P.Ld + rows_per_cta - 1) / rows_per_cta;
    const int64_t blocks = P.n_doc * chunks;
    const int smem = (kChunkFloats + kChunkRound) * static_cast<int>(sizeof(float));
    cudaError_t e = cudaFuncSetAttribute(grad_d_chunk_kernel<T, TO>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    grad_d_chunk_kernel<T, TO><<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(P, g, am, gD, rows_per_cta,
                                                                                          chunks, err);
    return cudaGetLastError();
}

}  // namespace

bool bwd_same_dtype_supported(const Problem& P) {
    const int64_t chunks = P.dim > 0 ? (P.Ld + kChunkFloats / P.dim - 1) / (kChunkFloats / P.dim) : 0;
    return (P.dtype == kF16 || P.dtype == kBF16) && P.dim % kVec == 0 && P.dim <= 2 * kOwnRowThreads * kVec &&
           P.n_doc * chunks < (int64_t(1) << 31) && P.n_query * P.Lq < (int64_t(1) << 31) &&
           P.n_pairs < (int64_t(1) << 31);
}

cudaError_t launch_bwd_grad_q_same(const Problem& P, const float* g, const int32_t* am, void* gQ,
                                   cudaStream_t stream) {
    if (P.n_query * P.Lq == 0) return cudaSuccess;
    unsigned int* err = device_error_word();
    if (P.dtype == kF16) return grad_q_typed<__half, __half>(P, g, am, static_cast<__half*>(gQ), stream, err);
    return grad_q_typed<__nv_bfloat16, __nv_bfloat16>(P, g, am, static_cast<__nv_bfloat16*>(gQ), stream, err);
}

bool grad_q_ce_fusable(const Problem& P) {
    const int64_t groups = (P.Lq + kRowsPerCta - 1) / kRowsPerCta;
    return P.Lq >= 1 && P.n_query >= 1 && P.pairs_per_query >= 1 && P.dim % kVec == 0 && P.dim <= 256 &&
           P.n_query * groups < (int64_t(1) << 31) && P.n_query * P.pairs_per_query <= (int64_t(1) << 20);
}

cudaError_t launch_bwd_grad_q_ce(const Problem& P, const float* scores, const int32_t* target, float scale,
                                 float* row_loss, float* grad_scores, const int32_t* am, void* gQ, bool same_dtype,
                                 cudaStream_t stream) {
    unsigned int* err = device_error_word();
    CeHead ce{scores, target, scale, row_loss, grad_scores};
    if (!same_dtype || P.dtype == kF32) {
        float* o = static_cast<float*>(gQ);
        switch (P.dtype) {
        case kF32: return grad_q_ce_typed<float, float>(P, ce, am, o, stream, err);
        case kF16: return grad_q_ce_typed<__half, float>(P, ce, am, o, stream, err);
        default: return grad_q_ce_typed<__nv_bfloat16, float>(P, ce, am, o, stream, err);
        }
    }
    if (P.dtype == kF16) return grad_q_ce_typed<__half, __half>(P, ce, am, static_cast<__half*>(gQ), stream, err);
    return grad_q_ce_typed<__nv_bfloat16, __nv_bfloat16>(P, ce, am, static_cast<__nv_bfloat16*>(gQ), stream, err);
}

cudaError_t launch_bwd_grad_d_same(const Problem& P, const float* g, const int32_t* am, void* gD,
                                   cudaStream_t stream) {
    if (P.n_doc * P.Ld * P.dim == 0) return cudaSuccess;
    unsigned int* err = device_error_word();
    if (P.dtype == kF16) return grad_d_same_typed<__half, __half>(P, g, am, static_cast<__half*>(gD), stream, err);
    return grad_d_same_typed<__nv_bfloat16, __nv_bfloat16>(P, g, am, static_cast<__nv_bfloat16*>(gD), stream, err);
}

}  // namespace lik
