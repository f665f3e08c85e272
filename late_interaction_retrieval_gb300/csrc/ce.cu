// ce.cu -- softmax cross-entropy head over MaxSim score rows.
//
// The in-batch ColBERT losses score every query against the batch's
// documents with the query's own document as the target, and the
// negative-document losses score each query against its own candidates with
// the positive first (colpali PR "Add support for late-interaction-kernels
// (LIK)", "What this PR adds"); the PR's "Results" time exactly that head,
// forward and backward.  For a row r of scores[rows, cols], logits
// z = scale * scores[r, :] and target t:
//     row_loss[r] = log(sum_c exp(z_c)) - z_t
//     grad[r, c]  = scale * (softmax(z)_c - [c == t]) / rows
//     loss        = mean over rows of row_loss
// A target outside [0, cols) leaves its row out (row_loss 0, zero gradient)
// but the mean still divides by rows.  Empty documents score -1e9, so their
// logits contribute exp(...) = 0.
#include "lik_internal.h"

namespace lik {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One warp per row: the row max, the sum of exponentials after subtracting
// it, the log-sum-exp, then the row's loss and gradient.
__global__ void __launch_bounds__(kThreads)
ce_rows_kernel(const float* __restrict__ scores, int64_t rows, int64_t cols, const int32_t* __restrict__ target,
               float scale, float* __restrict__ row_loss, float* __restrict__ grad) {
    const int lane = threadIdx.x & 31;
    const float inv_rows = 1.0f / static_cast<float>(rows);
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); r < rows;
         r += static_cast<int64_t>(gridDim.x) * kWarps) {
        const float* s = scores + r * cols;
        float* gr = grad ? grad + r * cols : nullptr;
        const int32_t t = target[r];
        if (t < 0 || t >= cols) {
            if (lane == 0) row_loss[r] = 0.0f;
            if (gr)
                for (int64_t c = lane; c < cols; c += 32) gr[c] = 0.0f;
            continue;
        }
        float m = -INFINITY;
        for (int64_t c = lane; c < cols; c += 32) m = fmaxf(m, scale * s[c]);
        m = warp_max(m);
        float sum = 0.0f;
        for (int64_t c = lane; c < cols; c += 32) sum += expf(scale * s[c] - m);
        sum = warp_sum(sum);
        const float lse = m + logf(sum);
        if (lane == 0) row_loss[r] = lse - scale * s[t];
        if (gr)
            for (int64_t c = lane; c < cols; c += 32)
                gr[c] = scale * (expf(scale * s[c] - lse) - (c == t ? 1.0f : 0.0f)) * inv_rows;
    }
}

// One block: loss = (sum of row_loss) / rows, summed in a fixed order (each
// thread a strided run of rows, then a fixed tree), so it is reproducible.
__global__ void __launch_bounds__(kThreads)
ce_mean_kernel(const float* __restrict__ row_loss, int64_t rows, float* __restrict__ loss) {
    __shared__ float part[kThreads];
    float acc = 0.0f;
    for (int64_t r = threadIdx.x; r < rows; r += kThreads) acc += row_loss[r];
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int w = kThreads / 2; w > 0; w >>= 1) {
        if (static_cast<int>(threadIdx.x) < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) *loss = rows > 0 ? part[0] / static_cast<float>(rows) : 0.0f;
}

}  // namespace

cudaError_t launch_ce_rows(const float* scores, int64_t rows, int64_t cols, const int32_t* target, float scale,
                           float* loss, float* row_loss, float* grad, cudaStream_t stream) {
    if (rows > 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        const int64_t cap = static_cast<int64_t>(device_info(dev).sm_count) * 8;
        int64_t blocks = (rows + kWarps - 1) / kWarps;
        if (blocks > cap) blocks = cap;
        ce_rows_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(scores, rows, cols, target, scale,
                                                                              row_loss, grad);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    ce_mean_kernel<<<1, kThreads, 0, stream>>>(row_loss, rows, loss);
    return cudaGetLastError();
}

}  // namespace lik
