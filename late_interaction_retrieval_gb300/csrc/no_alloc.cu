// no_alloc.cu -- the all-pairs backward that recomputes the argmax, for
// callers that cannot allocate device memory.
//
// lik_maxsim_allpairs_bwd_recompute needs an int32 argmax workspace
// [Nq, Nd, Lq] from its caller.  Some callers cannot provide one: a memory
// manager that reserves the whole device up front and hands out no
// third-party buffers, or a latency-critical loop that cannot afford
// cudaMalloc (it may synchronise the device).  For them,
// lik_maxsim_allpairs_bwd_recompute_noalloc uses a workspace that is part of
// the library itself: the file-scope array below, kNoAllocArgmaxEntries
// int32 entries (8 MiB) on every GPU that loads the library, held until the
// process exits.  Nothing is allocated per call.
//
// The array's name in host code is only a host-side stand-in: the device
// address comes from cudaGetSymbolAddress, once per device, on the first
// call made with that device current (so that first call should come before
// any stream capture).  Every call shares the one array and leaves the last
// call's argmax in it; nothing in it has to start at zero, because the
// forward writes every entry the backward then reads.  Calls whose work
// overlaps on the GPU (different streams, or different host threads) race
// on the array: the caller must order them.
#include <mutex>

#include "lik.h"
#include "lik_internal.h"

namespace lik {

// Defined in api.cu: sets the calling thread's lik_last_error_message().
lik_status report_status(lik_status s, const char* message);

constexpr int64_t kNoAllocArgmaxEntries = int64_t(1) << 21;  // Nq * Nd * Lq at most (8 MiB)

static __device__ __align__(256) int32_t g_noalloc_argmax[kNoAllocArgmaxEntries];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
int32_t* g_noalloc_address[kNoAllocMaxDevices];  // per device, set on its first call

// Device address of the array on the current device (set-up on first use).
cudaError_t noalloc_argmax_address(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_address[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_argmax);
        if (e != cudaSuccess) return e;
        g_noalloc_address[dev] = static_cast<int32_t*>(p);
    }
    *out = g_noalloc_address[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace lik

extern "C" lik_status lik_maxsim_allpairs_bwd_recompute_noalloc(const void* Q, const void* D, lik_dtype dtype,
                                                                int64_t Nq, int64_t Nd, int64_t Lq, int64_t Ld,
                                                                int64_t dim, const bool* qmask, const bool* dmask,
                                                                const float* grad_out, float* grad_Q,
                                                                float* grad_D, cudaStream_t stream) {
    using namespace lik;
    if (Nq > 0 && Nd > 0 && Lq > 0 && (Nq > kNoAllocArgmaxEntries || Nd > kNoAllocArgmaxEntries ||
                                        Lq > kNoAllocArgmaxEntries || Nq * Nd > kNoAllocArgmaxEntries / Lq))
        return report_status(LIK_ERR_UNSUPPORTED,
                             "lik_maxsim_allpairs_bwd_recompute_noalloc: Nq * Nd * Lq exceeds the built-in "
                             "argmax workspace of 2097152 entries; use lik_maxsim_allpairs_bwd_recompute "
                             "with a caller-allocated workspace");
    int32_t* ws = nullptr;
    const cudaError_t e = noalloc_argmax_address(&ws);
    if (e != cudaSuccess)
        return report_status(LIK_ERR_CUDA,
                             "lik_maxsim_allpairs_bwd_recompute_noalloc: cannot resolve the built-in "
                             "argmax workspace on the current device");
    return lik_maxsim_allpairs_bwd_recompute(Q, D, dtype, Nq, Nd, Lq, Ld, dim, qmask, dmask, grad_out, ws,
                                             grad_Q, grad_D, stream);
}
