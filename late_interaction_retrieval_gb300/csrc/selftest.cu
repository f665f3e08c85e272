// selftest.cu -- a self-test of the failure path of the bounded pipeline waits.
//
// Every mbarrier wait of the tensor-core kernels is bounded: when a wait
// runs out, the kernel sets the library's device error word, stops, and
// lik_check_device_error() reports LIK_ERR_TIMEOUT, so a broken pipeline
// surfaces as a status instead of a hung GPU (the colpali PR "Add support
// for late-interaction-kernels (LIK)", Design section: a real kernel failure
// is reported to the caller, never hidden).  In a healthy run no wait ever
// runs out, so this entry point makes one run out on purpose, safely: one
// thread waits, with the same bounded wait the pipelines use and a short
// limit, on an mbarrier that nothing ever arrives at.  No TMA copy, MMA or
// tensor memory is involved; the thread returns when the limit passes.
#include "lik.h"
#include "lik_internal.h"
#include "sm100_ptx.cuh"

namespace lik {

lik_status report_status(lik_status s, const char* message);

namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint64_t timeout_ns, unsigned int* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
    // nothing arrives on `bar`: its phase 0 never completes and the wait runs out
    ptx::mbar_wait_for(b, 0, err, timeout_ns);
}

}  // namespace
}  // namespace lik

extern "C" lik_status lik_selftest_bounded_wait(int64_t timeout_us, cudaStream_t stream) {
    using namespace lik;
    if (timeout_us < 1 || timeout_us > 1000000)
        return report_status(LIK_ERR_INVALID_ARG, "lik_selftest_bounded_wait: timeout_us must be in [1, 1000000]");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return report_status(LIK_ERR_CUDA, "lik_selftest_bounded_wait: no current CUDA device");
    const DeviceInfo& info = device_info(dev);
    if (info.major != 10 || info.minor != 3)
        return report_status(LIK_ERR_UNSUPPORTED, "lik_selftest_bounded_wait: the current device is not sm_103");
    unsigned int* err = device_error_word();
    if (!err) return report_status(LIK_ERR_CUDA, "lik_selftest_bounded_wait: cannot resolve the device error word");
    bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<uint64_t>(timeout_us) * 1000u, err);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return report_status(LIK_ERR_CUDA, "lik_selftest_bounded_wait: launch failed");
    return report_status(LIK_OK, "");
}
