// api.cu -- the C ABI of liblik (declared in include/lik.h): argument
// validation, kernel selection and error propagation.
//
// Validation mirrors the eligibility checks the colpali PR "Add support for
// late-interaction-kernels (LIK)" describes for its backend (Design section:
// device capability, embedding size, matching devices), with one difference:
// an ineligible call returns a status code and never falls back to another
// backend.  CUDA errors are always propagated (same section: a genuine
// kernel failure is never hidden behind a fallback).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "lik.h"
#include "lik_internal.h"

namespace lik {

// ---------------------------------------------------------- device state --

namespace {

constexpr int kMaxDevices = 64;

struct DeviceSlot {
    std::once_flag once;
    DeviceInfo info;
    cudaError_t init_error = cudaSuccess;
};
DeviceSlot g_devices[kMaxDevices];

// Set by kernels whose bounded waits expire or that meet an invalid saved
// argmax; read and cleared by lik_check_device_error().
__device__ unsigned int g_error_word;

struct ErrorWordSlot {
    std::once_flag once;
    unsigned int* ptr = nullptr;
};
ErrorWordSlot g_error_words[kMaxDevices];

thread_local char t_message[512];

lik_status fail(lik_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_message, sizeof t_message, fmt, ap);
    va_end(ap);
    return s;
}

lik_status cuda_fail(cudaError_t e, const char* what) {
    return fail(LIK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

}  // namespace

// For entry points defined in other files: records `message` as the calling
// thread's lik_last_error_message() and returns `s`.
lik_status report_status(lik_status s, const char* message) { return fail(s, "%s", message); }

const DeviceInfo& device_info(int device) {
    DeviceSlot& slot = g_devices[device % kMaxDevices];
    std::call_once(slot.once, [&] {
        DeviceInfo& d = slot.info;
        d.device = device;
        cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, device);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, device);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
        slot.init_error = e;
    });
    return slot.info;
}

unsigned int* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    ErrorWordSlot& slot = g_error_words[dev % kMaxDevices];
    std::call_once(slot.once, [&] {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess)
            slot.ptr = static_cast<unsigned int*>(p);
    });
    return slot.ptr;
}

// ------------------------------------------------------------ validation --

namespace {

bool known_dtype(lik_dtype t) { return t == LIK_F32 || t == LIK_F16 || t == LIK_BF16; }

// The current device must be a GB300 (sm_103): the kernels are built for
// sm_103a only.
lik_status check_device(int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const DeviceInfo& info = device_info(dev);
    if (g_devices[dev % kMaxDevices].init_error != cudaSuccess)
        return cuda_fail(g_devices[dev % kMaxDevices].init_error, "cudaDeviceGetAttribute");
    if (info.major != 10 || info.minor != 3)
        return fail(LIK_ERR_UNSUPPORTED, "device %d is sm_%d%d; liblik is built for sm_103a (GB300)",
                    dev, info.major, info.minor);
    if (!device_error_word()) return fail(LIK_ERR_CUDA, "cannot resolve the device error word");
    *dev_out = dev;
    return LIK_OK;
}

// A non-NULL pointer must be device (or managed) memory of device `dev`.
lik_status check_pointer(const void* p, int dev, const char* name) {
    if (!p) return LIK_OK;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of an unknown pointer
        return fail(LIK_ERR_INVALID_ARG, "%s is not a CUDA pointer", name);
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(LIK_ERR_INVALID_ARG, "%s is not device memory", name);
    if (attr.device != dev)
        return fail(LIK_ERR_INVALID_ARG, "%s lives on device %d, current device is %d", name,
                    attr.device, dev);
    return LIK_OK;
}

struct Spec {
    const char* name;
    const void* ptr;
    bool required;  // must be non-NULL when the buffer has elements
    int64_t elems;
};

lik_status check_common(lik_dtype dtype, int64_t n_query, int64_t n_doc, int64_t ppq,
                        int64_t Lq, int64_t Ld, int64_t dim, bool* nothing_to_do) {
    *nothing_to_do = false;
    if (!known_dtype(dtype)) return fail(LIK_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (n_query < 0 || n_doc < 0 || ppq < 0 || Lq < 0 || Ld < 0)
        return fail(LIK_ERR_INVALID_ARG, "negative size");
    if (dim < 1) return fail(LIK_ERR_INVALID_ARG, "dim must be >= 1 (got %lld)", (long long)dim);
    if (dim > 1024) return fail(LIK_ERR_UNSUPPORTED, "dim %lld > 1024", (long long)dim);
    if (Lq > 4096) return fail(LIK_ERR_UNSUPPORTED, "Lq %lld > 4096", (long long)Lq);
    if (Ld > (int64_t(1) << 30)) return fail(LIK_ERR_UNSUPPORTED, "Ld %lld > 2^30", (long long)Ld);
    *nothing_to_do = (n_query == 0 || ppq == 0);
    return LIK_OK;
}

lik_status check_buffers(int dev, const Spec* specs, int n) {
    for (int k = 0; k < n; ++k) {
        const Spec& s = specs[k];
        if (s.required && s.elems > 0 && !s.ptr) return fail(LIK_ERR_INVALID_ARG, "%s is NULL", s.name);
        if (s.elems > 0) {
            lik_status st = check_pointer(s.ptr, dev, s.name);
            if (st != LIK_OK) return st;
        }
    }
    return LIK_OK;
}

lik_status check_alignment(const void* Q, const void* D) {
    if ((reinterpret_cast<uintptr_t>(Q) & 15) || (reinterpret_cast<uintptr_t>(D) & 15))
        return fail(LIK_ERR_INVALID_ARG, "Q and D must be 16-byte aligned");
    return LIK_OK;
}

lik_status check_aligned(const void* p, uintptr_t bytes, const char* name) {
    if (reinterpret_cast<uintptr_t>(p) & (bytes - 1))
        return fail(LIK_ERR_INVALID_ARG, "%s must be %d-byte aligned", name, static_cast<int>(bytes));
    return LIK_OK;
}

Problem make_problem(int layout, lik_dtype dtype, const void* Q, const void* D,
                     const bool* qmask, const bool* dmask, int64_t n_query, int64_t n_doc,
                     int64_t ppq, int64_t n_pairs, int64_t Lq, int64_t Ld, int64_t dim) {
    Problem P;
    P.layout = layout;
    P.dtype = static_cast<int>(dtype);
    P.Q = Q;
    P.D = D;
    P.qmask = reinterpret_cast<const uint8_t*>(qmask);
    P.dmask = reinterpret_cast<const uint8_t*>(dmask);
    P.n_query = n_query;
    P.n_doc = n_doc;
    P.pairs_per_query = ppq;
    P.n_pairs = n_pairs;
    P.Lq = Lq;
    P.Ld = Ld;
    P.dim = dim;
    return P;
}

// A caller's workspace for the streaming forward (caller_ws): NULL is allowed
// only when the path needs none; otherwise it must be device memory of the
// current device, 16-byte aligned and at least the needed size.
struct CallerWorkspace {
    bool given = false;
    void* ptr = nullptr;
    size_t bytes = 0;
};

// scores may be NULL only for the backward's recompute (argmax_only): the
// kernels then write the argmax alone.
lik_status run_fwd(const Problem& P, const bool* qmask, const bool* dmask, float* scores,
                   int32_t* argmax, cudaStream_t stream, bool argmax_only = false,
                   CallerWorkspace ws = CallerWorkspace()) {
    int dev = 0;
    lik_status st = check_device(&dev);
    if (st != LIK_OK) return st;
    const int64_t q_elems = P.n_query * P.Lq * P.dim, d_elems = P.n_doc * P.Ld * P.dim;
    const Spec specs[] = {
        {"Q", P.Q, true, q_elems},
        {"D", P.D, true, d_elems},
        {"qmask", qmask, false, P.n_query * P.Lq},
        {"dmask", dmask, false, P.n_doc * P.Ld},
        {"scores", scores, !argmax_only, P.n_pairs},
        {"argmax", argmax, argmax_only, P.n_pairs * P.Lq},
    };
    if ((st = check_buffers(dev, specs, 6)) != LIK_OK) return st;
    if ((st = check_alignment(P.Q, P.D)) != LIK_OK) return st;
    if ((st = check_aligned(scores, 4, "scores")) != LIK_OK) return st;
    if ((st = check_aligned(argmax, 4, "argmax")) != LIK_OK) return st;
    // kernel choice by layout and shape (the FFMA kernel takes fp32 and shapes
    // outside the tensor-core kernels' limits)
    cudaError_t e;
    const char* what;
    if (tc_allpairs_eligible(P)) {
        e = launch_fwd_tc_allpairs(P, scores, argmax, stream);
        what = "tensor-core all-pairs forward launch";
    } else if (tc_stream_eligible(P)) {
        if (ws.given) {
            const size_t need = stream_workspace_bytes(P, dmask != nullptr);
            if (!ws.ptr || ws.bytes < need)
                return fail(LIK_ERR_INVALID_ARG, "workspace of %zu bytes given, this call needs %zu", ws.ptr ? ws.bytes : 0,
                            need);
            if ((st = check_pointer(ws.ptr, dev, "workspace")) != LIK_OK) return st;
            if ((st = check_aligned(ws.ptr, 16, "workspace")) != LIK_OK) return st;
        }
        e = launch_fwd_tc_stream(P, scores, argmax, ws.given ? ws.ptr : nullptr, ws.bytes, stream);
        what = "tensor-core streaming forward launch";
    } else if (tc_f32_eligible(P)) {
        e = launch_fwd_tc_f32(P, scores, argmax, stream);
        what = "tensor-core fp32 (split TF32) forward launch";
    } else {
        e = launch_fwd_simt(P, scores, argmax, stream);
        what = "forward launch";
    }
    if (e != cudaSuccess) return cuda_fail(e, what);
    return LIK_OK;
}

// The cross-entropy head of a one-call step, computed inside the grad_Q
// launch (grad_out is then its score gradient, written there).
struct FusedCe {
    const float* scores;
    const int32_t* target;
    float scale;
    float* row_loss;
};

lik_status run_bwd(const Problem& P, const float* grad_out, const int32_t* argmax, float* grad_Q,
                   float* grad_D, cudaStream_t stream, const FusedCe* ce = nullptr) {
    int dev = 0;
    lik_status st = check_device(&dev);
    if (st != LIK_OK) return st;
    const int64_t q_elems = P.n_query * P.Lq * P.dim, d_elems = P.n_doc * P.Ld * P.dim;
    const bool need_hits = P.n_pairs * P.Lq > 0 && (grad_Q || grad_D);
    if (need_hits && !argmax) return fail(LIK_ERR_INVALID_ARG, "argmax is NULL");
    if (need_hits && !grad_out) return fail(LIK_ERR_INVALID_ARG, "grad_out is NULL");
    const Spec specs[] = {
        {"Q", P.Q, grad_D != nullptr, q_elems},
        {"D", P.D, grad_Q != nullptr, d_elems},
        {"grad_out", grad_out, false, P.n_pairs},
        {"argmax", argmax, false, P.n_pairs * P.Lq},
        {"grad_Q", grad_Q, false, q_elems},
        {"grad_D", grad_D, false, d_elems},
    };
    if ((st = check_buffers(dev, specs, 6)) != LIK_OK) return st;
    if ((st = check_alignment(P.Q, P.D)) != LIK_OK) return st;
    if ((st = check_aligned(grad_out, 4, "grad_out")) != LIK_OK) return st;
    if ((st = check_aligned(argmax, 4, "argmax")) != LIK_OK) return st;
    if ((st = check_aligned(grad_Q, 16, "grad_Q")) != LIK_OK) return st;
    if ((st = check_aligned(grad_D, 16, "grad_D")) != LIK_OK) return st;
    cudaError_t e;
    if (grad_Q && grad_D && bwd_qd_fusable(P, ce != nullptr)) {  // one launch for both gradients
        e = ce ? launch_bwd_qd(P, nullptr, argmax, grad_Q, grad_D, ce->scores, ce->target, ce->scale,
                               ce->row_loss, const_cast<float*>(grad_out), stream)
               : launch_bwd_qd(P, grad_out, argmax, grad_Q, grad_D, nullptr, nullptr, 0.0f, nullptr, nullptr,
                               stream);
        if (e != cudaSuccess) return cuda_fail(e, "backward launch (grad_Q and grad_D)");
        return LIK_OK;
    }
    if (ce) {
        e = launch_bwd_grad_q_ce(P, ce->scores, ce->target, ce->scale, ce->row_loss,
                                 const_cast<float*>(grad_out), argmax, grad_Q, false, stream);
        if (e != cudaSuccess) return cuda_fail(e, "grad_Q launch (with the loss head)");
    } else if (grad_Q && (e = launch_bwd_grad_q(P, grad_out, argmax, grad_Q, stream)) != cudaSuccess) {
        return cuda_fail(e, "grad_Q launch");
    }
    if (grad_D && (e = launch_bwd_grad_d(P, grad_out, argmax, grad_D, stream)) != cudaSuccess)
        return cuda_fail(e, "grad_D launch");
    return LIK_OK;
}

// Backward with grad_Q / grad_D in the inputs' dtype.  fp32 inputs take the
// fp32 path unchanged.
lik_status run_bwd_same(const Problem& P, const float* grad_out, const int32_t* argmax, void* grad_Q,
                        void* grad_D, cudaStream_t stream, const FusedCe* ce = nullptr) {
    if (P.dtype == kF32)
        return run_bwd(P, grad_out, argmax, static_cast<float*>(grad_Q), static_cast<float*>(grad_D), stream, ce);
    int dev = 0;
    lik_status st = check_device(&dev);
    if (st != LIK_OK) return st;
    if (!bwd_same_dtype_supported(P))
        return fail(LIK_ERR_UNSUPPORTED,
                    "the backward with fp16/bf16 gradients needs dim %% 8 == 0 and dim <= 256 "
                    "(the fp32-gradient entry point takes any dim)");
    const int64_t q_elems = P.n_query * P.Lq * P.dim, d_elems = P.n_doc * P.Ld * P.dim;
    const bool need_hits = P.n_pairs * P.Lq > 0 && (grad_Q || grad_D);
    if (need_hits && !argmax) return fail(LIK_ERR_INVALID_ARG, "argmax is NULL");
    if (need_hits && !grad_out) return fail(LIK_ERR_INVALID_ARG, "grad_out is NULL");
    const Spec specs[] = {
        {"Q", P.Q, grad_D != nullptr, q_elems},
        {"D", P.D, grad_Q != nullptr, d_elems},
        {"grad_out", grad_out, false, P.n_pairs},
        {"argmax", argmax, false, P.n_pairs * P.Lq},
        {"grad_Q", grad_Q, false, q_elems},
        {"grad_D", grad_D, false, d_elems},
    };
    if ((st = check_buffers(dev, specs, 6)) != LIK_OK) return st;
    if ((st = check_alignment(P.Q, P.D)) != LIK_OK) return st;
    if ((st = check_aligned(grad_out, 4, "grad_out")) != LIK_OK) return st;
    if ((st = check_aligned(argmax, 4, "argmax")) != LIK_OK) return st;
    if ((st = check_aligned(grad_Q, 16, "grad_Q")) != LIK_OK) return st;
    if ((st = check_aligned(grad_D, 16, "grad_D")) != LIK_OK) return st;
    cudaError_t e;
    if (ce) {
        e = launch_bwd_grad_q_ce(P, ce->scores, ce->target, ce->scale, ce->row_loss,
                                 const_cast<float*>(grad_out), argmax, grad_Q, true, stream);
        if (e != cudaSuccess) return cuda_fail(e, "grad_Q launch (with the loss head)");
    } else if (grad_Q && (e = launch_bwd_grad_q_same(P, grad_out, argmax, grad_Q, stream)) != cudaSuccess) {
        return cuda_fail(e, "grad_Q launch");
    }
    if (grad_D && (e = launch_bwd_grad_d_same(P, grad_out, argmax, grad_D, stream)) != cudaSuccess)
        return cuda_fail(e, "grad_D launch");
    return LIK_OK;
}

// In a one-call step whose backward writes an fp32 grad_D on the same stream
// right after the forward, the tensor-core all-pairs forward zero-fills that
// grad_D on the side (HBM is mostly idle while it runs), and the backward
// skips its own zero-fill.  Only for a grad_D that the backward will accept
// (device memory of the current device, 16-byte aligned); otherwise nothing
// changes and the backward reports what is wrong.
void plan_fwd_zero(Problem& P, float* grad_D) {
    if (!grad_D || P.layout != kAllPairs || P.n_pairs * P.Lq == 0 || !tc_allpairs_eligible(P)) return;
    const int64_t elems = P.n_doc * P.Ld * P.dim;
    if (elems % 4 != 0 || (reinterpret_cast<uintptr_t>(grad_D) & 15) != 0) return;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    if (check_pointer(grad_D, dev, "grad_D") != LIK_OK) {
        t_message[0] = 0;
        return;
    }
    P.fwd_zero = grad_D;
    P.fwd_zero_bytes = elems * static_cast<int64_t>(sizeof(float));
    P.grad_d_zeroed = true;
}

// One loss-head step after the forward: with both gradients requested and the
// shape in range, the loss head runs inside the backward's launches (the row
// losses and the score gradient in the grad_Q gather, their mean in the grad_D
// launch); otherwise lik_ce_rows and then the backward.
lik_status ce_head_and_bwd(const Problem& P, const float* scores, const int32_t* target, float scale, float* loss,
                           float* row_loss, float* grad_scores, const int32_t* argmax, void* grad_Q, void* grad_D,
                           bool same_dtype, cudaStream_t stream, bool* fused) {
    *fused = false;
    if (!grad_Q || !grad_D || !grad_q_ce_fusable(P)) return LIK_OK;
    int dev = 0;
    lik_status st = check_device(&dev);
    if (st != LIK_OK) return st;
    const int64_t rows = P.n_query, cols = P.pairs_per_query;
    const Spec specs[] = {
        {"scores", scores, true, rows * cols},
        {"target", target, true, rows},
        {"loss", loss, true, 1},
        {"row_loss", row_loss, true, rows},
        {"grad_scores", grad_scores, true, rows * cols},
    };
    if ((st = check_buffers(dev, specs, 5)) != LIK_OK) return st;
    if ((st = check_aligned(target, 4, "target")) != LIK_OK) return st;
    if ((st = check_aligned(loss, 4, "loss")) != LIK_OK) return st;
    if ((st = check_aligned(row_loss, 4, "row_loss")) != LIK_OK) return st;
    if ((st = check_aligned(grad_scores, 4, "grad_scores")) != LIK_OK) return st;
    const FusedCe ce{scores, target, scale, row_loss};
    Problem Pc = P;  // the grad_D launch also writes the mean of the row losses
    Pc.ce_loss = loss;
    Pc.ce_row_loss = row_loss;
    *fused = true;
    if (same_dtype) return run_bwd_same(Pc, grad_scores, argmax, grad_Q, grad_D, stream, &ce);
    return run_bwd(Pc, grad_scores, argmax, static_cast<float*>(grad_Q), static_cast<float*>(grad_D), stream, &ce);
}

}  // namespace
}  // namespace lik

using namespace lik;

// ================================================================ C ABI ===

extern "C" {

const char* lik_status_string(lik_status s) {
    switch (s) {
    case LIK_OK: return "LIK_OK";
    case LIK_ERR_INVALID_ARG: return "LIK_ERR_INVALID_ARG";
    case LIK_ERR_UNSUPPORTED: return "LIK_ERR_UNSUPPORTED";
    case LIK_ERR_CUDA: return "LIK_ERR_CUDA";
    case LIK_ERR_TIMEOUT: return "LIK_ERR_TIMEOUT";
    default: return "LIK_ERR_UNKNOWN_STATUS";
    }
}

const char* lik_last_error_message(void) { return t_message; }

const char* lik_version(void) { return "0.1.0"; }

lik_status lik_check_device_error(cudaStream_t stream) {
    t_message[0] = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int* w = device_error_word();
    if (!w) return fail(LIK_ERR_CUDA, "cannot resolve the device error word");
    unsigned int word = 0;
    e = cudaMemcpy(&word, w, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word) {
        const unsigned int zero = 0;
        e = cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    }
    if (word & kErrTimeout) return fail(LIK_ERR_TIMEOUT, "a kernel's bounded wait expired");
    if (word & kErrBadIndex)
        return fail(LIK_ERR_INVALID_ARG, "a saved argmax held an index >= Ld (entries skipped)");
    return LIK_OK;
}

lik_status lik_maxsim_allpairs_fwd(const void* Q, const void* D, lik_dtype dtype, int64_t Nq,
                                   int64_t Nd, int64_t Lq, int64_t Ld, int64_t dim,
                                   const bool* qmask, const bool* dmask, float* scores,
                                   int32_t* argmax, cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, Nq, Nd, Nd, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    Problem P = make_problem(kAllPairs, dtype, Q, D, qmask, dmask, Nq, Nd, Nd, Nq * Nd, Lq, Ld, dim);
    return run_fwd(P, qmask, dmask, scores, argmax, stream);
}

lik_status lik_maxsim_allpairs_bwd(const void* Q, const void* D, lik_dtype dtype, int64_t Nq,
                                   int64_t Nd, int64_t Lq, int64_t Ld, int64_t dim,
                                   const float* grad_out, const int32_t* argmax, float* grad_Q,
                                   float* grad_D, cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, Nq, Nd, Nd, Lq, Ld, dim, &nothing);
    if (st != LIK_OK) return st;
    Problem P = make_problem(kAllPairs, dtype, Q, D, nullptr, nullptr, Nq, Nd, Nd, Nq * Nd, Lq, Ld, dim);
    // With no pairs the gradients are still defined: all zeros.
    if (nothing) P.n_pairs = 0;
    return run_bwd(P, grad_out, argmax, grad_Q, grad_D, stream);
}

lik_status lik_maxsim_pairwise_fwd(const void* Q, const void* D, lik_dtype dtype, int64_t B,
                                   int64_t Lq, int64_t Ld, int64_t dim, const bool* qmask,
                                   const bool* dmask, float* scores, int32_t* argmax,
                                   cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B, 1, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    Problem P = make_problem(kPairwise, dtype, Q, D, qmask, dmask, B, B, 1, B, Lq, Ld, dim);
    return run_fwd(P, qmask, dmask, scores, argmax, stream);
}

lik_status lik_maxsim_pairwise_bwd(const void* Q, const void* D, lik_dtype dtype, int64_t B,
                                   int64_t Lq, int64_t Ld, int64_t dim, const float* grad_out,
                                   const int32_t* argmax, float* grad_Q, float* grad_D,
                                   cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B, 1, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    Problem P = make_problem(kPairwise, dtype, Q, D, nullptr, nullptr, B, B, 1, B, Lq, Ld, dim);
    return run_bwd(P, grad_out, argmax, grad_Q, grad_D, stream);
}

lik_status lik_maxsim_kd_fwd(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t N,
                             int64_t Lq, int64_t Ld, int64_t dim, const bool* qmask,
                             const bool* dmask, float* scores, int32_t* argmax,
                             cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B * N, N, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    Problem P = make_problem(kKd, dtype, Q, D, qmask, dmask, B, B * N, N, B * N, Lq, Ld, dim);
    return run_fwd(P, qmask, dmask, scores, argmax, stream);
}

lik_status lik_maxsim_kd_bwd(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t N,
                             int64_t Lq, int64_t Ld, int64_t dim, const float* grad_out,
                             const int32_t* argmax, float* grad_Q, float* grad_D,
                             cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B * N, N, Lq, Ld, dim, &nothing);
    if (st != LIK_OK) return st;
    Problem P = make_problem(kKd, dtype, Q, D, nullptr, nullptr, B, B * N, N, B * N, Lq, Ld, dim);
    if (nothing) P.n_pairs = 0;
    return run_bwd(P, grad_out, argmax, grad_Q, grad_D, stream);
}

lik_status lik_maxsim_pairwise_fwd_workspace_bytes(lik_dtype dtype, int64_t B, int64_t Lq, int64_t Ld, int64_t dim,
                                                  int has_dmask, size_t* bytes) {
    t_message[0] = 0;
    if (!bytes) return fail(LIK_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B, 1, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    int dev = 0;
    if ((st = check_device(&dev)) != LIK_OK) return st;
    Problem P = make_problem(kPairwise, dtype, nullptr, nullptr, nullptr, nullptr, B, B, 1, B, Lq, Ld, dim);
    if (tc_stream_eligible(P)) *bytes = stream_workspace_bytes(P, has_dmask != 0);
    return LIK_OK;
}

lik_status lik_maxsim_kd_fwd_workspace_bytes(lik_dtype dtype, int64_t B, int64_t N, int64_t Lq, int64_t Ld,
                                            int64_t dim, int has_dmask, size_t* bytes) {
    t_message[0] = 0;
    if (!bytes) return fail(LIK_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B * N, N, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    int dev = 0;
    if ((st = check_device(&dev)) != LIK_OK) return st;
    Problem P = make_problem(kKd, dtype, nullptr, nullptr, nullptr, nullptr, B, B * N, N, B * N, Lq, Ld, dim);
    if (tc_stream_eligible(P)) *bytes = stream_workspace_bytes(P, has_dmask != 0);
    return LIK_OK;
}

lik_status lik_maxsim_pairwise_fwd_ws(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t Lq,
                                      int64_t Ld, int64_t dim, const bool* qmask, const bool* dmask,
                                      float* scores, int32_t* argmax, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B, 1, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    Problem P = make_problem(kPairwise, dtype, Q, D, qmask, dmask, B, B, 1, B, Lq, Ld, dim);
    CallerWorkspace ws;
    ws.given = true;
    ws.ptr = workspace;
    ws.bytes = workspace_bytes;
    return run_fwd(P, qmask, dmask, scores, argmax, stream, false, ws);
}

lik_status lik_maxsim_kd_fwd_ws(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t N, int64_t Lq,
                                int64_t Ld, int64_t dim, const bool* qmask, const bool* dmask, float* scores,
                                int32_t* argmax, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B * N, N, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    Problem P = make_problem(kKd, dtype, Q, D, qmask, dmask, B, B * N, N, B * N, Lq, Ld, dim);
    CallerWorkspace ws;
    ws.given = true;
    ws.ptr = workspace;
    ws.bytes = workspace_bytes;
    return run_fwd(P, qmask, dmask, scores, argmax, stream, false, ws);
}

lik_status lik_maxsim_allpairs_bwd_same_dtype(const void* Q, const void* D, lik_dtype dtype, int64_t Nq,
                                              int64_t Nd, int64_t Lq, int64_t Ld, int64_t dim,
                                              const float* grad_out, const int32_t* argmax, void* grad_Q,
                                              void* grad_D, cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, Nq, Nd, Nd, Lq, Ld, dim, &nothing);
    if (st != LIK_OK) return st;
    Problem P = make_problem(kAllPairs, dtype, Q, D, nullptr, nullptr, Nq, Nd, Nd, Nq * Nd, Lq, Ld, dim);
    if (nothing) P.n_pairs = 0;
    return run_bwd_same(P, grad_out, argmax, grad_Q, grad_D, stream);
}

lik_status lik_maxsim_pairwise_bwd_same_dtype(const void* Q, const void* D, lik_dtype dtype, int64_t B,
                                              int64_t Lq, int64_t Ld, int64_t dim, const float* grad_out,
                                              const int32_t* argmax, void* grad_Q, void* grad_D,
                                              cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B, 1, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    Problem P = make_problem(kPairwise, dtype, Q, D, nullptr, nullptr, B, B, 1, B, Lq, Ld, dim);
    return run_bwd_same(P, grad_out, argmax, grad_Q, grad_D, stream);
}

lik_status lik_maxsim_kd_bwd_same_dtype(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t N,
                                        int64_t Lq, int64_t Ld, int64_t dim, const float* grad_out,
                                        const int32_t* argmax, void* grad_Q, void* grad_D,
                                        cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B * N, N, Lq, Ld, dim, &nothing);
    if (st != LIK_OK) return st;
    Problem P = make_problem(kKd, dtype, Q, D, nullptr, nullptr, B, B * N, N, B * N, Lq, Ld, dim);
    if (nothing) P.n_pairs = 0;
    return run_bwd_same(P, grad_out, argmax, grad_Q, grad_D, stream);
}

lik_status lik_ce_rows(const float* scores, int64_t rows, int64_t cols, const int32_t* target, float scale,
                       float* loss, float* row_loss, float* grad_scores, cudaStream_t stream) {
    t_message[0] = 0;
    if (rows < 0 || cols < 0) return fail(LIK_ERR_INVALID_ARG, "negative size");
    int dev = 0;
    lik_status st = check_device(&dev);
    if (st != LIK_OK) return st;
    const Spec specs[] = {
        {"scores", scores, true, rows * cols},
        {"target", target, true, rows},
        {"loss", loss, true, 1},
        {"row_loss", row_loss, true, rows},
        {"grad_scores", grad_scores, false, rows * cols},
    };
    if ((st = check_buffers(dev, specs, 5)) != LIK_OK) return st;
    if ((st = check_aligned(scores, 4, "scores")) != LIK_OK) return st;
    if ((st = check_aligned(target, 4, "target")) != LIK_OK) return st;
    if ((st = check_aligned(loss, 4, "loss")) != LIK_OK) return st;
    if ((st = check_aligned(row_loss, 4, "row_loss")) != LIK_OK) return st;
    if ((st = check_aligned(grad_scores, 4, "grad_scores")) != LIK_OK) return st;
    const cudaError_t e = launch_ce_rows(scores, rows, cols, target, scale, loss, row_loss,
                                         cols > 0 ? grad_scores : nullptr, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cross-entropy launch");
    return LIK_OK;
}

lik_status lik_maxsim_allpairs_ce_step(const void* Q, const void* D, lik_dtype dtype, int64_t Nq, int64_t Nd,
                                       int64_t Lq, int64_t Ld, int64_t dim, const bool* qmask,
                                       const bool* dmask, const int32_t* target, float scale, float* scores,
                                       int32_t* argmax, float* loss, float* row_loss, float* grad_scores,
                                       void* grad_Q, void* grad_D, int grads_in_input_dtype,
                                       cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, Nq, Nd, Nd, Lq, Ld, dim, &nothing);
    if (st != LIK_OK) return st;
    Problem P = make_problem(kAllPairs, dtype, Q, D, qmask, dmask, Nq, Nd, Nd, Nq * Nd, Lq, Ld, dim);
    if (!nothing) {
        if (!grads_in_input_dtype || dtype == LIK_F32) plan_fwd_zero(P, static_cast<float*>(grad_D));
        if ((st = run_fwd(P, qmask, dmask, scores, argmax, stream)) != LIK_OK) return st;
    }
    if (Nq > 0 && Nd > 0 && !grad_scores) return fail(LIK_ERR_INVALID_ARG, "grad_scores is NULL");
    if (Nq > 0 && Nd > 0) {
        bool fused = false;
        st = ce_head_and_bwd(P, scores, target, scale, loss, row_loss, grad_scores, argmax, grad_Q, grad_D,
                             grads_in_input_dtype != 0, stream, &fused);
        if (st != LIK_OK || fused) return st;
    }
    st = lik_ce_rows(scores, Nq, Nd, target, scale, loss, row_loss, grad_scores, stream);
    if (st != LIK_OK) return st;
    if (grads_in_input_dtype)
        return lik_maxsim_allpairs_bwd_same_dtype(Q, D, dtype, Nq, Nd, Lq, Ld, dim, grad_scores, argmax, grad_Q,
                                                  grad_D, stream);
    return lik_maxsim_allpairs_bwd(Q, D, dtype, Nq, Nd, Lq, Ld, dim, grad_scores, argmax,
                                   static_cast<float*>(grad_Q), static_cast<float*>(grad_D), stream);
}

lik_status lik_maxsim_kd_ce_step(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t N, int64_t Lq,
                                 int64_t Ld, int64_t dim, const bool* qmask, const bool* dmask,
                                 const int32_t* target, float scale, float* scores, int32_t* argmax, float* loss,
                                 float* row_loss, float* grad_scores, void* grad_Q, void* grad_D,
                                 int grads_in_input_dtype, cudaStream_t stream) {
    lik_status st = lik_maxsim_kd_fwd(Q, D, dtype, B, N, Lq, Ld, dim, qmask, dmask, scores, argmax, stream);
    if (st != LIK_OK) return st;
    if (B > 0 && N > 0 && !grad_scores) return fail(LIK_ERR_INVALID_ARG, "grad_scores is NULL");
    if (B > 0 && N > 0) {
        const Problem P = make_problem(kKd, dtype, Q, D, qmask, dmask, B, B * N, N, B * N, Lq, Ld, dim);
        bool fused = false;
        st = ce_head_and_bwd(P, scores, target, scale, loss, row_loss, grad_scores, argmax, grad_Q, grad_D,
                             grads_in_input_dtype != 0, stream, &fused);
        if (st != LIK_OK || fused) return st;
    }
    st = lik_ce_rows(scores, B, N, target, scale, loss, row_loss, grad_scores, stream);
    if (st != LIK_OK) return st;
    if (grads_in_input_dtype)
        return lik_maxsim_kd_bwd_same_dtype(Q, D, dtype, B, N, Lq, Ld, dim, grad_scores, argmax, grad_Q, grad_D,
                                            stream);
    return lik_maxsim_kd_bwd(Q, D, dtype, B, N, Lq, Ld, dim, grad_scores, argmax, static_cast<float*>(grad_Q),
                             static_cast<float*>(grad_D), stream);
}

lik_status lik_maxsim_allpairs_bwd_recompute(const void* Q, const void* D, lik_dtype dtype, int64_t Nq,
                                             int64_t Nd, int64_t Lq, int64_t Ld, int64_t dim,
                                             const bool* qmask, const bool* dmask, const float* grad_out,
                                             int32_t* argmax_workspace, float* grad_Q, float* grad_D,
                                             cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, Nq, Nd, Nd, Lq, Ld, dim, &nothing);
    if (st != LIK_OK) return st;
    Problem P = make_problem(kAllPairs, dtype, Q, D, qmask, dmask, Nq, Nd, Nd, Nq * Nd, Lq, Ld, dim);
    if (nothing) P.n_pairs = 0;
    if (!nothing) {
        plan_fwd_zero(P, grad_D);
        if ((st = run_fwd(P, qmask, dmask, nullptr, argmax_workspace, stream, true)) != LIK_OK) return st;
    }
    return run_bwd(P, grad_out, argmax_workspace, grad_Q, grad_D, stream);
}

lik_status lik_maxsim_pairwise_bwd_recompute(const void* Q, const void* D, lik_dtype dtype, int64_t B,
                                             int64_t Lq, int64_t Ld, int64_t dim, const bool* qmask,
                                             const bool* dmask, const float* grad_out,
                                             int32_t* argmax_workspace, float* grad_Q, float* grad_D,
                                             cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B, 1, Lq, Ld, dim, &nothing);
    if (st != LIK_OK || nothing) return st;
    Problem P = make_problem(kPairwise, dtype, Q, D, qmask, dmask, B, B, 1, B, Lq, Ld, dim);
    if ((st = run_fwd(P, qmask, dmask, nullptr, argmax_workspace, stream, true)) != LIK_OK) return st;
    return run_bwd(P, grad_out, argmax_workspace, grad_Q, grad_D, stream);
}

lik_status lik_maxsim_kd_bwd_recompute(const void* Q, const void* D, lik_dtype dtype, int64_t B, int64_t N,
                                       int64_t Lq, int64_t Ld, int64_t dim, const bool* qmask,
                                       const bool* dmask, const float* grad_out, int32_t* argmax_workspace,
                                       float* grad_Q, float* grad_D, cudaStream_t stream) {
    t_message[0] = 0;
    bool nothing = false;
    lik_status st = check_common(dtype, B, B * N, N, Lq, Ld, dim, &nothing);
    if (st != LIK_OK) return st;
    Problem P = make_problem(kKd, dtype, Q, D, qmask, dmask, B, B * N, N, B * N, Lq, Ld, dim);
    if (nothing) P.n_pairs = 0;
    if (!nothing && (st = run_fwd(P, qmask, dmask, nullptr, argmax_workspace, stream, true)) != LIK_OK) return st;
    return run_bwd(P, grad_out, argmax_workspace, grad_Q, grad_D, stream);
}

}  // extern "C"
