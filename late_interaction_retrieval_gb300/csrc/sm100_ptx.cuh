// sm100_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family,
// built here for sm_103a) features the tensor-core kernels use: mbarriers,
// TMA tensor loads, tcgen05 MMA / TMEM, named barriers.  Written from the
// public PTX ISA; each wrapper is one instruction (or a bounded loop of one).
#pragma once

#include <cstdint>

#include <cuda.h>

#include "lik_internal.h"

namespace lik {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

// One test of the phase; if it has not completed, the thread may be
// suspended in hardware (up to the hint, in ns) until it does, instead of
// spinning on issue slots other warps need.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed.  Bounded: after
// `timeout_ns` it sets kErrTimeout in *err and returns false, so a broken
// pipeline ends the kernel instead of hanging the GPU.
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s; a healthy wait takes microseconds

__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned int* err,
                                              uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err) {
    return mbar_wait_for(bar, parity, err, kWaitTimeoutNs);
}

// Non-blocking test of a phase (no suspend).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait for warps that share their SM sub-partition with busy warps:
// between tests the waiting warp sleeps `nap_ns` (__nanosleep), so its polls
// do not take issue slots from them.  Bounded like mbar_wait.
__device__ __forceinline__ bool mbar_wait_nap(uint32_t bar, uint32_t parity, unsigned int* err, unsigned nap_ns) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
    while (true) {
        __nanosleep(nap_ns);
        if (mbar_test_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
}

// ------------------------------------------------------------------ TMA --

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, int32_t c0, int32_t c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, int32_t c0, int32_t c1,
                                            int32_t c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// -------------------------------------------------------------- tcgen05 --

// Allocate `ncols` TMEM columns (power of two >= 32); the base address is
// written to shared memory at `dst`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, fp32 accumulate, f16/bf16 inputs.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, fp32 accumulate, TF32 inputs
// (32-bit containers; the MMA reads the 19 TF32 bits).
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, fp32 accumulate, TF32 inputs, with
// A (M rows) read from tensor memory: row m in lane m, one TF32 per 32-bit
// column, the K-step's 8 columns starting at `a_tmem`.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued so far has
// completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored as rows
// of 128 bytes with the 128-byte swizzle (the layout a TMA load with
// CU_TENSOR_MAP_SWIZZLE_128B writes); groups of 8 rows are 1024 bytes apart.
// `addr` must lie in a 1024-byte aligned swizzle atom; moving along K inside
// the atom adds the byte offset to the start address.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                 // leading byte offset (unused for SW128 K-major)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 B
    d |= static_cast<uint64_t>(1) << 46;                 // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;                 // swizzle mode: 128-byte
    return d;
}

// One accumulator tile D = A . B^T over K = 16 * nk, issued as nk
// tcgen05.mma of K = 16.  A and B are SW128 K-major tiles split into atoms
// of 64 elements (128 B) along K; atom `a` of A starts at a_base + a * a_atom
// bytes (b likewise), and k-step k reads atom k / 4 at byte offset
// 32 * (k % 4).  The first step overwrites D, the rest accumulate.
// The chain is unrolled to kMaxK guarded steps (none left when nk is a
// compile-time kMaxK): the same instructions under a runtime-bounded loop
// ran about 1.5x slower on sm_103a (measured on a loop of MMAs alone).
template <int kMaxK>
__device__ __forceinline__ void mma_kchain(uint32_t d_tmem, uint32_t a_base, uint32_t a_atom, uint32_t b_base,
                                           uint32_t b_atom, int nk, uint32_t idesc) {
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < nk) {
            const uint32_t off = static_cast<uint32_t>(k & 3) * 32;
            const uint32_t atom = static_cast<uint32_t>(k >> 2);
            mma_f16(d_tmem, sw128_kmajor_desc(a_base + atom * a_atom + off),
                    sw128_kmajor_desc(b_base + atom * b_atom + off), idesc, k != 0);
        }
    }
}

// The same chain for TF32 operands: K = 8 per instruction, so a k-step is
// again 32 bytes of a 128-byte row (4 per swizzle atom of 32 fp32).  With
// `acc_first` the first step accumulates too (a later product of a split).
template <int kMaxK>
__device__ __forceinline__ void mma_tf32_kchain(uint32_t d_tmem, uint32_t a_base, uint32_t a_atom, uint32_t b_base,
                                                uint32_t b_atom, int nk, uint32_t idesc, bool acc_first) {
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < nk) {
            const uint32_t off = static_cast<uint32_t>(k & 3) * 32;
            const uint32_t atom = static_cast<uint32_t>(k >> 2);
            mma_tf32(d_tmem, sw128_kmajor_desc(a_base + atom * a_atom + off),
                     sw128_kmajor_desc(b_base + atom * b_atom + off), idesc, acc_first || k != 0);
        }
    }
}

// The same chain with A in tensor memory (columns a_col + 8k for k-step k).
template <int kMaxK>
__device__ __forceinline__ void mma_tf32_ts_kchain(uint32_t d_tmem, uint32_t a_col, uint32_t b_base, uint32_t b_atom,
                                                   int nk, uint32_t idesc, bool acc_first) {
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < nk) {
            const uint32_t off = static_cast<uint32_t>(k & 3) * 32;
            const uint32_t atom = static_cast<uint32_t>(k >> 2);
            mma_tf32_ts(d_tmem, a_col + 8u * static_cast<uint32_t>(k), sw128_kmajor_desc(b_base + atom * b_atom + off),
                        idesc, acc_first || k != 0);
        }
    }
}

// Instruction descriptor of tcgen05.mma .kind::tf32: fp32 accumulator, A and
// B TF32 (format code 2), both K-major, M x N.
__host__ __device__ constexpr uint32_t tf32_idesc(int M, int N) {
    return (1u << 4)                                   // D format: f32
           | (2u << 7)                                 // A format: tf32
           | (2u << 10)                                // B format: tf32
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Instruction descriptor of tcgen05.mma .kind::f16: fp32 accumulator,
// A and B of one type (bf16 when `bf16`, else fp16), both K-major, M x N.
__host__ __device__ constexpr uint32_t f16_idesc(int M, int N, bool bf16) {
    return (1u << 4)                                   // D format: f32
           | ((bf16 ? 1u : 0u) << 7)                   // A format
           | ((bf16 ? 1u : 0u) << 10)                  // B format
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

#define LIK_TMEM_LD_X32_OUT(v)                                                                    \
    "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),            \
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),    \
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),              \
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),              \
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-wide).  The
// load and its wait sit in one asm statement, so no use of the outputs can be
// scheduled before the data has arrived.
__device__ __forceinline__ void tmem_ld_32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : LIK_TMEM_LD_X32_OUT(v)
        : "r"(taddr)
        : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-wide), waited.
__device__ __forceinline__ void tmem_ld_16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

// Two 16-column loads (two TMEM addresses of this thread's lane) in flight
// together, one wait for both.
__device__ __forceinline__ void tmem_ld_16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, "
        "%26, %27, %28, %29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
          "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]),
          "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]),
          "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]),
          "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
        : "r"(ta), "r"(tb)
        : "memory");
}

// Two 32-column loads of this thread's lane in flight together, one wait.
__device__ __forceinline__ void tmem_ld_32x2(uint32_t ta, uint32_t tb, uint32_t (&a)[32], uint32_t (&b)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, "
        "%42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, "
        "%60, %61, %62, %63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : LIK_TMEM_LD_X32_OUT(a), LIK_TMEM_LD_X32_OUT(b)
        : "r"(ta), "r"(tb)
        : "memory");
}

// Store 32 consecutive 32-bit columns of this thread's lane (warp-wide; the
// warp's lanes are its TMEM lane quarter).  Completion: tmem_wait_st().
__device__ __forceinline__ void tmem_st_32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, "
        "%31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// tcgen05.ld.red (sm_103a): the 16 columns as tmem_ld_16 returns them, and
// in `mx` their maximum (IEEE max; +0 over -0), computed by the load.
__device__ __forceinline__ void tmem_ldmax_16(uint32_t taddr, uint32_t (&v)[16], float& mx) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15}, %16, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=f"(mx)
        : "r"(taddr)
        : "memory");
}

// Two tmem_ldmax_16 loads in flight together, one wait for both.
__device__ __forceinline__ void tmem_ldmax_16x2(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16],
                                                float& ma, float& mb) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15}, %32, [%34];\n\t"
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, "
        "%25, %26, %27, %28, %29, %30, %31}, %33, [%35];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
          "=r"(a[7]), "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]),
          "=r"(a[14]), "=r"(a[15]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]),
          "=r"(b[5]), "=r"(b[6]), "=r"(b[7]), "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]),
          "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]), "=f"(ma), "=f"(mb)
        : "r"(ta), "r"(tb)
        : "memory");
}

}  // namespace ptx
}  // namespace lik
