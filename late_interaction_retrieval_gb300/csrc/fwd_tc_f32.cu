// fwd_tc_f32.cu -- MaxSim forward for fp32 inputs on the sm_103a tensor cores.
//
// What it computes (Late Interaction Kernels README, "What does it compute?"
// and "Scoring interface"): for every pair p of query q and document d of the
// layout, score[p] = sum over valid i of max over valid j of Q[q,i].D[d,j],
// the lowest j reaching each max saved as argmax, -1e9 for a document with no
// valid token.  The README ("Precision and compatibility") accepts fp32
// inputs; its own accelerated path rounds them to half precision.  Here fp32
// inputs keep fp32 accuracy (scores within 1e-5 of an exact result), which
// rules out rounding them to 16 bits.
//
// Split precision.  Every fp32 element x is split into two TF32 values
// hi = round(x) and lo = round(x - hi) (round to nearest, 11 significant bits
// each), so x = hi + lo to about 2^-22 relative.  A similarity is then
//     Q.D = Ql.Dh + Qh.Dl + Qh.Dh   (+ Ql.Dl, about 2^-22 relative, dropped)
// three tcgen05.mma.kind::tf32 products into one fp32 TMEM accumulator, the
// two small ones first.
//
// Tiling.  A row block holds the 128 query tokens of floor(128/Lq) whole
// queries (all-pairs) or of one query (pairwise, per-query candidates; its
// rows past Lq belong to other queries and are ignored).  Documents are cut
// into tiles of 64 tokens from their first token (TMA zero-fills past Ld).
// One tile = S[128, 64] += Qblock[128, dim] . Dtile[64, dim]^T, issued as
// 3 * dim/8 tcgen05.mma (M=128, N=64, K=8) with the row block's hi and lo
// halves in tensor memory (A operand) and the tile's in shared memory (B):
// with both operands in shared memory, the 128-row A operand re-read by
// every K=8 step bounds the MMA by shared-memory bandwidth (measured: the
// tensor pipe 18% busy).  A work unit is a row block and a run of its
// documents; the CTAs (one per SM) take units round-robin.
//
// Tensor memory (512 columns): the row block's hi halves in columns
// [0, dim), lo in [128, 128 + dim), four accumulators of 64 columns from 256.
// Shared memory: 2..6 document stages, each a TMA-written fp32 tile
// converted to hi in place plus its lo half (64 KB at dim 128).
//
// Roles (352 threads, one CTA per SM):
//   warp 0      TMA producer: document tiles into the stages
//   warps 1, 10 MMA issuers of alternate tiles (warp 1 also allocates TMEM):
//               a thread issuing a chain waits for the tensor pipe, so with
//               one issuer its barrier checks between chains would leave the
//               pipe idle
//   warps 2-5   converters: split each landed tile into hi/lo in place and
//               hand the stage to the MMA (fence.proxy.async makes the writes
//               visible to the tensor core); per unit, once the previous
//               unit's MMAs are done, read the row block from global memory
//               (one row per thread), split it and store it into tensor
//               memory (each warp its lane quarter)
//   warps 6-9   epilogue: one accumulator row (query token) per thread; a
//               running (max, argmax) over the valid columns of each tile,
//               read with tcgen05.ld.red (each 16-column unit with its max,
//               so a fully valid unit needs no ALU work for its max);
//               at a document's end the valid tokens' maxima are summed per
//               query in a fixed order and score and argmax written
// Every mbarrier wait is bounded (ptx::mbar_wait); on expiry the kernel sets
// the library's error word, drains its own copies and MMAs, frees TMEM and
// returns.
#include <cfloat>

#include "lik_internal.h"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace lik {
namespace {

constexpr int kM = 128;            // accumulator rows (query tokens) per row block
constexpr int kT = 64;             // document tokens per tile (MMA N)
constexpr int kAtomBytes = 128;    // one 128-byte swizzle row = 32 fp32
constexpr int kAtomElems = 32;
constexpr int kMaxDim = 128;       // the row block's halves take 2 x 128 TMEM columns
constexpr int kMaxStages = 6;
constexpr int kAcc = 4;            // accumulator buffers of kT columns
constexpr int kTmemCols = 512;
constexpr uint32_t kQhiCol = 0, kQloCol = 128, kAccCol = 256;
constexpr int kConvWarps = 4;
constexpr int kEpiWarps = 4;
constexpr int kIssuers = 2;        // MMA issuing threads (warp 1 and the last warp), alternate tiles
constexpr int kThreads = 32 * (1 + kIssuers + kConvWarps + kEpiWarps);

struct Params {
    int64_t Nq, Nd, Lq, Ld;
    int64_t pairs_per_query;
    int layout, dim, atoms, nk, tiles_per_doc, qpt, n_rb, dpu, stages;
    int64_t n_units;
    uint32_t idesc, d_bytes;
    const float* Q;
    const uint8_t* qmask;
    const uint8_t* dmask;
    float* scores;
    int32_t* argmax;
    unsigned int* err;
};

struct Bars {
    uint64_t full_d[kMaxStages], conv_d[kMaxStages], empty_d[kMaxStages];
    uint64_t conv_q, empty_q;
    uint64_t acc_full[kAcc], acc_empty[kAcc];
    uint64_t xfull[2];   // every epilogue thread has written a document's per-row terms
    uint64_t mma_done;
    uint64_t exit_bar;   // every warp is done (one arrive per warp): TMEM may be released
    uint32_t tmem_base;
    uint32_t pad;
};

struct Exchange {
    float term[2][kM];   // per row: max of a valid query token of a non-empty document, else 0
};

// Work unit u: row block and document range [d0, d1).
struct Unit {
    int64_t rb, d0, d1;
};

__device__ __forceinline__ Unit unit_of(const Params& p, int64_t u) {
    Unit w;
    if (p.layout == kAllPairs) {
        w.rb = u % p.n_rb;
        w.d0 = (u / p.n_rb) * p.dpu;
        w.d1 = w.d0 + p.dpu < p.Nd ? w.d0 + p.dpu : p.Nd;
    } else {  // one query per unit, its own documents
        w.rb = u;
        w.d0 = u * p.pairs_per_query;
        w.d1 = w.d0 + p.pairs_per_query;
    }
    return w;
}

__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// Split `n16` 16-byte chunks at `hi` (fp32 written by TMA) into TF32 hi (in
// place) and lo (same offset at `lo`); thread t of the converter warps takes
// chunks t, t + 128, ...  Elementwise, so the swizzled layout is kept.
__device__ __forceinline__ void split_tile(uint8_t* hi, uint8_t* lo, int n16, int t) {
#pragma unroll 4
    for (int c = t; c < n16; c += 32 * kConvWarps) {
        float4 x = *reinterpret_cast<const float4*>(hi + 16 * c);
        const uint32_t h0 = tf32_rna(x.x), h1 = tf32_rna(x.y), h2 = tf32_rna(x.z), h3 = tf32_rna(x.w);
        const uint32_t l0 = tf32_rna(x.x - __uint_as_float(h0)), l1 = tf32_rna(x.y - __uint_as_float(h1));
        const uint32_t l2 = tf32_rna(x.z - __uint_as_float(h2)), l3 = tf32_rna(x.w - __uint_as_float(h3));
        *reinterpret_cast<uint4*>(hi + 16 * c) = make_uint4(h0, h1, h2, h3);
        *reinterpret_cast<uint4*>(lo + 16 * c) = make_uint4(l0, l1, l2, l3);
    }
}

// Generic-proxy writes to shared memory made visible to the tensor core.
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 elements [c0, c0 + 32) of this thread's Q row (zeros past dim or for a
// row past the last query token), as raw fp32 bits.
__device__ __forceinline__ void load_q_chunk(const Params& p, int64_t row, int c0, uint32_t (&x)[32]) {
    const bool in = row < p.Nq * p.Lq;
    const float* src = p.Q + row * p.dim + c0;
#pragma unroll
    for (int v = 0; v < 8; ++v) {
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in && c0 + 4 * v < p.dim) f = __ldg(reinterpret_cast<const float4*>(src + 4 * v));
        x[4 * v] = __float_as_uint(f.x);
        x[4 * v + 1] = __float_as_uint(f.y);
        x[4 * v + 2] = __float_as_uint(f.z);
        x[4 * v + 3] = __float_as_uint(f.w);
    }
}

// The tile's 64 columns: bit j of word h = document token t*kT + 32h + j is valid.
__device__ __forceinline__ uint8_t col_valid_byte(const Params& p, int64_t d, int t, int h, int lane) {
    const int64_t j = static_cast<int64_t>(t) * kT + 32 * h + lane;
    if (j >= p.Ld) return 0;
    return p.dmask ? p.dmask[d * p.Ld + j] : uint8_t(1);
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Folds 16 columns (values v, validity bits mw, first column col, the load's
// max of all 16 mred) into the row's running (max m, argmax am): the unit's
// max over its valid columns (mred when all are valid), and, only when it is
// strictly larger than m, its lowest column holding it.
__device__ __forceinline__ void fold16(const uint32_t* v, uint32_t mw, float mred, int col, float& m, int& am) {
    if (mw == 0) return;
    if (mw == 0xffffu) {  // every column valid: the load's own max
        if (mred > m) {
            int idx = 15;
#pragma unroll
            for (int c = 14; c >= 0; --c) idx = __uint_as_float(v[c]) == mred ? c : idx;
            m = mred;
            am = col + idx;
        }
        return;
    }
    float x[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) x[c] = ((mw >> c) & 1u) ? __uint_as_float(v[c]) : -FLT_MAX;
    const float a = max3f(x[0], x[1], x[2]), b = max3f(x[3], x[4], x[5]), c3 = max3f(x[6], x[7], x[8]);
    const float d = max3f(x[9], x[10], x[11]), e = max3f(x[12], x[13], x[14]);
    const float um = max3f(max3f(a, b, c3), fmaxf(d, e), x[15]);
    if (um > m) {
        int idx = 15;
#pragma unroll
        for (int c = 14; c >= 0; --c) idx = x[c] == um ? c : idx;
        m = um;
        am = col + idx;
    }
}

// The tile's four 16-column units with their maxima (tcgen05.ld.red, an
// sm_103a load-with-reduction), one wait for all four.
__device__ __forceinline__ void tmem_ldmax_16x4(uint32_t ta, uint32_t (&v)[4][16], float (&mx)[4]) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, "
        "%10, %11, %12, %13, %14, %15}, %64, [%68];\n\t"
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, "
        "%25, %26, %27, %28, %29, %30, %31}, %65, [%69];\n\t"
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, "
        "%41, %42, %43, %44, %45, %46, %47}, %66, [%70];\n\t"
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%48, %49, %50, %51, %52, %53, %54, %55, %56, "
        "%57, %58, %59, %60, %61, %62, %63}, %67, [%71];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0][0]), "=r"(v[0][1]), "=r"(v[0][2]), "=r"(v[0][3]), "=r"(v[0][4]), "=r"(v[0][5]),
          "=r"(v[0][6]), "=r"(v[0][7]), "=r"(v[0][8]), "=r"(v[0][9]), "=r"(v[0][10]), "=r"(v[0][11]),
          "=r"(v[0][12]), "=r"(v[0][13]), "=r"(v[0][14]), "=r"(v[0][15]),
          "=r"(v[1][0]), "=r"(v[1][1]), "=r"(v[1][2]), "=r"(v[1][3]), "=r"(v[1][4]), "=r"(v[1][5]),
          "=r"(v[1][6]), "=r"(v[1][7]), "=r"(v[1][8]), "=r"(v[1][9]), "=r"(v[1][10]), "=r"(v[1][11]),
          "=r"(v[1][12]), "=r"(v[1][13]), "=r"(v[1][14]), "=r"(v[1][15]),
          "=r"(v[2][0]), "=r"(v[2][1]), "=r"(v[2][2]), "=r"(v[2][3]), "=r"(v[2][4]), "=r"(v[2][5]),
          "=r"(v[2][6]), "=r"(v[2][7]), "=r"(v[2][8]), "=r"(v[2][9]), "=r"(v[2][10]), "=r"(v[2][11]),
          "=r"(v[2][12]), "=r"(v[2][13]), "=r"(v[2][14]), "=r"(v[2][15]),
          "=r"(v[3][0]), "=r"(v[3][1]), "=r"(v[3][2]), "=r"(v[3][3]), "=r"(v[3][4]), "=r"(v[3][5]),
          "=r"(v[3][6]), "=r"(v[3][7]), "=r"(v[3][8]), "=r"(v[3][9]), "=r"(v[3][10]), "=r"(v[3][11]),
          "=r"(v[3][12]), "=r"(v[3][13]), "=r"(v[3][14]), "=r"(v[3][15]),
          "=f"(mx[0]), "=f"(mx[1]), "=f"(mx[2]), "=f"(mx[3])
        : "r"(ta), "r"(ta + 16), "r"(ta + 32), "r"(ta + 48)
        : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
allpairs_fwd_tf32_kernel(const __grid_constant__ CUtensorMap tmd, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* dbuf = smem;                                  // stages x (hi d_bytes, lo d_bytes)
    Bars* bars = reinterpret_cast<Bars*>(dbuf + 2 * p.stages * p.d_bytes);
    Exchange* xc = reinterpret_cast<Exchange*>(bars + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned int* err = p.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->full_d[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->conv_d[s]), kConvWarps);
            ptx::mbar_init(ptx::smem_u32(&bars->empty_d[s]), 1);
        }
        ptx::mbar_init(ptx::smem_u32(&bars->conv_q), kConvWarps);
        ptx::mbar_init(ptx::smem_u32(&bars->empty_q), kIssuers);
        for (int b = 0; b < kAcc; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bars->acc_full[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->acc_empty[b]), kEpiWarps);
        }
        // one arrival per epilogue warp (lane 0, after __syncwarp)
        for (int b = 0; b < 2; ++b) ptx::mbar_init(ptx::smem_u32(&bars->xfull[b]), kEpiWarps);
        ptx::mbar_init(ptx::smem_u32(&bars->mma_done), kIssuers);
        ptx::mbar_init(ptx::smem_u32(&bars->exit_bar), kThreads / 32);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    const int tpd = p.tiles_per_doc;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane == 0) {
            ptx::prefetch_tmap(&tmd);
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_d = 0, last_ph_d = 0;
            bool ok = true;
            for (int64_t u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
                const Unit w = unit_of(p, u);
                for (int64_t d = w.d0; ok && d < w.d1; ++d) {
                    for (int t = 0; t < tpd; ++t) {
                        if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->empty_d[s]), ph ^ 1, err))) break;
                        const uint32_t fd = ptx::smem_u32(&bars->full_d[s]);
                        ptx::mbar_arrive_expect_tx(fd, p.d_bytes);
                        uint8_t* dh = dbuf + 2 * s * p.d_bytes;
                        for (int a = 0; a < p.atoms; ++a)
                            ptx::tma_load_3d(ptx::smem_u32(dh + a * kT * kAtomBytes), &tmd, a * kAtomElems, t * kT,
                                             static_cast<int32_t>(d), fd);
                        issued_d |= 1u << s;
                        last_ph_d = (last_ph_d & ~(1u << s)) | (ph << s);
                        if (++s == p.stages) { s = 0; ph ^= 1; }
                    }
                }
            }
            // every issued load must land before the CTA may exit
            for (int k = 0; k < p.stages; ++k)
                if (issued_d & (1u << k))
                    ptx::mbar_wait(ptx::smem_u32(&bars->full_d[k]), (last_ph_d >> k) & 1u, err);
        }
    } else if (warp == 1 || warp == 2 + kConvWarps + kEpiWarps) {
        // ----------------------------------------------------------- MMA --
        // Both issuers follow the whole tile sequence and issue every other
        // tile; each commits its own tiles, and both release the row block at
        // the end of a unit and take part in the final drain.
        if (lane == 0) {
            const int who = warp == 1 ? 0 : 1;
            int s = 0, ab = 0;
            uint32_t ph = 0, aph = 0, qph = 0;
            int64_t kt = 0;  // tile index in this CTA's sequence
            bool ok = true;
            const uint32_t qh_a = tmem_base + kQhiCol, ql_a = tmem_base + kQloCol;
            for (int64_t u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
                const Unit w = unit_of(p, u);
                if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->conv_q), qph, err))) break;
                qph ^= 1;
                ptx::tc_fence_after();
                for (int64_t d = w.d0; ok && d < w.d1; ++d) {
                    for (int t = 0; t < tpd; ++t, ++kt) {
                        if ((kt & 1) == who) {
                            if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->conv_d[s]), ph, err))) break;
                            if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->acc_empty[ab]), aph ^ 1, err))) break;
                            ptx::tc_fence_after();
                            const uint32_t dh_a = ptx::smem_u32(dbuf + 2 * s * p.d_bytes);
                            const uint32_t dl_a = dh_a + p.d_bytes;
                            const uint32_t acc = tmem_base + kAccCol + ab * kT;
                            constexpr uint32_t d_atom = kT * kAtomBytes;
                            // lo.hi and hi.lo first, then hi.hi
                            ptx::mma_tf32_ts_kchain<kMaxDim / 8>(acc, ql_a, dh_a, d_atom, p.nk, p.idesc, false);
                            ptx::mma_tf32_ts_kchain<kMaxDim / 8>(acc, qh_a, dl_a, d_atom, p.nk, p.idesc, true);
                            ptx::mma_tf32_ts_kchain<kMaxDim / 8>(acc, qh_a, dh_a, d_atom, p.nk, p.idesc, true);
                            ptx::mma_commit(ptx::smem_u32(&bars->empty_d[s]));
                            ptx::mma_commit(ptx::smem_u32(&bars->acc_full[ab]));
                        }
                        if (++s == p.stages) { s = 0; ph ^= 1; }
                        if (++ab == kAcc) { ab = 0; aph ^= 1; }
                    }
                }
                // the row block in tensor memory is free once the unit's MMAs complete
                ptx::mma_commit(ptx::smem_u32(&bars->empty_q));
            }
            ptx::mma_commit(ptx::smem_u32(&bars->mma_done));
            ptx::mbar_wait(ptx::smem_u32(&bars->mma_done), 0, err);
        }
    } else if (warp < 2 + kConvWarps) {
        // ---------------------------------------------------- converters --
        // Per unit: its first tiles (while the previous unit's last MMAs run),
        // the row block into tensor memory (once those MMAs are done), the
        // remaining tiles.  Warp w stores lane quarter w % 4.
        const int t = threadIdx.x - 64;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        int s = 0;
        uint32_t ph = 0, qph = 0;
        bool ok = true;
        const int d16 = kT * p.atoms * (kAtomBytes / 16);
        auto convert_tile = [&]() -> bool {
            bool w_ok = ptx::mbar_wait(ptx::smem_u32(&bars->full_d[s]), ph, err);
            w_ok = __all_sync(0xffffffffu, w_ok);
            if (!w_ok) return false;
            uint8_t* dh = dbuf + 2 * s * p.d_bytes;
            split_tile(dh, dh + p.d_bytes, d16, t);
            fence_async_shared();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->conv_d[s]));
            if (++s == p.stages) { s = 0; ph ^= 1; }
            return true;
        };
        for (int64_t u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
            const Unit w = unit_of(p, u);
            const int64_t ntiles = (w.d1 - w.d0) * tpd;
            const int64_t q_at = ntiles < p.stages ? ntiles : p.stages;
            const int64_t row = w.rb * p.qpt * p.Lq + r;
            uint32_t x[32];
            load_q_chunk(p, row, 0, x);  // in flight while the previous unit finishes
            int64_t k = 0;
            for (; ok && k < q_at; ++k) ok = convert_tile();
            if (!ok) break;
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->empty_q), qph ^ 1, err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            qph ^= 1;
            ptx::tc_fence_after();
            for (int c0 = 0; c0 < p.dim; c0 += 32) {
                if (c0 > 0) load_q_chunk(p, row, c0, x);
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    hi[e] = tf32_rna(__uint_as_float(x[e]));
                    lo[e] = tf32_rna(__uint_as_float(x[e]) - __uint_as_float(hi[e]));
                }
                ptx::tmem_st_32(tmem_base + lane_off + kQhiCol + c0, hi);
                ptx::tmem_st_32(tmem_base + lane_off + kQloCol + c0, lo);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->conv_q));
            for (; ok && k < ntiles; ++k) ok = convert_tile();
        }
    } else {
        // ------------------------------------------------------ epilogue --
        const int quarter = warp & 3;          // TMEM lane quarter of this warp
        const int r = quarter * 32 + lane;     // accumulator row of this thread
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int64_t Lq = p.Lq;
        const int rows_used = p.qpt * static_cast<int>(Lq);
        const int qloc = static_cast<int>(r / Lq);
        const int iq = static_cast<int>(r - static_cast<int64_t>(qloc) * Lq);
        int ab = 0, xb = 0;
        uint32_t aph = 0, xph = 0;  // xph bit b: phase of xfull[b]
        bool ok = true;
        for (int64_t u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
            const Unit w = unit_of(p, u);
            const int64_t q = w.rb * p.qpt + qloc;  // this row's query
            const bool row_ok = r < rows_used && q < p.Nq;
            const bool qvalid = row_ok && (p.qmask ? p.qmask[q * Lq + iq] != 0 : true);
            for (int64_t d = w.d0; ok && d < w.d1; ++d) {
                float m = -INFINITY;
                int am = -1;
                bool any = false;
                uint8_t pre0 = col_valid_byte(p, d, 0, 0, lane), pre1 = col_valid_byte(p, d, 0, 1, lane);
                for (int t = 0; t < tpd; ++t) {
                    const uint32_t mw0 = __ballot_sync(0xffffffffu, pre0 != 0);
                    const uint32_t mw1 = __ballot_sync(0xffffffffu, pre1 != 0);
                    if (t + 1 < tpd) {
                        pre0 = col_valid_byte(p, d, t + 1, 0, lane);
                        pre1 = col_valid_byte(p, d, t + 1, 1, lane);
                    }
                    any = any || (mw0 | mw1) != 0;
                    ok = ptx::mbar_wait(ptx::smem_u32(&bars->acc_full[ab]), aph, err);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    ptx::tc_fence_after();
                    uint32_t rv[4][16];
                    float rmax[4];
                    const uint32_t acc = tmem_base + kAccCol + ab * kT + lane_off;
                    tmem_ldmax_16x4(acc, rv, rmax);
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->acc_empty[ab]));
                    if (++ab == kAcc) { ab = 0; aph ^= 1; }
                    // ascending columns, strictly larger wins: the lowest index on ties
                    const int j0 = t * kT;
                    fold16(rv[0], mw0 & 0xffffu, rmax[0], j0, m, am);
                    fold16(rv[1], mw0 >> 16, rmax[1], j0 + 16, m, am);
                    fold16(rv[2], mw1 & 0xffffu, rmax[2], j0 + 32, m, am);
                    fold16(rv[3], mw1 >> 16, rmax[3], j0 + 48, m, am);
                }
                if (!ok) break;
                // ---- document end: sum each query's valid tokens in a fixed order
                const bool live = any && qvalid;
                if (Lq == 32) {
                    // the warp's 32 rows are one query's tokens: a butterfly, no exchange
                    float tsum = live ? m : 0.0f;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, off);
                    const int64_t pair = p.layout == kAllPairs ? q * p.Nd + d : d;
                    if (row_ok && lane == 0 && p.scores) p.scores[pair] = any ? tsum : kEmptyDocScore;
                    if (row_ok && p.argmax) p.argmax[pair * Lq + iq] = live ? am : -1;
                    continue;
                }
                xc->term[xb][r] = live ? m : 0.0f;
                // all rows written (bounded wait); the buffer is written again two
                // documents later, after every thread has passed the next one's wait
                __syncwarp();  // the warp's term writes precede lane 0's arrive (release)
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->xfull[xb]));
                ok = ptx::mbar_wait(ptx::smem_u32(&bars->xfull[xb]), (xph >> xb) & 1u, err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                xph ^= 1u << xb;
                const int64_t pair = p.layout == kAllPairs ? q * p.Nd + d : d;
                if (row_ok && iq == 0) {
                    const float* tt = xc->term[xb] + r;
                    float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
                    int64_t k4 = 0;
                    for (; k4 + 4 <= Lq; k4 += 4) {
                        s0 += tt[k4];
                        s1 += tt[k4 + 1];
                        s2 += tt[k4 + 2];
                        s3 += tt[k4 + 3];
                    }
                    for (; k4 < Lq; ++k4) s0 += tt[k4];
                    if (p.scores) p.scores[pair] = any ? (s0 + s1) + (s2 + s3) : kEmptyDocScore;
                }
                if (row_ok && p.argmax) p.argmax[pair * Lq + iq] = live ? am : -1;
                xb ^= 1;
            }
        }
    }

    // Release TMEM once every warp has finished with it: each warp arrives
    // once on an mbarrier after its last tensor-memory access, and the
    // allocating warp waits for all of them (bounded) before freeing the
    // columns.  In the producer and the two MMA issuers, lane 0 alone did the work:
    // it arrives for its warp and the other lanes leave (the allocating
    // warp's lanes wait for lane 0 first, since the free is warp-wide).  An
    // mbarrier rather than a CTA barrier: the warps arrive microseconds
    // apart, and timing of this kernel showed bar.sync letting warps through
    // before the last warp had arrived.
    ptx::tc_fence_before();
    if (warp <= 1 || warp == 2 + kConvWarps + kEpiWarps) {
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->exit_bar));
    } else {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->exit_bar));
    }
    if (warp == 1) {
        __syncwarp();
        ptx::mbar_wait(ptx::smem_u32(&bars->exit_bar), 0, p.err);
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

int ceil_div_i(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

size_t f32_misc_bytes() { return sizeof(Bars) + sizeof(Exchange); }

}  // namespace

bool tc_f32_eligible(const Problem& P) {
    if (P.dtype != kF32 || P.dim % 8 != 0 || P.dim > kMaxDim || P.Lq < 1 || P.Lq > kM || P.Ld < 1) return false;
    if (P.n_query * P.Lq >= (int64_t(1) << 31) || P.Ld >= (int64_t(1) << 31) || P.n_doc >= (int64_t(1) << 31))
        return false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const int atoms = static_cast<int>((P.dim + kAtomElems - 1) / kAtomElems);
    const size_t need = 1024 + 2 * 2 * static_cast<size_t>(atoms) * kT * kAtomBytes + f32_misc_bytes();
    return need <= static_cast<size_t>(device_info(dev).max_smem_optin);
}

cudaError_t launch_fwd_tc_f32(const Problem& P, float* scores, int32_t* argmax, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const DeviceInfo& info = device_info(dev);

    Params p{};
    p.Nq = P.n_query;
    p.Nd = P.n_doc;
    p.Lq = P.Lq;
    p.Ld = P.Ld;
    p.pairs_per_query = P.pairs_per_query;
    p.layout = P.layout;
    p.dim = static_cast<int>(P.dim);
    p.atoms = (p.dim + kAtomElems - 1) / kAtomElems;
    p.nk = p.dim / 8;
    p.d_bytes = static_cast<uint32_t>(p.atoms * kT * kAtomBytes);
    const size_t misc = f32_misc_bytes();
    const size_t budget = static_cast<size_t>(info.max_smem_optin) - 1024 - misc;
    p.stages = static_cast<int>(budget / (2 * static_cast<size_t>(p.d_bytes)));
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (p.stages < 2) return cudaErrorInvalidConfiguration;  // tc_f32_eligible rules this out
    p.tiles_per_doc = ceil_div_i(P.Ld, kT);
    if (P.layout == kAllPairs) {
        p.qpt = static_cast<int>(kM / P.Lq);
        p.n_rb = ceil_div_i(P.n_query, p.qpt);
        // units of about 64 tiles, at least one document each (the row block
        // is loaded into tensor memory once per unit), but enough of them for
        // every SM
        int dpu = ceil_div_i(64, p.tiles_per_doc);
        const int64_t chunks_min = (static_cast<int64_t>(info.sm_count) + p.n_rb - 1) / p.n_rb;
        while (dpu > 1 && ceil_div_i(P.n_doc, dpu) < chunks_min) --dpu;
        p.dpu = dpu;
        p.n_units = static_cast<int64_t>(p.n_rb) * ceil_div_i(P.n_doc, p.dpu);
    } else {
        p.qpt = 1;
        p.n_rb = static_cast<int>(P.n_query);
        p.dpu = static_cast<int>(P.pairs_per_query);
        p.n_units = P.n_query;
    }
    p.idesc = ptx::tf32_idesc(kM, kT);
    p.Q = static_cast<const float*>(P.Q);
    p.qmask = P.qmask;
    p.dmask = P.dmask;
    p.scores = scores;
    p.argmax = argmax;
    p.err = device_error_word();

    CUtensorMap tmd;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(P.dim), static_cast<uint64_t>(P.Ld),
                                  static_cast<uint64_t>(P.n_doc)};
        const uint64_t strides[2] = {static_cast<uint64_t>(P.dim) * 4, static_cast<uint64_t>(P.Ld * P.dim) * 4};
        const uint32_t box[3] = {kAtomElems, kT, 1};
        if (!encode_tmap_kmajor(&tmd, kF32, P.D, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const size_t smem = 1024 + 2 * static_cast<size_t>(p.stages) * p.d_bytes + misc;
    e = cudaFuncSetAttribute(allpairs_fwd_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const int64_t grid = p.n_units < info.sm_count ? p.n_units : info.sm_count;
    allpairs_fwd_tf32_kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tmd, p);
    return cudaGetLastError();
}

}  // namespace lik
