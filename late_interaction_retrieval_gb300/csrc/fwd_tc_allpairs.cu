// fwd_tc_allpairs.cu -- all-pairs MaxSim forward on the sm_103a tensor cores.
//
// What it computes (Late Interaction Kernels README, "What does it compute?"
// and "Scoring interface"): for every query q and document d,
//   score[q,d] = sum over valid i of max over valid j of Q[q,i].D[d,j]
// with the lowest j reaching each max saved as argmax, -1e9 for documents
// with no valid token.  The similarity grid is never written anywhere: it
// lives one tile at a time in tensor memory (LIK announcement thread, post
// 4/N: stream document tiles through on-chip memory and keep a running max;
// the design below is our own).
//
// Tiling.  Q is viewed as [Nq*Lq, dim]: a row block holds floor(128/Lq)
// whole queries (128 accumulator rows, one query token per row).  D is
// viewed as [Nd, Ld, dim]; every document is cut into tiles of T <= 256
// tokens that start at its first token, so a tile never straddles two
// documents (the last tile's columns past Ld are zero-filled by TMA and
// masked).  One tile is the MMA
//     S[128, T] = Qblock[128, dim] . Dtile[T, dim]^T      (fp32 in TMEM)
// issued as dim/16 tcgen05.mma (kind::f16, M=128, N=T, K=16).
//
// Warp roles (640 threads, one CTA per SM, persistent over work units):
//   warp 0      TMA producer: Q row blocks (2 buffers) and D tiles (S stages)
//   warp 1      TMEM allocator + MMA issuer of the even tiles
//   warps 2..17 epilogue: four warpgroups; warp w reads TMEM lanes
//               32*(w%4)..+31, i.e. one accumulator row per thread.  The
//               warpgroups split each tile's 16-column units round-robin
//               (unit u goes to group u % 4) and keep a running (max, argmax)
//               per row; at the end of a document each group hands its
//               (max, argmax) per row to the reducer through shared memory,
//               packed into one ordered 64-bit key, and goes on with the
//               next document.
//   warp 18     reducer: merges the four groups' keys per row (an unsigned
//               max), sums each query's valid rows and writes the score and
//               argmax, while the epilogue and the MMA continue.  It shares
//               a sub-partition with four epilogue warps, so its instruction
//               count is on the kernel's critical path: the key merge and,
//               for 32-token queries, a butterfly sum per query keep it short.
//   warp 19     MMA issuer of the odd tiles (one issuing thread leaves the
//               tensor pipe idle while it checks barriers between chains)
// Lanes 1-31 of the producer warp zero-fill a buffer of the backward that
// follows on the stream, when there is one (the fp32 grad_D of a one-call
// training step), while the tensor cores keep the kernel busy and HBM is
// mostly idle.
// The accumulator is multi-buffered in TMEM (512 columns split into 2..4
// buffers, as many as the tile width allows), so the MMA runs ahead of the
// epilogue.
//
// Epilogue per 16-column unit: the document mask as warp-uniform bits (one
// ballot per two units, loaded a tile ahead) and one tcgen05.ld.red, which
// returns the unit's 16 values together with their maximum (an sm_103a
// load-with-reduction), so a fully valid unit costs no ALU work for its max.
// A unit with masked columns takes its max over the valid ones instead.
// When argmax is wanted, a unit whose max is strictly larger than the row's
// running max keeps its 16 values in registers; at the document's end the
// lowest column equal to the max is picked from them.  Exact ties therefore
// go to the lowest token index, as in the oracle.  The reducer sums the
// maxima of the valid query tokens per query in a fixed order.
//
// Synchronisation: every hand-off is an mbarrier.  The epilogue warps and the
// reducer count one arrival per warp (after __syncwarp) and poll their waits
// with short naps, so that they take no issue slots from the MMA issuers,
// the producer and the reducer that share their sub-partitions.  TMEM is
// freed after an exit mbarrier that every warp arrives at once.
//
// Every mbarrier wait is bounded (ptx::mbar_wait); on expiry the kernel sets
// the library's error word, drains its own TMA loads and MMAs, frees TMEM and
// returns.
#include <cfloat>

#include "lik_internal.h"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace lik {
namespace {

constexpr int kEpiWarps = 16;         // 4 warpgroups of 4 warps
constexpr int kEpiGroups = kEpiWarps / 4;
constexpr int kRedWarps = 1;          // document-end reducer (one warp: it synchronises with __syncwarp)
constexpr int kIssuers = 2;           // MMA issuing threads (warp 1 and the last warp)
constexpr int kThreads = 32 * (2 + kEpiWarps + kRedWarps + 1);
constexpr int kSlots = 1;             // documents in flight between the epilogue and the reducers
constexpr int kM = 128;              // accumulator rows (query tokens) per tile
constexpr int kAtomBytes = 128;      // one 128-byte swizzle row = 64 fp16/bf16
constexpr int kMaxDim = 256;        // largest embedding size the tensor-core paths take
constexpr int kAtomElems = 64;
constexpr int kMaxStages = 6;
constexpr int kMaxTileCols = 256;     // widest document tile (MMA N)
// 16-column units of a tile per warpgroup, rounded up to pairs (one TMEM round trip each)
constexpr int kUnitsPerGroup = 2 * ((kMaxTileCols / 16 + 2 * kEpiGroups - 1) / (2 * kEpiGroups));
constexpr int kTmemCols = 512;        // all of TMEM; split into p.nacc accumulator buffers
constexpr int kMaxAcc = 4;

struct Params {
    int64_t Nq, Nd, Lq, Ld;
    int dim, atoms, T, tiles_per_doc, qpt, n_rb, dpu, stages;
    int nacc, acc_stride;  // accumulator buffers in TMEM and their column stride
    int64_t n_units;
    uint32_t idesc, q_bytes, d_bytes;
    const uint8_t* qmask;
    const uint8_t* dmask;
    float* scores;
    int32_t* argmax;
    unsigned int* err;
    float4* zero;           // a buffer the kernel zero-fills on the side (nullptr: none)
    int64_t zero_n16;       // its size in 16-byte words
};

// Barrier slots in the misc region.
struct Bars {
    uint64_t full_d[kMaxStages], empty_d[kMaxStages];
    uint64_t full_q[2], empty_q[2];
    uint64_t acc_full[kMaxAcc], acc_empty[kMaxAcc];
    uint64_t xfull[kSlots];   // every epilogue warp has published a document's (max, argmax)
    uint64_t xfree[kSlots];   // the reducer has read them
    uint64_t mma_done;
    uint64_t exit_bar;   // every warp is done (one arrive per warp): TMEM may be released
    uint32_t tmem_base;
    uint32_t pad;
};

// What the epilogue hands to the reducers at a document's end, per slot.
struct Exchange {
    // each warpgroup's (max, column) per accumulator row as one ordered key:
    // the larger key has the larger max, or the same max and the lower column
    uint64_t key[kSlots][kEpiGroups][kM];
    int stage_seq[kMaxStages];            // tile (index in the CTA's sequence) each D stage holds
    float term[kSlots][kM];               // merged per-row terms, summed per query
};

// (max m, column a) -> key.  m's bits are mapped to an unsigned integer of
// the same order (-0 taken as +0, so that equal maxima stay equal), and the
// column is inverted so that the lower column wins a tie; column -1 (none)
// gives the smallest low word.
__device__ __forceinline__ uint64_t max_key(float m, int a) {
    const uint32_t u = __float_as_uint(m + 0.0f);
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<uint64_t>(ord) << 32) | (0xffffffffu - static_cast<uint32_t>(a));
}
__device__ __forceinline__ float key_max(uint64_t k) {
    const uint32_t ord = static_cast<uint32_t>(k >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
}
__device__ __forceinline__ int key_col(uint64_t k) {
    return static_cast<int>(0xffffffffu - static_cast<uint32_t>(k));
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Max of 16 values with 3-input max (8 instructions).
__device__ __forceinline__ float max16(const float (&v)[16]) {
    const float a = max3f(v[0], v[1], v[2]), b = max3f(v[3], v[4], v[5]), c = max3f(v[6], v[7], v[8]);
    const float d = max3f(v[9], v[10], v[11]), e = max3f(v[12], v[13], v[14]);
    return max3f(max3f(a, b, c), fmaxf(d, e), v[15]);
}

// Max over the valid columns of a 16-column unit whose validity bits `mw`
// are not all set; invalid columns are overwritten with -FLT_MAX in `raw`,
// so that the saved values of a unit never hold a masked maximum.
__device__ __forceinline__ float masked_max16(uint32_t (&raw)[16], uint32_t mw) {
    float v[16];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        raw[t] = ((mw >> t) & 1u) ? raw[t] : 0xff7fffffu;  // -FLT_MAX
        v[t] = __uint_as_float(raw[t]);
    }
    return max16(v);
}

// Folds one loaded 16-column unit (validity bits `mw`, load max `mred`,
// first column `col`) into the row's running max `m`.  With kArg a strictly
// larger unit max also keeps the unit's values and first column; the column
// of the max is resolved once, at the document's end.
template <bool kArg>
__device__ __forceinline__ void fold_unit(uint32_t (&raw)[16], uint32_t mw, float mred, int col, float& m,
                                          int& bcol, uint32_t (&best)[16]) {
    if (mw == 0) return;
    // the load's own max, unless some of the unit's columns are masked
    const float cb = mw == 0xffffu ? mred : masked_max16(raw, mw);
    if constexpr (kArg) {
        if (cb > m) {
            m = cb;
            bcol = col;
#pragma unroll
            for (int t = 0; t < 16; ++t) best[t] = raw[t];
        }
    } else {
        m = fmaxf(m, cb);
    }
}

// Lowest t with v[t] == m (m is one of the 16 values).
__device__ __forceinline__ int first_equal16(const uint32_t (&v)[16], float m) {
    int idx = 15;
#pragma unroll
    for (int t = 14; t >= 0; --t) idx = (__uint_as_float(v[t]) == m) ? t : idx;
    return idx;
}

// Position in a CTA's sequence of (work unit, document, tile).
struct Cursor {
    int64_t u, d, d1;
    int t;
    bool valid;
};

__device__ __forceinline__ Cursor unit_cursor(const Params& p, int64_t u) {
    Cursor c;
    c.u = u;
    c.t = 0;
    c.valid = u < p.n_units;
    c.d = (u / p.n_rb) * p.dpu;
    c.d1 = c.d + p.dpu < p.Nd ? c.d + p.dpu : p.Nd;
    return c;
}

__device__ __forceinline__ Cursor first_cursor(const Params& p) { return unit_cursor(p, blockIdx.x); }

__device__ __forceinline__ Cursor next_cursor(const Params& p, Cursor c) {
    if (!c.valid) return c;
    if (++c.t < p.tiles_per_doc) return c;
    c.t = 0;
    if (++c.d < c.d1) return c;
    return unit_cursor(p, c.u + gridDim.x);
}

// Mask bytes of this warpgroup's 16-column units of the cursor's tile.
// Step m covers units wg + 4*(2m) (lanes 0..15) and wg + 4*(2m+1) (lanes
// 16..31), one column per lane (colb[m], the same in every tile); 0 past the
// tile or the document.
__device__ __forceinline__ void prefetch_mask(const Params& p, const Cursor& c, const int (&colb)[kUnitsPerGroup / 2],
                                              uint8_t (&out)[kUnitsPerGroup / 2]) {
    const int jt = c.t * p.T;
    const uint8_t* dm = p.dmask ? p.dmask + c.d * p.Ld + jt : nullptr;
    const int rest = static_cast<int>(p.Ld) - jt;
    const int lim = c.valid ? (rest < p.T ? rest : p.T) : 0;
#pragma unroll
    for (int m = 0; m < kUnitsPerGroup / 2; ++m)
        out[m] = colb[m] < lim ? (dm ? dm[colb[m]] : uint8_t(1)) : uint8_t(0);
}

template <bool kArg>
__global__ void __launch_bounds__(kThreads, 1)
allpairs_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmd,
                       const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qbuf = smem;                                   // 2 x q_bytes
    uint8_t* dbuf = smem + 2 * p.q_bytes;                   // stages x d_bytes
    Bars* bars = reinterpret_cast<Bars*>(dbuf + p.stages * p.d_bytes);
    Exchange* xc = reinterpret_cast<Exchange*>(bars + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned int* err = p.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->full_d[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->empty_d[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bars->full_q[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->empty_q[b]), kIssuers);
        }
        for (int b = 0; b < kMaxAcc; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bars->acc_full[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->acc_empty[b]), kEpiWarps);
        }
        for (int b = 0; b < kSlots; ++b) {
            // one arrival per warp, after __syncwarp: a barrier word takes its
            // arrivals one at a time, and a document end is on the epilogue's path
            ptx::mbar_init(ptx::smem_u32(&bars->xfull[b]), kEpiWarps);
            ptx::mbar_init(ptx::smem_u32(&bars->xfree[b]), 1);
        }
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

    const int64_t Lq = p.Lq;

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        if (lane != 0) {
            // the side zero-fill: 16-byte stores, 31 lanes of every CTA over
            // the buffer, each warp instruction 496 contiguous bytes
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int64_t i = static_cast<int64_t>(blockIdx.x) * 31 + lane - 1; i < p.zero_n16;
                 i += static_cast<int64_t>(gridDim.x) * 31)
                p.zero[i] = z;
        } else {
            ptx::prefetch_tmap(&tmq);
            ptx::prefetch_tmap(&tmd);
            int s = 0, qb = 0;
            uint32_t ph = 0, qph = 0;
            uint32_t issued_d = 0, issued_q = 0;  // bit i: slot i holds an issued load
            uint32_t last_ph_d = 0, last_ph_q = 0;
            bool ok = true;
            // Q row block of unit uq into the next Q buffer, once the MMAs of
            // the unit that used it before have completed
            auto issue_q = [&](int64_t uq) -> bool {
                if (!ptx::mbar_wait(ptx::smem_u32(&bars->empty_q[qb]), qph ^ 1, err)) return false;
                const uint32_t fq = ptx::smem_u32(&bars->full_q[qb]);
                ptx::mbar_arrive_expect_tx(fq, p.q_bytes);
                const int64_t rbq = uq % p.n_rb;
                const int32_t row0 = static_cast<int32_t>(rbq * p.qpt * Lq);
                for (int a = 0; a < p.atoms; ++a)
                    ptx::tma_load_2d(ptx::smem_u32(qbuf + qb * p.q_bytes + a * kM * kAtomBytes), &tmq,
                                     a * kAtomElems, row0, fq);
                issued_q |= 1u << qb;
                last_ph_q = (last_ph_q & ~(1u << qb)) | (qph << qb);
                if (++qb == 2) { qb = 0; qph ^= 1; }
                return true;
            };
            int64_t u = blockIdx.x, kseq = 0;
            if (u < p.n_units) ok = issue_q(u);
            for (; ok && u < p.n_units; u += gridDim.x) {
                const int64_t d0 = (u / p.n_rb) * p.dpu;
                const int64_t d1 = d0 + p.dpu < p.Nd ? d0 + p.dpu : p.Nd;
                // the next unit's Q goes out after this unit's first two D tiles,
                // so its load overlaps this unit's MMAs
                const int64_t un = u + gridDim.x;
                bool q_next = un < p.n_units;
                const int64_t ntiles = (d1 - d0) * p.tiles_per_doc;
                const int64_t q_at = ntiles < 2 ? ntiles : 2;
                int64_t k = 0;
                for (int64_t d = d0; ok && d < d1; ++d) {
                    for (int t = 0; t < p.tiles_per_doc; ++t) {
                        if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->empty_d[s]), ph ^ 1, err))) break;
                        xc->stage_seq[s] = static_cast<int>(kseq++);  // published by the arrive below
                        const uint32_t fd = ptx::smem_u32(&bars->full_d[s]);
                        ptx::mbar_arrive_expect_tx(fd, p.d_bytes);
                        for (int a = 0; a < p.atoms; ++a)
                            ptx::tma_load_3d(ptx::smem_u32(dbuf + s * p.d_bytes + a * p.T * kAtomBytes),
                                             &tmd, a * kAtomElems, t * p.T, static_cast<int32_t>(d), fd);
                        issued_d |= 1u << s;
                        last_ph_d = (last_ph_d & ~(1u << s)) | (ph << s);
                        if (++s == p.stages) { s = 0; ph ^= 1; }
                        if (q_next && ++k == q_at) {
                            if (!(ok = issue_q(un))) break;
                            q_next = false;
                        }
                    }
                }
            }
            // every issued load must land before the CTA may exit
            for (int k = 0; k < p.stages; ++k)
                if (issued_d & (1u << k))
                    ptx::mbar_wait(ptx::smem_u32(&bars->full_d[k]), (last_ph_d >> k) & 1u, err);
            for (int k = 0; k < 2; ++k)
                if (issued_q & (1u << k))
                    ptx::mbar_wait(ptx::smem_u32(&bars->full_q[k]), (last_ph_q >> k) & 1u, err);
        }
    } else if (warp == 1 || warp == 3 + kEpiWarps) {
        // ----------------------------------------------------------- MMA --
        // Two issuing threads take alternate tiles.  Issuing a chain blocks
        // until the tensor pipe has room, so a single thread is only a few
        // MMAs ahead of the pipe, and its barrier checks between chains (a few
        // hundred cycles) would leave the pipe idle; with two threads one
        // thread's chain runs while the other checks its barriers.  Each thread
        // commits its own tiles; at the end of every unit both arrive on the
        // unit's Q buffer, and both on the final drain barrier.
        if (lane == 0) {
            const int who = warp == 1 ? 0 : 1;
            int s = 0, qb = 0, ab = 0;
            uint32_t ph = 0, qph = 0, aph = 0;
            bool ok = true;
            int64_t k = 0;  // tile index in this CTA's sequence
            for (int64_t u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
                const int64_t d0 = (u / p.n_rb) * p.dpu;
                const int64_t d1 = d0 + p.dpu < p.Nd ? d0 + p.dpu : p.Nd;
                if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->full_q[qb]), qph, err))) break;
                ptx::tc_fence_after();
                const uint32_t qaddr = ptx::smem_u32(qbuf + qb * p.q_bytes);
                for (int64_t d = d0; ok && d < d1; ++d) {
                    for (int t = 0; t < p.tiles_per_doc; ++t, ++k) {
                        if ((k & 1) == who) {
                            if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->full_d[s]), ph, err))) break;
                            // With an odd stage count the stage's previous phase belongs to the
                            // other issuer's tile; if that load is still in flight (loads may
                            // complete out of order), the parity wait above has passed on it.
                            // The stage then still names the earlier tile: wait for that phase,
                            // then for this one.
                            if (xc->stage_seq[s] != static_cast<int>(k)) {
                                if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->full_d[s]), ph ^ 1, err))) break;
                                if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->full_d[s]), ph, err))) break;
                            }
                            if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->acc_empty[ab]), aph ^ 1, err))) break;
                            ptx::tc_fence_after();
                            const uint32_t daddr = ptx::smem_u32(dbuf + s * p.d_bytes);
                            const uint32_t acc = tmem_base + ab * p.acc_stride;
                            if (p.dim == 128)  // the common embedding size: no per-step guards
                                ptx::mma_kchain<8>(acc, qaddr, kM * kAtomBytes, daddr, p.T * kAtomBytes, 8, p.idesc);
                            else
                                ptx::mma_kchain<kMaxDim / 16>(acc, qaddr, kM * kAtomBytes, daddr, p.T * kAtomBytes,
                                                              p.dim / 16, p.idesc);
                            ptx::mma_commit(ptx::smem_u32(&bars->empty_d[s]));
                            ptx::mma_commit(ptx::smem_u32(&bars->acc_full[ab]));
                        }
                        if (++s == p.stages) { s = 0; ph ^= 1; }
                        if (++ab == p.nacc) { ab = 0; aph ^= 1; }
                    }
                }
                ptx::mma_commit(ptx::smem_u32(&bars->empty_q[qb]));
                if (++qb == 2) { qb = 0; qph ^= 1; }
            }
            // all MMAs of both threads complete before TMEM is released
            ptx::mma_commit(ptx::smem_u32(&bars->mma_done));
            ptx::mbar_wait(ptx::smem_u32(&bars->mma_done), 0, err);
        }
    } else if (warp < 2 + kEpiWarps) {
        // ------------------------------------------------------ epilogue --
        const int ew = warp - 2;            // 0..kEpiWarps-1
        const int wg = ew >> 2;             // warpgroup: units u with u % kEpiGroups == wg
        const int quarter = warp & 3;       // TMEM lane quarter of this warp
        const int r = quarter * 32 + lane;  // accumulator row of this thread
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        int ab = 0, slot = 0;
        uint32_t aph = 0, xph = 0;
        bool ok = true;

        // Flat cursor over this CTA's (unit, document, tile) sequence, so the
        // document-mask bytes of the next tile can be loaded while the
        // current tile is processed.
        Cursor cur = first_cursor(p), nxt;
        uint8_t pre[kUnitsPerGroup / 2], pre_next[kUnitsPerGroup / 2];
        int colb[kUnitsPerGroup / 2];  // this lane's column in each mask step (the same in every tile)
#pragma unroll
        for (int m = 0; m < kUnitsPerGroup / 2; ++m) colb[m] = (wg + kEpiGroups * (2 * m + (lane >> 4))) * 16 + (lane & 15);
        prefetch_mask(p, cur, colb, pre);
        float m = -INFINITY;   // running max of this row over the warpgroup's units
        int bcol = -1;         // first column of the unit that holds m
        uint32_t best[16];     // that unit's values (masked columns as -FLT_MAX)
#pragma unroll
        for (int t = 0; t < 16; ++t) best[t] = 0;
        while (ok && cur.valid) {
            uint32_t mw[kUnitsPerGroup / 2];
#pragma unroll
            for (int k = 0; k < kUnitsPerGroup / 2; ++k) mw[k] = __ballot_sync(0xffffffffu, pre[k] != 0);
            nxt = next_cursor(p, cur);
            prefetch_mask(p, nxt, colb, pre_next);
            if (cur.t == 0) {
                m = -INFINITY;
                bcol = -1;
            }

            // the 16 epilogue warps poll with naps: the MMA issuers, the producer
            // and the reducer share their SM sub-partitions
            ok = ptx::mbar_wait_nap(ptx::smem_u32(&bars->acc_full[ab]), aph, err, 32);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t acc = tmem_base + ab * p.acc_stride + lane_off;
            const int jt = cur.t * p.T;
            // units wg + 4k, two per TMEM round trip; a unit past the tile width is
            // never read (its columns may lie past this buffer, or past TMEM)
#pragma unroll
            for (int k2 = 0; k2 < kUnitsPerGroup; k2 += 2) {
                const uint32_t w2 = mw[k2 >> 1];
                if (w2 == 0) continue;
                const int u0 = wg + kEpiGroups * k2, u1 = u0 + kEpiGroups;
                uint32_t ra[16], rb[16];
                float ma, mb;
                if (u1 * 16 < p.T) {
                    ptx::tmem_ldmax_16x2(acc + u0 * 16, acc + u1 * 16, ra, rb, ma, mb);
                } else {
                    // w2 != 0 implies u0 lies inside the tile
                    ptx::tmem_ldmax_16(acc + u0 * 16, ra, ma);
                    mb = -INFINITY;
#pragma unroll
                    for (int t = 0; t < 16; ++t) rb[t] = 0;
                }
                fold_unit<kArg>(ra, w2 & 0xffffu, ma, jt + u0 * 16, m, bcol, best);
                fold_unit<kArg>(rb, w2 >> 16, mb, jt + u1 * 16, m, bcol, best);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->acc_empty[ab]));
            if (++ab == p.nacc) { ab = 0; aph ^= 1; }

            if (cur.t == p.tiles_per_doc - 1) {
                // ---- document end: hand this warpgroup's (max, argmax) of each
                // row to the reducers and go on; the lowest column of the first
                // unit holding the max is the group's argmax
                int am = -1;
                if constexpr (kArg) {
                    if (bcol >= 0) am = bcol + first_equal16(best, m);
                }
                ok = ptx::mbar_wait_nap(ptx::smem_u32(&bars->xfree[slot]), xph ^ 1, err, 32);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                xc->key[slot][wg][r] = max_key(m, am);
                __syncwarp();  // the warp's writes precede lane 0's arrive (release)
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->xfull[slot]));
                if (++slot == kSlots) { slot = 0; xph ^= 1; }
            }
            cur = nxt;
#pragma unroll
            for (int k = 0; k < kUnitsPerGroup / 2; ++k) pre[k] = pre_next[k];
        }
    } else {
        // ------------------------------------------------------ reducers --
        // Per document: merge the warpgroups' (max, argmax) per row (strictly
        // greater wins, equal maxima keep the lower column: the larger key),
        // sum the valid query tokens' maxima per query in a fixed order,
        // write score and argmax.  A thread owns rows rr + 32 * kRedWarps * k.
        static_assert(kRedWarps == 1, "the reducer synchronises its lanes with __syncwarp");
        constexpr int kRows = kM / (32 * kRedWarps);
        const int rr = (warp - 2 - kEpiWarps) * 32 + lane;  // the reducer warp(s) follow the epilogue
        const int64_t qrows = static_cast<int64_t>(p.qpt) * Lq;
        int slot = 0;
        uint32_t xph = 0;
        bool ok = true;
        // position of each owned row inside its query (the same in every unit)
        int qloc[kRows], iq[kRows];
#pragma unroll
        for (int k = 0; k < kRows; ++k) {
            const int r = rr + k * 32 * kRedWarps;
            qloc[k] = static_cast<int>(r / Lq);
            iq[k] = static_cast<int>(r - static_cast<int64_t>(qloc[k]) * Lq);
        }
        // query-mask bytes of a unit's rows (0 for rows past the last query);
        // the next unit's are loaded one unit ahead, off the document-end path
        auto load_qvalid = [&](int64_t uu, uint8_t (&out)[kRows]) {
            const int64_t rbq = uu % p.n_rb;
#pragma unroll
            for (int k = 0; k < kRows; ++k) {
                const int r = rr + k * 32 * kRedWarps;
                const int64_t qq = rbq * p.qpt + qloc[k];
                const bool in = r < qrows && qq < p.Nq;
                out[k] = in ? (p.qmask ? p.qmask[qq * Lq + iq[k]] : uint8_t(1)) : uint8_t(0);
            }
        };
        uint8_t qv_cur[kRows], qv_next[kRows];
        if (blockIdx.x < p.n_units) load_qvalid(blockIdx.x, qv_cur);
        for (int64_t u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
            if (u + gridDim.x < p.n_units) load_qvalid(u + gridDim.x, qv_next);
            const int rb = static_cast<int>(u % p.n_rb);
            const int64_t d0 = (u / p.n_rb) * p.dpu;
            const int64_t d1 = d0 + p.dpu < p.Nd ? d0 + p.dpu : p.Nd;
            int64_t q[kRows];
            bool row_ok[kRows], qvalid[kRows];
#pragma unroll
            for (int k = 0; k < kRows; ++k) {
                const int r = rr + k * 32 * kRedWarps;
                q[k] = static_cast<int64_t>(rb) * p.qpt + qloc[k];
                row_ok[k] = r < qrows && q[k] < p.Nq;
                qvalid[k] = qv_cur[k] != 0;
            }
            for (int64_t d = d0; ok && d < d1; ++d) {
                // a document takes several tiles: nap between polls, the reducer
                // shares its sub-partition with four epilogue warps
                ok = ptx::mbar_wait_nap(ptx::smem_u32(&bars->xfull[slot]), xph, err, 128);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                int am[kRows];
                float term[kRows];
                bool any_doc = false;
#pragma unroll
                for (int k = 0; k < kRows; ++k) {
                    const int r = rr + k * 32 * kRedWarps;
                    uint64_t kk = xc->key[slot][0][r];
#pragma unroll
                    for (int g = 1; g < kEpiGroups; ++g) {
                        const uint64_t k1 = xc->key[slot][g][r];
                        kk = k1 > kk ? k1 : kk;
                    }
                    const float mm = key_max(kk);
                    const int aa = key_col(kk);
                    // a row's max is finite exactly when the document has a valid
                    // column (the same for every row: validity is per column)
                    const bool an = mm != -INFINITY;
                    any_doc = an;
                    term[k] = (an && qvalid[k]) ? mm : 0.0f;
                    if (Lq != 32) xc->term[slot][r] = term[k];
                    am[k] = (an && qvalid[k]) ? aa : -1;
                }
                // the warp's reads of the slot and its term writes are complete:
                // release the slot, and make the terms visible to the summing lanes
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->xfree[slot]));
                if (Lq == 32) {
                    // row lane + 32k is token `lane` of the unit's query k: one
                    // butterfly per query, every lane ending with the sums
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                        for (int k = 0; k < kRows; ++k) term[k] += __shfl_xor_sync(0xffffffffu, term[k], off);
#pragma unroll
                    for (int k = 0; k < kRows; ++k) {
                        if (!row_ok[k]) continue;
                        const int64_t pair = q[k] * p.Nd + d;
                        if (lane == k && p.scores) p.scores[pair] = any_doc ? term[k] : kEmptyDocScore;
                        if (p.argmax) p.argmax[pair * Lq + lane] = am[k];
                    }
                    if (++slot == kSlots) { slot = 0; xph ^= 1; }
                    continue;
                }
#pragma unroll
                for (int k = 0; k < kRows; ++k) {
                    if (!row_ok[k]) continue;
                    const int r = rr + k * 32 * kRedWarps;
                    const int64_t pair = q[k] * p.Nd + d;
                    if (iq[k] == 0) {
                        // the query's rows r .. r + Lq - 1, four interleaved partial sums
                        const float* t = xc->term[slot] + r;
                        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
                        int64_t k4 = 0;
                        for (; k4 + 4 <= Lq; k4 += 4) {
                            s0 += t[k4];
                            s1 += t[k4 + 1];
                            s2 += t[k4 + 2];
                            s3 += t[k4 + 3];
                        }
                        for (; k4 < Lq; ++k4) s0 += t[k4];
                        if (p.scores) p.scores[pair] = any_doc ? (s0 + s1) + (s2 + s3) : kEmptyDocScore;
                    }
                    if (p.argmax) p.argmax[pair * Lq + iq[k]] = am[k];
                }
                if (++slot == kSlots) { slot = 0; xph ^= 1; }
            }
#pragma unroll
            for (int k = 0; k < kRows; ++k) qv_cur[k] = qv_next[k];
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
    if (warp <= 1 || warp == 3 + kEpiWarps) {
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

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Tiles of the busiest CTA when the n_rb x ceil(Nd/dpu) work units (unit u:
// row block u % n_rb, documents [dpu*(u/n_rb), +dpu)) are dealt round-robin
// to min(units, sms) persistent CTAs.  Only the last chunk of documents
// can be short.
int64_t busiest_tiles(int64_t n_rb, int64_t Nd, int64_t dpu, int64_t tiles, int64_t sms) {
    const int64_t chunks = (Nd + dpu - 1) / dpu, n = n_rb * chunks;
    const int64_t grid = n < sms ? n : sms;
    const int64_t short_by = (chunks * dpu - Nd) * tiles;  // missing tiles of a last-chunk unit
    const int64_t lo = n - n_rb;                           // first unit of the last chunk
    int64_t most = 0;
    for (int64_t b = 0; b < grid; ++b) {
        const int64_t cnt = (n - 1 - b) / grid + 1;
        const int64_t f = b >= lo ? b : b + ((lo - b + grid - 1) / grid) * grid;
        const int64_t n_short = f < n ? (n - 1 - f) / grid + 1 : 0;
        const int64_t load = cnt * dpu * tiles - n_short * short_by;
        most = load > most ? load : most;
    }
    return most;
}

// Documents per work unit.  A unit costs one Q row-block load and a short
// pipeline refill (about a quarter of a tile, measured), so units are kept
// long (up to ~24 tiles) unless shorter ones even out the CTAs' loads.
int choose_docs_per_unit(int64_t n_rb, int64_t Nd, int tiles, int sms) {
    const int dmax = ceil_div(24, tiles);
    int best = dmax;
    double best_cost = 0.0;
    for (int dpu = dmax; dpu >= 1; --dpu) {
        const int64_t chunks = (Nd + dpu - 1) / dpu, n = n_rb * chunks;
        const int64_t grid = n < sms ? n : sms;
        const double units_busiest = static_cast<double>((n + grid - 1) / grid);
        const double cost = static_cast<double>(busiest_tiles(n_rb, Nd, dpu, tiles, sms)) + 0.25 * units_busiest;
        if (dpu == dmax || cost < best_cost) {
            best = dpu;
            best_cost = cost;
        }
    }
    return best;
}

}  // namespace

bool tc_allpairs_eligible(const Problem& P) {
    return P.layout == kAllPairs && (P.dtype == kF16 || P.dtype == kBF16) && P.dim % 16 == 0 &&
           P.dim <= kMaxDim && P.Lq >= 1 && P.Lq <= kM && P.Ld >= 1 && P.n_query * P.Lq < (int64_t(1) << 31) &&
           P.Ld < (int64_t(1) << 31) && P.n_doc < (int64_t(1) << 31);
}

cudaError_t launch_fwd_tc_allpairs(const Problem& P, float* scores, int32_t* argmax, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const DeviceInfo& info = device_info(dev);

    Params p{};
    p.Nq = P.n_query;
    p.Nd = P.n_doc;
    p.Lq = P.Lq;
    p.Ld = P.Ld;
    p.dim = static_cast<int>(P.dim);
    p.atoms = (p.dim + kAtomElems - 1) / kAtomElems;
    p.q_bytes = static_cast<uint32_t>(p.atoms * kM * kAtomBytes);
    const size_t misc = sizeof(Bars) + sizeof(Exchange);
    const size_t budget = static_cast<size_t>(info.max_smem_optin) - 1024 - misc - 2 * p.q_bytes;
    // widest tile (<= 256 tokens) that leaves room for two D stages
    int tmax = kMaxTileCols;
    while (tmax > 16 && budget / (static_cast<size_t>(p.atoms) * tmax * kAtomBytes) < 2) tmax -= 16;
    p.tiles_per_doc = ceil_div(P.Ld, tmax);
    p.T = ((ceil_div(P.Ld, p.tiles_per_doc) + 15) / 16) * 16;
    // as many accumulator buffers as TMEM holds at a 32-column-aligned stride
    p.acc_stride = ((p.T + 31) / 32) * 32;
    p.nacc = kTmemCols / p.acc_stride;
    if (p.nacc > kMaxAcc) p.nacc = kMaxAcc;
    p.acc_stride = (kTmemCols / p.nacc) / 32 * 32;
    p.qpt = static_cast<int>(kM / P.Lq);
    p.n_rb = ceil_div(P.n_query, p.qpt);
    p.d_bytes = static_cast<uint32_t>(p.atoms * p.T * kAtomBytes);
    p.stages = static_cast<int>(budget / p.d_bytes);
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (p.stages < 2) return cudaErrorInvalidConfiguration;
    p.dpu = choose_docs_per_unit(p.n_rb, P.n_doc, p.tiles_per_doc, info.sm_count);
    p.n_units = static_cast<int64_t>(p.n_rb) * ceil_div(P.n_doc, p.dpu);
    p.idesc = ptx::f16_idesc(kM, p.T, P.dtype == kBF16);
    p.qmask = P.qmask;
    p.dmask = P.dmask;
    p.scores = scores;
    p.argmax = argmax;
    p.err = device_error_word();
    p.zero = static_cast<float4*>(P.fwd_zero);
    p.zero_n16 = P.fwd_zero ? P.fwd_zero_bytes / 16 : 0;

    CUtensorMap tmq, tmd;
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(P.dim), static_cast<uint64_t>(P.n_query * P.Lq)};
        const uint64_t strides[1] = {static_cast<uint64_t>(P.dim) * 2};
        const uint32_t box[2] = {kAtomElems, kM};
        if (!encode_tmap_kmajor(&tmq, P.dtype, P.Q, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(P.dim), static_cast<uint64_t>(P.Ld),
                                  static_cast<uint64_t>(P.n_doc)};
        const uint64_t strides[2] = {static_cast<uint64_t>(P.dim) * 2, static_cast<uint64_t>(P.Ld * P.dim) * 2};
        const uint32_t box[3] = {kAtomElems, static_cast<uint32_t>(p.T), 1};
        if (!encode_tmap_kmajor(&tmd, P.dtype, P.D, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }

    const size_t smem = 1024 + 2 * static_cast<size_t>(p.q_bytes) +
                        static_cast<size_t>(p.stages) * p.d_bytes + misc;
    // the max-only variant (no argmax requested: inference) skips the index work
    auto kernel = argmax ? allpairs_fwd_tc_kernel<true> : allpairs_fwd_tc_kernel<false>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int64_t grid = p.n_units < info.sm_count ? p.n_units : info.sm_count;
    kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(tmq, tmd, p);
    return cudaGetLastError();
}

}  // namespace lik
