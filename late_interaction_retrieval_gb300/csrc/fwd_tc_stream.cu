// fwd_tc_stream.cu -- pairwise and per-query-candidate (kd) MaxSim forward on
// the sm_103a tensor cores, streaming every document once from HBM.
//
// What it computes (Late Interaction Kernels README, "What does it compute?"
// and "Scoring interface"; per-query candidates: colpali PR "Add support for
// late-interaction-kernels (LIK)", Design section): for every pair p of
// query q(p) and document d(p),
//   score[p] = sum over valid i of max over valid j of Q[q,i].D[d,j]
// with the lowest j reaching each max saved as argmax, -1e9 for a document
// with no valid token.
//
// Each document is read once, so the work per byte of D is 2*Lq FLOP: the
// kernel is bound by HBM bandwidth, not by the tensor cores.  It still uses
// them: with CUDA-core FMA the Lq*dim multiply-adds per document token
// (4096 at Lq=32, dim=128) would cost more issue slots than streaming the
// token's 256 bytes takes at full bandwidth.
//
// Tiling.  A tile is 128 consecutive tokens of one document (TMA box of a
// 3D map [n_doc, Ld, dim]; tokens past Ld read as zero).  The MMA puts the
// document tokens on the M side and the query's tokens on the N side:
//     S[128, 32] = Dtile[128, dim] . Qb[32, dim]^T    (fp32 in TMEM)
// with the query's Lq <= 32 tokens in the first Lq columns (the rest are
// ignored).  So each accumulator lane is one document token and each column
// one query token.
//
// Schedule.  A document's work is its tiles up to the last one holding a
// valid token (at least one, so an empty document still gets its -1e9); a
// small plan kernel finds that count per pair from the mask.  The CTAs split
// the concatenated tile sequence of all pairs into equal contiguous ranges,
// so a long document may be cut between CTAs.  Each piece of a cut document
// leaves its per-query-token (max, argmax) in a workspace; the piece that
// arrives last (a counter per cut document) merges them in piece order,
// i.e. in token order, and writes the score and argmax.  The merged result
// is the one a single CTA would produce: maxima are exact, ties go to the
// lowest token index, and the sum over query tokens keeps its fixed order.
//
// Roles (one CTA per SM, persistent over its range of tiles; 224 threads):
//   warp 0      producer.  Finds the CTA's range (a search over the plan's
//               per-group sums).  Each lane loads the plan's row-validity
//               words of one tile of the window 8 tiles ahead; tiles with no
//               valid token are skipped (never loaded).  Lane 0 alone then
//               issues the window's TMA loads (a query's rows into one of two
//               buffers when the query changes, document tiles per stage) and
//               publishes, through a ring of tile records, the sequence the
//               epilogue follows: data tiles, one end record per document
//               piece, and an end-of-stream record.
//   warp 1      TMEM allocator + single-thread MMA issuer (4 accumulators).
//   warps 2-5   update warps.  Each thread owns one accumulator lane
//               (document token) and keeps a running (max, argmax) for each
//               of the 32 query tokens in registers across the piece's tiles.
//               At the end of a piece each warp reduces its 32 lanes with a
//               transposing butterfly (lane i ends with query token i) and
//               leaves 32 (max, argmax) pairs in a double-buffered dump, so
//               the dumps take 2 KB and the D stages get the shared memory.
//   warp 6      reducer.  Merges the four warps' partials per query token
//               (lowest token index on ties), sums the valid query tokens in
//               a fixed order and writes the score and argmax, or, for a
//               piece of a cut document, hands its partial to the merge.
// Every mbarrier wait is bounded; on expiry the kernel flags the library's
// error word, drains its own loads and MMAs, frees TMEM and returns.
#include <cfloat>
#include <cstdint>
#include <mutex>
#include <vector>

#include "lik_internal.h"
#include "sm100_ptx.cuh"
#include "tmap.h"

namespace lik {
namespace {

constexpr int kRows = 128;          // document tokens per tile (MMA M)
constexpr int kAtomBytes = 128;     // one 128-byte swizzle row = 64 fp16/bf16
constexpr int kMaxDim = 256;       // largest embedding size the tensor-core paths take
constexpr int kAtomElems = 64;
constexpr int kMaxStages = 8;
constexpr int kAccBufs = 4;
constexpr int kRing = 16;           // tile records in flight
constexpr int kWin = 8;             // tiles whose mask bytes the producer loads together
constexpr int kMaxLq = 32;          // query tokens: one per lane of the update and reducer warps

enum : int { kRecTile = 0, kRecDocEnd = 1, kRecStop = 2 };

struct Rec {
    int kind;
    int jt;                 // first document token of the tile
    int64_t pair;           // pair index (doc end) / unused
    uint32_t valid[4];      // row-validity bits of the tile (tile records)
    int nonempty;           // doc end: this piece of the document had a valid token
    int c_first, c_last;    // doc end: CTAs holding the document's first and last tile
    int first_tail;         // doc end: the document starts inside c_first's range (not at its start)
};

// Position of one tile in a CTA's range: the pair, the pair's first unit in
// the concatenated sequence, the tile's index within the pair, the pair's
// tile count.
struct Pos {
    int64_t pair;
    int64_t u_start;
    int t;
    int w;
};

struct StageMeta {
    int qb;                 // query buffer the tile multiplies
    int new_query;          // first tile with freshly loaded query rows: wait for them
    int stop;               // end of stream
    int pad;
};

struct Params {
    int64_t n_pairs, pairs_per_query, n_doc, Lq, Ld;
    int64_t tiles;          // 128-token tiles of a padded document
    int64_t n_groups;       // entries of group_units
    int layout, dim, atoms, np, stages, acc_cols;
    uint32_t idesc, q_bytes, d_bytes;
    const uint8_t* qmask;
    const uint8_t* dmask;
    float* scores;
    int32_t* argmax;
    unsigned int* err;
    // schedule and merge workspace (written by the plan kernel on the same stream)
    const int32_t* units;        // [n_pairs] tiles to visit per pair, or nullptr: all tiles
    const int32_t* group_units;  // [n_groups] sums of units over 32 consecutive pairs
    const uint4* words;          // [n_pairs * tiles] row-validity bits per tile, or nullptr: rows < Ld
    float* part_m;               // [2*grid][32] per-piece maxima of cut documents
    int32_t* part_a;             // [2*grid][32] per-piece argmax
    int32_t* part_ne;            // [2*grid] piece had a valid token
    unsigned int* arrivals;      // [grid] pieces arrived, per cut document (by its first CTA)
};

struct Bars {
    uint64_t full_d[kMaxStages], empty_d[kMaxStages];
    uint64_t full_q[2], empty_q[2];
    uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
    uint64_t rec_full[kRing], rec_empty[kRing];
    uint64_t dump_full[2], dump_empty[2];  // update warps -> reducer warp
    uint64_t mma_done;
    uint64_t exit_bar;   // every warp is done (one arrive per warp): TMEM may be released
    uint32_t tmem_base;
    uint32_t pad[3];     // Shared follows at a 16-byte boundary
};

// Per-document state handed from the update warps to the reducer warp
// (double-buffered): each update warp's (max, argmax) per query token over
// its 32 rows, already reduced across the warp's lanes.
struct Dump {
    float m[4][32];
    int a[4][32];
};

struct DumpInfo {
    int64_t pair;
    int nonempty;
    int stop;
    int c_first, c_last, first_tail;
    int pad;
};

static_assert(sizeof(Bars) % 16 == 0, "Shared follows Bars and holds 16-byte words");

struct alignas(16) Shared {
    uint4 win[kWin];         // producer: row-validity words of the current window
    Pos pos[kWin];           // producer: position of each tile of the current window
    Rec rec[kRing];
    StageMeta meta[kMaxStages];
    DumpInfo info[2];
    Dump dump[2];
};

__device__ __forceinline__ int64_t doc_of(const Params& p, int64_t pair) {
    return pair;  // pairwise: document b; kd: document b*N + n
}

__device__ __forceinline__ int64_t query_of(const Params& p, int64_t pair) {
    return pair / p.pairs_per_query;
}

// Index of the last nonzero byte of row[0, n), or -1 (one warp, every lane
// gets the result).  The bytes after the last 16-byte boundary, the last 128
// 16-byte words (four per lane) and the bytes before the first boundary are
// loaded together, then looked at from the end; further words (rows longer
// than 2 KB with a long invalid tail) 128 at a time.  Every access lies in
// row[0, n); n < 2^31 (the streaming kernels' limit on Ld), so offsets are
// 32-bit.
__device__ int last_nonzero_byte(const uint8_t* row, int n, int lane) {
    int head = static_cast<int>((16 - (reinterpret_cast<uintptr_t>(row) & 15)) & 15);
    if (head > n) head = n;
    const int words = (n - head) / 16;
    const int tail0 = head + 16 * words;
    const uint4* wv = reinterpret_cast<const uint4*>(row + head);
    auto load_words = [&](int top, uint4 (&v)[4], int (&wi)[4]) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            wi[k] = top - 1 - lane - 32 * k;
            v[k] = wi[k] >= 0 ? wv[wi[k]] : make_uint4(0, 0, 0, 0);
        }
    };
    auto last_in_words = [&](const uint4 (&v)[4], const int (&wi)[4]) {
        int best = -1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t x[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int e = 3; e >= 0; --e) {
                if (x[e] != 0) {
                    const int at = head + 16 * wi[k] + 4 * e + ((31 - __clz(static_cast<int>(x[e]))) >> 3);
                    best = at > best ? at : best;
                    break;
                }
            }
        }
        return __reduce_max_sync(0xffffffffu, best);
    };
    const uint8_t tb = tail0 + lane < n ? row[tail0 + lane] : uint8_t(0);
    const uint8_t hb = lane < head ? row[lane] : uint8_t(0);
    uint4 v[4];
    int wi[4];
    load_words(words, v, wi);
    int best = __reduce_max_sync(0xffffffffu, tb != 0 ? tail0 + lane : -1);
    if (best >= 0) return best;
    for (int top = words; top > 0; top -= 128) {
        if (top != words) load_words(top, v, wi);
        best = last_in_words(v, wi);
        if (best >= 0) return best;
    }
    return __reduce_max_sync(0xffffffffu, hb != 0 ? lane : -1);
}

// Plan kernel, two kinds of blocks of 1024 threads (with a document mask):
//  * blocks [0, n_groups): one warp per pair, 32 pairs per block:
//    units[p] = 1 + index of the last 128-token tile of pair p's document
//    that holds a valid token (1 for a document with none), and
//    group_units[b] = the sum over the block's pairs;
//  * the blocks after them: one warp per 8 consecutive tiles of all pairs'
//    padded tiles: words[t] = the tile's row-validity bits (bit l of word j
//    = row 32j + l), so the forward never reads mask bytes itself.
// Every block also zeroes its share of the forward's arrival counters.
struct PlanArgs {
    const uint8_t* dmask;
    int64_t n_pairs, Ld, tiles, n_groups;
    int32_t* units;
    int32_t* group_units;
    uint4* words;
    unsigned int* arrivals;
    int64_t n_arrivals;
};

__global__ void __launch_bounds__(1024) stream_plan_kernel(const PlanArgs a) {
    __shared__ int32_t per_warp[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the forward may be scheduled now: it waits for this grid before reading its output
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t z = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (z < a.n_arrivals) a.arrivals[z] = 0u;
    if (a.dmask == nullptr) return;
    if (blockIdx.x < a.n_groups) {
        const int64_t pair = static_cast<int64_t>(blockIdx.x) * 32 + warp;
        int32_t u = 0;
        if (pair < a.n_pairs) {
            const int last = last_nonzero_byte(a.dmask + pair * a.Ld, static_cast<int>(a.Ld), lane);
            u = last < 0 ? 1 : static_cast<int32_t>(last / kRows) + 1;
            if (lane == 0) a.units[pair] = u;
        }
        if (lane == 0) per_warp[warp] = u;
        __syncthreads();
        if (warp == 0) {
            int32_t s = lane < (blockDim.x >> 5) ? per_warp[lane] : 0;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (lane == 0) a.group_units[blockIdx.x] = s;
        }
        return;
    }
    const int64_t total = a.n_pairs * a.tiles;
    const int64_t t0 = ((static_cast<int64_t>(blockIdx.x) - a.n_groups) * 32 + warp) * 8;
    if (t0 >= total) return;
    // one row pointer per document and 32-bit offsets within it (Ld < 2^31)
    const int64_t pair = t0 / a.tiles;
    int tt = static_cast<int>(t0 - pair * a.tiles);
    const int ld = static_cast<int>(a.Ld), tiles = static_cast<int>(a.tiles);
    const int n_in = total - t0 < 8 ? static_cast<int>(total - t0) : 8;
    const uint8_t* row = a.dmask + pair * a.Ld;
    uint8_t b[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int j = tt * kRows + 32 * k + lane;
            b[i][k] = i < n_in && j < ld ? row[j] : uint8_t(0);
        }
        if (++tt == tiles) {
            tt = 0;
            row += a.Ld;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = __ballot_sync(0xffffffffu, b[i][k] != 0);
        if (lane == i && i < n_in) a.words[t0 + i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// This CTA's range of units [u0, u1), the pair p0 holding u0 and that pair's
// first unit (one warp; every lane gets the results).  The units are spread
// over ctas = min(grid, U) CTAs so that every working CTA has at least one
// (the merge of a cut document counts one arrival per CTA of its span).
struct Range {
    int64_t U, ctas, u0, u1, p0, p0_start;
    int64_t cache_base;  // lane l: units of pair cache_base + l (cache_val), when searched
    int32_t cache_val;
};

__device__ Range find_range(const Params& p, int lane) {
    Range r{};
    r.cache_base = -64;
    const int64_t c = blockIdx.x;
    constexpr int kPer = 8;  // group sums per lane per pass, all loads in flight together
    int32_t v[kPer];
    auto load = [&](int64_t base) {
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int64_t i = base + static_cast<int64_t>(lane) * kPer + k;
            v[k] = i < p.n_groups ? p.group_units[i] : 0;
        }
    };
    if (p.units == nullptr) {
        r.U = p.n_pairs * p.tiles;
    } else {
        int64_t s = 0;
        for (int64_t base = 0; base < p.n_groups; base += 32 * kPer) {
            load(base);
#pragma unroll
            for (int k = 0; k < kPer; ++k) s += v[k];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        r.U = s;
    }
    r.ctas = r.U < gridDim.x ? r.U : static_cast<int64_t>(gridDim.x);
    r.u0 = c < r.ctas ? c * r.U / r.ctas : r.U;
    r.u1 = c < r.ctas ? (c + 1) * r.U / r.ctas : r.U;
    if (r.u0 >= r.u1) return r;
    if (p.units == nullptr) {
        r.p0 = r.u0 / p.tiles;
        r.p0_start = r.p0 * p.tiles;
        return r;
    }
    // the group of 32 pairs holding u0: lane l scans groups [base + 8l, base + 8l + 8)
    int64_t grp = 0, grp_start = 0, carry = 0;
    for (int64_t base = 0; base < p.n_groups; base += 32 * kPer) {
        if (base > 0 || p.n_groups > 32 * kPer) load(base);  // one pass: v still holds it
        int64_t ls = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) ls += v[k];
        int64_t incl = ls;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t t = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += t;
        }
        int64_t at = carry + incl - ls;  // first unit of this lane's first group
        int hit = -1;
        int64_t hit_start = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            if (hit < 0 && v[k] > 0 && at <= r.u0 && r.u0 < at + v[k]) {
                hit = k;
                hit_start = at;
            }
            at += v[k];
        }
        const unsigned int found = __ballot_sync(0xffffffffu, hit >= 0);
        if (found) {
            const int src = __ffs(found) - 1;
            grp = base + static_cast<int64_t>(src) * kPer + __shfl_sync(0xffffffffu, hit, src);
            grp_start = __shfl_sync(0xffffffffu, hit_start, src);
            break;
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    // the pair within the group (every pair has at least one unit)
    const int64_t pair = grp * 32 + lane;
    const int64_t w = pair < p.n_pairs ? p.units[pair] : 0;
    int64_t incl = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    const int64_t ex = grp_start + incl - w;
    const unsigned int hit = __ballot_sync(0xffffffffu, w > 0 && ex <= r.u0 && r.u0 < ex + w);
    const int src = hit ? __ffs(hit) - 1 : 0;
    r.p0 = __shfl_sync(0xffffffffu, pair, src);
    r.p0_start = __shfl_sync(0xffffffffu, ex, src);
    r.cache_base = grp * 32;
    r.cache_val = static_cast<int32_t>(w);
    return r;
}

// CTA whose range holds unit u: the largest c with floor(c*U/G) <= u.
__device__ __forceinline__ int64_t cta_of_unit(int64_t u, int64_t U, int64_t G) {
    const int64_t c = ((u + 1) * G + U - 1) / U - 1;
    return c < G - 1 ? c : G - 1;
}

// One step of the warp's transposing max-reduction: m/a hold 2*kHalf query
// tokens per lane; afterwards the first kHalf entries hold the half this lane
// keeps (upper half if lane bit kHalf is set), merged with lane ^ kHalf's
// rows.  After the steps 16, 8, 4, 2, 1, lane l holds query token l over all
// 32 rows of the warp.  Ties go to the lower token index.
template <int kHalf>
__device__ __forceinline__ void fold_half(float (&m)[32], int (&a)[32], int lane) {
    const bool upper = (lane & kHalf) != 0;
#pragma unroll
    for (int c = 0; c < kHalf; ++c) {
        const float keep_v = upper ? m[c + kHalf] : m[c];
        const int keep_a = upper ? a[c + kHalf] : a[c];
        const float give_v = upper ? m[c] : m[c + kHalf];
        const int give_a = upper ? a[c] : a[c + kHalf];
        const float ov = __shfl_xor_sync(0xffffffffu, give_v, kHalf);
        const int oa = __shfl_xor_sync(0xffffffffu, give_a, kHalf);
        const bool take = ov > keep_v || (ov == keep_v && oa < keep_a);
        m[c] = take ? ov : keep_v;
        a[c] = take ? oa : keep_a;
    }
}

constexpr int kThreads = 32 * (2 + 4 + 1);  // producer, MMA, 4 update warps, reducer

__global__ void __launch_bounds__(kThreads, 1)
stream_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmd,
                     const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qbuf = smem;                          // 2 x q_bytes
    uint8_t* dbuf = smem + 2 * p.q_bytes;          // stages x d_bytes
    Bars* bars = reinterpret_cast<Bars*>(dbuf + p.stages * p.d_bytes);
    Shared* sh = reinterpret_cast<Shared*>(bars + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned int* err = p.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->full_d[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->empty_d[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bars->full_q[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->empty_q[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->dump_full[b]), 4);   // one arrive per update warp
            ptx::mbar_init(ptx::smem_u32(&bars->dump_empty[b]), 1);  // the reducer warp
        }
        for (int b = 0; b < kAccBufs; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bars->acc_full[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->acc_empty[b]), 4);
        }
        for (int r = 0; r < kRing; ++r) {
            ptx::mbar_init(ptx::smem_u32(&bars->rec_full[r]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->rec_empty[r]), 4);
        }
        ptx::mbar_init(ptx::smem_u32(&bars->mma_done), 1);
        ptx::mbar_init(ptx::smem_u32(&bars->exit_bar), kThreads / 32);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), p.acc_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    // launched as a programmatic dependent of the plan kernel: everything above
    // overlaps it; its output (and everything before it) is visible after this
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        // All lanes find the range and load the validity words of a window
        // of kWin tiles ahead; lane 0 alone publishes the window's tiles, so
        // a tile costs no warp-wide step.
        int s = 0, qb = 0, ri = 0;
        uint32_t ph = 0, qph = 0, rph = 0;
        uint32_t issued_d = 0, issued_q = 0, last_ph_d = 0, last_ph_q = 0;
        bool ok = true;
        // publish one record (lane 0), waiting for its ring slot
        auto publish = [&](const Rec& rec) -> bool {
            if (!ptx::mbar_wait(ptx::smem_u32(&bars->rec_empty[ri]), rph ^ 1, err)) return false;
            sh->rec[ri] = rec;
            ptx::mbar_arrive(ptx::smem_u32(&bars->rec_full[ri]));
            if (++ri == kRing) { ri = 0; rph ^= 1; }
            return true;
        };
        // hand one stage to the MMA (lane 0); data=false sends only metadata
        auto stage = [&](const StageMeta& meta, bool data, int64_t d, int64_t jt) -> bool {
            if (!ptx::mbar_wait(ptx::smem_u32(&bars->empty_d[s]), ph ^ 1, err)) return false;
            sh->meta[s] = meta;
            const uint32_t fd = ptx::smem_u32(&bars->full_d[s]);
            if (data) {
                ptx::mbar_arrive_expect_tx(fd, p.d_bytes);
                for (int a = 0; a < p.atoms; ++a)
                    ptx::tma_load_3d(ptx::smem_u32(dbuf + s * p.d_bytes + a * kRows * kAtomBytes), &tmd,
                                     a * kAtomElems, static_cast<int32_t>(jt), static_cast<int32_t>(d), fd);
                issued_d |= 1u << s;
                last_ph_d = (last_ph_d & ~(1u << s)) | (ph << s);
            } else {
                // the load this stage held before was consumed (its empty phase
                // completed above); forget it, or the drain below would wait on a
                // phase parity this arrive has moved past
                issued_d &= ~(1u << s);
                ptx::mbar_arrive(fd);
            }
            if (++s == p.stages) { s = 0; ph ^= 1; }
            return true;
        };

        const Range rg = find_range(p, lane);
        const int64_t G = rg.ctas, U = rg.U, u0 = rg.u0, u1 = rg.u1;
        // Units (tiles to visit) of pair pp; lane l caches the count of pair wc_base + l.
        int64_t wc_base = rg.cache_base;
        int32_t wc_val = rg.cache_val;
        auto units_of = [&](int64_t pp) -> int {
            if (p.units == nullptr) return static_cast<int>(p.tiles);
            if (pp < wc_base || pp >= wc_base + 32) {
                wc_base = pp;
                wc_val = pp + lane < p.n_pairs ? p.units[pp + lane] : 0;
            }
            return __shfl_sync(0xffffffffu, wc_val, static_cast<int>(pp - wc_base));
        };
        // Window loader: positions of the next kWin tiles (uniform) and, in
        // lane k, the validity words of slot k (loaded a window ahead).
        uint4 wq = make_uint4(0u, 0u, 0u, 0u);
        int64_t w_pair[kWin], w_start[kWin];
        int w_t[kWin], w_w[kWin];
        int64_t lp = 0, l_start = 0, lu = u0;  // next unit to load, its pair and the pair's first unit
        int lw = 0;
        if (u0 < u1) {
            lp = rg.p0;
            l_start = rg.p0_start;
            lw = units_of(lp);
        }
        auto load_window = [&]() {
            // lane k notes slot k's tile; one load per lane after the loop (predicated
            // loads into one register would wait for each other)
            int my_t = -1;
            int64_t my_idx = 0;
#pragma unroll
            for (int k = 0; k < kWin; ++k) {
                if (lu < u1) {
                    const int t = static_cast<int>(lu - l_start);
                    if (lane == k) {
                        my_t = t;
                        my_idx = lp * p.tiles + t;
                    }
                    w_pair[k] = lp;
                    w_start[k] = l_start;
                    w_t[k] = t;
                    w_w[k] = lw;
                    if (++lu == l_start + lw) {
                        ++lp;
                        l_start = lu;
                        if (lu < u1) lw = units_of(lp);
                    }
                } else {
                    w_pair[k] = w_start[k] = 0;
                    w_t[k] = w_w[k] = 0;
                }
            }
            if (my_t < 0) {
                wq = make_uint4(0u, 0u, 0u, 0u);
            } else if (p.words) {
                wq = p.words[my_idx];
            } else {  // no mask: rows below Ld are valid
                const int64_t nv64 = p.Ld - static_cast<int64_t>(my_t) * kRows;
                const int nv = nv64 < kRows ? static_cast<int>(nv64) : kRows;
                uint32_t wv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = nv - 32 * j;
                    wv[j] = n >= 32 ? 0xffffffffu : (n > 0 ? (1u << n) - 1u : 0u);
                }
                wq = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
        };
        load_window();
        const int64_t total = u1 - u0;
        int64_t q_loaded = -1, q_cur = -1, q_end = 0;
        int qb_cur = 0;
        bool any_tile = false;
        for (int64_t g0 = 0; ok && g0 < total; g0 += kWin) {
            // this window's words and positions to shared memory, then the next window's loads
            if (lane < kWin) sh->win[lane] = wq;
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < kWin; ++k) sh->pos[k] = Pos{w_pair[k], w_start[k], w_t[k], w_w[k]};
            }
            __syncwarp();
            load_window();
            if (lane == 0) {
                for (int k = 0; k < kWin && g0 + k < total; ++k) {
                    const Pos ps = sh->pos[k];
                    const int64_t unit = ps.u_start + ps.t;
                    const int64_t d = doc_of(p, ps.pair);
                    if (ps.t == 0 || unit == u0) any_tile = false;  // a piece starts
                    const uint4 wv = sh->win[k];
                    if ((wv.x | wv.y | wv.z | wv.w) != 0) {
                        StageMeta meta{};
                        if (!any_tile) {
                            any_tile = true;
                            // the pair's query, without a division while pairs stay within it
                            if (ps.pair >= q_end) {
                                q_cur = ps.pair < q_end + p.pairs_per_query ? q_cur + 1 : query_of(p, ps.pair);
                                q_end = (q_cur + 1) * p.pairs_per_query;
                            }
                            if (q_cur != q_loaded) {
                                // the query's rows, into the buffer the MMA released when it
                                // started the query before the previous one
                                if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->empty_q[qb]), qph ^ 1, err))) break;
                                const uint32_t fq = ptx::smem_u32(&bars->full_q[qb]);
                                ptx::mbar_arrive_expect_tx(fq, p.q_bytes);
                                for (int a = 0; a < p.atoms; ++a)
                                    ptx::tma_load_2d(ptx::smem_u32(qbuf + qb * p.q_bytes + a * p.np * kAtomBytes),
                                                     &tmq, a * kAtomElems, static_cast<int32_t>(q_cur * p.Lq), fq);
                                issued_q |= 1u << qb;
                                last_ph_q = (last_ph_q & ~(1u << qb)) | (qph << qb);
                                q_loaded = q_cur;
                                qb_cur = qb;
                                if (++qb == 2) { qb = 0; qph ^= 1; }
                                meta.new_query = 1;
                            }
                        }
                        meta.qb = qb_cur;
                        Rec rec{};
                        rec.kind = kRecTile;
                        rec.jt = ps.t * kRows;
                        rec.valid[0] = wv.x;
                        rec.valid[1] = wv.y;
                        rec.valid[2] = wv.z;
                        rec.valid[3] = wv.w;
                        if (!(ok = publish(rec))) break;
                        if (!(ok = stage(meta, true, d, static_cast<int64_t>(ps.t) * kRows))) break;
                    }
                    if (ps.t == ps.w - 1 || unit == u1 - 1) {
                        // the piece ends: the document's last tile, or the end of this CTA's range
                        Rec end{};
                        end.kind = kRecDocEnd;
                        end.pair = ps.pair;
                        end.nonempty = any_tile ? 1 : 0;
                        if (ps.u_start >= u0 && ps.u_start + ps.w <= u1) {
                            end.c_first = end.c_last = static_cast<int>(blockIdx.x);  // whole here
                        } else {  // only the first and the last pair of the range can be cut
                            const int64_t cf = cta_of_unit(ps.u_start, U, G);
                            end.c_first = static_cast<int>(cf);
                            end.c_last = static_cast<int>(cta_of_unit(ps.u_start + ps.w - 1, U, G));
                            end.first_tail = ps.u_start > cf * U / G ? 1 : 0;
                        }
                        if (!(ok = publish(end))) break;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            __syncwarp();  // the window's entries are read before the next window overwrites them
        }
        if (lane == 0) {
            if (ok) {
                StageMeta stop{};
                stop.stop = 1;
                ok = stage(stop, false, 0, 0);
                Rec r{};
                r.kind = kRecStop;
                if (ok) ok = publish(r);
            }
            for (int k = 0; k < p.stages; ++k)
                if (issued_d & (1u << k))
                    ptx::mbar_wait(ptx::smem_u32(&bars->full_d[k]), (last_ph_d >> k) & 1u, err);
            for (int k = 0; k < 2; ++k)
                if (issued_q & (1u << k))
                    ptx::mbar_wait(ptx::smem_u32(&bars->full_q[k]), (last_ph_q >> k) & 1u, err);
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMA --
        if (lane == 0) {
            int s = 0, ab = 0, prev_qb = -1;
            uint32_t ph = 0, aph = 0;
            uint32_t qph[2] = {0, 0};
            bool ok = true;
            while (ok) {
                if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->full_d[s]), ph, err))) break;
                const StageMeta meta = sh->meta[s];
                if (meta.stop) break;
                if (meta.new_query) {
                    // every MMA on the previous query's rows has been issued: release
                    // its buffer once they complete
                    if (prev_qb >= 0) ptx::mma_commit(ptx::smem_u32(&bars->empty_q[prev_qb]));
                    prev_qb = meta.qb;
                    if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->full_q[meta.qb]), qph[meta.qb], err))) break;
                    qph[meta.qb] ^= 1;
                }
                if (!(ok = ptx::mbar_wait(ptx::smem_u32(&bars->acc_empty[ab]), aph ^ 1, err))) break;
                ptx::tc_fence_after();
                const uint32_t daddr = ptx::smem_u32(dbuf + s * p.d_bytes);
                const uint32_t qaddr = ptx::smem_u32(qbuf + meta.qb * p.q_bytes);
                const uint32_t acc = tmem_base + ab * p.np;
                if (p.dim == 128)  // the common embedding size: no per-step guards
                    ptx::mma_kchain<8>(acc, daddr, kRows * kAtomBytes, qaddr, p.np * kAtomBytes, 8, p.idesc);
                else
                    ptx::mma_kchain<kMaxDim / 16>(acc, daddr, kRows * kAtomBytes, qaddr, p.np * kAtomBytes,
                                                  p.dim / 16, p.idesc);
                ptx::mma_commit(ptx::smem_u32(&bars->empty_d[s]));
                ptx::mma_commit(ptx::smem_u32(&bars->acc_full[ab]));
                if (++s == p.stages) { s = 0; ph ^= 1; }
                if (++ab == kAccBufs) { ab = 0; aph ^= 1; }
            }
            ptx::mma_commit(ptx::smem_u32(&bars->mma_done));
            ptx::mbar_wait(ptx::smem_u32(&bars->mma_done), 0, err);
        }
    } else if (warp < 6) {
        // ------------------------------------------------ update warps --
        const int quarter = warp & 3;         // TMEM lane quarter
        const int r = quarter * 32 + lane;    // tile row = document token jt + r
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        int ri = 0, ab = 0, db = 0;
        uint32_t rph = 0, aph = 0, dph = 0;
        bool ok = true;
        float m[32];
        int am[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            m[c] = -INFINITY;
            am[c] = -1;
        }
        while (ok) {
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->rec_full[ri]), rph, err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const Rec rec = sh->rec[ri];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->rec_empty[ri]));
            if (++ri == kRing) { ri = 0; rph ^= 1; }
            if (rec.kind == kRecTile) {
                ok = ptx::mbar_wait(ptx::smem_u32(&bars->acc_full[ab]), aph, err);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ptx::tc_fence_after();
                uint32_t raw[32];
                ptx::tmem_ld_32(tmem_base + ab * p.np + lane_off, raw);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->acc_empty[ab]));
                if (++ab == kAccBufs) { ab = 0; aph ^= 1; }
                if ((rec.valid[quarter] >> lane) & 1u) {
                    const int j = rec.jt + r;
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float v = __uint_as_float(raw[c]);
                        if (v > m[c]) {
                            m[c] = v;
                            am[c] = j;
                        }
                    }
                }
                continue;
            }
            // end of a document piece (or of the stream): hand the state to the reducer
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->dump_empty[db]), dph ^ 1, err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (rec.kind == kRecDocEnd) {
                fold_half<16>(m, am, lane);
                fold_half<8>(m, am, lane);
                fold_half<4>(m, am, lane);
                fold_half<2>(m, am, lane);
                fold_half<1>(m, am, lane);
                sh->dump[db].m[quarter][lane] = m[0];
                sh->dump[db].a[quarter][lane] = am[0];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    m[c] = -INFINITY;
                    am[c] = -1;
                }
            }
            if (r == 0) {
                sh->info[db].pair = rec.pair;
                sh->info[db].nonempty = rec.nonempty;
                sh->info[db].stop = rec.kind == kRecStop ? 1 : 0;
                sh->info[db].c_first = rec.c_first;
                sh->info[db].c_last = rec.c_last;
                sh->info[db].first_tail = rec.first_tail;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->dump_full[db]));
            if (++db == 2) { db = 0; dph ^= 1; }
            if (rec.kind == kRecStop) break;
        }
    } else if (warp == 6) {
        // ------------------------------------------------- reducer warp --
        // For each document piece: lane i merges the four update warps'
        // (max, argmax) of query token i (lowest token index on ties) and the
        // valid tokens' maxima are summed in a fixed order.  A piece of a cut
        // document goes to the workspace instead; the last piece to arrive
        // merges all pieces in token order.
        int db = 0;
        uint32_t dph = 0;
        bool ok = true;
        while (ok) {
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->dump_full[db]), dph, err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const DumpInfo info = sh->info[db];
            if (info.stop) break;
            float cm = -INFINITY;
            int ca = -1;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float v = sh->dump[db].m[w][lane];
                const int a = sh->dump[db].a[w][lane];
                if (v > cm || (v == cm && a < ca)) {
                    cm = v;
                    ca = a;
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->dump_empty[db]));  // read: release it
            if (++db == 2) { db = 0; dph ^= 1; }

            const int64_t pair = info.pair;
            bool writer = true;  // this CTA writes the pair's score and argmax
            int nonempty = info.nonempty;
            if (info.c_first != info.c_last) {
                // a piece of a cut document: leave (max, argmax) in this piece's slot
                const int c = blockIdx.x;
                const int slot = (c == info.c_first && info.first_tail) ? 2 * c + 1 : 2 * c;
                p.part_m[slot * 32 + lane] = cm;
                p.part_a[slot * 32 + lane] = ca;
                if (lane == 0) p.part_ne[slot] = info.nonempty;
                __threadfence();
                __syncwarp();
                unsigned int before = 0;
                if (lane == 0) before = atomicAdd(&p.arrivals[info.c_first], 1u);
                before = __shfl_sync(0xffffffffu, before, 0);
                writer = before == static_cast<unsigned int>(info.c_last - info.c_first);
                if (writer) {
                    __threadfence();
                    // pieces in CTA order = token order: ties keep the earlier piece
                    cm = -INFINITY;
                    ca = -1;
                    nonempty = 0;
                    for (int cc = info.c_first; cc <= info.c_last; ++cc) {
                        const int s = (cc == info.c_first && info.first_tail) ? 2 * cc + 1 : 2 * cc;
                        const float v = __ldcg(&p.part_m[s * 32 + lane]);
                        const int a = __ldcg(&p.part_a[s * 32 + lane]);
                        nonempty |= __ldcg(&p.part_ne[s]);
                        if (v > cm) {
                            cm = v;
                            ca = a;
                        }
                    }
                }
            }
            if (!writer) continue;
            const int64_t qi = query_of(p, pair);
            const bool qvalid = lane < p.Lq && (!p.qmask || p.qmask[qi * p.Lq + lane]);
            const bool live = nonempty && qvalid;
            if (lane < p.Lq && p.argmax) p.argmax[pair * p.Lq + lane] = live ? ca : -1;
            float total = live ? cm : 0.0f;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) total += __shfl_xor_sync(0xffffffffu, total, off);
            if (lane == 0 && p.scores) p.scores[pair] = nonempty ? total : kEmptyDocScore;
        }
    }

    // Release TMEM once every warp has finished with it: each warp arrives
    // once on an mbarrier after its last tensor-memory access, and the
    // allocating warp waits for all of them (bounded) before freeing the
    // columns.  In the MMA issuer, lane 0 alone did the work:
    // it arrives for its warp and the other lanes leave (the allocating
    // warp's lanes wait for lane 0 first, since the free is warp-wide).  An
    // mbarrier rather than a CTA barrier: the warps arrive microseconds
    // apart, and timing of this kernel showed bar.sync letting warps through
    // before the last warp had arrived.
    ptx::tc_fence_before();
    if (warp == 1) {
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->exit_bar));
    } else {
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&bars->exit_bar));
    }
    if (warp == 1) {
        __syncwarp();
        ptx::mbar_wait(ptx::smem_u32(&bars->exit_bar), 0, p.err);
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, p.acc_cols);
    }
}

}  // namespace

// D stages the kernel's shared memory holds for this problem (at least two
// are needed): the query rows (two buffers), the per-document dumps and the
// barriers come first.
int stream_stages(const Problem& P, int max_smem_optin) {
    const int atoms = static_cast<int>((P.dim + kAtomElems - 1) / kAtomElems);
    const size_t q_bytes = static_cast<size_t>(atoms) * 32 * kAtomBytes;
    const size_t d_bytes = static_cast<size_t>(atoms) * kRows * kAtomBytes;
    const size_t misc = sizeof(Bars) + sizeof(Shared);
    const size_t need = 1024 + misc + 2 * q_bytes;
    if (static_cast<size_t>(max_smem_optin) <= need) return 0;
    const size_t stages = (static_cast<size_t>(max_smem_optin) - need) / d_bytes;
    return stages > kMaxStages ? kMaxStages : static_cast<int>(stages);
}

bool tc_stream_eligible(const Problem& P) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    return (P.layout == kPairwise || P.layout == kKd) && (P.dtype == kF16 || P.dtype == kBF16) &&
           P.dim % 16 == 0 && P.dim <= kMaxDim && P.Lq >= 1 && P.Lq <= kMaxLq && P.Ld >= 1 &&
           P.n_query * P.Lq < (int64_t(1) << 31) && P.Ld < (int64_t(1) << 31) &&
           P.n_doc < (int64_t(1) << 31) && stream_stages(P, device_info(dev).max_smem_optin) >= 2;
}

// Byte offsets of the forward's schedule and merge workspace (plan outputs
// with a document mask, then the cut-document merge slots and counters),
// each 256-byte aligned from the workspace's start.
struct WsLayout {
    int64_t tiles, grid, n_groups;
    size_t o_units, o_groups, o_words, o_pm, o_pa, o_ne, o_arr, bytes;
};

static WsLayout ws_layout(const Problem& P, bool has_dmask, int sm_count) {
    WsLayout L{};
    L.tiles = (P.Ld + kRows - 1) / kRows;
    const int64_t all_tiles = P.n_pairs * L.tiles;
    // one CTA per SM, fewer only when there are fewer tiles than SMs
    L.grid = all_tiles < sm_count ? all_tiles : sm_count;
    L.n_groups = has_dmask ? (P.n_pairs + 31) / 32 : 0;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = (off + bytes + 255) & ~size_t(255);
        return at;
    };
    L.o_units = take(has_dmask ? static_cast<size_t>(P.n_pairs) * 4 : 0);
    L.o_groups = take(static_cast<size_t>(L.n_groups) * 4);
    L.o_words = take(has_dmask ? static_cast<size_t>(all_tiles) * 16 : 0);
    L.o_pm = take(static_cast<size_t>(2 * L.grid) * 32 * 4);
    L.o_pa = take(static_cast<size_t>(2 * L.grid) * 32 * 4);
    L.o_ne = take(static_cast<size_t>(2 * L.grid) * 4);
    L.o_arr = take(static_cast<size_t>(L.grid) * 4);
    L.bytes = off;
    return L;
}

// Library-owned memory pool of a device for the forward's schedule and merge
// workspace when the caller passes none: allocations are stream-ordered and
// freed on the stream after the kernel, and the pool keeps the memory it has
// mapped, so steady-state calls map nothing new.
static cudaError_t workspace_pool(int dev, cudaMemPool_t* out) {
    static std::mutex mu;
    static std::vector<cudaMemPool_t> pools;
    std::lock_guard<std::mutex> lock(mu);
    if (static_cast<int>(pools.size()) <= dev) pools.resize(dev + 1, nullptr);
    if (pools[dev] == nullptr) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        cudaError_t e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        pools[dev] = pool;
    }
    *out = pools[dev];
    return cudaSuccess;
}

size_t stream_workspace_bytes(const Problem& P, bool has_dmask) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    return ws_layout(P, has_dmask, device_info(dev).sm_count).bytes;
}

cudaError_t launch_fwd_tc_stream(const Problem& P, float* scores, int32_t* argmax, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const DeviceInfo& info = device_info(dev);

    Params p{};
    p.n_pairs = P.n_pairs;
    p.pairs_per_query = P.pairs_per_query;
    p.n_doc = P.n_doc;
    p.Lq = P.Lq;
    p.Ld = P.Ld;
    p.layout = P.layout;
    p.dim = static_cast<int>(P.dim);
    p.atoms = (p.dim + kAtomElems - 1) / kAtomElems;
    p.np = 32;  // the update warps read 32 columns (query tokens past Lq are zero rows)
    int cols = 32;
    while (cols < kAccBufs * p.np) cols <<= 1;
    p.acc_cols = cols;
    p.q_bytes = static_cast<uint32_t>(p.atoms * p.np * kAtomBytes);
    p.d_bytes = static_cast<uint32_t>(p.atoms * kRows * kAtomBytes);
    const size_t misc = sizeof(Bars) + sizeof(Shared);
    p.stages = stream_stages(P, info.max_smem_optin);
    if (p.stages < 2) return cudaErrorInvalidConfiguration;  // tc_stream_eligible rules this out
    p.idesc = ptx::f16_idesc(kRows, p.np, P.dtype == kBF16);
    p.qmask = P.qmask;
    p.dmask = P.dmask;
    p.scores = scores;
    p.argmax = argmax;
    p.err = device_error_word();

    CUtensorMap tmq, tmd;
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(P.dim), static_cast<uint64_t>(P.n_query * P.Lq)};
        const uint64_t strides[1] = {static_cast<uint64_t>(P.dim) * 2};
        const uint32_t box[2] = {kAtomElems, static_cast<uint32_t>(p.np)};
        if (!encode_tmap_kmajor(&tmq, P.dtype, P.Q, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(P.dim), static_cast<uint64_t>(P.Ld),
                                  static_cast<uint64_t>(P.n_doc)};
        const uint64_t strides[2] = {static_cast<uint64_t>(P.dim) * 2, static_cast<uint64_t>(P.Ld * P.dim) * 2};
        const uint32_t box[3] = {kAtomElems, kRows, 1};
        if (!encode_tmap_kmajor(&tmd, P.dtype, P.D, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const size_t smem = 1024 + 2 * static_cast<size_t>(p.q_bytes) + static_cast<size_t>(p.stages) * p.d_bytes + misc;
    e = cudaFuncSetAttribute(stream_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const WsLayout L = ws_layout(P, P.dmask != nullptr, info.sm_count);
    p.tiles = L.tiles;
    p.n_groups = L.n_groups;
    const int64_t grid = L.grid;

    // the caller's workspace, or one from the library's pool (freed on the
    // stream after the kernel)
    void* ws = workspace;
    if (ws == nullptr) {
        cudaMemPool_t pool = nullptr;
        if ((e = workspace_pool(dev, &pool)) != cudaSuccess) return e;
        if ((e = cudaMallocFromPoolAsync(&ws, L.bytes, pool, stream)) != cudaSuccess) return e;
    } else if (workspace_bytes < L.bytes) {
        return cudaErrorInvalidValue;  // the entry points check the size before calling
    }
    uint8_t* base = static_cast<uint8_t*>(ws);
    p.units = P.dmask ? reinterpret_cast<const int32_t*>(base + L.o_units) : nullptr;
    p.group_units = P.dmask ? reinterpret_cast<const int32_t*>(base + L.o_groups) : nullptr;
    p.words = P.dmask ? reinterpret_cast<const uint4*>(base + L.o_words) : nullptr;
    p.part_m = reinterpret_cast<float*>(base + L.o_pm);
    p.part_a = reinterpret_cast<int32_t*>(base + L.o_pa);
    p.part_ne = reinterpret_cast<int32_t*>(base + L.o_ne);
    p.arrivals = reinterpret_cast<unsigned int*>(base + L.o_arr);

    PlanArgs pa{};
    pa.dmask = P.dmask;
    pa.n_pairs = P.n_pairs;
    pa.Ld = P.Ld;
    pa.tiles = p.tiles;
    pa.n_groups = p.n_groups;
    pa.units = reinterpret_cast<int32_t*>(base + L.o_units);
    pa.group_units = reinterpret_cast<int32_t*>(base + L.o_groups);
    pa.words = reinterpret_cast<uint4*>(base + L.o_words);
    pa.arrivals = p.arrivals;
    pa.n_arrivals = grid;
    const int64_t all_tiles = P.n_pairs * p.tiles;
    const int64_t word_blocks = P.dmask ? (all_tiles + 255) / 256 : 0;
    const int64_t zero_blocks = (grid + 1023) / 1024;
    const int64_t plan_blocks =
        p.n_groups + word_blocks > zero_blocks ? p.n_groups + word_blocks : zero_blocks;
    stream_plan_kernel<<<static_cast<unsigned>(plan_blocks), 1024, 0, stream>>>(pa);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, stream_fwd_tc_kernel, tmq, tmd, p);
    }
    if (workspace == nullptr) {
        const cudaError_t ef = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess) e = ef;
    }
    return e;
}

}  // namespace lik
