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
//     S[128, Np] = Dtile[128, dim] . Qb[Np, dim]^T    (fp32 in TMEM)
// with Np = Lq rounded up to 16.  So each accumulator lane is one document
// token and each column one query token.
//
// Roles (one CTA per SM, persistent over a contiguous range of pairs):
//   warp 0      producer.  All 32 lanes read the document mask a window of
//               8 tiles ahead and build each tile's 128-bit row-validity mask
//               (one ballot per 32 rows); tiles with no
//               valid token are skipped (never loaded).  Lane 0 issues the
//               TMA loads (a query's rows into one of two buffers when the
//               query changes, document tiles per stage) and publishes,
//               through a ring of tile records, the sequence the epilogue
//               follows: data tiles, one end-of-document record per pair, and
//               an end-of-stream record.
//   warp 1      TMEM allocator + single-thread MMA issuer (4 accumulators).
//   update warps  one group of 4 warps per 32 query tokens.  Each thread
//               owns one accumulator lane (document token) and keeps a
//               running (max, argmax) for each of its group's 32 query
//               tokens in registers across the document's tiles.  At the end
//               of a document it dumps that state to shared memory (double-
//               buffered) and goes straight on with the next document.
//   reducer warps (4) reduce each dumped document over its 128 lanes per
//               query token (lowest token index on ties), sum the valid
//               query tokens in a fixed order, and write the score and
//               argmax, while the stream continues.
// Every mbarrier wait is bounded; on expiry the kernel flags the library's
// error word, drains its own loads and MMAs, frees TMEM and returns.
#include <cfloat>

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
constexpr int kMaxGroups = 1;       // Lq <= 32 (the double-buffered dump fits shared memory)

enum : int { kRecTile = 0, kRecDocEnd = 1, kRecStop = 2 };

struct Rec {
    int kind;
    int jt;                 // first document token of the tile
    int64_t pair;           // pair index (doc end) / unused
    uint32_t valid[4];      // row-validity bits of the tile (tile records)
    int nonempty;           // doc end: the document had a valid token
    int pad;
};

struct StageMeta {
    int qb;                 // query buffer the tile multiplies
    int new_query;          // first tile with freshly loaded query rows: wait for them
    int stop;               // end of stream
    int pad;
};

struct Params {
    int64_t n_pairs, pairs_per_query, n_doc, Lq, Ld;
    int layout, dim, atoms, np, groups, stages, acc_cols;
    uint32_t idesc, q_bytes, d_bytes;
    const uint8_t* qmask;
    const uint8_t* dmask;
    float* scores;
    int32_t* argmax;
    unsigned int* err;
};

struct Bars {
    uint64_t full_d[kMaxStages], empty_d[kMaxStages];
    uint64_t full_q[2], empty_q[2];
    uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
    uint64_t rec_full[kRing], rec_empty[kRing];
    uint64_t dump_full[2], dump_empty[2];  // update warps -> reducer warps
    uint64_t red_mid;                      // reducer warps: partials written
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t pad;
};

// Per-document state handed from the update warps to the reducer warps
// (double-buffered): every lane's running (max, argmax) per query token,
// rows padded to 33 words so both the row-wise writes and the column-wise
// reads are free of bank conflicts.
struct Dump {
    float m[kRows][33];
    int a[kRows][33];
};

struct DumpInfo {
    int64_t pair;
    int nonempty;
    int stop;
};

struct Shared {
    uint32_t win[kWin][4];   // producer: row-validity words of the current window
    Rec rec[kRing];
    StageMeta meta[kMaxStages];
    DumpInfo info[2];
    float part_m[4][32];
    int part_a[4][32];
    float gsum[kMaxGroups];
};

__device__ __forceinline__ int64_t doc_of(const Params& p, int64_t pair) {
    return pair;  // pairwise: document b; kd: document b*N + n
}

__device__ __forceinline__ int64_t query_of(const Params& p, int64_t pair) {
    return pair / p.pairs_per_query;
}

// Mask bytes of the tile starting at token jt of document d: lane l holds
// tokens jt + l, jt + 32 + l, jt + 64 + l, jt + 96 + l (0 past Ld).
__device__ __forceinline__ void load_tile_mask(const Params& p, int64_t d, int64_t jt, int lane,
                                               uint8_t (&b)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int64_t j = jt + 32 * k + lane;
        b[k] = j < p.Ld ? (p.dmask ? p.dmask[d * p.Ld + j] : uint8_t(1)) : uint8_t(0);
    }
}

__global__ void __launch_bounds__(32 * (2 + 4 * kMaxGroups + 4), 1)
stream_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmd,
                     const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qbuf = smem;                          // 2 x q_bytes
    uint8_t* dbuf = smem + 2 * p.q_bytes;          // stages x d_bytes
    Bars* bars = reinterpret_cast<Bars*>(dbuf + p.stages * p.d_bytes);
    Shared* sh = reinterpret_cast<Shared*>(bars + 1);
    Dump* dump = reinterpret_cast<Dump*>(sh + 1);  // [2][groups]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned int* err = p.err;

    // contiguous range of pairs for this CTA
    const int64_t per = (p.n_pairs + gridDim.x - 1) / gridDim.x;
    const int64_t pb = blockIdx.x * per;
    const int64_t pe = pb + per < p.n_pairs ? pb + per : p.n_pairs;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->full_d[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->empty_d[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bars->full_q[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->empty_q[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->dump_full[b]), 32 * 4 * p.groups);
            ptx::mbar_init(ptx::smem_u32(&bars->dump_empty[b]), 128);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bars->acc_full[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->acc_empty[b]), 4 * p.groups);
        }
        for (int r = 0; r < kRing; ++r) {
            ptx::mbar_init(ptx::smem_u32(&bars->rec_full[r]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->rec_empty[r]), 4 * p.groups);
        }
        ptx::mbar_init(ptx::smem_u32(&bars->red_mid), 128);
        ptx::mbar_init(ptx::smem_u32(&bars->mma_done), 1);
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

    if (warp == 0) {
        // ------------------------------------------------------ producer --
        int s = 0, qb = 0, ri = 0;
        uint32_t ph = 0, qph = 0, rph = 0;
        uint32_t issued_d = 0, issued_q = 0, last_ph_d = 0, last_ph_q = 0;
        bool ok = true;
        // publish one record (lane 0), waiting for its ring slot
        auto publish = [&](const Rec& rec) -> bool {
            bool good = true;
            if (lane == 0) {
                good = ptx::mbar_wait(ptx::smem_u32(&bars->rec_empty[ri]), rph ^ 1, err);
                if (good) {
                    sh->rec[ri] = rec;
                    ptx::mbar_arrive(ptx::smem_u32(&bars->rec_full[ri]));
                }
            }
            good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
            if (++ri == kRing) { ri = 0; rph ^= 1; }
            return good;
        };
        // hand one stage to the MMA (lane 0); data=false sends only metadata
        auto stage = [&](const StageMeta& meta, bool data, int64_t d, int64_t jt) -> bool {
            bool good = true;
            if (lane == 0) {
                good = ptx::mbar_wait(ptx::smem_u32(&bars->empty_d[s]), ph ^ 1, err);
                if (good) {
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
                }
            }
            good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
            if (++s == p.stages) { s = 0; ph ^= 1; }
            return good;
        };

        const int64_t tiles = (p.Ld + kRows - 1) / kRows;
        const int64_t total = (pe - pb) * tiles;  // flat (pair, tile) positions of this CTA
        // Document-mask bytes are read a window of kWin tiles ahead (4 bytes
        // per lane per tile, all loads in flight together), so the producer
        // never waits on a mask load while the stream needs tiles.
        uint8_t wb[kWin][4];
        int64_t lp = pb, lt = 0;  // position the next window load starts at
        auto load_window = [&]() {
#pragma unroll
            for (int k = 0; k < kWin; ++k) {
                if (lp < pe) {
                    load_tile_mask(p, doc_of(p, lp), lt * kRows, lane, wb[k]);
                    if (++lt == tiles) { lt = 0; ++lp; }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) wb[k][j] = 0;
                }
            }
        };
        load_window();
        int64_t cp = pb, ct = 0;  // position being published
        int64_t q_loaded = -1;
        int qb_cur = 0;
        bool any_tile = false;
        for (int64_t g0 = 0; ok && g0 < total; g0 += kWin) {
            // validity words of this window, then the next window's loads
#pragma unroll
            for (int k = 0; k < kWin; ++k)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w = __ballot_sync(0xffffffffu, wb[k][j] != 0);
                    if (lane == 0) sh->win[k][j] = w;
                }
            __syncwarp();
            load_window();
            for (int k = 0; ok && k < kWin && g0 + k < total; ++k) {
                const int64_t d = doc_of(p, cp);
                if (ct == 0) any_tile = false;
                uint32_t w[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) w[j] = sh->win[k][j];
                if ((w[0] | w[1] | w[2] | w[3]) != 0) {
                    StageMeta meta{};
                    if (!any_tile) {
                        any_tile = true;
                        const int64_t q = query_of(p, cp);
                        if (q != q_loaded) {
                            // the query's rows, into the buffer the MMA released when it
                            // started the query before the previous one
                            if (lane == 0) {
                                ok = ptx::mbar_wait(ptx::smem_u32(&bars->empty_q[qb]), qph ^ 1, err);
                                if (ok) {
                                    const uint32_t fq = ptx::smem_u32(&bars->full_q[qb]);
                                    ptx::mbar_arrive_expect_tx(fq, p.q_bytes);
                                    for (int a = 0; a < p.atoms; ++a)
                                        ptx::tma_load_2d(ptx::smem_u32(qbuf + qb * p.q_bytes + a * p.np * kAtomBytes),
                                                         &tmq, a * kAtomElems, static_cast<int32_t>(q * p.Lq), fq);
                                    issued_q |= 1u << qb;
                                    last_ph_q = (last_ph_q & ~(1u << qb)) | (qph << qb);
                                }
                            }
                            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                            if (!ok) break;
                            q_loaded = q;
                            qb_cur = qb;
                            if (++qb == 2) { qb = 0; qph ^= 1; }
                            meta.new_query = 1;
                        }
                    }
                    meta.qb = qb_cur;
                    Rec rec{};
                    rec.kind = kRecTile;
                    rec.jt = static_cast<int>(ct * kRows);
#pragma unroll
                    for (int j = 0; j < 4; ++j) rec.valid[j] = w[j];
                    if (!(ok = publish(rec))) break;
                    if (!(ok = stage(meta, true, d, ct * kRows))) break;
                }
                if (ct == tiles - 1) {
                    Rec end{};
                    end.kind = kRecDocEnd;
                    end.pair = cp;
                    end.nonempty = any_tile ? 1 : 0;
                    if (!(ok = publish(end))) break;
                }
                if (++ct == tiles) { ct = 0; ++cp; }
            }
            __syncwarp();  // the window's words are read before the next window overwrites them
        }
        if (ok) {
            StageMeta stop{};
            stop.stop = 1;
            ok = stage(stop, false, 0, 0);
            Rec r{};
            r.kind = kRecStop;
            if (ok) ok = publish(r);
        }
        if (lane == 0) {
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
    } else if (warp < 2 + 4 * p.groups) {
        // ------------------------------------------------ update warps --
        const int ew = warp - 2;
        const int g = ew >> 2;                // query-token group: columns 32g .. 32g+31
        const int quarter = warp & 3;         // TMEM lane quarter
        const int r = quarter * 32 + lane;    // tile row = document token jt + r
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const int col0 = 32 * g;
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
                ptx::tmem_ld_32(tmem_base + ab * p.np + col0 + lane_off, raw);
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
            // end of a document (or of the stream): hand the state to the reducer
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->dump_empty[db]), dph ^ 1, err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (rec.kind == kRecDocEnd) {
                Dump& dd = dump[db * p.groups + g];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    dd.m[r][c] = m[c];
                    dd.a[r][c] = am[c];
                    m[c] = -INFINITY;
                    am[c] = -1;
                }
            }
            if (g == 0 && r == 0) {
                sh->info[db].pair = rec.pair;
                sh->info[db].nonempty = rec.nonempty;
                sh->info[db].stop = rec.kind == kRecStop ? 1 : 0;
            }
            ptx::mbar_arrive(ptx::smem_u32(&bars->dump_full[db]));
            if (++db == 2) { db = 0; dph ^= 1; }
            if (rec.kind == kRecStop) break;
        }
    } else if (warp < 2 + 4 * p.groups + 4) {
        // ----------------------------------------------- reducer warps --
        // For each document: every (quarter, lane) thread takes query token
        // `lane` over rows 32*quarter .. +31 in ascending order, the four
        // partials are merged in row order (lowest token index on ties), the
        // valid tokens' maxima are summed per group in a fixed order, then
        // the groups' sums in group order.
        const int quarter = (warp - 2 - 4 * p.groups);
        int db = 0;
        uint32_t dph = 0, mph = 0;
        bool ok = true;
        while (ok) {
            ok = ptx::mbar_wait(ptx::smem_u32(&bars->dump_full[db]), dph, err);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const DumpInfo info = sh->info[db];
            if (info.stop) break;
            const int64_t pair = info.pair;
            const int64_t qi = query_of(p, pair);
            float total = 0.0f;
            for (int g = 0; g < p.groups; ++g) {
                const Dump& dd = dump[db * p.groups + g];
                float bm = -INFINITY;
                int ba = -1;
                for (int rr = 32 * quarter; rr < 32 * quarter + 32; ++rr) {
                    const float v = dd.m[rr][lane];
                    if (v > bm) {
                        bm = v;
                        ba = dd.a[rr][lane];
                    }
                }
                sh->part_m[quarter][lane] = bm;
                sh->part_a[quarter][lane] = ba;
                ptx::mbar_arrive(ptx::smem_u32(&bars->red_mid));
                ok = ptx::mbar_wait(ptx::smem_u32(&bars->red_mid), mph, err);
                ok = __all_sync(0xffffffffu, ok);
                mph ^= 1;
                if (!ok) break;
                if (quarter == 0) {
                    float cm = -INFINITY;
                    int ca = -1;
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float v = sh->part_m[w][lane];
                        if (v > cm) {
                            cm = v;
                            ca = sh->part_a[w][lane];
                        }
                    }
                    const int i = 32 * g + lane;
                    const bool qvalid = i < p.Lq && (!p.qmask || p.qmask[qi * p.Lq + i]);
                    const bool live = info.nonempty && qvalid;
                    if (i < p.Lq && p.argmax) p.argmax[pair * p.Lq + i] = live ? ca : -1;
                    float term = live ? cm : 0.0f;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) term += __shfl_xor_sync(0xffffffffu, term, off);
                    total += term;
                }
                // the partials of this group are read before the next group's overwrite them
                ptx::mbar_arrive(ptx::smem_u32(&bars->red_mid));
                ok = ptx::mbar_wait(ptx::smem_u32(&bars->red_mid), mph, err);
                ok = __all_sync(0xffffffffu, ok);
                mph ^= 1;
                if (!ok) break;
            }
            if (!ok) break;
            if (quarter == 0 && lane == 0 && p.scores) p.scores[pair] = info.nonempty ? total : kEmptyDocScore;
            ptx::mbar_arrive(ptx::smem_u32(&bars->dump_empty[db]));
            if (++db == 2) { db = 0; dph ^= 1; }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
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
    const int groups = static_cast<int>((P.Lq + 31) / 32);
    const size_t q_bytes = static_cast<size_t>(atoms) * 32 * groups * kAtomBytes;
    const size_t d_bytes = static_cast<size_t>(atoms) * kRows * kAtomBytes;
    const size_t misc = sizeof(Bars) + sizeof(Shared) + 2 * static_cast<size_t>(groups) * sizeof(Dump);
    const size_t need = 1024 + misc + 2 * q_bytes;
    if (static_cast<size_t>(max_smem_optin) <= need) return 0;
    const size_t stages = (static_cast<size_t>(max_smem_optin) - need) / d_bytes;
    return stages > kMaxStages ? kMaxStages : static_cast<int>(stages);
}

bool tc_stream_eligible(const Problem& P) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    return (P.layout == kPairwise || P.layout == kKd) && (P.dtype == kF16 || P.dtype == kBF16) &&
           P.dim % 16 == 0 && P.dim <= kMaxDim && P.Lq >= 1 && P.Lq <= 32 * kMaxGroups && P.Ld >= 1 &&
           P.n_query * P.Lq < (int64_t(1) << 31) && P.Ld < (int64_t(1) << 31) &&
           P.n_doc < (int64_t(1) << 31) && stream_stages(P, device_info(dev).max_smem_optin) >= 2;
}

cudaError_t launch_fwd_tc_stream(const Problem& P, float* scores, int32_t* argmax, cudaStream_t stream) {
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
    p.groups = static_cast<int>((P.Lq + 31) / 32);
    p.np = 32 * p.groups;  // every group reads 32 columns, so N covers whole groups
    int cols = 32;
    while (cols < kAccBufs * p.np) cols <<= 1;
    p.acc_cols = cols;
    p.q_bytes = static_cast<uint32_t>(p.atoms * p.np * kAtomBytes);
    p.d_bytes = static_cast<uint32_t>(p.atoms * kRows * kAtomBytes);
    const size_t misc = sizeof(Bars) + sizeof(Shared) + 2 * static_cast<size_t>(p.groups) * sizeof(Dump);
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
    const int64_t grid = P.n_pairs < info.sm_count ? P.n_pairs : info.sm_count;
    const int threads = 32 * (2 + 4 * p.groups + 4);
    stream_fwd_tc_kernel<<<static_cast<unsigned>(grid), threads, smem, stream>>>(tmq, tmd, p);
    return cudaGetLastError();
}

}  // namespace lik
