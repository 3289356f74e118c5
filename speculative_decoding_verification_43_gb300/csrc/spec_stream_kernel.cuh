// spec_stream_kernel: the per-position kernel of spec_verify for row slices of up to
// Geo<DT>::kMaxTiles tiles (included once, by spec_verify.cu; the rule and the exchange are those of
// spec_rows.cuh and spec_rows_kernel.cuh).
//
// One CTA per SM (clusters of C CTAs; C = 4 for bf16 V = 128256), rows streamed through shared
// memory in tiles of Geo<DT>::kVPT 16-byte vectors per data thread (three for bf16: 1440-vector
// tiles; two for f32: 960):
//   - a target ring of kTRing tiles carries, item after item, the target tiles of pass 1 of item
//     i (from HBM) and then those of pass 2 of item i - 1 (read again, from L2);
//   - a draft ring of kDRing tiles carries each pair's draft tiles; pass 1 reads them and leaves
//     them in place, pass 2 (one item later) reads them again and frees them tile by tile, so
//     the draft row crosses HBM once and never leaves the chip between the passes;
//   - pass 2 of item i - 1 runs after pass 1 of item i, so that item i - 1's exchange and
//     decision overlap item i's pass 1.
// Warp roles: the control warp (exchange, decision, draw), 15 data warps, and one producer warp
// per ring. A producer walks its ring's sequence and refills a slot as soon as the 15 data warps
// have arrived on the slot's "empty" barrier (bulk copy completing on its "full" barrier), so the
// data warps never issue copies. Thread t takes vectors t, t + 480, ... of every tile (one per
// vector of the thread), so chunk (r, warp), r = kVPT tile + u, covers vectors 480 r + 32 warp ...,
// the chunk numbering of the rows kernel, and the control warp's exchange, decision and draw code
// is shared with it.
#pragma once

#include "spec_rows_kernel.cuh"

namespace spec {

// Tile geometry per input type: vectors per data thread per tile (three for bf16; two for f32,
// whose wider vectors would not fit the registers three times over), ring depths and the
// dynamic shared memory (the rings, then the exchange slots).
template <int DT>
struct Geo {
    static constexpr int kVPT = (DT == SPEC_BF16) ? 3 : 2;
    static constexpr int kTileVecs = kVPT * kThreads;           // 1440 / 960 vectors
    static constexpr int kMaxTiles = kMaxStreamRows / kVPT;      // tiles of the largest slice
    static constexpr int kTRing = 3;                             // target tile slots
    static constexpr int kDRing = 2 * kMaxTiles;                 // draft tile slots: two items' slices
                                                                 // (pass 1 of item i + 1 runs while
                                                                 // item i's drafts wait for pass 2)
    static constexpr size_t kDynSmem = static_cast<size_t>(kTRing + kDRing) * kTileVecs * 16 +
                                       static_cast<size_t>(kNMS) * kMaxCluster * sizeof(Msg);
};
constexpr int kTRingMax = 3;
constexpr int kDRingMax = 2 * (kMaxStreamRows / 2);
constexpr int kStreamBlock = kBlock + 2 * kWarp;  // control, 15 data warps, two producers
// named barriers of the streaming kernel (BAR_BATCH: control and data warps)
enum : int { BAR_SHAPES = 2, BAR_PROD = 3 };
constexpr int kProdBarThreads = 3 * kWarp;     // control warp and the two producers

struct StreamShared {
    CtaShared c;                                // state shared with the exchange / draw helpers
    uint64_t tfull[kTRingMax], dfull[kDRingMax];    // a tile's bulk copy has landed
    uint64_t tempty[kTRingMax], dempty[kDRingMax];  // the 15 data warps are done with the slot
    int32_t rows[kMaxItems];                    // rows each item of the batch streams (0, 1, 2)
    long long t_issued, d_issued;               // tiles issued by each producer (all batches)
};

// A bounded wait of the streaming kernel: one plain test first (the common case: the phase is
// complete), then suspended tries. Once a wait of this CTA has given up (the results are already
// flagged), the later ones give up after a couple of tries, so that a CTA whose copies stopped
// landing leaves in milliseconds rather than seconds per wait.
__device__ __forceinline__ bool stream_wait(const CtaShared &sh, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const int tries = *reinterpret_cast<const volatile int32_t *>(&sh.timed_out) ? 2 : kMaxWaitTries;
    return mbar_wait_sleep_bounded(bar, parity, kSuspendNs, tries);
}

// Bytes of tile `t` of a row slice of nvec vectors.
template <int DT>
__device__ __forceinline__ uint32_t tile_bytes(int t, int nvec) {
    using G = Geo<DT>;
    return static_cast<uint32_t>(min(G::kTileVecs, nvec - t * G::kTileVecs)) * 16u;
}

// A data warp's position in a ring's sequence: the slot and the parity of its fill.
struct RingPos {
    int slot;
    uint32_t par;
};
template <int N>
__device__ __forceinline__ void ring_next(RingPos &p) {
    if (++p.slot == N) {
        p.slot = 0;
        p.par ^= 1u;
    }
}

// A data warp is done with a slot (its lanes' reads of it are complete).
__device__ __forceinline__ void slot_done(uint64_t *empty, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(empty);
}

// Producer lane: the next tile of a ring's sequence into slot pos % ring, once the data warps
// have emptied the slot's previous fill (position pos - ring).
template <int DT>
__device__ __forceinline__ void issue_tile(CtaShared &sh, uint64_t *full, uint64_t *empty, uint4 *ring, int nring,
                                           long long pos, const void *src, uint32_t bytes, uint64_t pol) {
    using G = Geo<DT>;
    const int slot = static_cast<int>(pos % nring);
    if (pos >= nring && !stream_wait(sh, &empty[slot], static_cast<uint32_t>((pos / nring - 1) & 1)))
        sh.timed_out = 1;
    mbar_arrive_expect_tx(&full[slot], bytes);
    bulk_g2s(ring + static_cast<size_t>(slot) * G::kTileVecs, src, bytes, &full[slot], pol);
}

// Target producer, one batch: for job i, the pass-1 tiles of item i (a pair's: evict-last, read
// again one item later; a plain row's: evict-first, its only use), then the pass-2 tiles of pair
// item i - kStreamLag (evict-first: the last use).
template <int DT>
__device__ __forceinline__ void produce_targets(StreamShared &ss, uint4 *tring, const RowsParams &P, int lo,
                                                int nvec, int ntiles, int nbatch) {
    using G = Geo<DT>;
    const size_t row_bytes = static_cast<size_t>(P.nvec_row) * 16;
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    long long pos = ss.t_issued;
    for (int i = 0; i < nbatch + kStreamLag; ++i) {
#pragma unroll 1
        for (int ph = 0; ph < 2; ++ph) {
            const int item = ph == 0 ? i : i - kStreamLag;
            if (item < 0 || item >= nbatch) continue;
            if (ph == 0 ? ss.rows[item] < 1 : ss.rows[item] != 2) continue;
            const unsigned char *src = static_cast<const unsigned char *>(P.target) +
                                       static_cast<size_t>(ss.c.desc[item].item) * row_bytes +
                                       static_cast<size_t>(lo) * 16;
#pragma unroll 1
            for (int t = 0; t < ntiles; ++t, ++pos)
                issue_tile<DT>(ss.c, ss.tfull, ss.tempty, tring, G::kTRing, pos, src + static_cast<size_t>(t) * G::kTileVecs * 16,
                           tile_bytes<DT>(t, nvec), (ph == 0 && ss.rows[item] == 2) ? keep : drop);
        }
    }
    ss.t_issued = pos;
}

// Draft producer, one batch: the tiles of each pair's draft row, in item order. A draft slot
// frees in pass 2 of the pair two items earlier; the tiles of pass 2 and of the pass 1 after it
// give the copy its lead.
template <int DT>
__device__ __forceinline__ void produce_drafts(StreamShared &ss, uint4 *dring, const RowsParams &P, int lo,
                                               int nvec, int ntiles, int nbatch) {
    using G = Geo<DT>;
    const size_t row_bytes = static_cast<size_t>(P.nvec_row) * 16;
    const uint64_t drop = policy_evict_first();
    long long pos = ss.d_issued;
    bool launch = pos == 0;  // the kernel's first pair
    for (int i = 0; i < nbatch; ++i) {
        if (ss.rows[i] != 2) continue;
        const unsigned char *src = static_cast<const unsigned char *>(P.draft) +
                                   static_cast<size_t>(ss.c.desc[i].drow) * row_bytes + static_cast<size_t>(lo) * 16;
#pragma unroll 1
        for (int t = 0; t < ntiles; ++t, ++pos)
            issue_tile<DT>(ss.c, ss.dfull, ss.dempty, dring, G::kDRing, pos, src + static_cast<size_t>(t) * G::kTileVecs * 16,
                       tile_bytes<DT>(t, nvec), drop);
        if (launch) {
            // at launch every CTA asks for its first tiles at once: the next pair's drafts wait until
            // the first pair's have landed, so that they do not queue ahead of the first items' tiles
            launch = false;
            const long long last = pos - 1;
            if (!stream_wait(ss.c, &ss.dfull[last % G::kDRing], static_cast<uint32_t>((last / G::kDRing) & 1)))
                ss.c.timed_out = 1;
        }
    }
    ss.d_issued = pos;
}

// Pass 1 state of one row in one thread: the integral reference b (-inf until a finite vector
// is seen) and the sum of 2^(y s - b) over the thread's vectors so far.
struct RowAcc {
    float b;
    float s;
};

// Sum of 2^(y s - b) over one vector (pairs of lanes packed, as in the rows kernel).
template <int DT>
__device__ __forceinline__ float vec_sum(const uint4 &w, float2 shi2, float2 slo2, float b) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    const float2 nb2 = f2splat(-b);
    float2 e[H];
#pragma unroll
    for (int h = 0; h < H; ++h) e[h] = ex2x2(exp_arg2(Elt<DT>::unpack_one(w, h), shi2, slo2, nb2));
    // a tree (H = 4 for bf16, 2 for f32): two dependent adds after the exponentials, not four
#pragma unroll
    for (int st = 1; st < H; st <<= 1)
#pragma unroll
        for (int h = 0; h + st < H; h += 2 * st) e[h] = __fadd2_rn(e[h], e[h + st]);
    return e[0].x + e[0].y;
}

// A vector's sum at the thread's reference b. While the thread has no reference (b = -inf) the
// terms are +inf (finite logits) or NaN (-inf logits): either sends the tile to the slow path.
template <int DT>
__device__ __forceinline__ float vec_share(const uint4 &w, float b, float2 shi2, float2 slo2) {
    return vec_sum<DT>(w, shi2, slo2, b);
}

// The slow path of a vector whose share overflowed (a term above 2^64, an infinite or NaN sum,
// or no reference yet): the reference rises to the vector's own floor(max y s) and the running
// sum is rescaled by the exact power of two; returns the share at the new reference. The fast
// path takes the reference from the thread's first vector, so no exponential waits on a running
// max.
template <int DT>
__device__ __forceinline__ float share_slow(RowAcc &A, const uint4 &w, float s_hi, float2 shi2, float2 slo2) {
    const float m = floorf(Elt<DT>::vmax(w) * s_hi);
    if (m > A.b || A.b == -INFINITY) {
        const float nb = fmaxf(A.b, m);
        const float sc = (A.b == -INFINITY) ? 0.0f : pow2i(A.b - nb);
        A.s *= sc;
        A.b = nb;
    }
    return (A.b == -INFINITY) ? 0.0f : vec_sum<DT>(w, shi2, slo2, A.b);
}

// Greedy rule, one vector: the largest logit and the smallest index attaining it; NaN / +inf
// make the row invalid.
template <int DT>
__device__ __forceinline__ void greedy_vec(const uint4 &w, int base, float &best, int &bidx, int &bad) {
    constexpr int E = Elt<DT>::kPerVec;
    constexpr int H = E / 2;
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const float2 y = Elt<DT>::unpack_one(w, h);
        bad |= (y.x != y.x) || (y.x == INFINITY) || (y.y != y.y) || (y.y == INFINITY);
    }
    const float mv = Elt<DT>::vmax(w);
    if (mv > best) {
        best = mv;
        for (int e = E - 1; e >= 0; --e)
            if (vec_elem<DT>(w, e) == mv) bidx = base + e;
    }
}

// A warp's greedy statistics of row r into ws (the record encoding of WarpStat).
__device__ __forceinline__ void warp_greedy_stats(CtaShared &sh, int wb, int r, int warp, int lane, float best,
                                                  int bidx, int bad) {
    const float wbest = warp_max(best);
    const int widx = warp_min_i32(best == wbest ? bidx : INT_MAX);
    const int wbad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        sh.ws[wb][warp].b[r] = wbad ? INFINITY : wbest;
        sh.ws[wb][warp].a[r] = wbad ? -1 : widx;
    }
}

// Bonus rows: chunk k (this warp's vectors of one chunk row) of p for a later draw, in units of
// 2^Bw, Bw the warp's largest reference (one per tile: the reference may rise between tiles).
__device__ __forceinline__ void chunk_of_tile(CtaShared &sh, int pb, int k, int lane, float b, float Bw, float a) {
    const float c = warp_sum(a > 0.0f ? a * pow2i(b - Bw) : 0.0f);
    if (lane == 0) {
        sh.pm[pb][k] = c;
        sh.pref[pb][k] = Bw;
    }
}

// Pass 1 of item g over its tiles (target tiles from the target ring; for a pair, draft tiles from
// the draft ring, left there for pass 2). TP / DP: this warp's positions in the two sequences.
// The descriptor's fields are read once, into registers. Vector u of a tile is chunk row
// r = G::kVPT t + u (vectors 480 r .. 480 r + 479 of the slice).
template <int DT>
__device__ __forceinline__ bool stream_pass1(StreamShared &ss, const uint4 *tring, const uint4 *dring,
                                             const Desc &dref, int V, int g, int lo, int nvec, int ntiles,
                                             RingPos &TP, RingPos &DP, int warp, int lane, int tid) {
    using G = Geo<DT>;
    constexpr int E = Elt<DT>::kPerVec;
    CtaShared &sh = ss.c;
    const int nr = desc_rows(dref), greedy = dref.greedy, trunc = dref.trunc, x = dref.x, cut_id = dref.cut_id;
    const uint32_t cut_tau = dref.cut_tau;
    const float s_hi = dref.s_hi, s_lo = dref.s_lo;
    const int wb = g % kWS, pb = g % kPM;
    const float2 shi2 = f2splat(s_hi), slo2 = f2splat(s_lo);
    int xv = (nr == 2 && x >= 0 && x < V) ? x / E - lo : -1;
    if (xv >= nvec) xv = -1;  // another CTA's slice
    // the tile, the thread and the vector of the tile that hold the draft token (none: tile -1)
    const int x_tile = xv >= 0 ? xv / G::kTileVecs : -1;
    const bool x_here = xv >= 0 && (xv % kThreads) == tid;
    const int x_u = xv >= 0 ? (xv % G::kTileVecs) / kThreads : 0;
    const int full_tiles = nvec / G::kTileVecs;  // tiles with no vector past the slice end
    RowAcc At = {-INFINITY, 0.0f}, Ad = {-INFINITY, 0.0f};
    float bt = -INFINITY, bd = -INFINITY;
    int it = INT_MAX, id = INT_MAX, badt = 0, badd = 0;
    bool ok = true;
    const int nt = nr >= 1 ? ntiles : 0;  // a bad shape streams no rows
    for (int t = 0; t < nt; ++t) {
        const int slot = TP.slot, ds = DP.slot;
        ok &= stream_wait(sh, &ss.tfull[slot], TP.par);
        if (nr == 2) ok &= stream_wait(sh, &ss.dfull[ds], DP.par);
        uint4 wt[G::kVPT], wd[G::kVPT];
        const uint4 *ts = tring + static_cast<size_t>(slot) * G::kTileVecs + tid;
        const uint4 *dsrc = dring + static_cast<size_t>(ds) * G::kTileVecs + tid;
        if (t < full_tiles) {  // a whole tile (warp-uniform)
#pragma unroll
            for (int u = 0; u < G::kVPT; ++u) {
                wt[u] = ts[u * kThreads];
                wd[u] = (nr == 2) ? dsrc[u * kThreads] : kNegInfVec<DT>();
            }
        } else {
#pragma unroll
            for (int u = 0; u < G::kVPT; ++u) {
                const bool in = t * G::kTileVecs + u * kThreads + tid < nvec;
                wt[u] = in ? ts[u * kThreads] : kNegInfVec<DT>();
                wd[u] = (nr == 2 && in) ? dsrc[u * kThreads] : kNegInfVec<DT>();
            }
        }
        // the target vectors are in registers: the slot may refill (the draft tile stays for pass 2)
        slot_done(&ss.tempty[slot], lane);
#pragma unroll
        for (int u = 0; u < G::kVPT; ++u)
            if (trunc) mask_cut<DT>(wt[u], lo + t * G::kTileVecs + u * kThreads + tid, cut_tau, cut_id);
        if (greedy) {
#pragma unroll
            for (int u = 0; u < G::kVPT; ++u) {
                const int base = (lo + t * G::kTileVecs + u * kThreads + tid) * E;
                greedy_vec<DT>(wt[u], base, bt, it, badt);
                if (nr == 2) greedy_vec<DT>(wd[u], base, bd, id, badd);
            }
        } else {
            // every share of the tile first (independent exponentials), one vote for the slow path
            if (t == 0) {
                At.b = floorf(Elt<DT>::vmax(wt[0]) * s_hi);
                Ad.b = floorf(Elt<DT>::vmax(wd[0]) * s_hi);
            }
            float a[G::kVPT], q[G::kVPT];
#pragma unroll
            for (int u = 0; u < G::kVPT; ++u) {
                a[u] = vec_share<DT>(wt[u], At.b, shi2, slo2);
                q[u] = (nr == 2) ? vec_share<DT>(wd[u], Ad.b, shi2, slo2) : 0.0f;
            }
            // one test on the tile's total: a NaN, an infinity or a share above 2^64 carries into it
            float ta = a[0], tq = q[0];
#pragma unroll
            for (int u = 1; u < G::kVPT; ++u) {
                ta += a[u];
                tq += q[u];
            }
            if (__any_sync(0xffffffffu, !(ta + tq <= 0x1p66f))) {
#pragma unroll
                for (int u = 0; u < G::kVPT; ++u) {
                    // a later vector's slow path may raise the reference: earlier shares rescale
                    const float b0 = At.b, d0 = Ad.b;
                    a[u] = share_slow<DT>(At, wt[u], s_hi, shi2, slo2);
                    if (nr == 2) q[u] = share_slow<DT>(Ad, wd[u], s_hi, shi2, slo2);
                    for (int w = 0; w < u; ++w) {
                        a[w] *= (At.b == b0) ? 1.0f : pow2i(b0 - At.b);
                        q[w] *= (Ad.b == d0) ? 1.0f : pow2i(d0 - Ad.b);
                    }
                }
                ta = a[0];
                tq = q[0];
#pragma unroll
                for (int u = 1; u < G::kVPT; ++u) {
                    ta += a[u];
                    tq += q[u];
                }
            }
            At.s += ta;
            Ad.s += tq;
            if (nr == 1) {
                const float Bw = warp_max(At.b);
#pragma unroll
                for (int u = 0; u < G::kVPT; ++u) {
                    const int r = t * G::kVPT + u;
                    if (r * kThreads + warp * kWarp < nvec)  // warp-uniform
                        chunk_of_tile(sh, pb, r * kWarps + warp, lane, At.b, Bw, a[u]);
                    else if (lane == 0) {
                        sh.pm[pb][r * kWarps + warp] = 0.0f;
                        sh.pref[pb][r * kWarps + warp] = -INFINITY;
                    }
                }
            }
        }
        if (t == x_tile && x_here) {
            // the thread holding the draft token: (y_t - y_d) s there, as a float pair
            const int u = x_u;
            uint4 xt = wt[0], xd = wd[0];
#pragma unroll
            for (int v = 1; v < G::kVPT; ++v)
                if (u == v) {
                    xt = wt[v];
                    xd = wd[v];
                }
            {
                const int e = x % E;
                const float yt = vec_elem<DT>(xt, e), yd = vec_elem<DT>(xd, e);
                const F2 Ex = f2_mul(f2_add({yt, 0.0f}, {-yd, 0.0f}), {s_hi, s_lo});
                sh.xE[wb][0] = Ex.hi;
                sh.xE[wb][1] = Ex.lo;
                sh.x_flags[wb] = XF_HAS | (yd == -INFINITY ? XF_QZERO : 0) | (yt == -INFINITY ? XF_PZERO : 0);
                sh.x_stamp[wb] = g + 1;
            }
        }
        ring_next<G::kTRing>(TP);
        if (nr == 2) ring_next<G::kDRing>(DP);
    }
    if (nr >= 1) {
        if (greedy) {
            warp_greedy_stats(sh, wb, 0, warp, lane, bt, it, badt);
            if (nr == 2) warp_greedy_stats(sh, wb, 1, warp, lane, bd, id, badd);
        } else {
            warp_row_stats(sh, wb, 0, warp, lane, At.s, At.b);
            if (nr == 2) warp_row_stats(sh, wb, 1, warp, lane, Ad.s, Ad.b);
        }
    }
    return ok;
}

// Pass 2 of pair item m (decision Dref) over its tiles: the target tiles again, from the target
// ring (re-read from L2), the draft tiles where pass 1 left them (draft sequence positions DB ..).
// The arithmetic is that of pass 2 in the rows kernel: where the position rejects, the residual
// max(e_t - lambda e_d, 0) per chunk and S_t min(p, q) = min(e_t, lambda e_d); where it accepts,
// only alpha, min(p, q) = 2^min(y_t s - c_t, y_d s - c_d). Every warp empties both slots.
template <int DT>
__device__ __forceinline__ bool stream_pass2(StreamShared &ss, const uint4 *tring, const uint4 *dring,
                                             const Decision &Dref, int rb, int lo, int nvec, int ntiles,
                                             RingPos &TP, RingPos DB, int warp, int lane, int tid) {
    using G = Geo<DT>;
    constexpr int H = Elt<DT>::kPerVec / 2;
    CtaShared &sh = ss.c;
    const bool work = Dref.status == 0 && Dref.pair && !Dref.greedy;
    const bool resid = work && Dref.kind == SAMPLE_RESIDUAL;
    const int trunc = Dref.trunc, cut_id = Dref.cut_id;
    const uint32_t cut_tau = Dref.cut_tau;
    const float2 shi2 = f2splat(Dref.s_hi), slo2 = f2splat(Dref.s_lo);
    // residual: 2^(y s - B) of both rows and lambda = S_t / S_d (a float pair); accept: the log2
    // normalisers c = integral + fraction
    const float2 nbt = f2splat(-Dref.B_t), nbd = f2splat(-Dref.B_d);
    const float2 nlh = f2splat(-Dref.lam.hi), nll = f2splat(-Dref.lam.lo);
    const float2 nct = f2splat(-Dref.c_t), ncd = f2splat(-Dref.c_d);
    const float2 nctf = f2splat(-Dref.c_tf), ncdf = f2splat(-Dref.c_df);
    const float inv_St = Dref.inv_St;
    float2 acc_a = make_float2(0.0f, 0.0f);
    float my_z = 0.0f;
    bool ok = true;
    if (!work) {
        // the greedy rule or a failed item: nothing to compute, the slots only go back to the rings
        for (int t = 0; t < ntiles; ++t) {
            ok &= stream_wait(sh, &ss.tfull[TP.slot], TP.par);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&ss.tempty[TP.slot]);
                mbar_arrive(&ss.dempty[DB.slot]);
            }
            ring_next<G::kTRing>(TP);
            ring_next<G::kDRing>(DB);
        }
        if (lane == 0) {
            sh.wal[rb][warp] = 0.0f;
            sh.wz[rb][warp] = 0.0f;
        }
        return ok;
    }
    const int full_tiles = nvec / G::kTileVecs;  // tiles with no vector past the slice end
    for (int t = 0; t < ntiles; ++t) {
        const int slot = TP.slot;
        const int ds = DB.slot;  // landed in pass 1, where this warp waited for it
        ok &= stream_wait(sh, &ss.tfull[slot], TP.par);
        uint4 wt[G::kVPT], wd[G::kVPT];
        const uint4 *ts = tring + static_cast<size_t>(slot) * G::kTileVecs + tid;
        const uint4 *dsrc = dring + static_cast<size_t>(ds) * G::kTileVecs + tid;
        if (t < full_tiles) {  // a whole tile (warp-uniform)
#pragma unroll
            for (int u = 0; u < G::kVPT; ++u) {
                wt[u] = ts[u * kThreads];
                wd[u] = dsrc[u * kThreads];
            }
        } else {
#pragma unroll
            for (int u = 0; u < G::kVPT; ++u) {
                const bool in = t * G::kTileVecs + u * kThreads + tid < nvec;
                wt[u] = in ? ts[u * kThreads] : kNegInfVec<DT>();
                wd[u] = in ? dsrc[u * kThreads] : kNegInfVec<DT>();
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&ss.tempty[slot]);
            mbar_arrive(&ss.dempty[ds]);
        }
        {
#pragma unroll
            for (int u = 0; u < G::kVPT; ++u) {
                const int r = t * G::kVPT + u;
                if (trunc) mask_cut<DT>(wt[u], lo + t * G::kTileVecs + u * kThreads + tid, cut_tau, cut_id);
                if (resid) {
                    float2 rv[H], mv[H];
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 yt = Elt<DT>::unpack_one(wt[u], h), yd = Elt<DT>::unpack_one(wd[u], h);
                        const float2 et = ex2x2(exp_arg2(yt, shi2, slo2, nbt));
                        const float2 ed = ex2x2(exp_arg2(yd, shi2, slo2, nbd));
                        const float2 rr = __ffma2_rn(ed, nll, __ffma2_rn(ed, nlh, et));
                        const float2 nq = __fmul2_rn(ed, nlh);  // -lambda_hi * e_d, for min(p, q)
                        rv[h] = make_float2(fmaxf(rr.x, 0.0f), fmaxf(rr.y, 0.0f));
                        mv[h] = make_float2(fminf(et.x, -nq.x), fminf(et.y, -nq.y));
                    }
#pragma unroll
                    for (int st = 1; st < H; st <<= 1)
#pragma unroll
                        for (int h = 0; h + st < H; h += 2 * st) {
                            rv[h] = __fadd2_rn(rv[h], rv[h + st]);
                            mv[h] = __fadd2_rn(mv[h], mv[h + st]);
                        }
                    acc_a = __fadd2_rn(acc_a, mv[0]);
                    if (r * kThreads + warp * kWarp < nvec) {  // warp-uniform
                        const float rs = warp_sum(rv[0].x + rv[0].y);
                        my_z += rs;
                        if (lane == 0) sh.rm[rb][r * kWarps + warp] = rs;
                    } else if (lane == 0) {
                        sh.rm[rb][r * kWarps + warp] = 0.0f;
                    }
                } else {
                    float2 mv[H];
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 at = __fadd2_rn(__ffma2_rn(Elt<DT>::unpack_one(wt[u], h), shi2, nct), nctf);
                        const float2 ad = __fadd2_rn(__ffma2_rn(Elt<DT>::unpack_one(wd[u], h), shi2, ncd), ncdf);
                        mv[h] = make_float2(ex2(fminf(at.x, ad.x)), ex2(fminf(at.y, ad.y)));
                    }
#pragma unroll
                    for (int st = 1; st < H; st <<= 1)
#pragma unroll
                        for (int h = 0; h + st < H; h += 2 * st) mv[h] = __fadd2_rn(mv[h], mv[h + st]);
                    acc_a = __fadd2_rn(acc_a, mv[0]);
                }
            }
        }
        ring_next<G::kTRing>(TP);
        ring_next<G::kDRing>(DB);
    }
    float my_alpha = acc_a.x + acc_a.y;
    if (resid) my_alpha *= inv_St;
    my_alpha = warp_sum(my_alpha);
    if (lane == 0) {
        sh.wal[rb][warp] = my_alpha;
        sh.wz[rb][warp] = my_z;
    }
    return ok;
}

template <int DT>
__global__ void __launch_bounds__(kStreamBlock, 1) spec_stream_kernel(const RowsParams P) {
    using G = Geo<DT>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ StreamShared ss;
    CtaShared &sh = ss.c;
    uint4 *const tring = reinterpret_cast<uint4 *>(smem_raw);
    uint4 *const dring = tring + static_cast<size_t>(G::kTRing) * G::kTileVecs;
    // the exchange slots follow the rings: kNMS exchanges x kMaxCluster records (C used)
    Msg *const slots = reinterpret_cast<Msg *>(dring + static_cast<size_t>(G::kDRing) * G::kTileVecs);

    // hardware warp 0: control; 1 .. 15: data (data thread t = 0 .. 479); 16, 17: producers of
    // the target and draft rings
    const int hw_warp = static_cast<int>(threadIdx.x) / kWarp, lane = static_cast<int>(threadIdx.x) % kWarp;
    const int warp = hw_warp == 0 ? kWarps : hw_warp - 1;
    const int tid = warp * kWarp + lane;
    griddep_launch_dependents();  // the selection kernel may be scheduled behind this grid
    const int C = static_cast<int>(cluster_nctarank());
    const int crank = static_cast<int>(cluster_ctarank());
    const int cid = static_cast<int>(cluster_id_x());
    const int lo = static_cast<int>((static_cast<int64_t>(P.nvec_row) * crank) / C);
    const int nvec = static_cast<int>((static_cast<int64_t>(P.nvec_row) * (crank + 1)) / C) - lo;
    const int ntiles = (nvec + G::kTileVecs - 1) / G::kTileVecs;
    const int nch = ntiles * G::kVPT * kWarps;  // chunks: G::kVPT rows of 15 per tile
    const int ncl = P.nclusters;
    const int nitems = cid < P.total_rows ? (P.total_rows - 1 - cid) / ncl + 1 : 0;

    if (tid == 0) {
        for (int k = 0; k < G::kTRing; ++k) {
            mbar_init(&ss.tfull[k], 1);
            mbar_init(&ss.tempty[k], kWarps);
        }
        for (int k = 0; k < G::kDRing; ++k) {
            mbar_init(&ss.dfull[k], 1);
            mbar_init(&ss.dempty[k], kWarps);
        }
        for (int k = 0; k < kNMS; ++k) mbar_init(&sh.msg_bar[k], 1);
        for (int k = 0; k < kSB; ++k) mbar_init(&sh.stats_bar[k], kWarps);
        for (int k = 0; k < kND; ++k) mbar_init(&sh.dec_bar[k], 1);
        for (int k = 0; k < kPB; ++k) mbar_init(&sh.p2_bar[k], kWarps);
        mbar_init(&sh.draw_bar, 1);
        fence_mbar_init();
        sh.timed_out = 0;
        sh.draw_pending = 0;
        sh.draw_phase = 0;
        for (int k = 0; k < kWS; ++k) sh.x_stamp[k] = 0;
        ss.t_issued = 0;
        ss.d_issued = 0;
    }
    __syncthreads();  // the barriers are initialised
    // every CTA of the cluster must run, its barriers ready, before any remote access
    cluster_arrive();

    if (hw_warp > kWarps) {
        // ================= producers: one ring each ==========================================
        const bool targets = hw_warp == kWarps + 1;
        for (int nb = 0; nb < nitems; nb += kMaxItems) {
            const int nbatch = min(kMaxItems, nitems - nb);
            bar_sync(BAR_SHAPES, kProdBarThreads);  // the batch's shapes are loaded
            if (lane == 0) {
                if (targets)
                    produce_targets<DT>(ss, tring, P, lo, nvec, ntiles, nbatch);
                else
                    produce_drafts<DT>(ss, dring, P, lo, nvec, ntiles, nbatch);
            }
            __syncwarp();
            bar_arrive(BAR_PROD, kProdBarThreads);  // done with the batch's descriptors
        }
        if (lane == 0 && sh.timed_out) {
            // a wait gave up: wait (bounded) for this ring's copies still in flight
            const long long n = targets ? ss.t_issued : ss.d_issued;
            const int nring = targets ? G::kTRing : G::kDRing;
            uint64_t *full = targets ? ss.tfull : ss.dfull;
            for (long long r = max(0LL, n - nring); r < n; ++r)
                mbar_wait_sleep_bounded(&full[r % nring], static_cast<uint32_t>((r / nring) & 1), kSuspendNs,
                                        kMaxWaitTries);
        }
        cluster_wait();
    } else if (warp < kWarps) {
        // ================= data warps: pass 1 of item i, then pass 2 of item i - 1 =============
        RingPos TP = {0, 0u}, DP = {0, 0u};  // this warp's positions in the target and draft sequences
        int g0 = 0;                // the batch's first item, counted over the whole list
        for (int nb = 0; nb < nitems; nb += kMaxItems) {
            const int nbatch = min(kMaxItems, nitems - nb);
            bar_sync(BAR_BATCH, kBlock);  // the control warp has the batch's descriptors
            RingPos db_prev = DP;         // draft position of the previous item's first tile
            for (int i = 0; i < nbatch + kStreamLag; ++i) {
                const RingPos db_cur = DP;
                if (i < nbatch) {
                    const int g = g0 + i;
                    if (!stream_pass1<DT>(ss, tring, dring, sh.desc[i], P.V, g, lo, nvec, ntiles, TP, DP, warp, lane,
                                          tid))
                        sh.timed_out = 1;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.stats_bar[g % kSB]);
                }
                if (i >= kStreamLag) {
                    const int m = i - kStreamLag, gm = g0 + m;
                    if (!stream_wait(sh, &sh.dec_bar[gm % kND], static_cast<uint32_t>((gm / kND) & 1)))
                        sh.timed_out = 1;
                    if (ss.rows[m] == 2) {
                        if (!stream_pass2<DT>(ss, tring, dring, sh.dec[gm % kND], gm % kRM, lo, nvec, ntiles, TP,
                                              db_prev, warp, lane, tid))
                            sh.timed_out = 1;
                    } else if (lane == 0) {
                        sh.wal[gm % kRM][warp] = 0.0f;
                        sh.wz[gm % kRM][warp] = 0.0f;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.p2_bar[gm % kPB]);
                }
                db_prev = db_cur;
            }
            g0 += nbatch;
        }
        cluster_wait();
    } else {
        // ================= control warp: exchanges, decisions, results, draws =================
        if (lane == 0 && nitems > 0) {
            // the first target row's slice into L2 while the descriptors load
            const size_t row_bytes = static_cast<size_t>(P.nvec_row) * 16;
            bulk_prefetch_l2(static_cast<const unsigned char *>(P.target) +
                                 static_cast<size_t>(cid) * row_bytes + static_cast<size_t>(lo) * 16,
                             static_cast<uint32_t>(nvec) * 16);
        }
        int e = 0;   // exchanges so far
        int g0 = 0;  // the batch's first item
        for (int nb = 0; nb < nitems; nb += kMaxItems) {
            const int nbatch = min(kMaxItems, nitems - nb);
            load_batch_shapes(sh, P, cid, nb, nbatch, lane);
            for (int s2 = lane; s2 < nbatch; s2 += kWarp) ss.rows[s2] = desc_rows(sh.desc[s2]);
            __syncwarp();
            bar_arrive(BAR_SHAPES, kProdBarThreads);  // the producers may start the batch's copies
            load_batch_values(sh, P, nbatch, lane);
            __syncwarp();
            bar_arrive(BAR_BATCH, kBlock);
            const int e0 = e;  // the exchange of the batch's item i is e0 + i
            // exchange j carries item j's record (j < nbatch) and the totals of item j - 2 (its pass
            // 2 ran before pass 1 of item j); two draining exchanges follow the batch's last item
            for (int j = 0; j < nbatch + kStreamLag + 1; ++j) {
                const int g = g0 + j, m = j - kStreamLag - 1;
                int nr = 0, greedy = 0;
                if (j < nbatch) {
                    nr = ss.rows[j];
                    greedy = sh.desc[j].greedy;
                    if (!stream_wait(sh, &sh.stats_bar[g % kSB], static_cast<uint32_t>((g / kSB) & 1)))
                        sh.timed_out = 1;
                }
                if (m >= 0 && !stream_wait(sh, &sh.p2_bar[(g0 + m) % kPB], static_cast<uint32_t>(((g0 + m) / kPB) & 1)))
                    sh.timed_out = 1;
                __syncwarp();
                uint4 rec[3];
                build_record(sh, greedy, nr, g, m >= 0 ? g0 + m : -1, lane, rec);
                if (e == 0) cluster_wait();  // the peers run and their barriers are ready
                Msg *const here = slots + (e % kNMS) * kMaxCluster;
                push_record(rec, here, &sh.msg_bar[e % kNMS], crank, C, lane);
                if (lane == 0) mbar_arrive_expect_tx(&sh.msg_bar[e % kNMS], static_cast<uint32_t>(C * kMsgBytes));
                complete_draw<DT>(sh, P, lo, lane);  // the draw fetched at the previous exchange
                if (!stream_wait(sh, &sh.msg_bar[e % kNMS], static_cast<uint32_t>((e / kNMS) & 1)))
                    sh.timed_out = 1;
                __syncwarp();
                if (j < nbatch) {
                    decide_item(sh, here, sh.desc[j], nr, g, C, P, lane);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.dec_bar[g % kND]);
                }
                if (m >= 0) {
                    const FinState f = finalize_head(sh, P, g0 + m, slots + ((e0 + m) % kNMS) * kMaxCluster, here,
                                                     C, crank, lane);
                    if (f.owner == crank) draw_chunk<DT>(sh, P, g0 + m, f, lane, nch, lo, nvec);
                }
                ++e;
            }
            complete_draw<DT>(sh, P, lo, lane);  // the batch's last draw
            // the producers are done with this batch's descriptors before the next batch's load
            bar_sync(BAR_PROD, kProdBarThreads);
            g0 += nbatch;
        }
        if (nitems == 0) cluster_wait();
    }
    __syncwarp();
    cluster_sync_all();  // no CTA leaves while another may still write into its shared memory
}

}  // namespace spec
