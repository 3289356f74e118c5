// spec_rows_kernel: see spec_rows.cuh for the design. Included once, by spec_verify.cu.
#pragma once

#include "spec_rows.cuh"

namespace spec {

// Static shared state of one CTA. Dynamic shared memory holds the row ring (kRing slices) and the
// exchange slots (kNMS x C records, written by every CTA of the cluster).
struct CtaShared {
    uint64_t full[kRing];                 // a ring slot's bulk copy has landed
    uint64_t draw_bar;                    // the draw chunk's bulk copy has landed
    uint64_t msg_bar[kNMS];               // all C records of an exchange have arrived
    uint64_t stats_bar[kSB];              // pass 1 of an item (or, held rows, the drain after the
                                          // last pass 2) done: one arrival per data warp
    uint64_t p2_bar[kPB];                 // kLag > 0: pass 2 of an item done (one arrival per data warp)
    uint64_t dec_bar[kND];                // the decision of an item is ready (control warp)
    Desc desc[kMaxItems];
    int32_t roff[kRoffMax];               // row_off, staged once when B + 1 entries fit
    WarpStat ws[kWS][kWarps];             // per-warp row statistics, by item % kWS
    float xE[kWS][2];                     // (y_t - y_d) s at the draft token, from the thread holding it
    int32_t x_flags[kWS];                 // XF_* bits of the draft token (XF_HAS when held here)
    int32_t x_stamp[kWS];                 // item number + 1 when this CTA holds the draft token
    float wal[kRM][kWarps];               // per-warp alpha partials, by item % kRM
    float wz[kRM][kWarps];                // per-warp residual mass (units 2^B_t), by item % kRM
    float rm[kRM][kMaxChunks];            // residual chunk sums (units 2^B_t), by item % kRM
    float pm[kPM][kMaxChunks];            // bonus-row chunk sums (units 2^pref), by item % kPM
    float pref[kPM][kMaxChunks];          // their integral reference exponents (one per chunk)
    Decision dec[kND];                    // by item % kND
    uint4 draw_buf[2][kChunkVecs];        // target / draft chunk of the pending draw
    int32_t timed_out;
    long long prod_issued;                // the producer (see release_row): rows copied; batch cursor
    int32_t prod_item, prod_row;
    int32_t free_cnt[kRing];              // data warps done with the row in each slot
    // the pending draw (owner CTA only)
    int32_t draw_pending, draw_chunk, draw_count, draw_clamped, draw_kind, draw_item, draw_dec;
    float draw_lt, draw_unit, draw_bg, draw_invZ;
    uint32_t draw_phase;
};

// Items of cluster `cid`: cid, cid + ncl, cid + 2 ncl, ... Batch `nb` holds list entries
// [nb, nb + nbatch). Every CTA of the cluster computes the same descriptors. Control warp, in two
// steps: the shapes (which request and position, the draft row), enough to issue the row copies,
// then the per-item values (temperature, draws, draft token).
__device__ void load_batch_shapes(CtaShared &sh, const RowsParams &P, int cid, int nb, int nbatch, int lane) {
    // row_off into shared memory once, eight independent loads per lane in flight
    const bool staged = P.B + 1 <= kRoffMax;
    if (nb == 0 && staged) {
        for (int base = 0; base <= P.B; base += 8 * kWarp) {
            int v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = base + k * kWarp + lane;
                v[k] = (i <= P.B) ? __ldg(P.row_off + i) : 0;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = base + k * kWarp + lane;
                if (i <= P.B) sh.roff[i] = v[k];
            }
        }
    }
    for (int s = lane; s < kMaxItems; s += kWarp) {
        Desc &d = sh.desc[s];
        d.item = cid + (nb + s) * P.nclusters;
        d.req = -1;
        d.pos = d.K = d.drow = -1;
        d.pair = 0;
        d.status = SPEC_REQ_BAD_SHAPE;  // until a request claims the item
        d.x = -1;
        d.greedy = 0;
        d.s_hi = d.s_lo = 0.0f;
        d.u_acc = d.u_s = {0.0f, 0.0f};
        d.cut_tau = 0u;
        d.cut_id = INT_MAX;
        d.trunc = 0;
    }
    __syncwarp();
    // every request writes the descriptors of its rows that belong to this batch
    const int first = cid + nb * P.nclusters;
    const int last = cid + (nb + nbatch) * P.nclusters;  // exclusive
    for (int i = lane; i < P.B; i += kWarp) {
        const int r0 = staged ? sh.roff[i] : __ldg(P.row_off + i);
        const int r1 = staged ? sh.roff[i + 1] : __ldg(P.row_off + i + 1);
        int lo = max(max(r0, first), 0);
        lo += ((cid - lo) % P.nclusters + P.nclusters) % P.nclusters;  // next item of this cluster
        const int hi = min(min(r1, last), P.total_rows);
        for (int it = lo; it < hi; it += P.nclusters) {
            const int s = (it - cid) / P.nclusters - nb;
            if (s < 0 || s >= nbatch) continue;
            Desc &d = sh.desc[s];
            const int K = r1 - r0 - 1, j = it - r0, dr = r0 - i + j;
            int status = 0;
            if (K < 0 || K > P.K_max || j < 0 || j > K || r1 > P.total_rows ||
                (j < K && (dr < 0 || dr >= P.total_rows - P.B)))
                status = SPEC_REQ_BAD_SHAPE;
            d.req = i;
            d.pos = j;
            d.K = K;
            d.drow = dr;
            d.pair = (status == 0 && j < K) ? 1 : 0;
            d.status = status;
            d.x = r1;  // the request's end row, for the frontier draw
        }
    }
    __syncwarp();
}

__device__ void load_batch_values(CtaShared &sh, const RowsParams &P, int nbatch, int lane) {
    // per item: temperature, draws and draft token (loads issued in parallel, one thread each)
    for (int s = lane; s < nbatch; s += kWarp) {
        Desc &d = sh.desc[s];
        int status = d.status;
        const int r1 = d.x;
        d.x = -1;
        // every load of the item at once (the shape decides which exist)
        const bool shaped = status == 0 && d.req >= 0;
        const float T = (d.req >= 0) ? (P.temperature ? __ldg(P.temperature + d.req) : P.temperature_scalar) : 1.0f;
        const double ua = shaped ? __ldg(P.uniforms + d.item) : 0.0;
        const double us = shaped ? __ldg(P.uniforms + r1 - 1) : 0.0;
        const int xt = (shaped && d.pair) ? __ldg(P.draft_tokens + d.drow) : -1;
        const int2 cut = (shaped && P.trunc) ? __ldg(P.trunc + d.item) : make_int2(0, INT_MAX);
        const float tp = (d.req >= 0 && P.top_p) ? __ldg(P.top_p + d.req) : 1.0f;
        if (!(T >= 0.0f) || isinf(T) || isnan(tp)) status |= SPEC_REQ_BAD_PARAM;
        d.cut_tau = static_cast<uint32_t>(cut.x);
        d.cut_id = cut.y;
        d.trunc = (cut.x != 0 || cut.y != INT_MAX) ? 1 : 0;
        d.greedy = (T == 0.0f) ? 1 : 0;
        F2 sv = {0.0f, 0.0f};
        if (T > 0.0f && !isinf(T)) sv = f2_div({kLog2eHi, kLog2eLo}, {T, 0.0f});
        if (sv.hi > 0.0f && sv.lo < 0.0f) {
            // s_hi moved toward zero so that s_lo > 0: a -inf logit then gives -inf in both terms
            // of exp_arg2 (a negative s_lo would make it NaN)
            const float down = __uint_as_float(__float_as_uint(sv.hi) - 1u);
            sv.lo += sv.hi - down;
            sv.hi = down;
        }
        d.s_hi = sv.hi;
        d.s_lo = fmaxf(sv.lo, 1.401298464e-45f);
        if (status == 0 && d.req >= 0) {
            d.u_acc = d2f2(ua);
            d.u_s = d2f2(us);
            if (d.pair) d.x = xt;
        }
        d.status = status;
    }
    __syncwarp();
}

// Rows an item streams through the ring: its target row, and its draft row for a pair. Only a bad
// shape has none (its rows may not exist); a bad temperature streams them and discards the
// result, so that the ring order is fixed before the temperatures are read.
__device__ __forceinline__ int desc_rows(const Desc &d) {
    return (d.status & SPEC_REQ_BAD_SHAPE) ? 0 : (d.pair ? 2 : 1);
}

// Data thread 0: issue the bulk copies of the cluster's row sequence up to row `limit`
// (exclusive). The sequence runs through the batch's items in order: target row, then draft row
// for a pair. With kLag > 0 pass 2 reads the rows again a few items later: the copies keep them in
// L2 (evict-last); otherwise each row is read once (evict-first).
__device__ __forceinline__ void produce_rows(CtaShared &sh, uint4 *ring, const RowsParams &P, int slice_max, int lo,
                                             int nvec, int nbatch, long long &issued, long long limit,
                                             int &cur_item, int &cur_row) {
    const size_t row_bytes = static_cast<size_t>(P.nvec_row) * 16;
    const uint64_t pol = kLag > 0 ? policy_evict_last() : policy_evict_first();
    while (issued < limit && cur_item < nbatch) {
        const Desc &d = sh.desc[cur_item];
        if (cur_row >= desc_rows(d)) {
            ++cur_item;
            cur_row = 0;
            continue;
        }
        const int slot = static_cast<int>(issued % kRing);
        const unsigned char *src =
            (cur_row == 0) ? static_cast<const unsigned char *>(P.target) + static_cast<size_t>(d.item) * row_bytes
                           : static_cast<const unsigned char *>(P.draft) + static_cast<size_t>(d.drow) * row_bytes;
        const uint32_t bytes = static_cast<uint32_t>(nvec) * 16;
        mbar_arrive_expect_tx(&sh.full[slot], bytes);
        bulk_g2s(ring + static_cast<size_t>(slot) * slice_max, src + static_cast<size_t>(lo) * 16, bytes,
                 &sh.full[slot], pol);
        ++issued;
        ++cur_row;
    }
}

// A data warp is done with ring row `row` (its lanes' reads of the slot are complete): the last
// of the 15 warps to get here refills the slot, issuing the copy of row + kRing. No warp waits
// for another; successive releases of a slot are ordered by the copies they issue (a warp reaches
// row + kRing only after the copy that the last release issued has landed).
__device__ __forceinline__ void release_row(CtaShared &sh, uint4 *ring, const RowsParams &P, int slice_max, int lo,
                                            int nvec, int nbatch, long long row, int lane) {
    __syncwarp();
    if (lane == 0) {
        const int slot = static_cast<int>(row % kRing);
        __threadfence_block();
        if (atomicAdd(&sh.free_cnt[slot], 1) == kWarps - 1) {
            sh.free_cnt[slot] = 0;
            __threadfence_block();
            fence_proxy_async_smem();
            produce_rows(sh, ring, P, slice_max, lo, nvec, nbatch, sh.prod_issued, row + 1 + kRing, sh.prod_item,
                         sh.prod_row);
        }
    }
}

// Whether warp `warp` has any vector v of the slice (its 32 vectors start at v * 480 + 32 warp):
// warps past the slice end skip the vector altogether (a warp-uniform branch).
__device__ __forceinline__ bool warp_has(int v, int warp, int nvec) { return v * kThreads + warp * kWarp < nvec; }

// A row of the item as pass 1 sees it, in registers: vector v of thread t is vector t + 480 v of
// the slice (a warp covers 32 contiguous vectors, a chunk).
template <int NVT>
struct RegRow {
    const uint4 (&vv)[NVT];
    __device__ __forceinline__ uint4 operator()(int v) const { return vv[v]; }
};
// The draft row as pass 1 sees it: in its ring slot, vector v of thread t at t + 480 v; past the
// slice end, -inf.
template <int DT>
struct SmemRow {
    const uint4 *src;
    int tid, nvec;
    __device__ __forceinline__ uint4 operator()(int v) const {
        const int vi = tid + v * kThreads;
        return vi < nvec ? src[vi] : kNegInfVec<DT>();
    }
};

// The sums of 2^(y*s - b) over a thread's vectors of one row, b an integral reference.
// Fast path: b comes from the thread's first vector alone, so no exponential waits on a running
// max; a larger value later in the row only makes its term larger than 1. Should the first vector
// be all -inf or the sum exceed 2^64 (so that every term later taken against the row's reference
// stays far inside float range; a +inf or NaN logit lands here too), the exact path takes b from
// the thread's max over all its vectors (a first sweep) and sums again.
// CHUNKS: also the per-vector sums, at the same reference.
// The exact path of the sums: b from the thread's max over all its vectors, then the sums.
template <int DT, int NVT, bool CHUNKS, class Row>
__device__ __forceinline__ float exact_sums(const Row &row, float s_hi, float2 shi2, float2 slo2, int warp, int nvec,
                                            float &b, float (&sv)[CHUNKS ? NVT : 1]) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    float m = -INFINITY;
#pragma unroll
    for (int v = 0; v < NVT; ++v)
        if (warp_has(v, warp, nvec)) m = fmaxf(m, Elt<DT>::vmax(row(v)));
    // an all -inf thread gets reference 0: its sum is 0 (or NaN if a NaN hides in it)
    b = (m == -INFINITY) ? 0.0f : floorf(m * s_hi);
    const float2 nb2 = f2splat(-b);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int v = 0; v < NVT; ++v) {
        if (CHUNKS) sv[CHUNKS ? v : 0] = 0.0f;
        if (!warp_has(v, warp, nvec)) continue;
        const uint4 w = row(v);
        float2 a = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int h = 0; h < H; ++h) a = __fadd2_rn(a, ex2x2(exp_arg2(Elt<DT>::unpack_one(w, h), shi2, slo2, nb2)));
        if (CHUNKS) sv[CHUNKS ? v : 0] = a.x + a.y;
        acc = __fadd2_rn(acc, a);
    }
    return acc.x + acc.y;
}

template <int DT, int NVT, bool CHUNKS, class Row>
__device__ __forceinline__ float sweep_sums(const Row &row, float s_hi, float2 shi2, float2 slo2, int warp, int nvec,
                                            float &b, float (&sv)[CHUNKS ? NVT : 1]) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    // an all -inf first vector gives b = -inf, hence inf or NaN sums: the exact path below
    b = floorf((warp_has(0, warp, nvec) ? Elt<DT>::vmax(row(0)) : -INFINITY) * s_hi);
    float s;
    {
        const float2 nb2 = f2splat(-b);
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int v = 0; v < NVT; ++v) {
            if (CHUNKS) sv[CHUNKS ? v : 0] = 0.0f;
            if (!warp_has(v, warp, nvec)) continue;
            const uint4 w = row(v);
            float2 a = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int h = 0; h < H; ++h) a = __fadd2_rn(a, ex2x2(exp_arg2(Elt<DT>::unpack_one(w, h), shi2, slo2, nb2)));
            if (CHUNKS) sv[CHUNKS ? v : 0] = a.x + a.y;
            acc = __fadd2_rn(acc, a);
        }
        s = acc.x + acc.y;
    }
    // the exact path, for the whole warp when any of its threads needs it (a warp-uniform branch:
    // a per-thread one costs the common path twice its time on this compiler)
    if (__any_sync(0xffffffffu, !(s <= 0x1p64f))) s = exact_sums<DT, NVT, CHUNKS>(row, s_hi, shi2, slo2, warp, nvec, b, sv);
    return s;
}

// Pass-1 statistics of one row: each thread's sum at its integral reference (sweep_sums), then
// a warp combines its threads by exact powers of two (one max and one sum across the lanes). For
// a row that a draw from p may need (CHUNKS), also the per-chunk sums (chunk (v, warp), units
// 2^B_w with B_w the warp's reference).
template <int DT, int NVT, bool CHUNKS, class Row>
__device__ __forceinline__ void row_stats(const Row &row, CtaShared &sh, int wb, int r, int pb, const Desc &d, int lo,
                                          int nvec, int warp, int lane, int tid) {
    constexpr int E = Elt<DT>::kPerVec;
    constexpr int H = E / 2;
    if (d.greedy) {
        // smallest index attaining the max; NaN / +inf make the row invalid. The running max
        // picks the thread's first vector attaining it, the element is found in that vector.
        float best = -INFINITY;
        int vbest = -1, bad = 0;
#pragma unroll
        for (int v = 0; v < NVT; ++v) {
            if (!warp_has(v, warp, nvec)) continue;
            const uint4 w = row(v);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const float2 y = Elt<DT>::unpack_one(w, h);
                bad |= (y.x != y.x) || (y.x == INFINITY) || (y.y != y.y) || (y.y == INFINITY);
            }
            const float mv = Elt<DT>::vmax(w);
            if (mv > best) {
                best = mv;
                vbest = v;
            }
        }
        int bidx = INT_MAX;
#pragma unroll
        for (int v = 0; v < NVT; ++v)
            if (v == vbest) {
                const uint4 w = row(v);
                for (int e = E - 1; e >= 0; --e)
                    if (vec_elem<DT>(w, e) == best) bidx = (lo + tid + v * kThreads) * E + e;
            }
        const float wbest = warp_max(best);
        const int widx = warp_min_i32(best == wbest ? bidx : INT_MAX);
        const int wbad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
            sh.ws[wb][warp].b[r] = wbad ? INFINITY : wbest;
            sh.ws[wb][warp].a[r] = wbad ? -1 : widx;
        }
        return;
    }
    const float2 shi2 = f2splat(d.s_hi), slo2 = f2splat(d.s_lo);
    float sv[CHUNKS ? NVT : 1];
    float b;
    float s = sweep_sums<DT, NVT, CHUNKS>(row, d.s_hi, shi2, slo2, warp, nvec, b, sv);
    const bool ok = s > 0.0f && !isinf(s);  // NaN, inf and empty are not ok
    const int bad = __any_sync(0xffffffffu, !(s >= 0.0f) || isinf(s));
    const float Bw = warp_max(ok ? b : -INFINITY);
    const float scale = ok ? pow2i(b - Bw) : 0.0f;
    const float Sw = warp_sum(ok ? s * scale : 0.0f);
    if (CHUNKS) {
#pragma unroll
        for (int v = 0; v < NVT; ++v) {
            const float c = warp_sum(ok ? sv[CHUNKS ? v : 0] * scale : 0.0f);
            if (lane == 0) sh.pm[pb][v * kWarps + warp] = c;
        }
    }
    if (lane == 0) {
        if (CHUNKS)
#pragma unroll
            for (int v = 0; v < NVT; ++v) sh.pref[pb][v * kWarps + warp] = Bw;
        // a reference beyond 2^28 (logits far outside any float32 softmax) reads as invalid
        const bool inval = bad || (Sw > 0.0f && !(fabsf(Bw) < 0x1p28f));
        sh.ws[wb][warp].a[r] = (Sw > 0.0f && !inval) ? static_cast<int>(Bw) : kNoRef;
        sh.ws[wb][warp].b[r] = inval ? NAN : Sw;
    }
}

// A warp's statistics of one row from each thread's sum s at its reference b.
__device__ __forceinline__ void warp_row_stats(CtaShared &sh, int wb, int r, int warp, int lane, float s, float b) {
    const bool ok = s > 0.0f && !isinf(s);  // NaN, inf and empty are not ok
    const int bad = __any_sync(0xffffffffu, !(s >= 0.0f) || isinf(s));
    const float Bw = warp_max(ok ? b : -INFINITY);
    const float Sw = warp_sum(ok ? s * pow2i(b - Bw) : 0.0f);
    if (lane == 0) {
        // a reference beyond 2^28 (logits far outside any float32 softmax) reads as invalid
        const bool inval = bad || (Sw > 0.0f && !(fabsf(Bw) < 0x1p28f));
        sh.ws[wb][warp].a[r] = (Sw > 0.0f && !inval) ? static_cast<int>(Bw) : kNoRef;
        sh.ws[wb][warp].b[r] = inval ? NAN : Sw;
    }
}

// Pass 1 of a pair under Rule 2: the target row in registers, the draft row in its ring slot, in
// one loop over both (the draft's loads and the target's exponentials hide each other's latency;
// both rows in registers would not fit 64 registers). References from each thread's first vectors
// (see sweep_sums).
template <int DT, int NVT>
__device__ __forceinline__ void pair_stats(const uint4 (&vt)[NVT], const SmemRow<DT> &rd, CtaShared &sh, int wb,
                                           const Desc &d, int nvec, int warp, int lane) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    const float2 shi2 = f2splat(d.s_hi), slo2 = f2splat(d.s_lo);
    const bool h0 = warp_has(0, warp, nvec);
    float bt = floorf((h0 ? Elt<DT>::vmax(vt[0]) : -INFINITY) * d.s_hi);
    float bd = floorf((h0 ? Elt<DT>::vmax(rd(0)) : -INFINITY) * d.s_hi);
    float st, sd;
    {
        const float2 nbt = f2splat(-bt), nbd = f2splat(-bd);
        float2 ta = make_float2(0.0f, 0.0f), qa = ta;
#pragma unroll
        for (int v = 0; v < NVT; ++v) {
            if (!warp_has(v, warp, nvec)) continue;
            const uint4 wt = vt[v], wd = rd(v);
#pragma unroll
            for (int h = 0; h < H; ++h) {
                ta = __fadd2_rn(ta, ex2x2(exp_arg2(Elt<DT>::unpack_one(wt, h), shi2, slo2, nbt)));
                qa = __fadd2_rn(qa, ex2x2(exp_arg2(Elt<DT>::unpack_one(wd, h), shi2, slo2, nbd)));
            }
        }
        st = ta.x + ta.y;
        sd = qa.x + qa.y;
    }
    float none[1];
    if (__any_sync(0xffffffffu, !(st <= 0x1p64f)))
        st = exact_sums<DT, NVT, false>(RegRow<NVT>{vt}, d.s_hi, shi2, slo2, warp, nvec, bt, none);
    if (__any_sync(0xffffffffu, !(sd <= 0x1p64f)))
        sd = exact_sums<DT, NVT, false>(rd, d.s_hi, shi2, slo2, warp, nvec, bd, none);
    warp_row_stats(sh, wb, 0, warp, lane, st, bt);
    warp_row_stats(sh, wb, 1, warp, lane, sd, bd);
}

// Sum over the 16-lane half of the warp (xor steps 8, 4, 2, 1; each half sums its own lanes).
__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float half_max(float v) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// Greedy rule: the larger logit, ties to the smaller index, over lanes xor o (o < n).
__device__ __forceinline__ void half_argmax(float &gm, int &ga, int n) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
        if (o < n) {
            const float og = __shfl_xor_sync(0xffffffffu, gm, o);
            const int oa = __shfl_xor_sync(0xffffffffu, ga, o);
            if (og > gm || (og == gm && oa < ga)) {
                gm = og;
                ga = oa;
            }
        }
}

// Control warp: this CTA's record for item g, in registers (the same in every lane): its row
// statistics over the data warps (row r in lanes 16r .. 16r + 14, lane 16r + w taking warp w:
// the max reference, then the sums scaled to it by exact powers of two), the ratio exponent at
// the draft token if this CTA holds it, and the totals of item m (its alpha share in the row-0
// lanes and its residual mass in the row-1 lanes, summed alongside; m < 0: none). nr = 0: no item
// (a draining exchange).
__device__ __forceinline__ void build_record(CtaShared &sh, int greedy, int nr, int g, int m, int lane,
                                             uint4 (&rec)[3]) {
    const int wb = g % kWS, r = lane >> 4, w = lane & 15;
    const bool use = w < kWarps && r < nr;
    const WarpStat &st = sh.ws[wb][use ? w : 0];
    int a = use ? st.a[r] : (greedy ? INT_MAX : kNoRef);
    float b = use ? st.b[r] : (greedy ? -INFINITY : 0.0f);
    float t = 0.0f;
    if (m >= 0 && w < kWarps) t = (r == 0) ? sh.wal[m % kRM][w] : sh.wz[m % kRM][w];
    if (greedy) {
        half_argmax(b, a, 16);
    } else {
        int Bm = a;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) Bm = max(Bm, __shfl_xor_sync(0xffffffffu, Bm, o));
        // no mass: 0 (a NaN sum stays NaN)
        b = (a == kNoRef) ? b * 0.0f : b * pow2_int(a - Bm);
        a = Bm;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
        if (!greedy) b += __shfl_xor_sync(0xffffffffu, b, o);
        t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    const int a1 = __shfl_sync(0xffffffffu, a, 16);
    const float b1 = __shfl_sync(0xffffffffu, b, 16);
    const float alpha = __shfl_sync(0xffffffffu, t, 0), Z = __shfl_sync(0xffffffffu, t, 16);
    const bool hx = nr > 0 && sh.x_stamp[wb] == g + 1;
    const int flags = (hx ? sh.x_flags[wb] : 0) | (sh.timed_out ? XF_TMO : 0);
    rec[0] = make_uint4(static_cast<uint32_t>(a), static_cast<uint32_t>(a1), __float_as_uint(b), __float_as_uint(b1));
    rec[1] = make_uint4(__float_as_uint(hx ? sh.xE[wb][0] : 0.0f), __float_as_uint(hx ? sh.xE[wb][1] : 0.0f),
                        static_cast<uint32_t>(flags), 0u);
    rec[2] = make_uint4(__float_as_uint(alpha), __float_as_uint(Z), 0u, 0u);
}

// Control warp, after the exchange of item g: combine the C records (lanes 0-15 take row 0,
// lanes 16-31 row 1, one lane per CTA, in CTA order; C is a power of two, so log2(C) butterfly
// steps combine them: the max reference, then the sums scaled to it by exact powers of two) and
// decide the accept test. Every lane then computes the whole scalar tail (the test, lambda, the
// log2 of both normalisers): independent chains that the compiler interleaves. Every CTA runs the
// same reductions on the same records, so all reach the same decision.
__device__ __forceinline__ void decide_item(CtaShared &sh, const Msg *M, const Desc &d, int nr, int g, int C,
                                            const RowsParams &P, int lane) {
    const int r = lane >> 4, c = lane & 15;
    const bool on = c < C && r < nr;
    const Msg &m = M[c];
    const int4 fx = *reinterpret_cast<const int4 *>(&m.E_hi);
    const int myflags = (r == 0 && c < C) ? fx.z : 0;
    const unsigned hx = __ballot_sync(0xffffffffu, myflags & XF_HAS);
    int flags = myflags;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) flags |= __shfl_xor_sync(0xffffffffu, flags, o);
    flags = __shfl_sync(0xffffffffu, flags, 0);
    const int lx = hx ? __ffs(hx) - 1 : 0;
    const float E_hi = __shfl_sync(0xffffffffu, __int_as_float(fx.x), lx);
    const float E_lo = __shfl_sync(0xffffffffu, __int_as_float(fx.y), lx);
    int a = on ? m.a[r] : (d.greedy ? INT_MAX : kNoRef);
    float b = on ? m.b[r] : (d.greedy ? -INFINITY : 0.0f);
    if (d.greedy) {
        half_argmax(b, a, C);
    } else {
        int Bm = a;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
            if (o < C) Bm = max(Bm, __shfl_xor_sync(0xffffffffu, Bm, o));
        b = (a == kNoRef) ? b * 0.0f : b * pow2_int(a - Bm);  // a NaN sum stays NaN
        a = Bm;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
            if (o < C) b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    // rows 0 and 1 from lanes 0 and 16, to every lane
    const int B0 = __shfl_sync(0xffffffffu, a, 0), B1 = __shfl_sync(0xffffffffu, a, 16);
    const float S0 = __shfl_sync(0xffffffffu, b, 0), S1 = __shfl_sync(0xffffffffu, b, 16);
    const int ga0 = B0, ga1 = B1;
    const float gm0 = S0, gm1 = S1;
    const bool tmo = (flags & XF_TMO) != 0;
    const int am0 = (nr >= 1 && ga0 >= 0 && gm0 != -INFINITY) ? ga0 : -1;
    const int am1 = (nr >= 2 && ga1 >= 0 && gm1 != -INFINITY) ? ga1 : -1;
    // a NaN sum marks a row that holds a NaN / +inf
    const float B_t = (nr >= 1 && B0 != kNoRef && !isnan(S0)) ? static_cast<float>(B0) : NAN;
    const float B_d = (nr >= 2 && B1 != kNoRef && !isnan(S1)) ? static_cast<float>(B1) : NAN;
    const float S_t = (nr >= 1) ? S0 : 0.0f, S_d = (nr >= 2) ? S1 : 0.0f;
    // the status, the same in every lane; row validity is reported together with a bad proposal
    // (both are preconditions)
    int status = d.status | (tmo ? REQ_TIMEOUT : 0);
    if (!(status & (SPEC_REQ_BAD_SHAPE | SPEC_REQ_BAD_PARAM | REQ_TIMEOUT))) {
        if (d.greedy) {
            if (am0 < 0 || (d.pair && am1 < 0)) status |= SPEC_REQ_BAD_LOGITS;
            if (d.pair && (d.x < 0 || d.x >= P.V)) status |= SPEC_REQ_BAD_PROPOSAL;
        } else {
            const bool ok_t = isfinite(B_t) && S_t > 0.0f && isfinite(S_t);
            const bool ok_d = !d.pair || (isfinite(B_d) && S_d > 0.0f && isfinite(S_d));
            if (!ok_t || !ok_d) status |= SPEC_REQ_BAD_LOGITS;
            // q(x) == 0 is a bad proposal for Rule 2 (checked before any draw)
            if (d.pair && (d.x < 0 || d.x >= P.V || (flags & XF_QZERO))) status |= SPEC_REQ_BAD_PROPOSAL;
        }
    }
    // the scalar tail in every lane (values of rows that are not there are computed and unused)
    const float inv_St = rcp_approx(S_t);
    const F2 lam = f2_div({S_t, 0.0f}, {S_d, 0.0f});
    const float2 ct = log2_split({S_t, 0.0f}, B_t), cd = log2_split({S_d, 0.0f}, B_d);
    int accept = 0, kind = SAMPLE_NONE, argmax_t = -1;
    float rho = 0.0f, alpha_g = 0.0f;
    if (status == 0) {
        if (d.greedy) {
            argmax_t = am0;
            if (d.pair) {
                accept = (d.x == am0);
                rho = accept ? 1.0f : 0.0f;
                alpha_g = (am0 == am1) ? 1.0f : 0.0f;
            }
        } else if (d.pair) {
            // rho = p(x)/q(x) = 2^E * S_d/S_t with E = (y_t - y_d) s - (B_t - B_d), in float
            // pairs; 2^E from ex2 of its fraction and an exact power of two
            if (!(flags & XF_PZERO)) {
                // (y_t - y_d) s came with the record of the CTA holding the draft token
                const F2 Ex = f2_add({E_hi, E_lo}, {-(B_t - B_d), 0.0f});
                const float nn = floorf(Ex.hi);
                const float f = (Ex.hi - nn) + Ex.lo;
                const F2 ratio = f2_div({S_d, 0.0f}, {S_t, 0.0f});
                const float mm = ex2(f) * (ratio.hi + ratio.lo);
                if (nn > 254.0f) {
                    rho = INFINITY;
                } else if (nn >= -252.0f) {
                    const float h = floorf(0.5f * nn);
                    rho = mm * pow2i(h) * pow2i(nn - h);
                }
            }
            accept = (rho > 0.0f) && !f2_gt(d.u_acc, {rho, 0.0f});
            if (!accept) kind = SAMPLE_RESIDUAL;
        } else {
            kind = SAMPLE_P;
        }
    }
    if (lane == 0) {
        Decision &D = sh.dec[g % kND];
        D.item = d.item;
        D.drow = d.drow;
        D.cut_tau = d.cut_tau;
        D.cut_id = d.cut_id;
        D.trunc = d.trunc;
        D.pair = d.pair;
        D.greedy = d.greedy;
        D.s_hi = d.s_hi;
        D.s_lo = d.s_lo;
        D.u_s = d.u_s;
        D.valid = 1;
        D.B_t = B_t;
        D.B_d = B_d;
        D.S_t = S_t;
        D.S_d = S_d;
        D.inv_St = inv_St;
        D.lam = lam;
        D.c_t = ct.x;
        D.c_tf = ct.y;
        D.c_d = cd.x;
        D.c_df = cd.y;
        D.argmax_t = argmax_t;
        D.alpha_g = alpha_g;
        D.rho = rho;
        D.accept = accept;
        D.kind = kind;
        D.status = status;
    }
}

// Pass 2 of a pair under Rule 2, from the registers and the ring slot of pass 1. Thread t takes
// vectors t + 480 v of the slice, as in pass 1. Where the position rejects:
// e_t = 2^(y_t s - B_t), e_d = 2^(y_d s - B_d), lambda = S_t / S_d; the residual
// max(e_t - lambda e_d, 0) per chunk and S_t * min(p, q) = min(e_t, lambda e_d) (no
// cancellation). Where it accepts, only alpha: min(p, q) = 2^min(y_t s - c_t, y_d s - c_d), c the
// log2 of the normaliser.
template <int DT, int NVT>
__device__ __forceinline__ void pass2_held(const uint4 (&vt)[NVT], const SmemRow<DT> &rd, CtaShared &sh,
                                      const Decision &D, int rb, int warp, int lane) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    float my_alpha = 0.0f, my_z = 0.0f;
    if (D.status == 0 && D.pair && !D.greedy) {
        const float2 shi2 = f2splat(D.s_hi), slo2 = f2splat(D.s_lo);
        if (D.kind == SAMPLE_RESIDUAL) {
            const float2 nbt = f2splat(-D.B_t), nbd = f2splat(-D.B_d);
            const float2 nlh = f2splat(-D.lam.hi), nll = f2splat(-D.lam.lo);
            float2 acc_a = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int v = 0; v < NVT; ++v) {
                if (!warp_has(v, warp, rd.nvec)) {
                    if (lane == 0) sh.rm[rb][v * kWarps + warp] = 0.0f;
                    continue;
                }
                const uint4 wd = rd(v);
                float2 racc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 yt = Elt<DT>::unpack_one(vt[v], h), yd = Elt<DT>::unpack_one(wd, h);
                    const float2 et = ex2x2(exp_arg2(yt, shi2, slo2, nbt));
                    const float2 ed = ex2x2(exp_arg2(yd, shi2, slo2, nbd));
                    const float2 r = __ffma2_rn(ed, nll, __ffma2_rn(ed, nlh, et));
                    const float2 nq = __fmul2_rn(ed, nlh);  // -lambda_hi * e_d, for min(p, q)
                    racc = __fadd2_rn(racc, make_float2(fmaxf(r.x, 0.0f), fmaxf(r.y, 0.0f)));
                    acc_a = __fadd2_rn(acc_a, make_float2(fminf(et.x, -nq.x), fminf(et.y, -nq.y)));
                }
                const float rs = warp_sum(racc.x + racc.y);
                my_z += rs;
                if (lane == 0) sh.rm[rb][v * kWarps + warp] = rs;
            }
            my_alpha = (acc_a.x + acc_a.y) * D.inv_St;
        } else {
            // y*s - c with c split: the product less the integral part rounds once (to a small
            // result near the top of the row), then the fraction
            const float2 nct = f2splat(-D.c_t), ncd = f2splat(-D.c_d);
            const float2 nctf = f2splat(-D.c_tf), ncdf = f2splat(-D.c_df);
            float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int v = 0; v < NVT; ++v) {
                if (!warp_has(v, warp, rd.nvec)) continue;
                const uint4 wd = rd(v);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 at = __fadd2_rn(__ffma2_rn(Elt<DT>::unpack_one(vt[v], h), shi2, nct), nctf);
                    const float2 ad = __fadd2_rn(__ffma2_rn(Elt<DT>::unpack_one(wd, h), shi2, ncd), ncdf);
                    acc = __fadd2_rn(acc, make_float2(ex2(fminf(at.x, ad.x)), ex2(fminf(at.y, ad.y))));
                }
            }
            my_alpha = acc.x + acc.y;
        }
    }
    my_alpha = warp_sum(my_alpha);
    if (lane == 0) {
        sh.wal[rb][warp] = my_alpha;
        sh.wz[rb][warp] = my_z;
    }
}

// kLag > 0: pass 2 of a pair under Rule 2, its two rows read again from global memory (pass 1's
// copies left them in L2 a few items earlier; these loads stream them out, evict-first). Thread t
// takes vectors t + 480 v of the slice, as in pass 1. The arithmetic is that of pass2_held.
template <int DT, int NVT>
__device__ __forceinline__ void pass2_l2(const RowsParams &P, CtaShared &sh, const Decision &D, int rb, int lo,
                                         int nvec, int warp, int lane, int tid) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    float my_alpha = 0.0f, my_z = 0.0f;
    if (D.status == 0 && D.pair && !D.greedy) {
        const uint4 *tr = static_cast<const uint4 *>(P.target) + static_cast<size_t>(D.item) * P.nvec_row + lo;
        const uint4 *dr = static_cast<const uint4 *>(P.draft) + static_cast<size_t>(D.drow) * P.nvec_row + lo;
        const float2 shi2 = f2splat(D.s_hi), slo2 = f2splat(D.s_lo);
        if (D.kind == SAMPLE_RESIDUAL) {
            const float2 nbt = f2splat(-D.B_t), nbd = f2splat(-D.B_d);
            const float2 nlh = f2splat(-D.lam.hi), nll = f2splat(-D.lam.lo);
            float2 acc_a = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int v = 0; v < NVT; ++v) {
                if (!warp_has(v, warp, nvec)) {
                    if (lane == 0) sh.rm[rb][v * kWarps + warp] = 0.0f;
                    continue;
                }
                const int vi = tid + v * kThreads;
                uint4 wt = vi < nvec ? __ldcs(tr + vi) : kNegInfVec<DT>();
                if (D.trunc) mask_cut<DT>(wt, lo + vi, D.cut_tau, D.cut_id);
                const uint4 wd = vi < nvec ? __ldcs(dr + vi) : kNegInfVec<DT>();
                float2 racc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 yt = Elt<DT>::unpack_one(wt, h), yd = Elt<DT>::unpack_one(wd, h);
                    const float2 et = ex2x2(exp_arg2(yt, shi2, slo2, nbt));
                    const float2 ed = ex2x2(exp_arg2(yd, shi2, slo2, nbd));
                    const float2 r = __ffma2_rn(ed, nll, __ffma2_rn(ed, nlh, et));
                    const float2 nq = __fmul2_rn(ed, nlh);  // -lambda_hi * e_d, for min(p, q)
                    racc = __fadd2_rn(racc, make_float2(fmaxf(r.x, 0.0f), fmaxf(r.y, 0.0f)));
                    acc_a = __fadd2_rn(acc_a, make_float2(fminf(et.x, -nq.x), fminf(et.y, -nq.y)));
                }
                const float rs = warp_sum(racc.x + racc.y);
                my_z += rs;
                if (lane == 0) sh.rm[rb][v * kWarps + warp] = rs;
            }
            my_alpha = (acc_a.x + acc_a.y) * D.inv_St;
        } else {
            const float2 nct = f2splat(-D.c_t), ncd = f2splat(-D.c_d);
            const float2 nctf = f2splat(-D.c_tf), ncdf = f2splat(-D.c_df);
            float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int v = 0; v < NVT; ++v) {
                if (!warp_has(v, warp, nvec)) continue;
                const int vi = tid + v * kThreads;
                uint4 wt = vi < nvec ? __ldcs(tr + vi) : kNegInfVec<DT>();
                if (D.trunc) mask_cut<DT>(wt, lo + vi, D.cut_tau, D.cut_id);
                const uint4 wd = vi < nvec ? __ldcs(dr + vi) : kNegInfVec<DT>();
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const float2 at = __fadd2_rn(__ffma2_rn(Elt<DT>::unpack_one(wt, h), shi2, nct), nctf);
                    const float2 ad = __fadd2_rn(__ffma2_rn(Elt<DT>::unpack_one(wd, h), shi2, ncd), ncdf);
                    acc = __fadd2_rn(acc, make_float2(ex2(fminf(at.x, ad.x)), ex2(fminf(at.y, ad.y))));
                }
            }
            my_alpha = acc.x + acc.y;
        }
    }
    my_alpha = warp_sum(my_alpha);
    if (lane == 0) {
        sh.wal[rb][warp] = my_alpha;
        sh.wz[rb][warp] = my_z;
    }
}

// The draw weights of one vector, exactly as the passes summed them: the residual in units of
// 2^B_t, or p in units of 2^bg (bg: the chunk's reference).
template <int DT>
__device__ __forceinline__ void draw_weights(int kind, const uint4 &wt, const uint4 &wd, const Decision &D, float bg,
                                             float *w) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    const float2 shi2 = f2splat(D.s_hi), slo2 = f2splat(D.s_lo);
    float2 yt[H];
    Elt<DT>::unpack2(wt, yt);
    if (kind == SAMPLE_RESIDUAL) {
        float2 yd[H];
        Elt<DT>::unpack2(wd, yd);
        const float2 nbt = f2splat(-D.B_t), nbd = f2splat(-D.B_d);
        const float2 nlh = f2splat(-D.lam.hi), nll = f2splat(-D.lam.lo);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float2 et = ex2x2(exp_arg2(yt[h], shi2, slo2, nbt));
            const float2 ed = ex2x2(exp_arg2(yd[h], shi2, slo2, nbd));
            const float2 r = __ffma2_rn(ed, nll, __ffma2_rn(ed, nlh, et));
            w[2 * h] = fmaxf(r.x, 0.0f);
            w[2 * h + 1] = fmaxf(r.y, 0.0f);
        }
    } else {
        const float2 nb = f2splat(-bg);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float2 e = ex2x2(exp_arg2(yt[h], shi2, slo2, nb));
            w[2 * h] = e.x;
            w[2 * h + 1] = e.y;
        }
    }
}

// Mass of CTA c's slice in the law a draw of item m uses (units 2^B_t).
__device__ __forceinline__ F2 cta_mass(const Msg &Mi, const Msg &Mn, int kind, float B_t) {
    if (kind == SAMPLE_RESIDUAL) return {Mn.prev_Z, 0.0f};
    // B_t is the cluster's max of the CTA references, an integer
    return (Mi.a[0] != kNoRef && Mi.b[0] > 0.0f) ? F2{Mi.b[0] * pow2_int(Mi.a[0] - static_cast<int>(B_t)), 0.0f}
                                                 : F2{0.0f, 0.0f};
}

// What the control warp knows about item m's draw after the exchange that carries its totals.
struct FinState {
    int kind, fb, owner;
    F2 local, Ztot;  // u*Z less the mass of the CTAs before the owner; Z (units 2^B_t)
};

// Control warp, once the exchange that carries item m's alpha and residual shares is done (Mi: the
// records of item m's own exchange, Mn: those of the exchange carrying its totals): the item's
// results. They are written by the owner of its draw (the CTA whose slice holds u*Z),
// else by CTA 0. Returns the draw's state in every lane.
__device__ __forceinline__ FinState finalize_head(CtaShared &sh, const RowsParams &P, int m, const Msg *Mi,
                                                  const Msg *Mn, int C, int crank, int lane) {
    const Decision &D = sh.dec[m % kND];
    FinState f;
    f.kind = D.kind;
    f.fb = 0;
    f.owner = -1;
    f.local = f.Ztot = {0.0f, 0.0f};
    // one lane per CTA record, in CTA order
    const bool on = lane < C;
    const Msg &mi = Mi[on ? lane : 0], &mn = Mn[on ? lane : 0];
    float alpha_sum = on ? mn.prev_alpha : 0.0f;
    float Zres = on ? mn.prev_Z : 0.0f;
    // sums over the C lanes (C a power of two: lane l < C meets only lanes below C)
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
        if (o < C) {
            alpha_sum += __shfl_xor_sync(0xffffffffu, alpha_sum, o);
            Zres += __shfl_xor_sync(0xffffffffu, Zres, o);
        }
    Zres = __shfl_sync(0xffffffffu, Zres, 0);  // the same in every lane: the branches below hold warp-wide shuffles
    if (f.kind == SAMPLE_RESIDUAL && !(Zres > 0.0f)) {
        f.kind = SAMPLE_P;  // zero residual mass: draw from p and say so
        f.fb = 1;
    }
    if (f.kind != SAMPLE_NONE) {
        // the first CTA whose running total exceeds u*Z (else the last with mass: rounding put
        // u*Z at the very end)
        const F2 mc = on ? cta_mass(mi, mn, f.kind, D.B_t) : F2{0.0f, 0.0f};
        // inclusive scan over the C lanes, in CTA order
        F2 incl = mc;
#pragma unroll
        for (int o = 1; o < kMaxCluster; o <<= 1)
            if (o < C) {
                const F2 w = {__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
                if (lane >= o) incl = f2_add(w, incl);
            }
        f.Ztot = shfl_f2(incl, C - 1);
        const F2 t = f2_mul(f.Ztot, D.u_s);
        const unsigned hit = __ballot_sync(0xffffffffu, on && mc.hi > 0.0f && f2_gt(incl, t));
        const unsigned posm = __ballot_sync(0xffffffffu, on && mc.hi > 0.0f);
        f.owner = hit ? __ffs(hit) - 1 : (posm ? 31 - __clz(static_cast<int>(posm)) : -1);
        if (f.owner >= 0) {
            const F2 prefix = shfl_f2(f2_sub(incl, mc), f.owner);
            f.local = f2_sub(t, prefix);
        }
    }
    if (lane == 0) {
        const int writer = f.owner >= 0 ? f.owner : 0;
        if (writer == crank) {
            const int item = D.item, st = D.status;
            P.item_status[item] = st;
            P.item_fb[item] = f.fb;
            if (D.pair) {
                const float alpha = D.greedy ? D.alpha_g : alpha_sum;
                P.item_flag[item] = (st == 0) ? D.accept : 0;
                P.alpha_ws[D.drow] = (st == 0) ? alpha : 0.0f;
                if (P.alpha_rows) P.alpha_rows[D.drow] = (st == 0) ? alpha : NAN;
                if (P.rho_rows) P.rho_rows[D.drow] = (st == 0) ? D.rho : NAN;
                if (P.resid_rows)
                    P.resid_rows[D.drow] =
                        (st == 0 && f.kind == SAMPLE_RESIDUAL && !D.greedy) ? Zres * D.inv_St : -1.0f;
            } else {
                P.item_flag[item] = 0;
            }
            if (f.owner < 0) {
                if (st == 0 && D.greedy && !(D.pair && D.accept)) {
                    // Rule 1: the correction (or the extra token) is argmax p
                    P.item_tok[item] = D.argmax_t;
                    P.item_prob[item] = 1.0f;
                } else {
                    P.item_tok[item] = -1;
                    P.item_prob[item] = NAN;
                }
                P.item_margin[item] = NAN;
            }
        }
    }
    f.local = shfl_f2(f.local, 0);
    f.Ztot = shfl_f2(f.Ztot, 0);
    return f;
}

// Control warp of the owner CTA, for a rejecting pair whose residual has no mass (p <= q at every
// token, up to rounding): the draw is from p, whose chunk masses (units 2^B_t) are computed here
// from the target row in global memory, in the place of the (zero) residual chunk sums. A path
// that ordinary inputs never take; it reads the slice once more.
template <int DT>
__device__ __noinline__ void fb_chunk_masses(CtaShared &sh, const RowsParams &P, const Decision &D, int rb, int lane,
                                             int nch, int lo, int nvec) {
    constexpr int E = Elt<DT>::kPerVec;
    const uint4 *row = static_cast<const uint4 *>(P.target) + static_cast<size_t>(D.item) * P.nvec_row + lo;
    for (int k = 0; k < nch; ++k) {
        const int vi = (k / kWarps) * kThreads + (k % kWarps) * kWarp + lane;
        float w[E];
        uint4 wt = vi < nvec ? row[vi] : kNegInfVec<DT>();
        if (D.trunc) mask_cut<DT>(wt, lo + vi, D.cut_tau, D.cut_id);
        draw_weights<DT>(SAMPLE_P, wt, kNegInfVec<DT>(), D, D.B_t, w);
        float a = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) a += w[e];
        a = warp_sum(a);
        if (lane == 0) sh.rm[rb][k] = a;
    }
    __syncwarp();
}

// Control warp of the owner CTA: the chunk that holds u*Z (an inclusive scan over the slice's
// chunk masses, in vocabulary order), fetched with a small bulk copy; `complete_draw` finds the
// token once it has landed.
template <int DT>
__device__ __noinline__ void draw_chunk(CtaShared &sh, const RowsParams &P, int m, const FinState &f, int lane,
                                           int nch, int lo, int nvec) {
    const int rb = m % kRM, pb = m % kPM;
    const Decision &D = sh.dec[m % kND];
    if (f.fb) fb_chunk_masses<DT>(sh, P, D, rb, lane, nch, lo, nvec);
    int ksel = -1, klast = -1;
    F2 before = {0.0f, 0.0f}, last_before = {0.0f, 0.0f}, run = {0.0f, 0.0f};
#pragma unroll 1
    for (int base = 0; base < nch; base += kWarp) {
        const int k = base + lane;
        float mk = 0.0f;
        if (k < nch) {
            if (f.kind == SAMPLE_RESIDUAL) {
                mk = sh.rm[rb][k];
            } else if (f.fb) {
                mk = sh.rm[rb][k];  // p masses, from fb_chunk_masses
            } else {
                const float pmk = sh.pm[pb][k];
                mk = pmk > 0.0f ? pmk * pow2i(sh.pref[pb][k] - D.B_t) : 0.0f;
            }
        }
        const bool pos = k < nch && mk > 0.0f;
        const F2 incl = f2_add(run, warp_scan_f2({mk, 0.0f}, lane));
        const unsigned hit = __ballot_sync(0xffffffffu, pos && f2_gt(incl, f.local));
        const unsigned posm = __ballot_sync(0xffffffffu, pos);
        if (hit) {
            const int l = __ffs(hit) - 1;
            ksel = base + l;
            before = shfl_f2(f2_sub(incl, {mk, 0.0f}), l);
            break;
        }
        if (posm) {
            const int l = 31 - __clz(static_cast<int>(posm));
            klast = base + l;
            last_before = shfl_f2(f2_sub(incl, {mk, 0.0f}), l);
        }
        run = shfl_f2(incl, kWarp - 1);
    }
    const int clamped = ksel < 0;  // rounding put u*Z past the last chunk with mass
    if (clamped) {
        ksel = klast;
        before = last_before;
    }
    if (lane == 0) {
        const int start = (ksel >= 0) ? (ksel / kWarps) * kThreads + (ksel % kWarps) * kWarp : 0;
        const int count = (ksel >= 0) ? max(0, min(kWarp, nvec - start)) : 0;
        float bg = 0.0f, unit = 1.0f, lt = 0.0f;
        const F2 rem = f2_sub(f.local, before);
        if (f.kind == SAMPLE_RESIDUAL || f.fb) {
            bg = D.B_t;
            lt = rem.hi + rem.lo;
        } else if (ksel >= 0) {
            // p weights of the chunk are in units of 2^bg: 2^(bg - B_t) cluster units
            bg = sh.pref[pb][ksel];
            unit = pow2i(bg - D.B_t);
            lt = (rem.hi + rem.lo) * pow2i(D.B_t - bg);
        }
        sh.draw_pending = 1;
        sh.draw_item = D.item;
        sh.draw_dec = m % kND;
        sh.draw_kind = f.kind;
        sh.draw_chunk = start;
        sh.draw_count = count;
        sh.draw_clamped = clamped;
        sh.draw_lt = lt;
        sh.draw_unit = unit;
        sh.draw_bg = bg;
        sh.draw_invZ = rcp_approx(f.Ztot.hi);
        if (count > 0) {
            const size_t row_bytes = static_cast<size_t>(P.nvec_row) * 16;
            const size_t off = static_cast<size_t>(lo + start) * 16;
            const uint32_t bytes = static_cast<uint32_t>(count) * 16;
            const bool two = f.kind == SAMPLE_RESIDUAL;
            mbar_arrive_expect_tx(&sh.draw_bar, two ? 2 * bytes : bytes);
            bulk_g2s(sh.draw_buf[0],
                     static_cast<const unsigned char *>(P.target) + static_cast<size_t>(D.item) * row_bytes + off,
                     bytes, &sh.draw_bar, policy_evict_first());
            if (two)
                bulk_g2s(sh.draw_buf[1],
                         static_cast<const unsigned char *>(P.draft) + static_cast<size_t>(D.drow) * row_bytes + off,
                         bytes, &sh.draw_bar, policy_evict_first());
        }
    }
    __syncwarp();
}

// Control warp of the owner CTA: the token of the pending draw within its chunk (one vector per
// lane).
template <int DT>
__device__ __noinline__ void complete_draw(CtaShared &sh, const RowsParams &P, int lo, int lane) {
    constexpr int E = Elt<DT>::kPerVec;
    if (!sh.draw_pending) return;
    const Decision &D = sh.dec[sh.draw_dec];
    const int kind = sh.draw_kind, count = sh.draw_count, clamped = sh.draw_clamped;
    bool ok = true;
    if (count > 0) {
        ok = mbar_wait_sleep_bounded(&sh.draw_bar, sh.draw_phase, kSuspendNs, kMaxWaitTries);
        ok = __all_sync(0xffffffffu, ok);
    }
    uint4 wt = lane < count ? sh.draw_buf[0][lane] : kNegInfVec<DT>();
    if (D.trunc) mask_cut<DT>(wt, lo + sh.draw_chunk + lane, D.cut_tau, D.cut_id);
    const uint4 wd = (lane < count && kind == SAMPLE_RESIDUAL) ? sh.draw_buf[1][lane] : kNegInfVec<DT>();
    float w[E];
    draw_weights<DT>(kind, wt, wd, D, sh.draw_bg, w);
    float ls = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) ls += w[e];
    float incl = ls;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    const float lt = sh.draw_lt;
    int found = -1, lastp = -1;
    float c = incl - ls, fprev = 0.0f, wf = 0.0f, wl = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if (w[e] > 0.0f) {
            if (found < 0 && !clamped && c + w[e] > lt) {
                found = e;
                fprev = c;
                wf = w[e];
            }
            lastp = e;
            wl = w[e];
        }
        c += w[e];
    }
    const unsigned hit = __ballot_sync(0xffffffffu, found >= 0);
    const unsigned posm = __ballot_sync(0xffffffffu, lastp >= 0);
    int tok = -1;
    float wsel = 0.0f, margin = 0.0f;
    const int base = lo + sh.draw_chunk;
    if (hit) {
        const int l = __ffs(hit) - 1;
        const float c0 = __shfl_sync(0xffffffffu, fprev, l);
        wsel = __shfl_sync(0xffffffffu, wf, l);
        tok = (base + l) * E + __shfl_sync(0xffffffffu, found, l);
        margin = fminf(lt - c0, c0 + wsel - lt) * sh.draw_unit * sh.draw_invZ;
    } else if (posm) {  // rounding: the last element with mass
        const int l = 31 - __clz(static_cast<int>(posm));
        wsel = __shfl_sync(0xffffffffu, wl, l);
        tok = (base + l) * E + __shfl_sync(0xffffffffu, lastp, l);
    }
    if (lane == 0) {
        const int item = sh.draw_item;
        if (ok) {
            P.item_tok[item] = tok;
            P.item_prob[item] = tok >= 0 ? wsel * sh.draw_unit * sh.draw_invZ : NAN;
            P.item_margin[item] = tok >= 0 ? margin : NAN;
        } else {
            P.item_status[item] = D.status | REQ_TIMEOUT;
            P.item_tok[item] = -1;
            P.item_prob[item] = NAN;
            P.item_margin[item] = NAN;
        }
        if (count > 0) sh.draw_phase ^= 1u;
        sh.draw_pending = 0;
    }
    __syncwarp();
}

// Control warp, exchange g: item g's record goes out with the totals of item g - 1 (pass 2 of
// g - 1 is done once every data warp has passed pass 1 of g); item g is decided and released to
// the data warps at once; then item g - 1 is finished (results, draw) from this exchange's totals.
// d == nullptr: the drain after the last item (totals only).
template <int DT>
__device__ __forceinline__ void control_item(CtaShared &sh, const RowsParams &P, const Desc *d, int g, Msg *slots,
                                             int C, int crank, int lo, int nvec, int nch, int lane) {
    const int nr = d ? desc_rows(*d) : 0, greedy = d ? d->greedy : 0;
    if (!mbar_wait_sleep_bounded(&sh.stats_bar[g % kSB], static_cast<uint32_t>((g / kSB) & 1), kSuspendNs,
                                 kMaxWaitTries))
        sh.timed_out = 1;
    __syncwarp();
    uint4 rec[3];
    build_record(sh, greedy, nr, g, g - 1, lane, rec);
    if (g == 0) cluster_wait();  // the peers run and their barriers are ready
    Msg *const here = slots + (g % kNMS) * kMaxCluster;
    push_record(rec, here, &sh.msg_bar[g % kNMS], crank, C, lane);
    if (lane == 0) mbar_arrive_expect_tx(&sh.msg_bar[g % kNMS], static_cast<uint32_t>(C * kMsgBytes));
    complete_draw<DT>(sh, P, lo, lane);  // the draw fetched at the previous exchange
    if (!mbar_wait_sleep_bounded(&sh.msg_bar[g % kNMS], static_cast<uint32_t>((g / kNMS) & 1), kSuspendNs,
                                 kMaxWaitTries))
        sh.timed_out = 1;
    __syncwarp();
    if (d) {
        decide_item(sh, here, *d, nr, g, C, P, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.dec_bar[g % kND]);
    }
    if (g >= 1) {
        const FinState f = finalize_head(sh, P, g - 1, slots + ((g - 1) % kNMS) * kMaxCluster, here, C, crank, lane);
        if (f.owner == crank) draw_chunk<DT>(sh, P, g - 1, f, lane, nch, lo, nvec);
    }
}

// Pass 1 of a pair: the thread that holds the draft token x records (y_t - y_d) s there as a float
// pair (for the accept ratio) and whether p(x) or q(x) is zero.
template <int DT, int NVT>
__device__ __forceinline__ void extract_x(CtaShared &sh, const Desc &d, const uint4 (&vt)[NVT], const SmemRow<DT> &rd,
                                          int wb, int g, int lo, int nvec, int V, int tid) {
    constexpr int E = Elt<DT>::kPerVec;
    const int x = d.x;
    if (x < 0 || x >= V) return;
    const int xv = x / E - lo;
    if (xv < 0 || xv >= nvec || (xv % kThreads) != tid) return;
    const int vx = xv / kThreads, e = x % E;
    float yt = 0.0f;
#pragma unroll
    for (int v = 0; v < NVT; ++v)
        if (v == vx) yt = vec_elem<DT>(vt[v], e);
    const float yd = vec_elem<DT>(rd.src[xv], e);
    const F2 Ex = f2_mul(f2_add({yt, 0.0f}, {-yd, 0.0f}), {d.s_hi, d.s_lo});
    sh.xE[wb][0] = Ex.hi;
    sh.xE[wb][1] = Ex.lo;
    sh.x_flags[wb] = XF_HAS | (yd == -INFINITY ? XF_QZERO : 0) | (yt == -INFINITY ? XF_PZERO : 0);
    sh.x_stamp[wb] = g + 1;
}

// Top-k / top-p: apply the target row's cut to this thread's vectors (vector v of thread t is
// vector lo + t + 480 v of the row).
template <int DT, int NVT>
__device__ __forceinline__ void mask_row(uint4 (&vt)[NVT], int lo, int tid, uint32_t tau, int id) {
#pragma unroll
    for (int v = 0; v < NVT; ++v) mask_cut<DT>(vt[v], lo + tid + v * kThreads, tau, id);
}

// Load the slice of one ring slot into registers: thread t takes vectors t, t + 480, ... so that
// a warp reads 32 contiguous vectors (a chunk); past the slice end, -inf.
template <int DT, int NVT>
__device__ __forceinline__ bool load_row(CtaShared &sh, const uint4 *ring, int slice_max, int nvec, long long row,
                                         int tid, uint4 (&vv)[NVT]) {
    const int slot = static_cast<int>(row % kRing);
    const bool ok =
        mbar_wait_sleep_bounded(&sh.full[slot], static_cast<uint32_t>((row / kRing) & 1), kSuspendNs, kMaxWaitTries);
    const uint4 *src = ring + static_cast<size_t>(slot) * slice_max;
#pragma unroll
    for (int v = 0; v < NVT; ++v) {
        const int vi = tid + v * kThreads;
        vv[v] = vi < nvec ? src[vi] : kNegInfVec<DT>();
    }
    return ok;
}

template <int DT, int NVT>
__global__ void __launch_bounds__(kBlock, 2) spec_rows_kernel(const RowsParams P) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ CtaShared sh;
    uint4 *ring = reinterpret_cast<uint4 *>(smem_raw);

    // The control warp is hardware warp 0 (the schedulers favour the lowest warps when several are
    // ready, and its chain of dependent steps gates every item); the data warps are hardware warps
    // 1 .. 15. Logical numbering: data thread t = 0 .. 479 in warps 0 .. 14, the control warp 15.
    const int hw_warp = static_cast<int>(threadIdx.x) / kWarp, lane = static_cast<int>(threadIdx.x) % kWarp;
    const int warp = hw_warp == 0 ? kWarps : hw_warp - 1;
    const int tid = warp * kWarp + lane;
    griddep_launch_dependents();  // the selection kernel may be scheduled behind this grid
    const int C = static_cast<int>(cluster_nctarank());
    const int crank = static_cast<int>(cluster_ctarank());
    const int cid = static_cast<int>(cluster_id_x());
    const int lo = static_cast<int>((static_cast<int64_t>(P.nvec_row) * crank) / C);
    const int nvec = static_cast<int>((static_cast<int64_t>(P.nvec_row) * (crank + 1)) / C) - lo;
    const int slice_max = P.slice_vecs_max;
    const int nch = NVT * kWarps;
    const int ncl = P.nclusters;
    const int nitems = cid < P.total_rows ? (P.total_rows - 1 - cid) / ncl + 1 : 0;
    // the exchange slots follow the ring: kNMS exchanges x kMaxCluster records (C used), the same
    // layout in every CTA
    Msg *const slots = reinterpret_cast<Msg *>(smem_raw + static_cast<size_t>(kRing) * slice_max * 16);

    if (tid == 0) {
        for (int k = 0; k < kRing; ++k) {
            mbar_init(&sh.full[k], 1);
            sh.free_cnt[k] = 0;
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
        sh.prod_issued = 0;
    }
    __syncthreads();  // the barriers are initialised
    // every CTA of the cluster must run, its barriers ready, before any remote access: all threads
    // arrive now; the control warp waits before its first remote store, the data warps at the end
    cluster_arrive();

    if (warp < kWarps) {
      if constexpr (kLag == 0) {
        // ================= data warps: pass 1, the decision, pass 2 (rows held on chip) ========
        long long R = 0;  // ring row of the item's target row
        int g0 = 0;       // the batch's first item, counted over the whole list
        for (int nb = 0; nb < nitems; nb += kMaxItems) {
            const int nbatch = min(kMaxItems, nitems - nb);
            bar_sync(BAR_BATCH, kBlock);  // the control warp has the batch's descriptors
            if (tid == 0 && nb > 0) {  // the first batch's copies went out with its shapes
                sh.prod_item = 0;
                sh.prod_row = 0;
                produce_rows(sh, ring, P, slice_max, lo, nvec, nbatch, sh.prod_issued, R + kRing, sh.prod_item,
                             sh.prod_row);
            }
            for (int i = 0; i < nbatch; ++i) {
                const int g = g0 + i, wb = g % kWS;
                const Desc &d = sh.desc[i];
                const int nr = desc_rows(d);
                uint4 vt[NVT];
                bool ok = true;
                if (nr >= 1) {
                    ok = load_row<DT, NVT>(sh, ring, slice_max, nvec, R, tid, vt);
                    // this warp holds the target row in registers: its slot may refill
                    release_row(sh, ring, P, slice_max, lo, nvec, nbatch, R, lane);
                    if (d.trunc) mask_row<DT, NVT>(vt, lo, tid, d.cut_tau, d.cut_id);
                }
                const SmemRow<DT> rd = {ring + static_cast<size_t>((R + 1) % kRing) * slice_max, tid, nvec};
                if (nr == 2)
                    ok &= mbar_wait_sleep_bounded(&sh.full[(R + 1) % kRing],
                                                  static_cast<uint32_t>(((R + 1) / kRing) & 1), kSuspendNs,
                                                  kMaxWaitTries);
                if (!ok) sh.timed_out = 1;
                if (nr == 1) row_stats<DT, NVT, true>(RegRow<NVT>{vt}, sh, wb, 0, g % kPM, d, lo, nvec, warp, lane, tid);
                if (nr == 2) {
                    if (d.greedy) {
                        row_stats<DT, NVT, false>(RegRow<NVT>{vt}, sh, wb, 0, 0, d, lo, nvec, warp, lane, tid);
                        row_stats<DT, NVT, false>(rd, sh, wb, 1, 0, d, lo, nvec, warp, lane, tid);
                    } else {
                        pair_stats<DT, NVT>(vt, rd, sh, wb, d, nvec, warp, lane);
                    }
                    extract_x<DT, NVT>(sh, d, vt, rd, wb, g, lo, nvec, P.V, tid);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.stats_bar[g % kSB]);
                // every item waits for its decision (pass 2 needs it; it also keeps the data warps
                // within one item of each other and of the control warp)
                if (!mbar_wait_sleep_bounded(&sh.dec_bar[g % kND], static_cast<uint32_t>((g / kND) & 1), kSuspendNs,
                                             kMaxWaitTries))
                    sh.timed_out = 1;
                if (nr == 2) {
                    pass2_held<DT, NVT>(vt, rd, sh, sh.dec[g % kND], g % kRM, warp, lane);
                    release_row(sh, ring, P, slice_max, lo, nvec, nbatch, R + 1, lane);  // the draft slot
                } else if (lane == 0) {
                    sh.wal[g % kRM][warp] = 0.0f;
                    sh.wz[g % kRM][warp] = 0.0f;
                }
                R += nr;
            }
            g0 += nbatch;
        }
        // the drain: the last pass 2 is done, its totals go out with one more exchange
        __syncwarp();
        if (nitems > 0 && lane == 0) mbar_arrive(&sh.stats_bar[nitems % kSB]);
      } else {
        // ================= data warps: pass 1 of item i, then pass 2 of item i - kLag =========
        long long R = 0;  // ring row of the item's target row
        int g0 = 0;       // the batch's first item, counted over the whole list
        for (int nb = 0; nb < nitems; nb += kMaxItems) {
            const int nbatch = min(kMaxItems, nitems - nb);
            bar_sync(BAR_BATCH, kBlock);  // the control warp has the batch's descriptors
            if (tid == 0 && nb > 0) {  // the first batch's copies went out with its shapes
                sh.prod_item = 0;
                sh.prod_row = 0;
                produce_rows(sh, ring, P, slice_max, lo, nvec, nbatch, sh.prod_issued, R + kRing, sh.prod_item,
                             sh.prod_row);
            }
            for (int i = 0; i < nbatch + kLag; ++i) {
                if (i < nbatch) {
                    const int g = g0 + i, wb = g % kWS;
                    const Desc &d = sh.desc[i];
                    const int nr = desc_rows(d);
                    uint4 vt[NVT];
                    bool ok = true;
                    if (nr >= 1) {
                        ok = load_row<DT, NVT>(sh, ring, slice_max, nvec, R, tid, vt);
                        // this warp holds the target row in registers: its slot may refill
                        release_row(sh, ring, P, slice_max, lo, nvec, nbatch, R, lane);
                        if (d.trunc) mask_row<DT, NVT>(vt, lo, tid, d.cut_tau, d.cut_id);
                    }
                    const SmemRow<DT> rd = {ring + static_cast<size_t>((R + 1) % kRing) * slice_max, tid, nvec};
                    if (nr == 2)
                        ok &= mbar_wait_sleep_bounded(&sh.full[(R + 1) % kRing],
                                                      static_cast<uint32_t>(((R + 1) / kRing) & 1), kSuspendNs,
                                                      kMaxWaitTries);
                    if (!ok) sh.timed_out = 1;
                    if (nr == 1)
                        row_stats<DT, NVT, true>(RegRow<NVT>{vt}, sh, wb, 0, g % kPM, d, lo, nvec, warp, lane, tid);
                    if (nr == 2) {
                        if (d.greedy) {
                            row_stats<DT, NVT, false>(RegRow<NVT>{vt}, sh, wb, 0, 0, d, lo, nvec, warp, lane, tid);
                            row_stats<DT, NVT, false>(rd, sh, wb, 1, 0, d, lo, nvec, warp, lane, tid);
                        } else {
                            pair_stats<DT, NVT>(vt, rd, sh, wb, d, nvec, warp, lane);
                        }
                        extract_x<DT, NVT>(sh, d, vt, rd, wb, g, lo, nvec, P.V, tid);
                        // pass 1 of this warp is done with the draft row
                        release_row(sh, ring, P, slice_max, lo, nvec, nbatch, R + 1, lane);
                    }
                    R += nr;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.stats_bar[g % kSB]);
                }
                if (i >= kLag) {
                    const int m = g0 + i - kLag;
                    if (!mbar_wait_sleep_bounded(&sh.dec_bar[m % kND], static_cast<uint32_t>((m / kND) & 1),
                                                 kSuspendNs, kMaxWaitTries))
                        sh.timed_out = 1;
                    pass2_l2<DT, NVT>(P, sh, sh.dec[m % kND], m % kRM, lo, nvec, warp, lane, tid);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sh.p2_bar[m % kPB]);
                }
            }
            g0 += nbatch;
        }
      }
        if (tid == 0 && sh.timed_out) {
            // a copy did not land in time: wait (bounded) once more so that none is left in flight
            for (long long r = max(0LL, sh.prod_issued - kRing); r < sh.prod_issued; ++r)
                mbar_wait_sleep_bounded(&sh.full[r % kRing], static_cast<uint32_t>((r / kRing) & 1), kSuspendNs,
                                        kMaxWaitTries);
        }
        cluster_wait();
    } else {
        // ================= control warp: exchanges, decisions, results, draws =================
        if (lane < kRing && lane < nitems) {
            // the first target rows' slices into L2 while the descriptors load
            const size_t row_bytes = static_cast<size_t>(P.nvec_row) * 16;
            bulk_prefetch_l2(static_cast<const unsigned char *>(P.target) +
                                 static_cast<size_t>(cid + lane * ncl) * row_bytes + static_cast<size_t>(lo) * 16,
                             static_cast<uint32_t>(nvec) * 16);
        }
      if constexpr (kLag == 0) {
        int g = 0;  // item (and exchange) number; exchange nitems is the drain
        for (int nb = 0; nb < nitems; nb += kMaxItems) {
            const int nbatch = min(kMaxItems, nitems - nb);
            load_batch_shapes(sh, P, cid, nb, nbatch, lane);
            if (nb == 0 && lane == 0) {
                // the first rows go out as soon as the shapes are known, while the values load (the
                // ring is empty; later batches are started by the data warps)
                sh.prod_item = 0;
                sh.prod_row = 0;
                produce_rows(sh, ring, P, slice_max, lo, nvec, nbatch, sh.prod_issued, kRing, sh.prod_item,
                             sh.prod_row);
            }
            load_batch_values(sh, P, nbatch, lane);
            __syncwarp();
            bar_arrive(BAR_BATCH, kBlock);
            for (int i = 0; i < nbatch; ++i, ++g)
                control_item<DT>(sh, P, &sh.desc[i], g, slots, C, crank, lo, nvec, nch, lane);
        }
        if (nitems > 0) {
            control_item<DT>(sh, P, nullptr, nitems, slots, C, crank, lo, nvec, nch, lane);
            complete_draw<DT>(sh, P, lo, lane);  // the last draw
        } else {
            cluster_wait();
        }
      } else {
        int e = 0;   // exchanges so far
        int g0 = 0;  // the batch's first item
        for (int nb = 0; nb < nitems; nb += kMaxItems) {
            const int nbatch = min(kMaxItems, nitems - nb);
            load_batch_shapes(sh, P, cid, nb, nbatch, lane);
            if (nb == 0 && lane == 0) {
                // the first rows go out as soon as the shapes are known, while the values load (the
                // ring is empty; later batches are started by the data warps)
                sh.prod_item = 0;
                sh.prod_row = 0;
                produce_rows(sh, ring, P, slice_max, lo, nvec, nbatch, sh.prod_issued, kRing, sh.prod_item,
                             sh.prod_row);
            }
            load_batch_values(sh, P, nbatch, lane);
            __syncwarp();
            bar_arrive(BAR_BATCH, kBlock);
            const int e0 = e;  // the exchange of the batch's item i is e0 + i
            // exchange j carries item j's record (j < nbatch) and the totals of item j - kLag - 1;
            // kLag + 1 draining exchanges follow the batch's last item
            for (int j = 0; j < nbatch + kLag + 1; ++j) {
                const int g = g0 + j, m = j - kLag - 1;
                int nr = 0, greedy = 0;
                if (j < nbatch) {
                    nr = desc_rows(sh.desc[j]);
                    greedy = sh.desc[j].greedy;
                    if (!mbar_wait_sleep_bounded(&sh.stats_bar[g % kSB], static_cast<uint32_t>((g / kSB) & 1),
                                                 kSuspendNs, kMaxWaitTries))
                        sh.timed_out = 1;
                }
                if (m >= 0 && !mbar_wait_sleep_bounded(&sh.p2_bar[(g0 + m) % kPB],
                                                       static_cast<uint32_t>(((g0 + m) / kPB) & 1), kSuspendNs,
                                                       kMaxWaitTries))
                    sh.timed_out = 1;
                __syncwarp();
                uint4 rec[3];
                build_record(sh, greedy, nr, g, m >= 0 ? g0 + m : -1, lane, rec);
                if (e == 0) cluster_wait();  // the peers run and their barriers are ready
                Msg *const here = slots + (e % kNMS) * kMaxCluster;
                push_record(rec, here, &sh.msg_bar[e % kNMS], crank, C, lane);
                if (lane == 0) mbar_arrive_expect_tx(&sh.msg_bar[e % kNMS], static_cast<uint32_t>(C * kMsgBytes));
                complete_draw<DT>(sh, P, lo, lane);  // the draw fetched at the previous exchange
                if (!mbar_wait_sleep_bounded(&sh.msg_bar[e % kNMS], static_cast<uint32_t>((e / kNMS) & 1),
                                             kSuspendNs, kMaxWaitTries))
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
            g0 += nbatch;
        }
        if (nitems == 0) cluster_wait();
      }
    }
    __syncwarp();
    cluster_sync_all();  // no CTA leaves while another may still write into its shared memory
}

}  // namespace spec
