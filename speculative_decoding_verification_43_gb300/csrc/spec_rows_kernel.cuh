// spec_rows_kernel: see spec_rows.cuh for the design. Included once, by spec_verify.cu.
#pragma once

#include "spec_rows.cuh"

namespace spec {

template <int DT>
__global__ void __launch_bounds__(kThreads, 3) spec_rows_kernel(const RowsParams P) {
    constexpr int E = Elt<DT>::kPerVec;
    constexpr int H = E / 2;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2][kMaxChunks];
    __shared__ Ex1 xch1[kMaxCluster];
    __shared__ Ex2 xch2[kMaxCluster];
    __shared__ Ex1 mine1;
    __shared__ Ex2 mine2;
    __shared__ ItemInfo I;
    __shared__ float red_f[kWarps];

    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    griddep_launch_dependents();  // the selection kernel may be scheduled behind the last wave
    const int C = static_cast<int>(cluster_nctarank());
    const int crank = static_cast<int>(cluster_ctarank());
    const int item = static_cast<int>(cluster_id_x());

    uint4 *buf_t = reinterpret_cast<uint4 *>(smem_raw);
    uint4 *buf_d = buf_t + P.slice_vecs_max;
    float *gref = reinterpret_cast<float *>(buf_d + P.slice_vecs_max);  // [2][groups_max]
    float *gsum = gref + 2 * P.groups_max;                              // [2][groups_max]
    float *gres = gsum + 2 * P.groups_max;                              // [groups_max]
    const size_t row_bytes = static_cast<size_t>(P.nvec_row) * 16;

    // ---- slice, barriers, target copies (the target row is known without any lookup) ----
    if (tid == 0) {
        const int lo = static_cast<int>((static_cast<int64_t>(P.nvec_row) * crank) / C);
        const int hi = static_cast<int>((static_cast<int64_t>(P.nvec_row) * (crank + 1)) / C);
        I.lo = lo;
        I.nvec = hi - lo;
        I.groups = (I.nvec + kGroupVecs - 1) / kGroupVecs;
        I.nchunk = max(1, min(kMaxChunks, I.groups / kWarps));
        for (int r = 0; r < 2; ++r)
            for (int k = 0; k < kMaxChunks; ++k) mbar_init(&bars[r][k], 1);
        fence_mbar_init();
        const uint64_t pol = policy_evict_first();
        const unsigned char *src = static_cast<const unsigned char *>(P.target) + static_cast<size_t>(item) * row_bytes +
                                   static_cast<size_t>(lo) * 16;
        for (int k = 0; k < I.nchunk; ++k) {
            int g0, g1, v0, v1;
            chunk_range(I.groups, I.nchunk, k, I.nvec, g0, g1, v0, v1);
            const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16;
            mbar_arrive_expect_tx(&bars[0][k], bytes);
            bulk_g2s(buf_t + v0, src + static_cast<size_t>(v0) * 16, bytes, &bars[0][k], pol);
        }
    }

    // ---- which request and position this item is (warp 0) ----
    // Loads whose values are needed only after pass 1 (the draft token, the uniforms) are
    // issued here and consumed later, so their latency hides behind the copies.
    int x_reg = -1;
    double u_acc_reg = 0.0, u_s_reg = 0.0;
    if (warp == 0) {
        int i;
        if (P.B < 8 * kWarp) {
            // one round trip: lane l holds row_off[8l .. 8l+7]; i + 1 offsets are <= item
            int cnt = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int idx = lane * 8 + k;
                cnt += (idx <= P.B ? __ldg(P.row_off + idx) : INT_MAX) <= item;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
            i = cnt - 1;
        } else {
            int lo = 0, hi = P.B;  // answer i in [lo, hi): row_off[i] <= item < row_off[i+1]
            while (hi - lo > kWarp) {
                const int step = (hi - lo + kWarp - 1) / kWarp;
                const int idx = lo + lane * step;
                const int v = idx < hi ? __ldg(P.row_off + idx) : INT_MAX;
                const unsigned m = __ballot_sync(0xffffffffu, v <= item);
                const int l = m ? 31 - __clz(static_cast<int>(m)) : 0;
                lo = lo + l * step;
                hi = min(lo + step, hi);
            }
            const int idx = lo + lane;
            const int v = idx < hi ? __ldg(P.row_off + idx) : INT_MAX;
            const unsigned m = __ballot_sync(0xffffffffu, v <= item);
            i = m ? lo + 31 - __clz(static_cast<int>(m)) : -1;
        }
        if (lane == 0) {
            int status = 0;
            if (i < 0 || i >= P.B) i = -1;
            int r0 = 0, r1 = 0, K = -1, j = -1, d = -1;
            if (i >= 0) {
                r0 = __ldg(P.row_off + i);
                r1 = __ldg(P.row_off + i + 1);
                K = r1 - r0 - 1;
                j = item - r0;
                d = r0 - i + j;
            }
            if (i < 0 || K < 0 || K > P.K_max || j < 0 || j > K || r1 > P.total_rows ||
                (j < K && (d < 0 || d >= P.total_rows - P.B)))
                status |= SPEC_REQ_BAD_SHAPE;
            I.req = i;
            I.pos = j;
            I.K = K;
            I.drow = d;
            I.pair = (status == 0 && j < K) ? 1 : 0;
            const float T = (i >= 0) ? (P.temperature ? __ldg(P.temperature + i) : P.temperature_scalar) : 1.0f;
            if (!(T >= 0.0f) || isinf(T)) status |= SPEC_REQ_BAD_PARAM;
            I.greedy = (T == 0.0f) ? 1 : 0;
            // s = log2(e)/T as a float pair, then s_hi moved toward zero so that s_lo > 0: a -inf
            // logit then gives -inf in both terms of exp_arg2 (a negative s_lo would make it NaN)
            F2 s = {0.0f, 0.0f};
            if (T > 0.0f && !isinf(T)) s = f2_div({kLog2eHi, kLog2eLo}, {T, 0.0f});
            if (s.hi > 0.0f && s.lo < 0.0f) {
                const float down = __uint_as_float(__float_as_uint(s.hi) - 1u);
                s.lo += s.hi - down;
                s.hi = down;
            }
            I.s_hi = s.hi;
            I.s_lo = fmaxf(s.lo, 1.401298464e-45f);
            if (status == 0) {
                u_acc_reg = __ldg(P.uniforms + item);
                u_s_reg = __ldg(P.uniforms + r1 - 1);
                if (I.pair) x_reg = __ldg(P.draft_tokens + d);
            }
            I.status = status;
            if (I.pair) {  // draft copies, once the draft row is known
                const uint64_t pol = policy_evict_first();
                const unsigned char *src = static_cast<const unsigned char *>(P.draft) +
                                           static_cast<size_t>(d) * row_bytes + static_cast<size_t>(I.lo) * 16;
                for (int k = 0; k < I.nchunk; ++k) {
                    int g0, g1, v0, v1;
                    chunk_range(I.groups, I.nchunk, k, I.nvec, g0, g1, v0, v1);
                    const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16;
                    mbar_arrive_expect_tx(&bars[1][k], bytes);
                    bulk_g2s(buf_d + v0, src + static_cast<size_t>(v0) * 16, bytes, &bars[1][k], pol);
                }
            }
        }
    }
    __syncthreads();

    const int nrows = 1 + I.pair;
    const int groups = I.groups, nvec = I.nvec, nchunk = I.nchunk;
    const bool greedy = I.greedy != 0;
    const float s_hi = I.s_hi, s_lo = I.s_lo;
    const float2 shi2 = f2splat(s_hi), slo2 = f2splat(s_lo);
    bool timed_out = false;

    // ---- pass 1: per-group statistics as the chunks land ----
    for (int r = 0; r < nrows; ++r) {
        const uint4 *buf = r ? buf_d : buf_t;
        for (int k = 0; k < nchunk; ++k) {
            if (!mbar_wait_sleep_bounded(&bars[r][k], 0, kSuspendNs, kMaxWaitTries)) timed_out = true;
            int g0, g1, v0, v1;
            chunk_range(groups, nchunk, k, nvec, g0, g1, v0, v1);
            for (int g = g0 + warp; g < g1; g += kWarps) {
                const int vbase = g * kGroupVecs + lane;
                if (greedy) {
                    // smallest index attaining the max; NaN / +inf make the row invalid
                    float best = -INFINITY;
                    int bidx = INT_MAX, bad = 0;
#pragma unroll
                    for (int q = 0; q < kVecPerLane; ++q) {
                        const int vi = vbase + q * kWarp;
                        float2 y[H];
                        load_vec2<DT>(buf, vi, nvec, y);
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const float v = (e & 1) ? y[e / 2].y : y[e / 2].x;
                            bad |= (v != v) || (v == INFINITY);
                            if (v > best) {
                                best = v;
                                bidx = (I.lo + vi) * E + e;
                            }
                        }
                    }
                    const float wbest = warp_max(best);
                    const int widx = warp_min_i32(best == wbest ? bidx : INT_MAX);
                    const int wbad = __any_sync(0xffffffffu, bad);
                    if (lane == 0) {
                        gref[r * P.groups_max + g] = wbest;
                        gsum[r * P.groups_max + g] = __int_as_float(wbad ? -1 : widx);
                    }
                } else {
                    // the group's vectors stay in registers between the max and the sums
                    uint4 wv[kVecPerLane];
                    float mx = -INFINITY;
#pragma unroll
                    for (int q = 0; q < kVecPerLane; ++q) {
                        const int vi = vbase + q * kWarp;
                        wv[q] = vi < nvec ? buf[vi] : kNegInfVec<DT>();
                        mx = fmaxf(mx, Elt<DT>::vmax(wv[q]));
                    }
                    mx = warp_max(mx);
                    // integral reference exponent: rescaling groups and CTAs is then exact; an
                    // all -inf group gets 0 (its sum is 0, or NaN if a NaN hides in it)
                    const float b = (mx == -INFINITY) ? 0.0f : floorf(mx * s_hi);
                    const float2 nb = f2splat(-b);
                    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int q = 0; q < kVecPerLane; ++q) {
                        float2 y[H];
                        Elt<DT>::unpack2(wv[q], y);
#pragma unroll
                        for (int h = 0; h < H; ++h) acc = __fadd2_rn(acc, ex2x2(exp_arg2(y[h], shi2, slo2, nb)));
                    }
                    const float a = warp_sum(acc.x + acc.y);
                    if (lane == 0) {
                        gref[r * P.groups_max + g] = b;
                        gsum[r * P.groups_max + g] = a;
                    }
                }
            }
        }
    }
    if (warp == 0 && lane == 0) I.x = x_reg;
    __syncthreads();

    // ---- this CTA's record: per-row statistics (lane 0 of warp r), the logits at x (warp 2) ----
    // One thread per row walks the group results in registers: a single wait on shared memory
    // instead of a chain of dependent warp shuffles, which queue behind the co-resident CTAs'
    // streaming loads.
    if (warp < nrows && lane == 0) {
        const int r = warp;
        const float *gr = gref + r * P.groups_max;
        const float *gs = gsum + r * P.groups_max;
        if (greedy) {
            float best = -INFINITY;
            int bidx = INT_MAX, bad = 0;
            for (int g = 0; g < groups; ++g) {
                const float v = gr[g];
                const int ix = __float_as_int(gs[g]);
                if (ix < 0) bad = 1;
                if (v > best || (v == best && ix < bidx)) {
                    best = v;
                    bidx = ix;
                }
            }
            mine1.gmax[r] = best;
            mine1.garg[r] = bidx;
            mine1.bad[r] = bad;
        } else {
            float Bc = -INFINITY;
            int bad = 0;
            for (int g = 0; g < groups; ++g) {
                const float sg = gs[g];
                if (!(sg >= 0.0f) || isinf(sg)) bad = 1;  // NaN or inf
                if (sg > 0.0f) Bc = fmaxf(Bc, gr[g]);
            }
            F2 acc = {0.0f, 0.0f};
            for (int g = 0; g < groups; ++g) {
                const float sg = gs[g];
                if (sg > 0.0f && !isinf(sg)) acc = f2_add(acc, {sg * pow2i(gr[g] - Bc), 0.0f});
            }
            mine1.B[r] = Bc;
            mine1.S_hi[r] = acc.hi;
            mine1.S_lo[r] = acc.lo;
            mine1.bad[r] = bad;
        }
    } else if (warp == 2 && lane == 0) {
        const int x = I.x;
        const int xl = x - I.lo * E;  // position of x in this slice
        const int has = I.pair && x >= 0 && xl >= 0 && xl < nvec * E;
        mine1.has_x = has;
        mine1.yx[0] = has ? Elt<DT>::at(buf_t, xl) : 0.0f;
        mine1.yx[1] = has ? Elt<DT>::at(buf_d, xl) : 0.0f;
    }
    __syncthreads();
    if (warp == 0) push_record(&mine1, xch1, crank, kEx1Words, C, lane);
    cluster_sync_all();  // #1: every slice's record is in every CTA

    // ---- combine the cluster (thread 0 walks the C records in CTA order), decide the accept test ----
    if (warp == 0) {
        float yx_t = 0.0f, yx_d = 0.0f;
        if (lane == 0) {
            for (int r = 0; r < nrows; ++r) {
                if (greedy) {
                    float best = -INFINITY;
                    int bidx = INT_MAX, bad = 0;
                    for (int c = 0; c < C; ++c) {
                        const float v = xch1[c].gmax[r];
                        const int ix = xch1[c].garg[r];
                        bad |= xch1[c].bad[r];
                        if (v > best || (v == best && ix < bidx)) {
                            best = v;
                            bidx = ix;
                        }
                    }
                    const int am = (bad || best == -INFINITY) ? -1 : bidx;
                    if (r == 0) I.argmax_t = am;
                    else I.argmax_d = am;
                } else {
                    float Bw = -INFINITY;
                    int bad = 0;
                    for (int c = 0; c < C; ++c) {
                        bad |= xch1[c].bad[r];
                        if (xch1[c].S_hi[r] > 0.0f) Bw = fmaxf(Bw, xch1[c].B[r]);
                    }
                    F2 S = {0.0f, 0.0f};
                    for (int c = 0; c < C; ++c) {
                        const F2 Sc = {xch1[c].S_hi[r], xch1[c].S_lo[r]};
                        if (Sc.hi > 0.0f) S = f2_add(S, f2_scale(Sc, xch1[c].B[r] - Bw));
                    }
                    if (r == 0) {
                        I.B_t = bad ? NAN : Bw;
                        I.S_t = S;
                    } else {
                        I.B_d = bad ? NAN : Bw;
                        I.S_d = S;
                    }
                }
            }
            for (int c = 0; c < C; ++c)
                if (xch1[c].has_x) {
                    yx_t = xch1[c].yx[0];
                    yx_d = xch1[c].yx[1];
                }
        }
        if (lane == 0) {
            int status = I.status | (timed_out ? REQ_TIMEOUT : 0);
            I.accept = 0;
            I.sample_kind = SAMPLE_NONE;
            I.rho = 0.0f;
            I.u_acc = d2f2(u_acc_reg);
            I.u_s = d2f2(u_s_reg);
            // row validity is reported together with a bad proposal (both are preconditions)
            if (!(status & (SPEC_REQ_BAD_SHAPE | SPEC_REQ_BAD_PARAM | REQ_TIMEOUT))) {
                if (greedy) {
                    if (I.argmax_t < 0 || (I.pair && I.argmax_d < 0)) status |= SPEC_REQ_BAD_LOGITS;
                    if (I.pair && (I.x < 0 || I.x >= P.V)) status |= SPEC_REQ_BAD_PROPOSAL;
                } else {
                    const bool ok_t = isfinite(I.B_t) && I.S_t.hi > 0.0f && isfinite(I.S_t.hi);
                    const bool ok_d = !I.pair || (isfinite(I.B_d) && I.S_d.hi > 0.0f && isfinite(I.S_d.hi));
                    if (!ok_t || !ok_d) status |= SPEC_REQ_BAD_LOGITS;
                    // q(x) == 0 is a bad proposal for Rule 2 (checked before any draw)
                    if (I.pair && (I.x < 0 || I.x >= P.V || yx_d == -INFINITY)) status |= SPEC_REQ_BAD_PROPOSAL;
                }
            }
            if (status == 0) {
                if (greedy) {
                    if (I.pair) {
                        I.accept = (I.x == I.argmax_t);
                        I.rho = I.accept ? 1.0f : 0.0f;
                        I.alpha = (I.argmax_t == I.argmax_d) ? 1.0f : 0.0f;
                    }
                } else {
                    I.inv_St = rcp_approx(I.S_t.hi);
                    if (I.pair) {
                        // rho = p(x)/q(x) = 2^E * S_d/S_t with E = (y_t - y_d) s - (B_t - B_d), all
                        // in float pairs; 2^E from ex2 of its fraction and an exact power of two
                        I.lam = f2_div(I.S_t, I.S_d);
                        float rho = 0.0f;
                        if (yx_t != -INFINITY) {
                            F2 Ex = f2_mul(f2_add({yx_t, 0.0f}, {-yx_d, 0.0f}), {s_hi, s_lo});
                            Ex = f2_add(Ex, {-(I.B_t - I.B_d), 0.0f});
                            const float n = floorf(Ex.hi);
                            const float f = (Ex.hi - n) + Ex.lo;
                            const F2 ratio = f2_div(I.S_d, I.S_t);
                            const float m = ex2(f) * (ratio.hi + ratio.lo);
                            if (n > 254.0f) {
                                rho = INFINITY;
                            } else if (n >= -252.0f) {
                                const float h = floorf(0.5f * n);
                                rho = m * pow2i(h) * pow2i(n - h);
                            }
                        }
                        I.rho = rho;
                        I.accept = (rho > 0.0f) && !f2_gt(I.u_acc, {rho, 0.0f});
                        I.c_t = I.B_t + __log2f(I.S_t.hi);
                        I.c_d = I.B_d + __log2f(I.S_d.hi);
                        if (!I.accept) I.sample_kind = SAMPLE_RESIDUAL;
                    } else {
                        I.sample_kind = SAMPLE_P;
                    }
                }
            }
            I.status = status;
        }
    }
    __syncthreads();
    // ---- pass 2 (pairs under Rule 2): alpha, and the residual where this position rejects ----
    float my_alpha = 0.0f;
    if (I.status == 0 && I.pair && !greedy) {
        if (I.sample_kind == SAMPLE_RESIDUAL) {
            const float2 nbt = f2splat(-I.B_t), nbd = f2splat(-I.B_d);
            const float2 nlh = f2splat(-I.lam.hi), nll = f2splat(-I.lam.lo), lh = f2splat(I.lam.hi);
            float2 acc_a = make_float2(0.0f, 0.0f);
            for (int g = warp; g < groups; g += kWarps) {
                float2 racc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int q = 0; q < kVecPerLane; ++q) {
                    const int vi = g * kGroupVecs + q * kWarp + lane;
                    float2 yt[H], yd[H];
                    load_vec2<DT>(buf_t, vi, nvec, yt);
                    load_vec2<DT>(buf_d, vi, nvec, yd);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 et = ex2x2(exp_arg2(yt[h], shi2, slo2, nbt));
                        const float2 ed = ex2x2(exp_arg2(yd[h], shi2, slo2, nbd));
                        const float2 r = __ffma2_rn(ed, nll, __ffma2_rn(ed, nlh, et));
                        racc = __fadd2_rn(racc, make_float2(fmaxf(r.x, 0.0f), fmaxf(r.y, 0.0f)));
                        const float2 m = __fmul2_rn(ed, lh);  // S_t * min(p, q): no cancellation
                        acc_a = __fadd2_rn(acc_a, make_float2(fminf(et.x, m.x), fminf(et.y, m.y)));
                    }
                }
                const float rs = warp_sum(racc.x + racc.y);
                if (lane == 0) gres[g] = rs;
            }
            my_alpha = (acc_a.x + acc_a.y) * I.inv_St;
        } else {
            const float2 nct = f2splat(-I.c_t), ncd = f2splat(-I.c_d);
            float2 acc = make_float2(0.0f, 0.0f);
            for (int g = warp; g < groups; g += kWarps) {
#pragma unroll
                for (int q = 0; q < kVecPerLane; ++q) {
                    const int vi = g * kGroupVecs + q * kWarp + lane;
                    if (vi >= nvec) continue;
                    float2 yt[H], yd[H];
                    Elt<DT>::unpack2(buf_t[vi], yt);
                    Elt<DT>::unpack2(buf_d[vi], yd);
#pragma unroll
                    for (int h = 0; h < H; ++h) {
                        const float2 at = __ffma2_rn(yt[h], shi2, nct), ad = __ffma2_rn(yd[h], shi2, ncd);
                        acc = __fadd2_rn(acc, make_float2(ex2(fminf(at.x, ad.x)), ex2(fminf(at.y, ad.y))));
                    }
                }
            }
            my_alpha = acc.x + acc.y;
        }
    }
    my_alpha = warp_sum(my_alpha);
    if (lane == 0) red_f[warp] = my_alpha;
    __syncthreads();
    if (warp == 0) {
        float a = lane < kWarps ? red_f[lane] : 0.0f;
        a = warp_sum(a);
        F2 z = {0.0f, 0.0f};
        if (I.sample_kind == SAMPLE_RESIDUAL)
            for (int g = lane; g < groups; g += kWarp) z = f2_add(z, {gres[g], 0.0f});
        z = warp_sum_f2(z);
        if (lane == 0) {
            mine2.alpha = a;
            mine2.Z_hi = z.hi;
            mine2.Z_lo = z.lo;
        }
        __syncwarp();
        push_record(&mine2, xch2, crank, kEx2Words, C, lane);
    }
    cluster_sync_all();  // #2: alpha and residual shares are in every CTA; no remote access after this

    // ---- cluster totals, the owner of the draw, item results (thread 0, CTAs in order) ----
    if (warp == 0) {
        float alpha_sum = 0.0f;
        int kind = I.sample_kind, fb = 0, owner = -1;
        F2 Zres = {0.0f, 0.0f}, Ztot = {0.0f, 0.0f}, t = {0.0f, 0.0f}, prefix = {0.0f, 0.0f};
        if (lane == 0) {
            for (int c = 0; c < C; ++c) {
                alpha_sum += xch2[c].alpha;
                Zres = f2_add(Zres, {xch2[c].Z_hi, xch2[c].Z_lo});
            }
            if (kind == SAMPLE_RESIDUAL && !(Zres.hi > 0.0f)) {
                kind = SAMPLE_P;  // zero residual mass: draw from p and say so
                fb = 1;
            }
            if (kind != SAMPLE_NONE && I.status == 0 && !greedy) {
                // masses of the law the draw uses, per CTA; the owner is the CTA whose running
                // total first exceeds u * Z (else the last CTA with mass, when rounding put u*Z
                // at the very end)
                for (int c = 0; c < C; ++c) {
                    const F2 Sc = {xch1[c].S_hi[0], xch1[c].S_lo[0]};
                    const F2 m = (kind == SAMPLE_RESIDUAL) ? F2{xch2[c].Z_hi, xch2[c].Z_lo}
                                                           : (Sc.hi > 0.0f ? f2_scale(Sc, xch1[c].B[0] - I.B_t)
                                                                           : F2{0.0f, 0.0f});
                    Ztot = f2_add(Ztot, m);
                }
                t = f2_mul(Ztot, I.u_s);
                F2 run = {0.0f, 0.0f}, last_run = {0.0f, 0.0f};
                int last = -1;
                for (int c = 0; c < C; ++c) {
                    const F2 Sc = {xch1[c].S_hi[0], xch1[c].S_lo[0]};
                    const F2 m = (kind == SAMPLE_RESIDUAL) ? F2{xch2[c].Z_hi, xch2[c].Z_lo}
                                                           : (Sc.hi > 0.0f ? f2_scale(Sc, xch1[c].B[0] - I.B_t)
                                                                           : F2{0.0f, 0.0f});
                    const F2 next = f2_add(run, m);
                    if (m.hi > 0.0f) {
                        last = c;
                        last_run = run;
                        if (owner < 0 && f2_gt(next, t)) {
                            owner = c;
                            prefix = run;
                        }
                    }
                    run = next;
                }
                if (owner < 0) {
                    owner = last;
                    prefix = last_run;
                }
            }
        }
        if (lane == 0) {
            I.sample_kind = kind;
            I.owner = owner;
            I.Ztot = Ztot;
            I.target_t = t;
            I.owner_prefix = prefix;
            if (crank == 0) {
                const int st = I.status;
                P.item_status[item] = st;
                P.item_fb[item] = fb;
                if (I.pair) {
                    const float alpha = greedy ? I.alpha : alpha_sum;
                    P.item_flag[item] = (st == 0) ? I.accept : 0;
                    P.alpha_ws[I.drow] = (st == 0) ? alpha : 0.0f;
                    if (P.alpha_rows) P.alpha_rows[I.drow] = (st == 0) ? alpha : NAN;
                    if (P.rho_rows) P.rho_rows[I.drow] = (st == 0) ? I.rho : NAN;
                    if (P.resid_rows)
                        P.resid_rows[I.drow] = (st == 0 && kind == SAMPLE_RESIDUAL && !greedy)
                                                   ? f2_div(Zres, I.S_t).hi
                                                   : -1.0f;
                } else {
                    P.item_flag[item] = 0;
                }
                if (st != 0 || (I.pair && I.accept)) {
                    P.item_tok[item] = -1;
                    P.item_prob[item] = NAN;
                    P.item_margin[item] = NAN;
                } else if (greedy) {
                    // Rule 1: the correction (or the extra token) is argmax p
                    P.item_tok[item] = I.argmax_t;
                    P.item_prob[item] = 1.0f;
                    P.item_margin[item] = NAN;
                } else if (owner < 0) {
                    P.item_tok[item] = -1;  // unreachable for a valid row: p always has mass
                    P.item_prob[item] = NAN;
                    P.item_margin[item] = NAN;
                }
            }
        }
    }
    __syncthreads();

    // ---- the draw: the owner CTA finds the group, then the vector, then the element ----
    if (warp == 0 && I.owner == crank) {
        const int kind = I.sample_kind;
        const F2 local = f2_sub(I.target_t, I.owner_prefix);
        int gsel = -1, last_g = -1;
        F2 before = {0.0f, 0.0f}, last_before = {0.0f, 0.0f}, run = {0.0f, 0.0f};
        for (int base = 0; base < groups; base += kWarp) {
            const int g = base + lane;
            float m = 0.0f;
            if (g < groups) {
                if (kind == SAMPLE_RESIDUAL) {
                    m = gres[g];
                } else {
                    const float sg = gsum[g];
                    m = (sg > 0.0f) ? sg * pow2i(gref[g] - I.B_t) : 0.0f;
                }
            }
            const F2 incl = f2_add(run, warp_scan_f2({m, 0.0f}, lane));
            const unsigned hit = __ballot_sync(0xffffffffu, g < groups && m > 0.0f && f2_gt(incl, local));
            const unsigned posm = __ballot_sync(0xffffffffu, g < groups && m > 0.0f);
            if (hit) {
                const int l = __ffs(hit) - 1;
                gsel = base + l;
                before = shfl_f2(f2_sub(incl, {m, 0.0f}), l);
                break;
            }
            if (posm) {
                const int l = 31 - __clz(static_cast<int>(posm));
                last_g = base + l;
                last_before = shfl_f2(f2_sub(incl, {m, 0.0f}), l);
            }
            run = shfl_f2(incl, kWarp - 1);
        }
        const bool clamped = gsel < 0;  // rounding put u*Z past the last group with mass
        if (clamped) {
            gsel = last_g;
            before = last_before;
        }
        int tok = -1;
        float wsel = 0.0f, margin = 0.0f, unit = 1.0f;
        if (gsel >= 0) {
            const float bg = (kind == SAMPLE_RESIDUAL) ? 0.0f : gref[gsel];
            // group units: residual weights are already in cluster units; P weights are in units
            // of 2^b_g, which is 2^(b_g - B_t) cluster units (an exact power of two)
            unit = (kind == SAMPLE_RESIDUAL) ? 1.0f : pow2i(bg - I.B_t);
            const F2 rem = f2_sub(local, before);
            const float lt = (rem.hi + rem.lo) * ((kind == SAMPLE_RESIDUAL) ? 1.0f : pow2i(I.B_t - bg));
            float run2 = 0.0f, last_w = 0.0f;
            int last_tok = -1;
            for (int q = 0; q < kVecPerLane; ++q) {
                const int vi = gsel * kGroupVecs + q * kWarp + lane;
                float w[E];
                vec_weights<DT>(kind, buf_t, buf_d, vi, nvec, I, bg, w);
                float ls = 0.0f;
#pragma unroll
                for (int e = 0; e < E; ++e) ls += w[e];
                float incl = ls;
#pragma unroll
                for (int o = 1; o < kWarp; o <<= 1) {
                    const float n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += n;
                }
                incl += run2;
                // this lane's element that takes the target, if any; and its last with mass
                int found = -1, lastp = -1;
                float fprev = 0.0f, c = incl - ls, wf = 0.0f, wl = 0.0f;
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
                if (hit) {
                    const int l = __ffs(hit) - 1;
                    const int e_sel = __shfl_sync(0xffffffffu, found, l);
                    const float c0 = __shfl_sync(0xffffffffu, fprev, l);
                    wsel = __shfl_sync(0xffffffffu, wf, l);
                    tok = (I.lo + gsel * kGroupVecs + q * kWarp + l) * E + e_sel;
                    margin = fminf(lt - c0, c0 + wsel - lt) * unit * rcp_approx(I.Ztot.hi);
                    break;
                }
                if (posm) {
                    const int l = 31 - __clz(static_cast<int>(posm));
                    last_tok = (I.lo + gsel * kGroupVecs + q * kWarp + l) * E + __shfl_sync(0xffffffffu, lastp, l);
                    last_w = __shfl_sync(0xffffffffu, wl, l);
                }
                run2 = __shfl_sync(0xffffffffu, incl, kWarp - 1);
            }
            if (tok < 0) {  // rounding: the last element with mass
                tok = last_tok;
                wsel = last_w;
                margin = 0.0f;
            }
        }
        if (lane == 0) {
            P.item_tok[item] = tok;
            P.item_prob[item] = tok >= 0 ? wsel * unit * rcp_approx(I.Ztot.hi) : NAN;
            P.item_margin[item] = tok >= 0 ? margin : NAN;
        }
    }
    if (timed_out) {
        // a copy did not land in time: wait (bounded) once more so none is left in flight
        for (int r = 0; r < nrows; ++r)
            for (int k = 0; k < nchunk; ++k) mbar_wait_sleep_bounded(&bars[r][k], 0, kSuspendNs, kMaxWaitTries);
    }
}

}  // namespace spec
