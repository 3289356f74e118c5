// The tail of a verification round on the device: the selection (spec_verify), the compaction
// (spec_compact) and the gamma choice (spec_choose_gamma), as device functions. Each entry point
// runs one of them as a kernel of its own; spec_verify_round runs all three in one kernel, one
// after another in one CTA (included by spec_verify.cu and spec_compact.cu).
#pragma once

#include <climits>
#include <cstdint>

#include "spec_device.cuh"
#include "spec_math.cuh"
#include "spec_verify.h"

namespace spec {

struct FinParams {
    const int32_t *row_off;
    const int32_t *draft_tokens;
    const int32_t *stop_token;
    const int32_t *max_new;
    int32_t B, K_max, total_rows;
    const int32_t *item_flag, *item_tok, *item_status, *item_fb;
    const float *item_prob, *item_margin, *alpha_ws;
    int32_t *accept_len, *n_emitted, *out_tokens, *req_status, *fallback, *alpha_count;
    float *frontier_prob, *frontier_margin;
    double *alpha_sum;
    int32_t *depth_reached, *depth_accepted;  // [K_max] each, or NULL
};

constexpr int kFinThreads = 1024;

// The selection of every request (one CTA of kFinThreads threads): the first rejection, the emitted
// tokens, stopping, the alpha reduction and the depth histogram. Waits for the kernel ahead of it
// in the stream (the per-position kernel) after reading the offsets.
__device__ __forceinline__ bool select_body(const FinParams &P) {
    __shared__ float red_hi[kFinThreads / kWarp];
    __shared__ float red_lo[kFinThreads / kWarp];
    __shared__ int red_n[kFinThreads / kWarp];
    // depth statistics ("M7.8 - Speculative Serving", 0x02D): requests that reached / accepted
    // depth j = 1..K_max
    __shared__ int hist_r[64], hist_a[64];
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    griddep_launch_dependents();
    if (threadIdx.x < 64) hist_r[threadIdx.x] = hist_a[threadIdx.x] = 0;
    // Inputs first (they do not depend on the per-position kernel): the offsets must start at 0,
    // end at total_rows and grow by at least one row per request; otherwise every request is
    // BAD_SHAPE and nothing is read through them.
    int bad_off = (__ldg(P.row_off) != 0) || (__ldg(P.row_off + P.B) != P.total_rows);
    for (int i = threadIdx.x; i < P.B && !bad_off; i += kFinThreads)
        if (__ldg(P.row_off + i + 1) <= __ldg(P.row_off + i)) bad_off = 1;
    const bool global_ok = !__syncthreads_or(bad_off);
    // The inputs of this warp's first kPre requests (offsets, budget, stop token, draft tokens)
    // also load before the wait: after it, a request costs one round of loads, not two.
    constexpr int kPre = 4;
    int pr_r0[kPre], pr_r1[kPre], pr_cap[kPre], pr_stop[kPre], pr_x0[kPre], pr_x1[kPre];
#pragma unroll
    for (int q = 0; q < kPre; ++q) {
        const int i = warp + q * (kFinThreads / kWarp);
        pr_r0[q] = pr_r1[q] = 0;
        pr_cap[q] = INT_MAX;
        pr_stop[q] = pr_x0[q] = pr_x1[q] = -1;
        if (i < P.B) {
            pr_r0[q] = __ldg(P.row_off + i);
            pr_r1[q] = __ldg(P.row_off + i + 1);
            if (P.max_new) pr_cap[q] = __ldg(P.max_new + i);
            if (P.stop_token) pr_stop[q] = __ldg(P.stop_token + i);
        }
    }
#pragma unroll
    for (int q = 0; q < kPre; ++q) {
        const int i = warp + q * (kFinThreads / kWarp);
        const int K = pr_r1[q] - pr_r0[q] - 1, d0 = pr_r0[q] - i;
        if (i < P.B && global_ok && K >= 0 && K <= P.K_max && pr_r0[q] >= 0 && pr_r1[q] <= P.total_rows && d0 >= 0) {
            if (lane < K) pr_x0[q] = __ldg(P.draft_tokens + d0 + lane);
            if (lane + kWarp < K) pr_x1[q] = __ldg(P.draft_tokens + d0 + lane + kWarp);
        }
    }
    griddep_wait();  // the per-position results are complete from here on
    F2 asum = {0.0f, 0.0f};
    int acnt = 0;
    // one request per warp at a time, lane j taking position j (K_max <= 64: two rounds at most);
    // every per-position value is fetched in one round of independent loads
    for (int i = warp, q = 0; i < P.B; i += kFinThreads / kWarp, ++q) {
        int r0 = 0, r1 = 0, n_cap = INT_MAX, stop = -1, px0 = -1, px1 = -1;
        if (q < kPre) {
#pragma unroll
            for (int k = 0; k < kPre; ++k)
                if (k == q) {
                    r0 = pr_r0[k];
                    r1 = pr_r1[k];
                    n_cap = pr_cap[k];
                    stop = pr_stop[k];
                    px0 = pr_x0[k];
                    px1 = pr_x1[k];
                }
        } else {
            r0 = __ldg(P.row_off + i);
            r1 = __ldg(P.row_off + i + 1);
            if (P.max_new) n_cap = __ldg(P.max_new + i);
            if (P.stop_token) stop = __ldg(P.stop_token + i);
        }
        const int K = r1 - r0 - 1;
        const int d0 = r0 - i;
        int status = 0;
        if (!global_ok || K < 0 || K > P.K_max || r0 < 0 || r1 > P.total_rows || d0 < 0) status |= SPEC_REQ_BAD_SHAPE;
        // positions j = lane and j = lane + 32
        int st_items = 0;
        unsigned rej_lo = 0u, rej_hi = 0u;
        int tok0 = -1, tok1 = -1, fb0 = 0, fb1 = 0, x0 = -1, x1 = -1;
        float pr0 = NAN, pr1 = NAN, mg0 = NAN, mg1 = NAN, al0 = 0.0f, al1 = 0.0f;
        int tok2 = -1, fb2 = 0;  // position 64 (lane 0), when K = 64
        float pr2 = NAN, mg2 = NAN;
        if (!status) {
            const int j0 = lane, j1 = lane + kWarp;
            const bool in0 = j0 <= K, in1 = j1 <= K;
            if (in0) {
                st_items |= P.item_status[r0 + j0];
                tok0 = P.item_tok[r0 + j0];
                pr0 = P.item_prob[r0 + j0];
                mg0 = P.item_margin[r0 + j0];
                fb0 = P.item_fb[r0 + j0];
                if (j0 < K) {
                    x0 = q < kPre ? px0 : __ldg(P.draft_tokens + d0 + j0);
                    al0 = P.alpha_ws[d0 + j0];
                }
            }
            if (in1) {
                st_items |= P.item_status[r0 + j1];
                tok1 = P.item_tok[r0 + j1];
                pr1 = P.item_prob[r0 + j1];
                mg1 = P.item_margin[r0 + j1];
                fb1 = P.item_fb[r0 + j1];
                if (j1 < K) {
                    x1 = q < kPre ? px1 : __ldg(P.draft_tokens + d0 + j1);
                    al1 = P.alpha_ws[d0 + j1];
                }
            }
            if (K == 2 * kWarp && lane == 0) {  // K_max <= 64: the frontier slot of K = 64
                st_items |= P.item_status[r0 + K];
                tok2 = P.item_tok[r0 + K];
                pr2 = P.item_prob[r0 + K];
                mg2 = P.item_margin[r0 + K];
                fb2 = P.item_fb[r0 + K];
            }
            rej_lo = __ballot_sync(0xffffffffu, j0 < K && P.item_flag[r0 + j0] == 0);
            rej_hi = __ballot_sync(0xffffffffu, j1 < K && P.item_flag[r0 + j1] == 0);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) st_items |= __shfl_xor_sync(0xffffffffu, st_items, o);
        }
        status |= st_items;
        if (status) {
            if (!(status & SPEC_REQ_BAD_SHAPE) || (K >= 0 && r1 <= P.total_rows && r0 >= 0))
                for (int j = lane; j <= K; j += kWarp) P.out_tokens[r0 + j] = -1;
            if (lane == 0) {
                P.req_status[i] = status;
                P.accept_len[i] = 0;
                if (P.n_emitted) P.n_emitted[i] = 0;
                if (P.frontier_prob) P.frontier_prob[i] = NAN;
                if (P.frontier_margin) P.frontier_margin[i] = NAN;
                if (P.fallback) P.fallback[i] = 0;
            }
            continue;
        }
        // A = index of the first rejected position (K when all are accepted)
        const int A = rej_lo ? __ffs(rej_lo) - 1 : (rej_hi ? kWarp + __ffs(rej_hi) - 1 : K);
        // the frontier's values, from the lane that holds position A
        const int la = A & (kWarp - 1), half = A >> 5;  // 0, 1, or 2 (A = 64, lane 0)
        const int frontier = __shfl_sync(0xffffffffu, half == 0 ? tok0 : half == 1 ? tok1 : tok2, la);
        const float fprob = __shfl_sync(0xffffffffu, half == 0 ? pr0 : half == 1 ? pr1 : pr2, la);
        const float fmarg = __shfl_sync(0xffffffffu, half == 0 ? mg0 : half == 1 ? mg1 : mg2, la);
        const int ffb = __shfl_sync(0xffffffffu, half == 0 ? fb0 : half == 1 ? fb1 : fb2, la);
        const int out0 = (lane < A) ? x0 : (lane == A ? frontier : -1);
        const int out1 = (lane + kWarp < A) ? x1 : (lane + kWarp == A ? frontier : -1);
        int n = min(A + 1, max(n_cap, 0));
        if (stop >= 0) {
            const unsigned h0 = __ballot_sync(0xffffffffu, lane < n && out0 == stop);
            const unsigned h1 = __ballot_sync(0xffffffffu, lane + kWarp < n && out1 == stop);
            if (h0)
                n = __ffs(h0);
            else if (h1)
                n = kWarp + __ffs(h1);
        }
        if (lane <= K) P.out_tokens[r0 + lane] = lane < n ? out0 : -1;
        if (lane + kWarp <= K) P.out_tokens[r0 + lane + kWarp] = lane + kWarp < n ? out1 : -1;
        if (lane == 0 && K == 2 * kWarp) P.out_tokens[r0 + K] = (A == K && n > K) ? frontier : -1;
        asum = f2_add(f2_add(asum, {al0, 0.0f}), {al1, 0.0f});
        // depth j + 1 was reached when the first j drafts were accepted, accepted when j < A
        if (P.depth_reached) {
            if (lane < K && lane <= A) atomicAdd(&hist_r[lane], 1);
            if (lane + kWarp < K && lane + kWarp <= A) atomicAdd(&hist_r[lane + kWarp], 1);
        }
        if (P.depth_accepted) {
            if (lane < K && lane < A) atomicAdd(&hist_a[lane], 1);
            if (lane + kWarp < K && lane + kWarp < A) atomicAdd(&hist_a[lane + kWarp], 1);
        }
        if (lane == 0) {
            acnt += K;
            P.req_status[i] = 0;
            P.accept_len[i] = A;
            if (P.n_emitted) P.n_emitted[i] = n;
            if (P.frontier_prob) P.frontier_prob[i] = fprob;
            if (P.frontier_margin) P.frontier_margin[i] = fmarg;
            if (P.fallback) P.fallback[i] = ffb;
        }
    }
    asum = warp_sum_f2(asum);
    if (lane == 0) {
        red_hi[warp] = asum.hi;
        red_lo[warp] = asum.lo;
        red_n[warp] = acnt;
    }
    __syncthreads();
    for (int j = threadIdx.x; j < P.K_max; j += kFinThreads) {
        if (P.depth_reached) P.depth_reached[j] = hist_r[j];
        if (P.depth_accepted) P.depth_accepted[j] = hist_a[j];
    }
    if (warp == 0) {
        F2 a = {red_hi[lane], red_lo[lane]};
        int c = red_n[lane];
        a = warp_sum_f2(a);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0) {
            // the one float64 operation of the call: the pair becomes the output double
            if (P.alpha_sum) *P.alpha_sum = static_cast<double>(a.hi) + static_cast<double>(a.lo);
            if (P.alpha_count) *P.alpha_count = c;
        }
    }
    return global_ok;  // the offsets passed their checks
}


constexpr int kCompactThreads = 1024;

struct CompactParams {
    int32_t B, page_size, max_blocks, total_rows;
    const int32_t *row_off, *accept_len, *n_emitted, *out_tokens, *req_status, *prefix_len,
        *cand_kv_rows, *block_table;
    int32_t *out_off, *packed_tokens, *packed_pos, *kv_off, *kv_src, *kv_dst, *new_seq_len,
        *new_kv_len, *new_draft_len, *compact_status;
};

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix and the total.
__device__ __forceinline__ int block_exscan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    int incl = v;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == kWarp - 1) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
        int ti = t;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += n;
        }
        warp_tot[lane] = ti - t;  // exclusive prefix of the warp totals
        if (lane == kWarp - 1) warp_tot[kWarp] = ti;
    }
    __syncthreads();
    const int ex = warp_tot[warp] + incl - v;
    total = warp_tot[kWarp];
    __syncthreads();
    return ex;
}

// The per-request values of one chunk of requests, for the copy phase.
struct CopyJob {
    int off_n, off_e, n, E, r0, Pi;
};

// The compaction of every request (one CTA of kCompactThreads threads). wait: call griddep_wait()
// once the caller's offsets are checked (a kernel of its own waits for the kernel ahead of it;
// the round's tail kernel has waited already). known_ok: 1 / 0 when the offsets were checked
// already (the selection of the same round, same array), -1 to check them here.
__device__ __forceinline__ void compact_body(const CompactParams &P, bool wait, int known_ok = -1) {
    __shared__ int tot_n[kWarp + 1];
    __shared__ int tot_e[kWarp + 1];
    __shared__ CopyJob job[kCompactThreads];
    int carry_n = 0, carry_e = 0;
    // offsets must start at 0, end at total_rows and grow by at least one row per request;
    // otherwise every request is BAD_SHAPE, so packed writes stay within their capacities. The
    // offsets are the caller's input, read while the kernel ahead of this one still runs.
    bool offsets_ok = known_ok == 1;
    if (known_ok < 0) {
        int bad_off = (__ldg(P.row_off) != 0) || (__ldg(P.row_off + P.B) != P.total_rows);
        for (int i = threadIdx.x; i < P.B && !bad_off; i += kCompactThreads)
            if (__ldg(P.row_off + i + 1) <= __ldg(P.row_off + i)) bad_off = 1;
        offsets_ok = !__syncthreads_or(bad_off);
    }
    if (wait) griddep_wait();  // the outputs of the kernel ahead are ready from here on
    for (int base = 0; base < P.B; base += kCompactThreads) {
        const int i = base + static_cast<int>(threadIdx.x);
        int n = 0, E = 0, status = 0, K = 0, r0 = 0, Pi = 0;
        if (i < P.B) {
            r0 = P.row_off[i];
            K = P.row_off[i + 1] - r0 - 1;
            Pi = P.prefix_len[i];
            status = P.req_status ? P.req_status[i] : 0;
            if (!offsets_ok || K < 0 || r0 < 0 || P.row_off[i + 1] > P.total_rows) status |= SPEC_REQ_BAD_SHAPE;
            if (!status) {
                const int A = P.accept_len[i];
                n = P.n_emitted ? P.n_emitted[i] : A + 1;
                if (A < 0 || A > K || n < 0 || n > K + 1) status |= SPEC_REQ_BAD_SHAPE;
                E = min(A, n);
                // every committed position P..P+E-1 needs a page of this request's table
                if (!status && E > 0) {
                    if (Pi < 0 || (Pi + E - 1) / P.page_size >= P.max_blocks) {
                        status |= SPEC_REQ_BAD_BLOCKS;
                    } else {
                        for (int pg = Pi / P.page_size; pg <= (Pi + E - 1) / P.page_size; ++pg)
                            if (P.block_table[static_cast<int64_t>(i) * P.max_blocks + pg] < 0) status |= SPEC_REQ_BAD_BLOCKS;
                    }
                }
                if (status) n = E = 0;
            }
        }
        int total_n, total_e;
        const int off_n = carry_n + block_exscan(n, tot_n, total_n);
        const int off_e = carry_e + block_exscan(E, tot_e, total_e);
        job[threadIdx.x] = {off_n, off_e, n, E, r0, Pi};
        if (i < P.B) {
            P.out_off[i] = off_n;
            P.kv_off[i] = off_e;
            P.new_seq_len[i] = Pi + n;
            P.new_kv_len[i] = Pi + E;
            if (P.new_draft_len) P.new_draft_len[i] = Pi + max(min(E, K - 1), 0);
            if (P.compact_status) P.compact_status[i] = status;
        }
        carry_n += total_n;
        carry_e += total_e;
        // the copies: one warp per request, one lane per position, so that a request's loads are
        // independent of each other (a thread per request would wait for each load in turn)
        __syncthreads();
        const int lane = threadIdx.x % kWarp;
        const int nreq = min(kCompactThreads, P.B - base);
        for (int q = threadIdx.x / kWarp; q < nreq; q += kCompactThreads / kWarp) {
            const CopyJob jb = job[q];
            const int req = base + q, d0 = jb.r0 - req;
            for (int j = lane; j < jb.n; j += kWarp) {
                P.packed_tokens[jb.off_n + j] = P.out_tokens[jb.r0 + j];
                P.packed_pos[jb.off_n + j] = jb.Pi + j;
            }
            for (int j = lane; j < jb.E; j += kWarp) {
                const int pos = jb.Pi + j;
                const int blk = P.block_table[static_cast<int64_t>(req) * P.max_blocks + pos / P.page_size];
                P.kv_src[jb.off_e + j] = P.cand_kv_rows[d0 + j];
                P.kv_dst[jb.off_e + j] = blk * P.page_size + pos % P.page_size;
            }
        }
        __syncthreads();  // job[] is rewritten by the next chunk
    }
    if (threadIdx.x == 0) {
        P.out_off[P.B] = carry_n;
        P.kv_off[P.B] = carry_e;
    }
}

// The objective in float pairs on the device (float64 is slow here): the committed count as the
// tail sum 1 + alpha + ... + alpha^gamma (M7.8 section 0x02), which needs no division and is
// gamma + 1 exactly at alpha = 1, and candidates compared by cross-multiplication:
// f(g1) > f(g2)  <=>  committed(g1) (g2 c + 1) > committed(g2) (g1 c + 1).
struct GammaParams {
    const double *alpha_sum;
    const int32_t *alpha_count;
    float prev_hi, prev_lo, c_hi, c_lo;
    int gmin, gmax;
    int32_t *gamma_out;
    double *alpha_out;
};

// One thread.
__device__ __forceinline__ void gamma_body(const GammaParams &G) {
    const double *alpha_sum = G.alpha_sum;
    const int32_t *alpha_count = G.alpha_count;
    const float prev_hi = G.prev_hi, prev_lo = G.prev_lo, c_hi = G.c_hi, c_lo = G.c_lo;
    const int gmin = G.gmin, gmax = G.gmax;
    int32_t *gamma_out = G.gamma_out;
    double *alpha_out = G.alpha_out;
    const int n = *alpha_count;
    const float n_hi = static_cast<float>(n);
    const F2 nf = f2_norm(n_hi, static_cast<float>(n - static_cast<int>(n_hi)));  // exact above 2^24 too
    F2 alpha = n > 0 ? f2_div(d2f2(*alpha_sum), nf) : F2{prev_hi, prev_lo};
    if (!(alpha.hi > 0.0f)) alpha = {0.0f, 0.0f};
    if (alpha.hi > 1.0f || (alpha.hi == 1.0f && alpha.lo > 0.0f)) alpha = {1.0f, 0.0f};
    const F2 c = {c_hi, c_lo};
    F2 pw = {1.0f, 0.0f}, committed = {1.0f, 0.0f};  // gamma = 0
    for (int g = 1; g <= gmin; ++g) {
        pw = f2_mul(pw, alpha);
        committed = f2_add(committed, pw);
    }
    int best = gmin;
    F2 best_c = committed;
    F2 best_den = f2_add(f2_mul({static_cast<float>(gmin), 0.0f}, c), {1.0f, 0.0f});
    for (int g = gmin + 1; g <= gmax; ++g) {
        pw = f2_mul(pw, alpha);
        committed = f2_add(committed, pw);
        const F2 den = f2_add(f2_mul({static_cast<float>(g), 0.0f}, c), {1.0f, 0.0f});
        if (f2_gt(f2_mul(committed, best_den), f2_mul(best_c, den))) {  // strict: a tie keeps the smaller
            best = g;
            best_c = committed;
            best_den = den;
        }
    }
    *gamma_out = best;
    *alpha_out = static_cast<double>(alpha.hi) + static_cast<double>(alpha.lo);
}


// Host (spec_compact.cu): the kernel parameters of the compaction and of the gamma choice from
// their arguments, SPEC_ERR_INVALID_ARG when the arguments are bad.
spec_status compact_params(const spec_compact_args *a, CompactParams &P);
spec_status gamma_params(const double *alpha_sum, const int32_t *alpha_count, double alpha_prev, double c,
                         int32_t gamma_min, int32_t gamma_max, int32_t *gamma_out, double *alpha_out, GammaParams &G);

}  // namespace spec
