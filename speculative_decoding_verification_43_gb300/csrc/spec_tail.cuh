// The tail of a verification round on the device: the compaction (spec_compact) and the gamma
// choice (spec_choose_gamma), as device functions. spec_compact and spec_choose_gamma run them as
// kernels of their own; spec_verify_round runs both in the last CTA of the verifier's kernel
// (included by spec_verify.cu and spec_compact.cu).
#pragma once

#include <climits>
#include <cstdint>

#include "spec_device.cuh"
#include "spec_math.cuh"
#include "spec_verify.h"

namespace spec {

constexpr int kCompactThreads = 1024;

struct CompactParams {
    int32_t B, page_size, max_blocks, total_rows;
    const int32_t *row_off, *accept_len, *n_emitted, *out_tokens, *req_status, *prefix_len,
        *cand_kv_rows, *block_table;
    int32_t *out_off, *packed_tokens, *packed_pos, *kv_off, *kv_src, *kv_dst, *new_seq_len,
        *new_kv_len, *new_draft_len, *compact_status;
};

// Block-wide exclusive scan of one int per thread over a CTA of NT threads (NT a multiple of 32,
// at most 1024); returns the exclusive prefix and the total. warp_tot: kWarp + 1 ints of scratch.
template <int NT>
__device__ __forceinline__ int block_exscan(int v, int *warp_tot, int &total) {
    constexpr int kNW = NT / kWarp;
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
        int t = lane < kNW ? warp_tot[lane] : 0;
        int ti = t;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += n;
        }
        if (lane < kNW) warp_tot[lane] = ti - t;  // exclusive prefix of the warp totals
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

// Scratch of the compaction in a CTA of NT threads (shared memory, supplied by the caller).
template <int NT>
struct CompactScratch {
    int tot_n[kWarp + 1];
    int tot_e[kWarp + 1];
    CopyJob job[NT];
};

// The compaction of every request by one CTA of NT threads. wait: call griddep_wait() once the
// caller's offsets are checked (a kernel of its own waits for the kernel ahead of it; a caller that
// has waited already passes false). known_ok: 1 / 0 when the offsets were checked already (the
// selection of the same round, same array), -1 to check them here.
template <int NT>
__device__ __forceinline__ void compact_body(const CompactParams &P, bool wait, int known_ok, CompactScratch<NT> &S) {
    int *const tot_n = S.tot_n;
    int *const tot_e = S.tot_e;
    CopyJob *const job = S.job;
    int carry_n = 0, carry_e = 0;
    // offsets must start at 0, end at total_rows and grow by at least one row per request;
    // otherwise every request is BAD_SHAPE, so packed writes stay within their capacities. The
    // offsets are the caller's input, read while the kernel ahead of this one still runs.
    bool offsets_ok = known_ok == 1;
    if (known_ok < 0) {
        int bad_off = (__ldg(P.row_off) != 0) || (__ldg(P.row_off + P.B) != P.total_rows);
        for (int i = threadIdx.x; i < P.B && !bad_off; i += NT)
            if (__ldg(P.row_off + i + 1) <= __ldg(P.row_off + i)) bad_off = 1;
        offsets_ok = !__syncthreads_or(bad_off);
    }
    if (wait) griddep_wait();  // the outputs of the kernel ahead are ready from here on
    for (int base = 0; base < P.B; base += NT) {
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
        const int off_n = carry_n + block_exscan<NT>(n, tot_n, total_n);
        const int off_e = carry_e + block_exscan<NT>(E, tot_e, total_e);
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
        const int nreq = min(NT, P.B - base);
        for (int q = threadIdx.x / kWarp; q < nreq; q += NT / kWarp) {
            const CopyJob jb = job[q];
            const int req = base + q, d0 = jb.r0 - req;
            for (int j = lane; j < jb.n; j += kWarp) {
                if (SPEC_IN(jb.off_n + j, P.total_rows, DBG_PACKED) && SPEC_IN(jb.r0 + j, P.total_rows, DBG_OUT_ROWS)) {
                    P.packed_tokens[jb.off_n + j] = P.out_tokens[jb.r0 + j];
                    P.packed_pos[jb.off_n + j] = jb.Pi + j;
                }
            }
            for (int j = lane; j < jb.E; j += kWarp) {
                const int pos = jb.Pi + j;
                const int blk = P.block_table[static_cast<int64_t>(req) * P.max_blocks + pos / P.page_size];
                if (SPEC_IN(jb.off_e + j, P.total_rows - P.B, DBG_PACKED) && SPEC_IN(d0 + j, P.total_rows - P.B, DBG_PACKED)) {
                    P.kv_src[jb.off_e + j] = P.cand_kv_rows[d0 + j];
                    P.kv_dst[jb.off_e + j] = blk * P.page_size + pos % P.page_size;
                }
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
