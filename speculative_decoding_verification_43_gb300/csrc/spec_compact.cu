// Ragged compaction of a verified round (spec_compact) and the gamma controller
// (spec_choose_gamma, spec_gamma_objective, and their per-depth forms spec_choose_gamma_depth,
// spec_depth_objective). See include/spec_verify.h for the contract.
//
// Compaction follows "M7.8 - Speculative Serving", sections 0x03C (L_out = P+A+1, L_kv = P+A;
// positions stay contiguous, padding never becomes history) and 0x09 (with stopping:
// L_out = P+E+F, L_target = P+E, L_draft = P+min(E, K-1)). One CTA scans the per-request
// counts in tiles of 1024 requests, carrying the running offsets, then scatters each request's
// tokens, positions and KV row moves.
//
// The gamma objective is the expected wall-time improvement of SOTA-227 ("Why it is free
// rather than a trade"): (1 - alpha^(gamma+1)) / ((1 - alpha)(gamma*c + 1)).
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
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

__global__ void __launch_bounds__(kCompactThreads) spec_compact_kernel(const CompactParams P) {
    __shared__ int tot_n[kWarp + 1];
    __shared__ int tot_e[kWarp + 1];
    griddep_launch_dependents();
    griddep_wait();  // launched behind the previous kernel of the stream: its outputs are ready now
    int carry_n = 0, carry_e = 0;
    // offsets must start at 0, end at total_rows and grow by at least one row per request;
    // otherwise every request is BAD_SHAPE, so packed writes stay within their capacities
    int bad_off = (P.row_off[0] != 0) || (P.row_off[P.B] != P.total_rows);
    for (int i = threadIdx.x; i < P.B && !bad_off; i += kCompactThreads)
        if (P.row_off[i + 1] <= P.row_off[i]) bad_off = 1;
    const bool offsets_ok = !__syncthreads_or(bad_off);
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
        if (i < P.B) {
            P.out_off[i] = off_n;
            P.kv_off[i] = off_e;
            for (int j = 0; j < n; ++j) {
                P.packed_tokens[off_n + j] = P.out_tokens[r0 + j];
                P.packed_pos[off_n + j] = Pi + j;
            }
            const int d0 = r0 - i;
            for (int j = 0; j < E; ++j) {
                const int pos = Pi + j;
                const int blk = P.block_table[static_cast<int64_t>(i) * P.max_blocks + pos / P.page_size];
                P.kv_src[off_e + j] = P.cand_kv_rows[d0 + j];
                P.kv_dst[off_e + j] = blk * P.page_size + pos % P.page_size;
            }
            P.new_seq_len[i] = Pi + n;
            P.new_kv_len[i] = Pi + E;
            if (P.new_draft_len) P.new_draft_len[i] = Pi + max(min(E, K - 1), 0);
            if (P.compact_status) P.compact_status[i] = status;
        }
        carry_n += total_n;
        carry_e += total_e;
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
__global__ void spec_gamma_kernel(const double *alpha_sum, const int32_t *alpha_count, float prev_hi, float prev_lo,
                                  float c_hi, float c_lo, int gmin, int gmax, int32_t *gamma_out, double *alpha_out) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    griddep_wait();
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


// Per-depth rates ("M7.8 - Speculative Serving", sections 0x02D and 0x07B): alpha_hat_j =
// n_accepted_j / n_reached_j; a depth nobody reached takes the pooled rate over all depths, and
// with no depth reached at all the previous estimate. E[A](gamma) = sum_{j<=gamma} prod_{m<=j}
// alpha_hat_m replaces the constant-alpha sum in the objective (1 + E[A]) / (gamma*c + 1). One
// thread, float pairs (no float64 arithmetic on the device).
__device__ __forceinline__ F2 int_f2(int n) {
    const float hi = static_cast<float>(n);
    return f2_norm(hi, static_cast<float>(n - static_cast<int>(hi)));  // exact above 2^24 too
}

__global__ void spec_gamma_depth_kernel(const int32_t *n_reached, const int32_t *n_accepted, int depth_max,
                                        float prev_hi, float prev_lo, float c_hi, float c_lo, int gmin, int gmax,
                                        int32_t *gamma_out, double *ea_out) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    griddep_wait();
    long long sr = 0, sa = 0;
    for (int j = 0; j < depth_max; ++j) {
        sr += n_reached[j];
        sa += n_accepted[j];
    }
    const F2 pooled = sr > 0 ? f2_div(int_f2(static_cast<int>(sa)), int_f2(static_cast<int>(sr))) : F2{prev_hi, prev_lo};
    const F2 c = {c_hi, c_lo};
    F2 prod = {1.0f, 0.0f}, ea = {0.0f, 0.0f};
    int best = -1;
    F2 best_num = {0.0f, 0.0f}, best_den = {1.0f, 0.0f}, best_ea = {0.0f, 0.0f};
    for (int g = 0; g <= gmax; ++g) {
        if (g > 0) {
            const int j = g - 1;
            const int r = j < depth_max ? n_reached[j] : 0;
            const F2 ah = r > 0 ? f2_div(int_f2(n_accepted[j]), int_f2(r)) : pooled;
            prod = f2_mul(prod, ah);
            ea = f2_add(ea, prod);
        }
        if (g < gmin) continue;
        const F2 num = f2_add({1.0f, 0.0f}, ea);
        const F2 den = f2_add(f2_mul({static_cast<float>(g), 0.0f}, c), {1.0f, 0.0f});
        if (best < 0 || f2_gt(f2_mul(num, best_den), f2_mul(best_num, den))) {  // strict: a tie keeps the smaller
            best = g;
            best_num = num;
            best_den = den;
            best_ea = ea;
        }
    }
    *gamma_out = best;
    *ea_out = static_cast<double>(best_ea.hi) + static_cast<double>(best_ea.lo);
}
}  // namespace spec

using namespace spec;

extern "C" spec_status spec_compact(const spec_compact_args *a, cudaStream_t stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 1 || a->page_size < 1 || a->max_blocks < 1 || a->total_rows < a->B) return SPEC_ERR_INVALID_ARG;
    if (!a->row_off || !a->accept_len || !a->out_tokens || !a->prefix_len || !a->block_table || !a->out_off ||
        !a->packed_tokens || !a->packed_pos || !a->kv_off || !a->new_seq_len || !a->new_kv_len)
        return SPEC_ERR_INVALID_ARG;
    if (a->total_rows > a->B && (!a->cand_kv_rows || !a->kv_src || !a->kv_dst)) return SPEC_ERR_INVALID_ARG;
    CompactParams P;
    P.B = a->B;
    P.page_size = a->page_size;
    P.max_blocks = a->max_blocks;
    P.total_rows = a->total_rows;
    P.row_off = a->row_off;
    P.accept_len = a->accept_len;
    P.n_emitted = a->n_emitted;
    P.out_tokens = a->out_tokens;
    P.req_status = a->req_status;
    P.prefix_len = a->prefix_len;
    P.cand_kv_rows = a->cand_kv_rows;
    P.block_table = a->block_table;
    P.out_off = a->out_off;
    P.packed_tokens = a->packed_tokens;
    P.packed_pos = a->packed_pos;
    P.kv_off = a->kv_off;
    P.kv_src = a->kv_src;
    P.kv_dst = a->kv_dst;
    P.new_seq_len = a->new_seq_len;
    P.new_kv_len = a->new_kv_len;
    P.new_draft_len = a->new_draft_len;
    P.compact_status = a->compact_status;
    return launch_after(spec_compact_kernel, dim3(1), dim3(kCompactThreads), stream, P) == cudaSuccess ? SPEC_OK
                                                                                                     : SPEC_ERR_CUDA;
}

// Host evaluation in double precision (the closed form of SOTA-227).
extern "C" double spec_gamma_objective(double alpha, double c, int32_t gamma) {
    if (alpha == 1.0) return (gamma + 1.0) / (gamma * c + 1.0);
    double pw = alpha;  // alpha^(gamma+1)
    for (int k = 0; k < gamma; ++k) pw *= alpha;
    return (1.0 - pw) / ((1.0 - alpha) * (gamma * c + 1.0));
}

extern "C" spec_status spec_choose_gamma(const double *alpha_sum, const int32_t *alpha_count, double alpha_prev,
                                         double c, int32_t gamma_min, int32_t gamma_max, int32_t *gamma_out,
                                         double *alpha_out, cudaStream_t stream) {
    if (!alpha_sum || !alpha_count || !gamma_out || !alpha_out) return SPEC_ERR_INVALID_ARG;
    if (gamma_min < 0 || gamma_max < gamma_min || gamma_max > 4096) return SPEC_ERR_INVALID_ARG;
    if (!(c >= 0.0) || !std::isfinite(c) || !(alpha_prev >= 0.0 && alpha_prev <= 1.0)) return SPEC_ERR_INVALID_ARG;
    // host splits of the two double parameters into float pairs
    const float ph = static_cast<float>(alpha_prev), pl = static_cast<float>(alpha_prev - static_cast<double>(ph));
    const float ch = static_cast<float>(c), cl = static_cast<float>(c - static_cast<double>(ch));
    return launch_after(spec_gamma_kernel, dim3(1), dim3(32), stream, alpha_sum, alpha_count, ph, pl, ch, cl,
                        static_cast<int>(gamma_min), static_cast<int>(gamma_max), gamma_out, alpha_out) == cudaSuccess
               ? SPEC_OK
               : SPEC_ERR_CUDA;
}

// Host evaluation in double precision of the depth-aware objective (for tests and callers that
// choose on the host). Host pointers.
extern "C" double spec_depth_objective(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                                       double alpha_prev, double c, int32_t gamma) {
    double sr = 0.0, sa = 0.0;
    for (int j = 0; j < depth_max; ++j) {
        sr += n_reached[j];
        sa += n_accepted[j];
    }
    const double pooled = sr > 0.0 ? sa / sr : alpha_prev;
    double prod = 1.0, ea = 0.0;
    for (int j = 0; j < gamma; ++j) {
        const int r = j < depth_max ? n_reached[j] : 0;
        prod *= r > 0 ? static_cast<double>(n_accepted[j]) / r : pooled;
        ea += prod;
    }
    return (1.0 + ea) / (gamma * c + 1.0);
}

extern "C" spec_status spec_choose_gamma_depth(const int32_t *n_reached, const int32_t *n_accepted, int32_t depth_max,
                                               double alpha_prev, double c, int32_t gamma_min, int32_t gamma_max,
                                               int32_t *gamma_out, double *ea_out, cudaStream_t stream) {
    if (!gamma_out || !ea_out || depth_max < 0 || (depth_max > 0 && (!n_reached || !n_accepted)))
        return SPEC_ERR_INVALID_ARG;
    if (gamma_min < 0 || gamma_max < gamma_min || gamma_max > 4096) return SPEC_ERR_INVALID_ARG;
    if (!(c >= 0.0) || !std::isfinite(c) || !(alpha_prev >= 0.0 && alpha_prev <= 1.0)) return SPEC_ERR_INVALID_ARG;
    const float ph = static_cast<float>(alpha_prev), pl = static_cast<float>(alpha_prev - static_cast<double>(ph));
    const float ch = static_cast<float>(c), cl = static_cast<float>(c - static_cast<double>(ch));
    return launch_after(spec_gamma_depth_kernel, dim3(1), dim3(32), stream, n_reached, n_accepted,
                        static_cast<int>(depth_max), ph, pl, ch, cl, static_cast<int>(gamma_min),
                        static_cast<int>(gamma_max), gamma_out, ea_out) == cudaSuccess
               ? SPEC_OK
               : SPEC_ERR_CUDA;
}
