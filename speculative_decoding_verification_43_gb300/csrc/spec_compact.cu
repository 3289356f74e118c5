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
#include "spec_tail.cuh"

namespace spec {

__global__ void __launch_bounds__(kCompactThreads) spec_compact_kernel(const CompactParams P) {
    __shared__ CompactScratch<kCompactThreads> scratch;
    griddep_launch_dependents();
    compact_body<kCompactThreads>(P, true, -1, scratch);
}

__global__ void spec_gamma_kernel(const GammaParams G) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    griddep_wait();
    gamma_body(G);
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

namespace spec {

// The compaction's kernel parameters from its arguments; SPEC_ERR_INVALID_ARG when they are bad.
spec_status compact_params(const spec_compact_args *a, CompactParams &P) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 1 || a->page_size < 1 || a->max_blocks < 1 || a->total_rows < a->B) return SPEC_ERR_INVALID_ARG;
    if (!a->row_off || !a->accept_len || !a->out_tokens || !a->prefix_len || !a->block_table || !a->out_off ||
        !a->packed_tokens || !a->packed_pos || !a->kv_off || !a->new_seq_len || !a->new_kv_len)
        return SPEC_ERR_INVALID_ARG;
    if (a->total_rows > a->B && (!a->cand_kv_rows || !a->kv_src || !a->kv_dst)) return SPEC_ERR_INVALID_ARG;
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
    return SPEC_OK;
}

// The gamma choice's kernel parameters; SPEC_ERR_INVALID_ARG when they are bad. The two double
// parameters are split into float pairs on the host.
spec_status gamma_params(const double *alpha_sum, const int32_t *alpha_count, double alpha_prev, double c,
                         int32_t gamma_min, int32_t gamma_max, int32_t *gamma_out, double *alpha_out, GammaParams &G) {
    if (!alpha_sum || !alpha_count || !gamma_out || !alpha_out) return SPEC_ERR_INVALID_ARG;
    if (gamma_min < 0 || gamma_max < gamma_min || gamma_max > 4096) return SPEC_ERR_INVALID_ARG;
    if (!(c >= 0.0) || !std::isfinite(c) || !(alpha_prev >= 0.0 && alpha_prev <= 1.0)) return SPEC_ERR_INVALID_ARG;
    G.alpha_sum = alpha_sum;
    G.alpha_count = alpha_count;
    G.prev_hi = static_cast<float>(alpha_prev);
    G.prev_lo = static_cast<float>(alpha_prev - static_cast<double>(G.prev_hi));
    G.c_hi = static_cast<float>(c);
    G.c_lo = static_cast<float>(c - static_cast<double>(G.c_hi));
    G.gmin = gamma_min;
    G.gmax = gamma_max;
    G.gamma_out = gamma_out;
    G.alpha_out = alpha_out;
    return SPEC_OK;
}

}  // namespace spec

extern "C" spec_status spec_compact(const spec_compact_args *a, cudaStream_t stream) {
    CompactParams P;
    const spec_status st = compact_params(a, P);
    if (st != SPEC_OK) return st;
    return launch_after(spec_compact_kernel, dim3(1), dim3(kCompactThreads), 0, stream, P) == cudaSuccess ? SPEC_OK
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
    GammaParams G;
    const spec_status st = gamma_params(alpha_sum, alpha_count, alpha_prev, c, gamma_min, gamma_max, gamma_out,
                                        alpha_out, G);
    if (st != SPEC_OK) return st;
    return launch_after(spec_gamma_kernel, dim3(1), dim3(32), 0, stream, G) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
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
    return launch_after(spec_gamma_depth_kernel, dim3(1), dim3(32), 0, stream, n_reached, n_accepted,
                        static_cast<int>(depth_max), ph, pl, ch, cl, static_cast<int>(gamma_min),
                        static_cast<int>(gamma_max), gamma_out, ea_out) == cudaSuccess
               ? SPEC_OK
               : SPEC_ERR_CUDA;
}

#ifdef SPEC_DEBUG
namespace spec {
// The debug words of this translation unit's kernels (the compaction and the gamma choice).
cudaError_t debug_take_compact(unsigned int out[4]) { return spec_dbg_take(out); }
}  // namespace spec
#endif
