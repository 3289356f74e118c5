// The verifier's kernels, launched back to back on one stream (included once, by spec_verify.cu):
// spec_stats_kernel (pass 1 over every logit), spec_decide_kernel (every position's accept test and
// each request's frontier), spec_pass2_kernel (pass 2 over the pairs: alpha, and the frontier's
// residual), spec_finish_kernel (the frontier draws, the requests' selections, and in the CTA that
// completes the batch its sums and, for spec_verify_round, the compaction and the gamma choice).
//
// The rule is that of "SOTA-227: Decode with a draft model and an accept-reject rule" ("What to
// do", steps 3-4) and SDCP Rules 1 and 2 ("Acceptance Rules"): accept x_j when u_j <= p_j(x_j) /
// q_j(x_j); at the first rejection draw from max(p_j - q_j, 0) normalised; with every draft
// accepted draw from p_{K+1}; with T = 0 the greedy rule.
//
// Work. An item is one target row (position j of request i; a pair with draft row j when j < K_i,
// else the row of the bonus or plain draw). Every row is cut into chunks of kChunkVecs 16-byte
// vectors (2 KB).
//
// spec_stats_kernel streams every logit once from HBM: a persistent grid whose warps each take a
// contiguous run of (item, chunk) pieces, with no cooperation between warps. A warp loads its
// chunk of the target row (and of the draft row, for a pair) with 128-bit loads, four vectors a
// lane, and reduces it to the chunk's statistics: per row an integral reference exponent and the
// sum of 2^(y s - ref) (s = log2(e) / T), or under the greedy rule the max and its smallest index.
// The lane whose vector holds the draft token also records (y_t - y_d) s there. A pair's rows are
// loaded with an L2 evict-last hint: pass 2 reads them again.
//
// spec_decide_kernel has one CTA per request and a warp per position: the warp combines the item's
// chunk statistics (references by exact powers of two) and decides the accept test; the CTA then
// records the request's first rejection A and status bits, marks its frontier (position A: the
// first rejection or, with every draft accepted, the bonus row), writes a bad request's outputs
// and adds the request to the batch's counts.
//
// spec_pass2_kernel walks the pairs' chunks again like the statistics kernel (contiguous runs per
// warp, from L2 where the rows stayed there): per chunk alpha = sum min(p, q) and, at the frontier,
// the residual mass sum max(p - q, 0). Rejections after the first need no residual: nothing after
// the first rejection is emitted.
//
// spec_finish_kernel has one warp per item: it sums the item's chunk shares, writes the item's
// per-draft outputs and adds its alpha to the batch's fixed-point sum; the frontier's warp draws
// the token (the chunk that holds u*Z by a scan over the chunk masses, then the token within it)
// and writes the request's outputs (accepted drafts, frontier token, stopping); the CTA holding
// the batch's last item runs the batch's tail.
//
// Each kernel after the first is launched with programmatic stream serialisation: its CTAs may
// start while the one before drains, and wait for it (griddepcontrol.wait) before reading anything
// it wrote. The statistics kernel zeroes the later kernels' counters, so a workspace needs no
// preparation between calls, whatever their shapes.
//
// The residual max(p - q, 0) is formed without cancellation: p (1 - 2^d) with d = log2(q/p) from
// the exact difference of the two logits, and 1 - 2^d from a series near d = 0, so that every
// residual weight is accurate to a few units in the last place of float32 however close q is to p.
#pragma once

#include <climits>
#include <cmath>
#include <cstdint>

#include "spec_device.cuh"
#include "spec_math.cuh"
#include "spec_tail.cuh"
#include "spec_verify.h"

namespace spec {
namespace vk {

constexpr int kVPT = 4;                          // 16-byte vectors of a chunk per lane and row
constexpr int kChunkVecs = kWarp * kVPT;         // 128 vectors: a chunk (2 KB)
constexpr int kStatsBlock = 256;                 // statistics kernel: threads per CTA
constexpr int kFinBlock = 256;                   // pass-2 and finishing kernels: threads per CTA
constexpr int kFinWarps = kFinBlock / kWarp;
constexpr int kDecWarps = 8;                     // decision kernel: warps per CTA (one request)
constexpr int kDrawRun = 16;                     // a draw's chunk masses per lane held at once

enum : int32_t { XF_QZERO = 1, XF_PZERO = 2 };   // draft token's flags: q(x) = 0, p(x) = 0
enum : int32_t { I_PAIR = 1, I_ROW = 2, I_SKIP = 3 };
enum : int32_t { SAMPLE_NONE = 0, SAMPLE_RESIDUAL = 1, SAMPLE_P = 2 };
enum : int32_t { REQ_TIMEOUT = SPEC_REQ_TIMEOUT };
enum : int { CTL_DONE = 0, CTL_BAD_OFFSETS = 1, kCtlWords = 4 };
// the batch's sums, accumulated by the requests' selections (zeroed by the statistics kernel): alpha
// in fixed point (an integer sum, the same in any order), the rows it counts, the depth counts
enum : int { AGG_ALPHA = 0, AGG_COUNT = 2, AGG_REACHED = 4, AGG_ACCEPTED = AGG_REACHED + 64, kAggWords = AGG_ACCEPTED + 64 };
constexpr double kAlphaFix = 1099511627776.0;  // 2^40: alpha's fixed-point unit is 2^-40
constexpr int32_t kNoRef = -(1 << 30);  // reference exponent of a row (or part) with no mass

constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963e-08f;

// An item as both kernels see it (computed from the inputs alone).
struct ItemDesc {
    int32_t kind;            // I_*
    int32_t item, req, pos, K, drow;
    int32_t greedy, trunc, status;
    int32_t x;               // a pair's draft token (-1: none)
    int32_t xchunk;          // the chunk holding x's vector (-1: x outside [0, V))
    float s_hi, s_lo;        // log2(e)/T as a float pair, s_hi rounded toward zero (s_lo > 0)
    uint32_t cut_tau;        // top-k / top-p cut of the target row (trunc = 0: none)
    int32_t cut_id;
    double ua, us;           // the position's accept draw and the request's frontier draw
};

// The decision of an item.
struct ItemDec {
    int32_t status, accept, kind, argmax_t;
    int32_t frontier;            // the request's frontier: its first rejection, or the bonus row
    float B_t, S_t;              // target: integral reference exponent and the sum at it
    float c_t, c_tf, c_d, c_df;  // log2 of each normaliser: integral part, fraction
    F2 dc;                       // c_d - c_t as a float pair
    float rho, alpha_g;
    F2 u_s;
};

struct VerifyParams {
    const void *target;
    const void *draft;
    const int32_t *row_off;
    const int32_t *draft_tokens;
    const double *uniforms;
    const float *temperature;
    float temperature_scalar;
    const float *top_p;      // read only for its NaN check (the cut is in trunc)
    const int2 *trunc;       // [T] cut of each target row, or NULL
    const int32_t *stop_token;
    const int32_t *max_new;
    int32_t B, V, K_max, total_rows;
    int32_t nvec_row;        // 16-byte vectors per row
    int32_t nchunk;          // chunks per row
    // workspace
    int4 *rec;               // [T][nchunk] each chunk's statistics (ref_t, sum_t, ref_d, sum_d)
    float4 *xrec;            // [T] the draft token's (E_hi, E_lo, flags, -)
    ItemDesc *desc;          // [T] each item's values, from the statistics kernel
    ItemDec *dec;            // [T] each item's decision, from the decision kernel
    float *alpha_c;          // [T][nchunk] each chunk's alpha share (a pair under Rule 2)
    float *zc;               // [T][nchunk] each chunk's residual mass (a frontier rejection)
    int32_t *req_first;      // [B] the request's first rejected position (K: none)
    int32_t *req_st;         // [B] the request's status bits
    uint32_t *ctl;           // [kCtlWords] items finalised; row offsets invalid
    uint32_t *agg;           // [kAggWords] the batch's sums
    // outputs
    int32_t *accept_len, *n_emitted, *out_tokens, *req_status, *fallback, *alpha_count;
    int32_t *depth_reached, *depth_accepted;
    float *alpha_rows, *rho_rows, *resid_rows, *frontier_prob, *frontier_margin;
    double *alpha_sum;
    // spec_verify_round: the compaction and the gamma choice after the selection
    int32_t round;
    CompactParams C;
    GammaParams G;
};

// ------------------------------------------------------------------------------------------------
// small helpers

__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// 2^d for an integer d <= 0 with integer operations only (0 below the normal range).
__device__ __forceinline__ float pow2_int(int d) { return d < -126 ? 0.0f : __int_as_float((d + 127) << 23); }

// The kernel's parameters copied into shared memory by the whole CTA (one word a thread, all at
// once): the functions that read many fields once (decisions, draws, selections, the batch's tail)
// then read them at shared-memory latency instead of missing the constant cache field by field.
template <int NT>
__device__ __forceinline__ void stage_params(const VerifyParams &src, VerifyParams &dst) {
    static_assert(sizeof(VerifyParams) % 4 == 0, "copied as words");
    constexpr int kWords = static_cast<int>(sizeof(VerifyParams) / 4);
    const uint32_t *s = reinterpret_cast<const uint32_t *>(&src);
    uint32_t *d = reinterpret_cast<uint32_t *>(&dst);
    for (int i = threadIdx.x; i < kWords; i += NT) d[i] = s[i];
    __syncthreads();
}

// Release/acquire fence at GPU scope: orders this thread's earlier memory operations before its
// later ones as seen by the other CTAs (the pattern of the last-arriver counters: write, fence,
// count; count, fence, read). Lighter than a sequentially consistent fence.
__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// A 16-byte load through L2 with an eviction hint, not kept in L1.
__device__ __forceinline__ uint4 ldg_hint(const uint4 *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

template <int DT>
__device__ __forceinline__ float vec_elem(const uint4 &w, int e) {
    float2 y[Elt<DT>::kPerVec / 2];
    Elt<DT>::unpack2(w, y);
    float r = 0.0f;
#pragma unroll
    for (int h = 0; h < Elt<DT>::kPerVec / 2; ++h) {
        if (e == 2 * h) r = y[h].x;
        if (e == 2 * h + 1) r = y[h].y;
    }
    return r;
}

// Top-k / top-p: the logits of vector `vi` of a target row outside the row's cut become -inf,
// which turns every later sum, ratio and draw into those of the truncated, renormalised law.
template <int DT>
__device__ __forceinline__ bool mask_cut(uint4 &w, int vi, uint32_t tau, int id) {
    // a vector wholly below the cut's logit (the common case after top-k) becomes -inf at once;
    // the largest element is taken with NaN propagating, so a NaN always takes the exact test
    // below and stays (it makes the row invalid)
    float vm, ct;
    if (DT == SPEC_BF16) {
        const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(w.x, w.y), bf16x2_max_nan(w.z, w.w));
        vm = fmax_nan(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
        const uint32_t b = (tau & 0x8000u) ? (tau & 0x7FFFu) : (~tau & 0xFFFFu);
        ct = __uint_as_float(b << 16);
    } else {
        vm = fmax_nan(fmax_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                      fmax_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
        ct = __uint_as_float((tau & 0x80000000u) ? (tau & 0x7FFFFFFFu) : ~tau);
    }
    if (vm < ct) {
        w = kNegInfVec<DT>();
        return true;
    }
    uint32_t x[4] = {w.x, w.y, w.z, w.w};
    if (DT == SPEC_BF16) {
        const int base = vi * 8;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const uint32_t lo = x[h] & 0xFFFFu, hi = x[h] >> 16;
            const uint32_t nlo = cut_keeps(key_bf16(lo), base + 2 * h, tau, id) ? lo : 0xFF80u;
            const uint32_t nhi = cut_keeps(key_bf16(hi), base + 2 * h + 1, tau, id) ? hi : 0xFF80u;
            x[h] = nlo | (nhi << 16);
        }
    } else {
        const int base = vi * 4;
#pragma unroll
        for (int h = 0; h < 4; ++h)
            if (!cut_keeps(key_f32(x[h]), base + h, tau, id)) x[h] = 0xFF800000u;
    }
    w = make_uint4(x[0], x[1], x[2], x[3]);
    return false;
}

// 2^d - 1 for d in [-1/4, 0] (and a little beyond) by its series in d: the coefficients are
// (ln 2)^k / k!, k = 1..7; the first term omitted is below 1e-9 relative. Accurate where
// 2^d - 1 computed as ex2(d) - 1 would cancel.
__device__ __forceinline__ float2 exp2m1_series(float2 d) {
    constexpr float c1 = 0.693147180559945309f, c2 = 0.240226506959100712f, c3 = 0.0555041086648215800f,
                    c4 = 0.00961812910762847717f, c5 = 0.00133335581464284434f, c6 = 0.000154035303933816100f,
                    c7 = 0.0000152527338040598403f;
    float2 p = __ffma2_rn(d, f2splat(c7), f2splat(c6));
    p = __ffma2_rn(d, p, f2splat(c5));
    p = __ffma2_rn(d, p, f2splat(c4));
    p = __ffma2_rn(d, p, f2splat(c3));
    p = __ffma2_rn(d, p, f2splat(c2));
    p = __ffma2_rn(d, p, f2splat(c1));
    return __fmul2_rn(d, p);
}

// The fraction term of -log2 of a row's normaliser, c_f, less y_top s_lo: in log2 p = y s_hi - c -
// c_f + y s_lo the term y s_lo is taken as y_top s_lo, one constant per row with y_top = (c + c_f)
// / s_hi (the log-normaliser over s, within log2(V) / s of the row's largest logit). It differs
// from y s_lo by (y - y_top) s_lo: at most about log2(V) 2^-24 relative on the terms that carry a
// sum, where dropping it would cost y s_lo (3e-5 at T = 0.01). Pass 2 and the residual draw use it
// alike, so a draw's weights are those pass 2 summed.
__device__ __forceinline__ float neg_frac_lo(float c, float cf, float s_hi, float s_lo) {
    return -cf + (c + cf) * (s_lo / s_hi);
}

// The residual weights max(p - q, 0) and min(p, q) of one pair of logits pairs, normalised: p =
// 2^(y_t s - c_t) and q / p = 2^d with d = (y_d - y_t) s - (c_d - c_t), the logit difference
// exact and its product with s a float pair, so that d is accurate even where p and q nearly
// agree; 1 - 2^d by the series near 0. A -inf logit gives weight 0 (fmin / fmax drop the NaNs of
// 0 * inf).
__device__ __forceinline__ void resid_weights(float2 yt, float2 yd, float2 shi2, float2 slo2, float2 nct,
                                              float2 nctf, float2 ndch, float2 ndcl, float2 &r, float2 &m) {
    const float2 at = __fadd2_rn(__ffma2_rn(yt, shi2, nct), nctf);  // log2 p
    const float2 diff = __fadd2_rn(yd, make_float2(-yt.x, -yt.y));
    const float2 d = __fadd2_rn(__ffma2_rn(diff, slo2, __ffma2_rn(diff, shi2, ndch)), ndcl);  // log2 (q / p)
    const float2 p = ex2x2(at);
    const float2 e = ex2x2(d);
    const float2 s = exp2m1_series(d);
    // 2^d - 1 (<= 0 where q <= p)
    const float em_x = (d.x > -0.25f) ? s.x : e.x - 1.0f;
    const float em_y = (d.y > -0.25f) ? s.y : e.y - 1.0f;
    const float2 rr = __fmul2_rn(p, make_float2(-em_x, -em_y));
    r = make_float2(fmaxf(rr.x, 0.0f), fmaxf(rr.y, 0.0f));
    m = __fmul2_rn(p, make_float2(fminf(1.0f, e.x), fminf(1.0f, e.y)));
}

// ------------------------------------------------------------------------------------------------
// data warps: pass 1

// Sum of 2^(y s - b) over one vector (pairs of lanes packed).
template <int DT>
__device__ __forceinline__ float vec_sum(const uint4 &w, float2 shi2, float2 slo2, float b) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    const float2 nb2 = f2splat(-b);
    float2 e[H];
#pragma unroll
    for (int h = 0; h < H; ++h) e[h] = ex2x2(exp_arg2(Elt<DT>::unpack_one(w, h), shi2, slo2, nb2));
#pragma unroll
    for (int st = 1; st < H; st <<= 1)
#pragma unroll
        for (int h = 0; h + st < H; h += 2 * st) e[h] = __fadd2_rn(e[h], e[h + st]);
    return e[0].x + e[0].y;
}

// Greedy rule, one thread's vectors of one row: the largest logit and the smallest index that
// attains it; a NaN or +inf makes the row invalid (max +inf, index -1).
template <int DT>
__device__ __forceinline__ void row_argmax(const uint4 (&v)[kVPT], int vbase, float &best, int &bidx) {
    constexpr int E = Elt<DT>::kPerVec;
    constexpr int H = E / 2;
    best = -INFINITY;
    bidx = INT_MAX;
    int bad = 0;
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float2 y = Elt<DT>::unpack_one(v[k], h);
            bad |= (y.x != y.x) || (y.x == INFINITY) || (y.y != y.y) || (y.y == INFINITY);
        }
        const float mv = Elt<DT>::vmax(v[k]);
        if (mv > best) {
            best = mv;
            for (int e = E - 1; e >= 0; --e)
                if (vec_elem<DT>(v[k], e) == mv) bidx = (vbase + k * kWarp) * E + e;
        }
    }
    if (bad) {
        best = INFINITY;
        bidx = -1;
    }
}

// Rule 2, one row, one (reference, sum) per lane over `width` lanes: the largest reference among
// lanes with mass and the sum scaled to it by exact powers of two. A sum that is NaN, +inf or
// negative in any lane (of the whole warp) makes the result's sum NaN; no mass gives (-inf, 0).
template <int W>
__device__ __forceinline__ float2 ref_sum(float b, float s) {
    const bool ok = s > 0.0f && !isinf(s);
    const int bad = __any_sync(0xffffffffu, !(s >= 0.0f) || isinf(s));
    float B = ok ? b : -INFINITY;
#pragma unroll
    for (int o = 1; o < W; o <<= 1) B = fmaxf(B, __shfl_xor_sync(0xffffffffu, B, o));
    float S = ok ? s * pow2i(b - B) : 0.0f;
#pragma unroll
    for (int o = 1; o < W; o <<= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    return make_float2(B, bad ? NAN : S);
}

// Greedy rule: the largest value and the smallest index attaining it over `width` lanes; an
// invalid part (+inf, index -1) wins every comparison.
template <int W>
__device__ __forceinline__ void arg_max(float &m, int &ix) {
#pragma unroll
    for (int o = 1; o < W; o <<= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const int oi = __shfl_xor_sync(0xffffffffu, ix, o);
        if (om > m || (om == m && oi < ix)) {
            m = om;
            ix = oi;
        }
    }
}

// ------------------------------------------------------------------------------------------------
// items

// Request of target row g: the i with row_off[i] <= g < row_off[i + 1]. Offsets that fail their
// checks still give some i in [0, B) (the call then reports every request BAD_SHAPE).
__device__ __forceinline__ int find_request(const VerifyParams &P, int g, int &r0, int &r1) {
    int lo = 0, hi = P.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(P.row_off + mid) <= g) lo = mid; else hi = mid - 1;
    }
    r0 = __ldg(P.row_off + lo);
    r1 = __ldg(P.row_off + lo + 1);
    return lo;
}

// Item g's values from the inputs (the same in every thread and kernel that computes them). An item
// whose request has a bad shape or bad parameters is I_SKIP: nothing of it is read.
template <int DT>
__device__ __forceinline__ ItemDesc item_desc(const VerifyParams &P, int g) {
    constexpr int E = Elt<DT>::kPerVec;
    int r0, r1;
    const int i = find_request(P, g, r0, r1);
    const int K = r1 - r0 - 1, pos = g - r0;
    const int drow = r0 - i + pos;
    // every index stays in range whatever the offsets hold
    const bool shaped = K >= 0 && K <= P.K_max && pos >= 0 && pos <= K && drow >= 0 &&
                        (pos == K || drow < P.total_rows - P.B) && r0 + K < P.total_rows;
    const float T = P.temperature ? __ldg(P.temperature + i) : P.temperature_scalar;
    const float tp = P.top_p ? __ldg(P.top_p + i) : 1.0f;
    const double ua = (shaped && pos < K) ? __ldg(P.uniforms + g) : 0.0;
    const double us = shaped ? __ldg(P.uniforms + r0 + K) : 0.0;
    const int x = (shaped && pos < K) ? __ldg(P.draft_tokens + drow) : -1;
    const int2 cut = (P.trunc && shaped) ? __ldg(P.trunc + g) : make_int2(0, INT_MAX);
    ItemDesc d = {};
    int status = shaped ? 0 : SPEC_REQ_BAD_SHAPE;
    if (!(T >= 0.0f) || isinf(T) || isnan(tp)) status |= SPEC_REQ_BAD_PARAM;
    d.kind = status ? I_SKIP : (pos < K ? I_PAIR : I_ROW);
    d.item = g;
    d.req = i;
    d.pos = pos;
    d.K = K;
    d.drow = drow;
    d.status = status;
    d.greedy = (T == 0.0f) ? 1 : 0;
    d.ua = ua;
    d.us = us;
    d.x = x;
    d.xchunk = (x >= 0 && x < P.V) ? (x / E) / kChunkVecs : -1;
    F2 sv = {0.0f, 0.0f};
    if (T > 0.0f && !isinf(T)) sv = f2_div({kLog2eHi, kLog2eLo}, {T, 0.0f});
    if (sv.hi > 0.0f && sv.lo < 0.0f) {
        // s_hi moved toward zero so that s_lo > 0: a -inf logit then gives -inf in both terms of
        // the exponent's argument (a negative s_lo would make it NaN)
        const float down = __uint_as_float(__float_as_uint(sv.hi) - 1u);
        sv.lo += sv.hi - down;
        sv.hi = down;
    }
    d.s_hi = sv.hi;
    d.s_lo = fmaxf(sv.lo, 1.401298464e-45f);
    d.cut_tau = static_cast<uint32_t>(cut.x);
    d.cut_id = cut.y;
    d.trunc = (!d.greedy && (cut.x != 0 || cut.y != INT_MAX)) ? 1 : 0;
    return d;
}

// Whether item d has pass 2: a pair under Rule 2 (alpha and the residual need both normalisers).
__device__ __forceinline__ bool has_p2(const ItemDesc &d) { return d.kind == I_PAIR && !d.greedy; }

// ------------------------------------------------------------------------------------------------
// spec_stats_kernel: each chunk's statistics

// A lane's sum of 2^(y s - b) over its vectors of one row in the exact form, for a warp in which a
// lane's fast sum overflowed (above 2^64: a later vector much larger than the first, an all -inf
// first vector, a NaN or +inf): b from the lane's max over all its vectors (0 for an all -inf
// lane, whose sum is then 0). Rare: out of line.
template <int DT>
__device__ __noinline__ float2 row_sum_exact(uint4 v0, uint4 v1, uint4 v2, uint4 v3, float s_hi, float s_lo) {
    static_assert(kVPT == 4, "the exact form takes a lane's four vectors");
    const float2 shi2 = f2splat(s_hi), slo2 = f2splat(s_lo);
    const float m = fmaxf(fmaxf(Elt<DT>::vmax(v0), Elt<DT>::vmax(v1)), fmaxf(Elt<DT>::vmax(v2), Elt<DT>::vmax(v3)));
    const float b = (m == -INFINITY) ? 0.0f : floorf(m * s_hi);
    const float s = vec_sum<DT>(v0, shi2, slo2, b) + vec_sum<DT>(v1, shi2, slo2, b) + vec_sum<DT>(v2, shi2, slo2, b) +
                    vec_sum<DT>(v3, shi2, slo2, b);
    return make_float2(b, s);
}

// A lane's (b, sum) of one row's vectors, b an integral reference from its first vector (so that no
// exponential waits on a running max); the warp takes the exact form where a sum overflowed.
template <int DT>
__device__ __forceinline__ float2 row_sum(const uint4 (&v)[kVPT], float s_hi, float s_lo) {
    const float2 shi2 = f2splat(s_hi), slo2 = f2splat(s_lo);
    // an all -inf first vector (masked vocabulary, a truncated row) takes 0 as its reference,
    // which keeps its -inf terms at 0 instead of sending the warp to the exact form
    const float m0 = Elt<DT>::vmax(v[0]);
    const float b = (m0 == -INFINITY) ? 0.0f : floorf(m0 * s_hi);
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kVPT; ++k) s += vec_sum<DT>(v[k], shi2, slo2, b);
    if (__any_sync(0xffffffffu, !(s <= 0x1p64f))) return row_sum_exact<DT>(v[0], v[1], v[2], v[3], s_hi, s_lo);
    return make_float2(b, s);
}

// The chunk's record from the warp's reduced values (every lane holds them): per row the reference
// (kNoRef: no mass) and the sum (NaN: invalid logits; a reference beyond 2^28 reads as invalid),
// or under the greedy rule (argmax, max) per row.
__device__ __forceinline__ int4 chunk_record(float4 w, bool greedy, bool pair) {
    if (greedy)
        return make_int4(__float_as_int(w.y), __float_as_int(w.x), __float_as_int(w.w), __float_as_int(w.z));
    const bool inval_t = isnan(w.y) || (w.y > 0.0f && !(fabsf(w.x) < 0x1p28f));
    const bool inval_d = isnan(w.w) || (w.w > 0.0f && !(fabsf(w.z) < 0x1p28f));
    return make_int4((w.y > 0.0f && !inval_t) ? static_cast<int>(w.x) : kNoRef, __float_as_int(inval_t ? NAN : w.y),
                     (pair && w.w > 0.0f && !inval_d) ? static_cast<int>(w.z) : kNoRef,
                     __float_as_int(pair ? (inval_d ? NAN : w.w) : 0.0f));
}

// Chunk c of item d (whole warp): lane l takes vectors c*128 + 32k + l, k < 4, of the target row
// and, for a pair, of the draft row (stats_load); the warp's statistics go to the chunk's record.
// The lane whose vector holds the draft token records (y_t - y_d) s there and the flags of a -inf
// logit.
template <int DT>
__device__ __forceinline__ void stats_load(const VerifyParams &P, const ItemDesc &d, int c, uint64_t keep, uint64_t drop,
                                           uint4 (&vt)[kVPT], uint4 (&vd)[kVPT]) {
    const int lane = threadIdx.x % kWarp;
    const bool pair = d.kind == I_PAIR;
    const uint4 *trow = static_cast<const uint4 *>(P.target) + static_cast<size_t>(d.item) * P.nvec_row;
    const uint4 *drow = static_cast<const uint4 *>(P.draft) + static_cast<size_t>(d.drow) * P.nvec_row;
    const uint64_t pol = has_p2(d) ? keep : drop;  // a pair's rows are read again by pass 2
    const bool rows_ok = SPEC_IN(d.item, P.total_rows, DBG_LOGITS) &&
                         (!pair || SPEC_IN(d.drow, P.total_rows - P.B, DBG_LOGITS));
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
        const int vi = c * kChunkVecs + k * kWarp + lane;
        const bool in = rows_ok && vi < P.nvec_row;
        vt[k] = in ? ldg_hint(trow + vi, pol) : kNegInfVec<DT>();
        vd[k] = (in && pair) ? ldg_hint(drow + vi, pol) : kNegInfVec<DT>();
    }
}
template <int DT>
__device__ __forceinline__ void chunk_stats(const VerifyParams &P, const ItemDesc &d, int c, uint4 (&vt)[kVPT],
                                            const uint4 (&vd)[kVPT]) {
    constexpr int E = Elt<DT>::kPerVec;
    const int lane = threadIdx.x % kWarp;
    const bool pair = d.kind == I_PAIR, greedy = d.greedy != 0;
    const int vbase = c * kChunkVecs + lane;
    bool t_empty = false;  // the target row's chunk lies wholly outside its top-k / top-p cut
    if (d.trunc) {
        bool all = true;
#pragma unroll
        for (int k = 0; k < kVPT; ++k) all &= mask_cut<DT>(vt[k], vbase + k * kWarp, d.cut_tau, d.cut_id);
        t_empty = __all_sync(0xffffffffu, all);
    }
    if (pair && !greedy && d.xchunk == c) {
        // x = E * (c*128 + 32k + l) + e for one lane l and one k
        const int xv = d.x / E - c * kChunkVecs;
        if (xv % kWarp == lane) {
            const int k = xv / kWarp;
            uint4 wt = vt[0], wd = vd[0];
#pragma unroll
            for (int q = 1; q < kVPT; ++q)
                if (q == k) {
                    wt = vt[q];
                    wd = vd[q];
                }
            const float yt = vec_elem<DT>(wt, d.x % E), yd = vec_elem<DT>(wd, d.x % E);
            const F2 Ex = f2_mul(f2_add({yt, 0.0f}, {-yd, 0.0f}), {d.s_hi, d.s_lo});
            const int flags = (yd == -INFINITY ? XF_QZERO : 0) | (yt == -INFINITY ? XF_PZERO : 0);
            if (SPEC_IN(d.item, P.total_rows, DBG_ROWS))
                P.xrec[d.item] = make_float4(Ex.hi, Ex.lo, __int_as_float(flags), 0.0f);
        }
    }
    float4 w;
    if (greedy) {
        float bt, bd = -INFINITY;
        int it, id = INT_MAX;
        row_argmax<DT>(vt, vbase, bt, it);
        if (pair) row_argmax<DT>(vd, vbase, bd, id);
        arg_max<kWarp>(bt, it);
        arg_max<kWarp>(bd, id);
        w = make_float4(bt, __int_as_float(it), bd, __int_as_float(id));
    } else {
        // a chunk with no target mass adds nothing to the target's sum: its exponentials are skipped
        const float2 t = t_empty ? make_float2(0.0f, 0.0f) : row_sum<DT>(vt, d.s_hi, d.s_lo);
        const float2 q = pair ? row_sum<DT>(vd, d.s_hi, d.s_lo) : make_float2(0.0f, 0.0f);
        const float2 rt = ref_sum<kWarp>(t.x, t.y);
        const float2 rd = pair ? ref_sum<kWarp>(q.x, q.y) : make_float2(-INFINITY, 0.0f);
        w = make_float4(rt.x, rt.y, rd.x, rd.y);
    }
    if (lane == 0 && SPEC_IN(static_cast<long long>(d.item) * P.nchunk + c, static_cast<long long>(P.total_rows) * P.nchunk,
                             DBG_RECORDS))
        P.rec[static_cast<size_t>(d.item) * P.nchunk + c] = chunk_record(w, greedy, pair);
}

// Pass 1: every chunk of every item, each warp a contiguous run of (item, chunk) pieces. The
// kernel also zeroes the later kernels' counters, and CTA 0 checks the row offsets (start at 0,
// end at total_rows, grow by at least one row).
template <int DT>
__global__ void __launch_bounds__(kStatsBlock) spec_stats_kernel(const __grid_constant__ VerifyParams P) {
    const int tid = threadIdx.x;
    const int nthreads = gridDim.x * kStatsBlock;
    for (int i = blockIdx.x * kStatsBlock + tid; i < kAggWords; i += nthreads) P.agg[i] = 0u;
    if (blockIdx.x == 0) {
        int bad = 0;
        for (int i = tid; i <= P.B; i += kStatsBlock) {
            const int v = __ldg(P.row_off + i);
            if (i == 0 && v != 0) bad = 1;
            if (i == P.B && v != P.total_rows) bad = 1;
            if (i < P.B && __ldg(P.row_off + i + 1) <= v) bad = 1;
        }
        bad = __syncthreads_or(bad);
        if (tid == 0) {
            P.ctl[CTL_DONE] = 0u;
            P.ctl[CTL_BAD_OFFSETS] = bad ? 1u : 0u;
        }
    }
    // the decision kernel may start its CTAs now; they wait for this grid before reading its output
    griddep_launch_dependents();
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    const long long warps = static_cast<long long>(gridDim.x) * (kStatsBlock / kWarp);
    const long long gw = static_cast<long long>(blockIdx.x) * (kStatsBlock / kWarp) + tid / kWarp;
    const long long total = static_cast<long long>(P.total_rows) * P.nchunk;
    const long long per = (total + warps - 1) / warps;
    const long long u1 = min(total, (gw + 1) * per);
    int cur = -1;
    ItemDesc d = {};
    const long long ub = gw * per;
    if (ub >= u1) return;
    // (item, chunk) stepped without divisions
    int item = static_cast<int>(ub / P.nchunk), c = static_cast<int>(ub % P.nchunk) - 1;
    for (long long u = ub; u < u1; ++u) {
        if (++c == P.nchunk) {
            c = 0;
            ++item;
        }
        if (item != cur) {
            d = item_desc<DT>(P, item);
            cur = item;
        }
        if (c == 0 && tid % kWarp == 0 && SPEC_IN(item, P.total_rows, DBG_ROWS))
            P.desc[item] = d;  // the item's values, for the later kernels
        if (d.kind == I_SKIP) continue;
        uint4 vt[kVPT], vd[kVPT];
        stats_load<DT>(P, d, c, keep, drop, vt, vd);
        chunk_stats<DT>(P, d, c, vt, vd);
    }
}

// The decision of item d from its combined statistics (every lane computes it; the same inputs
// give the same result in every CTA). Rule 2: (a0, s0) / (a1, s1)
// reference and sum of the target / draft row over the vocabulary; Ex = (y_t - y_d) s at the draft
// token and its flags. Greedy: (a0, s0) / (a1, s1) are (argmax, max) of each row.
__device__ __forceinline__ ItemDec decide_item(const VerifyParams &P, const ItemDesc &d, int status, int a0, float s0,
                                               int a1, float s1, F2 Ex, int xflags) {
    const bool pair = d.kind == I_PAIR;
    const int x = d.x;
    ItemDec D = {};
    D.kind = SAMPLE_NONE;
    D.argmax_t = -1;
    D.u_s = d2f2(d.us);
    if (d.greedy) {
        const int am0 = (a0 >= 0 && a0 != INT_MAX && s0 != -INFINITY) ? a0 : -1;
        const int am1 = (a1 >= 0 && a1 != INT_MAX && s1 != -INFINITY) ? a1 : -1;
        if (!(status & (SPEC_REQ_BAD_SHAPE | SPEC_REQ_BAD_PARAM | REQ_TIMEOUT))) {
            if (am0 < 0 || (pair && am1 < 0)) status |= SPEC_REQ_BAD_LOGITS;
            if (pair && (x < 0 || x >= P.V)) status |= SPEC_REQ_BAD_PROPOSAL;
        }
        D.status = status;
        if (status == 0) {
            D.argmax_t = am0;
            if (pair) {
                D.accept = (x == am0);
                D.rho = D.accept ? 1.0f : 0.0f;
                D.alpha_g = (am0 == am1) ? 1.0f : 0.0f;
            }
        }
        return D;
    }
    const float B_t = (a0 != kNoRef && !isnan(s0)) ? static_cast<float>(a0) : NAN;
    const float B_d = (pair && a1 != kNoRef && !isnan(s1)) ? static_cast<float>(a1) : NAN;
    const float S_t = s0, S_d = pair ? s1 : 0.0f;
    if (!(status & (SPEC_REQ_BAD_SHAPE | SPEC_REQ_BAD_PARAM | REQ_TIMEOUT))) {
        const bool ok_t = isfinite(B_t) && S_t > 0.0f && isfinite(S_t);
        const bool ok_d = !pair || (isfinite(B_d) && S_d > 0.0f && isfinite(S_d));
        if (!ok_t || !ok_d) status |= SPEC_REQ_BAD_LOGITS;
        // q(x) == 0 is a bad proposal for Rule 2 (checked before any draw)
        if (pair && (x < 0 || x >= P.V || (xflags & XF_QZERO))) status |= SPEC_REQ_BAD_PROPOSAL;
    }
    D.status = status;
    D.B_t = B_t;
    D.S_t = S_t;
    const float2 ct = log2_split({S_t, 0.0f}, B_t), cd = log2_split({S_d, 0.0f}, B_d);
    D.c_t = ct.x;
    D.c_tf = ct.y;
    D.c_d = cd.x;
    D.c_df = cd.y;
    D.dc = f2_add({cd.x - ct.x, 0.0f}, {cd.y - ct.y, 0.0f});  // the integral parts differ exactly
    if (status == 0) {
        if (pair) {
            // rho = p(x)/q(x) = 2^E S_d / S_t with E = (y_t - y_d) s - (B_t - B_d), in float pairs;
            // 2^E from ex2 of its fraction and an exact power of two
            float rho = 0.0f;
            if (!(xflags & XF_PZERO)) {
                const F2 E = f2_add(Ex, {-(B_t - B_d), 0.0f});
                const float nn = floorf(E.hi);
                const float f = (E.hi - nn) + E.lo;
                const F2 ratio = f2_div({S_d, 0.0f}, {S_t, 0.0f});
                const float mm = ex2(f) * (ratio.hi + ratio.lo);
                if (nn > 254.0f) {
                    rho = INFINITY;
                } else if (nn >= -252.0f) {
                    const float h = floorf(0.5f * nn);
                    rho = mm * pow2i(h) * pow2i(nn - h);
                }
            }
            D.rho = rho;
            D.accept = (rho > 0.0f) && !f2_gt(d2f2(d.ua), {rho, 0.0f});
            if (!D.accept) D.kind = SAMPLE_RESIDUAL;
        } else {
            D.kind = SAMPLE_P;
        }
    }
    return D;
}


// ------------------------------------------------------------------------------------------------
// spec_finish_kernel: decisions, pass 2, draws, selections, the batch's tail

// The decision of item d (whole warp) from its chunks' records and the draft token's words. Lane l
// combines chunks l, l + 32, ...; the parts combine by exact powers of two (argmax pairs under the
// greedy rule).
__device__ __noinline__ ItemDec decide_chunks(const VerifyParams &P, const ItemDesc &d) {
    const int lane = threadIdx.x % kWarp;
    const bool greedy = d.greedy != 0;
    const int4 *rec = P.rec + static_cast<size_t>(d.item) * P.nchunk;
    int la0 = greedy ? INT_MAX : kNoRef, la1 = la0;
    float ls0 = greedy ? -INFINITY : 0.0f, ls1 = ls0;
    // rounds of up to kRound records per lane, every load of a round in flight at once
    constexpr int kRound = 8;
    for (int base = 0; base < P.nchunk; base += kRound * kWarp) {
      int4 rr[kRound];
#pragma unroll
      for (int k = 0; k < kRound; ++k) {
        const int c = base + k * kWarp + lane;
        rr[k] = c < P.nchunk ? rec[c] : (greedy ? make_int4(INT_MAX, __float_as_int(-INFINITY), INT_MAX,
                                                             __float_as_int(-INFINITY))
                                                : make_int4(kNoRef, 0, kNoRef, 0));
      }
#pragma unroll
      for (int k = 0; k < kRound; ++k) {
        const int4 r = rr[k];
        const int ua0 = r.x, ua1 = r.z;
        const float us0 = __int_as_float(r.y), us1 = __int_as_float(r.w);
        if (greedy) {
            if (us0 > ls0 || (us0 == ls0 && ua0 < la0)) {
                ls0 = us0;
                la0 = ua0;
            }
            if (us1 > ls1 || (us1 == ls1 && ua1 < la1)) {
                ls1 = us1;
                la1 = ua1;
            }
        } else {
            // a NaN sum (an invalid part) stays NaN
            const int n0 = max(la0, ua0), n1 = max(la1, ua1);
            ls0 = ls0 * pow2_int(la0 - n0) + ((ua0 == kNoRef) ? us0 * 0.0f : us0 * pow2_int(ua0 - n0));
            ls1 = ls1 * pow2_int(la1 - n1) + ((ua1 == kNoRef) ? us1 * 0.0f : us1 * pow2_int(ua1 - n1));
            la0 = n0;
            la1 = n1;
        }
      }
    }
    int a0, a1;
    float s0, s1;
    if (greedy) {
        arg_max<kWarp>(ls0, la0);
        arg_max<kWarp>(ls1, la1);
        a0 = la0;
        a1 = la1;
        s0 = ls0;
        s1 = ls1;
    } else {
        int B0 = la0, B1 = la1;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            B0 = max(B0, __shfl_xor_sync(0xffffffffu, B0, o));
            B1 = max(B1, __shfl_xor_sync(0xffffffffu, B1, o));
        }
        float t0 = ls0 * pow2_int(la0 - B0), t1 = ls1 * pow2_int(la1 - B1);
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            t0 += __shfl_xor_sync(0xffffffffu, t0, o);
            t1 += __shfl_xor_sync(0xffffffffu, t1, o);
        }
        a0 = B0;
        a1 = B1;
        s0 = t0;
        s1 = t1;
    }
    F2 Ex = {0.0f, 0.0f};
    int xf = 0;
    if (d.kind == I_PAIR && !greedy && d.xchunk >= 0) {
        const float4 xr = P.xrec[d.item];
        Ex = {xr.x, xr.y};
        xf = __float_as_int(xr.z);
    }
    return decide_item(P, d, d.status, a0, s0, a1, s1, Ex, xf);
}

// A decision with nothing to decide (the item's request was rejected before any work).
__device__ __forceinline__ ItemDec skip_decision(const ItemDesc &d) {
    ItemDec D = {};
    D.status = d.status;
    D.kind = SAMPLE_NONE;
    D.argmax_t = -1;
    return D;
}

// A lane's vectors of chunk c of a pair's two rows (pass 2's loads, mostly from L2).
template <int DT>
__device__ __forceinline__ void load_chunk(const VerifyParams &P, const ItemDesc &d, int c, uint64_t drop,
                                           uint4 (&vt)[kVPT], uint4 (&vd)[kVPT]) {
    const int lane = threadIdx.x % kWarp;
    const uint4 *trow = static_cast<const uint4 *>(P.target) + static_cast<size_t>(d.item) * P.nvec_row;
    const uint4 *drow = static_cast<const uint4 *>(P.draft) + static_cast<size_t>(d.drow) * P.nvec_row;
    const bool rows_ok = SPEC_IN(d.item, P.total_rows, DBG_LOGITS) && SPEC_IN(d.drow, P.total_rows - P.B, DBG_LOGITS);
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
        const int vi = c * kChunkVecs + k * kWarp + lane;
        const bool in = rows_ok && vi < P.nvec_row;
        vt[k] = in ? ldg_hint(trow + vi, drop) : kNegInfVec<DT>();
        vd[k] = in ? ldg_hint(drow + vi, drop) : kNegInfVec<DT>();
    }
}

// Pass 2 of chunk c of a pair (whole warp, the chunk's vectors loaded): (alpha share, residual
// mass) of the chunk, both normalised. Where the position rejects, max(p - q, 0) and min(p, q) by
// resid_weights; where it accepts, only alpha: min(p, q) = 2^min(y_t s - c_t, y_d s - c_d), c the
// log2 of the normaliser.
template <int DT>
__device__ __forceinline__ float2 chunk_pass2(const ItemDesc &d, const ItemDec &D, int c, uint4 (&vt)[kVPT],
                                              const uint4 (&vd)[kVPT]) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    const int lane = threadIdx.x % kWarp;
    if (d.trunc) {
        bool all = true;
#pragma unroll
        for (int k = 0; k < kVPT; ++k) all &= mask_cut<DT>(vt[k], c * kChunkVecs + k * kWarp + lane, d.cut_tau, d.cut_id);
        // p is 0 on the whole chunk: min(p, q) and max(p - q, 0) are 0 there
        if (__all_sync(0xffffffffu, all)) return make_float2(0.0f, 0.0f);
    }
    const float2 shi2 = f2splat(d.s_hi);
    const float2 nct = f2splat(-D.c_t), nctf = f2splat(neg_frac_lo(D.c_t, D.c_tf, d.s_hi, d.s_lo));
    float a, z = 0.0f;
    if (D.kind == SAMPLE_RESIDUAL) {
        const float2 slo2 = f2splat(d.s_lo);
        const float2 ndch = f2splat(-D.dc.hi), ndcl = f2splat(-D.dc.lo);
        float2 racc = make_float2(0.0f, 0.0f), aacc = racc;
#pragma unroll
        for (int k = 0; k < kVPT; ++k) {
#pragma unroll
            for (int h = 0; h < H; ++h) {
                float2 r, m;
                resid_weights(Elt<DT>::unpack_one(vt[k], h), Elt<DT>::unpack_one(vd[k], h), shi2, slo2, nct, nctf, ndch,
                              ndcl, r, m);
                racc = __fadd2_rn(racc, r);
                aacc = __fadd2_rn(aacc, m);
            }
        }
        a = aacc.x + aacc.y;
        z = racc.x + racc.y;
    } else {
        // y s - c with c split: the product less the integral part rounds once (to a small result
        // near the top of the row), then the fraction with the row's s_lo term (neg_frac_lo)
        const float2 ncd = f2splat(-D.c_d), ncdf = f2splat(neg_frac_lo(D.c_d, D.c_df, d.s_hi, d.s_lo));
        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < kVPT; ++k) {
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const float2 at = __fadd2_rn(__ffma2_rn(Elt<DT>::unpack_one(vt[k], h), shi2, nct), nctf);
                const float2 ad = __fadd2_rn(__ffma2_rn(Elt<DT>::unpack_one(vd[k], h), shi2, ncd), ncdf);
                acc = __fadd2_rn(acc, make_float2(ex2(fminf(at.x, ad.x)), ex2(fminf(at.y, ad.y))));
            }
        }
        a = acc.x + acc.y;
    }
    return make_float2(warp_sum(a), warp_sum(z));
}

// The draw weights of one vector, exactly as the passes summed them: the residual (normalised),
// or p in units of 2^B_t.
template <int DT>
__device__ __forceinline__ void draw_weights(int kind, const uint4 &wt, const uint4 &wd, const ItemDesc &d,
                                             const ItemDec &D, float *w) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    const float2 shi2 = f2splat(d.s_hi), slo2 = f2splat(d.s_lo);
    if (kind == SAMPLE_RESIDUAL) {
        const float2 nct = f2splat(-D.c_t), nctf = f2splat(neg_frac_lo(D.c_t, D.c_tf, d.s_hi, d.s_lo));
        const float2 ndch = f2splat(-D.dc.hi), ndcl = f2splat(-D.dc.lo);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            float2 r, m;
            resid_weights(Elt<DT>::unpack_one(wt, h), Elt<DT>::unpack_one(wd, h), shi2, slo2, nct, nctf, ndch, ndcl, r, m);
            w[2 * h] = r.x;
            w[2 * h + 1] = r.y;
        }
    } else {
        const float2 nbt = f2splat(-D.B_t);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float2 e = ex2x2(exp_arg2(Elt<DT>::unpack_one(wt, h), shi2, slo2, nbt));
            w[2 * h] = e.x;
            w[2 * h + 1] = e.y;
        }
    }
}

// The mass of chunk c in the law of the draw: the residual's (normalised; written by the item's
// finishing CTAs), or p's in units of 2^B_t (from the chunk's statistics).
__device__ __forceinline__ float chunk_mass(const VerifyParams &P, const ItemDesc &d, const ItemDec &D, int kind, int c) {
    if (kind == SAMPLE_RESIDUAL) return __ldcg(P.zc + static_cast<size_t>(d.item) * P.nchunk + c);
    const int4 r = P.rec[static_cast<size_t>(d.item) * P.nchunk + c];
    const float cm = __int_as_float(r.y);
    return (r.x == kNoRef || !(cm > 0.0f)) ? 0.0f : cm * pow2_int(r.x - static_cast<int>(D.B_t));
}

// The draw of item d from the law `kind` (whole warp): the chunk that holds u*Z by an inclusive
// scan over the chunk masses in vocabulary order, then the token within it, the weights recomputed
// exactly as the passes summed them. Writes the token, its probability and the CDF margin. `dry`:
// every chunk mass reads as 1 (a rehearsal that only reads memory, see spec_finish_kernel).
template <int DT>
__device__ __noinline__ void draw_item(const VerifyParams &P, const ItemDesc &d, const ItemDec &D, int kind, int &tok,
                                       float &prob, float &margin, bool dry = false) {
    constexpr int E = Elt<DT>::kPerVec;
    const int lane = threadIdx.x % kWarp;
    const int nc = P.nchunk;
    F2 Z = {0.0f, 0.0f}, t, before = {0.0f, 0.0f};
    int csel = -1;
    bool clamped = false;  // rounding put u*Z past the last chunk with mass
    const int m = (nc + kWarp - 1) / kWarp;
    if (m <= kDrawRun) {
        // lanes take consecutive runs of m chunks: every mass is loaded at once, one scan over the
        // lanes finds the run that holds u*Z, and that lane's walk through its run the chunk
        const int c0 = lane * m;
        float mm[kDrawRun];
#pragma unroll
        for (int k = 0; k < kDrawRun; ++k)
            mm[k] = (k < m && c0 + k < nc) ? (dry ? 1.0f : chunk_mass(P, d, D, kind, c0 + k)) : 0.0f;
        F2 own = {0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < kDrawRun; ++k) own = f2_add(own, {mm[k], 0.0f});
        Z = warp_sum_f2(own);
        t = f2_mul(Z, D.u_s);
        const F2 incl = warp_scan_f2(own, lane);
        const bool pos = own.hi > 0.0f;
        const unsigned hit = __ballot_sync(0xffffffffu, pos && f2_gt(incl, t));
        const unsigned posm = __ballot_sync(0xffffffffu, pos);
        if (posm) {
            const int L = hit ? __ffs(hit) - 1 : 31 - __clz(static_cast<int>(posm));
            int c_sel = -1, last = -1, found = 0;
            F2 bef = {0.0f, 0.0f}, last_bef = {0.0f, 0.0f};
            if (lane == L) {
                F2 run = f2_sub(incl, own);
#pragma unroll
                for (int k = 0; k < kDrawRun; ++k) {
                    if (mm[k] > 0.0f) {
                        const F2 nxt = f2_add(run, {mm[k], 0.0f});
                        if (hit && c_sel < 0 && f2_gt(nxt, t)) {
                            c_sel = c0 + k;
                            bef = run;
                        }
                        last = c0 + k;
                        last_bef = run;
                        run = nxt;
                    }
                }
                found = c_sel >= 0;
                if (!found) {
                    c_sel = last;
                    bef = last_bef;
                }
            }
            csel = __shfl_sync(0xffffffffu, c_sel, L);
            before = shfl_f2(bef, L);
            clamped = __shfl_sync(0xffffffffu, found, L) == 0;
        }
    } else {
        // long rows: the masses in rounds of 32 chunks, read twice (once for Z, once for the scan)
        for (int base = 0; base < nc; base += kWarp) {
            const int c = base + lane;
            const float mv = c < nc ? chunk_mass(P, d, D, kind, c) : 0.0f;
            Z = f2_add(Z, warp_sum_f2({mv, 0.0f}));
        }
        t = f2_mul(Z, D.u_s);
        int clast = -1;
        F2 last_before = {0.0f, 0.0f}, run = {0.0f, 0.0f};
        for (int base = 0; base < nc; base += kWarp) {
            const int c = base + lane;
            const float mv = c < nc ? chunk_mass(P, d, D, kind, c) : 0.0f;
            const bool pos = mv > 0.0f;
            const F2 incl = f2_add(run, warp_scan_f2({mv, 0.0f}, lane));
            const unsigned hit = __ballot_sync(0xffffffffu, pos && f2_gt(incl, t));
            const unsigned posm = __ballot_sync(0xffffffffu, pos);
            if (hit) {
                const int l = __ffs(hit) - 1;
                csel = base + l;
                before = shfl_f2(f2_sub(incl, {mv, 0.0f}), l);
                break;
            }
            if (posm) {
                const int l = 31 - __clz(static_cast<int>(posm));
                clast = base + l;
                last_before = shfl_f2(f2_sub(incl, {mv, 0.0f}), l);
            }
            run = shfl_f2(incl, kWarp - 1);
        }
        clamped = csel < 0;
        if (clamped) {
            csel = clast;
            before = last_before;
        }
    }
    tok = -1;
    prob = NAN;
    margin = NAN;
    if (csel < 0) return;
    const F2 rem = f2_sub(t, before);
    const float lt = rem.hi + rem.lo;
    const float invZ = rcp_approx(Z.hi);
    const uint4 *trow = static_cast<const uint4 *>(P.target) + static_cast<size_t>(d.item) * P.nvec_row;
    const uint4 *drow = static_cast<const uint4 *>(P.draft) + static_cast<size_t>(d.drow) * P.nvec_row;
    // the chunk's vectors c*128 + 32k + lane, in vocabulary order k-major; a loop (not unrolled:
    // this code runs once per draw, and a compact body is fetched once), the next vector's loads in
    // flight while one is searched
    auto load = [&](int k, uint4 &wt, uint4 &wd) {
        const int vi = csel * kChunkVecs + k * kWarp + lane;
        wt = kNegInfVec<DT>();
        wd = kNegInfVec<DT>();
        if (vi < P.nvec_row && SPEC_IN(d.item, P.total_rows, DBG_LOGITS)) {
            wt = __ldcg(trow + vi);
            if (kind == SAMPLE_RESIDUAL && SPEC_IN(d.drow, P.total_rows - P.B, DBG_LOGITS)) wd = __ldcg(drow + vi);
        }
    };
    float c = 0.0f;  // mass before vector (k, lane) within the chunk
    int last_k = -1, last_e = -1, found_e = -1, hk = -1;
    float fprev = 0.0f, wf = 0.0f, wl = 0.0f;
    unsigned hit = 0u;
    uint4 wt, wd;
    load(0, wt, wd);
#pragma unroll 1
    for (int k = 0; k < kVPT; ++k) {
        uint4 nt = wt, nd = wd;
        if (k + 1 < kVPT) load(k + 1, nt, nd);
        if (d.trunc) mask_cut<DT>(wt, csel * kChunkVecs + k * kWarp + lane, d.cut_tau, d.cut_id);
        float w[E];
        draw_weights<DT>(kind, wt, wd, d, D, w);
        float vsk = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) vsk += w[e];
        float incl = vsk;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const float x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        float cc = c + incl - vsk;
        int fe = -1;
        float fp = 0.0f, fw = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (w[e] > 0.0f) {
                if (fe < 0 && !clamped && cc + w[e] > lt) {
                    fe = e;
                    fp = cc;
                    fw = w[e];
                }
                last_k = k;
                last_e = e;
                wl = w[e];
            }
            cc += w[e];
        }
        const unsigned h = __ballot_sync(0xffffffffu, fe >= 0);
        if (h) {
            hk = k;
            hit = h;
            found_e = fe;
            fprev = fp;
            wf = fw;
            break;
        }
        c += __shfl_sync(0xffffffffu, incl, kWarp - 1);
        wt = nt;
        wd = nd;
    }
    if (hk >= 0) {
        const int l = __ffs(hit) - 1;
        const float c0 = __shfl_sync(0xffffffffu, fprev, l);
        const float wsel = __shfl_sync(0xffffffffu, wf, l);
        const int e = __shfl_sync(0xffffffffu, found_e, l);
        tok = (csel * kChunkVecs + hk * kWarp + l) * E + e;
        prob = wsel * invZ;
        margin = fminf(lt - c0, c0 + wsel - lt) * invZ;
    } else {
        // rounding: the last element with mass (the largest vocabulary index holding mass)
        const int key = last_k >= 0 ? (last_k * kWarp + lane) * E + last_e : -1;
        int best = key;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
        if (best >= 0) {
            const int owner = (best / E) % kWarp;
            const float wsel = __shfl_sync(0xffffffffu, wl, owner);
            tok = csel * kChunkVecs * E + best;
            prob = wsel * invZ;
            margin = 0.0f;
        }
    }
}

// A request's outputs once its frontier token is known (whole warp, the frontier item's warp):
// the accepted drafts x_1 .. x_A, then the frontier token, cut by the stop token and the
// budget (SDCP "Verification and Commit" step 7), -1 past the emitted tokens. Lane j writes
// positions j and j + 32 (K_max <= 64: position 64 on lane 0).
__device__ __noinline__ void finish_request(const VerifyParams &P, int i, int r0, int K, int A, int frontier,
                                            float fprob, float fmarg, int ffb) {
    const int lane = threadIdx.x % kWarp;
    const int d0 = r0 - i;
    const int n_cap = P.max_new ? __ldg(P.max_new + i) : INT_MAX;
    const int stop = P.stop_token ? __ldg(P.stop_token + i) : -1;
    const int x0 = lane < A ? __ldg(P.draft_tokens + d0 + lane) : -1;
    const int x1 = lane + kWarp < A ? __ldg(P.draft_tokens + d0 + lane + kWarp) : -1;
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
    if (lane <= K && SPEC_IN(r0 + lane, P.total_rows, DBG_OUT_ROWS)) P.out_tokens[r0 + lane] = lane < n ? out0 : -1;
    if (lane + kWarp <= K && SPEC_IN(r0 + lane + kWarp, P.total_rows, DBG_OUT_ROWS))
        P.out_tokens[r0 + lane + kWarp] = lane + kWarp < n ? out1 : -1;
    if (lane == 0 && K == 2 * kWarp && SPEC_IN(r0 + K, P.total_rows, DBG_OUT_ROWS))
        P.out_tokens[r0 + K] = (A == K && n > K) ? frontier : -1;
    if (lane == 0 && SPEC_IN(i, P.B, DBG_OUT_REQS)) {
        P.req_status[i] = 0;
        P.accept_len[i] = A;
        if (P.n_emitted) P.n_emitted[i] = n;
        if (P.frontier_prob) P.frontier_prob[i] = fprob;
        if (P.frontier_margin) P.frontier_margin[i] = fmarg;
        if (P.fallback) P.fallback[i] = ffb;
    }
}

// The item's results (whole warp; alpha and the residual mass Zres from pass 2): its per-draft
// outputs and its share of the batch's alpha; at its request's frontier the draw and the request's
// outputs (finish_request). Then the batch's count: returns, in every lane, whether this was the
// batch's last item (its CTA then runs the batch's tail).
template <int DT>
__device__ __noinline__ bool finalize_item(const VerifyParams &P, const ItemDesc &d, const ItemDec &D, int rst, int A,
                                           float alpha, float Zres) {
    const int lane = threadIdx.x % kWarp;
    const bool pair = d.kind == I_PAIR;
    // the request's frontier: its first rejection, or its bonus row with every draft accepted
    const bool frontier = rst == 0 && d.pos == A;
    int kind = frontier ? D.kind : SAMPLE_NONE;
    int fb = 0;
    if (kind == SAMPLE_RESIDUAL && !(Zres > 0.0f)) {
        kind = SAMPLE_P;  // zero residual mass: draw from p and say so
        fb = 1;
    }
    int tok = -1;
    float prob = NAN, margin = NAN;
    if (kind != SAMPLE_NONE) {
        draw_item<DT>(P, d, D, kind, tok, prob, margin);
    } else if (frontier && d.greedy) {
        tok = D.argmax_t;  // Rule 1: the correction (or the extra token) is argmax p
        prob = 1.0f;
    }
    // a draft position: a pair, or a position of a request rejected before any work (every draft
    // row of a request with status bits gets the no-result values)
    const bool drow_item =
        pair || (d.kind == I_SKIP && d.pos < d.K && d.drow >= 0 && d.drow < P.total_rows - P.B);
    if (lane == 0 && drow_item && SPEC_IN(d.drow, P.total_rows - P.B, DBG_OUT_ROWS)) {
        const float a = d.greedy ? D.alpha_g : alpha;
        if (P.alpha_rows) P.alpha_rows[d.drow] = (rst == 0) ? a : NAN;
        if (P.rho_rows) P.rho_rows[d.drow] = (rst == 0) ? D.rho : NAN;
        if (P.resid_rows)
            P.resid_rows[d.drow] = (frontier && D.kind == SAMPLE_RESIDUAL && !d.greedy) ? Zres : -1.0f;
        if (rst == 0) {
            // the batch's alpha in fixed point: integer sums give the same result in any order
            atomicAdd(reinterpret_cast<unsigned long long *>(P.agg + AGG_ALPHA),
                      static_cast<unsigned long long>(__float2ll_rn(a * static_cast<float>(kAlphaFix))));
        }
    }
    if (frontier) finish_request(P, d.req, d.item - d.pos, d.K, A, tok, prob, margin, fb);
    __syncwarp();
    uint32_t done = 0;
    if (lane == 0) {
        fence_gpu();  // this item's writes before the batch's count
        done = atomicAdd(P.ctl + CTL_DONE, 1u);
    }
    done = __shfl_sync(0xffffffffu, done, 0);
    return done == static_cast<uint32_t>(P.total_rows - 1);
}

// ------------------------------------------------------------------------------------------------
// the batch's tail (the CTA that finalised the last item): the alpha sum and depth counts, then (a
// round) compaction and gamma

struct TailScratch {
    CompactScratch<kFinBlock> cs;
};

// The batch's tail, by the CTA that finalised the batch's last item: the alpha sum and depth
// counts (accumulated by the requests' selections), then, for a round, the compaction and the
// gamma choice. With row offsets that fail their checks, every request is reported BAD_SHAPE.
__device__ __noinline__ void batch_tail(const VerifyParams &P, TailScratch &S) {
    const int tid = threadIdx.x;
    const bool bad_off = __ldcg(P.ctl + CTL_BAD_OFFSETS) != 0;
    if (bad_off) {
        for (int i = tid; i < P.B; i += kFinBlock) {
            const int r0 = __ldg(P.row_off + i), r1 = __ldg(P.row_off + i + 1);
            const int K = r1 - r0 - 1;
            if (K >= 0 && r0 >= 0 && r1 <= P.total_rows)
                for (int j = 0; j <= K; ++j) P.out_tokens[r0 + j] = -1;
            P.req_status[i] = SPEC_REQ_BAD_SHAPE;
            P.accept_len[i] = 0;
            if (P.n_emitted) P.n_emitted[i] = 0;
            if (P.frontier_prob) P.frontier_prob[i] = NAN;
            if (P.frontier_margin) P.frontier_margin[i] = NAN;
            if (P.fallback) P.fallback[i] = 0;
        }
    }
    if (tid == 0) {
        const unsigned long long fx = __ldcg(reinterpret_cast<const unsigned long long *>(P.agg + AGG_ALPHA));
        // the one float64 operation of the call: the fixed-point sum becomes the output double
        if (P.alpha_sum) *P.alpha_sum = static_cast<double>(static_cast<long long>(fx)) / kAlphaFix;
        if (P.alpha_count) *P.alpha_count = static_cast<int32_t>(__ldcg(P.agg + AGG_COUNT));
    }
    for (int j = tid; j < P.K_max; j += kFinBlock) {
        if (P.depth_reached) P.depth_reached[j] = static_cast<int32_t>(__ldcg(P.agg + AGG_REACHED + j));
        if (P.depth_accepted) P.depth_accepted[j] = static_cast<int32_t>(__ldcg(P.agg + AGG_ACCEPTED + j));
    }
    fence_gpu();
    __syncthreads();
    if (P.round) {
        compact_body<kFinBlock>(P.C, false,
                                (P.C.row_off == P.row_off && P.C.B == P.B && P.C.total_rows == P.total_rows)
                                    ? (bad_off ? 0 : 1)
                                    : -1,
                                S.cs);
        __syncthreads();
        if (tid == 0) gamma_body(P.G);
    }
}

// Decisions: one CTA per request, a warp per position (the item's chunk statistics combined),
// then the request's frontier: its first rejected position, or its bonus row when every draft is
// accepted (only the frontier is drawn).
template <int DT>
__global__ void __launch_bounds__(kDecWarps * kWarp) spec_decide_kernel(const __grid_constant__ VerifyParams Pk) {
    __shared__ int s_first;   // the first rejected position (none: INT_MAX)
    __shared__ int s_status;  // the status bits of the request's positions
    __shared__ __align__(16) VerifyParams s_P;
    stage_params<kDecWarps * kWarp>(Pk, s_P);
    const VerifyParams &P = s_P;
    const int warp = static_cast<int>(threadIdx.x) / kWarp, lane = static_cast<int>(threadIdx.x) % kWarp;
    const int i = static_cast<int>(blockIdx.x);
    griddep_wait();  // the statistics kernel's records
    griddep_launch_dependents();
    if (__ldcg(P.ctl + CTL_BAD_OFFSETS) != 0) return;
    const int r0 = __ldg(P.row_off + i), r1 = __ldg(P.row_off + i + 1);
    const int n = r1 - r0;  // K + 1 positions (offsets checked)
    if (threadIdx.x == 0) {
        s_first = INT_MAX;
        s_status = 0;
    }
    __syncthreads();
    for (int j = warp; j < n; j += kDecWarps) {
        if (!SPEC_IN(r0 + j, P.total_rows, DBG_ROWS)) continue;
        const ItemDesc d = P.desc[r0 + j];
        const ItemDec D = (d.kind == I_SKIP) ? skip_decision(d) : decide_chunks(P, d);
        if (lane == 0) {
            if (d.kind == I_PAIR && D.status == 0 && !D.accept) atomicMin(&s_first, j);
            if (D.status) atomicOr(&s_status, D.status);
            P.dec[r0 + j] = D;
        }
    }
    __syncthreads();
    const int K = n - 1;
    const int A = min(s_first, K);  // drafts accepted before the first rejection
    const int status = s_status;
    if (threadIdx.x == 0) {
        // the frontier: the first rejection, else the bonus row
        if (SPEC_IN(r0 + A, P.total_rows, DBG_ROWS)) P.dec[r0 + A].frontier = 1;
        if (SPEC_IN(i, P.B, DBG_OUT_REQS)) {
            P.req_first[i] = A;
            P.req_st[i] = status;
        }
    }
    if (warp != 0) return;
    if (status) {
        // a request with any status bit emits nothing (its draft rows get their no-result values
        // from the finishing kernel)
        for (int j = lane; j <= K; j += kWarp)
            if (SPEC_IN(r0 + j, P.total_rows, DBG_OUT_ROWS)) P.out_tokens[r0 + j] = -1;
        if (lane == 0 && SPEC_IN(i, P.B, DBG_OUT_REQS)) {
            P.req_status[i] = status;
            P.accept_len[i] = 0;
            if (P.n_emitted) P.n_emitted[i] = 0;
            if (P.frontier_prob) P.frontier_prob[i] = NAN;
            if (P.frontier_margin) P.frontier_margin[i] = NAN;
            if (P.fallback) P.fallback[i] = 0;
        }
        return;
    }
    // the batch's counts ("M7.8 - Speculative Serving", sections 0x02D and 0x07B): the draft rows
    // in alpha's mean, and depth j + 1 reached when the first j drafts were accepted, accepted
    // when j < A
    if (lane == 0) atomicAdd(P.agg + AGG_COUNT, static_cast<uint32_t>(K));
    for (int j = lane; j < K; j += kWarp) {
        if (j <= A) atomicAdd(P.agg + AGG_REACHED + j, 1u);
        if (j < A) atomicAdd(P.agg + AGG_ACCEPTED + j, 1u);
    }
}

// Pass 2: every chunk of every pair under Rule 2, each warp a contiguous run of (pair, chunk)
// pieces, the bonus rows left out of the enumeration (the item's values and decision read once
// per item). A chunk's alpha share goes to
// alpha_c; at the request's frontier (its first rejection) its residual mass goes to zc.
template <int DT>
__global__ void __launch_bounds__(kFinBlock, 4) spec_pass2_kernel(const __grid_constant__ VerifyParams P) {
    const int lane = static_cast<int>(threadIdx.x) % kWarp;
    griddep_wait();  // the statistics and decision kernels' output
    griddep_launch_dependents();
    if (__ldcg(P.ctl + CTL_BAD_OFFSETS) != 0) return;
    const uint64_t drop = policy_evict_first();
    const long long warps = static_cast<long long>(gridDim.x) * kFinWarps;
    const long long gw = static_cast<long long>(blockIdx.x) * kFinWarps + threadIdx.x / kWarp;
    // units over the pairs only: unit u is chunk u % nchunk of draft row p = u / nchunk, whose
    // target row is p + i for the request i holding it (the bonus rows of requests before it
    // lie in between)
    const long long total = static_cast<long long>(P.total_rows - P.B) * P.nchunk;
    const long long per = (total + warps - 1) / warps;
    const long long u1 = min(total, (gw + 1) * per);
    int cur = -1;
    bool work = false, frontier = false;
    ItemDesc d = {};
    ItemDec D = {};
    const long long ub = gw * per;
    if (ub >= u1) return;
    int p = static_cast<int>(ub / P.nchunk), c = static_cast<int>(ub % P.nchunk) - 1;
    int i = 0;
    {
        int lo = 0, hi = P.B - 1;  // the last request whose first draft row is at most p
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(P.row_off + mid) - mid <= p) lo = mid; else hi = mid - 1;
        }
        i = lo;
    }
    int next_first = __ldg(P.row_off + i + 1) - (i + 1);  // the first draft row past request i
    while (p >= next_first && i + 1 < P.B) {
        ++i;
        next_first = __ldg(P.row_off + i + 1) - (i + 1);
    }
    for (long long u = ub; u < u1; ++u) {
        if (++c == P.nchunk) {
            c = 0;
            ++p;
            while (p >= next_first && i + 1 < P.B) {
                ++i;
                next_first = __ldg(P.row_off + i + 1) - (i + 1);
            }
        }
        const int item = p + i;
        if (item != cur) {
            cur = item;
            d = P.desc[item];
            D = P.dec[item];
            work = has_p2(d) && D.status == 0;
            frontier = D.frontier != 0;
            // alpha everywhere; the residual only where the request draws from it
            if (!frontier && D.kind == SAMPLE_RESIDUAL) D.kind = SAMPLE_NONE;
        }
        if (!work) continue;
        uint4 vt[kVPT], vd[kVPT];
        load_chunk<DT>(P, d, c, drop, vt, vd);
        const float2 r = chunk_pass2<DT>(d, D, c, vt, vd);
        if (lane == 0 && SPEC_IN(static_cast<long long>(item) * P.nchunk + c,
                                 static_cast<long long>(P.total_rows) * P.nchunk, DBG_RECORDS)) {
            P.alpha_c[static_cast<size_t>(item) * P.nchunk + c] = r.x;
            if (frontier) P.zc[static_cast<size_t>(item) * P.nchunk + c] = r.y;
        }
    }
}

// Draws and selections: one warp per item. Alpha and the residual mass are the item's chunk
// shares summed; the request's frontier draws its token; the item is counted for its request (the
// last item of a request runs its selection) and the batch (the CTA holding the last item runs the
// batch's tail).
template <int DT>
__global__ void __launch_bounds__(kFinBlock) spec_finish_kernel(const __grid_constant__ VerifyParams Pk) {
    __shared__ int s_tail;
    __shared__ TailScratch s_ts;
    __shared__ __align__(16) VerifyParams s_P;
    stage_params<kFinBlock>(Pk, s_P);
    const VerifyParams &P = s_P;
    const int lane = static_cast<int>(threadIdx.x) % kWarp;
    const int item = static_cast<int>(blockIdx.x) * kFinWarps + static_cast<int>(threadIdx.x) / kWarp;
    if (threadIdx.x == 0) s_tail = 0;
    if (threadIdx.x < kWarp && P.total_rows > 0) {
        // While pass 2 runs, one warp rehearses a draw on item 0's rows (reads only, its result
        // unused): the draws that follow then run from this SM's instruction cache instead of
        // fetching the code line by line.
        ItemDesc dd = {};
        dd.kind = I_PAIR;
        dd.s_hi = 1.0f;
        dd.s_lo = 0x1p-40f;
        ItemDec DD = {};
        DD.u_s = {0.5f, 0.0f};
        int tk;
        float pr, mg;
        draw_item<DT>(P, dd, DD, (P.total_rows > P.B) ? SAMPLE_RESIDUAL : SAMPLE_P, tk, pr, mg, true);
        if (tk == INT_MIN && threadIdx.x == 0) s_tail = 0;  // keeps the rehearsal
    }
    __syncthreads();
    griddep_wait();  // pass 2 (and, through it, the kernels before)
    if (__ldcg(P.ctl + CTL_BAD_OFFSETS) != 0) {
        // the row offsets fail their checks: no item is looked at; the batch's tail reports every
        // request BAD_SHAPE
        if (item < P.total_rows && lane == 0 &&
            atomicAdd(P.ctl + CTL_DONE, 1u) == static_cast<uint32_t>(P.total_rows - 1))
            s_tail = 1;
    } else if (item < P.total_rows) {
        const ItemDesc d = P.desc[item];
        const ItemDec D = P.dec[item];
        const int rst = P.req_st[d.req], A = P.req_first[d.req];  // from the decision kernel
        const bool frontier = rst == 0 && d.pos == A;
        float alpha = 0.0f, Zres = 0.0f;
        if (has_p2(d) && D.status == 0) {
            // sums over the chunks, lane-strided, then over the lanes (the same in every lane)
            float a = 0.0f, z = 0.0f;
            for (int c = lane; c < P.nchunk; c += kWarp) {
                a += P.alpha_c[static_cast<size_t>(item) * P.nchunk + c];
                if (frontier) z += P.zc[static_cast<size_t>(item) * P.nchunk + c];
            }
            alpha = warp_sum(a);
            Zres = warp_sum(z);
        }
        const bool tail = finalize_item<DT>(P, d, D, rst, A, alpha, Zres);
        if (lane == 0 && tail) s_tail = 1;
    }
    __syncthreads();
    if (s_tail) {
        fence_gpu();
        batch_tail(P, s_ts);
    }
}

}  // namespace vk
}  // namespace spec
