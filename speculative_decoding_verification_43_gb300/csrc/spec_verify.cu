// Batched speculative-decoding verifier for GB300 (sm_103a): spec_verify.
//
// The rule is the one of "SOTA-227: Decode with a draft model and an accept-reject rule"
// ("What to do", steps 3-4) and SDCP Rules 1 and 2 ("Acceptance Rules"); the C ABI and its
// conventions are documented in include/spec_verify.h.
//
// Design. The work unit is one target row ("item"): position j < K_i of request i is a pair
// (target row j, draft row j), position K_i is the target-only row that yields the bonus token
// (or the plain sample when K_i = 0). Each item is verified by one thread-block cluster of C
// CTAs; CTA c owns the c-th slice of the vocabulary of both rows and stages it in its own
// shared memory with 1-D bulk copies, so every logit is read from HBM exactly once:
//   pass 1 (while the copies land): per 1024-token group, max and sum of 2^(y*s - b) with the
//           group's own reference b; the cluster combines (b, S) through DSMEM;
//   accept test (fp64, identical in every CTA): rho = p(x)/q(x), accept when u <= rho;
//   pass 2 (pairs, from shared memory): alpha = sum min(p, q); if this position rejects, also
//           the residual r = max(p - q, 0) with its per-group sums. Every rejecting position
//           prepares its own candidate, so no item waits for another;
//   draw: the CTA whose slice holds u*Z walks its group sums, then one group's elements.
// A second kernel walks each request's accept flags left to right (a warp ballot), picks the
// candidate of the first rejection or the bonus, applies stop-token / max_new truncation and
// reduces alpha for the gamma controller.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "spec_device.cuh"
#include "spec_verify.h"

namespace spec {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / kWarp;
constexpr int kVecPerLane = 4;                   // 16-byte vectors per lane in one group
constexpr int kGroupVecs = kWarp * kVecPerLane;  // 128 vectors = 2 KiB per row per group
constexpr int kMaxChunks = 4;                    // bulk copies per row slice
constexpr int kMaxCluster = 16;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: a copy never takes this long
constexpr double kLog2e = 1.4426950408889634074;

enum : int32_t { REQ_TIMEOUT = 32 };  // internal: a bulk copy did not complete in time

template <int DT>
struct Elt;
template <>
struct Elt<SPEC_F32> {
    static constexpr int kPerVec = 4;
    __device__ static __forceinline__ void unpack(const uint4 &w, float *y) {
        y[0] = __uint_as_float(w.x);
        y[1] = __uint_as_float(w.y);
        y[2] = __uint_as_float(w.z);
        y[3] = __uint_as_float(w.w);
    }
    __device__ static __forceinline__ float at(const uint4 *buf, int e) {
        return reinterpret_cast<const float *>(buf)[e];
    }
};
template <>
struct Elt<SPEC_BF16> {
    static constexpr int kPerVec = 8;
    // bfloat16 is the upper half of a binary32: widening is a shift. The element at the lower
    // address is the low half of each 32-bit word.
    __device__ static __forceinline__ void unpack(const uint4 &w, float *y) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[2 * k] = __uint_as_float(u[k] << 16);
            y[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ float at(const uint4 *buf, int e) {
        const uint16_t b = reinterpret_cast<const uint16_t *>(buf)[e];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};

// ---- two-float arithmetic: a value hi + lo carried in float32 (about 48 significant bits).
// FP64 runs at a small fraction of the FP32 rate on this part, so sums that need more than
// float32 precision are kept as float pairs instead.
struct F2 {
    float hi, lo;
};
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    float e = (a.hi - (s - bb)) + (b.hi - bb);
    e += a.lo + b.lo;
    const float hi = s + e;
    return {hi, e - (hi - s)};
}
// a * 2^k, exact; k is clamped so that a wild exponent gives 0 rather than undefined behaviour
__device__ __forceinline__ F2 f2_scale(F2 a, float k) {
    const int kk = static_cast<int>(fminf(fmaxf(k, -300.0f), 300.0f));
    return {ldexpf(a.hi, kk), ldexpf(a.lo, kk)};
}
__device__ __forceinline__ float scale2(float a, float k) {
    return ldexpf(a, static_cast<int>(fminf(fmaxf(k, -300.0f), 300.0f)));
}
__device__ __forceinline__ F2 warp_sum_f2(F2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        F2 w;
        w.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        v = f2_add(v, w);
    }
    return v;
}
// a / b for positive a, b: a first quotient, then the quotient of the exact remainder
__device__ __forceinline__ F2 f2_div(F2 a, F2 b) {
    const float q1 = a.hi / b.hi;
    const float p_hi = q1 * b.hi;
    const float p_err = fmaf(q1, b.hi, -p_hi);
    const float r = ((a.hi - p_hi) - p_err) + a.lo - q1 * b.lo;
    const float q2 = r / b.hi;
    const float hi = q1 + q2;
    return {hi, q2 - (hi - q1)};
}
__device__ __forceinline__ double f2_d(F2 a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }

struct RowsParams {
    const void *target;
    const void *draft;
    const int32_t *row_off;
    const int32_t *draft_tokens;
    const double *uniforms;
    const float *temperature;
    float temperature_scalar;
    int32_t B, V, K_max, total_rows;
    int32_t nvec_row;        // 16-byte vectors per row
    int32_t slice_vecs_max;  // vectors of the largest slice
    int32_t groups_max;      // groups of the largest slice
    // per-item results (workspace), indexed by target row
    int32_t *item_flag;    // 1: the draft at this position is accepted
    int32_t *item_tok;     // candidate frontier token of this position (-1: none)
    int32_t *item_status;  // SPEC_REQ_* bits found by this item
    int32_t *item_fb;      // 1: residual had zero mass, drawn from p
    float *item_prob;      // probability of the candidate in its law
    float *item_margin;    // CDF margin of the candidate's draw
    float *alpha_ws;       // [T-B] alpha per draft row (always written)
    // optional outputs
    float *alpha_rows;
    float *rho_rows;
    float *resid_rows;
};

// What a CTA publishes after pass 1; it writes its record into slot `rank` of every CTA of
// the cluster (distributed shared memory), so that after the cluster barrier all reads are
// local. Fields are 32-bit words.
struct Ex1 {
    float B[2];      // integral reference exponent of S[r] (-inf: no mass)
    float S_hi[2];   // sum over the slice of 2^(y*s - B[r]), as a float pair
    float S_lo[2];
    int32_t bad[2];  // a NaN / +inf was seen in row r's slice
    float yx[2];     // target / draft logit at the draft token, from the CTA that holds it
    int32_t has_x;
    float gmax[2];   // greedy rule: max logit of the slice and the smallest index attaining it
    int32_t garg[2];
};
constexpr int kEx1Words = sizeof(Ex1) / 4;
// What a CTA publishes after pass 2.
struct Ex2 {
    float alpha;     // this slice's share of alpha (normalised)
    float Z_hi;      // this slice's residual mass, units of 2^B_t (float pair)
    float Z_lo;
};
constexpr int kEx2Words = sizeof(Ex2) / 4;

// Item-wide values, computed once and broadcast through shared memory.
struct ItemInfo {
    int32_t req, pos, K, drow, status, pair, greedy, accept, x, sample_kind;
    int32_t lo;      // first vector of this CTA's slice
    int32_t nvec;    // vectors in this CTA's slice
    int32_t groups;  // groups in this CTA's slice
    int32_t nchunk;
    int32_t owner;   // CTA that draws the candidate (-1: none)
    double u_acc, u_s;
    float s_hi, s_lo;  // log2(e)/T = s_hi + s_lo, s_hi rounded toward zero (s_lo > 0)
    float B_t, B_d;    // cluster-wide integral reference exponents
    F2 S_t, S_d;       // cluster-wide sums in those units
    float c_t, c_d;    // B + log2 S, for the alpha-only path
    F2 lam;            // S_t / S_d
    float rho, alpha, inv_St;
    double target_t, owner_prefix, Ztot, Zres;
    int32_t argmax_t, argmax_d;
};

enum { SAMPLE_NONE = 0, SAMPLE_RESIDUAL = 1, SAMPLE_P = 2 };

__device__ __forceinline__ void chunk_range(int groups, int nchunk, int k, int nvec, int &g0, int &g1,
                                            int &v0, int &v1) {
    g0 = (groups * k) / nchunk;
    g1 = (groups * (k + 1)) / nchunk;
    v0 = g0 * kGroupVecs;
    v1 = min(g1 * kGroupVecs, nvec);
}

// Vector vi of a slice (a 16-byte vector of E elements). Past the slice the elements read as
// -inf, which carries no mass and never wins a max.
template <int DT>
__device__ __forceinline__ void load_vec(const uint4 *buf, int vi, int nvec, float *y) {
    constexpr int E = Elt<DT>::kPerVec;
    if (vi < nvec) {
        Elt<DT>::unpack(buf[vi], y);
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) y[e] = -INFINITY;
    }
}

// Max of one vector, NaN ignored (NaN is caught later by the sums).
template <int DT>
__device__ __forceinline__ float vec_max(const uint4 &w) {
    if constexpr (DT == SPEC_BF16) {
        const uint32_t m01 = bf16x2_max(w.x, w.y), m23 = bf16x2_max(w.z, w.w);
        const uint32_t m = bf16x2_max(m01, m23);
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    } else {
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                     fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
}

// y*s - b with s = s_hi + s_lo (s_lo > 0): the product with s_hi and the subtraction of b round
// once, to the small result, then the s_lo term is added. y = -inf gives -inf.
__device__ __forceinline__ float exp_arg(float y, float s_hi, float s_lo, float b) {
    return fmaf(y, s_lo, fmaf(y, s_hi, -b));
}

// Weights of this lane's E elements of vector vi in the law the candidate is drawn from:
// RESIDUAL: max(e_t - lambda*e_d, 0) = S_t * max(p - q, 0) in units of 2^B_t;
// P: 2^(y*s - b_g), the pass-1 terms of the group (units of 2^b_g). The arithmetic is the same
// instruction sequence as in passes 1 and 2, so the values are bitwise those the sums saw.
template <int DT>
__device__ __forceinline__ void vec_weights(int kind, const uint4 *buf_t, const uint4 *buf_d, int vi, int nvec,
                                            const ItemInfo &I, float bg, float *w) {
    constexpr int E = Elt<DT>::kPerVec;
    float yt[E];
    load_vec<DT>(buf_t, vi, nvec, yt);
    if (kind == SAMPLE_RESIDUAL) {
        float yd[E];
        load_vec<DT>(buf_d, vi, nvec, yd);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const float et = ex2(exp_arg(yt[e], I.s_hi, I.s_lo, I.B_t));
            const float ed = ex2(exp_arg(yd[e], I.s_hi, I.s_lo, I.B_d));
            w[e] = fmaxf(fmaf(-I.lam.lo, ed, fmaf(-I.lam.hi, ed, et)), 0.0f);
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e) w[e] = ex2(exp_arg(yt[e], I.s_hi, I.s_lo, bg));
    }
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Lane l < C copies `words` 32-bit words of the local record into slot `rank` of CTA l.
__device__ __forceinline__ void push_record(const void *mine, void *slot_base, int rank, int words, int C,
                                            int lane) {
    if (lane < C) {
        const uint32_t *src = static_cast<const uint32_t *>(mine);
        const uint32_t dst = dsmem_map(static_cast<uint32_t *>(slot_base) + rank * words, lane);
        for (int w = 0; w < words; ++w) st_cluster_u32(dst + 4 * w, src[w]);
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 6) spec_rows_kernel(const RowsParams P) {
    constexpr int E = Elt<DT>::kPerVec;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bars[2][kMaxChunks];
    __shared__ Ex1 xch1[kMaxCluster];
    __shared__ Ex2 xch2[kMaxCluster];
    __shared__ Ex1 mine1;
    __shared__ Ex2 mine2;
    __shared__ ItemInfo I;
    __shared__ float red_f[kWarps];

    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
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
        const unsigned char *src = static_cast<const unsigned char *>(P.target) +
                                   static_cast<size_t>(item) * row_bytes + static_cast<size_t>(lo) * 16;
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
            int vals[8];
            int cnt = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int idx = lane * 8 + k;
                vals[k] = idx <= P.B ? __ldg(P.row_off + idx) : INT_MAX;
                cnt += vals[k] <= item;
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
            const double s64 = (T > 0.0f && !isinf(T)) ? kLog2e / static_cast<double>(T) : 0.0;
            // s = s_hi + s_lo with s_hi rounded toward zero, so s_lo > 0: then a -inf logit
            // gives -inf in both terms of exp_arg (a negative s_lo would make it NaN)
            I.s_hi = __double2float_rz(s64);
            I.s_lo = fmaxf(static_cast<float>(s64 - static_cast<double>(I.s_hi)), 1.401298464e-45f);
            if (status == 0) {
                u_acc_reg = __ldg(P.uniforms + item);
                u_s_reg = __ldg(P.uniforms + r1 - 1);
                if (I.pair) x_reg = __ldg(P.draft_tokens + d);
            }
            I.status = status;
            // draft copies, once the draft row is known
            if (I.pair) {
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
    bool timed_out = false;

    // ---- pass 1: per-group statistics as the chunks land ----
    for (int r = 0; r < nrows; ++r) {
        const uint4 *buf = r ? buf_d : buf_t;
        for (int k = 0; k < nchunk; ++k) {
            if (!mbar_wait_bounded(&bars[r][k], 0, kWaitLimitNs)) timed_out = true;
            int g0, g1, v0, v1;
            chunk_range(groups, nchunk, k, nvec, g0, g1, v0, v1);
            for (int g = g0 + warp; g < g1; g += kWarps) {
                const int vbase = g * kGroupVecs + lane;
                if (greedy) {
                    // smallest index attaining the max; NaN / +inf make the row invalid
                    float best = -INFINITY;
                    int bidx = INT_MAX;
                    int bad = 0;
#pragma unroll
                    for (int q = 0; q < kVecPerLane; ++q) {
                        float y[E];
                        const int vi = vbase + q * kWarp;
                        load_vec<DT>(buf, vi, nvec, y);
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            bad |= (y[e] != y[e]) || (y[e] == INFINITY);
                            if (y[e] > best) {
                                best = y[e];
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
                    float mx = -INFINITY;
#pragma unroll
                    for (int q = 0; q < kVecPerLane; ++q) {
                        const int vi = vbase + q * kWarp;
                        if (vi < nvec) mx = fmaxf(mx, vec_max<DT>(buf[vi]));
                    }
                    mx = warp_max(mx);
                    // integral reference exponent, so that rescaling groups is exact (ldexp);
                    // an all -inf group gets 0 (its sum is 0, or NaN if a NaN hides in it)
                    const float b = (mx == -INFINITY) ? 0.0f : floorf(mx * s_hi);
                    float acc = 0.0f;
#pragma unroll
                    for (int q = 0; q < kVecPerLane; ++q) {
                        float y[E];
                        load_vec<DT>(buf, vbase + q * kWarp, nvec, y);
#pragma unroll
                        for (int e = 0; e < E; ++e) acc += ex2(exp_arg(y[e], s_hi, s_lo, b));
                    }
                    acc = warp_sum(acc);
                    if (lane == 0) {
                        gref[r * P.groups_max + g] = b;
                        gsum[r * P.groups_max + g] = acc;
                    }
                }
            }
        }
    }
    if (warp == 0 && lane == 0) I.x = x_reg;
    __syncthreads();

    // ---- this CTA's record: per-row statistics (warp r), the logits at x (warp 2) ----
    if (warp < nrows) {
        const int r = warp;
        if (greedy) {
            float best = -INFINITY;
            int bidx = INT_MAX, bad = 0;
            for (int g = lane; g < groups; g += kWarp) {
                const float v = gref[r * P.groups_max + g];
                const int ix = __float_as_int(gsum[r * P.groups_max + g]);
                if (ix < 0) bad = 1;
                if (v > best || (v == best && ix < bidx)) {
                    best = v;
                    bidx = ix;
                }
            }
            const float wbest = warp_max(best);
            const int widx = warp_min_i32(best == wbest ? bidx : INT_MAX);
            const int wbad = __any_sync(0xffffffffu, bad);
            if (lane == 0) {
                mine1.gmax[r] = wbest;
                mine1.garg[r] = widx;
                mine1.bad[r] = wbad;
            }
        } else {
            float Bc = -INFINITY;
            int bad = 0;
            for (int g = lane; g < groups; g += kWarp) {
                const float sg = gsum[r * P.groups_max + g];
                if (!(sg >= 0.0f) || isinf(sg)) bad = 1;  // NaN or inf
                if (sg > 0.0f) Bc = fmaxf(Bc, gref[r * P.groups_max + g]);
            }
            Bc = warp_max(Bc);
            F2 acc = {0.0f, 0.0f};
            for (int g = lane; g < groups; g += kWarp) {
                const float sg = gsum[r * P.groups_max + g];
                if (sg > 0.0f && !isinf(sg)) acc = f2_add(acc, {scale2(sg, gref[r * P.groups_max + g] - Bc), 0.0f});
            }
            acc = warp_sum_f2(acc);
            const int wbad = __any_sync(0xffffffffu, bad);
            if (lane == 0) {
                mine1.B[r] = Bc;
                mine1.S_hi[r] = acc.hi;
                mine1.S_lo[r] = acc.lo;
                mine1.bad[r] = wbad;
            }
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

    // ---- combine the cluster (warp 0, lane c holds CTA c's record), decide the accept test ----
    if (warp == 0) {
        const bool in = lane < C;
        for (int r = 0; r < nrows; ++r) {
            if (greedy) {
                const float v = in ? xch1[lane].gmax[r] : -INFINITY;
                const int ix = in ? xch1[lane].garg[r] : INT_MAX;
                const int bad = in ? xch1[lane].bad[r] : 0;
                const float wv = warp_max(v);
                const int wix = warp_min_i32(v == wv ? ix : INT_MAX);
                const int wbad = __any_sync(0xffffffffu, bad);
                if (lane == 0) {
                    const int am = (wbad || wv == -INFINITY) ? -1 : wix;
                    if (r == 0) I.argmax_t = am;
                    else I.argmax_d = am;
                }
            } else {
                const F2 Sc = in ? F2{xch1[lane].S_hi[r], xch1[lane].S_lo[r]} : F2{0.0f, 0.0f};
                const float Bc = (in && Sc.hi > 0.0f) ? xch1[lane].B[r] : -INFINITY;
                const int bad = in ? xch1[lane].bad[r] : 0;
                const float Bw = warp_max(Bc);
                const F2 S = warp_sum_f2(Sc.hi > 0.0f ? f2_scale(Sc, Bc - Bw) : F2{0.0f, 0.0f});
                const int wbad = __any_sync(0xffffffffu, bad);
                if (lane == 0) {
                    if (r == 0) {
                        I.B_t = wbad ? NAN : Bw;
                        I.S_t = S;
                    } else {
                        I.B_d = wbad ? NAN : Bw;
                        I.S_d = S;
                    }
                }
            }
        }
        const unsigned xm = __ballot_sync(0xffffffffu, in && xch1[lane].has_x);
        const int xo = xm ? __ffs(xm) - 1 : 0;
        const float yx_t = __shfl_sync(0xffffffffu, in ? xch1[lane].yx[0] : 0.0f, xo);
        const float yx_d = __shfl_sync(0xffffffffu, in ? xch1[lane].yx[1] : 0.0f, xo);
        if (lane == 0) {
            int status = I.status | (timed_out ? REQ_TIMEOUT : 0);
            I.accept = 0;
            I.sample_kind = SAMPLE_NONE;
            I.rho = 0.0f;
            I.u_acc = u_acc_reg;
            I.u_s = u_s_reg;
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
                    I.inv_St = 1.0f / I.S_t.hi;
                    if (I.pair) {
                        // rho = p(x)/q(x) = 2^E * S_d/S_t with E = (y_t - y_d) s - (B_t - B_d):
                        // E in float64 (three operations), 2^E from the integer part and ex2 of
                        // the fraction with a first-order correction for its float rounding
                        const F2 lam = f2_div(I.S_t, I.S_d);
                        I.lam = lam;
                        float rho = 0.0f;
                        if (yx_t != -INFINITY) {
                            const double s64 = static_cast<double>(s_hi) + static_cast<double>(s_lo);
                            const double Ed = fma(static_cast<double>(yx_t) - static_cast<double>(yx_d), s64,
                                                  -(static_cast<double>(I.B_t) - static_cast<double>(I.B_d)));
                            const double n = floor(Ed);
                            const double fd = Ed - n;
                            const float f = static_cast<float>(fd);
                            const float flo = static_cast<float>(fd - static_cast<double>(f));
                            const float m = ex2(f) * fmaf(flo, 0.69314718f, 1.0f);
                            rho = scale2(m / lam.hi * (1.0f - lam.lo / lam.hi), static_cast<float>(fmax(fmin(n, 300.0), -300.0)));
                        }
                        I.rho = rho;
                        I.accept = (rho > 0.0f) && (I.u_acc <= static_cast<double>(rho));
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
            const float B_t = I.B_t, B_d = I.B_d, lam_hi = I.lam.hi, lam_lo = I.lam.lo;
            float acc_a = 0.0f;
            for (int g = warp; g < groups; g += kWarps) {
                float racc = 0.0f;
#pragma unroll
                for (int q = 0; q < kVecPerLane; ++q) {
                    const int vi = g * kGroupVecs + q * kWarp + lane;
                    float yt[E], yd[E];
                    load_vec<DT>(buf_t, vi, nvec, yt);
                    load_vec<DT>(buf_d, vi, nvec, yd);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const float et = ex2(exp_arg(yt[e], s_hi, s_lo, B_t));
                        const float ed = ex2(exp_arg(yd[e], s_hi, s_lo, B_d));
                        racc += fmaxf(fmaf(-lam_lo, ed, fmaf(-lam_hi, ed, et)), 0.0f);
                        acc_a += fminf(et, lam_hi * ed);  // S_t * min(p, q), no cancellation
                    }
                }
                racc = warp_sum(racc);
                if (lane == 0) gres[g] = racc;
            }
            my_alpha = acc_a * I.inv_St;
        } else {
            const float c_t = I.c_t, c_d = I.c_d;
            for (int g = warp; g < groups; g += kWarps) {
#pragma unroll
                for (int q = 0; q < kVecPerLane; ++q) {
                    const int vi = g * kGroupVecs + q * kWarp + lane;
                    if (vi >= nvec) continue;
                    float yt[E], yd[E];
                    Elt<DT>::unpack(buf_t[vi], yt);
                    Elt<DT>::unpack(buf_d[vi], yd);
#pragma unroll
                    for (int e = 0; e < E; ++e)
                        my_alpha += ex2(fminf(fmaf(yt[e], s_hi, -c_t), fmaf(yd[e], s_hi, -c_d)));
                }
            }
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

    // ---- cluster totals, the owner of the draw, item results ----
    if (warp == 0) {
        const bool in = lane < C;
        const float a = in ? xch2[lane].alpha : 0.0f;
        const F2 z = in ? F2{xch2[lane].Z_hi, xch2[lane].Z_lo} : F2{0.0f, 0.0f};
        F2 wp = {0.0f, 0.0f};
        if (in && I.sample_kind != SAMPLE_NONE && !greedy) {
            const F2 Sc = {xch1[lane].S_hi[0], xch1[lane].S_lo[0]};
            if (Sc.hi > 0.0f) wp = f2_scale(Sc, xch1[lane].B[0] - I.B_t);
        }
        const float alpha_sum = warp_sum(a);
        int kind = I.sample_kind;
        const F2 Zres = warp_sum_f2(z);
        int fb = 0;
        if (kind == SAMPLE_RESIDUAL && !(Zres.hi > 0.0f)) {
            kind = SAMPLE_P;  // zero residual mass: draw from p and say so
            fb = 1;
        }
        // masses of the law the draw uses, per CTA, accumulated in CTA order
        const double mine = (kind == SAMPLE_RESIDUAL) ? f2_d(z) : f2_d(wp);
        const double incl = warp_inclusive_scan_f64(in ? mine : 0.0, lane);
        const double Ztot = __shfl_sync(0xffffffffu, incl, C - 1);
        const double t = I.u_s * Ztot;
        const unsigned hit = __ballot_sync(0xffffffffu, in && mine > 0.0 && incl > t);
        const unsigned posm = __ballot_sync(0xffffffffu, in && mine > 0.0);
        int owner = -1;
        if (kind != SAMPLE_NONE && I.status == 0 && !greedy)
            owner = hit ? __ffs(hit) - 1 : (posm ? 31 - __clz(static_cast<int>(posm)) : -1);
        const double prefix = __shfl_sync(0xffffffffu, incl - mine, owner < 0 ? 0 : owner);
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
                                                   ? static_cast<float>(f2_d(Zres) / f2_d(I.S_t))
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
        const double local = I.target_t - I.owner_prefix;
        int gsel = -1, last_g = -1;
        double before = 0.0, last_before = 0.0, run = 0.0;
        for (int base = 0; base < groups; base += kWarp) {
            const int g = base + lane;
            double m = 0.0;
            if (g < groups) {
                if (kind == SAMPLE_RESIDUAL) {
                    m = static_cast<double>(gres[g]);
                } else {
                    const float sg = gsum[g];
                    m = (sg > 0.0f) ? static_cast<double>(scale2(sg, gref[g] - I.B_t)) : 0.0;
                }
            }
            const double incl = run + warp_inclusive_scan_f64(m, lane);
            const unsigned hit = __ballot_sync(0xffffffffu, g < groups && m > 0.0 && incl > local);
            const unsigned posm = __ballot_sync(0xffffffffu, g < groups && m > 0.0);
            if (hit) {
                const int l = __ffs(hit) - 1;
                gsel = base + l;
                before = __shfl_sync(0xffffffffu, incl - m, l);
                break;
            }
            if (posm) {
                const int l = 31 - __clz(static_cast<int>(posm));
                last_g = base + l;
                last_before = __shfl_sync(0xffffffffu, incl - m, l);
            }
            run = __shfl_sync(0xffffffffu, incl, kWarp - 1);
        }
        const bool clamped = gsel < 0;  // rounding put u*Z past the last group with mass
        if (clamped) {
            gsel = last_g;
            before = last_before;
        }
        int tok = -1;
        double wsel = 0.0, margin = 0.0, unit = 1.0;
        if (gsel >= 0) {
            const float bg = (kind == SAMPLE_RESIDUAL) ? 0.0f : gref[gsel];
            // group units: residual weights are already in cluster units; P weights are in
            // units of 2^b_g, 2^(b_g - B_t) cluster units each (exact power of two)
            unit = (kind == SAMPLE_RESIDUAL) ? 1.0 : static_cast<double>(scale2(1.0f, bg - I.B_t));
            const float lt = static_cast<float>((local - before) / unit);  // target inside the group
            float run2 = 0.0f;
            int last_tok = -1;
            float last_w = 0.0f;
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
                const float start = incl - ls;
                // this lane's element that takes the target, if any; and its last with mass
                int found = -1, lastp = -1;
                float fprev = 0.0f, c = start, wf = 0.0f, wl = 0.0f;
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
                    const float ws = __shfl_sync(0xffffffffu, wf, l);
                    wsel = ws;
                    tok = (I.lo + gsel * kGroupVecs + q * kWarp + l) * E + e_sel;
                    margin = fmin(static_cast<double>(lt - c0), static_cast<double>(c0 + ws - lt)) * unit / I.Ztot;
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
                margin = 0.0;
            }
        }
        if (lane == 0) {
            P.item_tok[item] = tok;
            P.item_prob[item] = tok >= 0 ? static_cast<float>(wsel * unit / I.Ztot) : NAN;
            P.item_margin[item] = tok >= 0 ? static_cast<float>(margin) : NAN;
        }
    }
    if (timed_out) {
        // a copy did not land in time: wait (bounded) once more so none is left in flight
        for (int r = 0; r < nrows; ++r)
            for (int k = 0; k < nchunk; ++k) mbar_wait_bounded(&bars[r][k], 0, kWaitLimitNs);
    }
}

// ------------------------------------------------------------------------------------------
// Per-request selection: the first rejection, the emitted tokens, stopping, alpha reduction.

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
};

constexpr int kFinThreads = 1024;

__global__ void __launch_bounds__(kFinThreads) spec_select_kernel(const FinParams P) {
    __shared__ double red_a[kFinThreads / kWarp];
    __shared__ int red_n[kFinThreads / kWarp];
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    // the offsets must start at 0, end at total_rows and grow by at least one row per request;
    // otherwise every request is BAD_SHAPE and nothing is read through them
    int bad_off = (__ldg(P.row_off) != 0) || (__ldg(P.row_off + P.B) != P.total_rows);
    for (int i = threadIdx.x; i < P.B && !bad_off; i += kFinThreads)
        if (__ldg(P.row_off + i + 1) <= __ldg(P.row_off + i)) bad_off = 1;
    const bool global_ok = !__syncthreads_or(bad_off);
    double asum = 0.0;
    int acnt = 0;
    for (int i = warp; i < P.B; i += kFinThreads / kWarp) {
        const int r0 = __ldg(P.row_off + i), r1 = __ldg(P.row_off + i + 1);
        const int K = r1 - r0 - 1;
        const int d0 = r0 - i;
        int status = 0;
        if (!global_ok || K < 0 || K > P.K_max || r0 < 0 || r1 > P.total_rows || d0 < 0) status |= SPEC_REQ_BAD_SHAPE;
        int st_items = 0;
        if (!status) {
            for (int j = lane; j <= K; j += kWarp) st_items |= P.item_status[r0 + j];
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
        // A = index of the first rejected position (K when all are accepted): ballots over
        // the accept flags, in position order
        int A = K;
        for (int base = 0; base < K; base += kWarp) {
            const int j = base + lane;
            const unsigned rej = __ballot_sync(0xffffffffu, j < K && P.item_flag[r0 + j] == 0);
            if (rej) {
                A = base + __ffs(rej) - 1;
                break;
            }
        }
        int n = A + 1;
        if (P.max_new) n = min(n, max(__ldg(P.max_new + i), 0));
        const int stop = P.stop_token ? __ldg(P.stop_token + i) : -1;
        const int frontier = P.item_tok[r0 + A];
        if (stop >= 0) {
            for (int base = 0; base < n; base += kWarp) {
                const int j = base + lane;
                int tok = -1;
                if (j < n) tok = (j < A) ? __ldg(P.draft_tokens + d0 + j) : frontier;
                const unsigned hit = __ballot_sync(0xffffffffu, j < n && tok == stop);
                if (hit) {
                    n = base + __ffs(hit);
                    break;
                }
            }
        }
        for (int j = lane; j <= K; j += kWarp) {
            int tok = -1;
            if (j < n) tok = (j < A) ? __ldg(P.draft_tokens + d0 + j) : frontier;
            P.out_tokens[r0 + j] = tok;
        }
        for (int j = lane; j < K; j += kWarp) asum += static_cast<double>(P.alpha_ws[d0 + j]);
        if (lane == 0) {
            acnt += K;
            P.req_status[i] = 0;
            P.accept_len[i] = A;
            if (P.n_emitted) P.n_emitted[i] = n;
            if (P.frontier_prob) P.frontier_prob[i] = P.item_prob[r0 + A];
            if (P.frontier_margin) P.frontier_margin[i] = P.item_margin[r0 + A];
            if (P.fallback) P.fallback[i] = P.item_fb[r0 + A];
        }
    }
    asum = warp_sum_f64(asum);
    if (lane == 0) {
        red_a[warp] = asum;
        red_n[warp] = acnt;
    }
    __syncthreads();
    if (warp == 0) {
        double a = red_a[lane];
        int c = red_n[lane];
        a = warp_sum_f64(a);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0) {
            if (P.alpha_sum) *P.alpha_sum = a;
            if (P.alpha_count) *P.alpha_count = c;
        }
    }
}

// ------------------------------------------------------------------------------------------
// Host side

struct WsLayout {
    size_t flag, tok, status, fb, prob, margin, alpha, total;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static WsLayout ws_layout(int32_t B, int32_t total_rows) {
    WsLayout L;
    const size_t T = static_cast<size_t>(total_rows > 0 ? total_rows : 0);
    const size_t nd = total_rows > B ? static_cast<size_t>(total_rows - B) : 0;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.flag = take(T * 4);
    L.tok = take(T * 4);
    L.status = take(T * 4);
    L.fb = take(T * 4);
    L.prob = take(T * 4);
    L.margin = take(T * 4);
    L.alpha = take((nd > 0 ? nd : 1) * 4);
    L.total = off;
    return L;
}

struct LaunchShape {
    int C = 0;
    int slice_vecs_max = 0;
    int groups_max = 0;
    size_t smem = 0;
};

static size_t rows_smem_bytes(int slice_vecs_max, int groups_max) {
    return static_cast<size_t>(2) * slice_vecs_max * 16 + static_cast<size_t>(5) * groups_max * 4;
}

template <int DT>
static cudaError_t pick_shape(int nvec_row, LaunchShape &out) {
    static std::mutex mu;
    static int cached_dev = -1, cached_nvec = -1;
    static LaunchShape cached;
    static size_t smem_set = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev == cached_dev && nvec_row == cached_nvec) {
        out = cached;
        return cudaSuccess;
    }
    int max_optin = 0;
    e = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    static bool nonportable_set = false;
    if (!nonportable_set) {
        e = cudaFuncSetAttribute(spec_rows_kernel<DT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        nonportable_set = true;
    }
    // the smallest cluster whose slices fit six CTAs per SM, else three, two, one
    const size_t budgets[4] = {36 * 1024, 72 * 1024, 110 * 1024, static_cast<size_t>(max_optin) - 4096};
    for (size_t budget : budgets) {
        for (int C = 1; C <= kMaxCluster; C *= 2) {
            if (C > nvec_row) break;
            LaunchShape s;
            s.C = C;
            s.slice_vecs_max = (nvec_row + C - 1) / C;
            s.groups_max = (s.slice_vecs_max + kGroupVecs - 1) / kGroupVecs;
            s.smem = rows_smem_bytes(s.slice_vecs_max, s.groups_max);
            if (s.smem > budget) continue;
            if (s.smem > smem_set) {
                e = cudaFuncSetAttribute(spec_rows_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(s.smem));
                if (e != cudaSuccess) return e;
                smem_set = s.smem;
            }
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = C;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(C * 16, 1, 1);
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = s.smem;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int nclusters = 0;
            e = cudaOccupancyMaxActiveClusters(&nclusters, spec_rows_kernel<DT>, &cfg);
            if (e != cudaSuccess) {
                cudaGetLastError();
                continue;
            }
            if (nclusters <= 0) continue;
            cached_dev = dev;
            cached_nvec = nvec_row;
            cached = s;
            out = s;
            return cudaSuccess;
        }
    }
    return cudaErrorInvalidConfiguration;
}

template <int DT>
static spec_status launch_rows(const RowsParams &P, cudaStream_t stream) {
    LaunchShape s;
    if (pick_shape<DT>(P.nvec_row, s) != cudaSuccess) return SPEC_ERR_UNSUPPORTED;
    RowsParams Q = P;
    Q.slice_vecs_max = s.slice_vecs_max;
    Q.groups_max = s.groups_max;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = s.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(P.total_rows) * s.C, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = s.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, spec_rows_kernel<DT>, Q) != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

}  // namespace spec

using namespace spec;

extern "C" size_t spec_verify_workspace_size(int32_t B, int32_t V, int32_t total_rows, spec_dtype dtype) {
    (void)V;
    (void)dtype;
    return ws_layout(B, total_rows).total;
}

extern "C" spec_status spec_verify(const spec_verify_args *a, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 1 || a->V < 1 || a->K_max < 0 || a->K_max > 64 || a->total_rows < a->B) return SPEC_ERR_INVALID_ARG;
    if (static_cast<int64_t>(a->total_rows) > static_cast<int64_t>(a->B) * (a->K_max + 1)) return SPEC_ERR_INVALID_ARG;
    if (a->dtype != SPEC_F32 && a->dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (!a->target_logits || !a->row_off || !a->uniforms || !a->accept_len || !a->out_tokens || !a->req_status)
        return SPEC_ERR_INVALID_ARG;
    const bool has_drafts = a->total_rows > a->B;
    if (has_drafts && (!a->draft_logits || !a->draft_tokens)) return SPEC_ERR_INVALID_ARG;
    const size_t eb = (a->dtype == SPEC_BF16) ? 2 : 4;
    const size_t row_bytes = eb * static_cast<size_t>(a->V);
    if (row_bytes % 16 != 0) return SPEC_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(a->target_logits) % 16 != 0) return SPEC_ERR_UNSUPPORTED;
    if (has_drafts && reinterpret_cast<uintptr_t>(a->draft_logits) % 16 != 0) return SPEC_ERR_UNSUPPORTED;
    if (row_bytes / 16 > static_cast<size_t>(INT_MAX)) return SPEC_ERR_UNSUPPORTED;
    if (!a->temperature && !(a->temperature_scalar >= 0.0f && std::isfinite(a->temperature_scalar)))
        return SPEC_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(a->B, a->total_rows);
    if (!workspace || workspace_bytes < L.total || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return SPEC_ERR_WORKSPACE;

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    RowsParams P = {};
    P.target = a->target_logits;
    P.draft = a->draft_logits;
    P.row_off = a->row_off;
    P.draft_tokens = a->draft_tokens;
    P.uniforms = a->uniforms;
    P.temperature = a->temperature;
    P.temperature_scalar = a->temperature_scalar;
    P.B = a->B;
    P.V = a->V;
    P.K_max = a->K_max;
    P.total_rows = a->total_rows;
    P.nvec_row = static_cast<int32_t>(row_bytes / 16);
    P.item_flag = reinterpret_cast<int32_t *>(ws + L.flag);
    P.item_tok = reinterpret_cast<int32_t *>(ws + L.tok);
    P.item_status = reinterpret_cast<int32_t *>(ws + L.status);
    P.item_fb = reinterpret_cast<int32_t *>(ws + L.fb);
    P.item_prob = reinterpret_cast<float *>(ws + L.prob);
    P.item_margin = reinterpret_cast<float *>(ws + L.margin);
    P.alpha_ws = reinterpret_cast<float *>(ws + L.alpha);
    P.alpha_rows = a->alpha_rows;
    P.rho_rows = a->rho_rows;
    P.resid_rows = a->resid_rows;

    if (a->rows_event_begin && cudaEventRecord(a->rows_event_begin, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    const spec_status st = (a->dtype == SPEC_BF16) ? launch_rows<SPEC_BF16>(P, stream) : launch_rows<SPEC_F32>(P, stream);
    if (st != SPEC_OK) return st;
    if (a->rows_event_end && cudaEventRecord(a->rows_event_end, stream) != cudaSuccess) return SPEC_ERR_CUDA;

    FinParams F = {};
    F.row_off = a->row_off;
    F.draft_tokens = a->draft_tokens;
    F.stop_token = a->stop_token;
    F.max_new = a->max_new;
    F.B = a->B;
    F.K_max = a->K_max;
    F.total_rows = a->total_rows;
    F.item_flag = P.item_flag;
    F.item_tok = P.item_tok;
    F.item_status = P.item_status;
    F.item_fb = P.item_fb;
    F.item_prob = P.item_prob;
    F.item_margin = P.item_margin;
    F.alpha_ws = P.alpha_ws;
    F.accept_len = a->accept_len;
    F.n_emitted = a->n_emitted;
    F.out_tokens = a->out_tokens;
    F.req_status = a->req_status;
    F.fallback = a->fallback;
    F.alpha_count = a->alpha_count;
    F.frontier_prob = a->frontier_prob;
    F.frontier_margin = a->frontier_margin;
    F.alpha_sum = a->alpha_sum;
    spec_select_kernel<<<1, kFinThreads, 0, stream>>>(F);
    if (cudaGetLastError() != cudaSuccess) return SPEC_ERR_CUDA;
    return SPEC_OK;
}

extern "C" const char *spec_version(void) { return "spec-verify-gb300 0.1 (sm_103a)"; }

// ------------------------------------------------------------------------------------------
// spec_verify_noalloc: spec_verify for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they verify a round: a serving
// engine whose memory planner has already reserved every byte of the device, a plugin that
// runs inside another runtime's allocator or scheduler callbacks, or a latency-critical loop
// where an allocation's implicit synchronisation and possible failure are not acceptable.
// For them this entry point takes its workspace from a fixed array in the library's own
// device memory instead of from the caller.
//
// The array lives in every GPU that loads the library until the process exits. Its address
// is looked up once per device, on the first call made with that device current; make that
// first call before any stream capture. All calls share the one array and it keeps the last
// call's contents (the kernels write every workspace entry before reading it, so nothing
// needs clearing); calls that overlap on the GPU, on two streams or from two threads, race
// on it and must be serialised by the caller.

namespace spec {
constexpr int32_t kNoallocMaxRows = 16384;  // target rows per call: T = sum_i (K_i + 1)
constexpr size_t kNoallocScratchBytes = 7 * 65536;  // = workspace of kNoallocMaxRows rows
static __device__ __align__(256) unsigned char noalloc_scratch[kNoallocScratchBytes];

static std::mutex noalloc_mu;
static void *noalloc_ptr[64] = {nullptr};
}  // namespace spec

extern "C" spec_status spec_verify_noalloc(const spec_verify_args *a, cudaStream_t stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->total_rows > kNoallocMaxRows) return SPEC_ERR_UNSUPPORTED;  // beyond the fixed scratch
    const size_t need = ws_layout(a->B, a->total_rows).total;
    if (need > kNoallocScratchBytes) return SPEC_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
    void *ptr = nullptr;
    {
        std::lock_guard<std::mutex> lock(noalloc_mu);
        if (!noalloc_ptr[dev]) {
            // host code must not use the array's name as a device address: ask the runtime
            if (cudaGetSymbolAddress(&noalloc_ptr[dev], noalloc_scratch) != cudaSuccess) {
                noalloc_ptr[dev] = nullptr;
                return SPEC_ERR_CUDA;
            }
        }
        ptr = noalloc_ptr[dev];
    }
    return spec_verify(a, ptr, kNoallocScratchBytes, stream);
}
