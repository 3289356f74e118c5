// The per-position kernel of spec_verify (included once, by spec_verify.cu).
//
// The rule is that of "SOTA-227: Decode with a draft model and an accept-reject rule" ("What to
// do", steps 3-4) and SDCP Rules 1 and 2 ("Acceptance Rules"): accept x_j when u_j <= p_j(x_j) /
// q_j(x_j); at the first rejection draw from max(p_j - q_j, 0) normalised; with all accepted draw
// from p_{K+1}; with T = 0, the greedy rule.
//
// Work unit: one target row ("item"). Position j < K_i of request i is a pair (target row j,
// draft row j); position K_i is the target-only row of the bonus (or plain) draw. One thread-block
// cluster of C CTAs verifies an item; CTA c owns the c-th 16-byte-aligned slice of the vocabulary
// of both rows and stages it in shared memory with 1-D bulk copies, so every logit crosses HBM
// exactly once:
//   pass 1 (as the copies land): per 1024-token group, max and sum of 2^(y*s - b) with an
//           integral reference b, so that combining groups and CTAs is exact scaling by 2^k;
//   exchange #1: each CTA writes its row statistics into every CTA's shared memory (DSMEM),
//           then one cluster barrier; the accept test is computed identically everywhere;
//   pass 2 (pairs, from shared memory): alpha = sum min(p, q), and only where this position
//           rejects, the residual max(p - q, 0) with per-group sums;
//   exchange #2: alpha and residual shares, then the CTA whose slice holds u*Z draws.
// Every rejecting position prepares its own candidate (the first rejection is known only per
// request); the selection kernel picks. Float math is packed two lanes per instruction.
#pragma once

#include <climits>
#include <cmath>
#include <cstdint>

#include "spec_device.cuh"
#include "spec_math.cuh"
#include "spec_verify.h"

namespace spec {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / kWarp;
constexpr int kVecPerLane = 4;                   // 16-byte vectors per lane in one group
constexpr int kGroupVecs = kWarp * kVecPerLane;  // 128 vectors = 2 KiB per row per group
constexpr int kMaxChunks = 4;                    // bulk copies per row slice
constexpr int kMaxCluster = 16;
constexpr uint32_t kSuspendNs = 1u << 20;        // one suspended wait: at most ~1 ms
constexpr int kMaxWaitTries = 2048;              // ~2 s in all: a copy never takes this long
// log2(e) as a float pair
constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963e-08f;

enum : int32_t { REQ_TIMEOUT = 32 };  // internal: a bulk copy did not complete in time

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

// A CTA's record after pass 1. It is written into slot `rank` of every CTA of the cluster, so
// that after the cluster barrier all reads are local. Fields are 32-bit words.
struct Ex1 {
    float B[2];      // integral reference exponent of S[r] (-inf: no mass)
    float S_hi[2];   // sum over the slice of 2^(y*s - B[r]), a float pair
    float S_lo[2];
    int32_t bad[2];  // a NaN / +inf was seen in row r's slice
    float yx[2];     // target / draft logit at the draft token, from the CTA that holds it
    int32_t has_x;
    float gmax[2];   // greedy rule: max logit of the slice and the smallest index attaining it
    int32_t garg[2];
};
constexpr int kEx1Words = sizeof(Ex1) / 4;
// A CTA's record after pass 2.
struct Ex2 {
    float alpha;  // this slice's share of alpha (normalised)
    float Z_hi;   // this slice's residual mass, units of 2^B_t (a float pair)
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
    F2 u_acc, u_s;     // the position's accept draw and the request's frontier draw
    float s_hi, s_lo;  // log2(e)/T = s_hi + s_lo, s_hi rounded toward zero (s_lo > 0)
    float B_t, B_d;    // cluster-wide integral reference exponents
    F2 S_t, S_d;       // cluster-wide sums in those units
    float c_t, c_d;    // B + log2 S, for the alpha-only pass
    F2 lam;            // S_t / S_d
    float rho, alpha, inv_St;
    F2 target_t, owner_prefix, Ztot;
    int32_t argmax_t, argmax_d;
};

enum { SAMPLE_NONE = 0, SAMPLE_RESIDUAL = 1, SAMPLE_P = 2 };

__device__ __forceinline__ void chunk_range(int groups, int nchunk, int k, int nvec, int &g0, int &g1, int &v0,
                                            int &v1) {
    g0 = (groups * k) / nchunk;
    g1 = (groups * (k + 1)) / nchunk;
    v0 = g0 * kGroupVecs;
    v1 = min(g1 * kGroupVecs, nvec);
}

// Lane l < C copies `words` 32-bit words of the local record into slot `rank` of CTA l.
__device__ __forceinline__ void push_record(const void *mine, void *slot_base, int rank, int words, int C, int lane) {
    if (lane < C) {
        const uint32_t *src = static_cast<const uint32_t *>(mine);
        const uint32_t dst = dsmem_map(static_cast<uint32_t *>(slot_base) + rank * words, lane);
        for (int w = 0; w < words; ++w) st_cluster_u32(dst + 4 * w, src[w]);
    }
}

// Weights of this lane's elements of vector vi in the law the candidate is drawn from:
// RESIDUAL: max(e_t - lambda*e_d, 0) = S_t * max(p - q, 0) in units of 2^B_t;
// P: 2^(y*s - b_g), the pass-1 terms of the group (units of 2^b_g).
// Same operations, in the same order, as passes 1 and 2: the values are bitwise those summed.
template <int DT>
__device__ __forceinline__ void vec_weights(int kind, const uint4 *buf_t, const uint4 *buf_d, int vi, int nvec,
                                            const ItemInfo &I, float bg, float *w) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    const float2 shi = f2splat(I.s_hi), slo = f2splat(I.s_lo);
    float2 yt[H];
    load_vec2<DT>(buf_t, vi, nvec, yt);
    if (kind == SAMPLE_RESIDUAL) {
        float2 yd[H];
        load_vec2<DT>(buf_d, vi, nvec, yd);
        const float2 nbt = f2splat(-I.B_t), nbd = f2splat(-I.B_d);
        const float2 nlh = f2splat(-I.lam.hi), nll = f2splat(-I.lam.lo);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float2 et = ex2x2(exp_arg2(yt[h], shi, slo, nbt));
            const float2 ed = ex2x2(exp_arg2(yd[h], shi, slo, nbd));
            const float2 r = __ffma2_rn(ed, nll, __ffma2_rn(ed, nlh, et));
            w[2 * h] = fmaxf(r.x, 0.0f);
            w[2 * h + 1] = fmaxf(r.y, 0.0f);
        }
    } else {
        const float2 nb = f2splat(-bg);
#pragma unroll
        for (int h = 0; h < H; ++h) {
            const float2 e = ex2x2(exp_arg2(yt[h], shi, slo, nb));
            w[2 * h] = e.x;
            w[2 * h + 1] = e.y;
        }
    }
}

}  // namespace spec
