// The per-position kernel of spec_verify (included once, by spec_verify.cu).
//
// The rule is that of "SOTA-227: Decode with a draft model and an accept-reject rule" ("What to
// do", steps 3-4) and SDCP Rules 1 and 2 ("Acceptance Rules"): accept x_j when u_j <= p_j(x_j) /
// q_j(x_j); at the first rejection draw from max(p_j - q_j, 0) normalised; with all accepted draw
// from p_{K+1}; with T = 0, the greedy rule.
//
// Work unit: one target row ("item"). Position j < K_i of request i is a pair (target row j,
// draft row j); position K_i is the target-only row of the bonus (or plain) draw.
//
// A persistent thread-block cluster of C CTAs (two CTAs per SM) walks a list of items. CTA c
// owns the c-th 16-byte-aligned slice of the vocabulary of every row. Each CTA has 15 data warps
// and one control warp.
//   pass 1 (data warps): the item's rows arrive in a ring of shared-memory slots by 1-D bulk
//           copies (issued by whichever data warp releases a slot last), the target row moves
//           into registers (its slot refills at once), and each thread sums 2^(y*s - b) with an
//           integral reference b of its own, so that combining threads, warps and CTAs is exact
//           scaling by powers of two;
//   exchange (control warp): the CTA's record (row statistics, the logits at the draft token, the
//           alpha / residual totals of the previous item) goes into every CTA's shared memory with
//           asynchronous stores completing on that CTA's barrier; every CTA then computes the
//           accept test identically;
//   pass 2 (data warps, pairs): from the same registers and slot: alpha = sum min(p, q) and, only
//           where the position rejects, the residual max(p - q, 0) per chunk (32 vectors);
//   draw (control warp): once an exchange has brought every CTA's residual (or p) mass, the CTA
//           whose slice holds u*Z fetches the one chunk that holds it and finds the token there.
// The roles meet at mbarriers keyed by item (statistics ready, decision ready): the control warp
// finishes an item (its results and draw) while the data warps run the next one.
// Every rejecting position prepares its own candidate (the first rejection is known only per
// request); the selection kernel picks. Float math is packed two lanes per instruction; no
// float64 instruction runs on the device (it is very slow on this part).
#pragma once

#include <climits>
#include <cmath>
#include <cstdint>

#include "spec_device.cuh"
#include "spec_math.cuh"
#include "spec_verify.h"

namespace spec {

// 15 data warps and one control warp (512 threads, 64 registers each), two CTAs per SM: each SM
// works on two items of two clusters at once, so that one CTA's exchange and decision latency
// hides behind the other's exponentials
constexpr int kWarps = 15;                   // data warps
constexpr int kThreads = kWarps * kWarp;     // data threads
constexpr int kBlock = kThreads + kWarp;     // plus the control warp
// named barrier (0 is __syncthreads): a batch's descriptors are loaded (all 512 threads)
enum : int { BAR_BATCH = 1 };
constexpr int kChunkVecs = kWarp;   // a chunk: 32 contiguous vectors, one per lane of a warp
constexpr int kRing = 3;            // row slots per CTA
constexpr int kMaxItems = 22;       // item descriptors held at once (one batch)
constexpr int kRoffMax = 520;       // row offsets staged in shared memory (B <= 519)
constexpr int kMaxCluster = 16;
constexpr int kMaxNvt = 5;          // 16-byte vectors per thread per row
constexpr int kMaxStreamRows = 10;  // streaming kernel: 480-vector rows of chunks per row slice
constexpr int kMaxChunks = (kMaxNvt > kMaxStreamRows ? kMaxNvt : kMaxStreamRows) * kWarps;
constexpr uint32_t kSuspendNs = 1u << 20;  // one suspended wait: at most ~1 ms
constexpr int kMaxWaitTries = 2048;        // ~2 s in all: a copy never takes this long
// log2(e) as a float pair
constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963e-08f;

enum : int32_t { REQ_TIMEOUT = 32 };  // internal: a bulk copy did not complete in time

// The pipeline. kLag = 0: an item's rows stay on chip from pass 1 to pass 2 (the target row in
// registers, the draft row in its ring slot), and the data warps wait for the item's decision
// between the passes while the other CTA on the SM computes. kLag > 0: pass 2 of item g runs
// after pass 1 of item g + kLag, so that the exchange and the decision overlap other items'
// passes; the rows of item g are read again (from L2, where pass 1's copies left them). The
// control warp decides item g, signals it, and only then finishes an earlier item (its results
// and draw). Ring depths of the per-item buffers follow from how far apart the roles may run:
constexpr int kLag = 0;
// The streaming kernel (spec_stream_kernel.cuh) runs pass 2 one item late; the depths below
// cover both kernels.
constexpr int kStreamLag = 1;
constexpr int kDepthLag = kLag > kStreamLag ? kLag : kStreamLag;
constexpr int kWS = kDepthLag + 2;       // pass-1 statistics (read by the item's exchange)
constexpr int kPM = 2 * kDepthLag + 4;   // bonus-row chunk sums (read by the draw, lag + 1 items later)
constexpr int kRM = kDepthLag + 3;       // pass-2 residual chunk sums and alpha partials
constexpr int kND = kDepthLag + 3;       // decisions (read by pass 2, the results and the draw)
constexpr int kNMS = kDepthLag + 3;      // exchange slots (a record is read again lag + 1 exchanges later)
constexpr int kSB = kDepthLag + 2;       // barriers: pass-1 statistics ready
constexpr int kPB = kDepthLag + 3;       // barriers: pass 2 done (lagged pipelines)

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
    int32_t nclusters;       // persistent clusters in the grid
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
    // top-k / top-p (each may be NULL): the cut of each target row, and the per-request top_p
    // (read only to flag a NaN as a bad parameter)
    const int2 *trunc;
    const float *top_p;
};

// One item of this cluster's list, prepared before its rows arrive.
struct Desc {
    int32_t item, req, pos, K, drow, pair, status, x;
    float s_hi, s_lo;  // log2(e)/T = s_hi + s_lo, s_hi rounded toward zero (s_lo > 0)
    int32_t greedy;
    F2 u_acc, u_s;     // the position's accept draw and the request's frontier draw
    uint32_t cut_tau;  // top-k / top-p cut of the target row (see cut_keeps); trunc = 0: none
    int32_t cut_id, trunc;
};

// Reference exponent of a row (or slice) with no mass.
constexpr int32_t kNoRef = -(1 << 30);
// Record flags: this CTA holds the draft token; a bulk copy timed out; q(x) = 0; p(x) = 0.
enum : int32_t { XF_HAS = 1, XF_TMO = 2, XF_QZERO = 4, XF_PZERO = 8 };

// A CTA's record for item k, stored into exchange slot k % kNMS of every CTA of the cluster
// (distributed shared memory, asynchronous stores that complete bytes on that CTA's barrier of
// the slot). Twelve 32-bit words, 16-byte aligned: three vector stores per destination. Sums are
// plain floats: a record adds a handful of roundings to sums of thousands of terms.
struct __align__(16) Msg {
    int32_t a[2];  // Rule 2: integral reference exponent B_r of row r (kNoRef: no mass);
                   // Rule 1: smallest index attaining the max (-1: the row holds a NaN / +inf)
    float b[2];    // Rule 2: sum S_r of 2^(y*s - B_r) (NaN: the row holds a NaN / +inf);
                   // Rule 1: max logit (+inf with a = -1: invalid row)
    float E_hi, E_lo;  // (y_t - y_d) s at the draft token, a float pair (from the CTA holding it)
    int32_t flags;     // XF_* bits
    int32_t pad0;
    float prev_alpha;  // the previous item: this slice's share of alpha (normalised)
    float prev_Z;      // the previous item: this slice's residual mass (units 2^B_t)
    int32_t pad1, pad2;
};
constexpr int kMsgBytes = sizeof(Msg);
static_assert(kMsgBytes == 48, "a record is three 16-byte vectors");

// The decision of an item, kept until its draw is finished (one item later).
struct Decision {
    int32_t item, drow, pair, greedy, status, accept, kind, valid;
    float B_t, B_d, s_hi, s_lo, rho, inv_St;
    float c_t, c_d, c_tf, c_df;  // log2 of each row's normaliser: integral part, fraction
    float S_t, S_d;  // each row's sum of 2^(y*s - B) over the whole vocabulary
    F2 lam, u_s;
    int32_t argmax_t;
    float alpha_g;  // greedy rule: alpha of the two point masses
    uint32_t cut_tau;  // the target row's top-k / top-p cut (trunc = 0: none)
    int32_t cut_id, trunc;
};

enum { SAMPLE_NONE = 0, SAMPLE_RESIDUAL = 1, SAMPLE_P = 2 };

// Per-warp statistics of both rows after pass 1, in the record's encoding (a[r], b[r] as in
// Msg), 16 bytes so that one vector load reads a warp's entry.
struct __align__(16) WarpStat {
    int32_t a[2];
    float b[2];
};

// 2^d for an integer d <= 0 with integer operations only (0 below the normal range).
__device__ __forceinline__ float pow2_int(int d) { return d < -126 ? 0.0f : __int_as_float((d + 127) << 23); }

// Lane l < C stores this CTA's record (three vectors in registers, the same in every lane) into
// slot `rank` of CTA l, each asynchronous store completing its bytes on CTA l's barrier.
__device__ __forceinline__ void push_record(const uint4 (&rec)[3], Msg *slot_base, uint64_t *bar, int rank, int C,
                                            int lane) {
    if (lane < C) {
        const uint32_t dst = dsmem_map(slot_base + rank, lane);
        const uint32_t rbar = dsmem_map(bar, lane);
#pragma unroll
        for (int q = 0; q < 3; ++q) st_async_v4(dst + 16 * q, rec[q], rbar);
    }
}

// Top-k / top-p: the logits of one 16-byte vector of a target row (vector `vi` of the row)
// that the row's cut removes become -inf, which turns every later sum, ratio and draw into
// those of the truncated, renormalised law.
template <int DT>
__device__ __forceinline__ void mask_cut(uint4 &w, int vi, uint32_t tau, int id) {
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

}  // namespace spec
