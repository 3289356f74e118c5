// spec_slice_kernel: the per-position kernel of spec_verify, with the round's selection, and for
// spec_verify_round its compaction and gamma choice, in one launch (included once, by
// spec_verify.cu).
//
// The rule is that of "SOTA-227: Decode with a draft model and an accept-reject rule" ("What to
// do", steps 3-4) and SDCP Rules 1 and 2 ("Acceptance Rules"): accept x_j when u_j <= p_j(x_j) /
// q_j(x_j); at the first rejection draw from max(p_j - q_j, 0) normalised; with every draft
// accepted draw from p_{K+1}; with T = 0 the greedy rule.
//
// Work. An item is one target row (position j of request i; a pair with draft row j when j < K_i,
// else the row of the bonus or plain draw). Every row is cut into slices of kSliceVecs 16-byte
// vectors (16 KB); a unit is one slice of one item: the target slice, and for a pair the draft
// slice at the same vocabulary offset. Units are numbered item-major and dealt round-robin: CTA c
// takes units c, c + G, c + 2G, ... (G CTAs), so at any time every CTA works on slices of the same
// few items, and no CTA holds two slices of one item (rows have at most G slices), which keeps
// the CTAs' waits on one another free of cycles.
//
// Grid. One persistent CTA per SM (every SM of the device), launched cooperatively so that all
// are resident at once (CTAs wait on one another's published statistics). Warp roles:
//   data warps (kDW): the jobs, in order: pass 1 of unit n, then pass 2 of unit n - kLag. Thread
//       (w, l) takes vectors w*128 + 32k + l, k < kVPT, of a slice (data warp w covers one
//       128-vector chunk);
//   producer: finds each unit's request and per-item values and writes the unit's descriptor;
//       issues each job's bulk copies (TMA, 1-D) into the job's pair of shared-memory slots: the
//       slices from HBM for pass 1, and again, kLag units later, from L2 for pass 2 (pass 1 copies
//       a pair's slices with an evict-last hint). Shared memory holds only the slices in flight, so
//       a late decision delays nothing but its own pass 2;
//   stats: reduces unit n's pass-1 partials to the unit's statistics (per row an integral
//       reference exponent and the sum of 2^(y s - ref); per 128-vector chunk of a target row its
//       share, for draws from p; the logits at the draft token, from the unit that holds it) and
//       publishes them in global memory as tagged words;
//   decide: four groups of eight lanes, each on its own unit, wait until every unit of the unit's
//       item has published, combine the records (the same reduction in every CTA, so every CTA
//       reaches the same decision) and decide the accept test; decisions may complete out of order;
//   finish: in order, reduces unit n's pass-2 partials (alpha and the residual per chunk) and
//       publishes them; the item's designated unit (slice item mod ns) hands the item to the final
//       warp;
//   final: the item's results and its draw (inverse CDF over the chunk masses, then within the one
//       chunk that holds u*Z, re-read from global memory); the last item of a request runs the
//       request's selection (first rejection, emitted tokens, stopping).
// The last CTA to finish writes the batch's alpha sum and depth counts and, for a round, runs the
// compaction and the gamma choice; it also resets the workspace's counters for the next call.
//
// Publication without fences: a published value is a 64-bit word (value, tag) written with one
// store; the tag is the call's epoch + 1 (the epoch lives in the workspace and grows by one per
// call), so a reader that polls the words sees either a stale tag or the whole value.
//
// The residual max(p - q, 0) is formed without cancellation: p (1 - 2^d) with d = log2(q/p) from
// the exact difference of the two logits, and 1 - 2^d from a series near d = 0, so that every
// residual weight is accurate to a few units in the last place of float32 however close q is to p.
//
// Every wait is bounded (mbarrier waits suspend between tries; global polls sleep between tries).
// A wait that gives up marks the CTA (and the items it touches) with SPEC_REQ_TIMEOUT; a request
// whose selection never ran is reported with SPEC_REQ_TIMEOUT by the last CTA.
#pragma once

#include <climits>
#include <cmath>
#include <cstdint>

#include "spec_device.cuh"
#include "spec_math.cuh"
#include "spec_tail.cuh"
#include "spec_verify.h"

namespace spec {
namespace slice {

constexpr int kDW = 16;                             // data warps
constexpr int kDataThreads = kDW * kWarp;           // 512
constexpr int kVPT = 2;                             // 16-byte vectors per data thread, row and slice
constexpr int kSliceVecs = kDataThreads * kVPT;     // 1024 vectors: 16 KB of one row
constexpr int kChunkVecs = kWarp * kVPT;            // 64 vectors: a data warp's share, a draw chunk
constexpr int kJobs = 6;                            // job ring: a job (pass 1 or pass 2 of a unit)
                                                    // owns two 16 KB slots
constexpr int kSlots = 2 * kJobs;                   // 16 KB slots
constexpr int kLag = 10;                            // pass 2 of unit n - kLag follows pass 1 of unit n
constexpr int kR = 16;                              // unit ring: descriptors
constexpr int kFQ = 16;                             // the final warp's queue
constexpr int kStage = 520;                         // row offsets staged in shared memory (B < kStage)
constexpr int kPrep = 8;                            // producer: descriptors prepared at once
static_assert(kR >= kLag + kJobs, "a unit's descriptor must outlive its last job");

// Warps: the data warps, the producer, the final warp. Eighteen warps put at most five on each of
// the four schedulers, whose register files (16384 each) then leave 96 registers to a thread.
enum : int { W_PROD = kDW, W_FINAL, kNumWarps };
constexpr int kBlock = kNumWarps * kWarp;  // 576 threads
constexpr int kMaxRegs = 96;

// Published records (64-bit tagged words), per data warp of a unit (one 128-vector chunk of each
// slice), contiguous per item: pass 1, the reference exponent and sum of its target and its draft
// chunk (greedy: argmax and max); pass 2, its alpha share and residual mass. Per item: the draft
// token's words (from the thread holding them) and the item's decision.
enum : int { W1_AT = 0, W1_ST = 1, W1_AD = 2, W1_SD = 3, kW1Words = 4 };
enum : int { W2_ALPHA = 0, W2_Z = 1, kW2Words = 2 };
enum : int { X_HI = 0, X_LO = 1, X_F = 2, kXWords = 4 };
// the decision: UnitDec's sixteen 32-bit fields in order
constexpr int kDecWords = 16;
// control words of the workspace
enum : int { CTL_DONE = 0, CTL_EPOCH = 1, kCtlWords = 4 };
enum : int32_t { XF_QZERO = 1, XF_PZERO = 2 };

enum : int32_t { U_END = 0, U_PAIR = 1, U_ROW = 2, U_SKIP = 3 };
// jobs: pass 1 of a unit; its pass 2 (slices again, with the item's decision); a unit without rows;
// the end
enum : int32_t { J_END = 0, J_P1 = 1, J_P2 = 2, J_SKIP = 3 };
enum : int32_t { SAMPLE_NONE = 0, SAMPLE_RESIDUAL = 1, SAMPLE_P = 2 };
enum : int32_t { REQ_TIMEOUT = SPEC_REQ_TIMEOUT };
constexpr int32_t kNoRef = -(1 << 30);  // reference exponent of a row (or part) with no mass

constexpr uint32_t kSuspendNs = 1u << 20;  // one suspended mbarrier try: at most ~1 ms
constexpr int kMaxWaitTries = 2048;        // ~2 s in all
constexpr uint64_t kPollNs = 200000000ull;  // a global poll gives up after 0.2 s (1 ms once a wait of
                                            // the CTA has given up)

constexpr float kLog2eHi = 1.44269502162933349609375f;
constexpr float kLog2eLo = 1.925963e-08f;

struct SliceParams {
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
    int32_t ns;              // slices per row
    int32_t nunits;          // total_rows * ns
    // workspace
    unsigned long long *p1w;       // [nunits][kDW][kW1Words]
    unsigned long long *p2w;       // [nunits][kDW][kW2Words]
    unsigned long long *xrec;      // [T][kXWords]
    unsigned long long *drec;      // [T][kDecWords]
    uint32_t *req_cnt;             // [B] items of the request finalised
    uint32_t *ctl;                 // [kCtlWords]
    int32_t *item_flag, *item_tok, *item_status, *item_fb;
    float *item_prob, *item_margin;
    float *alpha_ws;               // [T-B]
    float2 *req_alpha;             // [B] alpha summed over the request's draft rows (float pair)
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

// A unit, as the producer describes it.
struct UnitDesc {
    int32_t kind;            // U_*
    int32_t item, slice, req, pos, K, drow;
    int32_t nvec;            // vectors of this slice (the last slice of a row may be short)
    int32_t greedy, trunc, status;
    int32_t x;               // a pair's draft token (-1: none)
    int32_t xslice;          // the slice holding x's vector (-1: x outside [0, V))
    int32_t designated;      // this unit finalises the item (slice == item mod ns)
    float s_hi, s_lo;        // log2(e)/T as a float pair, s_hi rounded toward zero (s_lo > 0)
    uint32_t cut_tau;        // top-k / top-p cut of the target row (trunc = 0: none)
    int32_t cut_id;
    double ua, us;           // the position's accept draw and the request's frontier draw
};

// The decision of a unit's item (identical in every CTA that holds a unit of the item).
struct UnitDec {
    int32_t status, accept, kind, argmax_t;
    float B_t, S_t;              // target: integral reference exponent and the sum at it
    float c_t, c_tf, c_d, c_df;  // log2 of each normaliser: integral part, fraction
    F2 dc;                       // c_d - c_t as a float pair
    float rho, alpha_g;
    F2 u_s;
};

static_assert(sizeof(UnitDec) == kDecWords * 4, "the decision record holds UnitDec's fields");

// A job of the final warp: decide an item (its last unit has been through pass 1 in this CTA),
// or finalise it (results and draw) with its decision; or the end of the queue.
enum : int32_t { F_END = 0, F_DECIDE = 1, F_FINAL = 2 };
struct FinJob {
    int32_t op;
    UnitDesc d;
    UnitDec D;
};

// A job of the data warps, in the job's slots: pass 1 (the unit's slices), or pass 2 (the slices
// again and the item's decision record).
struct Job {
    int32_t type, unit;
};

struct Shared {
    unsigned long long drec[kJobs][kDecWords];  // a pass-2 job's copy of the item's decision
    UnitDesc desc[kR];
    FinJob fq[kFQ];
    Job jobs[kJobs];
    UnitDesc prep[kPrep];     // producer: the next batch of descriptors, prepared one per lane
    int32_t roff[kStage + 1];
    uint64_t desc_full[kR];   // producer: descriptor written
    uint64_t desc_empty[kR];  // every data warp is done with it
    uint64_t job_full[kJobs];     // producer: the job written, its copies landed
    uint64_t job_empty[kJobs];    // data warps: done with the job's slots
    uint64_t fq_full[kFQ], fq_empty[kFQ];
    int32_t fq_tail;          // tickets of the final warp's queue (several data warps push)
    int32_t end_cnt;          // data warps that reached the end
    int32_t timed_out;
    int32_t bad_offsets;      // row_off fails its checks: every request is BAD_SHAPE
    int32_t staged;           // row_off is in roff
    int32_t last_cta;
    uint32_t epoch;           // the workspace's epoch at launch
    uint32_t tag;             // the tag of this call's published words
};

// ------------------------------------------------------------------------------------------------
// small helpers

__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

__device__ __forceinline__ unsigned long long tagged(uint32_t value, uint32_t tag) {
    return (static_cast<unsigned long long>(value) << 32) | tag;
}
__device__ __forceinline__ void st_word(unsigned long long *p, uint32_t value, uint32_t tag) {
    const unsigned long long w = tagged(value, tag);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ld_word(const unsigned long long *p) {
    unsigned long long w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ ulonglong2 ld_word2(const unsigned long long *p) {
    ulonglong2 w;
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(w.x), "=l"(w.y) : "l"(p) : "memory");
    return w;
}
__device__ __forceinline__ uint32_t ld_u32_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t word_tag(unsigned long long w) { return static_cast<uint32_t>(w); }
__device__ __forceinline__ uint32_t word_val(unsigned long long w) { return static_cast<uint32_t>(w >> 32); }

// mbarrier expect-tx without an arrival (the producer arrives after writing the descriptor).
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// A bounded wait: one plain test first (the usual case: the phase is complete), then suspended
// tries. Once a wait of this CTA has given up, later ones give up after a couple of tries.
__device__ __forceinline__ bool wait_bar(Shared &sh, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const int tries = *reinterpret_cast<volatile int32_t *>(&sh.timed_out) ? 2 : kMaxWaitTries;
    if (mbar_wait_sleep_bounded(bar, parity, kSuspendNs, tries)) return true;
    sh.timed_out = 1;
    return false;
}

__device__ __forceinline__ void warp_arrive(uint64_t *bar, int lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// 2^d for an integer d <= 0 with integer operations only (0 below the normal range).
__device__ __forceinline__ float pow2_int(int d) { return d < -126 ? 0.0f : __int_as_float((d + 127) << 23); }

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

// Vector vi of a slice in its slot, or -inf past the slice's end (no mass, never a maximum).
template <int DT>
__device__ __forceinline__ uint4 slice_vec(const uint4 *slot, int vi, int nvec) {
    return vi < nvec ? slot[vi] : kNegInfVec<DT>();
}

// A thread's sum of 2^(y s - b) over its kVPT vectors of one row in the exact form, for a warp in
// which some thread's fast sum overflowed (above 2^64: a later vector much larger than the first,
// an all -inf first vector, a NaN or +inf): b from the thread's max over all its vectors (0 for an
// all -inf thread, whose sum is then 0). Rare: out of line, the vectors read again from the slot.
template <int DT>
__device__ __noinline__ float2 row_sum_exact(const UnitDesc &d, const uint4 *slot, int vbase, bool cut) {
    const int vglob = d.slice * kSliceVecs + vbase;
    const float2 shi2 = f2splat(d.s_hi), slo2 = f2splat(d.s_lo);
    uint4 v[kVPT];
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
        v[k] = slice_vec<DT>(slot, vbase + k * kWarp, d.nvec);
        if (cut) mask_cut<DT>(v[k], vglob + k * kWarp, d.cut_tau, d.cut_id);
        m = fmaxf(m, Elt<DT>::vmax(v[k]));
    }
    const float b = (m == -INFINITY) ? 0.0f : floorf(m * d.s_hi);
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < kVPT; ++k) s += vec_sum<DT>(v[k], shi2, slo2, b);
    return make_float2(b, s);
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

// Pass 1 of one unit under the greedy rule by one data thread: (max_t, argmax_t, max_d, argmax_d)
// of its vectors (indices as int bits). Out of line (the greedy rule is the rare one).
template <int DT>
__device__ __noinline__ float4 pass1_greedy(const UnitDesc &d, const uint4 *tslot, const uint4 *dslot, int vbase) {
    const bool pair = d.kind == U_PAIR;
    const int vglob = d.slice * kSliceVecs + vbase;
    uint4 vt[kVPT], vd[kVPT];
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
        vt[k] = slice_vec<DT>(tslot, vbase + k * kWarp, d.nvec);
        vd[k] = pair ? slice_vec<DT>(dslot, vbase + k * kWarp, d.nvec) : kNegInfVec<DT>();
    }
    float bt, bd = -INFINITY;
    int it, id = INT_MAX;
    row_argmax<DT>(vt, vglob, bt, it);
    if (pair) row_argmax<DT>(vd, vglob, bd, id);
    return make_float4(bt, __int_as_float(it), bd, __int_as_float(id));
}

// The draft token's words of a pair, published by the thread whose vectors hold it: (y_t - y_d) s
// at the token (a float pair) and the flags of a -inf logit. Out of line (one unit of a row holds
// it).
template <int DT>
__device__ __noinline__ void extract_x(const UnitDesc &d, const uint4 *tslot, const uint4 *dslot, int vbase,
                                       unsigned long long *xrec, uint32_t tag) {
    constexpr int E = Elt<DT>::kPerVec;
    // x = E * (vglob + 32 k) + e for one thread and one k
    const int xv = d.x / E - d.slice * kSliceVecs;  // its vector's index in the slice
    if (xv < vbase || xv >= vbase + kVPT * kWarp || (xv - vbase) % kWarp != 0) return;
    uint4 wt = tslot[xv];
    const uint4 wd = dslot[xv];
    if (d.trunc) mask_cut<DT>(wt, d.slice * kSliceVecs + xv, d.cut_tau, d.cut_id);
    const float yt = vec_elem<DT>(wt, d.x % E), yd = vec_elem<DT>(wd, d.x % E);
    const F2 Ex = f2_mul(f2_add({yt, 0.0f}, {-yd, 0.0f}), {d.s_hi, d.s_lo});
    const int flags = (yd == -INFINITY ? XF_QZERO : 0) | (yt == -INFINITY ? XF_PZERO : 0);
    st_word(xrec + X_HI, f2u(Ex.hi), tag);
    st_word(xrec + X_LO, f2u(Ex.lo), tag);
    st_word(xrec + X_F, static_cast<uint32_t>(flags), tag);
}

// Pass 1 of one unit under Rule 2 by one data thread: (b_t, s_t, b_d, s_d), per row the sum of
// 2^(y s - b) over its vectors with b an integral reference from its first vector (so that no
// exponential waits on a running max); a warp in which a sum overflowed takes the exact form.
// CUT: the target row's top-k / top-p cut (a separate, out-of-line instance).
template <int DT, bool CUT>
__device__ __forceinline__ float4 pass1_body(const UnitDesc &d, const uint4 *tslot, const uint4 *dslot, int vbase) {
    const bool pair = d.kind == U_PAIR;
    const int nvec = d.nvec;
    const float2 shi2 = f2splat(d.s_hi), slo2 = f2splat(d.s_lo);
    uint4 vt[kVPT], vd[kVPT];
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
        vt[k] = slice_vec<DT>(tslot, vbase + k * kWarp, nvec);
        if (CUT) mask_cut<DT>(vt[k], d.slice * kSliceVecs + vbase + k * kWarp, d.cut_tau, d.cut_id);
    }
    float bt = floorf(Elt<DT>::vmax(vt[0]) * d.s_hi);
    float st = 0.0f;
#pragma unroll
    for (int k = 0; k < kVPT; ++k) st += vec_sum<DT>(vt[k], shi2, slo2, bt);
    float bd = 0.0f, sd = 0.0f;
    if (pair) {
#pragma unroll
        for (int k = 0; k < kVPT; ++k) vd[k] = slice_vec<DT>(dslot, vbase + k * kWarp, nvec);
        bd = floorf(Elt<DT>::vmax(vd[0]) * d.s_hi);
#pragma unroll
        for (int k = 0; k < kVPT; ++k) sd += vec_sum<DT>(vd[k], shi2, slo2, bd);
    }
    if (__any_sync(0xffffffffu, !(st <= 0x1p64f))) {
        const float2 e = row_sum_exact<DT>(d, tslot, vbase, CUT);
        bt = e.x;
        st = e.y;
    }
    if (__any_sync(0xffffffffu, !(sd <= 0x1p64f))) {
        const float2 e = row_sum_exact<DT>(d, dslot, vbase, false);
        bd = e.x;
        sd = e.y;
    }
    return make_float4(bt, st, bd, sd);
}
template <int DT>
__device__ __noinline__ float4 pass1_cut(const UnitDesc &d, const uint4 *tslot, const uint4 *dslot, int vbase) {
    return pass1_body<DT, true>(d, tslot, dslot, vbase);
}

// ------------------------------------------------------------------------------------------------
// data warps: pass 2 (a pair under Rule 2)

// The partial (alpha share, residual mass) of one thread's vectors, both normalised. Where the
// position rejects, max(p - q, 0) and min(p, q) by resid_weights; where it accepts, only alpha:
// min(p, q) = 2^min(y_t s - c_t, y_d s - c_d), c the log2 of the normaliser.
template <int DT, bool CUT>
__device__ __forceinline__ float2 pass2_body(const UnitDesc &d, const UnitDec &D, const uint4 *tslot,
                                             const uint4 *dslot, int vbase) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    if (D.status != 0) return make_float2(0.0f, 0.0f);
    uint4 vt[kVPT], vd[kVPT];
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
        vt[k] = slice_vec<DT>(tslot, vbase + k * kWarp, d.nvec);
        vd[k] = slice_vec<DT>(dslot, vbase + k * kWarp, d.nvec);
        if (CUT) mask_cut<DT>(vt[k], d.slice * kSliceVecs + vbase + k * kWarp, d.cut_tau, d.cut_id);
    }
    const float2 shi2 = f2splat(d.s_hi);
    const float2 nct = f2splat(-D.c_t), nctf = f2splat(-D.c_tf);
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
        return make_float2(aacc.x + aacc.y, racc.x + racc.y);
    }
    // y s - c with c split: the product less the integral part rounds once (to a small result
    // near the top of the row), then the fraction
    const float2 ncd = f2splat(-D.c_d), ncdf = f2splat(-D.c_df);
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
    return make_float2(acc.x + acc.y, 0.0f);
}
template <int DT>
__device__ __noinline__ float2 pass2_cut(const UnitDesc &d, const UnitDec &D, const uint4 *tslot, const uint4 *dslot,
                                         int vbase) {
    return pass2_body<DT, true>(d, D, tslot, dslot, vbase);
}

// ------------------------------------------------------------------------------------------------
// reductions: a data warp's partial (its chunk), then the unit's (the eight warps, by the last data
// warp to finish the job)

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

// A data warp's pass-1 partial from its threads' (the warp's chunk of both slices).
__device__ __forceinline__ float4 warp_p1(float4 r, bool greedy, bool pair) {
    if (greedy) {
        float m0 = r.x, m1 = r.z;
        int i0 = __float_as_int(r.y), i1 = __float_as_int(r.w);
        arg_max<kWarp>(m0, i0);
        arg_max<kWarp>(m1, i1);
        return make_float4(m0, __int_as_float(i0), m1, __int_as_float(i1));
    }
    const float2 t = ref_sum<kWarp>(r.x, r.y);
    const float2 d = pair ? ref_sum<kWarp>(r.z, r.w) : make_float2(-INFINITY, 0.0f);
    return make_float4(t.x, t.y, d.x, d.y);
}

// A data warp's pass-1 record (lanes 0..3, one word each; w is the same in every lane): per row
// its reference (kNoRef: no mass) and sum (NaN: invalid logits; a reference beyond 2^28 reads as
// invalid), or under the greedy rule its argmax and max.
__device__ __forceinline__ void store_w1(unsigned long long *rec, float4 w, bool greedy, bool pair, uint32_t tag) {
    const int lane = threadIdx.x % kWarp;
    uint32_t v0, v1, v2, v3;
    if (greedy) {
        v0 = static_cast<uint32_t>(__float_as_int(w.y));
        v1 = f2u(w.x);
        v2 = static_cast<uint32_t>(__float_as_int(w.w));
        v3 = f2u(w.z);
    } else {
        const bool inval_t = isnan(w.y) || (w.y > 0.0f && !(fabsf(w.x) < 0x1p28f));
        const bool inval_d = isnan(w.w) || (w.w > 0.0f && !(fabsf(w.z) < 0x1p28f));
        v0 = static_cast<uint32_t>((w.y > 0.0f && !inval_t) ? static_cast<int>(w.x) : kNoRef);
        v1 = f2u(inval_t ? NAN : w.y);
        v2 = static_cast<uint32_t>((pair && w.w > 0.0f && !inval_d) ? static_cast<int>(w.z) : kNoRef);
        v3 = f2u(pair ? (inval_d ? NAN : w.w) : 0.0f);
    }
    if (lane < kW1Words) st_word(rec + lane, lane == 0 ? v0 : lane == 1 ? v1 : lane == 2 ? v2 : v3, tag);
}

// ------------------------------------------------------------------------------------------------
// the decision of an item

// The decision of unit d's item from its units' combined statistics (every lane of the group
// computes it; the same inputs give the same result in every CTA). Rule 2: (a0, s0) / (a1, s1)
// reference and sum of the target / draft row over the vocabulary; Ex = (y_t - y_d) s at the draft
// token and its flags. Greedy: (a0, s0) / (a1, s1) are (argmax, max) of each row.
__device__ __forceinline__ UnitDec decide_item(const SliceParams &P, const UnitDesc &d, int status, int a0, float s0,
                                               int a1, float s1, F2 Ex, int xflags) {
    const bool pair = d.kind == U_PAIR;
    const int x = d.x;
    UnitDec D = {};
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

// The decision of item d (whole warp) from the pass-1 records of every data warp of every unit of
// the item, and the draft token's words, polled until they carry the call's tag (every CTA that
// reads the item's records obtains the same values). Lane l combines records l, l + 32, ...; the
// parts combine like a unit's: references by exact powers of two (argmax pairs under the greedy
// rule).
__device__ __noinline__ UnitDec decide_records(const SliceParams &P, const UnitDesc &d, uint32_t tag, Shared &sh) {
    const int lane = threadIdx.x % kWarp;
    const bool greedy = d.greedy != 0;
    const int nrec = P.ns * kDW;
    const unsigned long long *g = P.p1w + static_cast<size_t>(d.item) * nrec * kW1Words;
    const uint64_t limit = *reinterpret_cast<volatile int32_t *>(&sh.timed_out) ? 1000000ull : kPollNs;
    uint64_t t0 = 0;
    bool gave_up = false;
    int la0 = greedy ? INT_MAX : kNoRef, la1 = la0;
    float ls0 = greedy ? -INFINITY : 0.0f, ls1 = ls0;
    // rounds of up to kRound records per lane, every load of a round in flight at once
    constexpr int kRound = 4;
    for (int base = 0; base < nrec; base += kRound * kWarp) {
        ulonglong2 w01[kRound], w23[kRound];
        for (bool first = true;; first = false) {
            bool ok = true;
#pragma unroll
            for (int k = 0; k < kRound; ++k) {
                const int u = base + k * kWarp + lane;
                if (u < nrec) {
                    w01[k] = ld_word2(g + static_cast<size_t>(u) * kW1Words + W1_AT);
                    w23[k] = ld_word2(g + static_cast<size_t>(u) * kW1Words + W1_AD);
                    ok &= (word_tag(w01[k].x) == tag) & (word_tag(w01[k].y) == tag) & (word_tag(w23[k].x) == tag) &
                          (word_tag(w23[k].y) == tag);
                }
            }
            if (__all_sync(0xffffffffu, ok) || gave_up) break;
            const uint64_t now = globaltimer_ns();
            if (first) t0 = now;
            gave_up = __shfl_sync(0xffffffffu, static_cast<int>(now - t0 > limit), 0) != 0;
            if (!gave_up) __nanosleep(64);
        }
#pragma unroll
        for (int k = 0; k < kRound; ++k) {
            if (base + k * kWarp + lane >= nrec) continue;
            const int ua0 = static_cast<int>(word_val(w01[k].x)), ua1 = static_cast<int>(word_val(w23[k].x));
            const float us0 = u2f(word_val(w01[k].y)), us1 = u2f(word_val(w23[k].y));
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
        float t0s = ls0 * pow2_int(la0 - B0), t1s = ls1 * pow2_int(la1 - B1);
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            t0s += __shfl_xor_sync(0xffffffffu, t0s, o);
            t1s += __shfl_xor_sync(0xffffffffu, t1s, o);
        }
        a0 = B0;
        a1 = B1;
        s0 = t0s;
        s1 = t1s;
    }
    // the draft token's words (Rule 2 pairs), by lane 0, then to every lane
    F2 Ex = {0.0f, 0.0f};
    int xf = 0;
    if (d.kind == U_PAIR && !greedy && d.xslice >= 0) {
        if (lane == 0) {
            const unsigned long long *r = P.xrec + static_cast<size_t>(d.item) * kXWords;
            unsigned long long x0 = 0, x1 = 0, x2 = 0;
            uint64_t tx = 0;
            for (bool first = true; !gave_up; first = false) {
                x0 = ld_word(r + X_HI);
                x1 = ld_word(r + X_LO);
                x2 = ld_word(r + X_F);
                if ((word_tag(x0) == tag) & (word_tag(x1) == tag) & (word_tag(x2) == tag)) break;
                const uint64_t now = globaltimer_ns();
                if (first) tx = now;
                if (now - tx > limit)
                    gave_up = true;
                else
                    __nanosleep(64);
            }
            Ex = {u2f(word_val(x0)), u2f(word_val(x1))};
            xf = __float_as_int(u2f(word_val(x2)));
        }
        gave_up = __shfl_sync(0xffffffffu, gave_up ? 1 : 0, 0) != 0;
        Ex.hi = __shfl_sync(0xffffffffu, Ex.hi, 0);
        Ex.lo = __shfl_sync(0xffffffffu, Ex.lo, 0);
        xf = __shfl_sync(0xffffffffu, xf, 0);
    }
    int status = d.status;
    if (gave_up) {
        status |= REQ_TIMEOUT;
        if (lane == 0) sh.timed_out = 1;
    }
    if (*reinterpret_cast<volatile int32_t *>(&sh.timed_out)) status |= REQ_TIMEOUT;
    return decide_item(P, d, status, a0, s0, a1, s1, Ex, xf);
}

// The decision as its record's words and back (the value of word k is UnitDec's field k).
__device__ __forceinline__ uint32_t dec_word(const UnitDec &D, int k) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&D);
    uint32_t v = 0;
#pragma unroll
    for (int i = 0; i < kDecWords; ++i)
        if (i == k) v = w[i];
    return v;
}

// A pass-2 job's decision (whole warp): the job's copy of the item's decision record, or, where a
// word of the copy is stale (the record was published after the copy), the record itself, polled.
// A wait that gives up yields a decision with SPEC_REQ_TIMEOUT.
__device__ __noinline__ UnitDec poll_decision(const SliceParams &P, const UnitDesc &d, uint32_t tag, Shared &sh) {
    const int lane = threadIdx.x % kWarp;
    const unsigned long long *r = P.drec + static_cast<size_t>(d.item) * kDecWords;
    const uint64_t limit = *reinterpret_cast<volatile int32_t *>(&sh.timed_out) ? 1000000ull : kPollNs;
    uint64_t t0 = 0;
    unsigned long long w = 0;
    for (bool first = true;; first = false) {
        if (lane < kDecWords) w = ld_word(r + lane);
        if (__all_sync(0xffffffffu, lane >= kDecWords || word_tag(w) == tag)) break;
        const uint64_t now = globaltimer_ns();
        if (first) t0 = now;
        if (__shfl_sync(0xffffffffu, static_cast<int>(now - t0 > limit), 0)) {
            if (lane == 0) sh.timed_out = 1;
            UnitDec D = {};
            D.status = d.status | REQ_TIMEOUT;
            D.kind = SAMPLE_NONE;
            D.argmax_t = -1;
            return D;
        }
        __nanosleep(64);
    }
    UnitDec D;
    uint32_t *dw = reinterpret_cast<uint32_t *>(&D);
#pragma unroll
    for (int k = 0; k < kDecWords; ++k) dw[k] = __shfl_sync(0xffffffffu, static_cast<uint32_t>(w >> 32), k);
    return D;
}
__device__ __forceinline__ UnitDec read_decision(const SliceParams &P, const UnitDesc &d,
                                                 const unsigned long long *copy, uint32_t tag, Shared &sh) {
    UnitDec D;
    uint32_t *dw = reinterpret_cast<uint32_t *>(&D);
    bool ok = true;
#pragma unroll
    for (int k = 0; k < kDecWords; k += 2) {
        const ulonglong2 w = *reinterpret_cast<const ulonglong2 *>(copy + k);
        ok &= (word_tag(w.x) == tag) & (word_tag(w.y) == tag);
        dw[k] = word_val(w.x);
        dw[k + 1] = word_val(w.y);
    }
    if (__all_sync(0xffffffffu, ok)) return D;
    return poll_decision(P, d, tag, sh);
}

// The decision of a unit without rows (its request was rejected before any work).
__device__ __forceinline__ UnitDec skip_decision(const UnitDesc &d) {
    UnitDec D = {};
    D.status = d.status;
    D.kind = SAMPLE_NONE;
    D.argmax_t = -1;
    return D;
}

// Hands an item to the final warp (whole warp; several data warps push: the tickets keep the
// queue in the order they were taken).
__device__ __forceinline__ void fq_push(Shared &sh, int op, const UnitDesc &d, const UnitDec &D) {
    const int lane = threadIdx.x % kWarp;
    int t = 0;
    if (lane == 0) t = atomicAdd(&sh.fq_tail, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    const int q = t % kFQ;
    if (t >= kFQ && !wait_bar(sh, &sh.fq_empty[q], static_cast<uint32_t>(((t / kFQ) - 1) & 1))) return;
    if (lane == 0) {
        sh.fq[q].op = op;
        sh.fq[q].d = d;
        sh.fq[q].D = D;
        mbar_arrive(&sh.fq_full[q]);
    }
    __syncwarp();
}

// ------------------------------------------------------------------------------------------------
// final warp: an item's results and draw, a request's selection

// Waits until words k < nw of units u < nunits (word k of unit u at base + u * stride + k; lane l
// reads units l, l + 32, ...) all carry the tag. Returns false once the wait gives up.
__device__ __forceinline__ bool poll_units(Shared &sh, const unsigned long long *base, int nunits, int stride, int nw,
                                           uint32_t tag) {
    const uint64_t limit = *reinterpret_cast<volatile int32_t *>(&sh.timed_out) ? 1000000ull : kPollNs;
    uint64_t t0 = 0;
    for (bool first = true;; first = false) {
        int ok = 1;
        for (int u = static_cast<int>(threadIdx.x % kWarp); u < nunits; u += kWarp)
            for (int k = 0; k < nw; ++k) ok &= word_tag(ld_word(base + static_cast<size_t>(u) * stride + k)) == tag;
        if (__all_sync(0xffffffffu, ok)) return true;
        const uint64_t now = globaltimer_ns();
        if (first) t0 = now;
        if (__shfl_sync(0xffffffffu, static_cast<int>(now - t0 > limit), 0)) return false;
        __nanosleep(64);
    }
}

// The draw weights of one vector, exactly as the passes summed them: the residual (normalised),
// or p in units of 2^B_t.
template <int DT>
__device__ __forceinline__ void draw_weights(int kind, const uint4 &wt, const uint4 &wd, const UnitDesc &d,
                                             const UnitDec &D, float *w) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    const float2 shi2 = f2splat(d.s_hi), slo2 = f2splat(d.s_lo);
    if (kind == SAMPLE_RESIDUAL) {
        const float2 nct = f2splat(-D.c_t), nctf = f2splat(-D.c_tf);
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

// The mass of chunk c (128 vectors of the row: data warp c mod kDW of unit c / kDW) in the law of
// the draw: the residual's (normalised), or p's in units of 2^B_t.
__device__ __forceinline__ float chunk_mass(const SliceParams &P, const UnitDesc &d, const UnitDec &D, int kind, int c) {
    const size_t rec = static_cast<size_t>(d.item) * P.ns * kDW + c;
    if (kind == SAMPLE_RESIDUAL) return u2f(word_val(ld_word(P.p2w + rec * kW2Words + W2_Z)));
    const int ref = static_cast<int>(word_val(ld_word(P.p1w + rec * kW1Words + W1_AT)));
    const float cm = u2f(word_val(ld_word(P.p1w + rec * kW1Words + W1_ST)));
    return (ref == kNoRef || !(cm > 0.0f)) ? 0.0f : cm * pow2_int(ref - static_cast<int>(D.B_t));
}

// The draw of item d from the law `kind` (whole warp): the chunk that holds u*Z by an inclusive
// scan over the chunk masses in vocabulary order, then the token within it, the weights recomputed
// exactly as the passes summed them. Writes the token, its probability and the CDF margin.
template <int DT>
__device__ __noinline__ void draw_item(const SliceParams &P, const UnitDesc &d, const UnitDec &D, int kind, int &tok,
                                       float &prob, float &margin) {
    constexpr int E = Elt<DT>::kPerVec;
    const int lane = threadIdx.x % kWarp;
    const int nc = (P.nvec_row + kChunkVecs - 1) / kChunkVecs;
    // the chunk masses are read twice: once for Z, once for the scan
    F2 Z = {0.0f, 0.0f};
    for (int base = 0; base < nc; base += kWarp) {
        const int c = base + lane;
        const float m = c < nc ? chunk_mass(P, d, D, kind, c) : 0.0f;
        Z = f2_add(Z, warp_sum_f2({m, 0.0f}));
    }
    const F2 t = f2_mul(Z, D.u_s);
    int csel = -1, clast = -1;
    F2 before = {0.0f, 0.0f}, last_before = {0.0f, 0.0f}, run = {0.0f, 0.0f};
    for (int base = 0; base < nc; base += kWarp) {
        const int c = base + lane;
        const float m = c < nc ? chunk_mass(P, d, D, kind, c) : 0.0f;
        const bool pos = m > 0.0f;
        const F2 incl = f2_add(run, warp_scan_f2({m, 0.0f}, lane));
        const unsigned hit = __ballot_sync(0xffffffffu, pos && f2_gt(incl, t));
        const unsigned posm = __ballot_sync(0xffffffffu, pos);
        if (hit) {
            const int l = __ffs(hit) - 1;
            csel = base + l;
            before = shfl_f2(f2_sub(incl, {m, 0.0f}), l);
            break;
        }
        if (posm) {
            const int l = 31 - __clz(static_cast<int>(posm));
            clast = base + l;
            last_before = shfl_f2(f2_sub(incl, {m, 0.0f}), l);
        }
        run = shfl_f2(incl, kWarp - 1);
    }
    const bool clamped = csel < 0;  // rounding put u*Z past the last chunk with mass
    if (clamped) {
        csel = clast;
        before = last_before;
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
    // the chunk's vectors c*128 + 32k + lane, in vocabulary order k-major
    float w[kVPT][E];
    float vs[kVPT];
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
        const int vi = csel * kChunkVecs + k * kWarp + lane;
        uint4 wt = kNegInfVec<DT>(), wd = kNegInfVec<DT>();
        if (vi < P.nvec_row) {
            wt = __ldcg(trow + vi);
            if (kind == SAMPLE_RESIDUAL) wd = __ldcg(drow + vi);
        }
        if (d.trunc) mask_cut<DT>(wt, vi, d.cut_tau, d.cut_id);
        draw_weights<DT>(kind, wt, wd, d, D, w[k]);
        float s = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) s += w[k][e];
        vs[k] = s;
    }
    float c = 0.0f;  // mass before vector (k, lane) within the chunk
    int last_k = -1, last_e = -1, found_e = -1;
    float fprev = 0.0f, wf = 0.0f, wl = 0.0f;
    unsigned hit = 0u;
    int hk = -1;
#pragma unroll
    for (int k = 0; k < kVPT; ++k) {
        float incl = vs[k];
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const float x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        float cc = c + incl - vs[k];
        int fe = -1;
        float fp = 0.0f, fw = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            if (w[k][e] > 0.0f) {
                if (fe < 0 && !clamped && cc + w[k][e] > lt) {
                    fe = e;
                    fp = cc;
                    fw = w[k][e];
                }
                last_k = k;
                last_e = e;
                wl = w[k][e];
            }
            cc += w[k][e];
        }
        const unsigned h = __ballot_sync(0xffffffffu, fe >= 0);
        if (h && hk < 0) {
            hk = k;
            hit = h;
            found_e = fe;
            fprev = fp;
            wf = fw;
        }
        c += __shfl_sync(0xffffffffu, incl, kWarp - 1);
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

// A request's selection (whole warp; every item of the request is finalised): the first rejection
// A, the emitted tokens (x_1 .. x_A, then the frontier), stop-token and max_new truncation, and
// the request's alpha sum. Lane j takes positions j and j + 32 (K_max <= 64: position 64 on lane 0).
__device__ __noinline__ void select_request(const SliceParams &P, int i) {
    const int lane = threadIdx.x % kWarp;
    const int r0 = __ldg(P.row_off + i), r1 = __ldg(P.row_off + i + 1);
    const int K = r1 - r0 - 1, d0 = r0 - i;
    const int n_cap = P.max_new ? __ldg(P.max_new + i) : INT_MAX;
    const int stop = P.stop_token ? __ldg(P.stop_token + i) : -1;
    int status = 0;
    if (K < 0 || K > P.K_max) status |= SPEC_REQ_BAD_SHAPE;
    int st_items = 0;
    unsigned rej_lo = 0u, rej_hi = 0u;
    int tok0 = -1, tok1 = -1, fb0 = 0, fb1 = 0, x0 = -1, x1 = -1, tok2 = -1, fb2 = 0;
    float pr0 = NAN, pr1 = NAN, mg0 = NAN, mg1 = NAN, al0 = 0.0f, al1 = 0.0f, pr2 = NAN, mg2 = NAN;
    if (!status) {
        const int j0 = lane, j1 = lane + kWarp;
        if (j0 <= K) {
            st_items |= __ldcg(P.item_status + r0 + j0);
            tok0 = __ldcg(P.item_tok + r0 + j0);
            pr0 = __ldcg(P.item_prob + r0 + j0);
            mg0 = __ldcg(P.item_margin + r0 + j0);
            fb0 = __ldcg(P.item_fb + r0 + j0);
            if (j0 < K) {
                x0 = __ldg(P.draft_tokens + d0 + j0);
                al0 = __ldcg(P.alpha_ws + d0 + j0);
            }
        }
        if (j1 <= K) {
            st_items |= __ldcg(P.item_status + r0 + j1);
            tok1 = __ldcg(P.item_tok + r0 + j1);
            pr1 = __ldcg(P.item_prob + r0 + j1);
            mg1 = __ldcg(P.item_margin + r0 + j1);
            fb1 = __ldcg(P.item_fb + r0 + j1);
            if (j1 < K) {
                x1 = __ldg(P.draft_tokens + d0 + j1);
                al1 = __ldcg(P.alpha_ws + d0 + j1);
            }
        }
        if (K == 2 * kWarp && lane == 0) {
            st_items |= __ldcg(P.item_status + r0 + K);
            tok2 = __ldcg(P.item_tok + r0 + K);
            pr2 = __ldcg(P.item_prob + r0 + K);
            mg2 = __ldcg(P.item_margin + r0 + K);
            fb2 = __ldcg(P.item_fb + r0 + K);
        }
        rej_lo = __ballot_sync(0xffffffffu, j0 < K && __ldcg(P.item_flag + r0 + min(j0, K)) == 0);
        rej_hi = __ballot_sync(0xffffffffu, j1 < K && __ldcg(P.item_flag + r0 + min(j1, K)) == 0);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) st_items |= __shfl_xor_sync(0xffffffffu, st_items, o);
    }
    status |= st_items;
    if (status) {
        if (K >= 0)
            for (int j = lane; j <= K; j += kWarp) P.out_tokens[r0 + j] = -1;
        if (lane == 0) {
            P.req_status[i] = status;
            P.accept_len[i] = 0;
            if (P.n_emitted) P.n_emitted[i] = 0;
            if (P.frontier_prob) P.frontier_prob[i] = NAN;
            if (P.frontier_margin) P.frontier_margin[i] = NAN;
            if (P.fallback) P.fallback[i] = 0;
            P.req_alpha[i] = make_float2(0.0f, 0.0f);
        }
        return;
    }
    const int A = rej_lo ? __ffs(rej_lo) - 1 : (rej_hi ? kWarp + __ffs(rej_hi) - 1 : K);
    const int la = A & (kWarp - 1), half = A >> 5;
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
    const F2 asum = warp_sum_f2(f2_add({al0, 0.0f}, {al1, 0.0f}));
    if (lane == 0) {
        P.req_status[i] = 0;
        P.accept_len[i] = A;
        if (P.n_emitted) P.n_emitted[i] = n;
        if (P.frontier_prob) P.frontier_prob[i] = fprob;
        if (P.frontier_margin) P.frontier_margin[i] = fmarg;
        if (P.fallback) P.fallback[i] = ffb;
        P.req_alpha[i] = make_float2(asum.hi, asum.lo);
    }
}

// The item's results and draw (whole warp), then the request's count; the last item of a request
// runs its selection.
template <int DT>
__device__ __noinline__ void finalize_item(const SliceParams &P, const FinJob &job, uint32_t tag, Shared &sh) {
    const UnitDesc &d = job.d;
    const UnitDec &D = job.D;
    const int lane = threadIdx.x % kWarp;
    const bool pair = d.kind == U_PAIR;
    int st = D.status;
    float alpha = 0.0f, Zres = 0.0f;
    const bool rule2_pair = pair && !d.greedy && st == 0;
    if (rule2_pair) {
        const int nrec = P.ns * kDW;
        const unsigned long long *rec = P.p2w + static_cast<size_t>(d.item) * nrec * kW2Words;
        if (!poll_units(sh, rec, nrec, kW2Words, kW2Words, tag)) {
            st |= REQ_TIMEOUT;
            sh.timed_out = 1;
        }
        // sums in record order over the lanes (the same in every lane)
        float a = 0.0f, z = 0.0f;
        for (int u = lane; u < nrec; u += kWarp) {
            a += u2f(word_val(ld_word(rec + static_cast<size_t>(u) * kW2Words + W2_ALPHA)));
            z += u2f(word_val(ld_word(rec + static_cast<size_t>(u) * kW2Words + W2_Z)));
        }
        alpha = warp_sum(a);
        Zres = warp_sum(z);
    }
    int kind = (st == 0) ? D.kind : SAMPLE_NONE;
    int fb = 0;
    if (kind == SAMPLE_RESIDUAL && !(Zres > 0.0f)) {
        kind = SAMPLE_P;  // zero residual mass: draw from p and say so
        fb = 1;
    }
    if (kind == SAMPLE_P) {
        // the draw from p reads the chunk shares of the target row (every data warp's pass-1 record)
        const int nrec = P.ns * kDW;
        if (!poll_units(sh, P.p1w + static_cast<size_t>(d.item) * nrec * kW1Words, nrec, kW1Words, kW1Words, tag)) {
            st |= REQ_TIMEOUT;
            sh.timed_out = 1;
            kind = SAMPLE_NONE;
        }
    }
    int tok = -1;
    float prob = NAN, margin = NAN;
    if (kind != SAMPLE_NONE) {
        draw_item<DT>(P, d, D, kind, tok, prob, margin);
    } else if (st == 0 && d.greedy && !(pair && D.accept)) {
        tok = D.argmax_t;  // Rule 1: the correction (or the extra token) is argmax p
        prob = 1.0f;
    }
    if (lane == 0) {
        const int item = d.item;
        P.item_status[item] = st;
        P.item_fb[item] = fb;
        P.item_tok[item] = tok;
        P.item_prob[item] = prob;
        P.item_margin[item] = margin;
        if (pair) {
            const float a = d.greedy ? D.alpha_g : alpha;
            P.item_flag[item] = (st == 0) ? D.accept : 0;
            P.alpha_ws[d.drow] = (st == 0) ? a : 0.0f;
            if (P.alpha_rows) P.alpha_rows[d.drow] = (st == 0) ? a : NAN;
            if (P.rho_rows) P.rho_rows[d.drow] = (st == 0) ? D.rho : NAN;
            if (P.resid_rows)
                P.resid_rows[d.drow] = (st == 0 && D.kind == SAMPLE_RESIDUAL && !d.greedy) ? Zres : -1.0f;
        } else {
            P.item_flag[item] = 0;
        }
        __threadfence();
    }
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(P.req_cnt + d.req, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    if (static_cast<int>(old) == d.K) {
        __threadfence();
        select_request(P, d.req);
        __threadfence();
    }
}

// ------------------------------------------------------------------------------------------------
// the last CTA: the batch's alpha sum and depth counts, then (a round) compaction and gamma

__device__ __noinline__ void batch_tail(const SliceParams &P, Shared &sh, unsigned char *scratch) {
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    float *red_hi = reinterpret_cast<float *>(scratch);
    float *red_lo = red_hi + kNumWarps;
    int *red_n = reinterpret_cast<int *>(red_lo + kNumWarps);
    int *hist_r = red_n + kNumWarps;
    int *hist_a = hist_r + 64;
    CompactScratch<kBlock> *cs = reinterpret_cast<CompactScratch<kBlock> *>(scratch + 4096);
    const bool bad_off = sh.bad_offsets != 0;
    for (int j = tid; j < 64; j += kBlock) hist_r[j] = hist_a[j] = 0;
    __syncthreads();
    // requests whose selection never ran: bad offsets (BAD_SHAPE) or a wait that gave up
    F2 asum = {0.0f, 0.0f};
    int acnt = 0;
    for (int i = tid; i < P.B; i += kBlock) {
        const int r0 = __ldg(P.row_off + i), r1 = __ldg(P.row_off + i + 1);
        const int K = r1 - r0 - 1;
        const bool done = !bad_off && K >= 0 && __ldcg(P.req_cnt + i) == static_cast<uint32_t>(K + 1);
        if (!done) {
            const int status = bad_off ? SPEC_REQ_BAD_SHAPE : REQ_TIMEOUT;
            if (!bad_off || (K >= 0 && r0 >= 0 && r1 <= P.total_rows))
                for (int j = 0; j <= K; ++j) P.out_tokens[r0 + j] = -1;
            P.req_status[i] = status;
            P.accept_len[i] = 0;
            if (P.n_emitted) P.n_emitted[i] = 0;
            if (P.frontier_prob) P.frontier_prob[i] = NAN;
            if (P.frontier_margin) P.frontier_margin[i] = NAN;
            if (P.fallback) P.fallback[i] = 0;
            continue;
        }
        if (__ldcg(P.req_status + i) != 0) continue;
        const float2 ra = __ldcg(P.req_alpha + i);
        asum = f2_add(asum, {ra.x, ra.y});
        acnt += K;
        const int A = __ldcg(P.accept_len + i);
        // depth j + 1 was reached when the first j drafts were accepted, accepted when j < A
        for (int j = 0; j < K; ++j) {
            if (j <= A) atomicAdd(&hist_r[j], 1);
            if (j < A) atomicAdd(&hist_a[j], 1);
        }
    }
    asum = warp_sum_f2(asum);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acnt += __shfl_xor_sync(0xffffffffu, acnt, o);
    if (lane == 0) {
        red_hi[warp] = asum.hi;
        red_lo[warp] = asum.lo;
        red_n[warp] = acnt;
    }
    __syncthreads();
    if (warp == 0) {
        F2 a = lane < kNumWarps ? F2{red_hi[lane], red_lo[lane]} : F2{0.0f, 0.0f};
        int c = lane < kNumWarps ? red_n[lane] : 0;
        a = warp_sum_f2(a);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
        if (lane == 0) {
            // the one float64 operation of the call: the pair becomes the output double
            if (P.alpha_sum) *P.alpha_sum = static_cast<double>(a.hi) + static_cast<double>(a.lo);
            if (P.alpha_count) *P.alpha_count = c;
        }
    }
    for (int j = tid; j < P.K_max; j += kBlock) {
        if (P.depth_reached) P.depth_reached[j] = hist_r[j];
        if (P.depth_accepted) P.depth_accepted[j] = hist_a[j];
    }
    __threadfence();
    __syncthreads();
    if (P.round) {
        compact_body<kBlock>(P.C, false,
                             (P.C.row_off == P.row_off && P.C.B == P.B && P.C.total_rows == P.total_rows) ? (bad_off ? 0 : 1)
                                                                                                         : -1,
                             *cs);
        __syncthreads();
        if (tid == 0) gamma_body(P.G);
    }
    // the workspace's counters back to zero and the next epoch, for the next call
    for (int i = tid; i < P.B; i += kBlock) P.req_cnt[i] = 0u;

    if (tid == 0) {
        P.ctl[CTL_DONE] = 0u;
        P.ctl[CTL_EPOCH] = sh.epoch + 1u;
    }
}

// ------------------------------------------------------------------------------------------------
// the kernel

// Request of target row g: the i with row_off[i] <= g < row_off[i + 1] (offsets checked).
__device__ __forceinline__ int find_request(const SliceParams &P, const Shared &sh, int g, int &r0, int &r1) {
    int lo = 0, hi = P.B - 1;
    if (sh.staged) {
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sh.roff[mid] <= g) lo = mid; else hi = mid - 1;
        }
        r0 = sh.roff[lo];
        r1 = sh.roff[lo + 1];
    } else {
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(P.row_off + mid) <= g) lo = mid; else hi = mid - 1;
        }
        r0 = __ldg(P.row_off + lo);
        r1 = __ldg(P.row_off + lo + 1);
    }
    return lo;
}

// The CTA's shared memory: the slots (dynamic) and the shared state (static), at file scope so
// that every role's function addresses them as shared memory.
extern __shared__ __align__(128) unsigned char s_dyn[];
__shared__ Shared s_sh;

// Whether unit d has pass 2: a pair under Rule 2 (alpha and the residual need the item's
// normalisers, so its slices are read again once every unit of the item is through pass 1).
__device__ __forceinline__ bool has_p2(const UnitDesc &d) { return d.kind == U_PAIR && !d.greedy; }

// Data warps: the jobs in order (pass 1 of unit n; pass 2 of unit n - kLag), each warp its chunk
// of the slices, its record published in global memory. The CTA holding an item's designated unit
// (slice item mod ns) hands the item to its final warp: after pass 1 to be decided, after pass 2
// to be finalised.
template <int DT>
__device__ __noinline__ void role_data(const SliceParams &P, uint32_t tag) {
    Shared &sh = s_sh;
    const uint4 *const slots = reinterpret_cast<const uint4 *>(s_dyn);
    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int vbase = warp * kChunkVecs + lane;  // this thread's first vector in a slice
    for (int j = 0;; ++j) {
        const int q = j % kJobs;
        if (!wait_bar(sh, &sh.job_full[q], static_cast<uint32_t>((j / kJobs) & 1))) break;
        const int type = sh.jobs[q].type, n = sh.jobs[q].unit;
        if (type == J_END) break;
        const int e = n % kR;
        const UnitDesc &d = sh.desc[e];
        const uint4 *ts = slots + static_cast<size_t>(2 * q) * kSliceVecs;
        const uint4 *ds = ts + kSliceVecs;
        const size_t wrec = (static_cast<size_t>(d.item) * P.ns + d.slice) * kDW + warp;  // this warp's record
        const bool hand = d.designated && warp == n % kDW;  // this warp hands the item over
        if (type == J_P1) {
            float4 r;
            if (warp * kChunkVecs >= d.nvec) {
                // this warp's chunk is past the end of a short last slice
                r = d.greedy ? make_float4(-INFINITY, __int_as_float(INT_MAX), -INFINITY, __int_as_float(INT_MAX))
                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            } else if (d.greedy) {
                r = pass1_greedy<DT>(d, ts, ds, vbase);
            } else if (d.trunc) {
                r = pass1_cut<DT>(d, ts, ds, vbase);
            } else {
                r = pass1_body<DT, false>(d, ts, ds, vbase);
            }
            if (d.kind == U_PAIR && !d.greedy && d.xslice == d.slice)
                extract_x<DT>(d, ts, ds, vbase, P.xrec + static_cast<size_t>(d.item) * kXWords, tag);
            const float4 w = warp_p1(r, d.greedy != 0, d.kind == U_PAIR);
            store_w1(P.p1w + wrec * kW1Words, w, d.greedy != 0, d.kind == U_PAIR, tag);
            warp_arrive(&sh.job_empty[q], lane);
            if (hand) fq_push(sh, F_DECIDE, d, skip_decision(d));
            if (!has_p2(d)) warp_arrive(&sh.desc_empty[e], lane);
        } else if (type == J_P2) {
            const UnitDec D = read_decision(P, d, sh.drec[q], tag, sh);
            const float2 r2 = d.trunc ? pass2_cut<DT>(d, D, ts, ds, vbase) : pass2_body<DT, false>(d, D, ts, ds, vbase);
            const float a = warp_sum(r2.x), z = warp_sum(r2.y);
            if (lane < kW2Words) st_word(P.p2w + wrec * kW2Words + lane, f2u(lane == W2_ALPHA ? a : z), tag);
            warp_arrive(&sh.job_empty[q], lane);
            if (hand) fq_push(sh, F_FINAL, d, D);
            warp_arrive(&sh.desc_empty[e], lane);
        } else {
            // a unit without rows
            warp_arrive(&sh.job_empty[q], lane);
            if (hand) fq_push(sh, F_FINAL, d, skip_decision(d));
            warp_arrive(&sh.desc_empty[e], lane);
        }
    }
    // the last data warp to finish closes the final warp's queue (after every push of the others)
    int last = 0;
    if (lane == 0) last = atomicAdd(&sh.end_cnt, 1) == kDW - 1;
    if (__shfl_sync(0xffffffffu, last, 0)) {
        UnitDesc d = {};
        d.kind = U_END;
        fq_push(sh, F_END, d, skip_decision(d));
    }
}

// Producer warp: descriptors, and the jobs' bulk copies.
template <int DT>
__device__ __noinline__ void role_producer(const SliceParams &P, uint32_t tag) {
    Shared &sh = s_sh;
    uint4 *const slots = reinterpret_cast<uint4 *>(s_dyn);
    const int lane = threadIdx.x % kWarp;
    const int G = gridDim.x;
    constexpr int E = Elt<DT>::kPerVec;
    const size_t row_bytes = static_cast<size_t>(P.nvec_row) * 16;
    const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
    int n = 0, j = 0;  // units described, jobs issued (lane 0)
    // the next job in the ring (once the data warps have left the slot): its slices (nrows rows)
    // and, for pass 2, the item's decision record, all completing on the job's barrier
    auto issue = [&](int type, int unit, const UnitDesc &d, int nrows, uint64_t pol) {
        const int q = j % kJobs;
        if (j >= kJobs && !wait_bar(sh, &sh.job_empty[q], static_cast<uint32_t>(((j / kJobs) - 1) & 1)))
            nrows = 0, type = (type == J_END) ? J_END : J_SKIP;
        const bool drec = type == J_P2;
        sh.jobs[q].type = type;
        sh.jobs[q].unit = unit;
        const uint32_t sbytes = static_cast<uint32_t>(d.nvec) * 16u;
        const uint32_t total = (nrows > 0 ? sbytes * nrows : 0u) + (drec ? kDecWords * 8u : 0u);
        if (total) mbar_expect_tx(&sh.job_full[q], total);
        if (nrows > 0) {
            const size_t off = static_cast<size_t>(d.slice) * kSliceVecs * 16;
            uint4 *dst = slots + static_cast<size_t>(2 * q) * kSliceVecs;
            bulk_g2s(dst, static_cast<const unsigned char *>(P.target) + static_cast<size_t>(d.item) * row_bytes + off,
                     sbytes, &sh.job_full[q], pol);
            if (nrows == 2)
                bulk_g2s(dst + kSliceVecs,
                         static_cast<const unsigned char *>(P.draft) + static_cast<size_t>(d.drow) * row_bytes + off,
                         sbytes, &sh.job_full[q], pol);
        }
        if (drec)
            bulk_g2s(sh.drec[q], P.drec + static_cast<size_t>(d.item) * kDecWords, kDecWords * 8u, &sh.job_full[q], drop);
        mbar_arrive(&sh.job_full[q]);
        ++j;
    };
    // pass 2 of unit m: its slices again (from L2) and the item's decision
    auto issue_second = [&](int m) {
        const UnitDesc &dm = sh.desc[m % kR];
        if (has_p2(dm)) issue(J_P2, m, dm, 2, drop);
    };
    for (bool end = false; !end;) {
        // lanes 0 .. kPrep-1 prepare the descriptors of units n .. n + kPrep - 1 at once, so that
        // their loads overlap
        if (lane < kPrep) {
            const long long u = sh.bad_offsets ? P.nunits : static_cast<long long>(blockIdx.x) + static_cast<long long>(n + lane) * G;
            UnitDesc d = {};
            if (u >= P.nunits) {
                d.kind = U_END;
            } else {
                const int g = static_cast<int>(u / P.ns), s = static_cast<int>(u % P.ns);
                int r0, r1;
                const int i = find_request(P, sh, g, r0, r1);
                const int K = r1 - r0 - 1, pos = g - r0;
                const int drow = r0 - i + pos;
                // the item's values, every load issued before any is used
                const float T = P.temperature ? __ldg(P.temperature + i) : P.temperature_scalar;
                const float tp = P.top_p ? __ldg(P.top_p + i) : 1.0f;
                const bool shaped = K <= P.K_max;
                const double ua = (shaped && pos < K) ? __ldg(P.uniforms + g) : 0.0;
                const double us = shaped ? __ldg(P.uniforms + r0 + K) : 0.0;
                const int x = (shaped && pos < K) ? __ldg(P.draft_tokens + drow) : -1;
                const int2 cut = (P.trunc && shaped) ? __ldg(P.trunc + g) : make_int2(0, INT_MAX);
                int status = shaped ? 0 : SPEC_REQ_BAD_SHAPE;
                if (!(T >= 0.0f) || isinf(T) || isnan(tp)) status |= SPEC_REQ_BAD_PARAM;
                d.kind = status ? U_SKIP : (pos < K ? U_PAIR : U_ROW);
                d.item = g;
                d.slice = s;
                d.req = i;
                d.pos = pos;
                d.K = K;
                d.drow = drow;
                d.nvec = min(kSliceVecs, P.nvec_row - s * kSliceVecs);
                d.status = status;
                d.greedy = (T == 0.0f) ? 1 : 0;
                d.designated = (s == g % P.ns) ? 1 : 0;
                d.ua = ua;
                d.us = us;
                d.x = x;
                d.xslice = (x >= 0 && x < P.V) ? (x / E) / kSliceVecs : -1;
                F2 sv = {0.0f, 0.0f};
                if (T > 0.0f && !isinf(T)) sv = f2_div({kLog2eHi, kLog2eLo}, {T, 0.0f});
                if (sv.hi > 0.0f && sv.lo < 0.0f) {
                    // s_hi moved toward zero so that s_lo > 0: a -inf logit then gives -inf in
                    // both terms of the exponent's argument (a negative s_lo would make it NaN)
                    const float down = __uint_as_float(__float_as_uint(sv.hi) - 1u);
                    sv.lo += sv.hi - down;
                    sv.hi = down;
                }
                d.s_hi = sv.hi;
                d.s_lo = fmaxf(sv.lo, 1.401298464e-45f);
                d.cut_tau = static_cast<uint32_t>(cut.x);
                d.cut_id = cut.y;
                d.trunc = (!d.greedy && (cut.x != 0 || cut.y != INT_MAX)) ? 1 : 0;
            }
            sh.prep[lane] = d;
        }
        __syncwarp();
        if (lane == 0) {
            for (int l = 0; l < kPrep; ++l, ++n) {
                const int e = n % kR;
                const bool ok = n < kR || wait_bar(sh, &sh.desc_empty[e], static_cast<uint32_t>(((n / kR) - 1) & 1));
                UnitDesc &d = sh.desc[e];
                d = sh.prep[l];
                if (!ok || sh.timed_out) d.kind = U_END;
                mbar_arrive(&sh.desc_full[e]);
                if (d.kind == U_END) {
                    end = true;
                    break;
                }
                // pass 1 of unit n: a pair's slices stay in L2 for its pass 2 (evict last)
                if (d.kind == U_SKIP)
                    issue(J_SKIP, n, d, 0, drop);
                else
                    issue(J_P1, n, d, d.kind == U_PAIR ? 2 : 1, (d.kind == U_PAIR && !d.greedy) ? keep : drop);
                if (n >= kLag) issue_second(n - kLag);
            }
            if (end) {
                // the last units' second jobs, then the end
                for (int m = max(0, n - kLag); m < n; ++m) issue_second(m);
                issue(J_END, n, sh.desc[n % kR], 0, drop);
                // copies still in flight (a wait gave up): wait for them, bounded, before leaving
                if (sh.timed_out)
                    for (int m = max(0, j - kJobs); m < j; ++m)
                        mbar_wait_sleep_bounded(&sh.job_full[m % kJobs], static_cast<uint32_t>((m / kJobs) & 1), kSuspendNs,
                                                4);
            }
        }
        n = __shfl_sync(0xffffffffu, n, 0);
        end = __shfl_sync(0xffffffffu, end ? 1 : 0, 0) != 0;
        __syncwarp();
    }
    (void)tag;
}

// Final warp: items' decisions (each item once in the whole grid, by the CTA that counted its
// last unit through pass 1), results and draws, requests' selections.
template <int DT>
__device__ __noinline__ void role_final(const SliceParams &P, uint32_t tag) {
    Shared &sh = s_sh;
    const int lane = threadIdx.x % kWarp;
    for (int j = 0;; ++j) {
        const int q = j % kFQ;
        if (!wait_bar(sh, &sh.fq_full[q], static_cast<uint32_t>((j / kFQ) & 1))) break;
        FinJob job = sh.fq[q];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.fq_empty[q]);
        if (job.op == F_END) break;
        if (job.op == F_DECIDE) {
            job.D = decide_records(P, job.d, tag, sh);
            // the decision record, for every CTA holding a unit of the item
            unsigned long long *r = P.drec + static_cast<size_t>(job.d.item) * kDecWords;
            if (lane < kDecWords) st_word(r + lane, dec_word(job.D, lane), tag);
            if (has_p2(job.d)) continue;  // finalised after pass 2
        }
        finalize_item<DT>(P, job, tag, sh);
    }
    __threadfence();
}

template <int DT>
__global__ void __maxnreg__(kMaxRegs) spec_slice_kernel(const __grid_constant__ SliceParams P) {
    Shared &sh = s_sh;
    const int tid = threadIdx.x, warp = tid / kWarp, lane = tid % kWarp;
    const int G = gridDim.x;

    if (tid == 0) {
        for (int k = 0; k < kR; ++k) {
            mbar_init(&sh.desc_full[k], 1);
            mbar_init(&sh.desc_empty[k], kDW);
        }
        for (int k = 0; k < kJobs; ++k) {
            mbar_init(&sh.job_full[k], 1);
            mbar_init(&sh.job_empty[k], kDW);
        }
        for (int k = 0; k < kFQ; ++k) {
            mbar_init(&sh.fq_full[k], 1);
            mbar_init(&sh.fq_empty[k], 1);
        }
        sh.fq_tail = 0;
        sh.end_cnt = 0;
        fence_mbar_init();
        sh.timed_out = 0;
        sh.last_cta = 0;
        const uint32_t epoch = ld_u32_relaxed(P.ctl + CTL_EPOCH);
        sh.epoch = epoch;
        sh.tag = epoch % 0x7fffffffu + 1u;  // never 0, the value of a zeroed workspace
    }
    // row offsets: checked by every CTA (start at 0, end at total_rows, grow by at least one row),
    // staged in shared memory when they fit
    const bool staged = P.B < kStage;
    int bad = 0;
    for (int i = tid; i <= P.B; i += kBlock) {
        const int v = __ldg(P.row_off + i);
        if (staged) sh.roff[i] = v;
        if (i == 0 && v != 0) bad = 1;
        if (i == P.B && v != P.total_rows) bad = 1;
        if (i < P.B && __ldg(P.row_off + i + 1) <= v) bad = 1;
    }
    bad = __syncthreads_or(bad);
    if (tid == 0) {
        sh.bad_offsets = bad;
        sh.staged = staged ? 1 : 0;
    }
    __syncthreads();
    const uint32_t tag = sh.tag;

    // each role in a function of its own (its own register allocation)
    if (warp < kDW)
        role_data<DT>(P, tag);
    else if (warp == W_PROD)
        role_producer<DT>(P, tag);
    else if (warp == W_FINAL)
        role_final<DT>(P, tag);

    // ================= the last CTA: batch-level results, compaction, gamma, reset ===================
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(P.ctl + CTL_DONE, 1u);
        sh.last_cta = (done == static_cast<uint32_t>(G - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (sh.last_cta) {
        __threadfence();
        batch_tail(P, sh, s_dyn);
    }
}

}  // namespace slice
}  // namespace spec
