// spec_trunc_kernel: top-k, then top-p, of each target row's law (included once, by
// spec_verify.cu).
//
// SDCP, section "Session Model": p is the target model's next-token distribution after
// temperature, top-k and top-p, in that order (the draft's q is not truncated). Tokens rank by
// logit, ties by ascending id; top-k keeps the first k; top-p then keeps the shortest head of
// the law renormalised over the top-k set whose mass reaches top_p. The kept set of a row is a
// prefix of that ranking, so it is one cut: token v is kept when key(v) > tau, or key(v) == tau
// and v <= id, with key the order-preserving integer image of the logit. The per-position
// kernel reads the cut and treats every other token of the row as a -inf logit, which is the
// truncated, renormalised law.
//
// One CTA per target row. With top-k of at most kTruncThreads tokens, two passes: each thread's
// largest key, whose k-th largest over the CTA bounds the row's top-k set from below (at least k
// tokens reach it); then every token at or above that bound is gathered into shared memory and
// sorted (bitonic, by key then id), which gives the top-k cut exactly and, for top-p, the masses
// of the top-k set in rank order for a prefix scan. Otherwise (no top-k, a larger k, or more
// candidates than fit): a radix select over the key, eight bits per pass, on counts (top-k) or
// on masses (top-p), then an ordered search among the tokens tied at the cut. Masses are
// 2^((z - z_max) s) in fixed point (2^-40 units, 64-bit integer sums): the sums, and so the cut,
// do not depend on the order of the atomic additions. Rows are read as 16-byte vectors; a row
// stays in L2 across its passes (bf16 V = 128256: about six passes over 256 KB).
#pragma once

#include <climits>
#include <cstdint>

#include "spec_device.cuh"
#include "spec_math.cuh"

namespace spec {

constexpr int kTruncThreads = 512;
constexpr int kTruncWarps = kTruncThreads / kWarp;
// the cut that keeps every token (every key is >= 0)
constexpr uint32_t kCutAllTau = 0u;
constexpr int32_t kCutAllId = INT_MAX;

struct TruncParams {
    const void *target;
    const int32_t *row_off;
    const float *temperature;
    float temperature_scalar;
    const int32_t *top_k;  // [B] or NULL
    const float *top_p;    // [B] or NULL
    int32_t B, V, total_rows;
    int2 *cut;             // [T] (tau, id) per target row
};

__device__ __forceinline__ float logit_of_key_bf16(uint32_t k) {
    const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return __uint_as_float(b << 16);
}
__device__ __forceinline__ float logit_of_key_f32(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

template <int DT>
struct TruncElt;
template <>
struct TruncElt<SPEC_BF16> {
    static constexpr int kBits = 16, kPerVec = 8;
    // key of element e of a 16-byte vector
    __device__ static __forceinline__ uint32_t key(const uint4 &w, int e) {
        const uint32_t x = (e >> 1) == 0 ? w.x : (e >> 1) == 1 ? w.y : (e >> 1) == 2 ? w.z : w.w;
        return key_bf16((e & 1) ? (x >> 16) : (x & 0xFFFFu));
    }
    __device__ static __forceinline__ float logit(uint32_t k) { return logit_of_key_bf16(k); }
};
template <>
struct TruncElt<SPEC_F32> {
    static constexpr int kBits = 32, kPerVec = 4;
    __device__ static __forceinline__ uint32_t key(const uint4 &w, int e) {
        return key_f32(e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w);
    }
    __device__ static __forceinline__ float logit(uint32_t k) { return logit_of_key_f32(k); }
};

// f(v, key) for every token of the row, each thread taking 16-byte vectors t, t + 512, ...
// (rows are 16-byte multiples).
template <int DT, class F>
__device__ __forceinline__ void for_each_key(const uint4 *row, int nv, int tid, F f) {
    constexpr int E = TruncElt<DT>::kPerVec;
    for (int i = tid; i < nv; i += kTruncThreads) {
        const uint4 w = __ldg(row + i);
#pragma unroll
        for (int e = 0; e < E; ++e) f(i * E + e, TruncElt<DT>::key(w, e));
    }
}

constexpr int kCandCap = 4096;  // candidates the two-pass top-k path holds (a power of two)

// Shared state of one row's selection.
struct TruncShared {
    unsigned long long cand[kCandCap];  // (key << 32) | (0xFFFFFFFF - id): larger ranks first
    uint32_t tmax[kTruncThreads];   // each warp's 32 thread maxima, sorted descending
    uint32_t bound;
    unsigned long long scan[kTruncWarps];
    uint32_t ncand;
    uint32_t hist[256];
    unsigned long long hmass[256];
    uint32_t wsum[kTruncWarps];
    uint32_t kmax;
    int32_t req, found;
    uint32_t chosen;
    unsigned long long need;
};


// Block-wide max of a key (every thread gets it).
__device__ __forceinline__ uint32_t block_max_u32(TruncShared &sh, uint32_t v, int tid) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (tid == 0) sh.kmax = 0u;
    __syncthreads();
    if ((tid & 31) == 0) atomicMax(&sh.kmax, v);
    __syncthreads();
    const uint32_t r = sh.kmax;
    __syncthreads();
    return r;
}

// Radix select from the top of the key order, eight bits per pass: the key tau at which the
// running total (counts when MASS is false, fixed-point masses otherwise) of the tokens ranked
// before it first reaches `need`; on return `need` is what remains to be taken among the
// tokens tied at tau. kept(v, key) filters the tokens that take part. With tp >= 0 (masses
// only), `need` comes from the first pass: ceil(tp * total), at least 1 (the top token).
// Histogram updates are aggregated per warp over lanes that hit the same bin.
template <int DT, bool MASS, class Kept, class Mass>
__device__ uint32_t radix_select(TruncShared &sh, const uint4 *row, int nv, unsigned long long &need, Kept kept,
                                 Mass mass, float tp, int tid) {
    constexpr int E = TruncElt<DT>::kPerVec;
    const int lane = tid & 31;
    uint32_t prefix = 0u, pmask = 0u;
    bool first = true;
    for (int shift = TruncElt<DT>::kBits - 8; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += kTruncThreads) {
            sh.hist[b] = 0u;
            sh.hmass[b] = 0ull;
        }
        __syncthreads();
        for (int base = tid & ~31; base < nv; base += kTruncThreads) {  // warp-uniform
            const int i = base + lane;
            const bool ok = i < nv;
            const uint4 w = ok ? __ldg(row + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const uint32_t k = TruncElt<DT>::key(w, e);
                const bool in = ok && (k & pmask) == prefix && kept(i * E + e, k);
                const uint32_t bin = in ? ((k >> shift) & 0xFFu) : 256u;
                const unsigned grp = __match_any_sync(0xffffffffu, bin);
                const bool leader = lane == __ffs(grp) - 1;
                if (MASS) {
                    // a mass is below 2^41: two 20-bit halves sum over 32 lanes without overflow
                    const unsigned long long m = in ? mass(k) : 0ull;
                    const unsigned hi = __reduce_add_sync(grp, static_cast<unsigned>(m >> 20));
                    const unsigned lo = __reduce_add_sync(grp, static_cast<unsigned>(m & 0xFFFFFull));
                    if (leader && bin < 256u)
                        atomicAdd(&sh.hmass[bin], (static_cast<unsigned long long>(hi) << 20) + lo);
                } else if (leader && bin < 256u) {
                    atomicAdd(&sh.hist[bin], static_cast<unsigned>(__popc(grp)));
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            if (MASS && first && tp >= 0.0f) {
                unsigned long long total = 0ull;
                for (int b = 0; b < 256; ++b) total += sh.hmass[b];
                need = 1ull;
                if (tp > 0.0f) {
                    const double t = ceil(static_cast<double>(tp) * static_cast<double>(total));
                    need = t < 1.0 ? 1ull : (t > static_cast<double>(total) ? total : static_cast<unsigned long long>(t));
                }
            }
            unsigned long long cum = 0ull, h_last = 0ull;
            int chosen = -1, last = 0;
            for (int b = 255; b >= 0; --b) {
                const unsigned long long h = MASS ? sh.hmass[b] : static_cast<unsigned long long>(sh.hist[b]);
                if (h == 0ull) continue;
                if (cum + h >= need) {
                    chosen = b;
                    break;
                }
                cum += h;
                last = b;
                h_last = h;
            }
            if (chosen >= 0) {
                sh.chosen = static_cast<uint32_t>(chosen);
                sh.need = need - cum;
            } else {
                // the total falls short of `need` (it can only by rounding): every token counts,
                // down to the lowest bin that holds any
                sh.chosen = static_cast<uint32_t>(last);
                sh.need = h_last;
            }
        }
        __syncthreads();
        prefix |= sh.chosen << shift;
        pmask |= 0xFFu << shift;
        need = sh.need;
        first = false;
        __syncthreads();
    }
    return prefix;
}

// The n-th (1-based) token in id order among those with key == tau that pass kept(v, key);
// -1 if there are fewer. Warp w scans the w-th contiguous run of vectors, 32 at a time.
template <int DT, class Kept>
__device__ int nth_tied(TruncShared &sh, const uint4 *row, int nv, uint32_t tau, uint32_t n, Kept kept, int tid) {
    constexpr int E = TruncElt<DT>::kPerVec;
    const int lane = tid & 31, wp = tid >> 5;
    const int cw = (nv + kTruncWarps - 1) / kTruncWarps;
    const int v0 = min(nv, wp * cw), v1 = min(nv, v0 + cw);
    auto ties = [&](int i, const uint4 &w) {
        uint32_t c = 0u;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const uint32_t k = TruncElt<DT>::key(w, e);
            c += (k == tau && kept(i * E + e, k)) ? 1u : 0u;
        }
        return c;
    };
    uint32_t c = 0u;
    for (int i = v0 + lane; i < v1; i += 32) c += ties(i, __ldg(row + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) sh.wsum[wp] = c;
    if (tid == 0) sh.found = -1;
    __syncthreads();
    uint32_t before = 0u;
    for (int k = 0; k < wp; ++k) before += sh.wsum[k];
    if (before < n && n <= before + c) {  // warp-uniform: this warp's run holds the n-th
        uint32_t seen = before;
        for (int base = v0; base < v1; base += 32) {
            const int i = base + lane;
            const bool ok = i < v1;
            const uint4 w = ok ? __ldg(row + i) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t mine = ok ? ties(i, w) : 0u;
            uint32_t incl = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += x;
            }
            const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
            if (seen + total >= n) {
                const uint32_t r = n - seen;  // 1-based rank within these 32 vectors
                if (mine > 0u && incl - mine < r && r <= incl) {
                    uint32_t left = r - (incl - mine);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const uint32_t k = TruncElt<DT>::key(w, e);
                        if (k == tau && kept(i * E + e, k) && --left == 0u) {
                            sh.found = i * E + e;
                            break;
                        }
                    }
                }
                break;
            }
            seen += total;
        }
    }
    __syncthreads();
    const int r = sh.found;
    __syncthreads();
    return r;
}

struct KeepAll {
    __device__ bool operator()(int, uint32_t) const { return true; }
};
// a cut (tau, id): the tokens ranked no later than it
struct KeepCut {
    uint32_t tau;
    int32_t id;
    __device__ bool operator()(int v, uint32_t k) const { return cut_keeps(k, v, tau, id); }
};
struct NoMass {
    __device__ unsigned long long operator()(uint32_t) const { return 0ull; }
};
// 2^((z - z_max) s) in units of 2^-40 (the top token weighs 2^40)
template <int DT>
struct FixedMass {
    float zmax, s;
    __device__ unsigned long long operator()(uint32_t k) const {
        const float m = ex2((TruncElt<DT>::logit(k) - zmax) * s);
        return __float2ull_rn(m * 0x1p40f);
    }
};

// Sorts a[0 .. n) (n a power of two, at most kCandCap) into descending order, the whole CTA.
template <class T>
__device__ __forceinline__ void bitonic_desc(T *a, int n, int tid) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n / 2; i += kTruncThreads) {
                // the pair (lo, lo + stride) of comparator i
                const int lo = 2 * stride * (i / stride) + (i % stride);
                const int hi = lo + stride;
                const bool desc = ((lo & size) == 0);
                const T x = a[lo], y = a[hi];
                if (desc ? (x < y) : (x > y)) {
                    a[lo] = y;
                    a[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

// Block-wide inclusive scan of one value per thread (every thread gets its prefix and the total).
__device__ __forceinline__ unsigned long long block_scan_u64(TruncShared &sh, unsigned long long v, int tid,
                                                             unsigned long long &total) {
    const int lane = tid & 31, wp = tid >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.scan[wp] = x;
    __syncthreads();
    unsigned long long before = 0ull;
    total = 0ull;
    for (int w = 0; w < kTruncWarps; ++w) {
        const unsigned long long t = sh.scan[w];
        if (w < wp) before += t;
        total += t;
    }
    __syncthreads();
    return before + x;
}

// The two-pass cut for top-k with k <= kTruncThreads (then top-p over the top-k set when use_p).
// Returns false, with nothing written, when the candidates at or above the bound exceed
// kCandCap (many tokens tied near the k-th key); the radix path then takes the row.
template <int DT>
__device__ bool cut_small_k(TruncShared &sh, const uint4 *row, int nv, int k, bool use_p, float tp, float T,
                            int tid, int2 &cut) {
    constexpr int E = TruncElt<DT>::kPerVec;
    const int lane = tid & 31;
    // pass 1: each thread's largest key (the key of its largest logit, NaN ignored: a row holding
    // a NaN is invalid whatever its cut); four loads in flight per thread
    float mx = -INFINITY;
    bool any = false;
    for (int i0 = tid; i0 < nv; i0 += 4 * kTruncThreads) {
        uint4 w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = i0 + q * kTruncThreads;
            w[q] = i < nv ? __ldg(row + i) : kNegInfVec<DT>();
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) mx = fmaxf(mx, Elt<DT>::vmax(w[q]));
        any = true;
    }
    uint32_t mk = any ? (DT == SPEC_BF16 ? key_bf16(__float_as_uint(mx) >> 16) : key_f32(__float_as_uint(mx))) : 0u;
    // each warp sorts its 32 maxima (descending, by shuffles); then the k-th largest of all 512
    // is the value with fewer than k larger and at least k not smaller, found by binary searches
    // in the 16 sorted lists
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, mk, stride);
            const bool lower = (lane & stride) == 0;   // this lane holds the pair's first slot
            const bool desc = (lane & size) == 0;      // this run sorts descending
            const uint32_t hi = max(mk, o), lo = min(mk, o);
            mk = (lower == desc) ? hi : lo;
        }
    }
    const int wp = tid >> 5;
    sh.tmax[wp * 32 + lane] = mk;
    if (tid == 0) {
        sh.ncand = 0u;
        sh.bound = 0u;
    }
    __syncthreads();
    {
        uint32_t gt = 0u, ge = 0u;  // values > mk and >= mk over all lists
        for (int l = 0; l < kTruncWarps; ++l) {
            const uint32_t *a = sh.tmax + l * 32;
            int lo = 0, hi = 32;  // count of a[j] > mk (a descending)
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (a[mid] > mk) lo = mid + 1; else hi = mid;
            }
            gt += static_cast<uint32_t>(lo);
            hi = 32;              // count of a[j] >= mk
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (a[mid] >= mk) lo = mid + 1; else hi = mid;
            }
            ge += static_cast<uint32_t>(lo);
        }
        if (gt < static_cast<uint32_t>(k) && static_cast<uint32_t>(k) <= ge) sh.bound = mk;  // the same value
    }
    __syncthreads();
    // at least k tokens (the k largest thread maxima) have a key >= L
    const uint32_t L = sh.bound;
    // pass 2: every token with key >= L, appended warp by warp; a vector whose largest logit lies
    // below L's is skipped whole (a NaN never reaches L: NaN compares false)
    const float Lz = TruncElt<DT>::logit(L);
    for (int base = tid & ~31; base < nv; base += 2 * kTruncThreads) {  // warp-uniform
        uint4 w2[2];
        bool ok2[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = base + q * kTruncThreads + lane;
            ok2[q] = i < nv;
            w2[q] = ok2[q] ? __ldg(row + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int i = base + q * kTruncThreads + lane;
            const uint4 w = w2[q];
            const bool ok = ok2[q];
            if (!__any_sync(0xffffffffu, ok && Elt<DT>::vmax(w) >= Lz)) continue;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const uint32_t key = TruncElt<DT>::key(w, e);
                const bool in = ok && key >= L;
                const unsigned m = __ballot_sync(0xffffffffu, in);
                if (m == 0u) continue;
                uint32_t at = 0u;
                if (lane == __ffs(m) - 1) at = atomicAdd(&sh.ncand, static_cast<uint32_t>(__popc(m)));
                at = __shfl_sync(0xffffffffu, at, __ffs(m) - 1) + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
                if (in && at < static_cast<uint32_t>(kCandCap)) {
                    const uint32_t id = static_cast<uint32_t>(i * E + e);
                    sh.cand[at] = (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - id);
                }
            }
        }
    }
    __syncthreads();
    const int n = static_cast<int>(sh.ncand);
    if (n > kCandCap) return false;  // uniform across the CTA
    if (n <= kTruncThreads) {
        // rank by counting (the candidates are distinct): thread t places candidate t
        const unsigned long long c = tid < n ? sh.cand[tid] : 0ull;
        int rank = 0;
        for (int j = 0; j < n; ++j) rank += sh.cand[j] > c ? 1 : 0;
        __syncthreads();
        if (tid < n) sh.cand[rank] = c;
        __syncthreads();
    } else {
        int np = 1;
        while (np < n) np <<= 1;
        for (int j = n + tid; j < np; j += kTruncThreads) sh.cand[j] = 0ull;  // ranks below every token
        __syncthreads();
        bitonic_desc(sh.cand, np, tid);
    }
    // the top-k set is cand[0 .. k): key, then id, descending rank
    const unsigned long long ck = sh.cand[k - 1];
    cut = make_int2(static_cast<int>(ck >> 32), static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(ck)));
    if (use_p) {
        // masses 2^((z - z_max) s) in 2^-40 units over the top-k set, in rank order; the cut is
        // the first token whose inclusive prefix reaches ceil(tp * total) (at least the top token)
        const FixedMass<DT> fm = {TruncElt<DT>::logit(static_cast<uint32_t>(sh.cand[0] >> 32)), 1.4426950408889634f / T};
        const unsigned long long m = tid < k ? fm(static_cast<uint32_t>(sh.cand[tid] >> 32)) : 0ull;
        unsigned long long total;
        const unsigned long long incl = block_scan_u64(sh, m, tid, total);
        unsigned long long need = 1ull;
        if (tp > 0.0f) {
            const double t = ceil(static_cast<double>(tp) * static_cast<double>(total));
            need = t < 1.0 ? 1ull : (t > static_cast<double>(total) ? total : static_cast<unsigned long long>(t));
        }
        if (tid == 0) sh.found = k - 1;
        __syncthreads();
        if (tid < k && incl >= need && incl - m < need) atomicMin(&sh.found, tid);
        __syncthreads();
        const unsigned long long cp = sh.cand[sh.found];
        cut = make_int2(static_cast<int>(cp >> 32), static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(cp)));
    }
    return true;
}

template <int DT>
__global__ void __launch_bounds__(kTruncThreads) spec_trunc_kernel(const TruncParams P) {
    __shared__ TruncShared sh;
    const int tid = static_cast<int>(threadIdx.x), row = static_cast<int>(blockIdx.x);
    if (tid == 0) {
        // the request owning target row `row`: the last i with row_off[i] <= row
        int lo = 0, hi = P.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(P.row_off + mid) <= row)
                lo = mid;
            else
                hi = mid - 1;
        }
        sh.req = lo;
    }
    __syncthreads();
    const int req = sh.req, V = P.V;
    const int32_t k = P.top_k ? __ldg(P.top_k + req) : 0;
    const float tp = P.top_p ? __ldg(P.top_p + req) : 1.0f;
    const float T = P.temperature ? __ldg(P.temperature + req) : P.temperature_scalar;
    const bool use_k = k > 0 && k < V;
    const bool use_p = tp < 1.0f;  // false for NaN (the request is then invalid)
    if ((!use_k && !use_p) || !(T > 0.0f) || isinf(T)) {  // the greedy rule ignores truncation
        if (tid == 0 && SPEC_IN(row, P.total_rows, DBG_CUT)) P.cut[row] = make_int2(static_cast<int>(kCutAllTau), kCutAllId);
        return;
    }
    const int nv = V / TruncElt<DT>::kPerVec;  // rows are 16-byte multiples
    const uint4 *rowp = static_cast<const uint4 *>(P.target) + static_cast<size_t>(row) * nv;

    if (use_k && k <= kTruncThreads) {
        int2 cut;
        if (cut_small_k<DT>(sh, rowp, nv, k, use_p, tp, T, tid, cut)) {
            if (tid == 0 && SPEC_IN(row, P.total_rows, DBG_CUT)) P.cut[row] = cut;
            return;
        }
    }
    // top-k: the k-th key from the top, then the tokens tied there in id order
    KeepCut kc = {kCutAllTau, kCutAllId};
    if (use_k) {
        unsigned long long need = static_cast<unsigned long long>(k);
        const uint32_t tau = radix_select<DT, false>(sh, rowp, nv, need, KeepAll{}, NoMass{}, -1.0f, tid);
        const int id = nth_tied<DT>(sh, rowp, nv, tau, static_cast<uint32_t>(need), KeepAll{}, tid);
        kc = {tau, id};
    }
    KeepCut fc = kc;
    if (use_p) {
        // masses relative to the top token; the shortest head of the top-k set whose mass reaches
        // top_p of the set's total (the first pass of the select sums it; at least the top token)
        uint32_t kmax = 0u;
        for_each_key<DT>(rowp, nv, tid, [&](int, uint32_t key) { kmax = max(kmax, key); });
        kmax = block_max_u32(sh, kmax, tid);
        const FixedMass<DT> fm = {TruncElt<DT>::logit(kmax), 1.4426950408889634f / T};
        unsigned long long need = 1ull;
        const uint32_t tau = radix_select<DT, true>(sh, rowp, nv, need, kc, fm, tp, tid);
        const unsigned long long mt = fm(tau);
        const uint32_t n = mt > 0ull ? static_cast<uint32_t>((need + mt - 1ull) / mt) : 1u;
        const int id = nth_tied<DT>(sh, rowp, nv, tau, n, kc, tid);
        fc = {tau, id};
    }
    if (tid == 0 && SPEC_IN(row, P.total_rows, DBG_CUT)) P.cut[row] = make_int2(static_cast<int>(fc.tau), fc.id);
}

}  // namespace spec
