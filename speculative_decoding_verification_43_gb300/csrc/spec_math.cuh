// Arithmetic helpers of the verifier kernels: logit vectors, float-pair sums, exact scaling by
// powers of two, and the packed (two-lane float32) exponent arguments used by every pass.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "spec_device.cuh"
#include "spec_verify.h"

namespace spec {

// One 16-byte vector of logits, unpacked to float pairs in token order.
template <int DT>
struct Elt;
template <>
struct Elt<SPEC_F32> {
    static constexpr int kPerVec = 4;
    __device__ static __forceinline__ void unpack2(const uint4 &w, float2 *y) {
        y[0] = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
        y[1] = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
    // the float pair of 32-bit word pair h (elements 2h, 2h + 1)
    __device__ static __forceinline__ float2 unpack_one(const uint4 &w, int h) {
        return h == 0 ? make_float2(__uint_as_float(w.x), __uint_as_float(w.y))
                      : make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
    }
    __device__ static __forceinline__ float at(const uint4 *buf, int e) {
        return reinterpret_cast<const float *>(buf)[e];
    }
    __device__ static __forceinline__ float vmax(const uint4 &w) {
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                     fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
};
template <>
struct Elt<SPEC_BF16> {
    static constexpr int kPerVec = 8;
    // bfloat16 is the upper half of a binary32: widening is a shift or a mask. The element at
    // the lower address is the low half of each 32-bit word.
    __device__ static __forceinline__ void unpack2(const uint4 &w, float2 *y) {
        y[0] = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
        y[1] = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
        y[2] = make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
        y[3] = make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
    }
    // the float pair of 32-bit word h (elements 2h, 2h + 1)
    __device__ static __forceinline__ float2 unpack_one(const uint4 &w, int h) {
        const uint32_t x = h == 0 ? w.x : h == 1 ? w.y : h == 2 ? w.z : w.w;
        return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
    }
    __device__ static __forceinline__ float at(const uint4 *buf, int e) {
        const uint16_t b = reinterpret_cast<const uint16_t *>(buf)[e];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    // NaN is ignored here (max.bf16x2 returns the other operand); the sums catch it later
    __device__ static __forceinline__ float vmax(const uint4 &w) {
        const uint32_t m = bf16x2_max(bf16x2_max(w.x, w.y), bf16x2_max(w.z, w.w));
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
};

// A vector of -inf logits (the bit patterns of -inf in either type).
template <int DT>
__device__ __forceinline__ uint4 kNegInfVec() {
    const uint32_t w = (DT == SPEC_BF16) ? 0xff80ff80u : 0xff800000u;
    return make_uint4(w, w, w, w);
}

// A 16-byte vector of a slice, or -inf past its end (no mass, never a maximum).
template <int DT>
__device__ __forceinline__ void load_vec2(const uint4 *buf, int vi, int nvec, float2 *y) {
    constexpr int H = Elt<DT>::kPerVec / 2;
    if (vi < nvec) {
        Elt<DT>::unpack2(buf[vi], y);
    } else {
#pragma unroll
        for (int h = 0; h < H; ++h) y[h] = make_float2(-INFINITY, -INFINITY);
    }
}

__device__ __forceinline__ float2 f2splat(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 ex2x2(float2 a) { return make_float2(ex2(a.x), ex2(a.y)); }

// y*s - b for a pair of logits, s = s_hi + s_lo with s_lo > 0: the product with s_hi and the
// subtraction of b round once (to the small result), then the s_lo term is added. -inf stays
// -inf. Both lanes round exactly as two scalar fmaf would.
__device__ __forceinline__ float2 exp_arg2(float2 y, float2 s_hi, float2 s_lo, float2 neg_b) {
    return __ffma2_rn(y, s_lo, __ffma2_rn(y, s_hi, neg_b));
}

// 2^k for an integral k (as float): exact for k >= -126, 0 below, +inf above 127.
__device__ __forceinline__ float pow2i(float k) {
    if (!(k >= -126.0f)) return 0.0f;
    if (k > 127.0f) return INFINITY;
    return __int_as_float((static_cast<int>(k) + 127) << 23);
}
// ---- two-float values hi + lo (about 48 significant bits), for sums that need more than
// float32: float64 runs at a small fraction of the float32 rate on this part.
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
__device__ __forceinline__ bool f2_gt(F2 a, F2 b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) { return f2_add(a, {-b.hi, -b.lo}); }
__device__ __forceinline__ F2 f2_norm(float hi, float lo) {
    const float s = hi + lo;
    return {s, lo - (s - hi)};
}
// a * b, the product of the high parts exact (fma), the cross terms to first order
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
    const float p = a.hi * b.hi;
    const float e = fmaf(a.hi, b.hi, -p) + (a.hi * b.lo + a.lo * b.hi);
    return f2_norm(p, e);
}
// 1/x on the special-function unit (about 1 ulp)
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// a / b for b > 0: the quotient from an approximate reciprocal, then the quotient of the
// remainder (computed exactly with fma) corrects it to float-pair precision. No division
// instruction: an IEEE float division is a long dependent sequence on this part.
__device__ __forceinline__ F2 f2_div(F2 a, F2 b) {
    const float r = rcp_approx(b.hi);
    const float q1 = a.hi * r;
    const float e = (fmaf(-q1, b.hi, a.hi) + a.lo) - q1 * b.lo;
    return f2_norm(q1, e * r);
}
// The value of a double as a float pair (about 48 bits), with integer operations only: the
// float64 instructions and conversions are very slow on this part. Values below 2^-126 read
// as 0; infinities and NaN go to hi.
__device__ __forceinline__ F2 d2f2(double x) {
    const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(x));
    const int ex = static_cast<int>((b >> 52) & 0x7ff);
    const float sgn = (b >> 63) ? -1.0f : 1.0f;
    if (ex == 0x7ff) return {sgn * ((b & 0xfffffffffffffull) ? NAN : INFINITY), 0.0f};
    const int e = ex - 1023;
    if (e < -126) return {0.0f, 0.0f};
    const unsigned long long full = (1ull << 52) | (b & 0xfffffffffffffull);
    const float hi = static_cast<float>(static_cast<uint32_t>(full >> 29)) * pow2i(static_cast<float>(e - 23));
    const float lo = static_cast<float>(static_cast<uint32_t>(full & ((1u << 29) - 1))) *
                     pow2i(static_cast<float>(e - 52));
    return f2_norm(sgn * hi, sgn * lo);
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
// inclusive scan over the lanes, in lane order
__device__ __forceinline__ F2 warp_scan_f2(F2 v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        F2 w;
        w.hi = __shfl_up_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_up_sync(0xffffffffu, v.lo, o);
        if (lane >= o) v = f2_add(w, v);
    }
    return v;
}
__device__ __forceinline__ F2 shfl_f2(F2 v, int src) {
    return {__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// log2(2^B * S) for S >= 1 a float pair and B integral, as an integral part (exact) and a
// fraction in [0, 1): the exponent of S.hi is split off exactly, the logarithm of its mantissa
// in [1, 2) is taken on the special-function unit (absolute error about 2^-22), and S.lo enters
// to first order. The error does not grow with the size of S.
__device__ __forceinline__ float2 log2_split(F2 S, float B) {
    const int bits = __float_as_int(S.hi);
    const int ex = ((bits >> 23) & 0xff) - 127;
    const float m = __int_as_float((bits & 0x007fffff) | 0x3f800000);
    const float frac = __log2f(m) + S.lo * rcp_approx(S.hi) * 1.44269504f;
    return make_float2(B + static_cast<float>(ex), frac);
}

__device__ __forceinline__ F2 f2_scale(F2 a, float k) {
    const float m = pow2i(k);
    return {a.hi * m, a.lo * m};
}

// ---- order-preserving integer keys of logits (a larger logit has a larger key; NaN sorts
// outside the finite range) and the top-k / top-p cut: token v is kept when its key is above
// tau, or equal to it with v <= id (ties rank by ascending token id).
__device__ __forceinline__ uint32_t key_bf16(uint32_t b) { return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u); }
__device__ __forceinline__ uint32_t key_f32(uint32_t u) { return (u & 0x80000000u) ? ~u : (u | 0x80000000u); }
__device__ __forceinline__ bool cut_keeps(uint32_t key, int v, uint32_t tau, int id) {
    return key > tau || (key == tau && v <= id);
}

}  // namespace spec
