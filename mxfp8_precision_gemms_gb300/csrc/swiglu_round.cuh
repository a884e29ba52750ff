// Correct BF16 rounding of the SwiGLU hidden value y = g sigma(g) u ("Olmo-core
// MoE report, Section 11: MXFP8 Training", Section 11.4.1, the "SwiGLU +
// activation Q" fusion) where the fused kernel's fp32 fast value lies too close
// to a BF16 rounding midpoint for its own rounding to be trusted.
//
// The exact y is irrational for g != 0 (e^-g is transcendental), so it is
// never a midpoint, and its BF16 value is the neighbour on its side of the
// midpoint m next to the fast value.  With p = g u (exact in fp32 when no
// bound is hit: two 8-bit significands) and t = e^-|g|:
//   g > 0:  |y| = |p| / (1 + t),      |y| > m  <=>  (|p| - m) - m t > 0;
//   g < 0:  |y| = |p| t / (1 + t),    |y| > m  <=>  t (|p| - m) - m > 0.
// |p| - m is formed exactly (Knuth's TwoSum), t in float-float arithmetic
// (pairs hi + lo of fp32 numbers: Dekker's exact product by FMA, TwoSum, and
// the renormalising FastTwoSum), so each form is known to about 2^-44 of its
// terms; a form closer to zero than 2^-40 of them reports `undecided` and the
// caller takes an FP64 evaluation instead.
//
// t = e^-a, a = |g| <= 81: a = k ln 2 - r with k the nearest integer to
// a / ln 2 (ln 2 split into three fp32 parts, the first with 12 significant
// bits so k times it is exact), r = j / 64 + s with |s| <= 1/128, so
// e^-a = 2^-k e^(j/64) e^s: e^(j/64) from a 47-entry table of float-float
// constants and e^s = 1 + m, m from the Taylor series of e^s - 1 through s^6
// (the first omitted term is below 2^-52 of m) evaluated by Horner's rule.
//
// The functions are __host__ __device__ so that the resolver can be checked
// on the CPU against high-precision arithmetic; the device build uses the
// round-to-nearest intrinsics, which the compiler never fuses or reorders.
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "ff_consts.h"

namespace mxfp8 {
namespace ff {

#define MXFP8_HD __host__ __device__ __forceinline__

MXFP8_HD float add(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fadd_rn(a, b);
#else
    return a + b;
#endif
}
MXFP8_HD float sub(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fsub_rn(a, b);
#else
    return a - b;
#endif
}
MXFP8_HD float mul(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}
MXFP8_HD float fma(float a, float b, float c) {
#if defined(__CUDA_ARCH__)
    return __fmaf_rn(a, b, c);
#else
    return std::fmaf(a, b, c);
#endif
}
MXFP8_HD uint32_t bits(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    return u;
}
MXFP8_HD float from_bits(uint32_t u) {
    float x;
    memcpy(&x, &u, 4);
    return x;
}

struct F2 {
    float hi, lo;
};

// s + e = a + b exactly.
MXFP8_HD F2 two_sum(float a, float b) {
    const float s = add(a, b);
    const float bb = sub(s, a);
    return {s, add(sub(a, sub(s, bb)), sub(b, bb))};
}
// Same when |a| >= |b| (or a == 0).
MXFP8_HD F2 fast_two_sum(float a, float b) {
    const float s = add(a, b);
    return {s, sub(b, sub(s, a))};
}
// p + e = a b exactly (no underflow).
MXFP8_HD F2 two_prod(float a, float b) {
    const float p = mul(a, b);
    return {p, fma(a, b, -p)};
}
MXFP8_HD F2 add(F2 x, F2 y) {
    F2 s = two_sum(x.hi, y.hi);
    const F2 t = two_sum(x.lo, y.lo);
    s = fast_two_sum(s.hi, add(s.lo, t.hi));
    return fast_two_sum(s.hi, add(s.lo, t.lo));
}
MXFP8_HD F2 add(F2 x, float b) {
    const F2 s = two_sum(x.hi, b);
    return fast_two_sum(s.hi, add(s.lo, x.lo));
}
MXFP8_HD F2 mul(F2 x, F2 y) {
    F2 p = two_prod(x.hi, y.hi);
    p.lo = fma(x.hi, y.lo, p.lo);
    p.lo = fma(x.lo, y.hi, p.lo);
    return fast_two_sum(p.hi, p.lo);
}
MXFP8_HD F2 mul(F2 x, float b) {
    const F2 p = two_prod(x.hi, b);
    return fast_two_sum(p.hi, fma(x.lo, b, p.lo));
}
// x 2^-k for 0 <= k <= 126 (exact while the parts stay normal).
MXFP8_HD F2 scale_down(F2 x, int k) {
    const float f = from_bits(static_cast<uint32_t>(127 - k) << 23);
    return {mul(x.hi, f), mul(x.lo, f)};
}

// e^-a = E 2^-k for 0 <= a <= 81 (a exact in fp32 with at most 8
// significant bits, as every BF16 magnitude is); E in [0.7, 1.42].
MXFP8_HD F2 exp_neg(float a, int* k_out) {
    const float kf = rintf(mul(a, 1.44269504f));
    *k_out = static_cast<int>(kf);
    // r = k ln2 - a: k C1 - a is exact (a multiple of 2^-12 below 2^-1 in
    // magnitude), k C2 exact as a pair, k C3 below 2^-27
    const F2 p2 = two_prod(kf, ffc::kLn2C2);
    F2 r = two_sum(fma(kf, ffc::kLn2C1, -a), p2.hi);
    r = two_sum(r.hi, add(r.lo, add(p2.lo, mul(kf, ffc::kLn2C3))));
    // r = j/64 + s; r.hi - j/64 is exact
    const float jf = rintf(mul(r.hi, 64.f));
    const F2 s = two_sum(sub(r.hi, mul(jf, 0.015625f)), r.lo);
    // m = e^s - 1 = s (1 + s (1/2 + s (1/6 + s (1/24 + s (1/120 + s / 720)))))
    const float w5 = fma(s.hi, 1.f / 720.f, 1.f / 120.f);
    const F2 c4 = add(F2{ffc::kInv24Hi, ffc::kInv24Lo}, mul(s.hi, w5));
    const F2 c3 = add(F2{ffc::kInv6Hi, ffc::kInv6Lo}, mul(s, c4));
    const F2 c2 = add(mul(s, c3), 0.5f);
    const F2 c1 = add(mul(s, c2), 1.f);
    const F2 m = mul(s, c1);
    const int j = static_cast<int>(jf) + 23;
    const F2 ej{ffc::kExp64[j][0], ffc::kExp64[j][1]};
    return add(ej, mul(ej, m));
}

// BF16 bits of the correctly rounded g sigma(g) u, given the fp32 fast value
// y of the same product whose low 16 bits lie near 0x8000 (so that the
// rounding may hinge on the error of y: |y - g sigma(g) u| is within a few
// dozen fp32 units of y).  Requires -80 <= g, g and u finite.  Sets
// *undecided (and returns 0) when the float-float forms cannot decide or a
// range bound below is hit; the caller then evaluates in FP64.
MXFP8_HD uint32_t swiglu_round_near(float g, float u, float y, bool* undecided) {
    *undecided = false;
    const float p = mul(g, u);
    const float ap = fabsf(p), ay = fabsf(y);
    // |p| <= 2^100 keeps E (|p| - m) finite; >= 2^-80 keeps p exact and every
    // low part of the forms above fp32's subnormal range
    if (!(g >= -80.f && ap <= 0x1p100f && ap >= 0x1p-80f && ay >= 0x1p-80f && ay <= 0x1p127f)) {
        *undecided = true;
        return 0;
    }
    const uint32_t yb = bits(ay);
    const uint32_t below = yb >> 16;                        // BF16 magnitude under m
    const float m = from_bits((yb & 0xFFFF0000u) | 0x8000u);  // the midpoint
    const float a = fabsf(g);
    const F2 d = two_sum(ap, -m);                           // |p| - m exactly
    bool up;
    if (g > 0.f) {
        if (d.hi == 0.f) {
            up = false;  // |y| = m / (1 + t) < m
        } else if (a > 12.f) {
            // a nonzero |p| - m is a multiple of 2^-16 m or more, above m t
            up = d.hi > 0.f;
        } else {
            int k;
            const F2 t = exp_neg(a, &k);  // k is set before it is read below
            const F2 mt = scale_down(mul(t, m), k);
            const F2 z = add(d, F2{-mt.hi, -mt.lo});
            if (fabsf(z.hi) <= mul(mt.hi, 0x1p-40f)) {
                *undecided = true;
                return 0;
            }
            up = z.hi > 0.f;
        }
    } else {
        int k;
        const F2 t = exp_neg(a, &k);
        const F2 td = scale_down(mul(t, d), k);
        const F2 z = add(td, -m);
        if (fabsf(z.hi) <= mul(m, 0x1p-40f)) {
            *undecided = true;
            return 0;
        }
        up = z.hi > 0.f;
    }
    return ((bits(p) & 0x80000000u) >> 16) | (up ? below + 1 : below);
}

}  // namespace ff
}  // namespace mxfp8
