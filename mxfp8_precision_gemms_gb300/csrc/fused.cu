// Kernels around the quantizer on the routed MXFP8 path ("Olmo-core MoE
// report, Section 11: MXFP8 Training", Sections 11.4.1-11.4.3 and Table 25):
//
//  - dequantize_mx_kernel: x^ = s q back to BF16 (Eq. 58), for a saved MXFP8
//    activation whose consumer needs BF16, and for the routed Wgrad operands.
//  - swiglu_quant_kernel: SwiGLU of the up/gate GEMM output rounded to BF16
//    and MX-quantized rowwise in the same pass, so the BF16 hidden tensor is
//    never written (the "SwiGLU + activation Q" fusion).
//  - weighted_quant_kernel: combine backward; each dispatched row's gradient
//    is its token's output gradient times the route weight, rounded to BF16
//    and MX-quantized rowwise in the same pass (the "route weighting +
//    gradient Q" fusion).
//  - weighted_quant_tokens_kernel: the same conversion walking tokens, so
//    each token's gradient row is read once for all of its routes.
//
// The first three share the row quantizer's 128 x 128 tile walk: blockIdx.x
// is a 128-row scale tile (group-padded when offsets are given), blockIdx.y a
// 128-column tile (or the first of several); each thread owns whole 32-value
// blocks.  The token walk gives each CTA 16 tokens.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "mx_common.cuh"
#include "ptx.cuh"
#include "swiglu_round.cuh"

namespace mxfp8 {

__device__ unsigned int g_status_fused = 0;

namespace {

__device__ __forceinline__ void record_status(unsigned code) {
    atomicCAS(&g_status_fused, 0u, code);
}

// Rows [begin, end) of row tile blockIdx.x.  Grouped: the tile's group is
// looked up from the offsets (validated; a violation is recorded once and
// every CTA returns false).  Returns false when the CTA has nothing to do.
template <bool GROUPED>
__device__ __forceinline__ bool tile_rows(const int32_t* offsets, int groups, int64_t rows,
                                          int64_t* begin, int64_t* end) {
    const int64_t rt = blockIdx.x;
    if constexpr (GROUPED) {
        __shared__ int64_t s_rows[2];
        __shared__ int s_ok;
        if (threadIdx.x < 32) locate_group_tile(offsets, groups, rows, rt, s_rows, &s_ok);
        __syncthreads();
        if (!s_ok) {
            if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
                record_status(MXFP8_ERR_DEVICE_CHECK);
            return false;
        }
        *begin = s_rows[0];
        *end = s_rows[1];
        return *begin >= 0;
    } else {
        *begin = rt * kTile;
        *end = min(rows, *begin + kTile);
        return true;
    }
}

// --------------------------------------------------------- dequantize --

// 2^(byte - 127) as fp32: byte 0 is the subnormal 2^-127, byte 255 is NaN.
__device__ __forceinline__ float e8m0_value(uint32_t byte) {
    if (byte == 0u) return __uint_as_float(0x00400000u);
    if (byte == 0xFFu) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(byte << 23);
}

// Two E4M3 codes (low byte first) times s, rounded to BF16 (low half first).
// E4M3 -> f16 is exact, and q * 2^k is exact in fp32 for every E4M3 q and
// |k| <= 127 (4 significant bits, 2^-136 <= |q s| < 2^136, overflow -> Inf),
// so the one rounding is the final fp32 -> BF16 RNE.
__device__ __forceinline__ uint32_t dq2(uint32_t codes, float s) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(codes)));
    float lo, hi;
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(static_cast<uint16_t>(h2 & 0xFFFFu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(static_cast<uint16_t>(h2 >> 16)));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__fmul_rn(hi, s)), "f"(__fmul_rn(lo, s)));
    return r;
}

// One thread per 32-value block: thread t of a 128 x 128 tile owns block
// (t & 3) of tile rows t/4 and t/4 + 64.  A CTA walks column tiles
// blockIdx.y, + gridDim.y, ... two at a time (both tiles' loads in flight
// before either is converted), so one group lookup serves several tiles.
template <bool GROUPED>
__global__ void __launch_bounds__(kThreads)
    dequantize_mx_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                         int64_t rows, int64_t cols, const int32_t* offsets, int groups,
                         uint16_t* __restrict__ out, int64_t ldo, int64_t nkc, bool v8) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    int64_t row_begin, row_end;
    if (!tile_rows<GROUPED>(offsets, groups, rows, &row_begin, &row_end)) return;
    const int tid = threadIdx.x;
    const int j = tid & 3;
    const int64_t n_row_tiles = GROUPED ? rows / kTile + groups : (rows + kTile - 1) / kTile;
    if (!MX_IN_BOUNDS(static_cast<int64_t>(blockIdx.x) < n_row_tiles)) return;
    for (int64_t ct0 = blockIdx.y; ct0 < nkc; ct0 += 2 * static_cast<int64_t>(gridDim.y)) {
        uint32_t qw[2][2][8];
        uint32_t sb[2][2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int64_t ct = ct0 + t * static_cast<int64_t>(gridDim.y);
            const int64_t col = ct * kTile + j * 32;
            const uint8_t* s_tile = s + (static_cast<int64_t>(blockIdx.x) * nkc + ct) * 512;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r = (tid >> 2) + 64 * i;
                const int64_t row = row_begin + r;
                if (ct < nkc && row < row_end && col < cols && MX_IN_BOUNDS(row < rows && col + 32 <= cols)) {
                    ld32_stream(q + row * cols + col, qw[t][i], v8);
                    sb[t][i] = __ldg(s_tile + swz_word(r) + j);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) qw[t][i][k] = 0u;
                    sb[t][i] = 0u;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int64_t ct = ct0 + t * static_cast<int64_t>(gridDim.y);
            const int64_t col = ct * kTile + j * 32;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int64_t row = row_begin + (tid >> 2) + 64 * i;
                if (ct < nkc && row < row_end && col < cols && MX_IN_BOUNDS(row < rows && col + 32 <= cols)) {
                    const float sc = e8m0_value(sb[t][i]);
                    uint32_t o[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        o[2 * k] = dq2(qw[t][i][k] & 0xFFFFu, sc);
                        o[2 * k + 1] = dq2(qw[t][i][k] >> 16, sc);
                    }
                    uint16_t* dst = out + row * ldo + col;
                    st32(dst, o, v8);
                    st32(dst + 16, o + 8, v8);
                }
            }
        }
    }
}

// ------------------------------------------------------ SwiGLU + Q ------

__device__ __forceinline__ uint32_t bf16_bits_rn(double v) {
    return __bfloat16_as_ushort(__double2bfloat16(v));
}

// Two fp32 values rounded to BF16 (RNE), `lo` in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// e^-|g| in fp32 from the special-function unit's 2^x, with the exponent
// -|g| log2(e) carried as an unevaluated sum p + d: p = RN(-a L2E), d = the
// product's exact residual (one FMA: Dekker's error-free product) plus
// -a * (log2(e) - L2E), the constant's own residual (the two-constant
// argument split of Cody and Waite), so e^-a = 2^p * 2^d with 2^d = 1 + d ln2
// to first order (|d| < 2^-17).  2^p flushes to 0 from a ~ 87.3 on; past
// a ~ 2.4e38 the product a L2E overflows and the result is NaN (the caller
// redoes such blocks in FP64).
__device__ __forceinline__ float exp_neg_abs(float g) {
    constexpr float kL2E = 1.44269502163f;       // RN(log2 e), 0x3FB8AA3B
    constexpr float kL2ELo = 1.92596303350e-08f;  // RN(log2 e - kL2E)
    constexpr float kLn2 = 0.693147182465f;       // RN(ln 2)
    const float a = fabsf(g);
    const float p = __fmul_rn(-a, kL2E);
    const float d = __fmaf_rn(-a, kL2ELo, __fmaf_rn(-a, kL2E, -p));
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(p));
    return __fmaf_rn(e, __fmul_rn(d, kLn2), e);
}

// g sigma(g) u in fp32, sigma(g) = 1 / (1 + e^-g), branch free, for
// g >= -80.  t = e^-|g| (exp_neg_abs) is a normal number there; r = 1/(1+t)
// (rcp.approx.ftz: within 1 ulp, and 1 + t lies in [1, 2]: one special-
// function instruction, 6 % faster than __fdividef on the routed workload
// with the same measured error); n = max(g, g t) is g for g >= 0
// (exact) and g e^g below; y = (n u) r.  With u = 1 the error of y against
// the exact g sigma(g) is below 4.5 * 2^-24 relative over every BF16 gate in
// [-80, inf) (measured exhaustively against double precision: 4.01 * 2^-24
// at most), and a general u adds at most three more half-ulp roundings
// (y = RN(RN(n u) r) against RN(n r)): below 7.5 * 2^-24, plus an absolute
// 2^-149 where n u underflows (for g >= 0, n u = g u is exact unless it underflows,
// which also covers BF16-subnormal gates; n u cannot overflow for g < 0).
// The BF16 rounding of y is therefore the correctly rounded value unless the
// exact value lies that close to a rounding midpoint, where it may be the
// neighbour.  NaN propagates (and |g| past ~2.4e38 gives NaN); g < -80 (e^g
// leaves fp32's normal range, including -Inf) takes the exact path below.
__device__ __forceinline__ float swiglu_fast(float g, float u) {
    const float t = exp_neg_abs(g);
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__fadd_rn(1.f, t)));
    const float n = fmaxf(g, __fmul_rn(g, t));
    return __fmul_rn(__fmul_rn(n, u), r);
}


// swiglu_fast for the two BF16 lanes of g2 and u2 (low half first), with the
// arithmetic in packed FP32.  Bit-identical to two swiglu_fast calls: the
// exponent residual is formed with the signs moved onto the constants,
// d' = fma(a, L2ELo, fma(a, L2E, p)) = -d exactly (each step is the negated
// scalar step, and rounding to nearest is symmetric), and d' (-ln 2) =
// d ln 2; the rest is the same operations lane by lane.
__device__ __forceinline__ void swiglu_fast2(uint32_t g2, uint32_t u2, float& y0, float& y1) {
    constexpr float kL2E = 1.44269502163f;
    constexpr float kL2ELo = 1.92596303350e-08f;
    constexpr float kLn2 = 0.693147182465f;
    const float g0 = bf16_lo(g2), g1 = bf16_hi(g2);
    const uint64_t G = f2_pack(g0, g1);
    const uint64_t U = f2_pack(bf16_lo(u2), bf16_hi(u2));
    const uint64_t A = f2_pack(fabsf(g0), fabsf(g1));
    const uint64_t P = f2_mul(A, f2_splat(-kL2E));                       // p = RN(-a L2E)
    const uint64_t D = f2_fma(A, f2_splat(kL2ELo), f2_fma(A, f2_splat(kL2E), P));  // -d
    float p0, p1, e0, e1;
    f2_unpack(P, p0, p1);
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(p0));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(p1));
    const uint64_t E = f2_pack(e0, e1);
    const uint64_t T = f2_fma(E, f2_mul(D, f2_splat(-kLn2)), E);         // t = e^-|g|
    float s0, s1, r0, r1, gt0, gt1;
    f2_unpack(f2_add(T, f2_splat(1.f)), s0, s1);
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(s0));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(s1));
    f2_unpack(f2_mul(G, T), gt0, gt1);
    const uint64_t N = f2_pack(fmaxf(g0, gt0), fmaxf(g1, gt1));
    f2_unpack(f2_mul(f2_mul(N, U), f2_pack(r0, r1)), y0, y1);
}

// Magnitude of BF16 bits 0..0x7F80 as a double (0x7F80 taken as 2^128, the
// value the rounding of the largest finite BF16 steps to).
__device__ __forceinline__ double bf16_mag(uint32_t b) {
    return b >= 0x7F80u ? 0x1p128 : static_cast<double>(__uint_as_float(b << 16));
}

// The correctly rounded BF16 value of g sigma(g) u evaluated in FP64 (the
// path for gates below -80, blocks holding Inf or NaN, and the few values the
// float-float resolver leaves undecided).  The FP64 value v is within a few
// 2^-53 of the exact one, so its rounding is the exact value's unless v lies
// next to a BF16 midpoint m; there the side is taken from the cancellation-
// free forms of swiglu_round.cuh ((|p| - m) - m t for g > 0, t (|p| - m) - m
// for g < 0, p = g u, t = e^-|g|), with |p| == m and g > 0 below m, and for
// |g| < 1 rewritten around |p| - 2m with expm1.
__device__ __noinline__ uint32_t swiglu_bf16_exact(float gf, float uf) {
    const double g = gf, u = uf, p = g * u;
    const double t = exp(-fabs(g));
    const double v = g >= 0.0 ? p / (1.0 + t) : p * t / (1.0 + t);
    uint16_t b;
    asm("cvt.rn.bf16.f64 %0, %1;" : "=h"(b) : "d"(v));
    if (!isfinite(v) || v == 0.0) return b;
    const double av = fabs(v);
    const uint32_t bm = b & 0x7FFFu;
    const uint32_t lo = bf16_mag(bm) > av ? bm - 1 : bm;  // BF16 magnitudes lo <= av < lo + 1
    if (lo >= 0x7F80u) return b;                         // at or past 2^128: Inf
    const double m = 0.5 * (bf16_mag(lo) + bf16_mag(lo + 1));
    if (fabs(av - m) > av * 0x1p-44) return b;
    const double ap = fabs(p);
    bool up;
    if (fabs(g) < 1.0) {
        // near g = 0 (e^-|g| rounds to 1 below 2^-54) the same forms around
        // |p| - 2m, which is exact here: the side of |p| == 2m is the sign of g
        const double e = g > 0.0 ? -m * expm1(-g) : expm1(g) * (ap - m);
        up = (ap - 2.0 * m) + e > 0.0;
    } else if (g > 0.0) {
        const double d = ap - m;
        up = d != 0.0 && d - m * t > 0.0;
    } else {
        up = t * (ap - m) - m > 0.0;
    }
    return (b & 0x8000u) | (up ? lo + 1 : lo);
}

// BF16 bits of one fast-path value next to a rounding midpoint: the
// float-float resolver, or FP64 where it cannot decide.
__device__ __noinline__ uint32_t swiglu_bf16_near(float g, float u, float y) {
    bool undecided;
    const uint32_t b = ff::swiglu_round_near(g, u, y, &undecided);
    return undecided ? swiglu_bf16_exact(g, u) : b;
}

// Near-midpoint test.  The fast value y is within 8.5 fp32 units of the
// exact one (7.5 2^-24 relative is at most 7.5 units of y's binade, plus one
// unit where fp32 underflows), so its BF16 rounding can be wrong only when
// its low 16 bits lie within 8 of 0x8000 (the midpoint pattern).  The test
// takes a window of kNearHalf = 10: low16 + 0x8000 + 10 (mod 2^16) <= 20.
constexpr uint32_t kNearHalf = 10;
constexpr uint32_t kNearOffset = (0x8000u + kNearHalf) * 0x10001u;

__device__ __forceinline__ bool near_one(float y) {
    return ((__float_as_uint(y) + 0x8000u + kNearHalf) & 0xFFFFu) <= 2 * kNearHalf;
}

// A running per-half minimum of the offset low halves of word pairs (see
// swiglu2) holds a near-midpoint value.  In the high half the carry out of
// the low half's addition can shift the window by one unit (to
// [0x8000 - 11, 0x8000 + 9]), still wider than the 8 units needed.
__device__ __forceinline__ bool near_any(uint32_t near) {
    return min(near & 0xFFFFu, near >> 16) <= 2 * kNearHalf;
}

// Two fast-path values rounded to BF16; `near` takes the per-half minimum of
// both values' low 16 bits (y0 in the low half) plus the window offset.
__device__ __forceinline__ uint32_t swiglu2(uint32_t g2, uint32_t u2, uint32_t& near) {
    float y0, y1;
    swiglu_fast2(g2, u2, y0, y1);
    uint32_t w;
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(w) : "r"(__float_as_uint(y0)), "r"(__float_as_uint(y1)));
    near = min_u16x2(near, w + kNearOffset);
    return bf16x2_rn(y0, y1);
}

// Column tiles per CTA of the fused row producers: the tile-row lookup (and,
// for gathers, the row indices) are paid once per CTA.
constexpr int kColTilesPerCta = 4;

// Any of 32 packed BF16 gates (16 words) below -80.
__device__ __forceinline__ bool swiglu_rare32(const uint32_t* g) {
    uint32_t m[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = max_u16x2(max_u16x2(g[4 * k], g[4 * k + 1]), max_u16x2(g[4 * k + 2], g[4 * k + 3]));
    const uint32_t t = max_u16x2(max_u16x2(m[0], m[1]), max_u16x2(m[2], m[3]));
    return max(t & 0xFFFFu, t >> 16) > 0xC2A0u;
}

__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    return v;
}

// E4M3 code of the BF16 value b (bits) under the block scale byte.
__device__ __forceinline__ uint32_t e4m3_of(uint32_t b, uint32_t byte) {
    if (byte == 0xFFu) return 0x7Fu;
    return cvt_fp8x2<FP8_E4M3>(__fmul_rn(bf16_lo(b), inv_scale(byte)), 0.f) & 0xFFu;
}

// Warp pass over one 32-value block (tile row `row`, columns col..col+31),
// one value per lane, read again from global memory, writing the block's
// payload and scale over what its owner wrote.  `exact`: every value in FP64
// (swiglu_bf16_exact).  Otherwise the fast values, where a value lies next to
// a BF16 midpoint (near_one) its side is taken only where it matters: when
// its upper candidate exceeds every settled value of the block (it may set
// the scale), or when its two candidates quantize to different E4M3 codes
// under the block's scale; any other near value quantizes the same either
// way.  All 32 lanes call it with the same arguments.
template <bool FLOOR>
__device__ __forceinline__ void swiglu_block_redo(const uint16_t* __restrict__ h, int64_t ld,
                                                  int64_t f, int64_t row, int64_t col, bool exact,
                                                  uint8_t* __restrict__ q, uint8_t* s_dst) {
    const int lane = threadIdx.x & 31;
    const uint16_t* hp = h + row * ld + col + lane;
    const float g = __uint_as_float(static_cast<uint32_t>(__ldg(hp)) << 16);
    const float u = __uint_as_float(static_cast<uint32_t>(__ldg(hp + f)) << 16);
    uint32_t b;
    float y = 0.f;
    bool near = false;
    if (exact) {
        b = swiglu_bf16_exact(g, u);
    } else {
        y = swiglu_fast(g, u);
        b = bf16x2_rn(y, 0.f) & 0xFFFFu;
        near = near_one(y);
    }
    // BF16 magnitude bits order like the magnitudes, Inf and NaN above all;
    // `below` is the magnitude under the midpoint next to y
    const uint32_t below = (__float_as_uint(y) >> 16) & 0x7FFFu;
    uint32_t am = warp_max(near ? 0u : (b & 0x7FFFu));
    const bool top = near && below + 1 > am;
    if (__any_sync(0xFFFFFFFFu, top)) {
        if (top) b = swiglu_bf16_near(g, u, y);
        near = near && !top;
        am = warp_max(near ? 0u : (b & 0x7FFFu));
    }
    const uint32_t byte = e8m0_byte(am, FLOOR);
    uint32_t code = e4m3_of(b, byte);
    if (near) {
        const uint32_t lo = (b & 0x8000u) | below;
        if (e4m3_of(lo, byte) != e4m3_of(lo + 1, byte)) code = e4m3_of(swiglu_bf16_near(g, u, y), byte);
    }
    q[row * f + col + lane] = static_cast<uint8_t>(code);
    if (lane == 0) *s_dst = static_cast<uint8_t>(byte);
}

// One thread per 32-value output block (thread t of a 128 x 128 tile owns
// block t & 3 of tile rows t/4 and t/4 + 64), several column tiles per CTA.
// The two rows are loaded and converted one after the other, which keeps the
// kernel at 64 registers: four CTAs (32 warps) per SM hide the load latency
// better than two CTAs holding both rows in flight (129.7 against 146 us on
// the 262144 x 512 routed workload).
//
// Exact rounding: every block is first quantized from its fast values; a
// block holding a fast value next to a BF16 midpoint (about one in 80), a
// gate below -80, or a maximum that is Inf or NaN (an input Inf or NaN, or
// g u past fp32's range where the exact value may still be finite) is then
// redone by its warp (swiglu_block_redo), in FP64 for the latter two.
template <bool FLOOR, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 4)
    swiglu_quant_kernel(const uint16_t* __restrict__ h, int64_t rows, int64_t f, int64_t ld,
                        const int32_t* offsets, int groups, uint8_t* __restrict__ q,
                        uint8_t* __restrict__ s, int64_t nkc, bool v8) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    int64_t row_begin, row_end;
    if (!tile_rows<GROUPED>(offsets, groups, rows, &row_begin, &row_end)) return;
    const int tid = threadIdx.x;
    const int j = tid & 3;
    const int64_t n_row_tiles = GROUPED ? rows / kTile + groups : (rows + kTile - 1) / kTile;
    if (!MX_IN_BOUNDS(static_cast<int64_t>(blockIdx.x) < n_row_tiles)) return;
    for (int64_t ct = blockIdx.y; ct < nkc; ct += gridDim.y) {
        const int64_t col = ct * kTile + j * 32;
        uint8_t* s_tile = s + (static_cast<int64_t>(blockIdx.x) * nkc + ct) * 512;
#pragma unroll 1
        for (int i = 0; i < 2; ++i) {
            const int r = (tid >> 2) + 64 * i;
            const int64_t row = row_begin + r;
            const bool in = row < row_end && col < f && MX_IN_BOUNDS(row < rows && col + 32 <= f && ld >= 2 * f);
            uint32_t gw[16], uw[16];
            if (in) {
                const uint16_t* src = h + row * ld + col;
                ld32_stream(src, gw, v8);
                ld32_stream(src + 16, gw + 8, v8);
                ld32_stream(src + f, uw, v8);
                ld32_stream(src + f + 16, uw + 8, v8);
            } else {
#pragma unroll
                for (int k = 0; k < 16; ++k) gw[k] = uw[k] = 0u;
            }
            {
                // this thread's next block (the tile's other row, else the next
                // column tile) into L2 while this one is converted: 2.3 % faster
                const int64_t nrow = i == 0 ? row + 64 : row_begin + (tid >> 2);
                const int64_t ncol = i == 0 ? col : col + static_cast<int64_t>(gridDim.y) * kTile;
                if (nrow < row_end && ncol < f) {
                    const uint16_t* nsrc = h + nrow * ld + ncol;
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(nsrc));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(nsrc + f));
                }
            }
            const bool rare = in && swiglu_rare32(gw);
            uint32_t v[16];
            uint32_t near = 0xFFFFFFFFu;
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = swiglu2(gw[k], uw[k], near);
            const uint32_t am = block32_amax_bits(v);
            mx_block32_amax<FLOOR>(v, am, in ? q + row * f + col : nullptr, s_tile + swz_word(r) + j, v8);
            // lanes out of range hold zeros: value 0, never near a midpoint
            const bool exact = rare || (in && am >= 0x7F80u);
            unsigned todo = __ballot_sync(0xFFFFFFFFu, exact || near_any(near));
            if (todo) {
                const unsigned ex = __ballot_sync(0xFFFFFFFFu, exact);
                __syncwarp();  // the owners' stores above come first
                do {
                    const int src = __ffs(todo) - 1;
                    todo &= todo - 1;
                    const int stid = (tid & ~31) | src;
                    const int rs = (stid >> 2) + 64 * i;
                    if (MX_IN_BOUNDS(row_begin + rs < rows && ct * kTile + (stid & 3) * 32 + 32 <= f))
                        swiglu_block_redo<FLOOR>(h, ld, f, row_begin + rs, ct * kTile + (stid & 3) * 32,
                                                 (ex >> src) & 1u, q, s_tile + swz_word(rs) + (stid & 3));
                } while (todo);
            }
        }
    }
}

// ------------------------------------------- route weighting + Q --------

// bf16_RNE(x w) of a BF16 x and an fp32 w, equal to one rounding of the
// exact product: p = fp32_RN(x w) is monotone in the exact value and every
// BF16 rounding midpoint is an fp32 number, so the BF16 rounding of p agrees
// with that of the exact product unless p lands exactly on a midpoint (its
// low 16 bits are 0x8000; this covers the fp32-subnormal range too, where
// fp32 still has 16 more fraction bits than BF16).  `mid` keeps the per-half
// minimum of both products' low halves xor 0x8000 (one prmt, one xor, one
// min.u16x2 per pair): a zero half marks such a product, and the caller
// redoes the pair exactly in double.  Overflow, Inf and NaN follow the fp32
// product, which agrees with the exact one in BF16.
__device__ __forceinline__ uint32_t weighted2(uint32_t x2, float w, uint32_t& mid) {
    const float p0 = __fmul_rn(bf16_lo(x2), w);
    const float p1 = __fmul_rn(bf16_hi(x2), w);
    uint32_t lows;
    asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(lows) : "r"(__float_as_uint(p0)), "r"(__float_as_uint(p1)));
    mid = min_u16x2(mid, lows ^ 0x80008000u);
    return bf16x2_rn(p0, p1);
}

// Either half of a `mid` accumulator zero: some product sat on a midpoint.
__device__ __forceinline__ bool weighted_tie(uint32_t mid) {
    return (mid & 0xFFFFu) == 0u || (mid >> 16) == 0u;
}

// p + a m with a 32-bit a m: one wide multiply-add (the FMA pipe) instead of
// a 64-bit add on the integer pipe.
__device__ __forceinline__ uint8_t* add_wide(uint8_t* p, uint32_t a, uint32_t m) {
    uint64_t r;
    asm("mad.wide.u32 %0, %1, %2, %3;" : "=l"(r) : "r"(a), "r"(m), "l"(reinterpret_cast<uint64_t>(p)));
    return reinterpret_cast<uint8_t*>(r);
}

// Per-half signed 16-bit minimum: 0x8000 is the smallest signed half, so a
// half of a running minimum is 0x8000 exactly when some input half was.
__device__ __forceinline__ uint32_t min_s16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bf16_RNE(x) as an fp32 value (the BF16 bits in the high half, zeros below).
__device__ __forceinline__ float bf16_round_f32(float x) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x), "f"(0.f));
    return __uint_as_float(r);
}

// One route of one block on the fast path: the 32 values as fp32 pairs xf(i)
// (i = 0..15, value 2i low), times ws two at a time, each product rounded to
// fp32, then to BF16, then to E4M3 (qv, 32 bytes).  The BF16 rounding of an
// fp32 product agrees with that of the exact product unless the product sits
// on a BF16 midpoint (low half 0x8000, see weighted2); the running signed
// minimum of the products' low halves finds that case.  Returns false then:
// the caller redoes the block exactly.
template <typename XF>
__device__ __forceinline__ bool weighted32_fast(const XF& xf, float ws, uint32_t* qv) {
    const uint64_t W = f2_splat(ws);
    uint32_t mn = 0x7FFF7FFFu;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        float r[4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            float p0, p1;
            f2_unpack(f2_mul(xf(2 * kk + t), W), p0, p1);
            uint32_t lows;
            asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(lows) : "r"(__float_as_uint(p0)), "r"(__float_as_uint(p1)));
            mn = min_s16x2(mn, lows);
            r[2 * t] = bf16_round_f32(p0);
            r[2 * t + 1] = bf16_round_f32(p1);
        }
        qv[kk] = cvt_fp8x4<FP8_E4M3>(r[0], r[1], r[2], r[3]);
    }
    return (mn & 0xFFFFu) != 0x8000u && (mn >> 16) != 0x8000u;
}

// bf16_RNE of the exact product x ws, as an fp32 value, for the values of a
// block that weighted32_fast flagged: p = fp32_RN(x ws), and when p sits on a
// BF16 midpoint the product's exact residual x ws - p (one FMA) moves p one
// fp32 unit toward the exact value, off the midpoint and onto the side the
// exact product rounds to.  The residual is exact for every product that can
// reach a nonzero E4M3 code (|p| >= 2^-11: its last bit lies far above
// fp32's underflow); a smaller p stays below 2^-10 after the one-unit move
// and quantizes to the same signed zero either way.
__device__ __forceinline__ float weighted_exact_f32(float x, float ws) {
    const float p = __fmul_rn(x, ws);
    const float r = __fmaf_rn(x, ws, -p);
    uint32_t pb = __float_as_uint(p);
    if ((pb & 0xFFFFu) == 0x8000u && r != 0.f) pb += ((r > 0.f) == (p > 0.f)) ? 1u : 0xFFFFFFFFu;
    return bf16_round_f32(__uint_as_float(pb));
}

// What the scale folding needs from a route's weight alone.  For a normal
// w with exponent field f, w' = w 2^(127 - byte) is the normal fp32 number
// with exponent field f + 127 - byte (bits: wbias - byte 2^23, exact) for
// byte in [f - 126, f + 126]; the fold also needs byte >= 11 (see
// weighted_block_quant) and a finite scale (byte <= 254).  The block takes
// the folded path iff byte - lo <= span (unsigned); a weight that is zero,
// subnormal, Inf or NaN never does (lo out of byte range).  Any narrower
// range gives the same bytes: the unfolded path is exact too.
struct WeightFold {
    float w;
    uint32_t wbias;  // bits(w) + 127 2^23
    uint32_t lo;
    uint32_t span;
};

__host__ __device__ __forceinline__ WeightFold weight_fold(float w, uint32_t wbits) {
    WeightFold f;
    f.w = w;
    f.wbias = wbits + (127u << 23);
    const int ef = static_cast<int>((wbits >> 23) & 0xFFu);
    const int lo = ef - 126 > 11 ? ef - 126 : 11;
    const int hi = ef + 126 < 254 ? ef + 126 : 254;
    const bool ok = ef != 0 && ef != 0xFF && lo <= hi;
    f.lo = ok ? static_cast<uint32_t>(lo) : 0x10000u;
    f.span = ok ? static_cast<uint32_t>(hi - lo) : 0u;
    return f;
}

// One weighted block: bf16_RNE(w x) of the 32 BF16 values given as fp32 pairs
// by xf(i) (value 2i low; rounded once from the exact products), MX-quantized
// into q_dst (32 bytes; skipped when null, which only QNULL callers pass) and
// *s_dst; ax is max |x| over the
// block as fp32 (the BF16 maximum, NaN or Inf as they are).  The block
// maximum of the weighted values is the correctly rounded |ax w|: the
// rounding is monotone, so one product replaces the maximum over the 32
// weighted values.  The rare forms (a flagged block, a scale outside the
// folded range, NaN / Inf) reread the block's 32 values from src four at a
// time, so that the values are all the registers they share with the fast
// path.
template <bool FLOOR, bool QNULL, typename XF>
__device__ __forceinline__ void weighted_block_quant(const XF& xf, const uint16_t* src,
                                                     float ax, const WeightFold& wf, uint8_t* q_dst,
                                                     uint8_t* s_dst, bool v8) {
    const float w = wf.w;
    // pa >= +0 or NaN, so am is the magnitude's bits (a NaN rounds to 0x7FFF)
    const float pa = __fmul_rn(ax, fabsf(w));
    const uint32_t am = (__float_as_uint(pa) & 0xFFFFu) == 0x8000u
                            ? bf16_bits_rn(static_cast<double>(ax) * fabs(static_cast<double>(w)))
                            : bf16x2_rn(pa, 0.f);
    // e8m0_byte's rule in one biased add and an arithmetic shift: am + 0x1F
    // carries into the exponent field exactly when the mantissa field is
    // above 0x60 (rceil), and a negative sum stands for a clamped byte 0
    const int t = static_cast<int>(am + (FLOOR ? 0u : 0x1Fu) - 0x400u) >> 7;
    const uint32_t byte = am >= 0x7F80u ? 0xFFu : static_cast<uint32_t>(max(t, 0));
    *s_dst = static_cast<uint8_t>(byte);
    // With the block scale 2^e known, w' = w 2^-e is exact while it is
    // a normal fp32 number, and bf16(x w') = bf16(x w) 2^-e for every
    // value that is BF16-normal; with e >= -116 a BF16-subnormal value
    // scales below 2^-10 and quantizes to a signed zero either way.
    // So the products x w' round straight to the scaled BF16 values.
    const bool folded = byte - wf.lo <= wf.span;
    const float ws = __uint_as_float(wf.wbias - (byte << 23));  // w 2^(127 - byte) where folded
    if (folded) {
        uint32_t qv[8];
        if (weighted32_fast(xf, ws, qv)) {
            if (!QNULL || q_dst != nullptr) st32(q_dst, qv, v8);  // one 32-byte store: each sector written once
            return;
        }
    }
    if (QNULL && q_dst == nullptr) return;
    const float f = inv_scale(byte);
#pragma unroll 1
    for (int kk = 0; kk < 8; ++kk) {
        const uint2 x = __ldg(reinterpret_cast<const uint2*>(src) + kk);
        uint32_t q4 = 0x7F7F7F7Fu;  // NaN scale: every payload byte NaN
        if (folded) {
            // a product on a BF16 midpoint: the exact residual settles it
            q4 = cvt_fp8x2<FP8_E4M3>(weighted_exact_f32(bf16_lo(x.x), ws), weighted_exact_f32(bf16_hi(x.x), ws)) |
                 (cvt_fp8x2<FP8_E4M3>(weighted_exact_f32(bf16_lo(x.y), ws), weighted_exact_f32(bf16_hi(x.y), ws))
                  << 16);
        } else if (byte != 0xFFu) {
            // the unscaled form: bf16(x w) rounded once (the double product
            // where the fp32 one sits on a midpoint; products here may be
            // fp32-subnormal), then times 1/s and rounded to E4M3
            uint32_t h[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const uint32_t word = t ? x.y : x.x;
                uint32_t mid = 0xFFFFFFFFu;
                uint32_t vb = weighted2(word, w, mid);
                if (weighted_tie(mid)) {
                    const double wd = w;
                    vb = bf16_bits_rn(static_cast<double>(bf16_lo(word)) * wd) |
                         (bf16_bits_rn(static_cast<double>(bf16_hi(word)) * wd) << 16);
                }
                h[t] = cvt_fp8x2<FP8_E4M3>(__fmul_rn(bf16_lo(vb), f), __fmul_rn(bf16_hi(vb), f));
            }
            q4 = h[0] | (h[1] << 16);
        }
        reinterpret_cast<uint32_t*>(q_dst)[kk] = q4;
    }
}

// Launch-bounded to 64 registers (four CTAs per SM): 252.6 against 273 us
// at the default three CTAs on the 262144 x 2048 combine-backward workload.
template <bool FLOOR, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 4)
    weighted_quant_kernel(const uint16_t* __restrict__ dy, int64_t tokens, int64_t ld,
                          const int32_t* __restrict__ row_token, const float* __restrict__ row_weight,
                          int64_t rows, int64_t cols, const int32_t* offsets, int groups,
                          uint8_t* __restrict__ q, uint8_t* __restrict__ s, int64_t nkc,
                          bool v8) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    int64_t row_begin, row_end;
    if (!tile_rows<GROUPED>(offsets, groups, rows, &row_begin, &row_end)) return;
    const int tid = threadIdx.x;
    const int j = tid & 3;
    const int64_t n_row_tiles = GROUPED ? rows / kTile + groups : (rows + kTile - 1) / kTile;
    if (!MX_IN_BOUNDS(static_cast<int64_t>(blockIdx.x) < n_row_tiles)) return;
    // token and weight of this thread's two rows, once for all column tiles
    int32_t tk[2];
    WeightFold wf[2];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int64_t row = row_begin + (tid >> 2) + 64 * i;
        const bool in = row < row_end && MX_IN_BOUNDS(row < rows);
        const int32_t t = in ? __ldg(row_token + row) : -1;
        const bool valid = t >= 0 && t < tokens;
        bad |= in && !valid;
        tk[i] = valid ? t : -1;
        const float w = valid ? __ldg(row_weight + row) : 0.f;
        wf[i] = weight_fold(w, __float_as_uint(w));
    }
    if (bad && blockIdx.y == 0) record_status(MXFP8_ERR_DEVICE_CHECK);
    for (int64_t ct = blockIdx.y; ct < nkc; ct += gridDim.y) {
        const int64_t col = ct * kTile + j * 32;
        uint32_t xw[2][16];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (tk[i] >= 0 && col < cols && MX_IN_BOUNDS(tk[i] < tokens && col + 32 <= cols)) {
                // cached: each token row is gathered by several dispatched rows
                const uint16_t* src = dy + static_cast<int64_t>(tk[i]) * ld + col;
                ld32_cached(src, xw[i], v8);
                ld32_cached(src + 16, xw[i] + 8, v8);
            } else {
#pragma unroll
                for (int k = 0; k < 16; ++k) xw[i][k] = 0u;
            }
        }
        uint8_t* s_tile = s + (static_cast<int64_t>(blockIdx.x) * nkc + ct) * 512;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = (tid >> 2) + 64 * i;
            const int64_t row = row_begin + r;
            uint8_t* const q_dst =
                row < row_end && col < cols && MX_IN_BOUNDS(row < rows && col + 32 <= cols) ? q + row * cols + col : nullptr;
            uint8_t* const s_dst = s_tile + swz_word(r) + j;
            if (tk[i] < 0 || col >= cols) {
                // no token (or padding, or past the last column): zeros
                const uint32_t z[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                if (q_dst != nullptr) st32(q_dst, z, v8);
                *s_dst = 0;
                continue;
            }
            const float ax = __uint_as_float(block32_amax_bits(xw[i]) << 16);
            weighted_block_quant<FLOOR, true>([&](int k) { return f2_pack(bf16_lo(xw[i][k]), bf16_hi(xw[i][k])); },
                                        dy + static_cast<int64_t>(tk[i]) * ld + col, ax, wf[i], q_dst, s_dst,
                                        v8);
        }
    }
}

// Token-walk form of the same conversion: each CTA takes kTokensPerCta
// tokens and reads each token's dY row once; a thread owns one 32-value
// block of one token and writes, for each of the token's k routes, the
// weighted block's E4M3 payload into the route's dispatched row and its scale
// byte into the (group-padded) scale array.  The per-value results are
// weighted_quant_kernel's, exact-product ties included.  The block is
// unpacked to fp32 pairs once for all of its routes (32 registers held
// across the route loop); launch-bounded to four CTAs per SM, which costs a
// few spilled words and still beats three CTAs without spills.
constexpr int kTokensPerCta = 16;
constexpr int kMaxRoutes = 16;

// One route of the CTA's table: its payload row and its row's place in the
// swizzled scale array (null: no route), and its weight's fold data; 32
// bytes, read as two 16-byte shared loads.
struct __align__(16) RouteEntry {
    uint8_t* qrow;
    uint8_t* srow;
    WeightFold wf;
};
static_assert(sizeof(RouteEntry) == 32, "two 16-byte loads per route");
constexpr int kMaxGroupsTok = 1024;

template <bool FLOOR, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 4)
    weighted_quant_tokens_kernel(const uint16_t* __restrict__ dy, int64_t tokens, int64_t ld,
                                 int k, const int32_t* __restrict__ token_rows,
                                 const float* __restrict__ token_weights, int64_t rows,
                                 int64_t cols, const int32_t* offsets, int groups,
                                 uint8_t* __restrict__ q, uint8_t* __restrict__ s, int64_t nkc,
                                 bool v8) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    // per route: its payload row (null: no route) and its row's place in the
    // swizzled scale array (block 0), so the item loop only adds offsets
    __shared__ RouteEntry s_route[kTokensPerCta * kMaxRoutes];
    __shared__ int32_t s_off[GROUPED ? kMaxGroupsTok + 1 : 1];
    __shared__ int64_t s_pstart[GROUPED ? kMaxGroupsTok + 1 : 1];
    __shared__ int s_ok;
    const int tid = threadIdx.x;
    const int64_t nb = cols / 32;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokensPerCta;
    const int nt = static_cast<int>(min(static_cast<int64_t>(kTokensPerCta), tokens - t0));
    // this thread's route entry (kTokensPerCta * kMaxRoutes == blockDim.x:
    // one at most) and its first (token, block) item's dY go out together
    static_assert(kTokensPerCta * kMaxRoutes == kThreads, "one route entry per thread");
    const bool has_route = tid < nt * k;
    int32_t r = -1;
    float wr = 0.f;
    if (has_route) {
        const int64_t idx = (t0 + tid / k) * k + tid % k;
        r = __ldg(token_rows + idx);
        wr = __ldg(token_weights + idx);
    }
    uint32_t xw[16];
    int64_t pi = tid;
    if (pi < nt * nb && MX_IN_BOUNDS(t0 + pi / nb < tokens && (pi % nb + 1) * 32 <= cols)) {
        const int tl = static_cast<int>(pi / nb);
        const uint16_t* src = dy + (t0 + tl) * ld + (pi - tl * nb) * 32;
        ld32_stream(src, xw, v8);
        ld32_stream(src + 16, xw + 8, v8);
    }
    if constexpr (GROUPED) {
        // offsets into shared memory (the whole CTA loads them at once),
        // validated (0 first, non-decreasing, rows last), and the padded
        // first scale row of every group (warp 0 scans them)
        for (int g = tid; g <= groups; g += blockDim.x) s_off[g] = offsets[g];
        __syncthreads();
        if (tid < 32) {
            bool ok = s_off[0] == 0 && static_cast<int64_t>(s_off[groups]) == rows;
            int64_t base = 0;
            for (int g0 = 0; g0 <= groups; g0 += 32) {
                const int g = g0 + tid;
                int64_t tiles = 0;
                if (g < groups) {
                    const int32_t gb = s_off[g], ge = s_off[g + 1];
                    if (ge < gb) ok = false;
                    tiles = ge > gb ? (ge - gb + kTile - 1) / kTile : 0;
                }
                int64_t incl = tiles;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                    if (tid >= d) incl += v;
                }
                if (g <= groups) s_pstart[g] = (base + incl - tiles) * kTile;
                base += __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (tid == 0) s_ok = ok ? 1 : 0;
        }
        __syncthreads();
        if (!s_ok) {
            if (blockIdx.x == 0 && tid == 0) record_status(MXFP8_ERR_DEVICE_CHECK);
            return;
        }
    }
    if (has_route) {
        int64_t row = -1, prow = -1;
        float w = 0.f;
        if (r >= rows) {
            record_status(MXFP8_ERR_DEVICE_CHECK);
        } else if (r >= 0) {
            row = r;
            w = wr;
            if constexpr (GROUPED) {
                int lo = 0, hi = groups - 1;  // the last group starting at or before r
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (s_off[mid] <= r) lo = mid; else hi = mid - 1;
                }
                prow = s_pstart[lo] + (r - s_off[lo]);
            } else {
                prow = r;
            }
        }
        // the padded scale row lies in the layout's row tiles
        const int64_t n_row_tiles = GROUPED ? rows / kTile + groups : (rows + kTile - 1) / kTile;
        if (row >= 0 && !MX_IN_BOUNDS(row < rows && prow / kTile < n_row_tiles)) row = -1;
        RouteEntry re;
        re.qrow = row >= 0 ? q + row * cols : nullptr;
        re.srow = row >= 0 ? s + (prow / kTile) * nkc * 512 + swz_word(static_cast<int>(prow % kTile)) : nullptr;
        re.wf = weight_fold(w, __float_as_uint(w));
        s_route[tid] = re;
    }
    __syncthreads();
    for (; pi < nt * nb; pi += blockDim.x) {
        const int tl = static_cast<int>(pi / nb);
        const int64_t b = pi - tl * nb;
        if (!MX_IN_BOUNDS(t0 + tl < tokens && (b + 1) * 32 <= cols)) continue;
        if (pi != tid) {
            const uint16_t* src = dy + (t0 + tl) * ld + b * 32;
            ld32_stream(src, xw, v8);
            ld32_stream(src + 16, xw + 8, v8);
        }
        // a route's block maximum is the correctly rounded |max |x| w|: the
        // rounding is monotone, so one product per route replaces the
        // maximum over the 32 weighted values (NaN and Inf carry over)
        const float ax = __uint_as_float(block32_amax_bits(xw) << 16);
        // the block's offsets in a route's payload row and scale rows (32
        // bits: cols <= 2^30), and the block as fp32 pairs, unpacked once for
        // all of its routes
        const uint32_t b32 = static_cast<uint32_t>(b);
        const uint32_t sb32 = ((b32 >> 2) << 9) | (b32 & 3u);
        uint64_t xf[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) xf[i] = f2_pack(bf16_lo(xw[i]), bf16_hi(xw[i]));
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
            const int e = tl * k + j;
            const RouteEntry re = s_route[e];
            if (re.qrow == nullptr) continue;
            weighted_block_quant<FLOOR, false>([&](int i) { return xf[i]; }, dy + (t0 + tl) * ld + b * 32, ax, re.wf,
                                               add_wide(re.qrow, b32, 32u), add_wide(re.srow, sb32, 1u), v8);
        }
    }
}

bool aligned32_host(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Grid of a tile walk: plain operands have ceil(rows/128) row tiles; a
// group-padded one at most floor(rows/128) + groups.
bool tile_grid(int64_t rows, int64_t cols, bool grouped, int groups, dim3* grid,
               int col_tiles_per_cta = 1) {
    const int64_t row_tiles = grouped ? rows / kTile + groups : (rows + kTile - 1) / kTile;
    const int64_t col_tiles = (cols + kTile - 1) / kTile;
    const int64_t col_ctas = (col_tiles + col_tiles_per_cta - 1) / col_tiles_per_cta;
    if (row_tiles > 0x7FFFFFFF || col_ctas > 65535) return false;
    *grid = dim3(static_cast<unsigned>(row_tiles), static_cast<unsigned>(col_ctas));
    return true;
}

}  // namespace

cudaError_t launch_dequantize_mx(const DequantArgs& a, cudaStream_t st) {
    dim3 grid;
    const bool grouped = a.offsets != nullptr;
    if (!tile_grid(a.rows, a.cols, grouped, a.groups, &grid, kColTilesPerCta)) return cudaErrorInvalidValue;
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    const int64_t nkc = (a.cols + kTile - 1) / kTile;
    const bool v8 = aligned32_host(a.q) && aligned32_host(a.out) && a.ldo % 16 == 0;
    if (grouped)
        return launch_pdl(dequantize_mx_kernel<true>, grid, dim3(kThreads), 0, st, a.q, a.s, a.rows,
                          a.cols, a.offsets, a.groups, a.out, a.ldo, nkc, v8);
    return launch_pdl(dequantize_mx_kernel<false>, grid, dim3(kThreads), 0, st, a.q, a.s, a.rows,
                      a.cols, nullptr, 0, a.out, a.ldo, nkc, v8);
}

cudaError_t launch_swiglu_quantize_mx(const SwigluQuantArgs& a, cudaStream_t st) {
    dim3 grid;
    const bool grouped = a.offsets != nullptr;
    const bool fl = a.flags & MX_SCALE_FLOOR;
    if (!tile_grid(a.rows, a.f, grouped, a.groups, &grid, kColTilesPerCta))
        return cudaErrorInvalidValue;
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    const int64_t nkc = (a.f + kTile - 1) / kTile;
    const bool v8 = aligned32_host(a.h) && a.ld % 16 == 0 && a.f % 16 == 0 && aligned32_host(a.q);
#define MXFP8_SWIGLU(FL, GR)                                                                   \
    launch_pdl(swiglu_quant_kernel<FL, GR>, grid, dim3(kThreads), 0, st, a.h, a.rows, a.f, a.ld, \
               a.offsets, a.groups, a.q, a.s, nkc, v8)
    cudaError_t e;
    if (grouped) {
        e = fl ? MXFP8_SWIGLU(true, true) : MXFP8_SWIGLU(false, true);
    } else {
        e = fl ? MXFP8_SWIGLU(true, false) : MXFP8_SWIGLU(false, false);
    }
#undef MXFP8_SWIGLU
    return e;
}

cudaError_t launch_weighted_quantize_mx(const WeightedQuantArgs& a, cudaStream_t st) {
    dim3 grid;
    const bool grouped = a.offsets != nullptr;
    const bool fl = a.flags & MX_SCALE_FLOOR;
    if (!tile_grid(a.rows, a.cols, grouped, a.groups, &grid, kColTilesPerCta))
        return cudaErrorInvalidValue;
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    const int64_t nkc = (a.cols + kTile - 1) / kTile;
    const bool v8 = aligned32_host(a.dy) && a.ld % 16 == 0 && aligned32_host(a.q);
#define MXFP8_WEIGHTED(FL, GR)                                                                \
    launch_pdl(weighted_quant_kernel<FL, GR>, grid, dim3(kThreads), 0, st, a.dy, a.tokens, a.ld, \
               a.row_token, a.row_weight, a.rows, a.cols, a.offsets, a.groups, a.q, a.s, nkc, v8)
    cudaError_t e;
    if (grouped) {
        e = fl ? MXFP8_WEIGHTED(true, true) : MXFP8_WEIGHTED(false, true);
    } else {
        e = fl ? MXFP8_WEIGHTED(true, false) : MXFP8_WEIGHTED(false, false);
    }
#undef MXFP8_WEIGHTED
    return e;
}

cudaError_t launch_weighted_quantize_tokens_mx(const WeightedTokensArgs& a, cudaStream_t st) {
    const bool grouped = a.offsets != nullptr;
    const bool fl = a.flags & MX_SCALE_FLOOR;
    if (a.k < 1 || a.k > kMaxRoutes || (grouped && a.groups > kMaxGroupsTok)) return cudaErrorInvalidValue;
    const int64_t nkc = (a.cols + kTile - 1) / kTile;
    // padding scale bytes (rows past a group's end, blocks past cols) read 0:
    // the token walk writes only the routed rows' blocks
    cudaError_t e = cudaMemsetAsync(a.s, 0, a.scale_bytes, st);
    if (e != cudaSuccess) return e;
    const int64_t ctas = (a.tokens + kTokensPerCta - 1) / kTokensPerCta;
    if (ctas == 0) return cudaSuccess;
    if (ctas > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const bool v8 = aligned32_host(a.dy) && a.ld % 16 == 0 && aligned32_host(a.q);
#define MXFP8_WTOK(FL, GR)                                                                      \
    weighted_quant_tokens_kernel<FL, GR><<<static_cast<unsigned>(ctas), kThreads, 0, st>>>(      \
        a.dy, a.tokens, a.ld, a.k, a.token_rows, a.token_weights, a.rows, a.cols, a.offsets,     \
        a.groups, a.q, a.s, nkc, v8)
    if (grouped) {
        if (fl) MXFP8_WTOK(true, true); else MXFP8_WTOK(false, true);
    } else {
        if (fl) MXFP8_WTOK(true, false); else MXFP8_WTOK(false, false);
    }
#undef MXFP8_WTOK
    return cudaGetLastError();
}

namespace {

// Test hook: the fast-path fp32 value g sigma(g) u per element (no BF16
// rounding, no quantization), for checking its error bound.
__global__ void swiglu_f32_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ u,
                                  int64_t n, float* __restrict__ y) {
    // pairs through the fused kernel's packed path (an odd last value alone);
    // each value is also computed by the scalar path the block redo uses, and
    // any difference in bits (other than two NaNs) is recorded as a device
    // check failure: the two paths are meant to be bit-identical
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; 2 * i < n; i += stride) {
        const int64_t k = 2 * i;
        const bool two = k + 1 < n;
        const uint32_t g2 = g[k] | (two ? static_cast<uint32_t>(g[k + 1]) << 16 : 0u);
        const uint32_t u2 = u[k] | (two ? static_cast<uint32_t>(u[k + 1]) << 16 : 0u);
        float y0, y1;
        swiglu_fast2(g2, u2, y0, y1);
        const float s0 = swiglu_fast(bf16_lo(g2), bf16_lo(u2));
        const float s1 = swiglu_fast(bf16_hi(g2), bf16_hi(u2));
        auto same = [](float a, float b) {
            return __float_as_uint(a) == __float_as_uint(b) || (isnan(a) && isnan(b));
        };
        if (!same(y0, s0) || (two && !same(y1, s1))) record_status(MXFP8_ERR_DEVICE_CHECK);
        y[k] = y0;
        if (two) y[k + 1] = y1;
    }
}

}  // namespace

cudaError_t launch_debug_swiglu_f32(const uint16_t* g, const uint16_t* u, int64_t n, float* y,
                                    cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 4096));
    swiglu_f32_kernel<<<blocks, 256, 0, s>>>(g, u, n, y);
    return cudaGetLastError();
}

cudaError_t take_status_fused(unsigned* out) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status_fused, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status_fused, &zero, sizeof(unsigned));
}

}  // namespace mxfp8
