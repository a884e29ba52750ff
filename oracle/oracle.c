/*
 * FP64 CPU oracle for MXFP8 / per-tensor FP8 quantization and scaled GEMMs.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link
 * or call this file.  Only the test suite, the smoke check of the build entry
 * point and the CPU-baseline leg of the benchmark use it.  It shares no code,
 * header, table or constant generator with the CUDA library: every number
 * here is derived from the format definitions written out below.
 *
 * Sources (page title, then section / equation / table / figure):
 *  [OLMO]  "Olmo-core MoE report, Section 11: MXFP8 Training"
 *          - Eq. 57 (33/32 bytes per value), Eq. 58 (q = E4M3(x/s), x^ = s q),
 *          - Figure 49 table (BF16 / E4M3 / E5M2 / E8M0 ranges),
 *          - Figure 50 (worked block value), Figure 52 (scale swizzle geometry:
 *            32-row groups, 4-column tiles, 128x4 scales per 512-byte tile),
 *          - Section 11.3.5 and Table 24 prose (OCP floor vs rceil scale rule),
 *          - Eq. 60 (forward / dgrad / wgrad orientations).
 *  [BOOK]  "3.8 Mixed Precision, bf16 & FP8 Training" (LLM stack book)
 *          - "The floating-point formats" (bf16 = RNE on the low 16 bits),
 *          - "Per-tensor scaling and the delayed-scaling recipe" and exercise 6
 *            (scale = 448 / max(amax, 1e-12), q = fp8(x * scale), GEMM output
 *            de-scaled by 1 / (s_x s_w)).
 *  [FP8LM] "FP8-LM: Training FP8 Large Language Models", Section 3.4
 *          (E4M3 / E5M2 ranges; FP8(x) = cast(s x), x ~ FP8(x) / s).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - all-zero block: scale byte 0 (2^-127), payload zeros (sign kept);
 *  - a block holding NaN or Inf: scale byte 0xFF, every payload byte 0x7F;
 *  - zero keeps its sign: -0 and negatives that round to zero encode as 0x80;
 *  - conversions saturate at the largest finite value (the Olmo page), never
 *    producing Inf (the FP8-LM summary's "overflow to infinity" is rejected);
 *  - padding bytes of the swizzled scale layout are 0;
 *  - the order of bytes inside a 512-byte scale tile is
 *      (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4),
 *    tiles ordered row-tile major with the K-tile index fastest.  The pages
 *    give only the tile geometry; this byte order is the library convention
 *    (the public 1D block-scaling-factor layout) and is pinned on the GPU by
 *    GEMM correctness.
 *
 * Parity status: every function here is pinned by tests that do not call the
 * oracle twice (worked values printed on the pages, torch's own float8
 * conversions, brute force over all codes and all bf16 patterns, closed forms
 * and a numpy matmul of independently dequantized operands), except the
 * intra-tile byte order of the swizzle, whose only pin is GEMM correctness.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_E4M3 0
#define ORC_E5M2 1
#define ORC_ROWWISE 1
#define ORC_COLWISE 2
#define ORC_FLOOR 4

/* ------------------------------------------------------------------------ */
/* Scalar codecs                                                             */
/* ------------------------------------------------------------------------ */

/* BF16: 1 sign, 8 exponent (bias 127), 7 mantissa bits; subnormals when the
 * exponent field is 0 ([OLMO] Figure 49 table: smallest subnormal 2^-133). */
double orc_bf16_decode(uint16_t b) {
    int sign = (b >> 15) & 1;
    int ef = (b >> 7) & 0xFF;
    int mf = b & 0x7F;
    double mag;
    if (ef == 0xFF) {
        mag = mf ? NAN : INFINITY;
    } else if (ef == 0) {
        mag = ldexp((double)mf, -126 - 7);
    } else {
        mag = ldexp(1.0 + mf / 128.0, ef - 127);
    }
    return sign ? -mag : mag;
}

/* E4M3 ("fn" variant): bias 7, no infinities, S.1111.111 is NaN, largest
 * finite 448 ([OLMO] Figure 49 table; [FP8LM] Section 3.4). */
double orc_e4m3_decode(uint8_t c) {
    int sign = c >> 7;
    int ef = (c >> 3) & 0xF;
    int mf = c & 7;
    double mag;
    if (ef == 0xF && mf == 7) {
        mag = NAN;
    } else if (ef == 0) {
        mag = ldexp((double)mf, -6 - 3);
    } else {
        mag = ldexp(1.0 + mf / 8.0, ef - 7);
    }
    return sign ? -mag : mag;
}

/* E5M2: bias 15, IEEE-like (exponent 31 is Inf / NaN), largest finite 57344. */
double orc_e5m2_decode(uint8_t c) {
    int sign = c >> 7;
    int ef = (c >> 2) & 0x1F;
    int mf = c & 3;
    double mag;
    if (ef == 0x1F) {
        mag = mf ? NAN : INFINITY;
    } else if (ef == 0) {
        mag = ldexp((double)mf, -14 - 2);
    } else {
        mag = ldexp(1.0 + mf / 4.0, ef - 15);
    }
    return sign ? -mag : mag;
}

double orc_fp8_decode(uint8_t c, int fmt) {
    return fmt == ORC_E5M2 ? orc_e5m2_decode(c) : orc_e4m3_decode(c);
}

/* E8M0: an unsigned power of two, byte = e + 127, 0xFF reserved for NaN
 * ([OLMO] Figure 49 table and Figure 50, "byte 120 = e + 127"). */
double orc_e8m0_decode(uint8_t b) {
    return b == 0xFF ? NAN : ldexp(1.0, (int)b - 127);
}

/* Largest finite positive code of each payload format. */
static int fp8_max_code(int fmt) { return fmt == ORC_E5M2 ? 0x7B : 0x7E; }

/* Saturating round-to-nearest-even encoder: the nearest of the finite codes,
 * ties to the code whose mantissa LSB is 0, magnitudes above the largest
 * finite value clamp to it, zero keeps the sign of v.  Implemented as a
 * binary search over the decoded positive code values (codes are monotone in
 * magnitude), not with bit manipulation. */
uint8_t orc_fp8_encode(double v, int fmt) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    int top = fp8_max_code(fmt);
    /* largest code lo with value(lo) <= a */
    int lo = 0, hi = top;
    if (a >= orc_fp8_decode((uint8_t)top, fmt)) return (uint8_t)(sign | top);
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_fp8_decode((uint8_t)mid, fmt) <= a) lo = mid; else hi = mid;
    }
    /* now value(lo) <= a < value(lo + 1) */
    double below = orc_fp8_decode((uint8_t)lo, fmt);
    double above = orc_fp8_decode((uint8_t)(lo + 1), fmt);
    int code;
    if (a - below < above - a) code = lo;
    else if (a - below > above - a) code = lo + 1;
    else code = (lo % 2 == 0) ? lo : lo + 1;
    return (uint8_t)(sign | code);
}

/* Round a double to BF16 with round-to-nearest-even ([BOOK] "The
 * floating-point formats").  Searches the sorted positive BF16 values. */
uint16_t orc_bf16_round(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    const int top = 0x7F7F; /* largest finite */
    double maxv = orc_bf16_decode((uint16_t)top);
    if (a >= maxv) {
        /* overflow threshold: max + half an ulp of max (2^120) rounds to Inf */
        double half_ulp = ldexp(1.0, 127 - 8);
        if (a >= maxv + half_ulp) return (uint16_t)(sign | 0x7F80);
        return (uint16_t)(sign | top);
    }
    int lo = 0, hi = top;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_bf16_decode((uint16_t)mid) <= a) lo = mid; else hi = mid;
    }
    double below = orc_bf16_decode((uint16_t)lo);
    double above = orc_bf16_decode((uint16_t)(lo + 1));
    int code;
    if (a - below < above - a) code = lo;
    else if (a - below > above - a) code = lo + 1;
    else code = (lo % 2 == 0) ? lo : lo + 1;
    return (uint16_t)(sign | code);
}

/* ------------------------------------------------------------------------ */
/* E8M0 block scale                                                          */
/* ------------------------------------------------------------------------ */

static int clamp_e(int e) { return e < -127 ? -127 : (e > 127 ? 127 : e); }

/* rceil ([OLMO] Section 11.3.5): the smallest power-of-two scale 2^e with
 * amax <= 448 * 2^e, i.e. the ratio amax / 448 rounded up to a power of two.
 * Evaluated exactly: amax = f * 2^x with f in [0.5, 1) (frexp is exact), and
 * 448 = 0.875 * 2^9, so e = x - 9 when f <= 0.875 and x - 8 otherwise.  The
 * candidate is checked against the definition with exact ldexp products.
 * All-zero blocks take the clamp (e = -127, byte 0). */
int orc_e8m0_rceil(double amax) {
    if (isnan(amax) || isinf(amax)) return 0xFF;
    if (amax == 0.0) return 0;
    int x;
    frexp(amax, &x);
    int e = x - 9;
    if (amax > ldexp(448.0, e)) e += 1;
    /* definition: amax <= 448 * 2^e and amax > 448 * 2^(e-1) */
    if (!(amax <= ldexp(448.0, e) && amax > ldexp(448.0, e - 1))) abort();
    return clamp_e(e) + 127;
}

/* OCP v1.0 floor ([OLMO] Section 11.3.5): round the block maximum down to a
 * power of two, then divide by 2^8 (the largest power of two in E4M3):
 * e = floor(log2 amax) - 8.  With amax = f * 2^x, f in [0.5, 1),
 * floor(log2 amax) = x - 1. */
int orc_e8m0_floor(double amax) {
    if (isnan(amax) || isinf(amax)) return 0xFF;
    if (amax == 0.0) return 0;
    int x;
    frexp(amax, &x);
    int e = (x - 1) - 8;
    if (!(ldexp(1.0, e + 8) <= amax && amax < ldexp(1.0, e + 9))) abort();
    return clamp_e(e) + 127;
}

/* ------------------------------------------------------------------------ */
/* Swizzled scale layout ([OLMO] Figure 52 geometry)                         */
/* ------------------------------------------------------------------------ */

/* Bytes of the padded swizzled scale array for a rows x k operand whose
 * 32-value blocks run along k: ceil(rows/128) row tiles x ceil(k/128) K tiles,
 * 512 bytes per tile. */
int64_t orc_scale_bytes(int64_t rows, int64_t k) {
    int64_t rt = (rows + 127) / 128;
    int64_t kt = (k + 127) / 128;
    return rt * kt * 512;
}

/* Byte offset of the logical scale (r, j): row r, K-block j. */
int64_t orc_swizzle_offset(int64_t r, int64_t j, int64_t k) {
    int64_t kt = (k + 127) / 128;
    int64_t tile = (r / 128) * kt + (j / 4);
    return tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4);
}

/* ------------------------------------------------------------------------ */
/* MX quantization ([OLMO] Eq. 58 and Section 11.3.5)                        */
/* ------------------------------------------------------------------------ */

/* Quantize one 32-value block given by a strided view of BF16 bits.  Writes
 * 32 payload bytes at q (stride 1) and returns the scale byte. */
static uint8_t quantize_block(const uint16_t* x, int64_t stride, int floor_rule,
                              uint8_t* q) {
    double vals[32];
    double amax = 0.0;
    int nonfinite = 0;
    for (int i = 0; i < 32; ++i) {
        vals[i] = orc_bf16_decode(x[i * stride]);
        if (isnan(vals[i]) || isinf(vals[i])) nonfinite = 1;
        else if (fabs(vals[i]) > amax) amax = fabs(vals[i]);
    }
    if (nonfinite) {
        for (int i = 0; i < 32; ++i) q[i] = 0x7F;
        return 0xFF;
    }
    int byte = floor_rule ? orc_e8m0_floor(amax) : orc_e8m0_rceil(amax);
    int e = byte - 127;
    for (int i = 0; i < 32; ++i) {
        double v = ldexp(vals[i], -e); /* x / s, exact in FP64 */
        q[i] = orc_fp8_encode(v, ORC_E4M3);
    }
    return (uint8_t)byte;
}

/* Rowwise output: q_row is rows x cols (row stride cols), blocks along cols,
 * scales in the swizzled layout of a rows x cols operand.
 * Colwise output: q_col is cols x rows (row stride rows) = the transposed
 * matrix, blocks along the original rows, scales in the swizzled layout of a
 * cols x rows operand.  Scale buffers are fully written (padding = 0). */
void orc_quantize_mx(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                     int flags, uint8_t* q_row, uint8_t* s_row,
                     uint8_t* q_col, uint8_t* s_col) {
    int floor_rule = (flags & ORC_FLOOR) != 0;
    if (flags & ORC_ROWWISE) {
        memset(s_row, 0, (size_t)orc_scale_bytes(rows, cols));
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            for (int64_t j = 0; j < cols / 32; ++j) {
                uint8_t byte = quantize_block(x + r * ld + j * 32, 1, floor_rule,
                                              q_row + r * cols + j * 32);
                s_row[orc_swizzle_offset(r, j, cols)] = byte;
            }
        }
    }
    if (flags & ORC_COLWISE) {
        memset(s_col, 0, (size_t)orc_scale_bytes(cols, rows));
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; ++c) {
            for (int64_t j = 0; j < rows / 32; ++j) {
                uint8_t byte = quantize_block(x + (j * 32) * ld + c, ld, floor_rule,
                                              q_col + c * rows + j * 32);
                s_col[orc_swizzle_offset(c, j, rows)] = byte;
            }
        }
    }
}

/* Grouped rowwise quantization of a row-sorted, expert-dispatched matrix:
 * group g owns rows [off[g], off[g+1]); its scale rows start at the padded row
 * P_g = sum_{h<g} ceil(m_h / 128) * 128 of one swizzled array whose row count
 * is the sum of the padded group sizes. */
void orc_quantize_mx_grouped(const uint16_t* x, int64_t cols, int64_t ld,
                             const int32_t* off, int32_t groups, int flags,
                             uint8_t* q_row, uint8_t* s_row, int64_t s_bytes) {
    int floor_rule = (flags & ORC_FLOOR) != 0;
    memset(s_row, 0, (size_t)s_bytes);
    int64_t padded = 0;
    for (int32_t g = 0; g < groups; ++g) {
        int64_t m = (int64_t)off[g + 1] - off[g];
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < m; ++i) {
            int64_t r = off[g] + i;
            for (int64_t j = 0; j < cols / 32; ++j) {
                uint8_t byte = quantize_block(x + r * ld + j * 32, 1, floor_rule,
                                              q_row + r * cols + j * 32);
                s_row[orc_swizzle_offset(padded + i, j, cols)] = byte;
            }
        }
        padded += (m + 127) / 128 * 128;
    }
}

/* MX dequantization to BF16 ([OLMO] Eq. 58, x^ = s q; Section 11.4.3: a
 * saved MXFP8 activation is dequantized when a BF16 consumer needs it).
 * out[r, c] = bf16_RNE(E4M3(q[r, c]) * 2^(byte(r, c/32) - 127)), computed
 * exactly in FP64 and rounded once (overflow to Inf, NaN codes / NaN scales
 * give NaN).  q is rows x cols (row stride cols); s is the swizzled array of
 * a rows x cols operand; out has row stride ldo. */
void orc_dequantize_mx(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t cols,
                       uint16_t* out, int64_t ldo) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t sb = s[orc_swizzle_offset(r, c / 32, cols)];
            double v = orc_e4m3_decode(q[r * cols + c]) * orc_e8m0_decode(sb);
            out[r * ldo + c] = orc_bf16_round(v);
        }
    }
}

/* Grouped form of orc_dequantize_mx: q rows keep their positions; row r of
 * group g reads its scales from padded row P_g + (r - off[g]) of the grouped
 * array (layout of orc_quantize_mx_grouped). */
void orc_dequantize_mx_grouped(const uint8_t* q, const uint8_t* s, const int32_t* off,
                               int32_t groups, int64_t cols, uint16_t* out, int64_t ldo) {
    int64_t padded = 0;
    for (int32_t g = 0; g < groups; ++g) {
        int64_t m = (int64_t)off[g + 1] - off[g];
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < m; ++i) {
            int64_t r = off[g] + i;
            for (int64_t c = 0; c < cols; ++c) {
                uint8_t sb = s[orc_swizzle_offset(padded + i, c / 32, cols)];
                double v = orc_e4m3_decode(q[r * cols + c]) * orc_e8m0_decode(sb);
                out[r * ldo + c] = orc_bf16_round(v);
            }
        }
        padded += (m + 127) / 128 * 128;
    }
}

/* SwiGLU of an up/gate output row pair ([OLMO] Section 11.4.1: the hidden
 * representation that feeds the down projection): y = g sigma(g) u with
 * sigma(g) = 1 / (1 + e^-g), gate g = h[r, c] and up u = h[r, f + c] for
 * c < f.  FP64; sigma is evaluated as e^g / (1 + e^g) for g < 0 so that no
 * intermediate overflows.  out is rows x f (row stride f). */
void orc_swiglu(const uint16_t* h, int64_t rows, int64_t f, int64_t ld, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < f; ++c) {
            double g = orc_bf16_decode(h[r * ld + c]);
            double u = orc_bf16_decode(h[r * ld + f + c]);
            double sig;
            if (g >= 0.0) {
                sig = 1.0 / (1.0 + exp(-g));
            } else {
                double e = exp(g);
                sig = e / (1.0 + e);
            }
            out[r * f + c] = g * sig * u;
        }
    }
}

/* Running count of SwiGLU values whose rounding side could not be decided in
 * FP64 (never observed; the Python wrapper raises when it grows). */
int64_t orc_swiglu_undecided = 0;

/* The correctly rounded BF16 value of y = g sigma(g) u ([OLMO] Section
 * 11.4.1; the hidden value an unfused SwiGLU stores in BF16).
 *
 * For a finite g != 0 and u != 0, e^-g is transcendental (g is rational;
 * Lindemann-Weierstrass), so y is irrational and never equals a BF16 rounding
 * midpoint: round-to-nearest never meets a tie.  The FP64 value v of
 * orc_swiglu lies within a few 2^-53 |y| of y, so wherever v is farther than
 * 2^-44 |v| from every midpoint, bf16_RNE(v) is the rounding of y.  Next to a
 * midpoint m the side of |y| against m is decided from forms without the
 * cancellation of |p| sigma(g) - m (p = g u, exact in FP64):
 *   g > 0:  |y| = |p| / (1 + e^-g),    |y| > m  <=>  (|p| - m) - m e^-g > 0,
 *           where |p| - m is exact (m lies within a factor of 2 of |p|) and
 *           |p| == m puts |y| below m whatever the size of e^-g > 0;
 *   g < 0:  |y| = |p| e^g / (1 + e^g), |y| > m  <=>  e^g (|p| - m) - m > 0;
 * for |g| < 1 the same forms are rewritten around |p| - 2m with expm1 (see
 * below), since e^-|g| rounds to 1 in FP64 for |g| < 2^-54.  A form whose
 * value lies within 2^-48 of the magnitude of its rounded term counts as
 * undecided (the result then falls back to bf16_RNE(v)). */
static uint16_t swiglu_bf16_one(double g, double u, int64_t* undecided) {
    double v;
    if (g >= 0.0) {
        v = g * (1.0 / (1.0 + exp(-g))) * u;
    } else {
        double e = exp(g);
        v = g * (e / (1.0 + e)) * u;
    }
    if (!isfinite(v) || v == 0.0) return orc_bf16_round(v);
    double a = fabs(v);
    /* consecutive BF16 magnitudes below <= a < above (2^128 past the largest) */
    int lo = 0, hi = 0x7F80;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_bf16_decode((uint16_t)mid) <= a) lo = mid; else hi = mid;
    }
    double below = orc_bf16_decode((uint16_t)lo);
    double above = lo == 0x7F7F ? ldexp(1.0, 128) : orc_bf16_decode((uint16_t)(lo + 1));
    double m = 0.5 * (below + above); /* exact: both are multiples of 2^-133 */
    if (fabs(a - m) > ldexp(a, -44)) return orc_bf16_round(v);
    double ap = fabs(g * u);
    int up;
    if (fabs(g) < 1.0) {
        /* near g = 0, with t = 1 + expm1(-|g|) the forms become
         *   g > 0:  (|p| - 2m) - m expm1(-g),   g < 0:  (|p| - 2m) + expm1(g) (|p| - m),
         * |p| - 2m exact (m lies between |p| / 4 and |p|); so |p| == 2m puts |y|
         * on the side of the sign of g however small g is */
        double e = g > 0.0 ? -m * expm1(-g) : expm1(g) * (ap - m);
        double z = (ap - 2.0 * m) + e;
        if (fabs(z) <= ldexp(fabs(e), -48)) {
            ++*undecided;
            return orc_bf16_round(v);
        }
        up = z > 0.0;
    } else if (g > 0.0) {
        double d = ap - m;
        if (d == 0.0) {
            up = 0;
        } else {
            double mt = m * exp(-g);
            double z = d - mt;
            if (fabs(z) <= ldexp(mt, -48)) {
                ++*undecided;
                return orc_bf16_round(v);
            }
            up = z > 0.0;
        }
    } else {
        double t = exp(g);
        double z = t * (ap - m) - m;
        if (fabs(z) <= ldexp(m, -48)) {
            ++*undecided;
            return orc_bf16_round(v);
        }
        up = z > 0.0;
    }
    return (uint16_t)((signbit(v) ? 0x8000 : 0) | (up ? lo + 1 : lo));
}

/* orc_swiglu rounded to BF16 bits with swiglu_bf16_one; out is rows x f. */
void orc_swiglu_bf16(const uint16_t* h, int64_t rows, int64_t f, int64_t ld, uint16_t* out) {
    int64_t undecided = 0;
#pragma omp parallel for schedule(static) reduction(+ : undecided)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < f; ++c) {
            double g = orc_bf16_decode(h[r * ld + c]);
            double u = orc_bf16_decode(h[r * ld + f + c]);
            out[r * f + c] = swiglu_bf16_one(g, u, &undecided);
        }
    }
    orc_swiglu_undecided += undecided;
}

/* Route-weighted gradient rows of combine backward ([OLMO] Section 11.4.1):
 * row i = bf16_RNE(w_i * dy[tok_i]); the product of a BF16 value and an fp32
 * weight is exact in FP64, so this is one rounding of the exact product.
 * An index outside [0, tokens) gives a zero row.  out is rows x cols. */
void orc_route_weight(const uint16_t* dy, int64_t tokens, int64_t ld, const int32_t* tok,
                      const float* w, int64_t rows, int64_t cols, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        int64_t t = tok[i];
        for (int64_t c = 0; c < cols; ++c) {
            double v = 0.0;
            if (t >= 0 && t < tokens) v = (double)w[i] * orc_bf16_decode(dy[t * ld + c]);
            out[i * cols + c] = orc_bf16_round(v);
        }
    }
}

/* Dequantize one operand row ([OLMO] Eq. 58: x^ = s q). */
static void deq_row(const uint8_t* q, const uint8_t* s, int64_t r, int64_t k,
                    int64_t s_row_base, double* out) {
    for (int64_t i = 0; i < k; ++i) {
        uint8_t sb = s[orc_swizzle_offset(s_row_base + r, i / 32, k)];
        out[i] = orc_e4m3_decode(q[r * k + i]) * orc_e8m0_decode(sb);
    }
}

/* ------------------------------------------------------------------------ */
/* Per-tensor FP8 quantization ([BOOK] exercise 6; [FP8LM] Section 3.4)      */
/* ------------------------------------------------------------------------ */

/* amax = max |x| (exact, then held as fp32); s = fp32(fmax / max(amax, 1e-12))
 * with fmax 448 (E4M3) or 57344 (E5M2), one rounding of the exact quotient;
 * y = fp32(x * s), one rounding of the exact product; q = saturating RNE FP8.
 * The product is exact in FP64 (8-bit times 24-bit significands), and the
 * quotient rounds correctly through FP64 then FP32 (53 >= 2 * 24 + 2). */
void orc_quantize_tensor(const uint16_t* x, int64_t n, int fmt,
                         float* amax_out, float* scale_out, uint8_t* q) {
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double a = fabs(orc_bf16_decode(x[i]));
        if (a > amax || isnan(a)) amax = a;
    }
    float amax_f = (float)amax; /* exact: a bf16 magnitude */
    double floor_v = (double)1e-12f;
    double denom = amax > floor_v ? amax : floor_v;
    double fmax = fmt == ORC_E5M2 ? 57344.0 : 448.0;
    float s = (float)(fmax / denom);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float y = (float)(orc_bf16_decode(x[i]) * (double)s);
        q[i] = orc_fp8_encode((double)y, fmt);
    }
    *amax_out = amax_f;
    *scale_out = s;
}

/* Number of payload codes equal to the largest finite code (either sign):
 * the numerator of [FP8LM]'s overflow ratio (Section 2.1, automatic scaling:
 * "values that hit the maximum representable value after the cast"). */
static int64_t count_saturated(const uint8_t* q, int64_t n, int fmt) {
    int64_t c = 0;
    int maxc = fp8_max_code(fmt);
    for (int64_t i = 0; i < n; ++i) c += (q[i] & 0x7F) == maxc;
    return c;
}

/* Per-tensor cast with a given scale ([BOOK] delayed-scaling sketch: the
 * cast uses a scale fixed before this tensor's amax is known; [FP8LM]
 * Section 2.1 Eq. 3, g' = mu g, is the case s = mu):
 * q = FP8(fp32(x s)), saturating RNE; also amax = max |x| (NaN wins) and the
 * number of saturated payloads. */
void orc_quantize_tensor_scaled(const uint16_t* x, int64_t n, int fmt, float s, uint8_t* q,
                                float* amax_out, int64_t* sat_out) {
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double a = fabs(orc_bf16_decode(x[i]));
        if (a > amax || isnan(a)) amax = a;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float y = (float)(orc_bf16_decode(x[i]) * (double)s); /* exact product, one rounding */
        q[i] = orc_fp8_encode((double)y, fmt);
    }
    *amax_out = (float)amax;
    *sat_out = count_saturated(q, n, fmt);
}

/* The delayed scale ([BOOK] sketch, compute_scale): a = the largest entry
 * of the amax history (NaN propagates), clamped below at fp32(1e-12);
 * s = fp32(fp32(fmax / a) * margin). */
float orc_delayed_scale(const float* hist, int32_t h, int fmt, float margin) {
    double a = 0.0;
    int seen = 0;
    for (int32_t i = 0; i < h; ++i) {
        double v = hist[i];
        if (!seen || v > a || isnan(v)) a = v;
        seen = 1;
        if (isnan(a)) break;
    }
    double floor_v = (double)1e-12f;
    if (!(a >= floor_v) && !isnan(a)) a = floor_v;
    double fmax = fmt == ORC_E5M2 ? 57344.0 : 448.0;
    float s = (float)(fmax / a);
    return (float)((double)s * (double)margin);
}

/* One delayed-scaling cast ([BOOK] sketch, cast_to_fp8): the scale from the
 * history as it stands, the cast of x with it, then history[pos] = amax(x)
 * and pos = (pos + 1) % h. */
void orc_quantize_tensor_delayed(const uint16_t* x, int64_t n, int fmt, float margin,
                                 float* hist, int32_t h, int32_t* pos, float* scale_out,
                                 uint8_t* q, float* amax_out, int64_t* sat_out) {
    float s = orc_delayed_scale(hist, h, fmt, margin);
    orc_quantize_tensor_scaled(x, n, fmt, s, q, amax_out, sat_out);
    hist[*pos] = *amax_out;
    *pos = (*pos + 1) % h;
    *scale_out = s;
}

/* Requantization to a shared scale ([FP8LM] Section 2.1, Eq. 4-5): with the
 * group's scale s_out = min over ranks of s_in, q'' = FP8(s_out (g' / s_in))
 * evaluated in that order in fp32: t = fp32(decode(q) / s_in),
 * y = fp32(s_out t), saturating RNE to fmt_out.  Also counts saturated
 * payloads. */
void orc_requantize_tensor(const uint8_t* q_in, int64_t n, int fmt_in, float s_in, float s_out,
                           int fmt_out, uint8_t* q_out, int64_t* sat_out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float t = (float)(orc_fp8_decode(q_in[i], fmt_in) / (double)s_in);
        float y = (float)((double)s_out * (double)t);
        q_out[i] = orc_fp8_encode((double)y, fmt_out);
    }
    *sat_out = count_saturated(q_out, n, fmt_out);
}

/* ------------------------------------------------------------------------ */
/* GEMMs: C = A B^T on dequantized operands, FP64 ([OLMO] Eq. 60 operands,  */
/* Section 11.1.1: block scales applied inside the product)                  */
/* ------------------------------------------------------------------------ */

/* MX GEMM on selected output rows.  A: M x K payload (row stride K) with its
 * swizzled scales, B: N x K likewise.  out: nrows x N (row i is C[rows[i]]).
 * rows == NULL means all M rows in order. */
void orc_gemm_mx_rows(const uint8_t* qa, const uint8_t* sa, const uint8_t* qb,
                      const uint8_t* sb, int64_t M, int64_t N, int64_t K,
                      const int64_t* rows, int64_t nrows, double* out) {
    (void)M;
    double* bd = (double*)malloc(sizeof(double) * (size_t)(N * K));
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) deq_row(qb, sb, n, K, 0, bd + n * K);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        double* ad = (double*)malloc(sizeof(double) * (size_t)K);
        deq_row(qa, sa, m, K, 0, ad);
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            const double* b = bd + n * K;
            for (int64_t k = 0; k < K; ++k) acc += ad[k] * b[k];
            out[i * N + n] = acc;
        }
        free(ad);
    }
    free(bd);
}

/* Per-tensor GEMM ([BOOK] exercise 6): C = (sum_k q_a q_b) / (s_a s_b). */
void orc_gemm_tensor_rows(const uint8_t* qa, int fa, float s_a, const uint8_t* qb,
                          int fb, float s_b, int64_t M, int64_t N, int64_t K,
                          const int64_t* rows, int64_t nrows, double* out) {
    (void)M;
    double* bd = (double*)malloc(sizeof(double) * (size_t)(N * K));
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) bd[n * K + k] = orc_fp8_decode(qb[n * K + k], fb);
    double descale = (double)s_a * (double)s_b;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t m = rows ? rows[i] : i;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += orc_fp8_decode(qa[m * K + k], fa) * bd[n * K + k];
            out[i * N + n] = acc / descale;
        }
    }
    free(bd);
}

/* Grouped MX GEMM: for each group g, C[off[g]:off[g+1]] = A_g W_g^T, where
 * A's scales use the grouped padded layout of orc_quantize_mx_grouped and
 * expert g's weight is the N x K matrix at qw + g*N*K with its own swizzled
 * scale array at sw + g * orc_scale_bytes(N, K).  Computes the output rows
 * listed in rows (global row indices, ascending); out row i is C[rows[i]].
 * rows == NULL means all rows in order (nrows = off[groups]). */
void orc_gemm_grouped_rows(const uint8_t* qa, const uint8_t* sa, const uint8_t* qw,
                           const uint8_t* sw, const int32_t* off, int32_t groups,
                           int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                           double* out) {
    int64_t wsb = orc_scale_bytes(N, K);
    int64_t padded = 0;
    int64_t next = 0; /* first entry of rows not yet computed */
    double* bd = (double*)malloc(sizeof(double) * (size_t)(N * K));
    for (int32_t g = 0; g < groups; ++g) {
        int64_t m = (int64_t)off[g + 1] - off[g];
        /* the wanted rows of this group: entries [first, last) of rows */
        int64_t first = next, last = next;
        if (rows) {
            while (last < nrows && rows[last] < off[g + 1]) ++last;
        } else {
            first = off[g];
            last = off[g + 1];
        }
        next = last;
        if (last > first) {
            const uint8_t* qg = qw + (int64_t)g * N * K;
            const uint8_t* sg = sw + (int64_t)g * wsb;
#pragma omp parallel for schedule(static)
            for (int64_t n = 0; n < N; ++n) deq_row(qg, sg, n, K, 0, bd + n * K);
#pragma omp parallel for schedule(static)
            for (int64_t i = first; i < last; ++i) {
                int64_t r = rows ? rows[i] : i;
                int64_t local = r - off[g];
                double* ad = (double*)malloc(sizeof(double) * (size_t)K);
                /* A row r is row `local` of group g, at padded scale row padded + local */
                for (int64_t k = 0; k < K; ++k) {
                    uint8_t s = sa[orc_swizzle_offset(padded + local, k / 32, K)];
                    ad[k] = orc_e4m3_decode(qa[r * K + k]) * orc_e8m0_decode(s);
                }
                for (int64_t n = 0; n < N; ++n) {
                    double acc = 0.0;
                    const double* b = bd + n * K;
                    for (int64_t k = 0; k < K; ++k) acc += ad[k] * b[k];
                    out[i * N + n] = acc;
                }
                free(ad);
            }
        }
        padded += (m + 127) / 128 * 128;
    }
    free(bd);
}

/* ------------------------------------------------------------------------ */
/* Array forms of the scalar codecs, for the Python wrapper                  */
/* ------------------------------------------------------------------------ */

void orc_bf16_decode_array(const uint16_t* b, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_decode(b[i]);
}
void orc_fp8_decode_array(const uint8_t* c, int64_t n, int fmt, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_decode(c[i], fmt);
}
void orc_fp8_encode_array(const double* v, int64_t n, int fmt, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_encode(v[i], fmt);
}
void orc_bf16_round_array(const double* v, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_round(v[i]);
}
void orc_e8m0_array(const double* amax, int64_t n, int floor_rule, int32_t* out) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = floor_rule ? orc_e8m0_floor(amax[i]) : orc_e8m0_rceil(amax[i]);
}

/* Threads the OpenMP loops above use (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int orc_num_threads(void) { return omp_get_max_threads(); }
#else
int orc_num_threads(void) { return 1; }
#endif
