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
//
// All three share the quantizer's 128 x 128 tile walk: blockIdx.x is a
// 128-row scale tile (group-padded when offsets are given), blockIdx.y a
// 128-column tile; a half-warp covers one tile row, 8 columns per lane.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "mx_common.cuh"

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

template <bool GROUPED>
__global__ void __launch_bounds__(kThreads)
    dequantize_mx_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                         int64_t rows, int64_t cols, const int32_t* offsets, int groups,
                         uint16_t* __restrict__ out, int64_t ldo, int64_t nkc) {
    int64_t row_begin, row_end;
    if (!tile_rows<GROUPED>(offsets, groups, rows, &row_begin, &row_end)) return;
    const int tid = threadIdx.x;
    const int seg = tid & 15;
    const int64_t col = static_cast<int64_t>(blockIdx.y) * kTile + seg * 8;
    const uint8_t* s_tile = s + (static_cast<int64_t>(blockIdx.x) * nkc + blockIdx.y) * 512;
    uint2 qv[8];
    uint32_t sw[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = it * 16 + (tid >> 4);
        const int64_t row = row_begin + r;
        const bool in = row < row_end && col < cols;
        qv[it] = in ? __ldcs(reinterpret_cast<const uint2*>(q + row * cols + col)) : make_uint2(0u, 0u);
        sw[it] = in ? __ldg(reinterpret_cast<const uint32_t*>(s_tile + swz_word(r))) : 0u;
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = it * 16 + (tid >> 4);
        const int64_t row = row_begin + r;
        if (row < row_end && col < cols) {
            const float sc = e8m0_value((sw[it] >> (8 * (seg >> 2))) & 0xFFu);
            uint4 o;
            o.x = dq2(qv[it].x & 0xFFFFu, sc);
            o.y = dq2(qv[it].x >> 16, sc);
            o.z = dq2(qv[it].y & 0xFFFFu, sc);
            o.w = dq2(qv[it].y >> 16, sc);
            *reinterpret_cast<uint4*>(out + row * ldo + col) = o;
        }
    }
}

// ------------------------------------------------------ SwiGLU + Q ------

__device__ __forceinline__ uint32_t bf16_bits_rn(float v) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ uint32_t bf16_bits_rn(double v) {
    return __bfloat16_as_ushort(__double2bfloat16(v));
}

// bf16_RNE(g sigma(g) u), sigma(g) = 1 / (1 + e^-g).  For g >= -80 the value
// is formed in fp32 from e^-|g| (never overflows; a normal number), with
// sigma = 1/(1+t) for g >= 0 and t/(1+t) below 0; with CUDA's expf error of
// at most 2 ulp the fp32 value is within 1.25 * 2^-21 relative of the exact
// one (plus an absolute 2^-149 where the product underflows), so the BF16
// result is the correctly rounded one unless the exact value lies that close
// to a rounding midpoint, where it may be the neighbour.  The product is
// taken as (g sigma) u, or (g u) sigma when |g| < 2^-100 so that g sigma never
// loses bits to fp32 underflow.  Below -80, where e^g leaves fp32's normal
// range, the value is formed in double and rounded once.
__device__ __forceinline__ uint32_t swiglu_bf16(float g, float u) {
    if (!(g >= -80.f)) {  // also NaN
        const double gd = g;
        const double e = exp(gd);
        return bf16_bits_rn(gd * (e / (1.0 + e)) * static_cast<double>(u));
    }
    const float t = expf(-fabsf(g));
    const float sig = __fdiv_rn(g >= 0.f ? 1.f : t, __fadd_rn(1.f, t));
    const float y = fabsf(g) < 0x1p-100f ? __fmul_rn(__fmul_rn(g, u), sig)
                                         : __fmul_rn(__fmul_rn(g, sig), u);
    return bf16_bits_rn(y);
}

__device__ __forceinline__ uint32_t swiglu2(uint32_t g2, uint32_t u2) {
    return swiglu_bf16(bf16_lo(g2), bf16_lo(u2)) | (swiglu_bf16(bf16_hi(g2), bf16_hi(u2)) << 16);
}

template <bool FLOOR, bool GROUPED>
__global__ void __launch_bounds__(kThreads)
    swiglu_quant_kernel(const uint16_t* __restrict__ h, int64_t rows, int64_t f, int64_t ld,
                        const int32_t* offsets, int groups, uint8_t* __restrict__ q,
                        uint8_t* __restrict__ s, int64_t nkc) {
    int64_t row_begin, row_end;
    if (!tile_rows<GROUPED>(offsets, groups, rows, &row_begin, &row_end)) return;
    const int tid = threadIdx.x;
    const int seg = tid & 15;
    const int64_t col = static_cast<int64_t>(blockIdx.y) * kTile + seg * 8;
    uint4 gv[8], uv[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int64_t row = row_begin + it * 16 + (tid >> 4);
        if (row < row_end && col < f) {
            gv[it] = __ldcs(reinterpret_cast<const uint4*>(h + row * ld + col));
            uv[it] = __ldcs(reinterpret_cast<const uint4*>(h + row * ld + f + col));
        } else {
            gv[it] = make_uint4(0u, 0u, 0u, 0u);
            uv[it] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    uint8_t* s_tile = s + (static_cast<int64_t>(blockIdx.x) * nkc + blockIdx.y) * 512;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = it * 16 + (tid >> 4);
        const int64_t row = row_begin + r;
        const bool in = row < row_end && col < f;
        uint4 v;
        v.x = swiglu2(gv[it].x, uv[it].x);
        v.y = swiglu2(gv[it].y, uv[it].y);
        v.z = swiglu2(gv[it].z, uv[it].z);
        v.w = swiglu2(gv[it].w, uv[it].w);
        mx_row_step<FLOOR>(v, r, in ? q + row * f + col : nullptr, s_tile);
    }
}

// ------------------------------------------- route weighting + Q --------

// bf16_RNE(x w) of a BF16 x and an fp32 w, rounded once from the exact
// product.  The product has at most 32 significant bits, so it is first
// rounded to fp32 toward zero with the lowest bit forced to 1 when inexact
// (round-to-odd; the FMA residual is exact for normal products), and the
// RNE rounding of that to BF16, 16 bits shorter, equals the RNE rounding of
// the exact product.  Products below fp32's normal range are formed in
// double (exact there) and rounded once.
__device__ __forceinline__ uint32_t weighted_bf16(float x, float w) {
    const float p = __fmul_rz(x, w);
    if (fabsf(p) < 0x1p-126f) {
        return bf16_bits_rn(static_cast<double>(x) * static_cast<double>(w));
    }
    uint32_t b = __float_as_uint(p);
    if (isfinite(p) && __fmaf_rn(x, w, -p) != 0.f) b |= 1u;
    return bf16_bits_rn(__uint_as_float(b));
}

__device__ __forceinline__ uint32_t weighted2(uint32_t x2, float w) {
    return weighted_bf16(bf16_lo(x2), w) | (weighted_bf16(bf16_hi(x2), w) << 16);
}

template <bool FLOOR, bool GROUPED>
__global__ void __launch_bounds__(kThreads)
    weighted_quant_kernel(const uint16_t* __restrict__ dy, int64_t tokens, int64_t ld,
                          const int32_t* __restrict__ row_token, const float* __restrict__ row_weight,
                          int64_t rows, int64_t cols, const int32_t* offsets, int groups,
                          uint8_t* __restrict__ q, uint8_t* __restrict__ s, int64_t nkc) {
    int64_t row_begin, row_end;
    if (!tile_rows<GROUPED>(offsets, groups, rows, &row_begin, &row_end)) return;
    const int tid = threadIdx.x;
    const int seg = tid & 15;
    const int64_t col = static_cast<int64_t>(blockIdx.y) * kTile + seg * 8;
    uint4 xv[8];
    float wv[8];
    bool bad = false;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int64_t row = row_begin + it * 16 + (tid >> 4);
        xv[it] = make_uint4(0u, 0u, 0u, 0u);
        wv[it] = 0.f;
        if (row < row_end && col < cols) {
            const int64_t t = __ldg(row_token + row);
            if (t >= 0 && t < tokens) {
                xv[it] = __ldcs(reinterpret_cast<const uint4*>(dy + t * ld + col));
                wv[it] = __ldg(row_weight + row);
            } else {
                bad = true;
            }
        }
    }
    if (bad) record_status(MXFP8_ERR_DEVICE_CHECK);
    uint8_t* s_tile = s + (static_cast<int64_t>(blockIdx.x) * nkc + blockIdx.y) * 512;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = it * 16 + (tid >> 4);
        const int64_t row = row_begin + r;
        const bool in = row < row_end && col < cols;
        uint4 v;
        v.x = weighted2(xv[it].x, wv[it]);
        v.y = weighted2(xv[it].y, wv[it]);
        v.z = weighted2(xv[it].z, wv[it]);
        v.w = weighted2(xv[it].w, wv[it]);
        mx_row_step<FLOOR>(v, r, in ? q + row * cols + col : nullptr, s_tile);
    }
}

// Grid of a tile walk: plain operands have ceil(rows/128) row tiles; a
// group-padded one at most floor(rows/128) + groups.
bool tile_grid(int64_t rows, int64_t cols, bool grouped, int groups, dim3* grid) {
    const int64_t row_tiles = grouped ? rows / kTile + groups : (rows + kTile - 1) / kTile;
    const int64_t col_tiles = (cols + kTile - 1) / kTile;
    if (row_tiles > 0x7FFFFFFF || col_tiles > 65535) return false;
    *grid = dim3(static_cast<unsigned>(row_tiles), static_cast<unsigned>(col_tiles));
    return true;
}

}  // namespace

cudaError_t launch_dequantize_mx(const DequantArgs& a, cudaStream_t st) {
    dim3 grid;
    const bool grouped = a.offsets != nullptr;
    if (!tile_grid(a.rows, a.cols, grouped, a.groups, &grid)) return cudaErrorInvalidValue;
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    const int64_t nkc = (a.cols + kTile - 1) / kTile;
    if (grouped) {
        dequantize_mx_kernel<true><<<grid, kThreads, 0, st>>>(a.q, a.s, a.rows, a.cols, a.offsets,
                                                             a.groups, a.out, a.ldo, nkc);
    } else {
        dequantize_mx_kernel<false><<<grid, kThreads, 0, st>>>(a.q, a.s, a.rows, a.cols, nullptr, 0,
                                                              a.out, a.ldo, nkc);
    }
    return cudaGetLastError();
}

cudaError_t launch_swiglu_quantize_mx(const SwigluQuantArgs& a, cudaStream_t st) {
    dim3 grid;
    const bool grouped = a.offsets != nullptr;
    const bool fl = a.flags & MX_SCALE_FLOOR;
    if (!tile_grid(a.rows, a.f, grouped, a.groups, &grid)) return cudaErrorInvalidValue;
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    const int64_t nkc = (a.f + kTile - 1) / kTile;
#define MXFP8_SWIGLU(FL, GR) \
    swiglu_quant_kernel<FL, GR><<<grid, kThreads, 0, st>>>(a.h, a.rows, a.f, a.ld, a.offsets, \
                                                            a.groups, a.q, a.s, nkc)
    if (grouped) {
        if (fl) MXFP8_SWIGLU(true, true); else MXFP8_SWIGLU(false, true);
    } else {
        if (fl) MXFP8_SWIGLU(true, false); else MXFP8_SWIGLU(false, false);
    }
#undef MXFP8_SWIGLU
    return cudaGetLastError();
}

cudaError_t launch_weighted_quantize_mx(const WeightedQuantArgs& a, cudaStream_t st) {
    dim3 grid;
    const bool grouped = a.offsets != nullptr;
    const bool fl = a.flags & MX_SCALE_FLOOR;
    if (!tile_grid(a.rows, a.cols, grouped, a.groups, &grid)) return cudaErrorInvalidValue;
    if (grid.x == 0 || grid.y == 0) return cudaSuccess;
    const int64_t nkc = (a.cols + kTile - 1) / kTile;
#define MXFP8_WEIGHTED(FL, GR)                                                               \
    weighted_quant_kernel<FL, GR><<<grid, kThreads, 0, st>>>(                                \
        a.dy, a.tokens, a.ld, a.row_token, a.row_weight, a.rows, a.cols, a.offsets, a.groups, \
        a.q, a.s, nkc)
    if (grouped) {
        if (fl) MXFP8_WEIGHTED(true, true); else MXFP8_WEIGHTED(false, true);
    } else {
        if (fl) MXFP8_WEIGHTED(true, false); else MXFP8_WEIGHTED(false, false);
    }
#undef MXFP8_WEIGHTED
    return cudaGetLastError();
}

cudaError_t take_status_fused(unsigned* out) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status_fused, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status_fused, &zero, sizeof(unsigned));
}

}  // namespace mxfp8
