// Device helpers shared by the MX quantizer kernels (quantize.cu) and the
// fused producers that quantize what they compute (fused.cu): the E8M0 rule
// from a BF16 amax, saturating FP8 conversion, the swizzled scale-tile
// position of a row, the row-tile lookup of group-padded (per-expert)
// operands, and one rowwise quantization step of a 128 x 128 tile.
//
// MX rule ("Olmo-core MoE report, Section 11: MXFP8 Training", Eq. 58 and
// Section 11.3.5): per 32-value block, amax -> E8M0 scale s = 2^e (rceil:
// smallest e with amax <= 448 * 2^e; floor: e = floor(log2 amax) - 8),
// clamped to [-127, 127]; payload q = E4M3(x / s), round to nearest even,
// saturating.  Scale tiles: 128 rows x 4 blocks in 512 bytes (Section 11.3.2).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/mxfp8.h"

namespace mxfp8 {

constexpr int kTile = 128;     // rows and columns of one quantizer tile
constexpr int kThreads = 256;  // 8 warps; each half-warp covers one tile row

// E8M0 byte (e + 127) of a block from the bit pattern of its largest BF16
// magnitude.  BF16 magnitude bits order like the magnitudes, with Inf and
// NaN (>= 0x7F80) above every finite value.  For a normal amax with exponent
// field f and mantissa field m: amax = (1 + m/128) 2^(f-127) and 448 = 1.75 2^8,
// so rceil gives e = f - 135 + (m > 0x60) and floor gives e = f - 135.
// Zero and subnormal amax fall below the clamp (byte 0).
__device__ __forceinline__ uint32_t e8m0_byte(uint32_t amax_bits, bool floor_rule) {
    if (amax_bits >= 0x7F80u) return 0xFFu;
    const int f = static_cast<int>(amax_bits >> 7);
    const int byte = f - 8 + ((!floor_rule && (amax_bits & 0x7Fu) > 0x60u) ? 1 : 0);
    return byte < 0 ? 0u : static_cast<uint32_t>(byte);
}

// 1 / s = 2^(127 - byte) as an fp32 power of two (byte <= 247 for finite
// BF16 input, so the exponent field 254 - byte stays normal).
__device__ __forceinline__ float inv_scale(uint32_t byte) {
    return __uint_as_float((254u - byte) << 23);
}

// Per-half unsigned 16-bit maximum (native on sm_90 and later).
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Per-half unsigned 16-bit minimum.
__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Per-half max(|a|, |b|) of packed BF16 (sign: the XOR of the inputs' signs;
// a NaN input gives the canonical NaN).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Largest BF16 magnitude bits among the 8 values of a 16-byte vector.
__device__ __forceinline__ uint32_t amax8(const uint4& v) {
    uint32_t m = max_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
    m = max_u16x2(m, v.z & 0x7FFF7FFFu);
    m = max_u16x2(m, v.w & 0x7FFF7FFFu);
    return max(m & 0xFFFFu, m >> 16);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 lanes in one 64-bit register pair, for sm_100's packed FP32
// instructions (each lane rounds to nearest exactly as the scalar one does).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_splat(float c) { return f2_pack(c, c); }

// Saturating RNE conversion of two fp32 values; `lo` lands in the low byte.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
    uint16_t r;
    if constexpr (FMT == FP8_E4M3) {
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    } else {
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    }
    return r;
}

// Saturating RNE conversion of four fp32 values into one word (a0 in the
// low byte): the two halves are written as one register pair, which the
// assembler can merge without a separate byte-permute.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x4(float a0, float a1, float b0, float b1) {
    uint32_t r;
    if constexpr (FMT == FP8_E4M3) {
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
            "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
            "mov.b32 %0, {lo, hi};\n\t}"
            : "=r"(r) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
    } else {
        asm("{\n\t.reg .b16 lo, hi;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 lo, %2, %1;\n\t"
            "cvt.rn.satfinite.e5m2x2.f32 hi, %4, %3;\n\t"
            "mov.b32 %0, {lo, hi};\n\t}"
            : "=r"(r) : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
    }
    return r;
}

// Four consecutive BF16 values (two words) times an fp32 factor, each
// product rounded to fp32 and then to FMT: four payload bytes.
template <int FMT>
__device__ __forceinline__ uint32_t quant4_scaled(uint32_t w0, uint32_t w1, float f) {
    const uint64_t F = f2_splat(f);
    float a0, a1, b0, b1;
    f2_unpack(f2_mul(f2_pack(bf16_lo(w0), bf16_hi(w0)), F), a0, a1);
    f2_unpack(f2_mul(f2_pack(bf16_lo(w1), bf16_hi(w1)), F), b0, b1);
    return cvt_fp8x4<FMT>(a0, a1, b0, b1);
}

// Four consecutive BF16 values (two words) times a factor -> four E4M3 bytes.
// The product by a power of two is exact (no FTZ in this file).  PACKED: the
// products in packed FP32 (lane by lane the scalar products; fewer issued
// instructions, but the register pairs cost registers in kernels already at
// their bound).
template <bool PACKED = true>
__device__ __forceinline__ uint32_t quant4_e4m3(uint32_t w0, uint32_t w1, float f) {
    if constexpr (PACKED) {
        return quant4_scaled<FP8_E4M3>(w0, w1, f);
    } else {
        return cvt_fp8x4<FP8_E4M3>(__fmul_rn(bf16_lo(w0), f), __fmul_rn(bf16_hi(w0), f),
                                   __fmul_rn(bf16_lo(w1), f), __fmul_rn(bf16_hi(w1), f));
    }
}

// Same for four values held in the low (or high) halves of four words
// (scalar products: the packed form's register pairs cost the colwise tile
// kernel 18 registers and a CTA per SM for no gain).
template <bool HIGH>
__device__ __forceinline__ uint32_t quant4_half(uint32_t w0, uint32_t w1, uint32_t w2,
                                                uint32_t w3, float f) {
    auto v = [](uint32_t w) { return HIGH ? bf16_hi(w) : bf16_lo(w); };
    return cvt_fp8x4<FP8_E4M3>(__fmul_rn(v(w0), f), __fmul_rn(v(w1), f), __fmul_rn(v(w2), f),
                               __fmul_rn(v(w3), f));
}

// Byte offset, inside its 512-byte tile, of the 4-byte group of scales of
// tile row r (0..127): 32-row groups x 4 K-blocks per tile.
__device__ __forceinline__ int swz_word(int r) { return (r & 31) * 16 + (r >> 5) * 4; }

// Warp 0 of a CTA finds the rows [begin, end) of padded row tile rt of a
// group-padded operand: group g owns ceil(m_g / 128) consecutive 128-row
// tiles, m_g = offsets[g+1] - offsets[g].  It also validates the offsets
// (offsets[0] == 0, non-decreasing, offsets[G] == total).  Results go to
// shared memory: rows[0..1] (-1 past the last tile) and *ok.  The caller
// synchronizes the CTA before reading them.
__device__ __forceinline__ void locate_group_tile(const int32_t* off, int G, int64_t total,
                                                  int64_t rt, int64_t* rows, int* ok_out) {
    const int lane = threadIdx.x & 31;
    bool ok = (off[0] == 0) && (static_cast<int64_t>(off[G]) == total);
    int64_t base = 0, found_begin = -1, found_end = -1;
    for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + lane;
        int64_t tiles = 0, b = 0, e = 0;
        if (g < G) {
            b = off[g];
            e = off[g + 1];
            if (e < b) ok = false;
            tiles = e > b ? (e - b + kTile - 1) / kTile : 0;
        }
        int64_t incl = tiles;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
        const int64_t excl = base + incl - tiles;
        if (g < G && rt >= excl && rt < excl + tiles) {
            found_begin = b + (rt - excl) * kTile;
            found_end = min(e, found_begin + kTile);
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    ok = __all_sync(0xffffffffu, ok);
    const unsigned who = __ballot_sync(0xffffffffu, found_begin >= 0);
    if (lane == 0) {
        *ok_out = ok ? 1 : 0;
        rows[0] = -1;
        rows[1] = -1;
    }
    __syncwarp();
    if (who && lane == __ffs(who) - 1) {
        rows[0] = found_begin;
        rows[1] = found_end;
    }
}

// 32-byte global accesses: one 256-bit instruction when `v8` (the caller
// has checked 32-byte alignment of every address it will use), else two
// 16-byte ones (the library's documented alignment is 16 bytes).  A thread
// owning a whole 32-value block touches whole 32-byte sectors either way,
// but a 256-bit access fetches each sector once per warp instruction.
// ld32_stream: data read once (evict-first); ld32_cached: data that other
// threads read again (gathers); st32: plain store.
__device__ __forceinline__ void ld32_stream(const void* p, uint32_t* r, bool v8) {
    if (v8) {
        asm("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7])
            : "l"(p));
    } else {
        const uint4 a = __ldcs(reinterpret_cast<const uint4*>(p));
        const uint4 b = __ldcs(reinterpret_cast<const uint4*>(p) + 1);
        r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
        r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
    }
}

__device__ __forceinline__ void ld32_cached(const void* p, uint32_t* r, bool v8) {
    if (v8) {
        asm("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
              "=r"(r[7])
            : "l"(p));
    } else {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
        r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
        r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
    }
}

__device__ __forceinline__ void st32(void* p, const uint32_t* r, bool v8) {
    if (v8) {
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r[0]),
                     "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
    } else {
        reinterpret_cast<uint4*>(p)[0] = make_uint4(r[0], r[1], r[2], r[3]);
        reinterpret_cast<uint4*>(p)[1] = make_uint4(r[4], r[5], r[6], r[7]);
    }
}

__device__ __forceinline__ bool aligned32(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 31u) == 0;
}

// Largest BF16 magnitude bits of a 32-value block held by one thread as 16
// words of packed BF16, with the packed BF16 abs-max (one instruction per
// pair of words): the magnitudes of non-NaN BF16 values order like their bit
// patterns, so the masked result is the largest magnitude's bits, and a NaN
// anywhere gives 0x7FFF, which e8m0_byte maps to the NaN scale as it does
// any NaN or Inf bits.
__device__ __forceinline__ uint32_t block32_amax_bits(const uint32_t* w) {
    uint32_t m8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = absmax_bf16x2(w[2 * i], w[2 * i + 1]);
#pragma unroll
    for (int i = 0; i < 4; ++i) m8[i] = absmax_bf16x2(m8[i], m8[i + 4]);
    const uint32_t m2 = absmax_bf16x2(absmax_bf16x2(m8[0], m8[1]), absmax_bf16x2(m8[2], m8[3])) & 0x7FFF7FFFu;
    return max(m2 & 0xFFFFu, m2 >> 16);
}

// MX quantization of one 32-value block held by one thread as 16 words of
// packed BF16 (value 2i in the low half of w[i]) whose largest magnitude's
// bits are amax_bits (block32_amax_bits).  Writes the 32 E4M3 bytes to q_dst
// (skipped when null; 32-byte aligned when v8) and the E8M0 byte to *s_dst.
template <bool FLOOR, bool PACKED = true>
__device__ __forceinline__ void mx_block32_amax(const uint32_t* w, uint32_t amax_bits,
                                                uint8_t* q_dst, uint8_t* s_dst, bool v8) {
    const uint32_t byte = e8m0_byte(amax_bits, FLOOR);
    uint32_t q[8];
    if (byte == 0xFFu) {
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = 0x7F7F7F7Fu;
    } else {
        const float f = inv_scale(byte);
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = quant4_e4m3<PACKED>(w[2 * k], w[2 * k + 1], f);
    }
    if (q_dst != nullptr) st32(q_dst, q, v8);
    *s_dst = static_cast<uint8_t>(byte);
}

// The same with the block maximum taken here.
template <bool FLOOR, bool PACKED = true>
__device__ __forceinline__ void mx_block32(const uint32_t* w, uint8_t* q_dst, uint8_t* s_dst,
                                           bool v8) {
    mx_block32_amax<FLOOR, PACKED>(w, block32_amax_bits(w), q_dst, s_dst, v8);
}

// One rowwise step of a 128 x 128 tile: the half-warp holding tile row r
// (lane & 16 selects the half) has 8 BF16 values per lane in v, lanes
// 4b..4b+3 of the half forming 32-value block b.  Writes the 8 E4M3 bytes to
// q_dst (skipped when null) and, from lane 4b, block b's scale byte into the
// 512-byte scale tile.  All 32 lanes must call it.
template <bool FLOOR>
__device__ __forceinline__ void mx_row_step(const uint4& v, int r, uint8_t* q_dst,
                                            uint8_t* s_tile) {
    const int lane = threadIdx.x & 31;
    uint32_t m = amax8(v);
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const uint32_t byte = e8m0_byte(m, FLOOR);
    uint2 q;
    if (byte == 0xFFu) {
        q = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
    } else {
        const float f = inv_scale(byte);
        q.x = quant4_e4m3(v.x, v.y, f);
        q.y = quant4_e4m3(v.z, v.w, f);
    }
    if (q_dst != nullptr) *reinterpret_cast<uint2*>(q_dst) = q;
    if ((lane & 3) == 0) s_tile[swz_word(r) + ((lane & 15) >> 2)] = static_cast<uint8_t>(byte);
}

}  // namespace mxfp8
