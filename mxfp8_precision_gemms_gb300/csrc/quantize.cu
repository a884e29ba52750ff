// Quantizer kernels: MXFP8 (32-value blocks, E8M0 scales written straight
// into the swizzled tensor-core layout, rowwise and/or colwise from one read
// of the BF16 input) and per-tensor current-scaling FP8 (amax + cast).
//
// MX rule ("Olmo-core MoE report, Section 11: MXFP8 Training", Eq. 58 and
// Section 11.3.5): per block, amax -> E8M0 scale s = 2^e (rceil: smallest e
// with amax <= 448 * 2^e; floor: e = floor(log2 amax) - 8), clamped to
// [-127, 127]; payload q = E4M3(x / s), round to nearest even, saturating.
// Per-tensor rule ("3.8 Mixed Precision, bf16 & FP8 Training", exercise 6):
// s = fp32(fmax / max(amax, 1e-12)), q = FP8(fp32(x * s)).
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "mx_common.cuh"
#include "ptx.cuh"

namespace mxfp8 {

__device__ unsigned int g_status_quant = 0;

namespace {

__device__ __forceinline__ void record_status(unsigned code) {
    atomicCAS(&g_status_quant, 0u, code);
}

// One CTA quantizes a 128 x 128 tile.  blockIdx.x = 128-row scale tile,
// blockIdx.y = 128-column tile.  Rowwise: a half-warp owns one tile row per
// step (16 lanes x 8 values), 4 lanes per 32-value block.  Colwise: the tile
// is staged in shared memory and each thread quantizes two columns of one
// 32-row block.
template <bool ROW, bool COL, bool FLOOR, bool GROUPED>
__global__ void __launch_bounds__(kThreads)
    quantize_mx_kernel(QuantMxArgs a, int64_t nkc_row, int64_t nkc_col) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    __shared__ __align__(16) uint32_t tile[COL ? kTile * kTile / 2 : 4];
    __shared__ __align__(16) uint8_t col_scales[COL ? kTile * 4 : 16];
    __shared__ int64_t s_rows[2];
    __shared__ int s_ok;

    const int tid = threadIdx.x;
    const int64_t rt = blockIdx.x;
    const int64_t ct = blockIdx.y;
    int64_t row_begin, row_end;

    if constexpr (GROUPED) {
        // Find the group owning padded row tile rt; validate the offsets.
        if (tid < 32) locate_group_tile(a.offsets, a.groups, a.rows, rt, s_rows, &s_ok);
        __syncthreads();
        if (!s_ok) {
            if (rt == 0 && ct == 0 && tid == 0) record_status(MXFP8_ERR_DEVICE_CHECK);
            return;
        }
        row_begin = s_rows[0];
        row_end = s_rows[1];
        if (row_begin < 0) return;  // past the last padded tile
    } else {
        row_begin = rt * kTile;
        row_end = min(a.rows, row_begin + kTile);
    }

    // ---- load the tile: 8 x 16 bytes per thread, all issued up front
    const int seg = tid & 15;
    const int64_t col = ct * kTile + seg * 8;
    uint4 v[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int r = it * 16 + (tid >> 4);
        const int64_t row = row_begin + r;
        if (row < row_end && col < a.cols && MX_IN_BOUNDS(row < a.rows && col + 8 <= a.cols)) {
            v[it] = __ldcs(reinterpret_cast<const uint4*>(a.x + row * a.ld + col));
        } else {
            v[it] = make_uint4(0u, 0u, 0u, 0u);
        }
    }

    // the scale layout's row tiles (grouped: every group padded to whole tiles)
    const int64_t n_row_tiles = GROUPED ? a.rows / kTile + a.groups : (a.rows + kTile - 1) / kTile;
    if (ROW && MX_IN_BOUNDS(rt < n_row_tiles && ct < nkc_row)) {
        uint8_t* s_tile = a.s_row + (rt * nkc_row + ct) * 512;
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int r = it * 16 + (tid >> 4);
            const int64_t row = row_begin + r;
            const bool in = row < row_end && col < a.cols && MX_IN_BOUNDS(row < a.rows && col + 8 <= a.cols);
            mx_row_step<FLOOR>(v[it], r, in ? a.q_row + row * a.cols + col : nullptr, s_tile);
        }
    }

    if constexpr (COL) {
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int r = it * 16 + (tid >> 4);
            reinterpret_cast<uint4*>(tile)[r * (kTile / 8) + seg] = v[it];
        }
        __syncthreads();
        const int cp = tid & 63;  // column pair: tile columns 2cp, 2cp+1
        const int j = tid >> 6;   // 32-row block of the tile
        uint32_t w[32];
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            w[i] = tile[(j * 32 + i) * (kTile / 2) + cp];
            m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
        }
        const uint32_t byte_lo = e8m0_byte(m & 0xFFFFu, FLOOR);
        const uint32_t byte_hi = e8m0_byte(m >> 16, FLOOR);
        col_scales[(2 * cp) * 4 + j] = static_cast<uint8_t>(byte_lo);
        col_scales[(2 * cp + 1) * 4 + j] = static_cast<uint8_t>(byte_hi);
        uint32_t qlo[8], qhi[8];
        const float flo = byte_lo == 0xFFu ? 0.f : inv_scale(byte_lo);
        const float fhi = byte_hi == 0xFFu ? 0.f : inv_scale(byte_hi);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            qlo[i] = byte_lo == 0xFFu
                         ? 0x7F7F7F7Fu
                         : quant4_half<false>(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3], flo);
            qhi[i] = byte_hi == 0xFFu
                         ? 0x7F7F7F7Fu
                         : quant4_half<true>(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3], fhi);
        }
        const int64_t k0 = ct * kTile + 2 * cp;  // output row (an input column)
        const int64_t r0 = rt * kTile + j * 32;  // output column (an input row)
        if (r0 < a.rows) {
            if (k0 < a.cols && MX_IN_BOUNDS(r0 + 32 <= a.rows)) {
                uint4* dst = reinterpret_cast<uint4*>(a.q_col + k0 * a.rows + r0);
                dst[0] = make_uint4(qlo[0], qlo[1], qlo[2], qlo[3]);
                dst[1] = make_uint4(qlo[4], qlo[5], qlo[6], qlo[7]);
            }
            if (k0 + 1 < a.cols && MX_IN_BOUNDS(r0 + 32 <= a.rows)) {
                uint4* dst = reinterpret_cast<uint4*>(a.q_col + (k0 + 1) * a.rows + r0);
                dst[0] = make_uint4(qhi[0], qhi[1], qhi[2], qhi[3]);
                dst[1] = make_uint4(qhi[4], qhi[5], qhi[6], qhi[7]);
            }
        }
        __syncthreads();
        if (tid < kTile && MX_IN_BOUNDS(ct < (a.cols + kTile - 1) / kTile && rt < nkc_col)) {
            uint8_t* s_tile = a.s_col + (ct * nkc_col + rt) * 512;
            *reinterpret_cast<uint32_t*>(s_tile + swz_word(tid)) =
                reinterpret_cast<const uint32_t*>(col_scales)[tid];
        }
    }
}

// Rowwise-only MX quantization, one thread per 32-value block: a CTA covers
// a 128 x 128 tile; thread t owns block (t & 3) of tile rows t/4 and t/4 + 64,
// reading each block as two 32-byte loads, computing its scale once and
// writing 32 payload bytes and one scale byte.
// One 128 x 128 tile of the rowwise quantization: thread t owns 32-value
// block t & 3 of tile rows t / 4 and t / 4 + 64 (rows from row_begin, below
// row_end; columns from ct * 128, below cols), reads it, and writes its 32
// payload bytes and its scale byte into the tile's 512-byte swizzled scale
// block s_tile.
template <bool FLOOR>
__device__ __forceinline__ void row_tile(const uint16_t* __restrict__ x, int64_t ld, int64_t rows,
                                         int64_t cols, uint8_t* __restrict__ q, uint8_t* __restrict__ s_tile,
                                         int64_t row_begin, int64_t row_end, int64_t ct, bool v8) {
    const int tid = threadIdx.x;
    const int j = tid & 3;
    const int64_t col = ct * kTile + j * 32;
    uint32_t w[2][16];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int64_t row = row_begin + (tid >> 2) + 64 * i;
        if (row < row_end && col < cols && MX_IN_BOUNDS(row < rows && col + 32 <= cols)) {
            const uint16_t* src = x + row * ld + col;
            ld32_stream(src, w[i], v8);
            ld32_stream(src + 16, w[i] + 8, v8);
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) w[i][k] = 0u;
        }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int r = (tid >> 2) + 64 * i;
        const int64_t row = row_begin + r;
        const bool in = row < row_end && col < cols && MX_IN_BOUNDS(row < rows && col + 32 <= cols);
        mx_block32<FLOOR>(w[i], in ? q + row * cols + col : nullptr, s_tile + swz_word(r) + j, v8);
    }
}

template <bool FLOOR, bool GROUPED>
__global__ void __launch_bounds__(kThreads)
    quantize_mx_row_kernel(QuantMxArgs a, int64_t nkc, bool v8) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    __shared__ int64_t s_rows[2];
    __shared__ int s_ok;
    const int tid = threadIdx.x;
    const int64_t rt = blockIdx.x;
    const int64_t ct = blockIdx.y;
    int64_t row_begin, row_end;
    if constexpr (GROUPED) {
        if (tid < 32) locate_group_tile(a.offsets, a.groups, a.rows, rt, s_rows, &s_ok);
        __syncthreads();
        if (!s_ok) {
            if (rt == 0 && ct == 0 && tid == 0) record_status(MXFP8_ERR_DEVICE_CHECK);
            return;
        }
        row_begin = s_rows[0];
        row_end = s_rows[1];
        if (row_begin < 0) return;
    } else {
        row_begin = rt * kTile;
        row_end = min(a.rows, row_begin + kTile);
    }
    const int64_t n_row_tiles = GROUPED ? a.rows / kTile + a.groups : (a.rows + kTile - 1) / kTile;
    if (!MX_IN_BOUNDS(rt < n_row_tiles && ct < nkc)) return;
    row_tile<FLOOR>(a.x, a.ld, a.rows, a.cols, a.q_row, a.s_row + (rt * nkc + ct) * 512, row_begin,
                    row_end, ct, v8);
}

// Rowwise MX quantization of several tensors in one launch: a 1D grid over
// all tensors' 128 x 128 tiles (tensor t owns blocks [tile_end[t-1],
// tile_end[t]), row tiles fastest), each tile done as above.
struct MxRowBatch {
    const uint16_t* x[kMaxBatch];
    uint8_t* q[kMaxBatch];
    uint8_t* s[kMaxBatch];
    int64_t rows[kMaxBatch], cols[kMaxBatch], ld[kMaxBatch];
    int64_t row_tiles[kMaxBatch], nkc[kMaxBatch], tile_end[kMaxBatch];
    uint8_t v8[kMaxBatch];
    int count;
};

template <bool FLOOR>
__global__ void __launch_bounds__(kThreads)
    quantize_mx_row_batch_kernel(const __grid_constant__ MxRowBatch b) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    const int64_t blk = blockIdx.x;
    int t = 0;
    while (t + 1 < b.count && blk >= b.tile_end[t]) ++t;
    const int64_t local = blk - (t ? b.tile_end[t - 1] : 0);
    const int64_t rt = local % b.row_tiles[t];
    const int64_t ct = local / b.row_tiles[t];
    const int64_t row_begin = rt * kTile;
    const int64_t row_end = min(b.rows[t], row_begin + kTile);
    if (!MX_IN_BOUNDS(rt < (b.rows[t] + kTile - 1) / kTile && ct < (b.cols[t] + kTile - 1) / kTile)) return;
    row_tile<FLOOR>(b.x[t], b.ld[t], b.rows[t], b.cols[t], b.q[t], b.s[t] + (rt * b.nkc[t] + ct) * 512,
                    row_begin, row_end, ct, b.v8[t] != 0);
}

// Rowwise + colwise (or colwise only) MX quantization of a 128 x 128 tile
// staged by TMA: two 64-column boxes with 128-byte swizzle (16-byte chunk k
// of a 128-byte half-row r sits at chunk k ^ (r % 8)), so both access
// patterns below are free of bank conflicts.
//   colwise: thread t owns columns 4g..4g+3 (g = t % 32) of the 32-row block
//            j = t / 32, read as 32 64-bit loads (two BF16 pairs per row);
//            each column's 32 E4M3 bytes are one output row segment of q_col.
//   rowwise: thread t owns tile row t, its four 32-value blocks read as
//            16-byte chunks.
// The E8M0 rule and packing are the row kernel's; 128 threads per CTA.
constexpr int kTileThreads = 128;
constexpr uint32_t kTileSmem = kTile * kTile * 2;

// What one tile kernel needs to know about its tensor.
struct TileArgs {
    int64_t rows, cols;
    uint8_t* q_row;
    uint8_t* s_row;
    uint8_t* q_col;
    uint8_t* s_col;
    int64_t nkc_row;  // 128-wide K tiles of the rowwise operand (column tiles)
    int64_t nkc_col;  // ... of the colwise one (row tiles)
    bool row;         // rowwise outputs too
    bool v8;          // 32-byte aligned outputs: 256-bit stores
};

// One 128 x 128 tile (row tile rt, column tile ct) of tensor `map` / `a`,
// staged in the CTA's 32 KB shared tile `st` through mbarrier `bb` whose
// next phase has parity `parity`.  Returns false when the copy did not land
// in time (the status is recorded).
template <bool FLOOR>
__device__ __forceinline__ bool tile_quantize(const CUtensorMap* map, const TileArgs& a, int64_t rt,
                                              int64_t ct, uint32_t st, uint32_t bb, uint32_t parity,
                                              uint64_t limit_ns) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_arrive_expect_tx(bb, kTileSmem);
        tma_load_2d(st, map, bb, static_cast<int32_t>(ct * kTile), static_cast<int32_t>(rt * kTile));
        tma_load_2d(st + kTileSmem / 2, map, bb, static_cast<int32_t>(ct * kTile + 64),
                    static_cast<int32_t>(rt * kTile));
    }
    const int never = 0;
    if (!mbar_wait(bb, parity, limit_ns, &never)) {
        if (tid == 0) record_status(MXFP8_ERR_TIMEOUT);
        mbar_wait(bb, parity, limit_ns, &never);  // the copy may still land: give it time
        return false;
    }
    // 16-byte chunk k (0..15) of tile row r
    auto chunk_addr = [&](int r, int k) {
        return st + (k >> 3) * (kTileSmem / 2) + r * 128 + (((k & 7) ^ (r & 7)) << 4);
    };

    if (a.row) {
        const int r = tid;
        const int64_t row = rt * kTile + r;
        uint8_t* s_tile = a.s_row + (rt * a.nkc_row + ct) * 512;
        uint32_t bytes = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w[4 * k]), "=r"(w[4 * k + 1]), "=r"(w[4 * k + 2]), "=r"(w[4 * k + 3])
                             : "r"(chunk_addr(r, 4 * b + k)));
            }
            const int64_t col = ct * kTile + 32 * b;
            uint8_t byte;
            const bool in = row < a.rows && col < a.cols && MX_IN_BOUNDS(col + 32 <= a.cols);
            mx_block32<FLOOR>(w, in ? a.q_row + row * a.cols + col : nullptr, &byte, a.v8);
            bytes |= static_cast<uint32_t>(byte) << (8 * b);
        }
        if (MX_IN_BOUNDS(rt < (a.rows + kTile - 1) / kTile && ct < a.nkc_row))
            *reinterpret_cast<uint32_t*>(s_tile + swz_word(r)) = bytes;
    }

    // colwise
    {
        const int g = tid & 31, j = tid >> 5;
        uint32_t lo[32], hi[32];  // columns 4g, 4g+1 (lo) and 4g+2, 4g+3 (hi) of rows 32j + i
        const int k = g >> 1;     // 16-byte chunk holding this column group
        const uint32_t sub = (g & 1) * 8;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int r = 32 * j + i;
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                         : "=r"(lo[i]), "=r"(hi[i])
                         : "r"(chunk_addr(r, k) + sub));
        }
        uint32_t mlo = 0, mhi = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            mlo = max_u16x2(mlo, lo[i] & 0x7FFF7FFFu);
            mhi = max_u16x2(mhi, hi[i] & 0x7FFF7FFFu);
        }
        const uint32_t bc[4] = {e8m0_byte(mlo & 0xFFFFu, FLOOR), e8m0_byte(mlo >> 16, FLOOR),
                                e8m0_byte(mhi & 0xFFFFu, FLOOR), e8m0_byte(mhi >> 16, FLOOR)};
        const int64_t r0 = rt * kTile + 32 * j;  // output column (an input row)
        uint8_t* s_tile = a.s_col + (ct * a.nkc_col + rt) * 512;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t* src = c < 2 ? lo : hi;
            const bool high = c & 1;
            uint32_t q[8];
            if (bc[c] == 0xFFu) {
#pragma unroll
                for (int t = 0; t < 8; ++t) q[t] = 0x7F7F7F7Fu;
            } else {
                const float f = inv_scale(bc[c]);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    q[t] = high ? quant4_half<true>(src[4 * t], src[4 * t + 1], src[4 * t + 2], src[4 * t + 3], f)
                                : quant4_half<false>(src[4 * t], src[4 * t + 1], src[4 * t + 2], src[4 * t + 3], f);
                }
            }
            const int64_t k0 = ct * kTile + 4 * g + c;  // output row (an input column)
            if (k0 < a.cols && r0 < a.rows && MX_IN_BOUNDS(r0 + 32 <= a.rows)) st32(a.q_col + k0 * a.rows + r0, q, a.v8);
            if (MX_IN_BOUNDS(ct < (a.cols + kTile - 1) / kTile && rt < a.nkc_col))
                s_tile[swz_word(4 * g + c) + j] = static_cast<uint8_t>(bc[c]);
        }
    }
    return true;
}

// Rowwise + colwise (or colwise only) MX quantization of a 128 x 128 tile
// staged by TMA: two 64-column boxes with 128-byte swizzle (16-byte chunk k
// of a 128-byte half-row r sits at chunk k ^ (r % 8)), so both access
// patterns are free of bank conflicts.
//   colwise: thread t owns columns 4g..4g+3 (g = t % 32) of the 32-row block
//            j = t / 32, read as 32 64-bit loads (two BF16 pairs per row);
//            each column's 32 E4M3 bytes are one output row segment of q_col.
//   rowwise: thread t owns tile row t, its four 32-value blocks read as
//            16-byte chunks.
// The E8M0 rule and packing are the row kernel's; 128 threads per CTA, one
// tile per CTA (grid: row tiles x column tiles).
template <bool FLOOR>
__global__ void __launch_bounds__(kTileThreads)
    quantize_mx_tile_kernel(const __grid_constant__ CUtensorMap tm_x, TileArgs a, uint64_t limit_ns) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    extern __shared__ uint8_t tile_raw[];
    __shared__ __align__(8) uint64_t bar;
    uint8_t* tile = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(tile_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t bb = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(bb, 1);
        fence_mbar_init();
    }
    __syncthreads();
    tile_quantize<FLOOR>(&tm_x, a, blockIdx.x, blockIdx.y, smem_u32(tile), bb, 0, limit_ns);
}

// The same over several tensors in one launch: a 1D grid over all their
// tiles (tensor t owns blocks [tile_end[t-1], tile_end[t]), row tiles
// fastest), each CTA one tile.
constexpr int kMaxTileBatch = 8;
struct MxTileBatch {
    CUtensorMap map[kMaxTileBatch];
    TileArgs arg[kMaxTileBatch];
    int64_t row_tiles[kMaxTileBatch];
    int64_t tile_end[kMaxTileBatch];
    int count;
};

template <bool FLOOR>
__global__ void __launch_bounds__(kTileThreads)
    quantize_mx_tile_batch_kernel(const __grid_constant__ MxTileBatch b, uint64_t limit_ns) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    extern __shared__ uint8_t tile_raw[];
    __shared__ __align__(8) uint64_t bar;
    uint8_t* tile = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(tile_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t bb = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(bb, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int64_t blk = blockIdx.x;
    int t = 0;
    while (t + 1 < b.count && blk >= b.tile_end[t]) ++t;
    const int64_t local = blk - (t ? b.tile_end[t - 1] : 0);
    tile_quantize<FLOOR>(&b.map[t], b.arg[t], local % b.row_tiles[t], local / b.row_tiles[t],
                         smem_u32(tile), bb, 0, limit_ns);
}

// ---------------------------------------------------------- per-tensor --

__device__ __forceinline__ uint32_t warp_max(uint32_t m) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, d));
    return m;
}

// amax of |x| as BF16 magnitude bits, merged into *amax_bits (pre-zeroed) as
// the fp32 bit pattern (positive fp32 patterns order like their values).
__global__ void __launch_bounds__(256)
    tensor_amax_kernel(const uint16_t* __restrict__ x, int64_t n, unsigned* amax_bits) {
    __shared__ uint32_t red[8];
    const int64_t n8 = n / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    uint32_t m = 0;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n8 && MX_IN_BOUNDS((i + 3 * stride + 1) * 8 <= n); i += 4 * stride) {
        const uint4 a0 = x8[i], a1 = x8[i + stride], a2 = x8[i + 2 * stride],
                    a3 = x8[i + 3 * stride];
        m = max(m, max(max(amax8(a0), amax8(a1)), max(amax8(a2), amax8(a3))));
    }
    for (; i < n8 && MX_IN_BOUNDS((i + 1) * 8 <= n); i += stride) m = max(m, amax8(x8[i]));
    for (int64_t t = n8 * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
         t += stride)
        m = max(m, static_cast<uint32_t>(x[t] & 0x7FFFu));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0u;
        m = warp_max(m);
        if (threadIdx.x == 0 && m) atomicMax(amax_bits, m << 16);
    }
}

template <int FMT>
__global__ void __launch_bounds__(256)
    tensor_cast_kernel(const uint16_t* __restrict__ x, int64_t n, const unsigned* amax_bits,
                       float* scale_out, uint8_t* __restrict__ q) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    const float amax = __uint_as_float(*amax_bits);
    const float fmax = FMT == FP8_E4M3 ? 448.0f : 57344.0f;
    const float s = __fdiv_rn(fmax, amax > 1e-12f ? amax : 1e-12f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s;
    const int64_t n8 = n / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += stride) {
        if (!MX_IN_BOUNDS((i + 1) * 8 <= n)) break;
        const uint4 v = x8[i];
        uint2 o;
        o.x = quant4_scaled<FMT>(v.x, v.y, s);
        o.y = quant4_scaled<FMT>(v.z, v.w, s);
        reinterpret_cast<uint2*>(q)[i] = o;
    }
    for (int64_t t = n8 * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
         t += stride) {
        const float y = __fmul_rn(__uint_as_float(static_cast<uint32_t>(x[t]) << 16), s);
        q[t] = static_cast<uint8_t>(cvt_fp8x2<FMT>(y, 0.0f) & 0xFFu);
    }
}

// Single-launch per-tensor quantization of a batch of tensors (one grid
// barrier for all of them, e.g. a linear layer's activation and weight):
// every CTA reduces its share of |x_t| into ws[t] (atomicMax on the fp32 bit
// pattern), the CTAs meet at a grid barrier (ws[kMaxBatch] counts arrivals;
// the launch is cooperative so all CTAs are resident; the wait is bounded),
// then each CTA computes every tensor's scale and casts its share, re-reading
// x_t (from L2 when it fits there).  ws[0 .. kMaxBatch] must be zero at launch.
constexpr int kFusedThreads = 512;

struct TensorBatch {
    const uint16_t* x[kMaxBatch];
    uint8_t* q[kMaxBatch];
    float* amax[kMaxBatch];   // device scalars (outputs)
    float* scale[kMaxBatch];
    int64_t n[kMaxBatch];
    uint8_t v8[kMaxBatch];    // x 32-byte aligned: 256-bit loads
    int count;
};

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// |x| maximum of one tensor over this thread's grid-stride share, as BF16
// magnitude bits.
// This thread's share of max |x| (as BF16 magnitude bits) over 32-byte
// chunks first, first + stride, ...: four chunks in flight per round, kept
// in L2 (normal caching) for the cast that re-reads them.
__device__ __forceinline__ uint32_t amax_share(const uint16_t* __restrict__ x, int64_t n,
                                               int64_t first, int64_t stride, bool v8) {
    const int64_t n16 = n / 16;
    uint32_t m = 0;
    for (int64_t i = first; i < n16; i += 4 * stride) {
        uint32_t w[4][8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t c = i + k * stride;
            if (c < n16) {
                ld32_cached(x + c * 16, w[k], v8);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) w[k][e] = 0u;
            }
        }
        // the next round's chunks into L2 meanwhile (no registers held)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t c = i + (4 + k) * stride;
            if (c < n16) asm volatile("prefetch.global.L2 [%0];" ::"l"(x + c * 16));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m = max(m, max(amax8(make_uint4(w[k][0], w[k][1], w[k][2], w[k][3])),
                           amax8(make_uint4(w[k][4], w[k][5], w[k][6], w[k][7]))));
    }
    for (int64_t t = n16 * 16 + first; t < n; t += stride) m = max(m, static_cast<uint32_t>(x[t] & 0x7FFFu));
    return m;
}

// Cast this thread's share (the same chunks as amax_share) with scale s:
// four 32-byte chunks in flight, 16 payload bytes stored per chunk.
template <int FMT>
__device__ __forceinline__ void cast_share(const uint16_t* __restrict__ x, uint8_t* __restrict__ q,
                                           int64_t n, float s, int64_t first, int64_t stride,
                                           bool v8) {
    const int64_t n16 = n / 16;
    for (int64_t i = first; i < n16; i += 4 * stride) {
        uint32_t w[4][8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t c = i + k * stride;
            if (c < n16) ld32_stream(x + c * 16, w[k], v8);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int64_t c = i + k * stride;
            if (c < n16 && MX_IN_BOUNDS((c + 1) * 16 <= n)) {
                uint4 o;
                uint32_t* po = &o.x;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    po[e] = quant4_scaled<FMT>(w[k][2 * e], w[k][2 * e + 1], s);
                reinterpret_cast<uint4*>(q)[c] = o;
            }
        }
    }
    for (int64_t r = n16 * 16 + first; r < n; r += stride) {
        const float y = __fmul_rn(__uint_as_float(static_cast<uint32_t>(x[r]) << 16), s);
        q[r] = static_cast<uint8_t>(cvt_fp8x2<FMT>(y, 0.0f) & 0xFFu);
    }
}

template <int FMT>
__global__ void __launch_bounds__(kFusedThreads)
    tensor_quant_batch_kernel(const TensorBatch b, uint32_t* ws, uint64_t limit_ns) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    __shared__ uint32_t red[kMaxBatch][kFusedThreads / 32];
    __shared__ int s_ok;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t first = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int t = 0; t < b.count; ++t) {
        const uint32_t m = warp_max(amax_share(b.x[t], b.n[t], first, stride, b.v8[t] != 0));
        if (lane == 0) red[t][warp] = m;
    }
    __syncthreads();
    if (warp == 0) {
        for (int t = 0; t < b.count; ++t) {
            uint32_t m = lane < kFusedThreads / 32 ? red[t][lane] : 0u;
            m = warp_max(m);
            if (lane == 0 && m) atomicMax(ws + t, m << 16);
        }
        if (lane == 0) {
            __threadfence();
            atomicAdd(ws + kMaxBatch, 1u);
            bool ok = ld_acquire_gpu(ws + kMaxBatch) >= gridDim.x;
            if (!ok) {
                const uint64_t t0 = globaltimer_ns();
                for (uint32_t it = 1;; ++it) {
                    if (ld_acquire_gpu(ws + kMaxBatch) >= gridDim.x) {
                        ok = true;
                        break;
                    }
                    if ((it & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) break;
                }
            }
            s_ok = ok ? 1 : 0;
        }
    }
    __syncthreads();
    if (!s_ok) {
        if (threadIdx.x == 0) record_status(MXFP8_ERR_TIMEOUT);
        return;
    }
    const float fmax = FMT == FP8_E4M3 ? 448.0f : 57344.0f;
    for (int t = 0; t < b.count; ++t) {
        const float amax = __uint_as_float(ld_acquire_gpu(ws + t));
        const float s = __fdiv_rn(fmax, amax > 1e-12f ? amax : 1e-12f);
        if (blockIdx.x == 0 && threadIdx.x == 0) {
            *b.amax[t] = amax;
            *b.scale[t] = s;
        }
        cast_share<FMT>(b.x[t], b.q[t], b.n[t], s, first, stride, b.v8[t] != 0);
    }
}

// ------------------------------------- delayed and automatic scaling --

// True when the saturating RNE cast of y gives the largest finite code:
// E4M3 448 for |y| >= 432 (the tie with 416 goes to 448, the even code),
// E5M2 57344 for |y| > 53248 (that tie goes to 49152).  False for NaN.
template <int FMT>
__device__ __forceinline__ uint32_t saturates(float y) {
    const float a = fabsf(y);
    return (FMT == FP8_E4M3 ? (a >= 432.f) : (a > 53248.f)) ? 1u : 0u;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
    return __reduce_add_sync(0xffffffffu, v);
}

// Block reduction of (amax bits, saturated count) into the global
// accumulators: the amax as fp32 bits of a BF16 magnitude (positive fp32
// patterns order like their values, NaN above Inf), the count 64-bit.
__device__ __forceinline__ void reduce_amax_sat(uint32_t m, uint32_t cnt, unsigned* amax_bits,
                                                unsigned long long* sat) {
    __shared__ uint32_t red_m[8], red_c[8];
    m = warp_max(m);
    cnt = warp_sum(cnt);
    if ((threadIdx.x & 31) == 0) {
        red_m[threadIdx.x >> 5] = m;
        red_c[threadIdx.x >> 5] = cnt;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < blockDim.x / 32 ? red_m[threadIdx.x] : 0u;
        cnt = threadIdx.x < blockDim.x / 32 ? red_c[threadIdx.x] : 0u;
        m = warp_max(m);
        cnt = warp_sum(cnt);
        if (threadIdx.x == 0) {
            if (m) atomicMax(amax_bits, m << 16);
            if (cnt) atomicAdd(sat, static_cast<unsigned long long>(cnt));
        }
    }
}

// Cast with a scale read from device memory ("3.8 Mixed Precision", the
// delayed-scaling sketch; FP8-LM Section 2.1 Eq. 3 with s = mu): q =
// FP8(fp32(x s)); accumulates amax(x) and the saturated count (both zeroed
// on the stream before the launch).
template <int FMT>
__global__ void __launch_bounds__(256)
    tensor_cast_scaled_kernel(const uint16_t* __restrict__ x, int64_t n, const float* scale,
                              uint8_t* __restrict__ q, unsigned* amax_bits,
                              unsigned long long* sat) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    const float s = *scale;
    const int64_t n8 = n / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    uint32_t m = 0, cnt = 0;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += stride) {
        if (!MX_IN_BOUNDS((i + 1) * 8 <= n)) break;
        const uint4 v = x8[i];
        m = max(m, amax8(v));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float y[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            y[2 * k] = __fmul_rn(bf16_lo(w[k]), s);
            y[2 * k + 1] = __fmul_rn(bf16_hi(w[k]), s);
            cnt += saturates<FMT>(y[2 * k]) + saturates<FMT>(y[2 * k + 1]);
        }
        reinterpret_cast<uint2*>(q)[i] = make_uint2(cvt_fp8x4<FMT>(y[0], y[1], y[2], y[3]),
                                                    cvt_fp8x4<FMT>(y[4], y[5], y[6], y[7]));
    }
    for (int64_t t = n8 * 8 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
         t += stride) {
        m = max(m, static_cast<uint32_t>(x[t] & 0x7FFFu));
        const float y = __fmul_rn(__uint_as_float(static_cast<uint32_t>(x[t]) << 16), s);
        cnt += saturates<FMT>(y);
        q[t] = static_cast<uint8_t>(cvt_fp8x2<FMT>(y, 0.0f) & 0xFFu);
    }
    reduce_amax_sat(m, cnt, amax_bits, sat);
}

// The delayed scale from the amax history ("3.8 Mixed Precision", the
// delayed-scaling sketch): a = max(history) (NaN propagates), clamped below
// at 1e-12, s = fp32(fp32(fmax / a) * margin).  One thread; also zeroes
// the accumulators of the cast that follows.
__global__ void delayed_scale_kernel(const float* hist, int h, int fmt, float margin,
                                     float* scale_out, unsigned* amax_bits,
                                     unsigned long long* sat) {
    float a = hist[0];
    for (int i = 1; i < h && !isnan(a); ++i) {
        const float v = hist[i];
        if (isnan(v) || v > a) a = v;
    }
    if (!(a >= 1e-12f) && !isnan(a)) a = 1e-12f;
    const float fmax = fmt == FP8_E5M2 ? 57344.0f : 448.0f;
    *scale_out = __fmul_rn(__fdiv_rn(fmax, a), margin);
    *amax_bits = 0u;
    *sat = 0ull;
}

// history[pos] = this step's amax; pos = (pos + 1) % h.  One thread.
__global__ void delayed_record_kernel(float* hist, int h, int* pos, const unsigned* amax_bits) {
    int p = *pos;
    if (p < 0 || p >= h) {  // a corrupted pointer: record and restart the ring
        record_status(MXFP8_ERR_DEVICE_CHECK);
        p = 0;
    }
    hist[p] = __uint_as_float(*amax_bits);
    *pos = (p + 1) % h;
}

// Two FP8 codes (low byte first) to fp32, exactly (both formats fit f16).
template <int FMT>
__device__ __forceinline__ float2 fp8x2_to_f32(uint32_t codes) {
    uint32_t h2;
    if constexpr (FMT == FP8_E4M3) {
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(codes)));
    } else {
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(codes)));
    }
    float lo, hi;
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"(static_cast<uint16_t>(h2 & 0xFFFFu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"(static_cast<uint16_t>(h2 >> 16)));
    return make_float2(lo, hi);
}

// Requantization to a shared scale (FP8-LM Section 2.1, Eq. 4-5): q'' =
// FP8(fp32(s_out * fp32(decode(q) / s_in))), in the equation's order;
// accumulates the saturated count (zeroed before the launch).  An FP8 input
// has 256 codes, so every CTA first evaluates that expression once per code
// into a shared-memory table (the division correctly rounded, as stated) and
// then maps bytes through the table: the same result for every byte at a
// fraction of the arithmetic.
template <int FIN, int FOUT>
__global__ void __launch_bounds__(256)
    requantize_kernel(const uint8_t* __restrict__ q_in, int64_t n, const float* s_in_p,
                      const float* s_out_p, uint8_t* __restrict__ q_out, unsigned long long* sat) {
    griddep_launch_dependents();  // a dependent GEMM may launch now
    griddep_wait();               // the previous kernel's results are visible
    // one output code per input code, in four copies shifted to the four byte
    // positions of a word, so that a word is three ORs of looked-up values
    __shared__ uint32_t lut[4][256];
    {
        const float s_in = *s_in_p, s_out = *s_out_p;
        const uint32_t c = threadIdx.x;  // blockDim.x == 256
        const float v = fp8x2_to_f32<FIN>(c).x;
        const float y = __fmul_rn(s_out, __fdiv_rn(v, s_in));
        const uint32_t code = cvt_fp8x2<FOUT>(y, 0.0f) & 0xFFu;
#pragma unroll
        for (int b = 0; b < 4; ++b) lut[b][c] = code << (8 * b);
    }
    __syncthreads();
    constexpr uint32_t kMaxCode = FOUT == FP8_E4M3 ? 0x7Eu : 0x7Bu;
    const int64_t n16 = n / 16;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const uint4* in16 = reinterpret_cast<const uint4*>(q_in);
    uint32_t cnt = 0;
    auto map4 = [&](uint32_t w) {
        const uint32_t o = lut[0][w & 0xFFu] | lut[1][(w >> 8) & 0xFFu] | lut[2][(w >> 16) & 0xFFu] |
                           lut[3][w >> 24];
        // bytes equal to the largest finite code (either sign): zero bytes of x
        const uint32_t x = (o & 0x7F7F7F7Fu) ^ (kMaxCode * 0x01010101u);
        const uint32_t z = ~(((x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | x | 0x7F7F7F7Fu);
        cnt += __popc(z);
        return o;
    };
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += stride) {
        if (!MX_IN_BOUNDS((i + 1) * 16 <= n)) break;
        const uint4 v = __ldcs(in16 + i);
        uint4 o;
        o.x = map4(v.x);
        o.y = map4(v.y);
        o.z = map4(v.z);
        o.w = map4(v.w);
        reinterpret_cast<uint4*>(q_out)[i] = o;
    }
    for (int64_t t = n16 * 16 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n;
         t += stride) {
        const uint32_t o = lut[0][q_in[t]];
        cnt += (o & 0x7Fu) == kMaxCode;
        q_out[t] = static_cast<uint8_t>(o);
    }
    __shared__ uint32_t red_c[8];
    cnt = warp_sum(cnt);
    if ((threadIdx.x & 31) == 0) red_c[threadIdx.x >> 5] = cnt;
    __syncthreads();
    if (threadIdx.x < 32) {
        cnt = threadIdx.x < blockDim.x / 32 ? red_c[threadIdx.x] : 0u;
        cnt = warp_sum(cnt);
        if (threadIdx.x == 0 && cnt) atomicAdd(sat, static_cast<unsigned long long>(cnt));
    }
}

int elementwise_blocks(int64_t n, int per_thread) {
    const int64_t chunks = n / per_thread + 1;
    const int64_t max_blocks = static_cast<int64_t>(sm_count_current_device()) * 8;
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((chunks + 255) / 256, max_blocks)));
}

template <bool ROW, bool COL, bool FLOOR, bool GROUPED>
cudaError_t launch_mx(const QuantMxArgs& a, int64_t row_tiles, cudaStream_t s) {
    const int64_t col_tiles = (a.cols + kTile - 1) / kTile;
    const int64_t nkc_row = col_tiles;                   // K tiles of the rowwise operand
    const int64_t nkc_col = (a.rows + kTile - 1) / kTile;  // K tiles of the transposed one
    if (row_tiles <= 0 || col_tiles <= 0) return cudaSuccess;
    if (col_tiles > 65535 || row_tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(row_tiles), static_cast<unsigned>(col_tiles));
    if constexpr (ROW && !COL) {
        // 256-bit accesses when every block start is 32-byte aligned
        const bool v8 = (reinterpret_cast<uintptr_t>(a.x) % 32 == 0) && (a.ld % 16 == 0) &&
                        (reinterpret_cast<uintptr_t>(a.q_row) % 32 == 0);
        return launch_pdl(quantize_mx_row_kernel<FLOOR, GROUPED>, grid, dim3(kThreads), 0, s, a,
                          nkc_row, v8);
    }
    return launch_pdl(quantize_mx_kernel<ROW, COL, FLOOR, GROUPED>, grid, dim3(kThreads), 0, s, a,
                      nkc_row, nkc_col);
}

}  // namespace

cudaError_t launch_quantize_mx_rows_batch(int count, const QuantMxArgs* a, cudaStream_t s) {
    if (count < 1 || count > kMaxBatch) return cudaErrorInvalidValue;
    MxRowBatch b{};
    int64_t tiles = 0;
    bool floor = false;
    int n = 0;
    for (int t = 0; t < count; ++t) {
        if (a[t].rows <= 0 || a[t].cols <= 0) continue;  // nothing to do for an empty tensor
        const int64_t row_tiles = (a[t].rows + kTile - 1) / kTile;
        const int64_t col_tiles = (a[t].cols + kTile - 1) / kTile;
        b.x[n] = a[t].x;
        b.q[n] = a[t].q_row;
        b.s[n] = a[t].s_row;
        b.rows[n] = a[t].rows;
        b.cols[n] = a[t].cols;
        b.ld[n] = a[t].ld;
        b.row_tiles[n] = row_tiles;
        b.nkc[n] = col_tiles;
        tiles += row_tiles * col_tiles;
        b.tile_end[n] = tiles;
        b.v8[n] = (reinterpret_cast<uintptr_t>(a[t].x) % 32 == 0) && (a[t].ld % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(a[t].q_row) % 32 == 0);
        floor = (a[t].flags & MX_SCALE_FLOOR) != 0;
        ++n;
    }
    if (n == 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
    b.count = n;
    const dim3 grid(static_cast<unsigned>(tiles));
    return floor ? launch_pdl(quantize_mx_row_batch_kernel<true>, grid, dim3(kThreads), 0, s, b)
                 : launch_pdl(quantize_mx_row_batch_kernel<false>, grid, dim3(kThreads), 0, s, b);
}

// The tile kernels' view of a tensor; false when its TMA map cannot be made.
bool tile_args(const QuantMxArgs& a, CUtensorMap* map, TileArgs* t) {
    const int64_t row_tiles = (a.rows + kTile - 1) / kTile;
    const int64_t col_tiles = (a.cols + kTile - 1) / kTile;
    if (col_tiles > 65535 || row_tiles > 0x7FFFFFFF) return false;
    // the tensor map wants a 16-byte aligned base and row stride (checked by the API)
    if (!encode_tensor_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, a.rows, a.cols, a.ld * 2,
                              64, kTile, CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    const bool row = (a.flags & MX_ROWWISE) != 0;
    t->rows = a.rows;
    t->cols = a.cols;
    t->q_row = a.q_row;
    t->s_row = a.s_row;
    t->q_col = a.q_col;
    t->s_col = a.s_col;
    t->nkc_row = col_tiles;
    t->nkc_col = row_tiles;
    t->row = row;
    t->v8 = (reinterpret_cast<uintptr_t>(a.q_col) % 32 == 0) &&
            (!row || reinterpret_cast<uintptr_t>(a.q_row) % 32 == 0);
    return true;
}

cudaError_t launch_mx_tile(const QuantMxArgs& a, const CUtensorMap& map, const TileArgs& t,
                           cudaStream_t s) {
    dim3 grid(static_cast<unsigned>(t.nkc_col), static_cast<unsigned>(t.nkc_row));
    const uint64_t limit = wait_limit_ns();
    return (a.flags & MX_SCALE_FLOOR)
               ? launch_pdl(quantize_mx_tile_kernel<true>, grid, dim3(kTileThreads), kTileSmem + 1024, s,
                            map, t, limit)
               : launch_pdl(quantize_mx_tile_kernel<false>, grid, dim3(kTileThreads), kTileSmem + 1024, s,
                            map, t, limit);
}

cudaError_t launch_quantize_mx(const QuantMxArgs& a, cudaStream_t s) {
    const bool row = a.flags & MX_ROWWISE, col = a.flags & MX_COLWISE;
    const bool fl = a.flags & MX_SCALE_FLOOR;
    const int64_t row_tiles = (a.rows + kTile - 1) / kTile;
    if (col && a.rows > 0 && a.cols > 0) {
        // colwise (with or without rowwise): TMA-staged tile kernel
        CUtensorMap map;
        TileArgs t;
        if (tile_args(a, &map, &t)) return launch_mx_tile(a, map, t, s);
    }
    if (row && col) {
        return fl ? launch_mx<true, true, true, false>(a, row_tiles, s)
                  : launch_mx<true, true, false, false>(a, row_tiles, s);
    }
    if (row) {
        return fl ? launch_mx<true, false, true, false>(a, row_tiles, s)
                  : launch_mx<true, false, false, false>(a, row_tiles, s);
    }
    return fl ? launch_mx<false, true, true, false>(a, row_tiles, s)
              : launch_mx<false, true, false, false>(a, row_tiles, s);
}

cudaError_t launch_quantize_mx_cols_batch(int count, const QuantMxArgs* a, cudaStream_t s) {
    MxTileBatch b{};
    int n = 0;
    int64_t tiles = 0;
    bool floor = false;
    cudaError_t e = cudaSuccess;
    auto flush = [&]() -> cudaError_t {
        if (n == 0) return cudaSuccess;
        b.count = n;
        const dim3 grid(static_cast<unsigned>(tiles));
        const uint64_t limit = wait_limit_ns();
        const cudaError_t r =
            floor ? launch_pdl(quantize_mx_tile_batch_kernel<true>, grid, dim3(kTileThreads),
                               kTileSmem + 1024, s, b, limit)
                  : launch_pdl(quantize_mx_tile_batch_kernel<false>, grid, dim3(kTileThreads),
                               kTileSmem + 1024, s, b, limit);
        n = 0;
        tiles = 0;
        return r;
    };
    for (int t = 0; t < count && e == cudaSuccess; ++t) {
        if (a[t].rows <= 0 || a[t].cols <= 0) continue;
        floor = (a[t].flags & MX_SCALE_FLOOR) != 0;
        if (!tile_args(a[t], &b.map[n], &b.arg[n])) {
            e = launch_quantize_mx(a[t], s);  // no TMA map for this tensor: the register-staged kernel
            continue;
        }
        const int64_t t_tiles = b.arg[n].nkc_col * b.arg[n].nkc_row;
        if (tiles + t_tiles > 0x7FFFFFFF) {
            if ((e = flush()) != cudaSuccess) break;
            if (!tile_args(a[t], &b.map[0], &b.arg[0])) return cudaErrorInvalidValue;
        }
        b.row_tiles[n] = b.arg[n].nkc_col;
        tiles += t_tiles;
        b.tile_end[n] = tiles;
        if (++n == kMaxTileBatch) e = flush();
    }
    if (e == cudaSuccess) e = flush();
    return e;
}

cudaError_t launch_quantize_mx_grouped(const QuantMxArgs& a, cudaStream_t s) {
    // sum_g ceil(m_g / 128) <= floor(total / 128) + groups
    const int64_t row_tiles = a.rows / kTile + a.groups;
    return (a.flags & MX_SCALE_FLOOR) ? launch_mx<true, false, true, true>(a, row_tiles, s)
                                      : launch_mx<true, false, false, true>(a, row_tiles, s);
}

cudaError_t launch_quantize_tensor(const uint16_t* x, int64_t n, int fmt, float* amax,
                                   float* scale, uint8_t* q, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
    const int64_t chunks = n / 8 + 1;
    const int64_t max_blocks = static_cast<int64_t>(sm_count_current_device()) * 8;
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((chunks + 255) / 256, max_blocks)));
    unsigned* bits = reinterpret_cast<unsigned*>(amax);
    if (n > 0) tensor_amax_kernel<<<blocks, 256, 0, s>>>(x, n, bits);
    if (fmt == FP8_E5M2) {
        tensor_cast_kernel<FP8_E5M2><<<blocks, 256, 0, s>>>(x, n, bits, scale, q);
    } else {
        tensor_cast_kernel<FP8_E4M3><<<blocks, 256, 0, s>>>(x, n, bits, scale, q);
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize_tensor_batch(int count, const uint16_t* const* x, const int64_t* n,
                                         int fmt, float* amax, float* scale, uint8_t* const* q,
                                         uint32_t* ws, cudaStream_t s) {
    if (count < 1 || count > kMaxBatch) return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(ws, 0, kTensorScratchBytes, s);
    if (e != cudaSuccess) return e;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    // resident blocks per SM, queried once per device and format
    static std::atomic<int> per_sm[2][64];
    const int f = fmt == FP8_E5M2 ? 1 : 0;
    const void* k = f ? reinterpret_cast<const void*>(tensor_quant_batch_kernel<FP8_E5M2>)
                      : reinterpret_cast<const void*>(tensor_quant_batch_kernel<FP8_E4M3>);
    int bps = dev >= 0 && dev < 64 ? per_sm[f][dev].load() : 0;
    if (bps <= 0) {
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, k, kFusedThreads, 0)) != cudaSuccess)
            return e;
        if (bps <= 0) return cudaErrorInvalidConfiguration;
        if (dev >= 0 && dev < 64) per_sm[f][dev].store(bps);
    }
    TensorBatch b{};
    int64_t chunks = 1;
    for (int t = 0; t < count; ++t) {
        b.x[t] = x[t];
        b.q[t] = q[t];
        b.amax[t] = amax + t;
        b.scale[t] = scale + t;
        b.n[t] = n[t];
        b.v8[t] = reinterpret_cast<uintptr_t>(x[t]) % 32 == 0;
        chunks = std::max<int64_t>(chunks, n[t] / 16 + 1);
    }
    b.count = count;
    const int64_t resident = static_cast<int64_t>(sm_count_current_device()) * bps;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((chunks + kFusedThreads - 1) / kFusedThreads, resident)));
    uint64_t limit = wait_limit_ns();
    void* args[] = {&b, &ws, &limit};
    e = cudaLaunchCooperativeKernel(k, dim3(grid), dim3(kFusedThreads), args, 0, s);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_quantize_tensor_fused(const uint16_t* x, int64_t n, int fmt, float* amax,
                                         float* scale, uint8_t* q, uint32_t* ws, cudaStream_t s) {
    return launch_quantize_tensor_batch(1, &x, &n, fmt, amax, scale, &q, ws, s);
}

// Scratch of fp8_quantize_tensor_noalloc: a file-scope device array, so that
// entry point needs no memory from its caller.  Every GPU that loads this
// library holds these 256 bytes until the process exits; all calls on a
// device share them (the launch clears the first kTensorScratchBytes = 68).
constexpr size_t kNoAllocScratchBytes = kTensorWorkspaceBytes;
static_assert(kTensorScratchBytes <= kNoAllocScratchBytes, "per-tensor scratch exceeds the static array");
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / 4];

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress, once per device, while that device is current.
// The cached address belongs to the device's context of that moment: a
// cudaDeviceReset (or any other teardown of that context) invalidates it.
cudaError_t noalloc_scratch_address(uint32_t** out) {
    constexpr int kDevices = 64;
    static std::mutex mu;
    static uint32_t* addr[kDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<uint32_t*>(p);
    }
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_quantize_tensor_scaled(const uint16_t* x, int64_t n, int fmt, const float* scale,
                                          uint8_t* q, float* amax, unsigned long long* sat,
                                          cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(sat, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return e;
    if (n == 0) return cudaSuccess;
    const int blocks = elementwise_blocks(n, 8);
    unsigned* bits = reinterpret_cast<unsigned*>(amax);
    if (fmt == FP8_E5M2) {
        tensor_cast_scaled_kernel<FP8_E5M2><<<blocks, 256, 0, s>>>(x, n, scale, q, bits, sat);
    } else {
        tensor_cast_scaled_kernel<FP8_E4M3><<<blocks, 256, 0, s>>>(x, n, scale, q, bits, sat);
    }
    return cudaGetLastError();
}

cudaError_t launch_quantize_tensor_delayed(const uint16_t* x, int64_t n, int fmt, float margin,
                                           float* hist, int h, int* pos, float* scale,
                                           uint8_t* q, float* amax, unsigned long long* sat,
                                           cudaStream_t s) {
    unsigned* bits = reinterpret_cast<unsigned*>(amax);
    delayed_scale_kernel<<<1, 1, 0, s>>>(hist, h, fmt, margin, scale, bits, sat);
    if (n > 0) {
        const int blocks = elementwise_blocks(n, 8);
        if (fmt == FP8_E5M2) {
            tensor_cast_scaled_kernel<FP8_E5M2><<<blocks, 256, 0, s>>>(x, n, scale, q, bits, sat);
        } else {
            tensor_cast_scaled_kernel<FP8_E4M3><<<blocks, 256, 0, s>>>(x, n, scale, q, bits, sat);
        }
    }
    delayed_record_kernel<<<1, 1, 0, s>>>(hist, h, pos, bits);
    return cudaGetLastError();
}

cudaError_t launch_requantize_tensor(const uint8_t* q_in, int64_t n, int fmt_in, const float* s_in,
                                     const float* s_out, int fmt_out, uint8_t* q_out,
                                     unsigned long long* sat, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(sat, 0, sizeof(unsigned long long), s);
    if (e != cudaSuccess) return e;
    if (n == 0) return cudaSuccess;
    const int blocks = elementwise_blocks(n, 16);
#define MXFP8_REQ(FI, FO) requantize_kernel<FI, FO><<<blocks, 256, 0, s>>>(q_in, n, s_in, s_out, q_out, sat)
    if (fmt_in == FP8_E4M3) {
        if (fmt_out == FP8_E4M3) MXFP8_REQ(FP8_E4M3, FP8_E4M3); else MXFP8_REQ(FP8_E4M3, FP8_E5M2);
    } else {
        if (fmt_out == FP8_E4M3) MXFP8_REQ(FP8_E5M2, FP8_E4M3); else MXFP8_REQ(FP8_E5M2, FP8_E5M2);
    }
#undef MXFP8_REQ
    return cudaGetLastError();
}

cudaError_t take_status_quant(unsigned* out) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status_quant, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status_quant, &zero, sizeof(unsigned));
}

}  // namespace mxfp8
