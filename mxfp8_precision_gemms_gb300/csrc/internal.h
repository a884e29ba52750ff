// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mxfp8.h"

namespace mxfp8 {

// Kernel launch with programmatic stream serialization: the kernel may start
// while the kernel before it on the stream is finishing, so it must call
// griddep_wait() (ptx.cuh) before its first global memory access.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Index checks of the bounds-checked build (compiled with
// -DMXFP8_BOUNDS_CHECK into libmxfp8_bc.so): each guards one global access
// with the extent of the tensor it touches, stated independently of the
// kernel's own tile arithmetic; a failed check records
// MXFP8_ERR_DEVICE_CHECK through the kernel file's own record_status and the
// access is skipped.  In the product build every check is the constant true
// and compiles away.
#ifdef MXFP8_BOUNDS_CHECK
#define MX_IN_BOUNDS(cond) ((cond) || (record_status(MXFP8_ERR_DEVICE_CHECK), false))
#else
#define MX_IN_BOUNDS(cond) true
#endif

// Launch parameters of the MX quantizer (plain or grouped rows).
struct QuantMxArgs {
    const uint16_t* x;
    int64_t rows;       // plain: rows of x; grouped: total rows
    int64_t cols;
    int64_t ld;
    uint8_t* q_row;
    uint8_t* s_row;
    uint8_t* q_col;
    uint8_t* s_col;
    const int32_t* offsets;  // grouped only (device)
    int32_t groups;          // grouped only
    unsigned flags;
};

cudaError_t launch_quantize_mx(const QuantMxArgs& a, cudaStream_t s);
cudaError_t launch_quantize_mx_grouped(const QuantMxArgs& a, cudaStream_t s);
// Rowwise MX quantization of count (<= kMaxBatch) tensors in one launch;
// every a[t].flags carries the same MX_SCALE_FLOOR choice.
cudaError_t launch_quantize_mx_rows_batch(int count, const QuantMxArgs* a, cudaStream_t s);
// Colwise (or both-orientation) MX quantization of count tensors with as few
// launches as possible (one per 8 tensors); every a[t].flags includes
// MX_COLWISE and carries the same MX_SCALE_FLOOR choice.
cudaError_t launch_quantize_mx_cols_batch(int count, const QuantMxArgs* a, cudaStream_t s);
cudaError_t launch_quantize_tensor(const uint16_t* x, int64_t n, int fmt, float* amax,
                                   float* scale, uint8_t* q, cudaStream_t s);
// Tensors one batched per-tensor launch accepts.
constexpr int kMaxBatch = 16;

// Scratch of the single-launch per-tensor path: kMaxBatch + 1 uint32 words
// (one amax word per tensor, then the grid barrier's arrival count), cleared
// on the stream before each launch.  kTensorWorkspaceBytes is what
// mxfp8_tensor_workspace_bytes() reports (the documented size, with room
// to spare) and what the allocation-free entry point's static array holds.
constexpr size_t kTensorScratchBytes = (kMaxBatch + 1) * sizeof(uint32_t);
constexpr size_t kTensorWorkspaceBytes = 256;
static_assert(kTensorScratchBytes <= kTensorWorkspaceBytes,
              "the per-tensor scratch must fit the documented workspace");

// Single cooperative launch for `count` tensors (amax[t], scale[t] are
// consecutive device floats); ws: kMaxBatch + 1 uint32 of device scratch
// (zeroed here).
cudaError_t launch_quantize_tensor_batch(int count, const uint16_t* const* x, const int64_t* n,
                                         int fmt, float* amax, float* scale, uint8_t* const* q,
                                         uint32_t* ws, cudaStream_t s);

// Single cooperative launch; ws: kMaxBatch + 1 uint32 of device scratch (zeroed here).
// The scratch it needs, whatever n is: mxfp8_tensor_workspace_bytes().
cudaError_t launch_quantize_tensor_fused(const uint16_t* x, int64_t n, int fmt, float* amax,
                                         float* scale, uint8_t* q, uint32_t* ws, cudaStream_t s);

// The kernels around the quantizer (fused.cu).  offsets == nullptr selects
// the plain layout; otherwise scales are group-padded as in the grouped
// quantizer.
struct DequantArgs {
    const uint8_t* q;
    const uint8_t* s;
    int64_t rows, cols;
    const int32_t* offsets;
    int32_t groups;
    uint16_t* out;
    int64_t ldo;
};

struct SwigluQuantArgs {
    const uint16_t* h;  // rows x 2f: gate columns [0, f), up columns [f, 2f)
    int64_t rows, f, ld;
    const int32_t* offsets;
    int32_t groups;
    unsigned flags;
    uint8_t* q;
    uint8_t* s;
};

struct WeightedQuantArgs {
    const uint16_t* dy;  // tokens x cols, leading dimension ld
    int64_t tokens, ld;
    const int32_t* row_token;
    const float* row_weight;
    int64_t rows, cols;
    const int32_t* offsets;
    int32_t groups;
    unsigned flags;
    uint8_t* q;
    uint8_t* s;
};

struct WeightedTokensArgs {
    const uint16_t* dy;  // tokens x cols, leading dimension ld
    int64_t tokens, ld;
    int k;                        // routes per token
    const int32_t* token_rows;    // tokens x k dispatched rows (-1: none)
    const float* token_weights;   // tokens x k
    int64_t rows, cols;
    const int32_t* offsets;
    int32_t groups;
    unsigned flags;
    uint8_t* q;
    uint8_t* s;
    size_t scale_bytes;           // size of s (zeroed first)
};

cudaError_t launch_dequantize_mx(const DequantArgs& a, cudaStream_t s);
cudaError_t launch_weighted_quantize_tokens_mx(const WeightedTokensArgs& a, cudaStream_t s);
cudaError_t launch_swiglu_quantize_mx(const SwigluQuantArgs& a, cudaStream_t s);
cudaError_t launch_weighted_quantize_mx(const WeightedQuantArgs& a, cudaStream_t s);
// Test hook: the SwiGLU fast path's fp32 value per element.
cudaError_t launch_debug_swiglu_f32(const uint16_t* g, const uint16_t* u, int64_t n, float* y,
                                    cudaStream_t s);
cudaError_t take_status_fused(unsigned* out);

// Delayed / automatic scaling (quantize.cu).  sat: 64-bit saturated count.
cudaError_t launch_quantize_tensor_scaled(const uint16_t* x, int64_t n, int fmt, const float* scale,
                                          uint8_t* q, float* amax, unsigned long long* sat,
                                          cudaStream_t s);
cudaError_t launch_quantize_tensor_delayed(const uint16_t* x, int64_t n, int fmt, float margin,
                                           float* hist, int h, int* pos, float* scale,
                                           uint8_t* q, float* amax, unsigned long long* sat,
                                           cudaStream_t s);
cudaError_t launch_requantize_tensor(const uint8_t* q_in, int64_t n, int fmt_in, const float* s_in,
                                     const float* s_out, int fmt_out, uint8_t* q_out,
                                     unsigned long long* sat, cudaStream_t s);

struct GemmArgs {
    int mode;          // GEMM_MX or GEMM_TENSOR
    int a_fmt, b_fmt;  // FP8_E4M3 / FP8_E5M2
    const uint8_t* a;
    const void* a_scale;
    const uint8_t* b;
    const void* b_scale;
    int64_t M, N, K;   // grouped: M = total rows
    uint16_t* c;
    int64_t ldc;
    const int32_t* offsets;  // grouped only (device)
    int32_t groups;          // grouped: number of experts; plain: 0
};

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t s);
// Two plain GEMMs of one mode (M, N, K > 0 each) in one persistent launch,
// the CTA pairs split between them.
cudaError_t launch_gemm_dual(const GemmArgs& g0, const GemmArgs& g1, cudaStream_t s);
cudaError_t launch_zero_fill_bf16(uint16_t* c, int64_t rows, int64_t cols, int64_t ldc,
                                  cudaStream_t s);

// Per-translation-unit device status words: read (and clear) after a sync.
cudaError_t take_status_quant(unsigned* out);

// The allocation-free per-tensor path's static device scratch: its size and
// its address on the current device (looked up once per device).
size_t noalloc_scratch_bytes();
cudaError_t noalloc_scratch_address(uint32_t** out);
cudaError_t take_status_gemm(unsigned* out);

// Time limit for device waits (ns) and the one-shot timeout-injection hook.
uint64_t wait_limit_ns();
bool take_inject_timeout();

int sm_count_current_device();

// 2D tensor map (TMA descriptor) over a rows x width matrix of `dtype`
// elements with the given row stride in bytes; box of box_w x box_rows
// elements.  Returns false when the driver rejects it.
bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                          int64_t rows, int64_t width, int64_t row_stride_bytes, uint32_t box_w,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle);

// A row-major rows x k byte matrix (row stride k, k % 128 == 0) seen as
// [k / 128 chunks][rows][128 bytes]: one box of box_rows x box_chunks lands
// as box_chunks consecutive (box_rows x 128)-byte tiles, 128-byte swizzled.
bool encode_kchunk_map_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t k,
                          uint32_t box_rows, uint32_t box_chunks);

}  // namespace mxfp8
