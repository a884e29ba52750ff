// C ABI of the library (declared in include/mxfp8.h): argument validation,
// then stream-ordered kernel launches.  Nothing here allocates device memory
// or synchronizes, except mxfp8_last_device_status().
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"

namespace mxfp8 {

namespace {

thread_local char g_err[256] = "";
std::atomic<uint64_t> g_wait_limit{2000000000ull};
std::atomic<int> g_inject{0};

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

mxfp8_status fail(mxfp8_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mxfp8_status fail(mxfp8_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

mxfp8_status ok() {
    g_err[0] = '\0';
    return MXFP8_OK;
}

mxfp8_status cuda_result(cudaError_t e, const char* what) {
    if (e != cudaSuccess) return fail(MXFP8_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Optional group offsets of the routed entry points: NULL with groups == 0
// selects the plain layout; otherwise 1 <= groups <= 1024 and rows < 2^31.
mxfp8_status check_groups(const int32_t* offsets, int32_t groups, int64_t rows) {
    if (!offsets) {
        if (groups != 0) return fail(MXFP8_ERR_INVALID_ARG, "groups given without group_offsets");
        return ok();
    }
    if (groups <= 0) return fail(MXFP8_ERR_INVALID_ARG, "groups must be >= 1 with group_offsets");
    if (groups > 1024) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "groups > 1024");
    if (rows > 0x7FFFFFFF) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "grouped rows >= 2^31");
    return ok();
}

}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit.load(); }
bool take_inject_timeout() { return g_inject.exchange(0) != 0; }

int sm_count_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = g_sm_count[dev].load();
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        g_sm_count[dev].store(n);
    }
    return n;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        }
    });
    return fn;
}

}  // namespace

bool encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                          int64_t rows, int64_t width, int64_t row_stride_bytes, uint32_t box_w,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride_bytes)};
    const cuuint32_t box[2] = {box_w, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_kchunk_map_u8(CUtensorMap* map, const void* base, int64_t rows, int64_t k,
                          uint32_t box_rows, uint32_t box_chunks) {
    if (k % 128) return false;
    auto enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(k / 128)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(k), 128};
    const cuuint32_t box[3] = {128, box_rows, box_chunks};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// What a checked GEMM call needs: a launch, nothing (M or N is 0) or a zero
// fill of C (K == 0).
enum GemmKind { kGemmLaunch, kGemmNothing, kGemmZero };

mxfp8_status check_gemm(int mode, int a_fmt, int b_fmt, const void* a, const void* a_scale,
                        const void* b, const void* b_scale, int64_t M, int64_t N, int64_t K,
                        void* c_bf16, int64_t ldc, GemmArgs* g, GemmKind* kind) {
    if (mode != GEMM_MX && mode != GEMM_TENSOR) return fail(MXFP8_ERR_INVALID_ARG, "unknown mode %d", mode);
    if ((a_fmt != FP8_E4M3 && a_fmt != FP8_E5M2) || (b_fmt != FP8_E4M3 && b_fmt != FP8_E5M2))
        return fail(MXFP8_ERR_INVALID_ARG, "unknown format");
    if (mode == GEMM_MX && (a_fmt != FP8_E4M3 || b_fmt != FP8_E4M3))
        return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "MX mode takes E4M3 payloads");
    if (M < 0 || N < 0 || K < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    *g = GemmArgs{};
    g->M = M;
    g->N = N;
    g->c = static_cast<uint16_t*>(c_bf16);
    g->ldc = ldc;
    if (M == 0 || N == 0) {
        *kind = kGemmNothing;
        return MXFP8_OK;
    }
    if (!c_bf16) return fail(MXFP8_ERR_INVALID_ARG, "c is NULL");
    if (ldc < N) return fail(MXFP8_ERR_INVALID_ARG, "ldc < N");
    if (N % 8 || ldc % 8 || !aligned16(c_bf16))
        return fail(MXFP8_ERR_MISALIGNED, "N, ldc or c not 16-byte aligned");
    if (K == 0) {
        *kind = kGemmZero;
        return MXFP8_OK;
    }
    if (!a || !b || !a_scale || !b_scale) return fail(MXFP8_ERR_INVALID_ARG, "operand or scale is NULL");
    if (mode == GEMM_MX && K % 32) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "MX mode needs K %% 32 == 0");
    if (K % 16) return fail(MXFP8_ERR_MISALIGNED, "K %% 16 != 0 (row stride of A/B)");
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF)
        return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "dimension >= 2^31");
    if (!aligned16(a) || !aligned16(b)) return fail(MXFP8_ERR_MISALIGNED, "operand not 16-byte aligned");
    if (mode == GEMM_MX && (!aligned16(a_scale) || !aligned16(b_scale)))
        return fail(MXFP8_ERR_MISALIGNED, "scale array not 16-byte aligned");
    if (mode == GEMM_TENSOR &&
        ((reinterpret_cast<uintptr_t>(a_scale) & 3u) || (reinterpret_cast<uintptr_t>(b_scale) & 3u)))
        return fail(MXFP8_ERR_MISALIGNED, "scale scalar not 4-byte aligned");
    g->mode = mode;
    g->a_fmt = a_fmt;
    g->b_fmt = b_fmt;
    g->a = static_cast<const uint8_t*>(a);
    g->a_scale = a_scale;
    g->b = static_cast<const uint8_t*>(b);
    g->b_scale = b_scale;
    g->K = K;
    *kind = kGemmLaunch;
    return MXFP8_OK;
}

// One checked GEMM on its own.
mxfp8_status run_gemm(const GemmArgs& g, GemmKind kind, cudaStream_t s, const char* what) {
    if (kind == kGemmNothing) return ok();
    if (kind == kGemmZero) return cuda_result(launch_zero_fill_bf16(g.c, g.M, g.N, g.ldc, s), "zero fill");
    return cuda_result(launch_gemm(g, s), what);
}

}  // namespace

}  // namespace mxfp8

using namespace mxfp8;

extern "C" {

size_t mxfp8_scale_bytes(int64_t rows, int64_t k) {
    if (rows <= 0 || k <= 0) return 0;
    return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((k + 127) / 128) * 512u;
}

size_t mxfp8_grouped_scale_bytes(int64_t total_rows, int64_t k, int32_t groups) {
    if (total_rows < 0 || k <= 0 || groups <= 0) return 0;
    return static_cast<size_t>((total_rows + 127) / 128 + groups) *
           static_cast<size_t>((k + 127) / 128) * 512u;
}

mxfp8_status fp8_quantize_mx(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                             unsigned flags, void* q_row, void* s_row, void* q_col, void* s_col,
                             mxfp8_stream_t stream) {
    const bool row = flags & MX_ROWWISE, col = flags & MX_COLWISE;
    if (flags & ~7u) return fail(MXFP8_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
    if (!row && !col) return fail(MXFP8_ERR_INVALID_ARG, "flags select no orientation");
    if (rows < 0 || cols < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (rows == 0 || cols == 0) return ok();
    if (!x_bf16) return fail(MXFP8_ERR_INVALID_ARG, "x is NULL");
    if (row && (!q_row || !s_row)) return fail(MXFP8_ERR_INVALID_ARG, "rowwise output is NULL");
    if (col && (!q_col || !s_col)) return fail(MXFP8_ERR_INVALID_ARG, "colwise output is NULL");
    if (cols % 32) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "cols %% 32 != 0 (cols=%lld)", (long long)cols);
    if (col && rows % 32)
        return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "colwise needs rows %% 32 == 0 (rows=%lld)", (long long)rows);
    if (ld < cols) return fail(MXFP8_ERR_INVALID_ARG, "ld < cols");
    if (ld % 8 || !aligned16(x_bf16)) return fail(MXFP8_ERR_MISALIGNED, "x or ld not 16-byte aligned");
    if ((row && (!aligned16(q_row) || !aligned16(s_row))) || (col && (!aligned16(q_col) || !aligned16(s_col))))
        return fail(MXFP8_ERR_MISALIGNED, "output pointer not 16-byte aligned");
    QuantMxArgs a{};
    a.x = static_cast<const uint16_t*>(x_bf16);
    a.rows = rows;
    a.cols = cols;
    a.ld = ld;
    a.q_row = static_cast<uint8_t*>(q_row);
    a.s_row = static_cast<uint8_t*>(s_row);
    a.q_col = static_cast<uint8_t*>(q_col);
    a.s_col = static_cast<uint8_t*>(s_col);
    a.flags = flags;
    return cuda_result(launch_quantize_mx(a, reinterpret_cast<cudaStream_t>(stream)), "fp8_quantize_mx launch");
}

mxfp8_status fp8_quantize_mx_batch(int32_t count, const void* const* x_bf16, const int64_t* rows,
                                   const int64_t* cols, const int64_t* ld, const unsigned* flags,
                                   void* const* q_row, void* const* s_row, void* const* q_col,
                                   void* const* s_col, mxfp8_stream_t stream) {
    if (count < 1 || count > kMaxBatch)
        return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "count must be in [1, %d]", kMaxBatch);
    if (!x_bf16 || !rows || !cols || !ld || !flags)
        return fail(MXFP8_ERR_INVALID_ARG, "an argument array is NULL");
    QuantMxArgs row_only[kMaxBatch] = {}, with_col[kMaxBatch] = {};
    int n_row = 0, n_col = 0;
    int floor_bit = -1;
    for (int t = 0; t < count; ++t) {
        const unsigned f = flags[t];
        const bool row = f & MX_ROWWISE, col = f & MX_COLWISE;
        if (f & ~7u) return fail(MXFP8_ERR_INVALID_ARG, "unknown flag bits 0x%x (tensor %d)", f, t);
        if (!row && !col) return fail(MXFP8_ERR_INVALID_ARG, "flags of tensor %d select no orientation", t);
        if (rows[t] < 0 || cols[t] < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size (tensor %d)", t);
        if (rows[t] == 0 || cols[t] == 0) continue;
        const int fb = (f & MX_SCALE_FLOOR) ? 1 : 0;
        if (floor_bit >= 0 && fb != floor_bit)
            return fail(MXFP8_ERR_INVALID_ARG, "MX_SCALE_FLOOR must be the same for every tensor");
        floor_bit = fb;
        if (!x_bf16[t]) return fail(MXFP8_ERR_INVALID_ARG, "x of tensor %d is NULL", t);
        if (row && (!q_row || !s_row || !q_row[t] || !s_row[t]))
            return fail(MXFP8_ERR_INVALID_ARG, "rowwise output of tensor %d is NULL", t);
        if (col && (!q_col || !s_col || !q_col[t] || !s_col[t]))
            return fail(MXFP8_ERR_INVALID_ARG, "colwise output of tensor %d is NULL", t);
        if (cols[t] % 32)
            return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "cols %% 32 != 0 (tensor %d, cols=%lld)", t, (long long)cols[t]);
        if (col && rows[t] % 32)
            return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "colwise needs rows %% 32 == 0 (tensor %d)", t);
        if (ld[t] < cols[t]) return fail(MXFP8_ERR_INVALID_ARG, "ld < cols (tensor %d)", t);
        if (ld[t] % 8 || !aligned16(x_bf16[t]))
            return fail(MXFP8_ERR_MISALIGNED, "x or ld of tensor %d not 16-byte aligned", t);
        if ((row && (!aligned16(q_row[t]) || !aligned16(s_row[t]))) ||
            (col && (!aligned16(q_col[t]) || !aligned16(s_col[t]))))
            return fail(MXFP8_ERR_MISALIGNED, "an output of tensor %d is not 16-byte aligned", t);
        if ((cols[t] + 127) / 128 > 65535 || rows[t] > 0x7FFFFFFF)
            return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "tensor %d too large", t);
        QuantMxArgs& a = col ? with_col[n_col++] : row_only[n_row++];
        a.x = static_cast<const uint16_t*>(x_bf16[t]);
        a.rows = rows[t];
        a.cols = cols[t];
        a.ld = ld[t];
        a.q_row = row ? static_cast<uint8_t*>(q_row[t]) : nullptr;
        a.s_row = row ? static_cast<uint8_t*>(s_row[t]) : nullptr;
        a.q_col = col ? static_cast<uint8_t*>(q_col[t]) : nullptr;
        a.s_col = col ? static_cast<uint8_t*>(s_col[t]) : nullptr;
        a.flags = f;
    }
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (n_row) e = launch_quantize_mx_rows_batch(n_row, row_only, st);
    if (e == cudaSuccess && n_col) e = launch_quantize_mx_cols_batch(n_col, with_col, st);
    return cuda_result(e, "fp8_quantize_mx_batch launch");
}

mxfp8_status fp8_quantize_mx_grouped(const void* x_bf16, int64_t total_rows, int64_t cols,
                                     int64_t ld, const int32_t* group_offsets_dev, int32_t groups,
                                     unsigned flags, void* q, void* s, mxfp8_stream_t stream) {
    if (flags & ~(unsigned)(MX_ROWWISE | MX_SCALE_FLOOR))
        return fail(MXFP8_ERR_INVALID_ARG, "grouped quantization is rowwise only");
    if (groups <= 0) return fail(MXFP8_ERR_INVALID_ARG, "groups must be >= 1");
    if (groups > 1024) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "groups > 1024");
    if (total_rows < 0 || cols < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (total_rows > 0x7FFFFFFF) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "total_rows >= 2^31");
    if (!group_offsets_dev) return fail(MXFP8_ERR_INVALID_ARG, "group_offsets is NULL");
    if (cols == 0 || total_rows == 0) return ok();
    if (!x_bf16) return fail(MXFP8_ERR_INVALID_ARG, "x is NULL");
    if (!q || !s) return fail(MXFP8_ERR_INVALID_ARG, "output is NULL");
    if (cols % 32) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "cols %% 32 != 0");
    if (ld < cols) return fail(MXFP8_ERR_INVALID_ARG, "ld < cols");
    if (ld % 8 || !aligned16(x_bf16) || !aligned16(q) || !aligned16(s))
        return fail(MXFP8_ERR_MISALIGNED, "pointer or ld not 16-byte aligned");
    QuantMxArgs a{};
    a.x = static_cast<const uint16_t*>(x_bf16);
    a.rows = total_rows;
    a.cols = cols;
    a.ld = ld;
    a.q_row = static_cast<uint8_t*>(q);
    a.s_row = static_cast<uint8_t*>(s);
    a.offsets = group_offsets_dev;
    a.groups = groups;
    a.flags = flags | MX_ROWWISE;
    return cuda_result(launch_quantize_mx_grouped(a, reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_quantize_mx_grouped launch");
}

size_t mxfp8_tensor_workspace_bytes(void) { return kTensorWorkspaceBytes; }

mxfp8_status fp8_quantize_tensor_scaled(const void* x_bf16, int64_t n, int fmt,
                                        const float* scale_dev, void* q, float* amax_dev,
                                        uint64_t* sat_count_dev, mxfp8_stream_t stream) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(MXFP8_ERR_INVALID_ARG, "unknown format %d", fmt);
    if (n < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (!scale_dev || !amax_dev || !sat_count_dev)
        return fail(MXFP8_ERR_INVALID_ARG, "scale, amax or sat_count is NULL");
    if (n > 0 && (!x_bf16 || !q)) return fail(MXFP8_ERR_INVALID_ARG, "x or q is NULL");
    if ((n > 0 && (!aligned16(x_bf16) || !aligned16(q))) ||
        (reinterpret_cast<uintptr_t>(scale_dev) & 3u) || (reinterpret_cast<uintptr_t>(amax_dev) & 3u) ||
        (reinterpret_cast<uintptr_t>(sat_count_dev) & 7u))
        return fail(MXFP8_ERR_MISALIGNED, "pointer misaligned");
    return cuda_result(launch_quantize_tensor_scaled(static_cast<const uint16_t*>(x_bf16), n, fmt,
                                                     scale_dev, static_cast<uint8_t*>(q), amax_dev,
                                                     reinterpret_cast<unsigned long long*>(sat_count_dev),
                                                     reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_quantize_tensor_scaled launch");
}

mxfp8_status fp8_quantize_tensor_delayed(const void* x_bf16, int64_t n, int fmt, float margin,
                                         float* amax_history_dev, int32_t history_len,
                                         int32_t* history_pos_dev, float* scale_dev, void* q,
                                         float* amax_dev, uint64_t* sat_count_dev,
                                         mxfp8_stream_t stream) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(MXFP8_ERR_INVALID_ARG, "unknown format %d", fmt);
    if (n < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (history_len < 1 || history_len > 65536)
        return fail(MXFP8_ERR_INVALID_ARG, "history_len must be in [1, 65536]");
    if (!amax_history_dev || !history_pos_dev || !scale_dev || !amax_dev || !sat_count_dev)
        return fail(MXFP8_ERR_INVALID_ARG, "a state or output pointer is NULL");
    if (n > 0 && (!x_bf16 || !q)) return fail(MXFP8_ERR_INVALID_ARG, "x or q is NULL");
    if ((n > 0 && (!aligned16(x_bf16) || !aligned16(q))) ||
        ((reinterpret_cast<uintptr_t>(amax_history_dev) | reinterpret_cast<uintptr_t>(history_pos_dev) |
          reinterpret_cast<uintptr_t>(scale_dev) | reinterpret_cast<uintptr_t>(amax_dev)) & 3u) ||
        (reinterpret_cast<uintptr_t>(sat_count_dev) & 7u))
        return fail(MXFP8_ERR_MISALIGNED, "pointer misaligned");
    return cuda_result(
        launch_quantize_tensor_delayed(static_cast<const uint16_t*>(x_bf16), n, fmt, margin,
                                       amax_history_dev, history_len, history_pos_dev, scale_dev,
                                       static_cast<uint8_t*>(q), amax_dev,
                                       reinterpret_cast<unsigned long long*>(sat_count_dev),
                                       reinterpret_cast<cudaStream_t>(stream)),
        "fp8_quantize_tensor_delayed launch");
}

mxfp8_status fp8_requantize_tensor(const void* q_in, int64_t n, int fmt_in, const float* scale_in_dev,
                                   const float* scale_out_dev, int fmt_out, void* q_out,
                                   uint64_t* sat_count_dev, mxfp8_stream_t stream) {
    if ((fmt_in != FP8_E4M3 && fmt_in != FP8_E5M2) || (fmt_out != FP8_E4M3 && fmt_out != FP8_E5M2))
        return fail(MXFP8_ERR_INVALID_ARG, "unknown format");
    if (n < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (!scale_in_dev || !scale_out_dev || !sat_count_dev)
        return fail(MXFP8_ERR_INVALID_ARG, "a scale or sat_count is NULL");
    if (n > 0 && (!q_in || !q_out)) return fail(MXFP8_ERR_INVALID_ARG, "q_in or q_out is NULL");
    if ((n > 0 && (!aligned16(q_in) || !aligned16(q_out))) ||
        ((reinterpret_cast<uintptr_t>(scale_in_dev) | reinterpret_cast<uintptr_t>(scale_out_dev)) & 3u) ||
        (reinterpret_cast<uintptr_t>(sat_count_dev) & 7u))
        return fail(MXFP8_ERR_MISALIGNED, "pointer misaligned");
    return cuda_result(launch_requantize_tensor(static_cast<const uint8_t*>(q_in), n, fmt_in, scale_in_dev,
                                                scale_out_dev, fmt_out, static_cast<uint8_t*>(q_out),
                                                reinterpret_cast<unsigned long long*>(sat_count_dev),
                                                reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_requantize_tensor launch");
}

mxfp8_status fp8_dequantize_mx(const void* q, const void* s, int64_t rows, int64_t cols,
                               const int32_t* group_offsets_dev, int32_t groups, void* out_bf16,
                               int64_t ldo, mxfp8_stream_t stream) {
    if (rows < 0 || cols < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    mxfp8_status st = check_groups(group_offsets_dev, groups, rows);
    if (st != MXFP8_OK) return st;
    if (rows == 0 || cols == 0) return ok();
    if (!q || !s || !out_bf16) return fail(MXFP8_ERR_INVALID_ARG, "q, s or out is NULL");
    if (cols % 32) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "cols %% 32 != 0 (cols=%lld)", (long long)cols);
    if (ldo < cols) return fail(MXFP8_ERR_INVALID_ARG, "ldo < cols");
    if (ldo % 8 || !aligned16(q) || !aligned16(s) || !aligned16(out_bf16))
        return fail(MXFP8_ERR_MISALIGNED, "pointer or ldo not 16-byte aligned");
    DequantArgs a{};
    a.q = static_cast<const uint8_t*>(q);
    a.s = static_cast<const uint8_t*>(s);
    a.rows = rows;
    a.cols = cols;
    a.offsets = group_offsets_dev;
    a.groups = groups;
    a.out = static_cast<uint16_t*>(out_bf16);
    a.ldo = ldo;
    return cuda_result(launch_dequantize_mx(a, reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_dequantize_mx launch");
}

mxfp8_status fp8_swiglu_quantize_mx(const void* h_bf16, int64_t rows, int64_t f, int64_t ld,
                                    const int32_t* group_offsets_dev, int32_t groups,
                                    unsigned flags, void* q, void* s, mxfp8_stream_t stream) {
    if (flags & ~(unsigned)(MX_ROWWISE | MX_SCALE_FLOOR))
        return fail(MXFP8_ERR_INVALID_ARG, "SwiGLU quantization is rowwise only");
    if (rows < 0 || f < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    mxfp8_status st = check_groups(group_offsets_dev, groups, rows);
    if (st != MXFP8_OK) return st;
    if (rows == 0 || f == 0) return ok();
    if (!h_bf16 || !q || !s) return fail(MXFP8_ERR_INVALID_ARG, "h, q or s is NULL");
    if (f % 32) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "f %% 32 != 0 (f=%lld)", (long long)f);
    if (ld < 2 * f) return fail(MXFP8_ERR_INVALID_ARG, "ld < 2 f");
    if (ld % 8 || !aligned16(h_bf16) || !aligned16(q) || !aligned16(s))
        return fail(MXFP8_ERR_MISALIGNED, "pointer or ld not 16-byte aligned");
    SwigluQuantArgs a{};
    a.h = static_cast<const uint16_t*>(h_bf16);
    a.rows = rows;
    a.f = f;
    a.ld = ld;
    a.offsets = group_offsets_dev;
    a.groups = groups;
    a.flags = flags;
    a.q = static_cast<uint8_t*>(q);
    a.s = static_cast<uint8_t*>(s);
    return cuda_result(launch_swiglu_quantize_mx(a, reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_swiglu_quantize_mx launch");
}

mxfp8_status fp8_route_weight_quantize_mx(const void* dy_bf16, int64_t tokens, int64_t ld,
                                          const int32_t* row_token_dev,
                                          const float* row_weight_dev, int64_t rows,
                                          int64_t cols, const int32_t* group_offsets_dev,
                                          int32_t groups, unsigned flags, void* q, void* s,
                                          mxfp8_stream_t stream) {
    if (flags & ~(unsigned)(MX_ROWWISE | MX_SCALE_FLOOR))
        return fail(MXFP8_ERR_INVALID_ARG, "route-weighted quantization is rowwise only");
    if (rows < 0 || cols < 0 || tokens < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    mxfp8_status st = check_groups(group_offsets_dev, groups, rows);
    if (st != MXFP8_OK) return st;
    if (rows == 0 || cols == 0) return ok();
    if (!dy_bf16 || !row_token_dev || !row_weight_dev || !q || !s)
        return fail(MXFP8_ERR_INVALID_ARG, "dy, row_token, row_weight, q or s is NULL");
    if (tokens == 0) return fail(MXFP8_ERR_INVALID_ARG, "rows to fill but no tokens");
    if (cols % 32) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "cols %% 32 != 0 (cols=%lld)", (long long)cols);
    if (ld < cols) return fail(MXFP8_ERR_INVALID_ARG, "ld < cols");
    if (ld % 8 || !aligned16(dy_bf16) || !aligned16(q) || !aligned16(s))
        return fail(MXFP8_ERR_MISALIGNED, "pointer or ld not 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(row_token_dev) | reinterpret_cast<uintptr_t>(row_weight_dev)) & 3u)
        return fail(MXFP8_ERR_MISALIGNED, "row_token or row_weight not 4-byte aligned");
    WeightedQuantArgs a{};
    a.dy = static_cast<const uint16_t*>(dy_bf16);
    a.tokens = tokens;
    a.ld = ld;
    a.row_token = row_token_dev;
    a.row_weight = row_weight_dev;
    a.rows = rows;
    a.cols = cols;
    a.offsets = group_offsets_dev;
    a.groups = groups;
    a.flags = flags;
    a.q = static_cast<uint8_t*>(q);
    a.s = static_cast<uint8_t*>(s);
    return cuda_result(launch_weighted_quantize_mx(a, reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_route_weight_quantize_mx launch");
}

mxfp8_status fp8_quantize_tensor(const void* x_bf16, int64_t n, int fmt, float* amax_dev,
                                 float* scale_dev, void* q, void* workspace,
                                 mxfp8_stream_t stream) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(MXFP8_ERR_INVALID_ARG, "unknown format %d", fmt);
    if (n < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (!amax_dev || !scale_dev) return fail(MXFP8_ERR_INVALID_ARG, "amax/scale is NULL");
    if (n > 0 && (!x_bf16 || !q)) return fail(MXFP8_ERR_INVALID_ARG, "x or q is NULL");
    if ((n > 0 && (!aligned16(x_bf16) || !aligned16(q))) ||
        (reinterpret_cast<uintptr_t>(amax_dev) & 3u) || (reinterpret_cast<uintptr_t>(scale_dev) & 3u) ||
        (workspace && !aligned16(workspace)))
        return fail(MXFP8_ERR_MISALIGNED, "pointer misaligned");
    const auto s = reinterpret_cast<cudaStream_t>(stream);
    const auto xs = static_cast<const uint16_t*>(x_bf16);
    const auto qs = static_cast<uint8_t*>(q);
    if (workspace) {
        return cuda_result(launch_quantize_tensor_fused(xs, n, fmt, amax_dev, scale_dev, qs,
                                                        static_cast<uint32_t*>(workspace), s),
                           "fp8_quantize_tensor (fused) launch");
    }
    return cuda_result(launch_quantize_tensor(xs, n, fmt, amax_dev, scale_dev, qs, s),
                       "fp8_quantize_tensor launch");
}

mxfp8_status fp8_quantize_tensor_batch(int32_t count, const void* const* x_bf16, const int64_t* n,
                                       int fmt, float* amax_dev, float* scale_dev, void* const* q,
                                       void* workspace, mxfp8_stream_t stream) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(MXFP8_ERR_INVALID_ARG, "unknown format %d", fmt);
    if (count < 1 || count > kMaxBatch)
        return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "count must be in [1, %d]", kMaxBatch);
    if (!x_bf16 || !n || !q) return fail(MXFP8_ERR_INVALID_ARG, "x, n or q array is NULL");
    if (!amax_dev || !scale_dev || !workspace)
        return fail(MXFP8_ERR_INVALID_ARG, "amax, scale or workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(amax_dev) & 3u) || (reinterpret_cast<uintptr_t>(scale_dev) & 3u) ||
        !aligned16(workspace))
        return fail(MXFP8_ERR_MISALIGNED, "amax/scale/workspace misaligned");
    const uint16_t* xs[kMaxBatch];
    uint8_t* qs[kMaxBatch];
    for (int t = 0; t < count; ++t) {
        if (n[t] < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size (tensor %d)", t);
        if (n[t] > 0 && (!x_bf16[t] || !q[t])) return fail(MXFP8_ERR_INVALID_ARG, "x or q of tensor %d is NULL", t);
        if (n[t] > 0 && (!aligned16(x_bf16[t]) || !aligned16(q[t])))
            return fail(MXFP8_ERR_MISALIGNED, "x or q of tensor %d not 16-byte aligned", t);
        xs[t] = static_cast<const uint16_t*>(x_bf16[t]);
        qs[t] = static_cast<uint8_t*>(q[t]);
    }
    return cuda_result(launch_quantize_tensor_batch(count, xs, n, fmt, amax_dev, scale_dev, qs,
                                                    static_cast<uint32_t*>(workspace),
                                                    reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_quantize_tensor_batch launch");
}

mxfp8_status fp8_quantize_tensor_noalloc(const void* x_bf16, int64_t n, int fmt, float* amax_dev,
                                         float* scale_dev, void* q, mxfp8_stream_t stream) {
    if (fmt != FP8_E4M3 && fmt != FP8_E5M2) return fail(MXFP8_ERR_INVALID_ARG, "unknown format %d", fmt);
    if (n < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (!amax_dev || !scale_dev) return fail(MXFP8_ERR_INVALID_ARG, "amax/scale is NULL");
    if (n > 0 && (!x_bf16 || !q)) return fail(MXFP8_ERR_INVALID_ARG, "x or q is NULL");
    if ((n > 0 && (!aligned16(x_bf16) || !aligned16(q))) ||
        (reinterpret_cast<uintptr_t>(amax_dev) & 3u) || (reinterpret_cast<uintptr_t>(scale_dev) & 3u))
        return fail(MXFP8_ERR_MISALIGNED, "pointer misaligned");
    // the scratch this path needs must fit the library's static array
    const size_t need = kTensorScratchBytes;
    if (need > noalloc_scratch_bytes())
        return fail(MXFP8_ERR_UNSUPPORTED_SHAPE,
                    "needs %zu bytes of scratch, the static device array holds %zu", need,
                    noalloc_scratch_bytes());
    uint32_t* ws = nullptr;
    cudaError_t e = noalloc_scratch_address(&ws);
    if (e != cudaSuccess)
        return fail(MXFP8_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
    return cuda_result(launch_quantize_tensor_fused(static_cast<const uint16_t*>(x_bf16), n, fmt,
                                                    amax_dev, scale_dev, static_cast<uint8_t*>(q), ws,
                                                    reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_quantize_tensor_noalloc launch");
}

mxfp8_status fp8_scaled_gemm(int mode, int a_fmt, int b_fmt, const void* a, const void* a_scale,
                             const void* b, const void* b_scale, int64_t M, int64_t N, int64_t K,
                             void* c_bf16, int64_t ldc, mxfp8_stream_t stream) {
    GemmArgs g;
    GemmKind kind;
    const mxfp8_status st =
        check_gemm(mode, a_fmt, b_fmt, a, a_scale, b, b_scale, M, N, K, c_bf16, ldc, &g, &kind);
    if (st != MXFP8_OK) return st;
    return run_gemm(g, kind, reinterpret_cast<cudaStream_t>(stream), "fp8_scaled_gemm launch");
}

mxfp8_status fp8_scaled_gemm_pair(int mode, int a_fmt0, int b_fmt0, const void* a0,
                                  const void* a_scale0, const void* b0, const void* b_scale0,
                                  int64_t M0, int64_t N0, int64_t K0, void* c0_bf16, int64_t ldc0,
                                  int a_fmt1, int b_fmt1, const void* a1, const void* a_scale1,
                                  const void* b1, const void* b_scale1, int64_t M1, int64_t N1,
                                  int64_t K1, void* c1_bf16, int64_t ldc1, mxfp8_stream_t stream) {
    GemmArgs g0, g1;
    GemmKind k0, k1;
    mxfp8_status st = check_gemm(mode, a_fmt0, b_fmt0, a0, a_scale0, b0, b_scale0, M0, N0, K0,
                                 c0_bf16, ldc0, &g0, &k0);
    if (st != MXFP8_OK) return st;
    st = check_gemm(mode, a_fmt1, b_fmt1, a1, a_scale1, b1, b_scale1, M1, N1, K1, c1_bf16, ldc1, &g1, &k1);
    if (st != MXFP8_OK) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (k0 == kGemmLaunch && k1 == kGemmLaunch)
        return cuda_result(launch_gemm_dual(g0, g1, s), "fp8_scaled_gemm_pair launch");
    st = run_gemm(g0, k0, s, "fp8_scaled_gemm_pair launch (first)");
    if (st != MXFP8_OK) return st;
    return run_gemm(g1, k1, s, "fp8_scaled_gemm_pair launch (second)");
}

mxfp8_status fp8_grouped_gemm(const void* a, const void* a_scale, const void* b, const void* b_scale,
                              const int32_t* group_offsets_dev, int32_t groups, int64_t total_rows,
                              int64_t N, int64_t K, void* c_bf16, int64_t ldc, mxfp8_stream_t stream) {
    if (groups <= 0) return fail(MXFP8_ERR_INVALID_ARG, "groups must be >= 1");
    if (groups > 1024) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "groups > 1024");
    if (total_rows < 0 || N < 0 || K < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (!group_offsets_dev) return fail(MXFP8_ERR_INVALID_ARG, "group_offsets is NULL");
    if (total_rows == 0 || N == 0) return ok();
    if (!c_bf16) return fail(MXFP8_ERR_INVALID_ARG, "c is NULL");
    if (ldc < N) return fail(MXFP8_ERR_INVALID_ARG, "ldc < N");
    if (N % 8 || ldc % 8 || !aligned16(c_bf16))
        return fail(MXFP8_ERR_MISALIGNED, "N, ldc or c not 16-byte aligned");
    if (K == 0) return cuda_result(launch_zero_fill_bf16(static_cast<uint16_t*>(c_bf16), total_rows, N, ldc,
                                                         reinterpret_cast<cudaStream_t>(stream)),
                                   "zero fill");
    if (!a || !b || !a_scale || !b_scale) return fail(MXFP8_ERR_INVALID_ARG, "operand or scale is NULL");
    if (K % 32) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "K %% 32 != 0");
    if (total_rows > 0x7FFFFFFF || static_cast<int64_t>(groups) * N > 0x7FFFFFFF || K > 0x7FFFFFFF)
        return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "dimension >= 2^31");
    if (!aligned16(a) || !aligned16(b) || !aligned16(a_scale) || !aligned16(b_scale))
        return fail(MXFP8_ERR_MISALIGNED, "pointer not 16-byte aligned");
    GemmArgs g{};
    g.mode = GEMM_MX;
    g.a_fmt = g.b_fmt = FP8_E4M3;
    g.a = static_cast<const uint8_t*>(a);
    g.a_scale = a_scale;
    g.b = static_cast<const uint8_t*>(b);
    g.b_scale = b_scale;
    g.M = total_rows;
    g.N = N;
    g.K = K;
    g.c = static_cast<uint16_t*>(c_bf16);
    g.ldc = ldc;
    g.offsets = group_offsets_dev;
    g.groups = groups;
    return cuda_result(launch_gemm(g, reinterpret_cast<cudaStream_t>(stream)), "fp8_grouped_gemm launch");
}

mxfp8_status fp8_route_weight_quantize_mx_tokens(const void* dy_bf16, int64_t tokens, int64_t ld,
                                                 int32_t k, const int32_t* token_rows_dev,
                                                 const float* token_weights_dev, int64_t rows,
                                                 int64_t cols, const int32_t* group_offsets_dev,
                                                 int32_t groups, unsigned flags, void* q, void* s,
                                                 mxfp8_stream_t stream) {
    if (flags & ~(unsigned)(MX_ROWWISE | MX_SCALE_FLOOR))
        return fail(MXFP8_ERR_INVALID_ARG, "route-weighted quantization is rowwise only");
    if (rows < 0 || cols < 0 || tokens < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (k < 1 || k > 16) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "k must be in [1, 16] (k=%d)", k);
    mxfp8_status st = check_groups(group_offsets_dev, groups, rows);
    if (st != MXFP8_OK) return st;
    if (rows == 0 || cols == 0) return ok();
    if (!dy_bf16 || !token_rows_dev || !token_weights_dev || !q || !s)
        return fail(MXFP8_ERR_INVALID_ARG, "dy, token_rows, token_weights, q or s is NULL");
    if (cols % 32) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "cols %% 32 != 0 (cols=%lld)", (long long)cols);
    if (cols > (int64_t{1} << 30)) return fail(MXFP8_ERR_UNSUPPORTED_SHAPE, "cols > 2^30 (cols=%lld)", (long long)cols);
    if (ld < cols) return fail(MXFP8_ERR_INVALID_ARG, "ld < cols");
    if (ld % 8 || !aligned16(dy_bf16) || !aligned16(q) || !aligned16(s))
        return fail(MXFP8_ERR_MISALIGNED, "pointer or ld not 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(token_rows_dev) | reinterpret_cast<uintptr_t>(token_weights_dev)) & 3u)
        return fail(MXFP8_ERR_MISALIGNED, "token_rows or token_weights not 4-byte aligned");
    WeightedTokensArgs a{};
    a.dy = static_cast<const uint16_t*>(dy_bf16);
    a.tokens = tokens;
    a.ld = ld;
    a.k = k;
    a.token_rows = token_rows_dev;
    a.token_weights = token_weights_dev;
    a.rows = rows;
    a.cols = cols;
    a.offsets = group_offsets_dev;
    a.groups = groups;
    a.flags = flags;
    a.q = static_cast<uint8_t*>(q);
    a.s = static_cast<uint8_t*>(s);
    a.scale_bytes = group_offsets_dev ? mxfp8_grouped_scale_bytes(rows, cols, groups)
                                      : mxfp8_scale_bytes(rows, cols);
    return cuda_result(launch_weighted_quantize_tokens_mx(a, reinterpret_cast<cudaStream_t>(stream)),
                       "fp8_route_weight_quantize_mx_tokens launch");
}

mxfp8_status mxfp8_last_device_status(mxfp8_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(MXFP8_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
    unsigned q = 0, g = 0, fu = 0;
    if ((e = take_status_quant(&q)) != cudaSuccess || (e = take_status_gemm(&g)) != cudaSuccess ||
        (e = take_status_fused(&fu)) != cudaSuccess)
        return fail(MXFP8_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    const unsigned st = q ? q : (g ? g : fu);
    if (st) return fail(static_cast<mxfp8_status>(st), "device reported %s",
                        mxfp8_status_string(static_cast<mxfp8_status>(st)));
    return ok();
}

const char* mxfp8_status_string(mxfp8_status s) {
    switch (s) {
        case MXFP8_OK: return "ok";
        case MXFP8_ERR_INVALID_ARG: return "invalid argument";
        case MXFP8_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MXFP8_ERR_MISALIGNED: return "misaligned pointer or stride";
        case MXFP8_ERR_CUDA: return "CUDA error";
        case MXFP8_ERR_DEVICE_CHECK: return "device-side check failed";
        case MXFP8_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

const char* mxfp8_last_error(void) { return g_err; }

void mxfp8_set_wait_limit_ns(uint64_t ns) { g_wait_limit.store(ns ? ns : 2000000000ull); }

mxfp8_status mxfp8_debug_swiglu_f32(const void* g_bf16, const void* u_bf16, int64_t n, float* y,
                                    mxfp8_stream_t stream) {
    if (n < 0) return fail(MXFP8_ERR_INVALID_ARG, "negative size");
    if (n == 0) return ok();
    if (!g_bf16 || !u_bf16 || !y) return fail(MXFP8_ERR_INVALID_ARG, "NULL pointer");
    return cuda_result(launch_debug_swiglu_f32(static_cast<const uint16_t*>(g_bf16),
                                               static_cast<const uint16_t*>(u_bf16), n, y,
                                               reinterpret_cast<cudaStream_t>(stream)),
                       "mxfp8_debug_swiglu_f32 launch");
}

void mxfp8_debug_inject_wait_timeout(int enable) { g_inject.store(enable ? 1 : 0); }

}  // extern "C"
