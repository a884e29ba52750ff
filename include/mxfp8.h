/*
 * mxfp8.h - C ABI of the GB300 (sm_103a) MXFP8 / per-tensor FP8 library.
 *
 * The library turns BF16 operands into FP8 payloads plus scales and runs the
 * scaled GEMMs that consume them, all as hand-written CUDA kernels launched
 * on the caller's stream.
 *
 * Conventions shared by every entry point
 *  - Pointers named *_dev or documented as device pointers are CUDA device
 *    memory owned and allocated by the caller.  The library allocates
 *    nothing, frees nothing and keeps no reference after the call returns.
 *  - Work is stream ordered on `stream` (NULL = the legacy default stream).
 *    Calls never synchronize, except mxfp8_last_device_status().  A call
 *    issues only kernel launches and memsets on `stream`, so a sequence of
 *    calls can be captured into a CUDA graph and replayed; make each kind
 *    of call once on the device before capturing it (its first use sets
 *    kernel attributes and caches occupancy queries).  Calls on different
 *    streams may run concurrently when they share no output buffer (and,
 *    for the entry points that take one, no workspace or history state).
 *  - Kernels use programmatic dependent launch: the GEMMs and most
 *    quantizers are launched with programmatic stream serialization, so
 *    they may start while the kernel before them on the stream finishes,
 *    and each waits for that kernel's completion (griddepcontrol.wait)
 *    before touching global memory; every kernel signals early launch of
 *    the kernel after it.  A kernel of the caller's own that follows a call
 *    and is itself launched with programmatic stream serialization must
 *    therefore wait (cudaGridDependencySynchronize) before reading the
 *    call's outputs, as programmatic dependent launch always requires;
 *    kernels launched without that attribute are unaffected.
 *  - Errors the host can see (null pointers, bad shapes, misaligned pointers
 *    or strides) are returned at once and launch nothing.  Errors only the
 *    device can see (inconsistent group offsets, a wait that exceeded its
 *    time limit) are recorded in a per-device status word that
 *    mxfp8_last_device_status() reads; the kernels never trap.
 *  - BF16 matrices are row-major with a leading dimension in elements.
 *    "Alignment" below means the byte address is a multiple of 16.
 *  - A GEMM computes C = A . B^T with A M x K and B N x K, both K-major
 *    (the 32-value scale blocks run along K).  The forward, dgrad and wgrad
 *    products of a linear layer (Y = X W^T, dX = dY W, dW = dY^T X) are all
 *    expressed this way by quantizing each operand in the orientation whose
 *    blocks run along that product's reduction axis ("Olmo-core MoE report,
 *    Section 11: MXFP8 Training", Section 11.3.2, Eq. 60).
 *
 * Swizzled scale layout ("Olmo-core MoE report", Section 11.2.1, Figure 52):
 *  the E8M0 scales of a rows x k operand (one per row and 32-value K-block j)
 *  are stored in 512-byte tiles of 128 rows x 4 K-blocks; tile (r/128, j/4)
 *  sits at byte ((r/128) * ceil(k/128) + j/4) * 512 and inside it scale (r, j)
 *  sits at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4).  This is the
 *  order in which the tensor cores read block scales.  Padding rows and
 *  blocks hold 0.  Size: mxfp8_scale_bytes(rows, k).
 */
#ifndef MXFP8_H
#define MXFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* mxfp8_stream_t;

typedef enum {
    MXFP8_OK = 0,
    MXFP8_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum  */
    MXFP8_ERR_UNSUPPORTED_SHAPE = 2, /* divisibility or size limit violated   */
    MXFP8_ERR_MISALIGNED = 3,        /* pointer or stride not 16-byte aligned */
    MXFP8_ERR_CUDA = 4,              /* a CUDA runtime / driver call failed   */
    MXFP8_ERR_DEVICE_CHECK = 5,      /* device-side validation failed         */
    MXFP8_ERR_TIMEOUT = 6            /* a device wait exceeded its time limit */
} mxfp8_status;

/* fp8_quantize_mx flags.  Scale rule default: rceil. */
enum {
    MX_ROWWISE = 1,     /* blocks along cols; q_row is rows x cols           */
    MX_COLWISE = 2,     /* blocks along rows; q_col is cols x rows (= X^T)    */
    MX_SCALE_FLOOR = 4  /* OCP v1.0 floor rule instead of rceil               */
};

/* FP8 payload formats. */
enum { FP8_E4M3 = 0, FP8_E5M2 = 1 };

/* fp8_scaled_gemm modes. */
enum { GEMM_MX = 0, GEMM_TENSOR = 1 };

/* Bytes of the swizzled E8M0 scale array of a rows x k operand whose blocks
 * run along k: ceil(rows/128) * ceil(k/128) * 512.  Returns 0 for
 * non-positive sizes.  ("Olmo-core MoE report", Section 11.2.1, Figure 52.) */
size_t mxfp8_scale_bytes(int64_t rows, int64_t k);

/* Upper bound on the bytes of a grouped scale array (see
 * fp8_quantize_mx_grouped): (ceil(total_rows/128) + groups) * ceil(k/128) * 512. */
size_t mxfp8_grouped_scale_bytes(int64_t total_rows, int64_t k, int32_t groups);

/*
 * fp8_quantize_mx - MXFP8 quantization of a BF16 matrix.
 * ("Olmo-core MoE report", Section 11.2.1 Eq. 58 and Figure 50; scale rule
 *  Section 11.3.5 / Table 24; one read emits both orientations, Section
 *  11.1.4 and Figure 55.)
 *
 * Each 32-value block gets the E8M0 scale s = 2^e chosen from its largest
 * magnitude amax:
 *   rceil (default): the smallest e with amax <= 448 * 2^e;
 *   MX_SCALE_FLOOR:  e = floor(log2 amax) - 8 (may saturate);
 * e is clamped to [-127, 127] (an all-zero block gets byte 0); the payload is
 * q = E4M3(x / s), round-to-nearest-even, saturating at +-448, zero keeps its
 * sign.  A block holding NaN or Inf gets scale byte 0xFF and payload 0x7F.
 *
 *  x_bf16  device, rows x cols BF16, leading dimension ld (elements).
 *  flags   MX_ROWWISE and/or MX_COLWISE, optionally MX_SCALE_FLOOR.
 *  q_row   device, rows x cols bytes (row stride cols), when MX_ROWWISE.
 *  s_row   device, mxfp8_scale_bytes(rows, cols) bytes, when MX_ROWWISE.
 *  q_col   device, cols x rows bytes (row stride rows), when MX_COLWISE.
 *  s_col   device, mxfp8_scale_bytes(cols, rows) bytes, when MX_COLWISE.
 * Requirements: cols % 32 == 0; rows % 32 == 0 when MX_COLWISE; ld >= cols
 * and ld % 8 == 0; every pointer 16-byte aligned.  Unused outputs may be NULL.
 * Every byte of the scale arrays is written (padding = 0).
 */
mxfp8_status fp8_quantize_mx(const void* x_bf16, int64_t rows, int64_t cols, int64_t ld,
                             unsigned flags, void* q_row, void* s_row, void* q_col,
                             void* s_col, mxfp8_stream_t stream);

/*
 * fp8_quantize_mx_batch - fp8_quantize_mx for up to 16 tensors with as few
 * launches as possible (a linear layer's activation and weight rowwise for
 * the forward GEMM, or the backward's dY both ways and W and X colwise:
 * "Olmo-core MoE report, Section 11: MXFP8 Training", Section 11.3.2, Eq. 60).
 * Each tensor gets exactly what fp8_quantize_mx(x[t], rows[t], cols[t],
 * ld[t], flags[t], ...) gives it.  Rowwise-only tensors share one launch;
 * tensors with MX_COLWISE share one launch per 8.
 *
 *  count                  1 .. 16.
 *  x_bf16                 HOST array of count DEVICE pointers to the BF16
 *                         inputs (row stride ld[t] elements), 16-byte aligned.
 *  rows, cols, ld, flags  HOST arrays of count values, with fp8_quantize_mx's
 *                         rules per tensor; MX_SCALE_FLOOR must be the same for
 *                         every non-empty tensor.  A tensor with no rows or no
 *                         columns is skipped (its pointers unused).
 *  q_row, s_row           HOST arrays of count DEVICE pointers (rowwise
 *                         outputs of the tensors whose flags have MX_ROWWISE;
 *                         the arrays may be NULL when none has).
 *  q_col, s_col           the same for MX_COLWISE.
 */
mxfp8_status fp8_quantize_mx_batch(int32_t count, const void* const* x_bf16, const int64_t* rows,
                                   const int64_t* cols, const int64_t* ld, const unsigned* flags,
                                   void* const* q_row, void* const* s_row, void* const* q_col,
                                   void* const* s_col, mxfp8_stream_t stream);

/*
 * fp8_quantize_mx_grouped - rowwise MXFP8 quantization of an expert-dispatched
 * matrix whose rows are sorted by expert ("Olmo-core MoE report", Section
 * 11.4.1: dispatch places each token row's qdata and scales in its expert's
 * buffer).
 *
 * Group g owns rows [off[g], off[g+1]) of x.  Payload rows keep their
 * positions (q is total_rows x cols).  Scales: each group is padded to a
 * multiple of 128 rows, and group g's scales occupy rows
 * P_g .. P_g + m_g - 1 of one swizzled array, P_g = sum_{h<g} ceil(m_h/128)*128;
 * its padding rows are written as 0.  Bytes past the last padded group are
 * not written.
 *
 *  group_offsets_dev  device, groups + 1 int32, off[0] = 0, non-decreasing,
 *                     off[groups] = total_rows.  Checked on the device: a
 *                     violation records MXFP8_ERR_DEVICE_CHECK and writes nothing.
 *  s                  device, at least
 *                     mxfp8_grouped_scale_bytes(total_rows, cols, groups) bytes.
 * flags may hold MX_SCALE_FLOOR (MX_ROWWISE is implied).  1 <= groups <= 1024.
 * Other requirements as fp8_quantize_mx.
 */
mxfp8_status fp8_quantize_mx_grouped(const void* x_bf16, int64_t total_rows, int64_t cols,
                                     int64_t ld, const int32_t* group_offsets_dev,
                                     int32_t groups, unsigned flags, void* q, void* s,
                                     mxfp8_stream_t stream);

/*
 * fp8_quantize_tensor - per-tensor current-scaling FP8 quantization.
 * ("3.8 Mixed Precision, bf16 & FP8 Training", "Per-tensor scaling and the
 *  delayed-scaling recipe" and exercise 6; "FP8-LM: Training FP8 Large
 *  Language Models", Section 3.4 tensor scaling.)
 *
 *   amax = max |x|;  s = fp32(fmax / max(amax, 1e-12));  q = FP8(fp32(x * s))
 * with fmax = 448 (FP8_E4M3) or 57344 (FP8_E5M2, gradient operands), the FP8
 * cast round-to-nearest-even and saturating.  x ~ q / s.
 *
 *  x_bf16     device, n BF16 values, 16-byte aligned.
 *  amax_dev   device fp32 scalar, written (overwritten: not accumulated).
 *  scale_dev  device fp32 scalar s, written.
 *  q          device, n bytes, 16-byte aligned.
 *  workspace  NULL: two kernels (amax reduction, then the cast).  Otherwise
 *             device scratch of mxfp8_tensor_workspace_bytes() bytes, 16-byte
 *             aligned, owned by the caller: one cooperative kernel reduces the
 *             amax, meets at a grid barrier kept in the workspace, and casts
 *             (the library zeroes the workspace on the stream first).  Calls
 *             sharing one workspace must not overlap on the GPU.
 * n == 0 writes amax = 0 and s = fmax / 1e-12.
 */
mxfp8_status fp8_quantize_tensor(const void* x_bf16, int64_t n, int fmt, float* amax_dev,
                                 float* scale_dev, void* q, void* workspace,
                                 mxfp8_stream_t stream);

/* Bytes of device scratch fp8_quantize_tensor takes as its workspace. */
size_t mxfp8_tensor_workspace_bytes(void);

/*
 * fp8_quantize_tensor_noalloc - fp8_quantize_tensor's single-launch path for
 * callers that cannot allocate device memory.  The pages have no counterpart
 * to this entry point; it exists for the library's users.
 *
 * Some callers cannot call cudaMalloc (or any allocating routine) at the
 * point where they quantize: code running inside a host application that
 * owns every device allocation, or hot loops that are forbidden to allocate
 * after start-up.  Those callers still pass x, q, amax_dev and scale_dev, but
 * no workspace: the scratch comes from a static 256-byte device array inside
 * the library, which every GPU that loads the library holds until the
 * process exits.
 *
 * Results are identical to fp8_quantize_tensor (same kernel, same rule).
 * The scratch this path needs does not grow with n (it is
 * mxfp8_tensor_workspace_bytes()); a need larger than the static array would
 * be rejected with MXFP8_ERR_UNSUPPORTED_SHAPE before anything runs.
 * The path uses 68 bytes of the array (one amax word and a grid-barrier
 * counter, sized for the batched kernel's 16 tensors).
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it for the life of the process; make that
 * first call before any stream capture.  The address belongs to the device's
 * context at that moment: after a cudaDeviceReset, or any other teardown of
 * that context, do not call this entry point again in the same process.
 * All calls on a device share the array and each clears the words it needs
 * on its stream first: calls that overlap on the GPU (e.g. on two streams)
 * race and must not be issued.  Allocates nothing (no cudaMalloc, cudaFree
 * or allocating library routine).
 */
mxfp8_status fp8_quantize_tensor_noalloc(const void* x_bf16, int64_t n, int fmt,
                                         float* amax_dev, float* scale_dev, void* q,
                                         mxfp8_stream_t stream);

/*
 * fp8_scaled_gemm - C = A . B^T with FP32 accumulation and a BF16 epilogue
 * (round to nearest even).
 * ("Olmo-core MoE report", Section 11.1.1: block-scaled tcgen05.mma with an
 *  epilogue converting the accumulator to BF16; "3.8 Mixed Precision, bf16 &
 *  FP8 Training", exercise 6: per-tensor GEMM de-scaled by 1 / (s_x s_w).)
 *
 * GEMM_MX:     a, b E4M3 payloads (a_fmt = b_fmt = FP8_E4M3); a_scale, b_scale
 *              device swizzled E8M0 arrays of mxfp8_scale_bytes(M, K) and
 *              mxfp8_scale_bytes(N, K) bytes, as written by fp8_quantize_mx.
 *              C[m,n] = bf16( sum_k s_a[m,k/32] q_a[m,k] * s_b[n,k/32] q_b[n,k] ).
 *              K % 32 == 0.
 * GEMM_TENSOR: a, b payloads in a_fmt / b_fmt (E4M3 or E5M2); a_scale, b_scale
 *              device fp32 scalars s_a, s_b as written by fp8_quantize_tensor.
 *              C[m,n] = bf16( (sum_k q_a[m,k] q_b[n,k]) / (s_a s_b) ).  K % 16 == 0.
 *
 *  a   device, M x K bytes (row stride K);  b  device, N x K bytes.
 *  c   device BF16, M x N with leading dimension ldc (elements).
 * Requirements: N % 8 == 0, ldc >= N, ldc % 8 == 0, all pointers 16-byte
 * aligned.  M, N may be 0 (no work); K == 0 writes C = 0.
 */
mxfp8_status fp8_scaled_gemm(int mode, int a_fmt, int b_fmt, const void* a,
                             const void* a_scale, const void* b, const void* b_scale,
                             int64_t M, int64_t N, int64_t K, void* c_bf16, int64_t ldc,
                             mxfp8_stream_t stream);

/*
 * fp8_scaled_gemm_pair - two independent fp8_scaled_gemm calls of one mode in
 * one launch, e.g. the two products of a linear layer's backward: dgrad
 * dX = dY . W and wgrad dW = dY^T . X ("Olmo-core MoE report", Section
 * 11.3.2, Eq. 60, with the operands quantized in the orientation each GEMM
 * consumes).
 *
 * Problem i (i = 0, 1) takes a_fmt_i, b_fmt_i, a_i, a_scale_i, b_i,
 * b_scale_i, M_i, N_i, K_i, c_i, ldc_i with exactly the meaning, layout,
 * requirements and result of fp8_scaled_gemm's arguments: each C_i is
 * bit-identical to what fp8_scaled_gemm writes (the same dot products in the
 * same K order).  The persistent kernel gives each problem its own share of
 * the SMs' CTA pairs, chosen on the host so that both finish together, which
 * fills the partial last waves two separate launches would each leave.  If
 * either problem has M, N or K == 0, the two are run as separate calls.
 * Argument errors of either problem return before anything is launched.
 * C_0 and C_1 must not overlap.
 */
mxfp8_status fp8_scaled_gemm_pair(int mode, int a_fmt0, int b_fmt0, const void* a0,
                                  const void* a_scale0, const void* b0, const void* b_scale0,
                                  int64_t M0, int64_t N0, int64_t K0, void* c0_bf16, int64_t ldc0,
                                  int a_fmt1, int b_fmt1, const void* a1, const void* a_scale1,
                                  const void* b1, const void* b_scale1, int64_t M1, int64_t N1,
                                  int64_t K1, void* c1_bf16, int64_t ldc1, mxfp8_stream_t stream);

/*
 * fp8_grouped_gemm - per-expert MXFP8 GEMM over ragged, row-sorted groups.
 * ("Olmo-core MoE report", Section 11.1.1 and 11.4.1: the grouped expert
 *  GEMMs consume the dispatched activation and the cached expert weights.)
 *
 * For each group g with rows [off[g], off[g+1]):
 *   C[off[g]:off[g+1], :] = MX-GEMM(A[off[g]:off[g+1], :], W_g)
 *
 *  a        device, total_rows x K E4M3 payload (row stride K).
 *  a_scale  device, grouped swizzled scales as written by
 *           fp8_quantize_mx_grouped with the same offsets.
 *  b        device, groups x N x K E4M3 payload (expert g at b + g*N*K).
 *  b_scale  device, groups consecutive swizzled arrays of
 *           mxfp8_scale_bytes(N, K) bytes (expert g's at g times that size);
 *           equivalently fp8_quantize_mx of the (groups*N) x K stack when
 *           N % 128 == 0.
 *  group_offsets_dev  as in fp8_quantize_mx_grouped; a violation records
 *           MXFP8_ERR_DEVICE_CHECK and no output is written.
 *  c        device BF16, total_rows x N, leading dimension ldc.
 * Requirements: 1 <= groups <= 1024, K % 32 == 0, N % 8 == 0, ldc % 8 == 0,
 * pointers 16-byte aligned.  Empty groups are allowed.
 */
mxfp8_status fp8_grouped_gemm(const void* a, const void* a_scale, const void* b,
                              const void* b_scale, const int32_t* group_offsets_dev,
                              int32_t groups, int64_t total_rows, int64_t N, int64_t K,
                              void* c_bf16, int64_t ldc, mxfp8_stream_t stream);

/*
 * fp8_quantize_tensor_batch - fp8_quantize_tensor for `count` tensors in one
 * cooperative launch with one grid barrier (a linear layer's activation and
 * weight, say; "3.8 Mixed Precision, bf16 & FP8 Training", exercise 6 casts
 * both operands before the FP8 matmul).  Each tensor t gets its own amax,
 * scale and payload exactly as fp8_quantize_tensor computes them.
 *
 *  count            1 .. 16.
 *  x_bf16, n, q     HOST arrays of count entries: device pointers to the
 *                   BF16 inputs and payload outputs (16-byte aligned) and the
 *                   element counts (n[t] == 0 allowed).
 *  amax_dev         device fp32[count], written.
 *  scale_dev        device fp32[count], written.
 *  workspace        device scratch of mxfp8_tensor_workspace_bytes() bytes,
 *                   16-byte aligned (zeroed by the library on the stream);
 *                   calls sharing one workspace must not overlap on the GPU.
 */
mxfp8_status fp8_quantize_tensor_batch(int32_t count, const void* const* x_bf16, const int64_t* n,
                                       int fmt, float* amax_dev, float* scale_dev, void* const* q,
                                       void* workspace, mxfp8_stream_t stream);

/*
 * fp8_quantize_tensor_scaled - per-tensor FP8 cast with a scale the caller
 * already holds on the device ("3.8 Mixed Precision, bf16 & FP8 Training",
 * "Per-tensor scaling and the delayed-scaling recipe": the cast uses a scale
 * chosen before this tensor's amax is known; "FP8-LM: Training FP8 Large
 * Language Models", Section 2.1 Eq. 3: the gradient cast g' = mu g is the
 * case s = mu).
 *
 *   q = FP8(fp32(x * s)), round-to-nearest-even, saturating at +-fmax.
 *
 *  scale_dev      device fp32 scalar s (read).
 *  amax_dev       device fp32 scalar, written: max |x| (NaN if any x is NaN).
 *  sat_count_dev  device uint64, written: how many payloads are the largest
 *                 finite code (+-448 / +-57344) - FP8-LM's overflow count.
 *  x_bf16, q      n values, 16-byte aligned.  n == 0 writes amax = 0, count 0.
 */
mxfp8_status fp8_quantize_tensor_scaled(const void* x_bf16, int64_t n, int fmt,
                                        const float* scale_dev, void* q, float* amax_dev,
                                        uint64_t* sat_count_dev, mxfp8_stream_t stream);

/*
 * fp8_quantize_tensor_delayed - one delayed-scaling cast ("3.8 Mixed
 * Precision", "Per-tensor scaling and the delayed-scaling recipe"): the scale
 * comes from a rolling history of past amax values, the cast runs without
 * waiting for this tensor's amax, and that amax is recorded for later steps.
 *
 *   a = max(history) (NaN propagates), clamped below at 1e-12;
 *   s = fp32(fp32(fmax / a) * margin);  q = FP8(fp32(x * s)) saturating;
 *   history[pos] = max |x|;  pos = (pos + 1) % history_len.
 *
 *  amax_history_dev  device fp32[history_len], read and updated (state the
 *                    caller keeps across steps; all zeros at the start, which
 *                    makes the first cast saturate, as in the recipe).
 *  history_pos_dev   device int32 ring position, read and updated; a value
 *                    outside [0, history_len) records MXFP8_ERR_DEVICE_CHECK
 *                    and restarts the ring at 0.
 *  scale_dev         device fp32, written: the s used.
 *  amax_dev, sat_count_dev  as in fp8_quantize_tensor_scaled.
 * 1 <= history_len <= 65536.  Three kernels on `stream`; calls on one state
 * must be stream ordered.
 */
mxfp8_status fp8_quantize_tensor_delayed(const void* x_bf16, int64_t n, int fmt, float margin,
                                         float* amax_history_dev, int32_t history_len,
                                         int32_t* history_pos_dev, float* scale_dev, void* q,
                                         float* amax_dev, uint64_t* sat_count_dev,
                                         mxfp8_stream_t stream);

/*
 * fp8_requantize_tensor - rescale a per-tensor FP8 payload to another scale
 * ("FP8-LM", Section 2.1, Eq. 4-5: before the gradient all-reduce every rank
 * requantizes to the group's shared scale s'_g = min_i s'_i).
 *
 *   q'' = FP8(fp32(s_out * fp32(decode(q) / s_in))), in that order,
 *         round-to-nearest-even, saturating; fmt_in and fmt_out independent.
 *
 *  scale_in_dev, scale_out_dev  device fp32 scalars (read).
 *  sat_count_dev                device uint64, written: payloads at the
 *                               largest finite code of fmt_out.
 *  q_in, q_out                  n bytes, 16-byte aligned; may not overlap.
 */
mxfp8_status fp8_requantize_tensor(const void* q_in, int64_t n, int fmt_in, const float* scale_in_dev,
                                   const float* scale_out_dev, int fmt_out, void* q_out,
                                   uint64_t* sat_count_dev, mxfp8_stream_t stream);

/*
 * Routed-path kernels around the quantizer ("Olmo-core MoE report", Section
 * 11.4.1 and Table 25).  Each takes optional group offsets: NULL with
 * groups == 0 gives the plain rows x cols layout of fp8_quantize_mx's rowwise
 * output; a device array of groups + 1 int32 (1 <= groups <= 1024, rows <
 * 2^31, same rules and device check as fp8_quantize_mx_grouped) gives that
 * entry point's group-padded scale layout.
 */

/*
 * fp8_dequantize_mx - BF16 x^ = s q of a rowwise MXFP8 operand ("Olmo-core
 * MoE report", Section 11.2.1 Eq. 58; used where a saved MXFP8 activation
 * meets a BF16 consumer, Section 11.4.3, and for the routed Wgrad operands,
 * Section 11.4.1).  A colwise output (q_col, s_col) is itself a rowwise
 * operand of the transpose and dequantizes to X^T.
 *
 *  q        device, rows x cols E4M3 bytes (row stride cols).
 *  s        device, its scales (mxfp8_scale_bytes(rows, cols), or the
 *           group-padded array when offsets are given).
 *  out_bf16 device, rows x cols BF16 with leading dimension ldo (>= cols).
 * out[r][c] = bf16_RNE(E4M3(q[r][c]) * 2^(byte - 127)), the product being
 * exact before that one rounding (overflow gives Inf; an E4M3 NaN code or
 * scale byte 0xFF gives NaN).  Requirements: cols % 32 == 0, ldo % 8 == 0,
 * every pointer 16-byte aligned.
 */
mxfp8_status fp8_dequantize_mx(const void* q, const void* s, int64_t rows, int64_t cols,
                               const int32_t* group_offsets_dev, int32_t groups, void* out_bf16,
                               int64_t ldo, mxfp8_stream_t stream);

/*
 * fp8_swiglu_quantize_mx - SwiGLU of the up/gate GEMM output, MXFP8-quantized
 * rowwise in the same pass ("Olmo-core MoE report", Section 11.4.1: the fused
 * SwiGLU-plus-quantization step that feeds the down projection; Table 25).
 *
 *  h_bf16  device, rows x 2f BF16 (leading dimension ld >= 2f): gate in
 *          columns [0, f), up in columns [f, 2f).
 *  q, s    outputs as fp8_quantize_mx's rowwise ones for a rows x f operand
 *          (or the group-padded scale array).
 * The hidden value a = bf16_RNE(g * sigma(g) * u), sigma(g) = 1/(1+e^-g), is
 * what an unfused SwiGLU would store in BF16; it is formed in fp32 within
 * 7.5 * 2^-24 relative of the exact value (in double, rounded once, for
 * g < -80), so a is the correctly rounded BF16 value except within that
 * distance of a rounding midpoint, where it may be the neighbour.  a is then quantized by the MX rule
 * of fp8_quantize_mx (flags: MX_SCALE_FLOOR optional, rowwise implied) and
 * never written.  Requirements: f % 32 == 0, ld % 8 == 0, pointers 16-byte
 * aligned.
 */
mxfp8_status fp8_swiglu_quantize_mx(const void* h_bf16, int64_t rows, int64_t f, int64_t ld,
                                    const int32_t* group_offsets_dev, int32_t groups,
                                    unsigned flags, void* q, void* s, mxfp8_stream_t stream);

/*
 * fp8_route_weight_quantize_mx - combine backward: the route-weighted output
 * gradient of every dispatched row, MXFP8-quantized rowwise in the same pass
 * ("Olmo-core MoE report", Section 11.4.1: combine backward applies the route
 * weights while quantizing the output gradient; Table 25).
 *
 *  dy_bf16         device, tokens x cols BF16 output gradient, leading
 *                  dimension ld (>= cols).
 *  row_token_dev   device, rows int32: the token each dispatched row came
 *                  from.  An index outside [0, tokens) records
 *                  MXFP8_ERR_DEVICE_CHECK; that row is quantized as zeros.
 *  row_weight_dev  device, rows fp32 route weights.
 *  q, s            rowwise outputs for the rows x cols dispatched gradient
 *                  (or the group-padded scale array).
 * Row i is g_i = bf16_RNE(w_i * dy[row_token[i]]), rounded once from the exact
 * product, then quantized by the MX rule (MX_SCALE_FLOOR optional).  The
 * route-expanded BF16 gradient is never written.  Requirements: cols % 32 ==
 * 0, ld % 8 == 0, dy/q/s 16-byte aligned, row_token/row_weight 4-byte aligned.
 */
mxfp8_status fp8_route_weight_quantize_mx(const void* dy_bf16, int64_t tokens, int64_t ld,
                                          const int32_t* row_token_dev,
                                          const float* row_weight_dev, int64_t rows,
                                          int64_t cols, const int32_t* group_offsets_dev,
                                          int32_t groups, unsigned flags, void* q, void* s,
                                          mxfp8_stream_t stream);

/*
 * fp8_route_weight_quantize_mx_tokens - fp8_route_weight_quantize_mx with the
 * routing given per token: each token's gradient row is read once and its k
 * route-weighted copies are quantized into their dispatched rows ("Olmo-core
 * MoE report", Section 11.4.1 and Table 25, route weighting + gradient Q in
 * combine backward).
 *
 *  dy_bf16            device, tokens x cols BF16, leading dimension ld.
 *  k                  routes per token, 1..16.
 *  token_rows_dev     device, tokens x k int32: the dispatched row of each of
 *                     the token's routes (-1: no route in that slot).  A row
 *                     >= rows records MXFP8_ERR_DEVICE_CHECK and is skipped.
 *  token_weights_dev  device, tokens x k fp32 route weights.
 *  rows, cols, group_offsets_dev, groups, flags, q, s: as in
 *                     fp8_route_weight_quantize_mx (s holds
 *                     mxfp8_scale_bytes(rows, cols) or, with offsets,
 *                     mxfp8_grouped_scale_bytes(rows, cols, groups) bytes).
 * Dispatched row i = (token t, slot j) with token_rows[t k + j] = i gets
 * bf16_RNE(token_weights[t k + j] * dy[t]), rounded once from the exact
 * product, MX-quantized rowwise: the same bytes as
 * fp8_route_weight_quantize_mx with row_token[i] = t and row_weight[i] equal
 * to that weight.  Every row in [0, rows) must be some token's route
 * exactly once: a row no token names keeps its previous payload and gets
 * zero scale bytes (the scale array is zeroed first, so padding reads 0).
 * Requirements as fp8_route_weight_quantize_mx; groups <= 1024 and
 * cols <= 2^30 (else MXFP8_ERR_UNSUPPORTED_SHAPE).
 */
mxfp8_status fp8_route_weight_quantize_mx_tokens(const void* dy_bf16, int64_t tokens, int64_t ld,
                                                 int32_t k, const int32_t* token_rows_dev,
                                                 const float* token_weights_dev, int64_t rows,
                                                 int64_t cols, const int32_t* group_offsets_dev,
                                                 int32_t groups, unsigned flags, void* q, void* s,
                                                 mxfp8_stream_t stream);

/*
 * mxfp8_last_device_status - synchronize `stream`, then return and clear the
 * device status word of the current device: MXFP8_OK, MXFP8_ERR_DEVICE_CHECK
 * or MXFP8_ERR_TIMEOUT (the first one recorded since the last call), or
 * MXFP8_ERR_CUDA if the synchronization itself failed.
 */
mxfp8_status mxfp8_last_device_status(mxfp8_stream_t stream);

/* Static English text for a status code. */
const char* mxfp8_status_string(mxfp8_status status);

/* Detail of the most recent error returned on the calling thread ("" if none). */
const char* mxfp8_last_error(void);

/*
 * Test hook: the time limit, in nanoseconds, after which a device-side wait
 * gives up, records MXFP8_ERR_TIMEOUT and lets the kernel exit (default
 * 2e9).  0 restores the default.  Affects launches issued after the call.
 */
void mxfp8_set_wait_limit_ns(uint64_t ns);

/*
 * Test hook: when nonzero, the next GEMM launch makes its MMA-issuing thread
 * wait on a barrier that nothing signals, so the wait runs out after the
 * limit above and the kernel exits with MXFP8_ERR_TIMEOUT recorded.  The hook
 * resets itself after one launch.
 */
void mxfp8_debug_inject_wait_timeout(int enable);

/*
 * Test hook: y[i] = the fp32 value g[i] sigma(g[i]) u[i] that
 * fp8_swiglu_quantize_mx forms on its fast path (gates >= -80), before the
 * BF16 rounding, so its error bound can be checked.  g, u: device BF16[n];
 * y: device fp32[n].  The fast path runs two values at a time in packed
 * FP32; each value is also formed one at a time (as the per-block redo
 * does), and a difference in bits other than two NaNs records
 * MXFP8_ERR_DEVICE_CHECK for mxfp8_last_device_status().
 */
mxfp8_status mxfp8_debug_swiglu_f32(const void* g_bf16, const void* u_bf16, int64_t n, float* y,
                                    mxfp8_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP8_H */
