// Scaled FP8 GEMMs on the sm_103a tensor cores: C = A . B^T, both operands
// K-major, FP32 accumulation in tensor memory, BF16 (RNE) epilogue.
//
//   GEMM_MX      tcgen05.mma kind::mxf8f6f4 block_scale: one E8M0 scale per
//                32 K-values of each row of A and B, read by the tensor core
//                from TMEM ("Olmo-core MoE report, Section 11: MXFP8
//                Training", Section 11.1.1 and 11.2.3).
//   GEMM_TENSOR  tcgen05.mma kind::f8f6f4 on per-tensor scaled E4M3/E5M2
//                payloads; the epilogue multiplies by 1 / (s_a s_b) ("3.8
//                Mixed Precision, bf16 & FP8 Training", exercise 6).
//   grouped      the MX GEMM over ragged, row-sorted expert groups, expert g
//                using its own weight ("Olmo-core MoE report", Section 11.4.1).
//
// Structure: a persistent kernel, one CTA per SM, 128 x 256 output tiles.
//   warp 0       TMA producer: 128 x 128 A box + 256 x 128 B box (128-byte
//                swizzle) and the 512-byte scale tiles per K step, into a
//                4-stage shared-memory ring guarded by mbarriers.
//   warp 1       TMEM allocator and MMA issuer: tcgen05.cp of the block scales
//                into TMEM, 4 MMAs of K = 32 per stage, tcgen05.commit frees the
//                stage and, after the last K step, hands the accumulator over.
//   warps 2-9    epilogue: tcgen05.ld of the 128 x 256 FP32 accumulator (each
//                warp one 32-lane quarter x 128 columns), release TMEM, convert
//                to BF16 and store, overlapping the next tile's main loop.
// Every wait is bounded; a wait that runs out records MXFP8_ERR_TIMEOUT,
// the CTA drains its outstanding copies and MMAs, frees TMEM and exits.
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp8 {

__device__ unsigned int g_status_gemm = 0;

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // bytes = FP8 elements per K step (one 128-byte swizzle row)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int SFA_BYTES = 512;   // one 128-row x 4-block scale tile
constexpr int SFB_BYTES = 1024;  // two of them (256 rows)
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr int MAX_GROUPS = 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = BN;        // 128 lanes x 256 FP32 columns
constexpr uint32_t SF_COLS_PER_STAGE = 12;  // A: 4 columns, B: 8 columns

// Shared memory map (offsets from a 1024-byte aligned base).
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
constexpr uint32_t OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
constexpr uint32_t NUM_BARS = 2 * STAGES + 4;  // full, empty, tmem_full, tmem_empty, drain, never
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_PREFIX = OFF_MISC + 32;
constexpr uint32_t SMEM_PLAIN = OFF_PREFIX;
constexpr uint32_t SMEM_GROUPED = OFF_PREFIX + 2 * (MAX_GROUPS + 1) * 4;

static_assert(OFF_B % 1024 == 0 && OFF_SFA % 1024 == 0, "swizzled tiles need 1024B alignment");
static_assert(ACC_COLS + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");

struct KParams {
    int64_t M, N, K;
    int32_t num_m_tiles, num_n_tiles, num_k_tiles;
    int32_t n_scale_tiles;       // ceil(N / 128): 128-row scale tiles of one B
    const uint8_t* sfa;
    const uint8_t* sfb;
    int64_t sfb_group_stride;    // bytes between experts' B scale arrays
    const float* s_a;            // GEMM_TENSOR scalars
    const float* s_b;
    uint16_t* c;
    int64_t ldc;
    const int32_t* offsets;      // grouped
    int32_t groups;
    uint64_t wait_limit_ns;
    int32_t inject_timeout;
    uint32_t idesc_tensor;
};

struct Tile {
    int64_t a_row;     // first row of A (and of C)
    int64_t row_end;   // rows of C valid below this
    int64_t sfa_tile;  // 128-row tile index in A's scale array
    int64_t b_row;     // first row of B (grouped: of the experts' stack)
    int32_t n_tile;
    int32_t group;
};

__device__ __forceinline__ void record_status(unsigned code) {
    atomicCAS(&g_status_gemm, 0u, code);
}

template <bool GROUPED>
__device__ __forceinline__ Tile decode_tile(const KParams& p, int64_t t, const int32_t* prefix,
                                            const int32_t* offs) {
    Tile tl;
    if constexpr (GROUPED) {
        const int64_t gm = t / p.num_n_tiles;
        tl.n_tile = static_cast<int32_t>(t % p.num_n_tiles);
        int lo = 0, hi = p.groups - 1;  // largest g with prefix[g] <= gm
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= gm) lo = mid; else hi = mid - 1;
        }
        tl.group = lo;
        tl.a_row = offs[lo] + (gm - prefix[lo]) * BM;
        tl.row_end = min(static_cast<int64_t>(offs[lo + 1]), tl.a_row + BM);
        tl.sfa_tile = gm;
        tl.b_row = static_cast<int64_t>(lo) * p.N + static_cast<int64_t>(tl.n_tile) * BN;
    } else {
        const int64_t mt = t % p.num_m_tiles;
        tl.n_tile = static_cast<int32_t>(t / p.num_m_tiles);
        tl.group = 0;
        tl.a_row = mt * BM;
        tl.row_end = min(p.M, tl.a_row + BM);
        tl.sfa_tile = mt;
        tl.b_row = static_cast<int64_t>(tl.n_tile) * BN;
    }
    return tl;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

template <bool MX, bool GROUPED>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const KParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    auto bar = [&](uint32_t i) { return sbase + OFF_BAR + 8 * i; };
    const uint32_t BAR_FULL = 0, BAR_EMPTY = STAGES, BAR_TMEM_FULL = 2 * STAGES,
                   BAR_TMEM_EMPTY = 2 * STAGES + 1, BAR_DRAIN = 2 * STAGES + 2,
                   BAR_NEVER = 2 * STAGES + 3;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + OFF_PREFIX);
    int32_t* offs = prefix + (MAX_GROUPS + 1);
    __shared__ int64_t s_total_tiles;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            mbar_init(bar(BAR_FULL + s), 1);
            mbar_init(bar(BAR_EMPTY + s), 1);
        }
        mbar_init(bar(BAR_TMEM_FULL), 1);
        mbar_init(bar(BAR_TMEM_EMPTY), EPI_WARPS);
        mbar_init(bar(BAR_DRAIN), 1);
        mbar_init(bar(BAR_NEVER), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if constexpr (GROUPED) {
        // Validate the offsets and build the prefix of 128-row tiles per group.
        if (warp == 0) {
            const int G = p.groups;
            bool ok = (p.offsets[0] == 0) && (static_cast<int64_t>(p.offsets[G]) == p.M);
            int32_t base = 0;
            for (int g0 = 0; g0 <= G; g0 += 32) {
                const int g = g0 + lane;
                int32_t tiles = 0;
                if (g <= G) offs[g] = p.offsets[g];
                if (g < G) {
                    const int32_t m = p.offsets[g + 1] - p.offsets[g];
                    if (m < 0) ok = false;
                    tiles = m > 0 ? (m + BM - 1) / BM : 0;
                }
                int32_t incl = tiles;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
                    if (lane >= d) incl += v;
                }
                if (g <= G) prefix[g] = base + incl - tiles;
                base += __shfl_sync(0xffffffffu, incl, 31);
            }
            ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) {
                s_total_tiles = ok ? static_cast<int64_t>(base) * p.num_n_tiles : 0;
                if (!ok && blockIdx.x == 0) record_status(MXFP8_ERR_DEVICE_CHECK);
            }
        }
    } else {
        if (threadIdx.x == 0)
            s_total_tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(misc), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int64_t total = s_total_tiles;

    auto fail = [&]() {
        *abort_flag = 1;
        record_status(MXFP8_ERR_TIMEOUT);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_b);
            uint32_t stage = 0, phase = 0;
            uint32_t issued = 0, issued_parity = 0;  // per-stage bit masks
            bool ok = true;
            for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile tl = decode_tile<GROUPED>(p, t, prefix, offs);
                const uint8_t* sfb_g = p.sfb + static_cast<int64_t>(tl.group) * p.sfb_group_stride;
                const bool two_sfb = (2 * tl.n_tile + 1) < p.n_scale_tiles;
                for (int kt = 0; kt < p.num_k_tiles; ++kt) {
                    if (!mbar_wait(bar(BAR_EMPTY + stage), phase ^ 1u, p.wait_limit_ns, abort_flag)) {
                        fail();
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar(BAR_FULL + stage);
                    uint32_t bytes = A_BYTES + B_BYTES;
                    if constexpr (MX) bytes += SFA_BYTES + (two_sfb ? 1024u : 512u);
                    mbar_arrive_expect_tx(fb, bytes);
                    tma_load_2d(sbase + OFF_A + stage * A_BYTES, &tm_a, fb, kt * BK,
                                static_cast<int32_t>(tl.a_row));
                    tma_load_2d(sbase + OFF_B + stage * B_BYTES, &tm_b, fb, kt * BK,
                                static_cast<int32_t>(tl.b_row));
                    if constexpr (MX) {
                        bulk_load(sbase + OFF_SFA + stage * SFA_BYTES,
                                  p.sfa + (tl.sfa_tile * p.num_k_tiles + kt) * 512, 512, fb);
                        const int64_t nb = 2 * static_cast<int64_t>(tl.n_tile);
                        bulk_load(sbase + OFF_SFB + stage * SFB_BYTES,
                                  sfb_g + (nb * p.num_k_tiles + kt) * 512, 512, fb);
                        if (two_sfb) {
                            bulk_load(sbase + OFF_SFB + stage * SFB_BYTES + 512,
                                      sfb_g + ((nb + 1) * p.num_k_tiles + kt) * 512, 512, fb);
                        }
                    }
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let every copy already in flight land before the CTA exits
                const int never = 0;
                for (uint32_t s = 0; s < STAGES; ++s) {
                    if (issued & (1u << s))
                        mbar_wait(bar(BAR_FULL + s), (issued_parity >> s) & 1u, p.wait_limit_ns,
                                  &never);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const int never = 0;
            bool ok = true;
            if (p.inject_timeout) {
                // test hook: a wait on a barrier nothing signals
                if (!mbar_wait(bar(BAR_NEVER), 0, p.wait_limit_ns, &never)) {
                    fail();
                    ok = false;
                }
            }
            uint32_t stage = 0, phase = 0, acc_phase = 0;
            const uint64_t sf_desc_base = smem_desc(0, 0, 128, SWZ_NONE);
            for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(bar(BAR_TMEM_EMPTY), acc_phase ^ 1u, p.wait_limit_ns, abort_flag)) {
                    fail();
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < p.num_k_tiles; ++kt) {
                    if (!mbar_wait(bar(BAR_FULL + stage), phase, p.wait_limit_ns, abort_flag)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = smem_desc(sbase + OFF_A + stage * A_BYTES, 16, 1024, SWZ_128B);
                    const uint64_t db = smem_desc(sbase + OFF_B + stage * B_BYTES, 16, 1024, SWZ_128B);
                    if constexpr (MX) {
                        const uint32_t sfa_t = tmem + ACC_COLS + stage * SF_COLS_PER_STAGE;
                        const uint32_t sfb_t = sfa_t + 4;
                        const uint32_t sa = sbase + OFF_SFA + stage * SFA_BYTES;
                        const uint32_t sb = sbase + OFF_SFB + stage * SFB_BYTES;
                        tc_cp_32x128b_warpx4(sfa_t, sf_desc_base | ((sa & 0x3FFFFu) >> 4));
                        tc_cp_32x128b_warpx4(sfb_t, sf_desc_base | ((sb & 0x3FFFFu) >> 4));
                        tc_cp_32x128b_warpx4(sfb_t + 4, sf_desc_base | (((sb + 512) & 0x3FFFFu) >> 4));
#pragma unroll
                        for (uint32_t kk = 0; kk < BK / 32; ++kk) {
                            mma_mxf8(tmem, da + 2 * kk, db + 2 * kk, idesc_mxf8(BM, BN, kk), sfa_t,
                                     sfb_t, (kt | kk) != 0);
                        }
                    } else {
#pragma unroll
                        for (uint32_t kk = 0; kk < BK / 32; ++kk) {
                            mma_f8(tmem, da + 2 * kk, db + 2 * kk, p.idesc_tensor, (kt | kk) != 0);
                        }
                    }
                    tc_commit(bar(BAR_EMPTY + stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(bar(BAR_TMEM_FULL));
                acc_phase ^= 1u;
            }
            // every MMA / copy this thread issued completes before teardown
            tc_commit(bar(BAR_DRAIN));
            mbar_wait(bar(BAR_DRAIN), 0, p.wait_limit_ns, &never);
        }
    } else {
        // ------------------------------------------------ epilogue
        const int quarter = warp & 3;        // TMEM lanes this warp may read
        const int half = (warp - 2) >> 2;    // which 128 accumulator columns
        float alpha = 1.0f;
        if constexpr (!MX) alpha = __fdiv_rn(1.0f, *p.s_a) * __fdiv_rn(1.0f, *p.s_b);
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
            const Tile tl = decode_tile<GROUPED>(p, t, prefix, offs);
            if (!mbar_wait(bar(BAR_TMEM_FULL), acc_phase, p.wait_limit_ns, abort_flag)) {
                fail();
                break;
            }
            tc_fence_after();
            uint32_t v[128];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * 128;
            tmem_ld_x32(taddr + 0, v + 0);
            tmem_ld_x32(taddr + 32, v + 32);
            tmem_ld_x32(taddr + 64, v + 64);
            tmem_ld_x32(taddr + 96, v + 96);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_TMEM_EMPTY));
            const int64_t row = tl.a_row + quarter * 32 + lane;
            if (row < tl.row_end) {
                uint16_t* crow = p.c + row * p.ldc;
                const int64_t col0 = static_cast<int64_t>(tl.n_tile) * BN + half * 128;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int64_t col = col0 + j * 8;
                    if (col < p.N) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * alpha,
                                          __uint_as_float(v[8 * j + 1]) * alpha);
                        o.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * alpha,
                                          __uint_as_float(v[8 * j + 3]) * alpha);
                        o.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * alpha,
                                          __uint_as_float(v[8 * j + 5]) * alpha);
                        o.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * alpha,
                                          __uint_as_float(v[8 * j + 7]) * alpha);
                        *reinterpret_cast<uint4*>(crow + col) = o;
                    }
                }
            }
            acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

__global__ void zero_fill_kernel(uint16_t* c, int64_t rows, int64_t cols, int64_t ldc) {
    const int64_t total = rows * cols;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        c[(i / cols) * ldc + (i % cols)] = 0;
    }
}

// ------------------------------------------------------------ host side --

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

// 2D tensor map over a rows x k byte matrix (row stride k), box_rows x 128.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t k, uint32_t box_rows) {
    auto enc = get_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool MX, bool GROUPED>
cudaError_t launch_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const KParams& p,
                          int grid, cudaStream_t s) {
    const uint32_t smem = (GROUPED ? SMEM_GROUPED : SMEM_PLAIN) + 1024;
    auto k = gemm_kernel<MX, GROUPED>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    k<<<grid, THREADS, smem, s>>>(ta, tb, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t s) {
    const bool grouped = g.groups > 0;
    const bool mx = g.mode == GEMM_MX;
    const int64_t b_rows = grouped ? static_cast<int64_t>(g.groups) * g.N : g.N;
    CUtensorMap ta, tb;
    if (!make_map(&ta, g.a, g.M, g.K, BM) || !make_map(&tb, g.b, b_rows, g.K, BN))
        return cudaErrorInvalidValue;
    KParams p{};
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.num_m_tiles = static_cast<int32_t>((g.M + BM - 1) / BM);
    p.num_n_tiles = static_cast<int32_t>((g.N + BN - 1) / BN);
    p.num_k_tiles = static_cast<int32_t>((g.K + BK - 1) / BK);
    p.n_scale_tiles = static_cast<int32_t>((g.N + 127) / 128);
    if (mx) {
        p.sfa = static_cast<const uint8_t*>(g.a_scale);
        p.sfb = static_cast<const uint8_t*>(g.b_scale);
        p.sfb_group_stride = static_cast<int64_t>(p.n_scale_tiles) * p.num_k_tiles * 512;
    } else {
        p.s_a = static_cast<const float*>(g.a_scale);
        p.s_b = static_cast<const float*>(g.b_scale);
        p.idesc_tensor = idesc_f8(BM, BN, static_cast<uint32_t>(g.a_fmt), static_cast<uint32_t>(g.b_fmt));
    }
    p.c = g.c;
    p.ldc = g.ldc;
    p.offsets = g.offsets;
    p.groups = g.groups;
    p.wait_limit_ns = wait_limit_ns();
    p.inject_timeout = take_inject_timeout() ? 1 : 0;
    const int sms = sm_count_current_device();
    int grid;
    if (grouped) {
        grid = sms;
    } else {
        const int64_t tiles = static_cast<int64_t>(p.num_m_tiles) * p.num_n_tiles;
        grid = static_cast<int>(std::min<int64_t>(tiles, sms));
    }
    if (mx) {
        return grouped ? launch_kernel<true, true>(ta, tb, p, grid, s)
                       : launch_kernel<true, false>(ta, tb, p, grid, s);
    }
    return launch_kernel<false, false>(ta, tb, p, grid, s);
}

cudaError_t launch_zero_fill_bf16(uint16_t* c, int64_t rows, int64_t cols, int64_t ldc,
                                  cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int64_t total = rows * cols;
    const int blocks = static_cast<int>(std::min<int64_t>((total + 255) / 256, 4096));
    zero_fill_kernel<<<blocks, 256, 0, s>>>(c, rows, cols, ldc);
    return cudaGetLastError();
}

cudaError_t take_status_gemm(unsigned* out) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status_gemm, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status_gemm, &zero, sizeof(unsigned));
}

}  // namespace mxfp8
