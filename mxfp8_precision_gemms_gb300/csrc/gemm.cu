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
// Structure: a persistent kernel, one CTA per SM.  In the default PAIR form
// two CTAs of a cluster drive one 2-SM tensor-core operation (cta_group::2)
// on a 256 x 256 output tile: each CTA holds 128 rows of A and 128 rows of B
// per K step (32 KB instead of the 48 KB a single-SM 128 x 256 tile needs),
// so the same shared memory keeps 6 stages in flight and each staged byte
// feeds 1.5x the FLOPs.  The kernel is limited by how many bytes can be in
// flight from L2, not by raw L2 bandwidth (multicasting B across CTAs did
// not help), which is why the 2-SM form pays.  Work units run M-group
// fastest: the resident pairs cover every 256-row group of A for one or two
// 256-column tiles of B at a time, so each B tile is read by ~32 pairs at
// once and A stays in L2.  Banded (4-16 M groups) and diagonal orders were
// 1-27 % slower under a sustained load and drew more power per GEMM.
//   warp 0       TMA producer (both CTAs): A box, this CTA's half of the B box
//                (128-byte swizzle) and the 512-byte scale tiles into a
//                shared-memory ring of slots, one slot per K step; one "full" /
//                "empty" mbarrier pair covers two slots, and every load of both
//                CTAs completes on the leader CTA's "full" mbarrier.  When K
//                splits into whole slot pairs each operand's pair is one copy
//                (3D K-chunk maps for A and B): each TMA instruction costs the
//                issuing thread 70-80 cycles whatever its size (measured), so
//                five copies per pair instead of ten.
//   warp 1       TMEM allocator (both CTAs, collectively) and, in the leader
//                only, the MMA issuer: per K step tcgen05.cp of the block
//                scales into TMEM and 4 MMAs of K = 32 (in issue order, so the
//                MMAs see the scales without a wait), per slot pair one
//                tcgen05.commit releasing the pair in both CTAs and, after the
//                last K step, handing the accumulators over.  Measured in
//                isolation, each tcgen05 instruction costs the issuing thread
//                about 45 cycles (the 3 copies + 4 MMAs of a K step: ~315
//                cycles against 512 of tensor work), a completed try_wait 48
//                and a commit 46; the pipe stays full only while the thread is
//                not waiting, hence one barrier per two K steps and
//                constant-stride address updates.  Moving the copies to another
//                thread was slower: they then have to be waited for, and they
//                queue behind the MMAs already issued.
//   warps 2-9    epilogue (both CTAs): tcgen05.ld of this CTA's 128 x 256 FP32
//                accumulator, release it to the leader, convert to BF16 and
//                store while the next tile's main loop runs: through a 2 KB
//                swizzled staging tile per warp and TMA stores (plain GEMM;
//                direct stores cost the main loop ~7 %), or with direct
//                stores masked to the expert's rows (grouped GEMM).
// Short last wave (plain GEMM): when the tiles left after the full waves
// fill at most half the resident pairs (a 4096 x 4096 output: 256 tiles, 28
// left over on 76 pairs), each of them becomes two units of 128 columns
// (N = 128 MMAs, half the B rows and one B scale tile per K step), so the last
// wave runs on twice as many pairs in a little over half the time.  Every
// output element is the same dot product in the same K order either way.
// Measured: 4096^3 per-tensor GEMM 47.7 -> 46.1 us, the backward row 2 %.
// The single-SM form (PAIR = false) is the same pipeline with one CTA.
// Every wait is bounded; a wait that runs out records MXFP8_ERR_TIMEOUT,
// the CTA drains its outstanding copies and MMAs, frees TMEM and exits.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp8 {

__device__ unsigned int g_status_gemm = 0;

namespace {

constexpr int BM = 128;  // rows of A / C per CTA
constexpr int BN = 256;  // columns of C per tile
constexpr int BK = 128;  // bytes = FP8 elements per K step (one 128-byte swizzle row)
constexpr int A_BYTES = BM * BK;
constexpr int SFA_BYTES = 512;   // one 128-row x 4-block scale tile
constexpr int SFB_BYTES = 1024;  // two of them (the tile's 256 B rows)
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr uint32_t EPI_TILE_BYTES = 32 * 32 * 2;  // 32 rows x 32 BF16 columns
constexpr int SLOTS_PER_BAR = 2;              // K steps covered by one full/empty barrier
constexpr int MAX_GROUPS = 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = BN;           // 128 lanes x 256 FP32 columns
constexpr uint32_t SF_COLS_PER_STAGE = 12;  // A: 4 columns, B: 8 columns

#ifndef GEMM_PAIR
#define GEMM_PAIR 1
#endif

template <bool PAIR>
struct Cfg {
    static constexpr int CG = PAIR ? 2 : 1;  // CTAs per tensor-core operation
    static constexpr int STAGES = PAIR ? 6 : 4;   // shared-memory slots of one K step
    static constexpr int NBARS = STAGES / SLOTS_PER_BAR;
    static constexpr int B_ROWS = BN / CG;   // B rows one CTA holds
    static constexpr int B_BYTES = B_ROWS * BK;
    // shared memory map (offsets from a 1024-byte aligned base)
    static constexpr uint32_t OFF_A = 0;
    static constexpr uint32_t OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr uint32_t OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr uint32_t OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_SFB + STAGES * SFB_BYTES;
    // full, empty per slot pair; tmem_full/empty, drain, never
    static constexpr uint32_t NUM_BARS = 2 * NBARS + 4;
    static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr uint32_t OFF_PREFIX = OFF_MISC + 32;
    // plain GEMM: per epilogue warp a 2 KB staging tile for the TMA stores of C
    static constexpr uint32_t OFF_EPI = (OFF_PREFIX + 1023) / 1024 * 1024;
    static constexpr uint32_t SMEM_PLAIN = OFF_EPI + EPI_WARPS * EPI_TILE_BYTES;
    // grouped GEMM: two prefix tables (tiles and units per expert group), then
    // the staging tiles (512-byte aligned: the 64-byte swizzle's period)
    static constexpr uint32_t OFF_EPI_G = (OFF_PREFIX + 2 * (MAX_GROUPS + 1) * 4 + 511) / 512 * 512;
    static constexpr uint32_t SMEM_GROUPED = OFF_EPI_G + EPI_WARPS * EPI_TILE_BYTES;
    static_assert(OFF_B % 1024 == 0 && OFF_SFA % 1024 == 0, "swizzled tiles need 1024B alignment");
    static_assert(ACC_COLS + STAGES * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
    static_assert(STAGES % SLOTS_PER_BAR == 0, "slots come in barrier pairs");
    // + 1024: the base is aligned up at run time; + 16: the static variables
    static_assert(SMEM_GROUPED + 1024 + 16 <= 232448, "shared memory budget");
    static_assert(SMEM_PLAIN + 1024 + 16 <= 232448, "shared memory budget");
};

struct KParams {
    int64_t M, N, K;
    int32_t num_m_tiles, num_n_tiles, num_k_tiles;
    int32_t num_m_groups;        // ceil(num_m_tiles / CG) (plain GEMM)
    int32_t n_scale_tiles;       // ceil(N / 128): 128-row scale tiles of one B
    int64_t sfb_group_chunks;    // 512-byte scale tiles between experts' B scales
    const float* s_a;            // GEMM_TENSOR scalars
    const float* s_b;
    uint16_t* c;
    int64_t ldc;
    const int32_t* offsets;      // grouped
    int32_t groups;
    uint64_t wait_limit_ns;
    int32_t inject_timeout;
    uint32_t idesc_tensor;
    uint32_t idesc_tensor_half;  // the same with N = 128
    int32_t merged;              // 1: one copy per operand loads a whole slot pair
    // plain GEMM: units [0, split_from) are whole tiles; from split_from on,
    // each remaining tile is two units of 128 columns (a short last wave
    // spread over twice as many pairs); INT64_MAX: no split
    int64_t split_from;
    int64_t total_units;
};

// One CTA's share of a work unit: the unit covers CG consecutive 128-row
// tiles of A (one per CTA of the pair) and one 256-column tile of B.
struct Tile {
    int64_t a_row;     // first row of A (and of C) of this CTA
    int64_t row_end;   // rows of C valid below this
    int64_t sfa_tile;  // 128-row tile index in A's scale array
    int64_t b_row;     // first row of the unit's B rows (grouped: of the experts' stack)
    int64_t n_col;     // first column of C of the unit
    int32_t n_tile;
    int32_t n_half;    // -1: all 256 columns; 0 / 1: that 128-column half only
    int32_t group;
    bool a_valid;      // false: a padding tile (nothing to store)
};

__device__ __forceinline__ void record_status(unsigned code) {
    atomicCAS(&g_status_gemm, 0u, code);
}

template <bool GROUPED, int CG>
__device__ __forceinline__ Tile decode_unit(const KParams& p, int64_t u, uint32_t rank,
                                            const int32_t* mtile_prefix,
                                            const int32_t* mgroup_prefix, const int32_t* offs) {
    Tile tl;
    if constexpr (GROUPED) {
        const int64_t gmg = u / p.num_n_tiles;
        tl.n_tile = static_cast<int32_t>(u % p.num_n_tiles);
        int lo = 0, hi = p.groups - 1;  // largest g with mgroup_prefix[g] <= gmg
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (mgroup_prefix[mid] <= gmg) lo = mid; else hi = mid - 1;
        }
        const int64_t mt = (gmg - mgroup_prefix[lo]) * CG + rank;
        tl.group = lo;
        tl.a_valid = mt < mtile_prefix[lo + 1] - mtile_prefix[lo];
        tl.a_row = offs[lo] + mt * BM;
        tl.row_end = min(static_cast<int64_t>(offs[lo + 1]), tl.a_row + BM);
        tl.sfa_tile = mtile_prefix[lo] + mt;
        tl.b_row = static_cast<int64_t>(lo) * p.N + static_cast<int64_t>(tl.n_tile) * BN;
        tl.n_half = -1;
        tl.n_col = static_cast<int64_t>(tl.n_tile) * BN;
    } else {
        tl.n_half = -1;
        if (u >= p.split_from) {  // half of one of the last tiles
            const int64_t v = u - p.split_from;
            tl.n_half = static_cast<int32_t>(v & 1);
            u = p.split_from + (v >> 1);
        }
        const int64_t mt = (u % p.num_m_groups) * CG + rank;
        tl.n_tile = static_cast<int32_t>(u / p.num_m_groups);
        tl.group = 0;
        tl.a_valid = mt < p.num_m_tiles;
        tl.a_row = mt * BM;
        tl.row_end = min(p.M, tl.a_row + BM);
        tl.sfa_tile = mt;
        tl.n_col = static_cast<int64_t>(tl.n_tile) * BN + (tl.n_half > 0 ? BN / 2 : 0);
        tl.b_row = tl.n_col;
    }
    return tl;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// tm_a / tm_b: payload boxes (128 x 128 and B_ROWS x 128 bytes, 128-byte
// swizzle); with p.merged, 3D K-chunk maps whose box is SLOTS_PER_BAR such
// tiles (one copy fills a slot pair).  tm_sa / tm_sb: the scale arrays seen as
// rows of 256 bytes, boxes of 2 rows = one 512-byte scale tile, or of
// 2 * SLOTS_PER_BAR rows with p.merged (out-of-range tiles read as 0).
// tm_c: C as BF16, 32 x 32 boxes with 64-byte swizzle (plain GEMM only; the
// store clips rows and columns outside M x N).
// The kernel body for one problem, run by the CTA pairs pair_id of
// num_pairs (a persistent round robin over the problem's work units).
template <bool MX, bool GROUPED, bool PAIR>
__device__ __forceinline__ void gemm_body(const CUtensorMap* tm_a, const CUtensorMap* tm_b,
                                          const CUtensorMap* tm_bh, const CUtensorMap* tm_sa,
                                          const CUtensorMap* tm_sb, const CUtensorMap* tm_c,
                                          const KParams& p, int64_t pair_id, int64_t num_pairs) {
    using C = Cfg<PAIR>;
    constexpr int CG = C::CG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_ctarank() : 0;
    const bool leader = rank == 0;

    auto bar = [&](uint32_t i) { return sbase + C::OFF_BAR + 8 * i; };
    constexpr uint32_t NB = C::NBARS;
    const uint32_t BAR_FULL = 0, BAR_EMPTY = NB, BAR_TMEM_FULL = 2 * NB,
                   BAR_TMEM_EMPTY = 2 * NB + 1, BAR_DRAIN = 2 * NB + 2, BAR_NEVER = 2 * NB + 3;
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
    int32_t* mtile_prefix = reinterpret_cast<int32_t*>(smem + C::OFF_PREFIX);
    int32_t* mgroup_prefix = mtile_prefix + (MAX_GROUPS + 1);
    const int32_t* offs = p.offsets;  // validated below before any use
    __shared__ int64_t s_total_units;

    if (threadIdx.x == 0) {
        for (uint32_t b = 0; b < NB; ++b) {
            mbar_init(bar(BAR_FULL + b), 1);
            mbar_init(bar(BAR_EMPTY + b), 1);
        }
        mbar_init(bar(BAR_TMEM_FULL), 1);
        mbar_init(bar(BAR_TMEM_EMPTY), EPI_WARPS * CG);  // both CTAs' epilogues
        mbar_init(bar(BAR_DRAIN), 1);
        mbar_init(bar(BAR_NEVER), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // Launched with programmatic stream serialization: everything above
    // touches only shared memory; from here on the kernel reads what the
    // kernels before it wrote (operands, scales, offsets, per-tensor scales).
    griddep_wait();
    if constexpr (GROUPED) {
        // Validate the offsets; prefix sums of 128-row tiles and of units of
        // CG tiles per expert group.
        if (warp == 0) {
            const int G = p.groups;
            bool ok = (p.offsets[0] == 0) && (static_cast<int64_t>(p.offsets[G]) == p.M);
            int32_t tbase = 0, gbase = 0;
            for (int g0 = 0; g0 <= G; g0 += 32) {
                const int g = g0 + lane;
                int32_t tiles = 0;
                if (g < G) {
                    const int32_t m = p.offsets[g + 1] - p.offsets[g];
                    if (m < 0) ok = false;
                    tiles = m > 0 ? (m + BM - 1) / BM : 0;
                }
                const int32_t mgs = (tiles + CG - 1) / CG;
                int32_t ti = tiles, gi = mgs;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int32_t v = __shfl_up_sync(0xffffffffu, ti, d);
                    const int32_t w = __shfl_up_sync(0xffffffffu, gi, d);
                    if (lane >= d) {
                        ti += v;
                        gi += w;
                    }
                }
                if (g <= G) {
                    mtile_prefix[g] = tbase + ti - tiles;
                    mgroup_prefix[g] = gbase + gi - mgs;
                }
                tbase += __shfl_sync(0xffffffffu, ti, 31);
                gbase += __shfl_sync(0xffffffffu, gi, 31);
            }
            ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) {
                s_total_units = ok ? static_cast<int64_t>(gbase) * p.num_n_tiles : 0;
                if (!ok && blockIdx.x == 0) record_status(MXFP8_ERR_DEVICE_CHECK);
            }
        }
    } else {
        if (threadIdx.x == 0)
            s_total_units = p.total_units;
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(misc), TMEM_COLS);  // with CG = 2: both CTAs, same columns
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the peer's barriers exist before any remote use
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int64_t total = s_total_units;

    auto fail = [&]() {
        *abort_flag = 1;
        record_status(MXFP8_ERR_TIMEOUT);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(tm_a);
            tma_prefetch_desc(tm_b);
            if (p.split_from < p.total_units) tma_prefetch_desc(tm_bh);
            if constexpr (MX) {
                tma_prefetch_desc(tm_sa);
                tma_prefetch_desc(tm_sb);
            }
            uint32_t pb = 0, phase = 0;              // slot pair (barrier) and its parity
            uint32_t issued = 0, issued_parity = 0;  // per-barrier bit masks (leader's drain)
            bool ok = true;
            constexpr uint32_t kSlotTx =
                CG * (A_BYTES + C::B_BYTES + (MX ? SFA_BYTES + SFB_BYTES : 0));
            // a half unit: half the B rows and one of the two B scale tiles
            constexpr uint32_t kSlotTxHalf =
                CG * (A_BYTES + C::B_BYTES / 2 + (MX ? SFA_BYTES + SFB_BYTES / 2 : 0));
            for (int64_t u = pair_id; u < total && ok; u += num_pairs) {
                const Tile tl = decode_unit<GROUPED, CG>(p, u, rank, mtile_prefix, mgroup_prefix, offs);
                const bool hu = tl.n_half >= 0;
                // B scale tiles: the unit's first 128 rows at sfb_base, the
                // next 128 (whole tiles only) num_k_tiles tiles further on
                const int64_t sfb_base = static_cast<int64_t>(tl.group) * p.sfb_group_chunks +
                                         (2 * static_cast<int64_t>(tl.n_tile) + (hu ? tl.n_half : 0)) *
                                             p.num_k_tiles;
                const int32_t b_row =
                    static_cast<int32_t>(tl.b_row + rank * (hu ? C::B_ROWS / 2 : C::B_ROWS));
                const CUtensorMap* mb = hu ? tm_bh : tm_b;  // 2D maps (per-slot copies)
                const uint32_t slot_tx = hu ? kSlotTxHalf : kSlotTx;
                for (int kt0 = 0; kt0 < p.num_k_tiles; kt0 += SLOTS_PER_BAR) {
                    const int nslots = min(SLOTS_PER_BAR, p.num_k_tiles - kt0);
                    if (!mbar_wait(bar(BAR_EMPTY + pb), phase ^ 1u, p.wait_limit_ns, abort_flag)) {
                        fail();
                        ok = false;
                        break;
                    }
                    const uint32_t fb_local = bar(BAR_FULL + pb);
                    if (leader) mbar_arrive_expect_tx(fb_local, slot_tx * nslots);
                    const uint32_t slot0 = pb * SLOTS_PER_BAR;
                    // B scales of a slot pair: [half 0 of each slot][half 1 of each slot]
                    const uint32_t dSBp = sbase + C::OFF_SFB + slot0 * SFB_BYTES;
                    if (p.merged) {
                        // K % (BK * SLOTS_PER_BAR) == 0: the pair is full and each
                        // operand's SLOTS_PER_BAR K steps are one box (A, B: 3D K-chunk
                        // maps; scales: consecutive 512-byte tiles)
                        const uint32_t dA = sbase + C::OFF_A + slot0 * A_BYTES;
                        const uint32_t dB = sbase + C::OFF_B + slot0 * C::B_BYTES;
                        const uint32_t dSA = sbase + C::OFF_SFA + slot0 * SFA_BYTES;
                        const int32_t ya = static_cast<int32_t>(2 * (tl.sfa_tile * p.num_k_tiles + kt0));
                        const int32_t yb0 = static_cast<int32_t>(2 * (sfb_base + kt0));
                        const int32_t yb1 = static_cast<int32_t>(2 * (sfb_base + p.num_k_tiles + kt0));
                        if constexpr (PAIR) {
                            const uint32_t fb = mapa_shared(fb_local, 0);  // the leader's barrier
                            tma_load_3d_pair(dA, tm_a, fb, 0, static_cast<int32_t>(tl.a_row), kt0);
                            if (!hu) {
                                tma_load_3d_pair(dB, tm_b, fb, 0, b_row, kt0);
                            } else {  // 2D boxes of B_ROWS / 2 rows, one per slot
                                for (int j = 0; j < SLOTS_PER_BAR; ++j)
                                    tma_load_2d_pair(dB + j * C::B_BYTES, tm_bh, fb, (kt0 + j) * BK, b_row);
                            }
                            if constexpr (MX) {
                                tma_load_2d_pair(dSA, tm_sa, fb, 0, ya);
                                tma_load_2d_pair(dSBp, tm_sb, fb, 0, yb0);
                                if (!hu) tma_load_2d_pair(dSBp + SLOTS_PER_BAR * 512, tm_sb, fb, 0, yb1);
                            }
                        } else {
                            tma_load_3d(dA, tm_a, fb_local, 0, static_cast<int32_t>(tl.a_row), kt0);
                            if (!hu) {
                                tma_load_3d(dB, tm_b, fb_local, 0, b_row, kt0);
                            } else {
                                for (int j = 0; j < SLOTS_PER_BAR; ++j)
                                    tma_load_2d(dB + j * C::B_BYTES, tm_bh, fb_local, (kt0 + j) * BK, b_row);
                            }
                            if constexpr (MX) {
                                tma_load_2d(dSA, tm_sa, fb_local, 0, ya);
                                tma_load_2d(dSBp, tm_sb, fb_local, 0, yb0);
                                if (!hu) tma_load_2d(dSBp + SLOTS_PER_BAR * 512, tm_sb, fb_local, 0, yb1);
                            }
                        }
                    } else {
                        for (int j = 0; j < nslots; ++j) {
                            const int kt = kt0 + j;
                            const uint32_t slot = slot0 + j;
                            const uint32_t dA = sbase + C::OFF_A + slot * A_BYTES;
                            const uint32_t dB = sbase + C::OFF_B + slot * C::B_BYTES;
                            const uint32_t dSA = sbase + C::OFF_SFA + slot * SFA_BYTES;
                            const uint32_t dSB0 = dSBp + j * 512;
                            const uint32_t dSB1 = dSBp + (SLOTS_PER_BAR + j) * 512;
                            const int32_t ya = static_cast<int32_t>(2 * (tl.sfa_tile * p.num_k_tiles + kt));
                            const int32_t yb0 = static_cast<int32_t>(2 * (sfb_base + kt));
                            const int32_t yb1 = static_cast<int32_t>(2 * (sfb_base + p.num_k_tiles + kt));
                            if constexpr (PAIR) {
                                const uint32_t fb = mapa_shared(fb_local, 0);  // the leader's barrier
                                tma_load_2d_pair(dA, tm_a, fb, kt * BK, static_cast<int32_t>(tl.a_row));
                                tma_load_2d_pair(dB, mb, fb, kt * BK, b_row);
                                if constexpr (MX) {
                                    tma_load_2d_pair(dSA, tm_sa, fb, 0, ya);
                                    tma_load_2d_pair(dSB0, tm_sb, fb, 0, yb0);
                                    if (!hu) tma_load_2d_pair(dSB1, tm_sb, fb, 0, yb1);
                                }
                            } else {
                                tma_load_2d(dA, tm_a, fb_local, kt * BK, static_cast<int32_t>(tl.a_row));
                                tma_load_2d(dB, mb, fb_local, kt * BK, b_row);
                                if constexpr (MX) {
                                    tma_load_2d(dSA, tm_sa, fb_local, 0, ya);
                                    tma_load_2d(dSB0, tm_sb, fb_local, 0, yb0);
                                    if (!hu) tma_load_2d(dSB1, tm_sb, fb_local, 0, yb1);
                                }
                            }
                        }
                    }
                    issued |= 1u << pb;
                    issued_parity = (issued_parity & ~(1u << pb)) | (phase << pb);
                    if (++pb == NB) {
                        pb = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && leader) {
                // let every copy already in flight land before the CTA exits
                const int never = 0;
                for (uint32_t b = 0; b < NB; ++b) {
                    if (issued & (1u << b))
                        mbar_wait(bar(BAR_FULL + b), (issued_parity >> b) & 1u, p.wait_limit_ns,
                                  &never);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader)
        if (lane == 0 && leader) {
            const int never = 0;
            bool ok = true;
            if (p.inject_timeout) {
                // test hook: a wait on a barrier nothing signals
                if (!mbar_wait(bar(BAR_NEVER), 0, p.wait_limit_ns, &never)) {
                    fail();
                    ok = false;
                }
            }
            constexpr uint16_t kPairMask = PAIR ? 3 : 1;
            uint32_t pb = 0, phase = 0, acc_phase = 0;
            // Descriptors and TMEM addresses of slot pair pb, advanced by
            // constants (a single thread issues everything: its dependent
            // bookkeeping, not the tensor pipe, sets the pace).  The smem
            // start-address fields (bits 0-13, address >> 4) never carry:
            // shared memory stays below 256 KB.
            constexpr uint32_t kPairA = SLOTS_PER_BAR * A_BYTES >> 4;
            constexpr uint32_t kPairB = SLOTS_PER_BAR * C::B_BYTES >> 4;
            constexpr uint32_t kPairSfa = SLOTS_PER_BAR * SFA_BYTES >> 4;
            constexpr uint32_t kPairSfb = SLOTS_PER_BAR * SFB_BYTES >> 4;
            constexpr uint32_t kPairCols = SLOTS_PER_BAR * SF_COLS_PER_STAGE;
            const uint64_t desc_a0 = smem_desc(sbase + C::OFF_A, 16, 1024, SWZ_128B);
            const uint64_t desc_b0 = smem_desc(sbase + C::OFF_B, 16, 1024, SWZ_128B);
            const uint64_t sfa_d0 = smem_desc(sbase + C::OFF_SFA, 0, 128, SWZ_NONE);
            const uint64_t sfb_d0 = smem_desc(sbase + C::OFF_SFB, 0, 128, SWZ_NONE);
            const uint32_t sf_t0 = tmem + ACC_COLS;
            uint64_t da = desc_a0, db = desc_b0, dsa = sfa_d0, dsb = sfb_d0;
            uint32_t sft = sf_t0;
            for (int64_t u = pair_id; u < total && ok; u += num_pairs) {
                if (!mbar_wait(bar(BAR_TMEM_EMPTY), acc_phase ^ 1u, p.wait_limit_ns, abort_flag)) {
                    fail();
                    break;
                }
                tc_fence_after();
                // one unit's K loop; HALF: 128 columns (N = 128, one B scale tile)
                auto k_loop = [&](auto half_c) {
                    constexpr bool HALF = decltype(half_c)::value;
                    uint32_t acc = 0;  // the first MMA of a unit overwrites the accumulator
                    for (int kt0 = 0; kt0 < p.num_k_tiles; kt0 += SLOTS_PER_BAR) {
                        const int nslots = min(SLOTS_PER_BAR, p.num_k_tiles - kt0);
                        if (!mbar_wait(bar(BAR_FULL + pb), phase, p.wait_limit_ns, abort_flag)) {
                            fail();
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int j = 0; j < SLOTS_PER_BAR; ++j) {
                            if (j < nslots) {
                                const uint64_t dja = da + j * (A_BYTES >> 4);
                                const uint64_t djb = db + j * (C::B_BYTES >> 4);
                                if constexpr (MX) {
                                    const uint32_t sfa_t = sft + j * SF_COLS_PER_STAGE;
                                    // scales of this K step into TMEM; issued in order with
                                    // the MMAs below, which therefore see them
                                    tc_cp_32x128b_warpx4<CG>(sfa_t, dsa + j * (SFA_BYTES >> 4));
                                    tc_cp_32x128b_warpx4<CG>(sfa_t + 4, dsb + j * (512 >> 4));
                                    if constexpr (!HALF)
                                        tc_cp_32x128b_warpx4<CG>(sfa_t + 8,
                                                                 dsb + (SLOTS_PER_BAR + j) * (512 >> 4));
#pragma unroll
                                    for (uint32_t kk = 0; kk < BK / 32; ++kk) {
                                        mma_mxf8<CG>(tmem, dja + 2 * kk, djb + 2 * kk,
                                                     idesc_mxf8(BM * CG, HALF ? BN / 2 : BN, kk), sfa_t,
                                                     sfa_t + 4, acc);
                                        acc = 1;
                                    }
                                } else {
                                    const uint32_t idesc = HALF ? p.idesc_tensor_half : p.idesc_tensor;
#pragma unroll
                                    for (uint32_t kk = 0; kk < BK / 32; ++kk) {
                                        mma_f8<CG>(tmem, dja + 2 * kk, djb + 2 * kk, idesc, acc);
                                        acc = 1;
                                    }
                                }
                            }
                        }
                        // the slot pair is free in both CTAs once these MMAs completed
                        if constexpr (PAIR) tc_commit_multicast<CG>(bar(BAR_EMPTY + pb), kPairMask);
                        else tc_commit<CG>(bar(BAR_EMPTY + pb));
                        if (++pb == NB) {
                            pb = 0;
                            phase ^= 1u;
                            da = desc_a0;
                            db = desc_b0;
                            dsa = sfa_d0;
                            dsb = sfb_d0;
                            sft = sf_t0;
                        } else {
                            da += kPairA;
                            db += kPairB;
                            dsa += kPairSfa;
                            dsb += kPairSfb;
                            sft += kPairCols;
                        }
                    }
                };
                if (u >= p.split_from) k_loop(std::true_type{});
                else k_loop(std::false_type{});
                if (!ok) break;
                if constexpr (PAIR) tc_commit_multicast<CG>(bar(BAR_TMEM_FULL), kPairMask);
                else tc_commit<CG>(bar(BAR_TMEM_FULL));
                acc_phase ^= 1u;
            }
            // every MMA / copy this thread issued completes before teardown
            tc_commit<CG>(bar(BAR_DRAIN));
            mbar_wait(bar(BAR_DRAIN), 0, p.wait_limit_ns, &never);
        }
    } else {
        // ------------------------------------------------ epilogue
        const int quarter = warp & 3;        // TMEM lanes this warp may read
        const int half = (warp - 2) >> 2;    // which 128 accumulator columns (warps 2-9)
        const uint32_t empty_bar = PAIR ? mapa_shared(bar(BAR_TMEM_EMPTY), 0) : bar(BAR_TMEM_EMPTY);
        float alpha = 1.0f;
        if constexpr (!MX) alpha = __fdiv_rn(1.0f, *p.s_a) * __fdiv_rn(1.0f, *p.s_b);
        uint32_t acc_phase = 0;
        for (int64_t u = pair_id; u < total; u += num_pairs) {
            const Tile tl = decode_unit<GROUPED, CG>(p, u, rank, mtile_prefix, mgroup_prefix, offs);
            if (!mbar_wait(bar(BAR_TMEM_FULL), acc_phase, p.wait_limit_ns, abort_flag)) {
                fail();
                break;
            }
            tc_fence_after();
            uint32_t v[128];
            // a half unit's 128 columns sit in accumulator columns 0..127
            const bool idle = tl.n_half >= 0 && half == 1;
            if (!idle) {
                const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + half * 128;
                tmem_ld_x32(taddr + 0, v + 0);
                tmem_ld_x32(taddr + 32, v + 32);
                tmem_ld_x32(taddr + 64, v + 64);
                tmem_ld_x32(taddr + 96, v + 96);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(empty_bar);
                else mbar_arrive(empty_bar);
            }
            // This warp's 32 rows go out through TMA stores when they are all
            // rows of C this tile owns (always, for a valid plain tile; for an
            // expert group's last tile only the warps inside the group), else
            // with masked direct stores.
            bool staged = tl.a_valid && !idle;
            if constexpr (GROUPED) staged = staged && tl.a_row + quarter * 32 + 32 <= tl.row_end;
            {
                // BF16 through a swizzled 32 x 32 staging tile and TMA stores:
                // lane = row; 16-byte chunk j of a 64-byte row goes to chunk
                // j ^ ((row >> 1) & 3), the 64-byte swizzle the store undoes,
                // which also keeps each 8-lane phase on distinct banks
                const uint32_t stile =
                    sbase + (GROUPED ? C::OFF_EPI_G : C::OFF_EPI) + (warp - 2) * EPI_TILE_BYTES;
                const uint32_t srow = stile + lane * 64;
                const uint32_t sw = (lane >> 1) & 3;
                if (staged) {
                    const int32_t y = static_cast<int32_t>(tl.a_row + quarter * 32);
                    const int32_t x0 = static_cast<int32_t>(tl.n_col + half * 128);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            w[i] = pack_bf16x2(__uint_as_float(v[32 * c + 2 * i]) * alpha,
                                               __uint_as_float(v[32 * c + 2 * i + 1]) * alpha);
                        if (lane == 0) bulk_wait_group_read0();  // the tile is free again
                        __syncwarp();
#pragma unroll
                        for (uint32_t j = 0; j < 4; ++j) {
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                             srow + 16 * (j ^ sw)),
                                         "r"(w[4 * j]), "r"(w[4 * j + 1]), "r"(w[4 * j + 2]),
                                         "r"(w[4 * j + 3])
                                         : "memory");
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(tm_c, stile, x0 + 32 * c, y);
                            bulk_commit_group();
                        }
                    }
                }
            }
            if (GROUPED && !staged) {
                const int64_t row = tl.a_row + quarter * 32 + lane;
                if (tl.a_valid && row < tl.row_end) {
                    uint16_t* crow = p.c + row * p.ldc;
                    const int64_t col0 = tl.n_col + half * 128;
    #pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int64_t col = col0 + j * 8;
                        if (col < p.N && MX_IN_BOUNDS(row < p.M && col + 8 <= p.N)) {
                            uint4 o;
                            o.x = pack_bf16x2(__uint_as_float(v[8 * j + 0]) * alpha,
                                              __uint_as_float(v[8 * j + 1]) * alpha);
                            o.y = pack_bf16x2(__uint_as_float(v[8 * j + 2]) * alpha,
                                              __uint_as_float(v[8 * j + 3]) * alpha);
                            o.z = pack_bf16x2(__uint_as_float(v[8 * j + 4]) * alpha,
                                              __uint_as_float(v[8 * j + 5]) * alpha);
                            o.w = pack_bf16x2(__uint_as_float(v[8 * j + 6]) * alpha,
                                              __uint_as_float(v[8 * j + 7]) * alpha);
                            // evict-first: C streams out to HBM while the GEMM
                            // runs instead of lingering in L2 as dirty lines
                            __stcs(reinterpret_cast<uint4*>(crow + col), o);
                        }
                    }
                }
            }
            acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait_group0();  // every store of C has completed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // the leader's MMAs (which also write the peer's TMEM) have drained and
    // both epilogues are done before either CTA frees its TMEM
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem, TMEM_COLS);
    }
    if constexpr (PAIR) cluster_sync();
}

template <bool MX, bool GROUPED, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_bh, const __grid_constant__ CUtensorMap tm_sa,
                const __grid_constant__ CUtensorMap tm_sb, const __grid_constant__ CUtensorMap tm_c,
                const __grid_constant__ KParams p) {
    constexpr int CG = Cfg<PAIR>::CG;
    gemm_body<MX, GROUPED, PAIR>(&tm_a, &tm_b, &tm_bh, &tm_sa, &tm_sb, &tm_c, p, blockIdx.x / CG,
                                 gridDim.x / CG);
}

// Two independent plain GEMMs in one persistent launch: pairs0 of the CTA
// pairs, spread evenly over the grid, run problem 0, the others problem 1,
// each with the pipeline
// above over its own work units (the host picks pairs0 so that both finish
// together: the backward's dgrad and wgrad, whose last waves would otherwise
// each leave pairs idle, and one launch boundary less).
template <bool MX, bool PAIR>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_dual_kernel(const __grid_constant__ CUtensorMap a0, const __grid_constant__ CUtensorMap b0,
                     const __grid_constant__ CUtensorMap bh0, const __grid_constant__ CUtensorMap sa0,
                     const __grid_constant__ CUtensorMap sb0, const __grid_constant__ CUtensorMap c0,
                     const __grid_constant__ CUtensorMap a1, const __grid_constant__ CUtensorMap b1,
                     const __grid_constant__ CUtensorMap bh1, const __grid_constant__ CUtensorMap sa1,
                     const __grid_constant__ CUtensorMap sb1, const __grid_constant__ CUtensorMap c1,
                     const __grid_constant__ KParams p0, const __grid_constant__ KParams p1,
                     int32_t pairs0) {
    constexpr int CG = Cfg<PAIR>::CG;
    const int64_t pair = blockIdx.x / CG;
    const int64_t pairs = gridDim.x / CG;
    // problem 0's pairs spread evenly over the grid (and so over both dies):
    // c(q) = floor(q pairs0 / pairs) of the pairs below q are problem 0's
    const int64_t c = pair * pairs0 / pairs;
    if ((pair + 1) * pairs0 / pairs > c)
        gemm_body<MX, false, PAIR>(&a0, &b0, &bh0, &sa0, &sb0, &c0, p0, c, pairs0);
    else
        gemm_body<MX, false, PAIR>(&a1, &b1, &bh1, &sa1, &sb1, &c1, p1, pair - c, pairs - pairs0);
}

__global__ void zero_fill_kernel(uint16_t* c, int64_t rows, int64_t cols, int64_t ldc) {
    const int64_t total = rows * cols;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        c[(i / cols) * ldc + (i % cols)] = 0;
    }
}

// ------------------------------------------------------------ host side --

// 2D tensor map over a rows x width byte matrix (row stride width).
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t width, uint32_t box_w,
              uint32_t box_rows, CUtensorMapSwizzle swz) {
    return encode_tensor_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rows, width, width, box_w,
                                box_rows, swz);
}

// Per device: the dynamic shared memory attribute is set once and the number
// of co-resident clusters is queried once (both are host-side driver calls
// too slow to repeat on every launch).
constexpr int kMaxDevices = 64;

template <bool MX, bool GROUPED, bool PAIR>
cudaError_t launch_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbh,
                          const CUtensorMap& tsa, const CUtensorMap& tsb, const CUtensorMap& tc,
                          const KParams& p_in, int64_t units, bool can_split, cudaStream_t s) {
    using C = Cfg<PAIR>;
    static std::atomic<int> resident[kMaxDevices];  // 0 = not yet queried
    const uint32_t smem = (GROUPED ? C::SMEM_GROUPED : C::SMEM_PLAIN) + 1024;
    auto k = gemm_kernel<MX, GROUPED, PAIR>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // the kernel may start while the previous kernel on the stream finishes
    // (it waits for that kernel's results after its prologue)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int max_clusters = resident[dev].load(std::memory_order_relaxed);
    if (max_clusters <= 0) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        // persistent grid: as many pairs (or CTAs) as can be resident at once
        cfg.gridDim = dim3(C::CG * 64, 1, 1);
        e = cudaOccupancyMaxActiveClusters(&max_clusters, k, &cfg);
        if (e != cudaSuccess || max_clusters <= 0) {
            (void)cudaGetLastError();
            max_clusters = sm_count_current_device() / C::CG;
        }
        resident[dev].store(max_clusters, std::memory_order_relaxed);
    }
    KParams p = p_in;
    p.split_from = INT64_MAX;
    p.total_units = units;
    if (!GROUPED && can_split) {
        // A last wave that fills at most half the pairs: its tiles become
        // two 128-column units each, on twice as many pairs (same dot
        // products, same K order: the same C)
        const int64_t tail = units % max_clusters;
        if (tail > 0 && 2 * tail <= max_clusters) {
            p.split_from = units - tail;
            p.total_units = units + tail;
        }
    }
    const int64_t clusters = std::max<int64_t>(1, std::min<int64_t>(p.total_units, max_clusters));
    cfg.gridDim = dim3(static_cast<unsigned>(clusters * C::CG), 1, 1);
    e = cudaLaunchKernelEx(&cfg, k, ta, tb, tbh, tsa, tsb, tc, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

constexpr bool kPair = GEMM_PAIR != 0;

}  // namespace

namespace {

// Tensor maps, parameters and unit count of one GEMM.
struct Prepared {
    CUtensorMap ta, tb, tbh, tsa, tsb, tc;
    KParams p;
    int64_t units;
    bool can_split;
};

cudaError_t prepare_gemm(const GemmArgs& g, Prepared* out) {
    using C = Cfg<kPair>;
    const bool grouped = g.groups > 0;
    const bool mx = g.mode == GEMM_MX;
    const int64_t b_rows = grouped ? static_cast<int64_t>(g.groups) * g.N : g.N;
    KParams p{};
    p.M = g.M;
    p.N = g.N;
    p.K = g.K;
    p.num_m_tiles = static_cast<int32_t>((g.M + BM - 1) / BM);
    p.num_n_tiles = static_cast<int32_t>((g.N + BN - 1) / BN);
    p.num_k_tiles = static_cast<int32_t>((g.K + BK - 1) / BK);
    p.num_m_groups = (p.num_m_tiles + C::CG - 1) / C::CG;
    p.n_scale_tiles = static_cast<int32_t>((g.N + 127) / 128);
    p.sfb_group_chunks = static_cast<int64_t>(p.n_scale_tiles) * p.num_k_tiles;
    CUtensorMap& ta = out->ta;
    CUtensorMap& tb = out->tb;
    CUtensorMap& tsa = out->tsa;
    CUtensorMap& tsb = out->tsb;
    // whole slot pairs in one copy per operand when K splits into full pairs
    p.merged = g.K % (BK * SLOTS_PER_BAR) == 0 &&
               encode_kchunk_map_u8(&ta, g.a, g.M, g.K, BM, SLOTS_PER_BAR) &&
               encode_kchunk_map_u8(&tb, g.b, b_rows, g.K, C::B_ROWS, SLOTS_PER_BAR);
    if (!p.merged &&
        (!make_map(&ta, g.a, g.M, g.K, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
         !make_map(&tb, g.b, b_rows, g.K, BK, C::B_ROWS, CU_TENSOR_MAP_SWIZZLE_128B)))
        return cudaErrorInvalidValue;
    // half units (plain GEMM): B in boxes of half the rows, one per K step
    CUtensorMap& tbh = out->tbh;
    tbh = tb;
    const bool can_split =
        !grouped && make_map(&tbh, g.b, b_rows, g.K, BK, C::B_ROWS / 2, CU_TENSOR_MAP_SWIZZLE_128B);
    const uint32_t sf_box_rows = p.merged ? 2 * SLOTS_PER_BAR : 2;
    if (mx) {
        // scale arrays as 256-byte rows; a 512-byte scale tile is 2 rows, the
        // tiles of consecutive K steps are consecutive
        const int64_t a_tiles = grouped ? (g.M + 127) / 128 + g.groups : p.num_m_tiles;
        const int64_t a_chunks = a_tiles * p.num_k_tiles;
        const int64_t b_chunks = (grouped ? g.groups : 1) * p.sfb_group_chunks;
        if (!make_map(&tsa, g.a_scale, 2 * a_chunks, 256, 256, sf_box_rows, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map(&tsb, g.b_scale, 2 * b_chunks, 256, 256, sf_box_rows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        tsa = ta;  // unused
        tsb = tb;
        p.s_a = static_cast<const float*>(g.a_scale);
        p.s_b = static_cast<const float*>(g.b_scale);
        p.idesc_tensor = idesc_f8(BM * C::CG, BN, static_cast<uint32_t>(g.a_fmt),
                                  static_cast<uint32_t>(g.b_fmt));
        p.idesc_tensor_half = idesc_f8(BM * C::CG, BN / 2, static_cast<uint32_t>(g.a_fmt),
                                       static_cast<uint32_t>(g.b_fmt));
    }
    p.c = g.c;
    p.ldc = g.ldc;
    // C as BF16 32 x 32 boxes (grouped: only warps whose rows all lie in one
    // expert group store through it)
    CUtensorMap& tc = out->tc;
    if (!encode_tensor_map_2d(&tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.c, g.M, g.N, g.ldc * 2, 32, 32,
                              CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    p.offsets = g.offsets;
    p.groups = g.groups;
    p.wait_limit_ns = wait_limit_ns();
    p.inject_timeout = take_inject_timeout() ? 1 : 0;
    // grouped: the unit count depends on device offsets; this bound only caps the grid
    const int64_t units = grouped
        ? (static_cast<int64_t>(p.num_m_tiles) / C::CG + g.groups + 1) * p.num_n_tiles
        : static_cast<int64_t>(p.num_m_groups) * p.num_n_tiles;
    out->p = p;
    out->units = units;
    out->can_split = can_split;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t s) {
    Prepared d;
    cudaError_t e = prepare_gemm(g, &d);
    if (e != cudaSuccess) return e;
    const bool mx = g.mode == GEMM_MX;
    if (g.groups > 0)
        return launch_kernel<true, true, kPair>(d.ta, d.tb, d.tbh, d.tsa, d.tsb, d.tc, d.p, d.units, false, s);
    if (mx)
        return launch_kernel<true, false, kPair>(d.ta, d.tb, d.tbh, d.tsa, d.tsb, d.tc, d.p, d.units,
                                                 d.can_split, s);
    return launch_kernel<false, false, kPair>(d.ta, d.tb, d.tbh, d.tsa, d.tsb, d.tc, d.p, d.units,
                                              d.can_split, s);
}

namespace {

// Units a problem gives `pairs` CTA pairs, as the launcher arranges them: a
// last wave filling at most half the pairs is split into half units.
void plan_units(const KParams& p_in, int64_t units, bool can_split, int64_t pairs, KParams* p) {
    *p = p_in;
    p->split_from = INT64_MAX;
    p->total_units = units;
    if (can_split && pairs > 0) {
        const int64_t tail = units % pairs;
        if (tail > 0 && 2 * tail <= pairs) {
            p->split_from = units - tail;
            p->total_units = units + tail;
        }
    }
}

// Time of a problem on `pairs` pairs in units of one K step: whole waves of
// num_k_tiles steps, a split last wave at a little over half of that.
double plan_cost(const KParams& p, int64_t units, bool can_split, int64_t pairs) {
    if (pairs <= 0) return 1e300;
    const int64_t waves = units / pairs, tail = units % pairs;
    double w = static_cast<double>(waves);
    if (tail > 0) w += (can_split && 2 * tail <= pairs) ? 0.55 : 1.0;
    return w * p.num_k_tiles;
}

template <bool MX>
cudaError_t launch_dual(const Prepared& d0, const Prepared& d1, cudaStream_t s) {
    using C = Cfg<kPair>;
    static std::atomic<int> resident[kMaxDevices];
    const uint32_t smem = C::SMEM_PLAIN + 1024;
    auto k = gemm_dual_kernel<MX, kPair>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    // the kernel may start while the previous kernel on the stream finishes
    // (it waits for that kernel's results after its prologue)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int max_clusters = resident[dev].load(std::memory_order_relaxed);
    if (max_clusters <= 0) {
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(C::CG * 64, 1, 1);
        e = cudaOccupancyMaxActiveClusters(&max_clusters, k, &cfg);
        if (e != cudaSuccess || max_clusters <= 0) {
            (void)cudaGetLastError();
            max_clusters = sm_count_current_device() / C::CG;
        }
        resident[dev].store(max_clusters, std::memory_order_relaxed);
    }
    if (max_clusters < 2) return cudaErrorInvalidConfiguration;
    // the split of the pairs whose slower problem finishes first
    int64_t best = 1;
    double best_cost = 1e300;
    for (int64_t p0 = 1; p0 < max_clusters; ++p0) {
        const double c = std::max(plan_cost(d0.p, d0.units, d0.can_split, p0),
                                  plan_cost(d1.p, d1.units, d1.can_split, max_clusters - p0));
        if (c < best_cost) {
            best_cost = c;
            best = p0;
        }
    }
    KParams p0, p1;
    plan_units(d0.p, d0.units, d0.can_split, best, &p0);
    plan_units(d1.p, d1.units, d1.can_split, max_clusters - best, &p1);
    cfg.gridDim = dim3(static_cast<unsigned>(max_clusters * C::CG), 1, 1);
    const int32_t pairs0 = static_cast<int32_t>(best);
    e = cudaLaunchKernelEx(&cfg, k, d0.ta, d0.tb, d0.tbh, d0.tsa, d0.tsb, d0.tc, d1.ta, d1.tb, d1.tbh,
                           d1.tsa, d1.tsb, d1.tc, p0, p1, pairs0);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_dual(const GemmArgs& g0, const GemmArgs& g1, cudaStream_t s) {
    Prepared d0, d1;
    cudaError_t e = prepare_gemm(g0, &d0);
    if (e == cudaSuccess) e = prepare_gemm(g1, &d1);
    if (e != cudaSuccess) return e;
    // the inject hook applies to the next launch once: give it to problem 0
    d1.p.inject_timeout = 0;
    return g0.mode == GEMM_MX ? launch_dual<true>(d0, d1, s) : launch_dual<false>(d0, d1, s);
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
