// Blockwise-scaled FP8 GEMM on tcgen05 (sm_103a).
//
//   D[i][j] = bf16_rn( sum_c  sA[c][i] * sB(c, j) * sum_{t in chunk c} A[i][t] * B[j][t] )
//
// A and B hold E4M3 codes; the contraction axis is cut into 128-wide chunks,
// each with its own FP32 scales: one per row of A (1x128 activation tiles) and,
// for B, either one per 128-column block (128x128 weight blocks, "scalar" mode)
// or one per column (1x128 tiles of the other operand, "vector" mode). This is
// the fine-grained block scaling the Puro-2B recipe takes from DeepSeek-V3
// (Puro-2B article on en.roboind.com, section "FP8 takes advantage of the
// RTX 5090's low precision efficiency"): every chunk's partial product is
// accumulated by the tensor core in FP32, then promoted into an FP32 register
// accumulator with the product of the two chunk scales.
//
// Structure (one 128 x BN output tile per CTA):
//   warp 0      TMA producer: A tile 128x128, B tile BNx128 (K-major) or
//               128xBN (MN-major), the chunk's A scales (and B scales in vector
//               mode) into a STAGES-deep shared-memory ring;
//   warp 1      allocates TMEM; one thread issues 4 tcgen05.mma (K = 32 each)
//               per chunk into one of two TMEM accumulators (double buffer);
//   warps 4..   promotion: each warp owns 32 TMEM lanes (= 32 output rows) and
//               128 columns; per chunk it loads the partial sums with
//               tcgen05.ld, frees the TMEM buffer and does
//               acc = fma(partial, sA * sB, acc) in registers; at the end the
//               accumulators are rounded to BF16, staged in shared memory
//               (128-byte swizzle) and written with TMA stores (rows or columns
//               outside D are dropped by the TMA unit).
// Every mbarrier wait is bounded (see mbar_wait); a timeout sets the library's
// device status word and the kernel unwinds without hanging.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace bfp8 {

template <int BN_, int STAGES_, bool B_MN_, bool SB_VEC_>
struct GemmConfig {
    static constexpr int BM = 128;
    static constexpr int BN = BN_;
    static constexpr int BK = 128;
    static constexpr int STAGES = STAGES_;
    static constexpr bool B_MN = B_MN_;      // B stored MN-major (contraction axis strided)
    static constexpr bool SB_VEC = SB_VEC_;  // B scales per column (else per 128-column block)
    static constexpr int PROMO_WG = BN / 128;
    static constexpr int PROMO_WARPS = 4 * PROMO_WG;
    static constexpr int THREADS = 128 + 32 * PROMO_WARPS;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int SA_BYTES = BM * 4;
    static constexpr int SB_BYTES = SB_VEC ? BN * 4 : 0;
    static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES + SA_BYTES + SB_BYTES;
    // shared-memory layout (offsets from a 1024-byte-aligned base)
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SB = OFF_SA + STAGES * SA_BYTES;
    static constexpr int OFF_BAR = OFF_SB + STAGES * SB_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
    // epilogue staging (reuses the operand ring once the main loop is done):
    // per promotion warpgroup two 64-column slabs of 128 rows x 128 bytes
    static constexpr int SLAB_BYTES = 128 * 128;
    static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
    static_assert(PROMO_WG * 2 * SLAB_BYTES <= STAGES * (A_BYTES + B_BYTES), "staging must fit in the ring");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct GemmArgs {
    int gm, gn, num_chunks;
    const float* sb_scalar;   // scalar mode: sB(c, j) = sb_scalar[(j/128) * sb_col_stride + c * sb_chunk_stride]
    int64_t sb_col_stride, sb_chunk_stride;
    unsigned* status;
};

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    bfp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                     const __grid_constant__ CUtensorMap tmD, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + Cfg::OFF_A;
    uint8_t* sB = smem + Cfg::OFF_B;
    float* sSA = reinterpret_cast<float*>(smem + Cfg::OFF_SA);
    float* sSB = reinterpret_cast<float*>(smem + Cfg::OFF_SB);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + Cfg::STAGES;
    uint64_t* tfull = bars + 2 * Cfg::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* mma_done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * Cfg::BN;
    const int m0 = blockIdx.y * Cfg::BM;
    const int nc = args.num_chunks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + Cfg::PROMO_WARPS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::PROMO_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmSA);
        if (Cfg::SB_VEC)
            tma_prefetch_desc(&tmSB);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        tmem_alloc<Cfg::TMEM_COLS>(tmem_slot);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nc; ++c) {
                const int s = c % Cfg::STAGES;
                const uint32_t ph = (c / Cfg::STAGES) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, args.status))
                    break;
                mbar_arrive_expect_tx(&full[s], Cfg::TX_BYTES);
                tma_load_2d(sA + s * Cfg::A_BYTES, &tmA, &full[s], c * Cfg::BK, m0);
                if (Cfg::B_MN) {
#pragma unroll
                    for (int a = 0; a < Cfg::BN / 128; ++a)
                        tma_load_2d(sB + s * Cfg::B_BYTES + a * 128 * Cfg::BK, &tmB, &full[s], n0 + a * 128,
                                    c * Cfg::BK);
                } else {
                    tma_load_2d(sB + s * Cfg::B_BYTES, &tmB, &full[s], c * Cfg::BK, n0);
                }
                tma_load_2d(sSA + s * Cfg::BM, &tmSA, &full[s], m0, c);
                if (Cfg::SB_VEC)
                    tma_load_2d(sSB + s * Cfg::BN, &tmSB, &full[s], n0, c);
                ++issued;
            }
            // make sure no copy is still landing in shared memory before exit
            for (int c = issued - Cfg::STAGES < 0 ? 0 : issued - Cfg::STAGES; c < issued; ++c) {
                volatile int never = 0;
                mbar_wait(&full[c % Cfg::STAGES], (c / Cfg::STAGES) & 1, &never, args.status);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(Cfg::BM, Cfg::BN, Cfg::B_MN);
            const uint32_t a_base = smem_u32(sA);
            const uint32_t b_base = smem_u32(sB);
            for (int c = 0; c < nc; ++c) {
                const int s = c % Cfg::STAGES;
                const uint32_t ph = (c / Cfg::STAGES) & 1;
                const int b = c & 1;
                const uint32_t bph = (c >> 1) & 1;
                if (!mbar_wait(&full[s], ph, abort_flag, args.status))
                    break;
                if (!mbar_wait(&tempty[b], bph ^ 1, abort_flag, args.status))
                    break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * Cfg::BN;
#pragma unroll
                for (int kk = 0; kk < Cfg::BK / 32; ++kk) {
                    const uint64_t ad = smem_desc_sw128(a_base + s * Cfg::A_BYTES + kk * 32, 16, 1024);
                    const uint64_t bd =
                        Cfg::B_MN ? smem_desc_sw128(b_base + s * Cfg::B_BYTES + kk * 32 * 128, 128 * Cfg::BK, 1024)
                                  : smem_desc_sw128(b_base + s * Cfg::B_BYTES + kk * 32, 16, 1024);
                    mma_e4m3(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&empty[s]);
                mma_commit(&tfull[b]);
            }
            // all issued MMAs must be complete before TMEM is released
            mma_commit(mma_done);
            volatile int never = 0;
            mbar_wait(mma_done, 0, &never, args.status);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- promotion + epilogue
        const int pw = warp - 4;            // 0 .. PROMO_WARPS-1
        const int g = pw >> 2;              // which 128-column half of the tile
        const int quarter = warp & 3;       // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const int col0 = n0 + g * 128;      // first output column of this warpgroup
        const bool cols_valid = col0 < args.gn;

        float acc[128];
#pragma unroll
        for (int i = 0; i < 128; ++i)
            acc[i] = 0.0f;

        // scalar-mode B scale for chunk c (same for the whole warpgroup)
        auto load_sb = [&](int c) -> float {
            if (Cfg::SB_VEC || !cols_valid || c >= nc)
                return 0.0f;
            return __ldg(args.sb_scalar + (int64_t)(col0 / 128) * args.sb_col_stride + (int64_t)c * args.sb_chunk_stride);
        };
        float sb_next = load_sb(0);
        bool ok = true;
        for (int c = 0; c < nc; ++c) {
            const int s = c % Cfg::STAGES;
            const uint32_t ph = (c / Cfg::STAGES) & 1;
            const int b = c & 1;
            const uint32_t bph = (c >> 1) & 1;
            const float sb_c = sb_next;
            sb_next = load_sb(c + 1);
            if (!mbar_wait(&tfull[b], bph, abort_flag, args.status)) {
                ok = false;
                break;
            }
            // the scales in stage s landed with full[s]; its phase cannot move on
            // before this warp arrives on empty[s], so this wait returns at once
            if (!mbar_wait(&full[s], ph, abort_flag, args.status)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const float sa = sSA[s * Cfg::BM + row];
            const uint32_t t_base = tmem_base + ((uint32_t)(quarter * 32) << 16) + b * Cfg::BN + g * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_base + j * 32, r);
                tmem_ld_wait();
                if (j == 3) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&tempty[b]);
                }
                if (Cfg::SB_VEC) {
                    const float* sbv = sSB + s * Cfg::BN + g * 128 + j * 32;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        acc[j * 32 + i] = fmaf(__uint_as_float(r[i]) * sbv[i], sa, acc[j * 32 + i]);
                } else {
                    const float sc = sa * sb_c;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        acc[j * 32 + i] = fmaf(__uint_as_float(r[i]), sc, acc[j * 32 + i]);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[s]);
        }
        // all promotion warps take the same decision on whether to write the tile
        const bool give_up = named_barrier_or(1, 32 * Cfg::PROMO_WARPS, !ok || *abort_flag != 0);
        if (!give_up) {
            // BF16 epilogue: two 64-column slabs per warpgroup, 128-byte swizzled
            uint8_t* stage_base = smem + g * 2 * Cfg::SLAB_BYTES;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint8_t* slab = stage_base + h * Cfg::SLAB_BYTES;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float* a = acc + h * 64 + k * 8;
                    uint4 pk;
                    pk.x = cvt_bf16x2(a[0], a[1]);
                    pk.y = cvt_bf16x2(a[2], a[3]);
                    pk.z = cvt_bf16x2(a[4], a[5]);
                    pk.w = cvt_bf16x2(a[6], a[7]);
                    *reinterpret_cast<uint4*>(slab + row * 128 + ((k ^ (row & 7)) * 16)) = pk;
                }
            }
            fence_proxy_async_smem();
            named_barrier_sync(2 + g, 128);
            if (quarter == 0 && lane == 0 && cols_valid) {
                tma_store_2d(&tmD, stage_base, col0, m0);
                if (col0 + 64 < args.gn)
                    tma_store_2d(&tmD, stage_base + Cfg::SLAB_BYTES, col0 + 64, m0);
                tma_store_commit();
                tma_store_wait_read_all();
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<Cfg::TMEM_COLS>(tmem_base);
    }
}

}  // namespace bfp8
