// BF16 GEMM with a scaled-sum epilogue on tcgen05 (sm_103a), for the Newton-Schulz
// iterations of the MuonH update (Puro-2B article on en.roboind.com, section "From
// ordinary learning to effective learning": the update is standardised on top of
// Muon, whose orthogonalisation runs these products):
//
//   D[m][n] = bf16_rn( alpha * sum_k A[m][k] * B(k, n)  +  beta * C[m][n] )
//
// A is BF16 [M][K] with K contiguous; B is BF16 either [N][K] (K contiguous, B(k, n)
// = B[n][k]) or [K][N] (N contiguous, B(k, n) = B[k][n]); C (optional, beta != 0) and
// D are BF16 [M][N]. The products are summed by the tensor core in FP32 over the whole
// contraction (no per-chunk scaling here), in TMEM; the epilogue applies alpha and
// beta in FP32 and rounds once to BF16.
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles in a static round-robin.
//   warp 0      TMA producer: a ring of STAGES stages of 64-deep K slices
//               (A 128 x 64, B 256 x 64, 128-byte swizzle);
//   warp 1      allocates TMEM (2 x 256 columns) and issues, from one thread, four
//               tcgen05.mma.kind::f16 (K = 16) per stage into the tile's accumulator;
//               consecutive tiles alternate between the two accumulators, so the
//               epilogue of one tile overlaps the MMAs of the next;
//   warps 4..7  epilogue: warp w reads TMEM lanes 32 (w%4) .. +31 (rows) in
//               32-column pieces, adds beta * C read from global memory, rounds to
//               BF16 into a 128-byte-swizzled shared-memory slab and stores it with TMA.
// Every mbarrier wait is bounded (mbar_wait); a timeout sets the library's device
// status word and the kernel unwinds.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace bfp8 {

template <bool B_MN_>
struct Bf16GemmConfig {
    static constexpr int BM = 128;
    static constexpr int BN = 256;
    static constexpr int BK = 64;        // K elements per stage (128 bytes of BF16)
    static constexpr int STAGES = 3;
    static constexpr bool B_MN = B_MN_;  // B stored [K][N]
    static constexpr int THREADS = 256;
    static constexpr int EPI_WARPS = 4;
    static constexpr int NBUF = 2;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr uint32_t OP_TX = A_BYTES + B_BYTES;
    static constexpr int BOX_BYTES = 32 * 128;                     // 32 rows x 64 BF16 columns
    static constexpr int OUT_BYTES = EPI_WARPS * (BN / 64) * BOX_BYTES;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_OUT = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_OUT + OUT_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * NBUF + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

struct Bf16GemmArgs {
    int gm, gn, gk;
    int tiles_m, tiles_n, kblocks;
    float alpha, beta;
    const uint16_t* c;  // beta * C is added when c != nullptr
    int64_t ldc;
    unsigned* status;
    unsigned long long wait_ns;
    int stall;  // test switch: the producer issues no copies
};

// Instruction descriptor of tcgen05.mma .kind::f16 with BF16 A and B and an FP32
// accumulator; A K-major, B K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool b_mn_major)
{
    return (1u << 4)                          // D format: F32
           | (1u << 7) | (1u << 10)           // A, B format: BF16
           | (0u << 15)                       // A: K-major
           | ((b_mn_major ? 1u : 0u) << 16)   // B major-ness
           | ((N >> 3) << 17)                 // N / 8
           | ((M >> 4) << 24);                // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T for BF16 operands, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <class Cfg>
__device__ __forceinline__ void bf16_tile_origin(const Bf16GemmArgs& args, int t, int& m0, int& n0)
{
    const int id = static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x);
    m0 = (id % args.tiles_m) * Cfg::BM;
    n0 = (id / args.tiles_m) * Cfg::BN;
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    bf16_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmD, const Bf16GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + Cfg::OFF_A;
    uint8_t* sB = smem + Cfg::OFF_B;
    uint8_t* sOut = smem + Cfg::OFF_OUT;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* full = bars;                  // stage landed (TMA)
    uint64_t* empty = full + Cfg::STAGES;   // stage consumed (MMA commit)
    uint64_t* tfull = empty + Cfg::STAGES;  // accumulator holds a finished tile
    uint64_t* tempty = tfull + Cfg::NBUF;   // accumulator read out by the epilogue
    uint64_t* mma_done = tempty + Cfg::NBUF;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_tiles = args.tiles_m * args.tiles_n;
    const int cta = static_cast<int>(blockIdx.x);
    const int my_tiles = total_tiles > cta ? (total_tiles - 1 - cta) / static_cast<int>(gridDim.x) + 1 : 0;
    const int nkb = args.kblocks;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < Cfg::NBUF; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        tmem_alloc<512>(tmem_slot);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const int total = args.stall ? 0 : my_tiles * nkb;
            int issued = 0, t = 0, kb = 0, m0 = 0, n0 = 0;
            bf16_tile_origin<Cfg>(args, 0, m0, n0);
            for (int g = 0; g < total; ++g) {
                const int s = g % Cfg::STAGES;
                if (!mbar_wait(&empty[s], ((g / Cfg::STAGES) & 1) ^ 1, abort_flag, args.status, args.wait_ns))
                    break;
                mbar_arrive_expect_tx(&full[s], Cfg::OP_TX);
                const int k0 = kb * Cfg::BK;
                tma_load_2d(sA + s * Cfg::A_BYTES, &tmA, &full[s], k0, m0);
                if (Cfg::B_MN) {
                    // four boxes of 64 N-columns x 64 K-rows
#pragma unroll
                    for (int a = 0; a < Cfg::BN / 64; ++a)
                        tma_load_2d(sB + s * Cfg::B_BYTES + a * 64 * Cfg::BK * 2, &tmB, &full[s], n0 + a * 64, k0);
                } else {
                    tma_load_2d(sB + s * Cfg::B_BYTES, &tmB, &full[s], k0, n0);
                }
                ++issued;
                if (++kb == nkb) {
                    kb = 0;
                    ++t;
                    bf16_tile_origin<Cfg>(args, t, m0, n0);
                }
            }
            volatile int never = 0;
            for (int g = issued - Cfg::STAGES < 0 ? 0 : issued - Cfg::STAGES; g < issued; ++g)
                mbar_wait(&full[g % Cfg::STAGES], (g / Cfg::STAGES) & 1, &never, args.status, args.wait_ns);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(Cfg::BM, Cfg::BN, Cfg::B_MN);
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
            // MN-major B: 64-column boxes of 64 K-rows x 128 bytes, 8 KB apart
            const uint64_t b_desc0 = Cfg::B_MN ? smem_desc_sw128(smem_u32(sB), 64 * Cfg::BK * 2, 1024)
                                               : smem_desc_sw128(smem_u32(sB), 16, 1024);
            constexpr uint32_t kBStep = (Cfg::B_MN ? 16 * 128 : 32) / 16;  // 16-byte units per K step of 16
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = 0; t < my_tiles && ok; ++t) {
                const int b = t & 1;
                if (!mbar_wait(&tempty[b], ((t >> 1) & 1) ^ 1, abort_flag, args.status, args.wait_ns))
                    break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * Cfg::BN;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[s], ph, abort_flag, args.status, args.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < Cfg::BK / 16; ++kk) {
                        const uint64_t ad = a_desc0 + ((s * Cfg::A_BYTES) >> 4) + kk * 2;
                        const uint64_t bd = b_desc0 + ((s * Cfg::B_BYTES) >> 4) + kk * kBStep;
                        mma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&empty[s]);
                    if (++s == Cfg::STAGES) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                if (ok)
                    mma_commit(&tfull[b]);
            }
            mma_commit(mma_done);
            volatile int never = 0;
            mbar_wait(mma_done, 0, &never, args.status, args.wait_ns);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        uint8_t* my_out = sOut + quarter * (Cfg::BN / 64) * Cfg::BOX_BYTES;
        int m0 = 0, n0 = 0;
        for (int t = 0; t < my_tiles; ++t) {
            bf16_tile_origin<Cfg>(args, t, m0, n0);
            const int b = t & 1;
            if (!mbar_wait(&tfull[b], (t >> 1) & 1, abort_flag, args.status, args.wait_ns))
                break;
            tc_fence_after_sync();
            if (lane == 0)
                tma_store_wait_read_all();  // the previous tile's stores have left the slab
            __syncwarp();
            const int grow = m0 + quarter * 32 + lane;
            const bool row_ok = grow < args.gm;
            const uint16_t* crow = args.c ? args.c + static_cast<int64_t>(grow) * args.ldc + n0 : nullptr;
            const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * Cfg::BN;
#pragma unroll 1
            for (int j = 0; j < Cfg::BN / 32; ++j) {
                uint32_t r[32];
                tmem_ld32_start(t_base + j * 32, r);
                tmem_ld_wait(r);
                if (j == Cfg::BN / 32 - 1) {  // the whole accumulator is in registers
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&tempty[b]);
                }
                // beta * C for these 32 columns (zero past the matrix)
                uint4 cv[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                               make_uint4(0, 0, 0, 0)};
                if (crow && row_ok) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (n0 + j * 32 + q * 8 < args.gn)
                            cv[q] = __ldg(reinterpret_cast<const uint4*>(crow + j * 32 + q * 8));
                }
                uint8_t* box = my_out + (j >> 1) * Cfg::BOX_BYTES;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t cw[4] = {cv[q].x, cv[q].y, cv[q].z, cv[q].w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a0 = __uint_as_float(r[q * 8 + 2 * e]);
                        const float a1 = __uint_as_float(r[q * 8 + 2 * e + 1]);
                        const float v0 = fmaf(args.beta, bf16_lo(cw[e]), args.alpha * a0);
                        const float v1 = fmaf(args.beta, bf16_hi(cw[e]), args.alpha * a1);
                        o[e] = cvt_bf16x2(v0, v1);
                    }
                    // 16-byte chunk (j & 1) * 4 + q of the 128-byte row, swizzled by the row
                    const int chunk = ((j & 1) << 2) + q;
                    *reinterpret_cast<uint4*>(box + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int bx = 0; bx < Cfg::BN / 64; ++bx)
                    if (n0 + bx * 64 < args.gn && m0 + quarter * 32 < args.gm)
                        tma_store_2d(&tmD, my_out + bx * Cfg::BOX_BYTES, n0 + bx * 64, m0 + quarter * 32);
                tma_store_commit();
            }
        }
        if (lane == 0)
            tma_store_wait_read_all();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<512>(tmem_base);
    }
}

}  // namespace bfp8
