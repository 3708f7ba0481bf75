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
// Persistent kernel, one CTA per SM, output tiles of 128 x BN visited in a
// static round-robin order (the smaller operand is re-read from L2, the larger
// one streamed once). When the tiles do not fill the last round of the grid,
// that last partial round (the tail) can be split along the contraction axis:
// the whole rounds run in one launch, and a second launch of the same kernel
// in piece mode (SPLIT) cuts the tail tiles' chunks into one contiguous range
// per CTA. Its CTAs start on the SMs that the first launch frees (a
// programmatic dependent launch: the pieces need nothing from the whole
// tiles). A piece that covers a whole tile is stored as usual; every other
// piece is stored as an FP32 partial tile in a caller workspace, two slots per
// CTA (its first and its last tail tile), and gemm_tail_reduce_kernel adds
// the partial tiles of each split tile in CTA order and stores it in BF16. So
// the tail costs about (tail tiles / CTAs) of a round instead of a whole one,
// and the result is deterministic. Two shared-memory rings:
//   operand ring (STAGES deep): the A tile 128x128 and the B tile (BNx128
//     K-major, or 128-column boxes of an MN-major operand) of one chunk; a
//     stage is handed back to the producer by the MMA completion alone;
//   scale ring (SSTAGES deep): the scales of a group of SGROUP chunks of one
//     tile (128 A scales per chunk; BN B scales per chunk in vector mode, one
//     per 128 columns in scalar mode); a stage is handed back by the promotion
//     warps once per group, so that their per-chunk work holds one barrier
//     wait (the TMEM buffer) instead of two.
// Warp roles:
//   warp 0      TMA producer of the operand ring;
//   warp 1      allocates TMEM; one thread issues 4 tcgen05.mma (K = 32 each)
//               per chunk into one of two TMEM accumulators of BN columns;
//   warp 2      producer of the scale ring (TMA for the per-row A scales; plain
//               loads for the B scales, shared with warp 3 for per-column ones,
//               which it stores permuted for the promotion's 16x256b layout);
//   warps 4..   promotion (8 warps; 12 with 192-wide tiles): warp w owns
//               TMEM lanes 32 (w%4) .. +31 (output rows) and BN/(PW/4)
//               columns; per chunk it reads the partial sums with tcgen05.ld
//               (scalar B scales: 32x32b, in quarters of 32 columns, later
//               quarters loading while earlier ones are promoted; per-column B
//               scales: 16x256b, in two 64-column blocks), releases the TMEM
//               buffer once its last load has landed, and accumulates
//               acc += partial * (sA * sB)  in FP32
//               registers with packed two-lane FP32 instructions (scalar FP32
//               instructions issued at this rate halve the tensor core's MMA
//               rate on sm_103; the packed form leaves it at full speed); after
//               the last chunk of a
//               tile it rounds acc to BF16, stages it in its own 128-byte-
//               swizzled shared-memory slab and issues TMA stores (the TMA unit
//               drops rows and columns outside D), overlapping the MMAs of the
//               next tile. The accumulate epilogue instead stages acc as FP32
//               and has the TMA unit add it into an FP32 D (D += acc).
// With BN = 256 the promotion warps need more than the 168 registers a
// 384-thread CTA gets; setmaxnreg moves registers from the producer/MMA
// warpgroup to the promotion warpgroups (56/224, or 40/232 with per-column
// B scales), within the launch budget of 384 x 168 (12 promotion warps at
// BN = 192: 56/152 within 512 x 128).
// Every mbarrier wait is bounded (mbar_wait); a timeout sets the library's
// device status word and the kernel unwinds without hanging.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace bfp8 {

// Epilogue kinds: what the promotion warps do with a finished tile.
enum GemmEpilogue {
    EPI_BF16_TMA = 1,  // round to BF16, stage in shared memory, TMA store (default)
    EPI_F32_ADD = 2,   // keep FP32, stage in shared memory, TMA reduce-add into an FP32 D
};

template <int BN_, int STAGES_, bool B_MN_, bool SB_VEC_, int EPI_ = EPI_BF16_TMA, int PW_ = 8>
struct GemmConfig {
    static constexpr int BM = 128;
    static constexpr int BN = BN_;
    static constexpr int BK = 128;
    static constexpr int STAGES = STAGES_;
    static constexpr int SGROUP = 4;   // chunks per scale stage
    static constexpr int SSTAGES = 2;  // scale stages
    static constexpr bool B_MN = B_MN_;      // B stored MN-major (contraction axis strided)
    static constexpr bool SB_VEC = SB_VEC_;  // B scales per column (else per 128-column block)
    // epilogue: EPI_BF16_TMA stages BF16 tiles in shared memory and stores them
    // with TMA; EPI_F32_ADD stages FP32 boxes in the same slab and adds them into
    // an FP32 D with TMA reduce-add (D += result, no BF16 rounding)
    static constexpr int EPI = EPI_;
    // Promotion warps: PW/4 column groups per TMEM lane quarter. More warps hide the
    // TMEM-load latency behind other warps' arithmetic; fewer leave more registers.
    static constexpr int PROMO_WARPS = PW_;
    static constexpr int GROUPS = PW_ / 4;
    static constexpr int CPW = BN / GROUPS;  // output columns per promotion warp
    static constexpr int THREADS = 128 + 32 * PROMO_WARPS;
    static constexpr bool REG_SPLIT = (BN >= 192);
    // TMEM accumulator buffers: as many BN-column buffers as the 512 columns hold
    // (2 at BN = 256, 4 at BN = 128), i.e. that many chunks in flight between the
    // MMA issuer and the promotion warps
    static constexpr int NBUF = 512 / BN;
    // TMEM columns between buffers: 192-wide accumulators start on 256-column boundaries
    static constexpr int BUF_STRIDE = BN == 192 ? 256 : BN;
    static constexpr int TMEM_COLS = 512;
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int SA_BYTES = BM * 4;               // A scales of one chunk
    // Vector-mode B scales of one chunk, stored permuted for the promotion's
    // 16x256b TMEM layout (thread i holds columns 8g + 2(i%4), +1 of its column
    // group): per column group h, per lane class q4 = i % 4, the 2G scales of that
    // class's columns (G = CPW / 8 column pairs), each class padded by 4 floats so
    // that the four classes' 16-byte reads fall on distinct banks.
    static constexpr int SBV_G = CPW / 8;
    static constexpr int SBV_QSTRIDE = 2 * SBV_G + 4;
    static constexpr int SBV_HSTRIDE = 4 * SBV_QSTRIDE;
    static constexpr int SBV_CHUNK = GROUPS * SBV_HSTRIDE;  // floats per chunk
    static constexpr int SB_BYTES = SB_VEC ? SBV_CHUNK * 4 : 0;
    // scalar-mode B scales of one chunk: the 128-column blocks a tile touches (a
    // 192-wide tile at a multiple of 192 touches two)
    static constexpr int SBS_PER_CHUNK = BN == 128 ? 1 : 2;
    static constexpr uint32_t OP_TX = A_BYTES + B_BYTES;
    static constexpr uint32_t SC_TX = SGROUP * SA_BYTES;  // TMA bytes of one scale stage (A scales)
    // scale-producer warps: with per-column B scales, warps 2 and 3 each fetch half of
    // a group's column scales with plain loads, all in flight at once
    static constexpr int SCALE_WARPS = SB_VEC ? 2 : 1;
    // epilogue staging: per promotion warp CPW/64 boxes of 32 rows x 128 bytes
    // (64 BF16 or 32 FP32 columns; 4 KB, 128-byte swizzle)
    static constexpr int BOX_BYTES = 32 * 128;
    static constexpr int STAGE_OUT_BYTES = PROMO_WARPS * (CPW / 64) * BOX_BYTES;
    // shared-memory layout (offsets from a 1024-byte-aligned base)
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_OUT = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SA = OFF_OUT + STAGE_OUT_BYTES;
    static constexpr int OFF_SB = OFF_SA + SSTAGES * SGROUP * SA_BYTES;
    static constexpr int OFF_SBS = OFF_SB + SSTAGES * SGROUP * SB_BYTES;
    static constexpr int OFF_BAR = (OFF_SBS + SSTAGES * SGROUP * SBS_PER_CHUNK * 4 + 7) / 8 * 8;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * SSTAGES + 2 * NBUF + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
    static_assert(BN == 128 || BN == 192 || BN == 256, "BN must be 128, 192 or 256");
    static_assert(BN != 192 || (!B_MN && CPW == 64), "192-wide tiles: K-major B, 64 columns per promotion warp");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    // registers per thread at launch (65536 / THREADS, rounded down to a multiple of 8)
    static constexpr int LAUNCH_REGS = (65536 / THREADS) / 8 * 8;
    // setmaxnreg split between the producer/MMA warpgroup and the two promotion
    // warpgroups, chosen so that neither side spills (per-column B scales: the
    // promotion's 16x256b path needs 232, and the producers then fit in 40)
    static constexpr int REG_LOW = PW_ == 12 ? 56 : (SB_VEC ? 40 : 56);
    static constexpr int REG_HIGH = PW_ == 12 ? 152 : (SB_VEC ? 232 : 224);
    static_assert(PW_ == 8 || PW_ == 12, "8 or 12 promotion warps");
    static_assert(CPW % 64 == 0, "promotion works on pairs of 32-column quarters");
    static_assert(!REG_SPLIT || 128 * REG_LOW + 32 * PW_ * REG_HIGH <= THREADS * LAUNCH_REGS, "register split");
};

struct GemmArgs {
    int gm, gn, num_chunks;
    int tiles_m, tiles_n;
    int n_fastest;            // tile order: 1 = sweep the N tiles of a row block first
    const float* sb_scalar;   // scalar mode: sB(c, j) = sb_scalar[(j/128) * sb_col_stride + c * sb_chunk_stride]
    int64_t sb_col_stride, sb_chunk_stride;
    const float* sb_vec;      // vector mode: sB(c, j) = sb_vec[c * ld_sb + j]
    int64_t ld_sb;
    unsigned* status;
    unsigned long long wait_ns;  // limit of one mbarrier wait
    int stall;                   // test switch: the operand producer issues no copies
    // Tiles 0 .. tail_tile0 - 1 are whole tiles, handed out round-robin by the
    // whole-tile launch. The piece-mode launch cuts the tail_units =
    // (tiles - tail_tile0) * num_chunks chunks of the other tiles into gridDim.x
    // equal contiguous ranges; pieces that are not a whole tile go to ws as FP32
    // partial tiles, [2 * gridDim.x][BM][BN] row-major (through the tensor map
    // tmW): slot 2i for CTA i's first tail tile, 2i + 1 for its last one.
    int tail_tile0;
    long long tail_units;
};

// The tail range of chunk units of CTA `cta` out of `ncta`.
__host__ __device__ __forceinline__ void tail_range(long long units, int cta, int ncta, long long& u0, long long& u1)
{
    u0 = units * cta / ncta;
    u1 = units * (cta + 1) / ncta;
}

// Origin of the t-th tile of this CTA: tiles are handed out in a static
// round-robin over the CTAs.
template <class Cfg>
__device__ __forceinline__ void tile_origin(const GemmArgs& args, int t, int& m0, int& n0)
{
    const int id = static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x);
    int mb, nb;
    if (args.n_fastest) {
        nb = id % args.tiles_n;
        mb = id / args.tiles_n;
    } else {
        mb = id % args.tiles_m;
        nb = id / args.tiles_m;
    }
    m0 = mb * Cfg::BM;
    n0 = nb * Cfg::BN;
}

// The t-th piece of work of this CTA: whole-tile mode, its t-th tile (chunks
// 0 .. nc - 1); piece mode, the t-th tile its tail range touches, chunks
// c0 .. c1 - 1 of it, and the piece's workspace slot (-1: the whole tile).
template <class Cfg, bool SPLIT>
__device__ __forceinline__ void piece_origin(const GemmArgs& args, int t, int& m0, int& n0, int& c0, int& c1,
                                             int& slot)
{
    if constexpr (!SPLIT) {
        tile_origin<Cfg>(args, t, m0, n0);
        c0 = 0;
        c1 = args.num_chunks;
        slot = -1;
    } else {
        const int nc = args.num_chunks;
        long long u0, u1;
        tail_range(args.tail_units, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), u0, u1);
        const int j = static_cast<int>(u0 / nc) + t;  // tile of the tail
        const long long base = static_cast<long long>(j) * nc;
        c0 = u0 > base ? static_cast<int>(u0 - base) : 0;
        c1 = u1 - base < nc ? static_cast<int>(u1 - base) : nc;
        slot = (c0 == 0 && c1 == nc) ? -1 : 2 * static_cast<int>(blockIdx.x) + (t == 0 ? 0 : 1);
        const int id = args.tail_tile0 + j;
        int mb, nb;
        if (args.n_fastest) {
            nb = id % args.tiles_n;
            mb = id / args.tiles_n;
        } else {
            mb = id % args.tiles_m;
            nb = id / args.tiles_m;
        }
        m0 = mb * Cfg::BM;
        n0 = nb * Cfg::BN;
    }
}

template <class Cfg, bool SPLIT = false>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    bfp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ CUtensorMap tmW, const GemmArgs args)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem + Cfg::OFF_A;
    uint8_t* sB = smem + Cfg::OFF_B;
    uint8_t* sOut = smem + Cfg::OFF_OUT;
    float* sSA = reinterpret_cast<float*>(smem + Cfg::OFF_SA);
    float* sSB = reinterpret_cast<float*>(smem + Cfg::OFF_SB);
    float* sSBs = reinterpret_cast<float*>(smem + Cfg::OFF_SBS);  // scalar-mode B scales
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::OFF_BAR);
    uint64_t* full = bars;                       // operand stage landed (TMA)
    uint64_t* empty = full + Cfg::STAGES;        // operand stage consumed (MMA commit)
    uint64_t* sfull = empty + Cfg::STAGES;       // scale stage landed (TMA)
    uint64_t* sempty = sfull + Cfg::SSTAGES;     // scale stage consumed (promotion warps)
    uint64_t* tfull = sempty + Cfg::SSTAGES;     // TMEM buffer holds a finished chunk
    uint64_t* tempty = tfull + Cfg::NBUF;        // TMEM buffer read out
    uint64_t* mma_done = tempty + Cfg::NBUF;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nc = args.num_chunks;
    // whole tiles handed out round-robin over the CTAs (whole-tile mode), or this
    // CTA's range of the tail's chunks, in one or more pieces (piece mode)
    const int ncta = static_cast<int>(gridDim.x);
    const int cta = static_cast<int>(blockIdx.x);
    int my_tiles, my_chunks;
    if constexpr (!SPLIT) {
        const int total_tiles = args.tail_tile0;
        my_tiles = total_tiles > cta ? (total_tiles - 1 - cta) / ncta + 1 : 0;
        my_chunks = my_tiles * nc;
    } else {
        long long u0, u1;
        tail_range(args.tail_units, cta, ncta, u0, u1);
        my_chunks = static_cast<int>(u1 - u0);
        my_tiles = u1 > u0 ? static_cast<int>((u1 - 1) / nc - u0 / nc) + 1 : 0;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);  // one MMA completion
        }
        for (int s = 0; s < Cfg::SSTAGES; ++s) {
            mbar_init(&sfull[s], Cfg::SCALE_WARPS);  // one arrival per scale-producer warp
            mbar_init(&sempty[s], Cfg::PROMO_WARPS);
        }
        for (int b = 0; b < Cfg::NBUF; ++b) {
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
        tma_prefetch_desc(&tmD);
        if (SPLIT)
            tma_prefetch_desc(&tmW);
    }
    // The launch after this one on the stream, if it is a programmatic dependent
    // (the piece-mode launch after the whole tiles; the tail reduce after the
    // pieces), may be scheduled from now on.
    grid_launch_dependents();
    if (warp == 1) {
        tmem_alloc<Cfg::TMEM_COLS>(tmem_slot);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    // The register split sits inside each role's branch so that the compiler
    // allocates every role's code under that role's budget.
    if (warp < 4) {
        if (Cfg::REG_SPLIT)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::REG_LOW));
    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            int t = 0, c = 0, c_end = nc, m0 = 0, n0 = 0, slot;
            piece_origin<Cfg, SPLIT>(args, 0, m0, n0, c, c_end, slot);
            // with the test switch on, nothing is loaded: the MMA issuer's first wait
            // runs out, and every role unwinds through its bounded waits
            const int to_issue = args.stall ? 0 : my_chunks;
            for (int g = 0; g < to_issue; ++g) {
                const int s = g % Cfg::STAGES;
                const uint32_t ph = (g / Cfg::STAGES) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, args.status, args.wait_ns))
                    break;
                mbar_arrive_expect_tx(&full[s], Cfg::OP_TX);
                tma_load_2d(sA + s * Cfg::A_BYTES, &tmA, &full[s], c * Cfg::BK, m0);
                if (Cfg::B_MN) {
#pragma unroll
                    for (int a = 0; a < Cfg::BN / 128; ++a)
                        tma_load_2d(sB + s * Cfg::B_BYTES + a * 128 * Cfg::BK, &tmB, &full[s], n0 + a * 128,
                                    c * Cfg::BK);
                } else {
                    tma_load_2d(sB + s * Cfg::B_BYTES, &tmB, &full[s], c * Cfg::BK, n0);
                }
                ++issued;
                if (++c == c_end) {
                    ++t;
                    piece_origin<Cfg, SPLIT>(args, t, m0, n0, c, c_end, slot);
                }
            }
            // make sure no copy is still landing in shared memory before exit: wait
            // for the last phase of every stage that was filled
            volatile int never = 0;
            for (int g = issued - Cfg::STAGES < 0 ? 0 : issued - Cfg::STAGES; g < issued; ++g)
                mbar_wait(&full[g % Cfg::STAGES], (g / Cfg::STAGES) & 1, &never, args.status, args.wait_ns);
        }
    } else if (warp == 2 || (Cfg::SCALE_WARPS == 2 && warp == 3)) {
        // ---------------------------------------------------------------- scale producer
        const int sp = warp - 2;  // this warp's share of the per-column scales
        // Groups of SGROUP chunks of one tile, or of one piece in piece mode (the
        // last group may be shorter: its rows past the end hold other chunks'
        // scales, or TMA's zero fill past the last chunk, and the promotion warps
        // never read them).
        constexpr int NSBS = Cfg::SGROUP * Cfg::SBS_PER_CHUNK;
        static_assert(NSBS <= 32, "one lane per scalar B scale of a group");
        int issued = 0;
        bool ok = true;
        for (int t = 0; t < my_tiles && ok; ++t) {
            int m0, n0, cb, ce, slot;
            piece_origin<Cfg, SPLIT>(args, t, m0, n0, cb, ce, slot);
            for (int c0 = cb; c0 < ce; c0 += Cfg::SGROUP) {
                const int qs = issued % Cfg::SSTAGES;
                const uint32_t qph = (issued / Cfg::SSTAGES) & 1;
                // lane 0 waits and the warp follows its verdict, so that no lane can
                // leave the loop while the others reach the __syncwarp below
                int ready = 1;
                if (lane == 0)
                    ready = mbar_wait(&sempty[qs], qph ^ 1, abort_flag, args.status, args.wait_ns) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, ready, 0)) {
                    ok = false;
                    break;
                }
                if constexpr (Cfg::SB_VEC) {
                    // this warp's half of the group's per-column scales, a column pair
                    // per lane and step, written in the promotion's permuted layout
                    // (zero past the edges)
                    float* dst = sSB + qs * Cfg::SGROUP * Cfg::SBV_CHUNK;
                    constexpr int PAIRS = Cfg::BN / 2;
                    constexpr int HALF = Cfg::SGROUP * PAIRS / 2;
                    static_assert(HALF % 32 == 0, "whole steps of 32 column pairs");
#pragma unroll 4
                    for (int k = 0; k < HALF / 32; ++k) {
                        const int u = sp * HALF + lane + 32 * k;
                        const int cc = u / PAIRS, n = 2 * (u % PAIRS);
                        const int c = c0 + cc;
                        float2 v = make_float2(0.0f, 0.0f);
                        if (c < nc && n0 + n < args.gn)
                            v = __ldg(reinterpret_cast<const float2*>(args.sb_vec + static_cast<int64_t>(c) * args.ld_sb +
                                                                      n0 + n));
                        const int h = n / Cfg::CPW, w = n % Cfg::CPW;
                        *reinterpret_cast<float2*>(dst + cc * Cfg::SBV_CHUNK + h * Cfg::SBV_HSTRIDE +
                                                   ((w & 7) >> 1) * Cfg::SBV_QSTRIDE + 2 * (w >> 3)) = v;
                    }
                    __syncwarp();  // the stores above happen before lane 0's arrive (release)
                } else {
                    // lane i: chunk c0 + i / SBS_PER_CHUNK, the tile's 128-column block i % SBS_PER_CHUNK
                    if (lane < NSBS) {
                        const int c = c0 + lane / Cfg::SBS_PER_CHUNK;
                        const int col = ((n0 >> 7) + lane % Cfg::SBS_PER_CHUNK) * 128;
                        float v = 0.0f;
                        if (c < nc && col < args.gn)
                            v = __ldg(args.sb_scalar + static_cast<int64_t>(col >> 7) * args.sb_col_stride +
                                      static_cast<int64_t>(c) * args.sb_chunk_stride);
                        sSBs[qs * NSBS + lane] = v;
                    }
                    __syncwarp();  // the stores above happen before lane 0's arrive (release)
                }
                if (lane == 0) {
                    if (sp == 0) {
                        mbar_arrive_expect_tx(&sfull[qs], Cfg::SC_TX);
                        tma_load_2d(sSA + qs * Cfg::SGROUP * Cfg::BM, &tmSA, &sfull[qs], m0, c0);
                    } else {
                        mbar_arrive(&sfull[qs]);
                    }
                }
                ++issued;
            }
        }
        // no copy may still be landing in shared memory at exit (warp 2 issued them)
        if (lane == 0 && sp == 0) {
            volatile int never = 0;
            for (int q = issued - Cfg::SSTAGES < 0 ? 0 : issued - Cfg::SSTAGES; q < issued; ++q)
                mbar_wait(&sfull[q % Cfg::SSTAGES], (q / Cfg::SSTAGES) & 1, &never, args.status, args.wait_ns);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(Cfg::BM, Cfg::BN, Cfg::B_MN);
            // Descriptors of stage 0, K step 0; the others differ only in the start
            // address field (bits 0-13 of the low word, in 16-byte units), which never
            // carries over because shared-memory addresses stay below 256 KB. The loop
            // keeps its ring positions as counters, so it issues no integer multiply
            // or division: this thread shares its SM sub-partition with promotion
            // warps whose packed FMAs keep the FMA pipe busy.
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA), 16, 1024);
            const uint64_t b_desc0 = Cfg::B_MN ? smem_desc_sw128(smem_u32(sB), 128 * Cfg::BK, 1024)
                                               : smem_desc_sw128(smem_u32(sB), 16, 1024);
            const uint32_t a_lo = static_cast<uint32_t>(a_desc0), a_hi = static_cast<uint32_t>(a_desc0 >> 32);
            const uint32_t b_lo = static_cast<uint32_t>(b_desc0), b_hi = static_cast<uint32_t>(b_desc0 >> 32);
            constexpr uint32_t kBStep = (Cfg::B_MN ? 32 * 128 : 32) / 16;  // 16-byte units per K step of 32
            int s = 0, b = 0;
            uint32_t ph = 0, bph = 0, a_off = 0, b_off = 0, d_tmem = tmem_base;
            for (int g = 0; g < my_chunks; ++g) {
                if (!mbar_wait(&full[s], ph, abort_flag, args.status, args.wait_ns))
                    break;
                if (!mbar_wait(&tempty[b], bph ^ 1, abort_flag, args.status, args.wait_ns))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < Cfg::BK / 32; ++kk) {
                    uint64_t ad, bd;
                    asm("mov.b64 %0, {%1, %2};" : "=l"(ad) : "r"(a_lo + a_off + kk * 2), "r"(a_hi));
                    asm("mov.b64 %0, {%1, %2};" : "=l"(bd) : "r"(b_lo + b_off + kk * kBStep), "r"(b_hi));
                    mma_e4m3(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(&empty[s]);
                mma_commit(&tfull[b]);
                if (++s == Cfg::STAGES) {
                    s = 0;
                    ph ^= 1;
                    a_off = 0;
                    b_off = 0;
                } else {
                    a_off += Cfg::A_BYTES / 16;
                    b_off += Cfg::B_BYTES / 16;
                }
                if (++b == Cfg::NBUF) {
                    b = 0;
                    bph ^= 1;
                    d_tmem = tmem_base;
                } else {
                    d_tmem += Cfg::BUF_STRIDE;
                }
            }
            // all issued MMAs must be complete before TMEM is released
            mma_commit(mma_done);
            volatile int never = 0;
            mbar_wait(mma_done, 0, &never, args.status, args.wait_ns);
        }
    }
    } else {
        if (Cfg::REG_SPLIT)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::REG_HIGH));
        // ---------------------------------------------------------------- promotion + epilogue
        constexpr int CPW = Cfg::CPW;
        const int pw = warp - 4;            // 0 .. PROMO_WARPS-1
        const int half = pw >> 2;           // which column group of the tile
        const int quarter = warp & 3;       // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        uint8_t* my_out = sOut + pw * (CPW / 64) * Cfg::BOX_BYTES;

        // FP32 accumulators of the thread's row, as packed pairs of neighbouring columns
        uint64_t acc[CPW / 2];
#pragma unroll
        for (int i = 0; i < CPW / 2; ++i)
            acc[i] = 0;

        int t = 0, c = 0, c_end = nc, m0 = 0, n0 = 0, wslot = -1;
        piece_origin<Cfg, SPLIT>(args, 0, m0, n0, c, c_end, wslot);
        int qs = 0, gi = 0;  // scale stage and chunk index within its group
        uint32_t qph = 0;
        for (int g = 0; g < my_chunks; ++g) {
            const int b = g % Cfg::NBUF;
            const uint32_t bph = (g / Cfg::NBUF) & 1;
            if (gi == 0 && !mbar_wait(&sfull[qs], qph, abort_flag, args.status, args.wait_ns))
                break;
            if (!mbar_wait(&tfull[b], bph, abort_flag, args.status, args.wait_ns))
                break;
            tc_fence_after_sync();
            const int slot = qs * Cfg::SGROUP + gi;  // this chunk's row of the scale stage
            const uint32_t t_base =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + b * Cfg::BUF_STRIDE + half * CPW;
            auto release = [&]() {  // to the MMA issuer
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&tempty[b]);
            };
            uint32_t ra[32], rb[32];
            if constexpr (Cfg::SB_VEC) {
                // Per-column B scales. TMEM is read in the 16x256b layout: a load of the
                // warp's lanes 0-15 (ra) or 16-31 (rb) over 64 columns gives thread i
                // the rows i/4 and i/4 + 8 of those lanes and, for each 8-column step,
                // the column pair 2(i%4), +1; so the thread's 128 values are 4 rows x 16
                // column pairs, and it needs the scales of 32 columns, not 128. Both
                // lane halves use the same columns: one 16-byte read serves 16 values.
                constexpr int G = Cfg::SBV_G;
                constexpr int NB = CPW / 64;
                static_assert(NB == 1 || NB == 2, "one or two 64-column blocks per warp");
                uint64_t sa2[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float v = sSA[slot * Cfg::BM + quarter * 32 + (lane >> 2) + 8 * k];
                    sa2[k] = pack_f32x2(v, v);
                }
                const float* sbq = sSB + slot * Cfg::SBV_CHUNK + half * Cfg::SBV_HSTRIDE + (lane & 3) * Cfg::SBV_QSTRIDE;
                auto promote_block = [&](const uint32_t(&lo)[32], const uint32_t(&hi)[32], int j) {
                    const ulonglong2* v2 = reinterpret_cast<const ulonglong2*>(sbq + 16 * j);
#pragma unroll
                    for (int t2 = 0; t2 < 4; ++t2) {
                        const ulonglong2 v = v2[t2];  // scales of pairs 8j + 2t2 (x) and 8j + 2t2 + 1 (y)
                        const int gp = 8 * j + 2 * t2;
                        const int r0 = 8 * t2;        // registers of the 8-column steps 2t2 and 2t2 + 1
                        ffma2(acc[0 * G + gp], fmul2(pair(lo[r0], lo[r0 + 1]), v.x), sa2[0]);
                        ffma2(acc[1 * G + gp], fmul2(pair(lo[r0 + 2], lo[r0 + 3]), v.x), sa2[1]);
                        ffma2(acc[0 * G + gp + 1], fmul2(pair(lo[r0 + 4], lo[r0 + 5]), v.y), sa2[0]);
                        ffma2(acc[1 * G + gp + 1], fmul2(pair(lo[r0 + 6], lo[r0 + 7]), v.y), sa2[1]);
                        ffma2(acc[2 * G + gp], fmul2(pair(hi[r0], hi[r0 + 1]), v.x), sa2[2]);
                        ffma2(acc[3 * G + gp], fmul2(pair(hi[r0 + 2], hi[r0 + 3]), v.x), sa2[3]);
                        ffma2(acc[2 * G + gp + 1], fmul2(pair(hi[r0 + 4], hi[r0 + 5]), v.y), sa2[2]);
                        ffma2(acc[3 * G + gp + 1], fmul2(pair(hi[r0 + 6], hi[r0 + 7]), v.y), sa2[3]);
                    }
                };
                const uint32_t t_hi = t_base + (16u << 16);
                tmem_ld16x256_start(t_base, ra);
                tmem_ld16x256_start(t_hi, rb);
                tmem_ld_wait(ra);
                tmem_ld_wait(rb);
                if constexpr (NB == 1) {
                    release();
                    promote_block(ra, rb, 0);
                } else {
                    promote_block(ra, rb, 0);
                    tmem_ld16x256_start(t_base + 64, ra);
                    tmem_ld16x256_start(t_hi + 64, rb);
                    tmem_ld_wait(ra);
                    tmem_ld_wait(rb);
                    release();
                    promote_block(ra, rb, 1);
                }
            } else {
                // Scalar B scales (one per 128-column block): the 32x32b layout, thread =
                // row, one scale product per chunk. The warp's CPW columns go in quarters
                // of 32 through two register buffers. The first two quarters are loaded
                // together; each later one is loaded into the buffer just promoted, while
                // the other buffer is promoted. The TMEM buffer goes back to the MMA
                // issuer as soon as its last quarter has landed in registers.
                constexpr int NQ = CPW / 32;
                static_assert(NQ == 2 || NQ == 4, "two or four quarters per warp");
                const float sa = sSA[slot * Cfg::BM + row];
                const float sb_c = sSBs[slot * Cfg::SBS_PER_CHUNK + ((n0 + half * CPW) >> 7) - (n0 >> 7)];
                const float sc = sa * sb_c;
                const uint64_t sc2 = pack_f32x2(sc, sc);
                auto promote = [&](const uint32_t(&r)[32], int j) {
                    uint64_t* a = acc + j * 16;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        ffma2(a[i], pair(r[2 * i], r[2 * i + 1]), sc2);
                };
                tmem_ld32_start(t_base, ra);
                tmem_ld32_start(t_base + 32, rb);
                tmem_ld_wait(ra);
                tmem_ld_wait(rb);
                if constexpr (NQ == 2) {
                    release();
                    promote(ra, 0);
                    promote(rb, 1);
                } else {
                    promote(ra, 0);
                    tmem_ld32_start(t_base + 64, ra);
                    promote(rb, 1);
                    tmem_ld32_start(t_base + 96, rb);
                    tmem_ld_wait(ra);
                    tmem_ld_wait(rb);
                    release();
                    promote(ra, 2);
                    promote(rb, 3);
                }
            }
            // the group's last chunk (or the tile's): this warp is done with the stage
            if (gi == Cfg::SGROUP - 1 || c == c_end - 1) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sempty[qs]);
                gi = 0;
                if (++qs == Cfg::SSTAGES) {
                    qs = 0;
                    qph ^= 1;
                }
            } else {
                ++gi;
            }

            if (++c == c_end) {
                // ------------------------------------------------ BF16 epilogue of tile t
                const int col0 = n0 + half * CPW;
                bool f32_piece = false;  // a partial tile of piece mode: FP32 to the workspace
                if constexpr (SPLIT)
                    f32_piece = wslot >= 0;
                if (f32_piece) {
                    // FP32 boxes of 32 columns x 32 rows into the piece's workspace slot
                    // (rows wslot * BM + ..., columns of the tile): the slab holds CPW/64
                    // boxes, so the warp's CPW/32 boxes go out in two rounds.
                    constexpr int SLAB = CPW / 64;
                    const int y0 = wslot * Cfg::BM + quarter * 32;
#pragma unroll
                    for (int round = 0; round < 2; ++round) {
                        if (lane == 0)
                            tma_store_wait_read_all();  // earlier stores have read the slab
                        __syncwarp();
                        if constexpr (Cfg::SB_VEC) {
                            // 16x256b layout (4 rows x G column pairs per thread)
                            constexpr int G = Cfg::SBV_G;
                            const int q4 = lane & 3, rs = lane >> 2;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int r = rs + 8 * k;
#pragma unroll
                                for (int gg = 0; gg < SLAB * 4; ++gg) {
                                    const int chunk16 = 2 * (gg & 3) + (q4 >> 1);
                                    *reinterpret_cast<uint64_t*>(my_out + (gg >> 2) * Cfg::BOX_BYTES + r * 128 +
                                                                 ((chunk16 ^ (r & 7)) << 4) + 8 * (q4 & 1)) =
                                        acc[k * G + round * SLAB * 4 + gg];
                                }
                            }
                        } else {
                            // 32x32b layout: the thread's row; box b holds pairs 16 b .. 16 b + 15
#pragma unroll
                            for (int bx = 0; bx < SLAB; ++bx) {
                                const uint64_t* v = acc + (round * SLAB + bx) * 16;
#pragma unroll
                                for (int q = 0; q < 8; ++q)
                                    *reinterpret_cast<ulonglong2*>(my_out + bx * Cfg::BOX_BYTES + lane * 128 +
                                                                   ((q ^ (lane & 7)) << 4)) =
                                        make_ulonglong2(v[2 * q], v[2 * q + 1]);
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
#pragma unroll
                            for (int bx = 0; bx < SLAB; ++bx)
                                tma_store_2d(&tmW, my_out + bx * Cfg::BOX_BYTES, half * CPW + (round * SLAB + bx) * 32,
                                             y0);
                            tma_store_commit();
                        }
                    }
                } else if constexpr (Cfg::EPI == EPI_F32_ADD) {
                    // FP32 boxes of 32 columns: the slab holds CPW/64 of them, so the
                    // CPW/32 boxes of the row go out in two rounds. The accumulators are
                    // in the 16x256b layout (4 rows x G column pairs per thread): each pair
                    // goes to its row and column of a 128-byte-swizzled box.
                    static_assert(Cfg::SB_VEC, "the FP32 accumulate epilogue serves the weight gradient");
                    constexpr int SLAB = CPW / 64;
                    constexpr int G = Cfg::SBV_G;
                    const int q4 = lane & 3, rs = lane >> 2;
#pragma unroll
                    for (int round = 0; round < 2; ++round) {
                        if (lane == 0)
                            tma_store_wait_read_all();  // earlier adds have read the slab
                        __syncwarp();
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int r = rs + 8 * k;
#pragma unroll
                            for (int gg = 0; gg < SLAB * 4; ++gg) {
                                const int chunk16 = 2 * (gg & 3) + (q4 >> 1);
                                *reinterpret_cast<uint64_t*>(my_out + (gg >> 2) * Cfg::BOX_BYTES + r * 128 +
                                                             ((chunk16 ^ (r & 7)) << 4) + 8 * (q4 & 1)) =
                                    acc[k * G + round * SLAB * 4 + gg];
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
#pragma unroll
                            for (int bx = 0; bx < SLAB; ++bx) {
                                const int x = col0 + (round * SLAB + bx) * 32;
                                if (x < args.gn && m0 + quarter * 32 < args.gm)
                                    tma_reduce_add_2d(&tmD, my_out + bx * Cfg::BOX_BYTES, x, m0 + quarter * 32);
                            }
                            tma_store_commit();
                        }
                    }
                } else {
                    if (lane == 0)
                        tma_store_wait_read_all();  // this warp's previous stores have left the slab
                    __syncwarp();
                    if constexpr (Cfg::SB_VEC) {
                        // 16x256b layout: each BF16 pair goes to its row and column of a
                        // 128-byte-swizzled 32 x 64 box
                        constexpr int G = Cfg::SBV_G;
                        const int q4 = lane & 3, rs = lane >> 2;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int r = rs + 8 * k;
#pragma unroll
                            for (int gp = 0; gp < G; ++gp)
                                *reinterpret_cast<uint32_t*>(my_out + (gp >> 3) * Cfg::BOX_BYTES + r * 128 +
                                                             (((gp & 7) ^ (r & 7)) << 4) + 4 * q4) =
                                    cvt_bf16x2(acc[k * G + gp]);
                        }
                    } else {
#pragma unroll
                        for (int bx = 0; bx < CPW / 64; ++bx) {
                            uint8_t* box = my_out + bx * Cfg::BOX_BYTES;
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const uint64_t* v = acc + bx * 32 + k * 4;
                                uint4 pk;
                                pk.x = cvt_bf16x2(v[0]);
                                pk.y = cvt_bf16x2(v[1]);
                                pk.z = cvt_bf16x2(v[2]);
                                pk.w = cvt_bf16x2(v[3]);
                                *reinterpret_cast<uint4*>(box + lane * 128 + ((k ^ (lane & 7)) * 16)) = pk;
                            }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
#pragma unroll
                        for (int bx = 0; bx < CPW / 64; ++bx)
                            if (col0 + bx * 64 < args.gn && m0 + quarter * 32 < args.gm)
                                tma_store_2d(&tmD, my_out + bx * Cfg::BOX_BYTES, col0 + bx * 64, m0 + quarter * 32);
                        tma_store_commit();
                    }
                }
#pragma unroll
                for (int i = 0; i < CPW / 2; ++i)
                    acc[i] = 0;
                ++t;
                piece_origin<Cfg, SPLIT>(args, t, m0, n0, c, c_end, wslot);
            }
        }
        if (lane == 0)
            tma_store_wait_read_all();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<Cfg::TMEM_COLS>(tmem_base);
    }
    // piece mode runs beside the whole-tile launch before it; it completes only
    // after that launch has, so that work after it on the stream finds every tile
    if constexpr (SPLIT)
        grid_dependency_wait();
}

// ---------------------------------------------------------------------------
// The split tail tiles: tile j of the tail (tile tail_tile0 + j) was cut between
// the CTAs whose ranges meet its chunk units j nc .. (j + 1) nc - 1; each wrote
// its piece to its slot (2i for the CTA's first tail tile, 2i + 1 for its last).
// This kernel adds the pieces in CTA order and stores the BF16 tile. A tile that
// one CTA did whole was stored by that CTA and is skipped; CTAs between the
// first and the last owner of a tile whose range is empty (possible when the
// tail has fewer chunks than there are CTAs) wrote nothing and are skipped.
// It is launched as a programmatic dependent of the piece-mode GEMM, so its
// CTAs are staged while the GEMM finishes and start as soon as it has
// completed. One CTA of 256 threads per 8 rows of a tail tile.
struct TailReduceArgs {
    const float* ws;
    uint16_t* d;  // BF16 output
    long long ldd;
    int gm, gn, num_chunks, tail_tile0, grid;
    long long tail_units;
    int tiles_m, tiles_n, n_fastest;
};

// The CTA (of `grid`) whose tail range holds chunk unit u.
__device__ __forceinline__ int tail_owner(long long u, long long units, int grid)
{
    return static_cast<int>(((u + 1) * grid - 1) / units);
}

template <int BN>
__global__ void __launch_bounds__(256) gemm_tail_reduce_kernel(const TailReduceArgs a)
{
    constexpr int BM = 128, ROWS = 8, VEC = 4, MAXP = 256;
    __shared__ int slots[MAXP];
    // launched as a programmatic dependent of the GEMM: wait until that grid has
    // completed and its workspace stores are visible
    grid_dependency_wait();
    const int j = blockIdx.x;
    const long long first = static_cast<long long>(j) * a.num_chunks;
    const int i0 = tail_owner(first, a.tail_units, a.grid);
    const int i1 = tail_owner(first + a.num_chunks - 1, a.tail_units, a.grid);
    if (i0 == i1)
        return;
    // the tile's pieces in CTA order, one CTA per thread: slot of CTA i0 + t (2i for
    // its first tail tile, 2i + 1 for its last), or -1 for a CTA with an empty range
    const int np = i1 - i0 + 1;  // at most the grid size, which the host keeps <= MAXP
    if (threadIdx.x < np) {
        const int i = i0 + threadIdx.x;
        long long s0, s1;
        tail_range(a.tail_units, i, a.grid, s0, s1);
        slots[threadIdx.x] = s0 == s1 ? -1 : 2 * i + (s0 / a.num_chunks == j ? 0 : 1);
    }
    __syncthreads();
    const int id = a.tail_tile0 + j;
    int mb, nb;
    if (a.n_fastest) {
        nb = id % a.tiles_n;
        mb = id / a.tiles_n;
    } else {
        mb = id % a.tiles_m;
        nb = id / a.tiles_m;
    }
    const int m0 = mb * BM, n0 = nb * BN;
    for (int v = threadIdx.x; v < ROWS * BN / VEC; v += 256) {  // 4-column groups of this CTA's rows
        const int r = blockIdx.y * ROWS + v / (BN / VEC), col = (v % (BN / VEC)) * VEC;
        const float* base = a.ws + r * BN + col;
        float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int p = 0; p < np; p += 4) {
            // four pieces' loads in flight, added in order
            float4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (p + u < np && slots[p + u] >= 0)
                    q[u] = *reinterpret_cast<const float4*>(base + static_cast<long long>(slots[p + u]) * (BM * BN));
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (p + u < np && slots[p + u] >= 0) {
                    sum.x += q[u].x;
                    sum.y += q[u].y;
                    sum.z += q[u].z;
                    sum.w += q[u].w;
                }
        }
        const int gr = m0 + r, gc = n0 + col;
        if (gr < a.gm && gc < a.gn) {
            uint2 o;
            o.x = cvt_bf16x2(sum.x, sum.y);
            o.y = cvt_bf16x2(sum.z, sum.w);
            *reinterpret_cast<uint2*>(a.d + static_cast<long long>(gr) * a.ldd + gc) = o;
        }
    }
}

}  // namespace bfp8
