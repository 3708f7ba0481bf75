// Blockwise-FP8 quantisers: BF16 in, E4M3 codes plus one FP32 scale per tile out.
//
// The Puro-2B recipe runs its main linear layers in FP8 with DeepSeek-V3's
// fine-grained block quantisation (Puro-2B article on en.roboind.com, section
// "FP8 takes advantage of the RTX 5090's low precision efficiency"). The
// convention implemented here: activation tiles of 1x128 along the contraction
// axis, weight blocks of 128x128, scale s = fl32(amax / 448), code =
// e4m3_rn_satfinite(fl32(x / s)); an all-zero tile gets s = 0 and signed-zero
// codes. Both divisions are IEEE binary32 divisions, so codes and scales are
// reproducible bit for bit.
//
// Exact quotients without a division instruction per element (Markstein's
// method: P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990; also the Handbook of
// Floating-Point Arithmetic, Muller et al., section on division with an FMA).
// With y = RN(1/s) (one correctly rounded reciprocal per tile) and the
// remainder r = a - s q, which an FMA computes exactly when q is within an ulp
// of a/s and nothing underflows, the step q' = RN(q + r y) returns RN(a/s)
// whenever q is a faithful approximation of a/s. The first product q0 = RN(a y)
// is within 1.5 ulp of a/s, so one step first brings it within a hair of a/s
// (faithful), and a second step makes it the correctly rounded quotient,
// identical to the IEEE division. To keep the remainders clear of the
// subnormal range, tiles with a scale below 2^-60 (including binary32
// subnormal scales) work on a and s both multiplied by 2^64, which changes
// neither the quotient nor any rounding. The quotient is taken of |x| and given
// x's sign afterwards, so that -0 keeps its sign; an all-zero tile (s = 0)
// runs the same instructions with y = 0 and yields the inputs' signed zeros.
// Where a is so small against s that a remainder still underflows, the
// quotient is below 2^-40 and its code is a signed zero either way.
//
// All four kernels are HBM-bound (2 B read + 1 B written per element and per
// code layout): reads are 16-byte vector loads that cover whole 128-byte lines,
// amax reductions use warp shuffles (or a shared-memory column pass for the
// transposed layout).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace bfp8 {

// A tile's scale and what the division-free quotient needs.
struct TileScale {
    float s;    // fl32(amax / 448), 0 for an all-zero tile: the stored scale
    float pre;  // 2^64 for tiny scales, else 1 (applied to both operands)
    float sp;   // s * pre (exact), or 1 for an all-zero tile
    float y;    // RN(1 / sp), or 0 for an all-zero tile
};

__device__ __forceinline__ TileScale tile_scale(float amax)
{
    TileScale t;
    t.s = __fdiv_rn(amax, 448.0f);
    t.pre = t.s < 0x1p-60f ? 0x1p64f : 1.0f;
    t.sp = t.s == 0.0f ? 1.0f : t.s * t.pre;
    t.y = t.s == 0.0f ? 0.0f : __frcp_rn(t.sp);
    return t;
}

// RN(x / s) by two Markstein steps.
__device__ __forceinline__ float quotient(float x, const TileScale& ts)
{
    const float a = fabsf(x) * ts.pre;
    float q = a * ts.y;
    float r = fmaf(-q, ts.sp, a);
    q = fmaf(r, ts.y, q);
    r = fmaf(-q, ts.sp, a);
    q = fmaf(r, ts.y, q);
    return copysignf(q, x);
}

// Codes of N values (N a multiple of 4); out[i] packs codes 4i .. 4i+3, first value in the low byte.
template <int N>
__device__ __forceinline__ void encode(const float (&x)[N], const TileScale& ts, uint32_t (&out)[N / 4])
{
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        t[i] = quotient(x[i], ts);
#pragma unroll
    for (int i = 0; i < N / 4; ++i)
        out[i] = cvt_e4m3x2(t[4 * i], t[4 * i + 1]) | (cvt_e4m3x2(t[4 * i + 2], t[4 * i + 3]) << 16);
}

__device__ __forceinline__ float amax_word(uint32_t w)
{
    return fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w)));
}

__device__ __forceinline__ float amax_v4(const uint4& v)
{
    return fmaxf(fmaxf(amax_word(v.x), amax_word(v.y)), fmaxf(amax_word(v.z), amax_word(v.w)));
}

// 8 BF16 values -> 8 codes (one 64-bit word, first value in the low byte).
__device__ __forceinline__ uint2 codes8(const uint4& v, const TileScale& ts)
{
    const float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                        bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
    uint32_t o[2];
    encode<8>(x, ts, o);
    return make_uint2(o[0], o[1]);
}

// amax over the 16 lanes that share one 1x128 tile (lanes 0-15 or 16-31).
__device__ __forceinline__ float amax16(float a)
{
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    return a;
}

// ---------------------------------------------------------------------------
// 1x128 activation tiles along the columns of x [R][C] (C a multiple of 128).
// 16 threads own one tile (8 values each); a warp covers two neighbouring
// tiles, i.e. 512 contiguous bytes of a row. Each thread handles UNROLL tiles
// (all loads issued first for memory-level parallelism).
// q [R][C] (ldq), s [C/128][R] (lds).
// ---------------------------------------------------------------------------
template <int UNROLL>
__global__ void __launch_bounds__(256) quant_act_kernel(const uint16_t* __restrict__ x, int64_t ldx,
                                                        uint8_t* __restrict__ q, int64_t ldq,
                                                        float* __restrict__ s, int64_t lds,
                                                        int64_t nchunks, int64_t ntiles)
{
    const int sub = threadIdx.x & 15;
    const int64_t first = (int64_t)blockIdx.x * (16 * UNROLL) + (threadIdx.x >> 4);
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const int64_t t = first + u * 16;
        if (t < ntiles) {
            const int64_t r = t / nchunks, c = t - r * nchunks;
            v[u] = ld_stream_v4(x + r * ldx + c * 128 + sub * 8);
        } else {
            v[u] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
        const float a = amax16(amax_v4(v[u]));
        const int64_t t = first + u * 16;
        if (t < ntiles) {
            const int64_t r = t / nchunks, c = t - r * nchunks;
            const TileScale ts = tile_scale(a);
            *reinterpret_cast<uint2*>(q + r * ldq + c * 128 + sub * 8) = codes8(v[u], ts);
            if (sub == 0)
                s[c * lds + r] = ts.s;
        }
    }
}

// ---------------------------------------------------------------------------
// 128x128 weight blocks: one CTA (256 threads) per block. Thread t reads 8
// values of column group t%16 in rows t/16 + 16 i (i < 8); the block amax is
// reduced with shuffles and then across the 8 warps in shared memory.
// q [N][K] (ldq), s [N/128][K/128] dense.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_weight_kernel(const uint16_t* __restrict__ w, int64_t ldw,
                                                           uint8_t* __restrict__ q, int64_t ldq,
                                                           float* __restrict__ s, int64_t kblocks)
{
    __shared__ float red[8];
    const int tid = threadIdx.x;
    const int cg = tid & 15, r0 = tid >> 4;
    const int64_t bi = blockIdx.y, bj = blockIdx.x;
    const uint16_t* base = w + (bi * 128 + r0) * ldw + bj * 128 + cg * 8;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = ld_stream_v4(base + (int64_t)(16 * i) * ldw);
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        a = fmaxf(a, amax_v4(v[i]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    if ((tid & 31) == 0)
        red[tid >> 5] = a;
    __syncthreads();
    a = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
        a = fmaxf(a, red[i]);
    const TileScale ts = tile_scale(a);
    uint8_t* qb = q + (bi * 128 + r0) * ldq + bj * 128 + cg * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        *reinterpret_cast<uint2*>(qb + (int64_t)(16 * i) * ldq) = codes8(v[i], ts);
    if (tid == 0)
        s[bi * kblocks + bj] = ts.s;
}

// ---------------------------------------------------------------------------
// Column pass shared by the transposed and the dual kernel. The 128x128 BF16
// block sits row-major in shared memory (rows past R hold +0). Warp w takes
// rows 32 (w%4) .. +31 of the column pair 64 (w/4) + 2 lane, +1 (conflict-free
// 4-byte reads); the four row quarters combine their amax through shared
// memory. Codes go to qt [C][R128] (row = input column), scales to
// st [R128/128][C]. Pad rows hold +0 and so get code 0x00.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void column_pass(const uint32_t (*tile)[64], float (*part)[128], int64_t cb, int64_t rb,
                                            uint8_t* __restrict__ qt, int64_t ldqt, float* __restrict__ st,
                                            int64_t ldst)
{
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    const int col = (warp >> 2) * 64 + 2 * lane;  // first of the thread's two columns
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t w = tile[quarter * 32 + i][col >> 1];
        a0 = fmaxf(a0, fabsf(bf16_lo(w)));
        a1 = fmaxf(a1, fabsf(bf16_hi(w)));
    }
    *reinterpret_cast<float2*>(&part[quarter][col]) = make_float2(a0, a1);
    __syncthreads();
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const float2 p = *reinterpret_cast<const float2*>(&part[qq][col]);
        a0 = fmaxf(a0, p.x);
        a1 = fmaxf(a1, p.y);
    }
    const TileScale s0 = tile_scale(a0), s1 = tile_scale(a1);

    // column col: low halves; column col+1: high halves. 32 rows -> 32 codes each,
    // re-read from shared memory and encoded 8 at a time to bound register use.
    uint32_t c0[8], c1[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float x0[8], x1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w = tile[quarter * 32 + 8 * j + i][col >> 1];
            x0[i] = bf16_lo(w);
            x1[i] = bf16_hi(w);
        }
        uint32_t o0[2], o1[2];
        encode<8>(x0, s0, o0);
        encode<8>(x1, s1, o1);
        c0[2 * j] = o0[0];
        c0[2 * j + 1] = o0[1];
        c1[2 * j] = o1[0];
        c1[2 * j + 1] = o1[1];
    }
    uint8_t* out0 = qt + (cb * 128 + col) * ldqt + rb * 128 + quarter * 32;
    uint8_t* out1 = out0 + ldqt;
    reinterpret_cast<uint4*>(out0)[0] = make_uint4(c0[0], c0[1], c0[2], c0[3]);
    reinterpret_cast<uint4*>(out0)[1] = make_uint4(c0[4], c0[5], c0[6], c0[7]);
    reinterpret_cast<uint4*>(out1)[0] = make_uint4(c1[0], c1[1], c1[2], c1[3]);
    reinterpret_cast<uint4*>(out1)[1] = make_uint4(c1[4], c1[5], c1[6], c1[7]);
    if (quarter == 0)
        *reinterpret_cast<float2*>(st + rb * ldst + cb * 128 + col) = make_float2(s0.s, s1.s);
}

// ---------------------------------------------------------------------------
// Transposed 1x128 tiles: tiles run down the columns of x [R][C] (along R, the
// contraction axis of the weight-gradient GEMM); codes are written transposed,
// qt [C][R128] (ldqt), scales st [R128/128][C] (ldst). One CTA per 128x128
// input block: the block is staged row-major in shared memory (coalesced
// 16-byte loads, zero rows past R), then the column pass.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 3) quant_transpose_kernel(const uint16_t* __restrict__ x, int64_t R,
                                                              int64_t ldx, uint8_t* __restrict__ qt,
                                                              int64_t ldqt, float* __restrict__ st,
                                                              int64_t ldst)
{
    __shared__ __align__(16) uint32_t tile[128][64];  // 128 rows x 128 bf16
    __shared__ __align__(16) float part[4][128];
    const int tid = threadIdx.x;
    const int64_t cb = blockIdx.x, rb = blockIdx.y;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = tid + 256 * i;
        const int row = idx >> 4, cv = idx & 15;
        const int64_t gr = rb * 128 + row;
        v[i] = (gr < R) ? ld_stream_v4(x + gr * ldx + cb * 128 + cv * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = tid + 256 * i;
        *reinterpret_cast<uint4*>(&tile[idx >> 4][(idx & 15) * 4]) = v[i];
    }
    __syncthreads();
    column_pass(tile, part, cb, rb, qt, ldqt, st, ldst);
}

// ---------------------------------------------------------------------------
// Both layouts of one activation in a single pass over HBM: the 1x128 tiles
// along the columns (q [R][C], s [C/128][R], as quant_act_kernel) and the
// transposed tiles along the rows (qt [C][R128], st [R128/128][C], as
// quant_transpose_kernel). One CTA per 128x128 block; thread t's i-th 16-byte
// load holds 8 values of row t/16 + 16 i, so the 16 lanes of a half-warp own
// one 1x128 row tile and reduce its amax with shuffles while the block is
// staged in shared memory for the column pass.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 3) quant_dual_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t ldx,
                                                         uint8_t* __restrict__ q, int64_t ldq,
                                                         float* __restrict__ s, int64_t lds,
                                                         uint8_t* __restrict__ qt, int64_t ldqt,
                                                         float* __restrict__ st, int64_t ldst)
{
    __shared__ __align__(16) uint32_t tile[128][64];
    __shared__ __align__(16) float part[4][128];
    const int tid = threadIdx.x;
    const int sub = tid & 15;
    const int64_t cb = blockIdx.x, rb = blockIdx.y;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = tid + 256 * i;
        const int row = idx >> 4;
        const int64_t gr = rb * 128 + row;
        v[i] = (gr < R) ? ld_stream_v4(x + gr * ldx + cb * 128 + sub * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int idx = tid + 256 * i;
        *reinterpret_cast<uint4*>(&tile[idx >> 4][sub * 4]) = v[i];
    }
    // row tiles (1x128 along the columns) from the registers
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = (tid >> 4) + 16 * i;
        const int64_t gr = rb * 128 + row;
        const float a = amax16(amax_v4(v[i]));
        if (gr < R) {
            const TileScale ts = tile_scale(a);
            *reinterpret_cast<uint2*>(q + gr * ldq + cb * 128 + sub * 8) = codes8(v[i], ts);
            if (sub == 0)
                s[cb * lds + gr] = ts.s;
        }
    }
    __syncthreads();
    column_pass(tile, part, cb, rb, qt, ldqt, st, ldst);
}

}  // namespace bfp8
