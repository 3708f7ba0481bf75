// Blockwise-FP8 quantisers: BF16 in, E4M3 codes plus one FP32 scale per tile out.
//
// The Puro-2B recipe runs its main linear layers in FP8 with DeepSeek-V3's
// fine-grained block quantisation (Puro-2B article on en.roboind.com, section
// "FP8 takes advantage of the RTX 5090's low precision efficiency"). The
// convention implemented here: activation tiles of 1x128 along the contraction
// axis, weight blocks of 128x128, scale s = fl32(amax / 448), code =
// e4m3_rn_satfinite(fl32(x / s)); an all-zero tile gets s = 0 and signed-zero
// codes. Both divisions are IEEE binary32 divisions (__fdiv_rn), so codes and
// scales are reproducible bit for bit.
//
// All three kernels are HBM-bound (2 B read + 1 B written per element): reads
// are 16-byte vector loads that cover whole 128-byte lines, amax reductions
// use warp shuffles (or a shared-memory column pass in the transposed kernel).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace bfp8 {

// Scale of a tile from its amax; 0 for an all-zero tile.
__device__ __forceinline__ float tile_scale(float amax)
{
    return __fdiv_rn(amax, 448.0f);
}

// Codes of two BF16 values (packed in one word) under scale s.
__device__ __forceinline__ uint32_t codes2(uint32_t w, float s)
{
    if (s == 0.0f) {
        // signed zeros: the sign bits of the two inputs
        return ((w >> 8) & 0x80u) | ((w >> 16) & 0x8000u);
    }
    return cvt_e4m3x2(__fdiv_rn(bf16_lo(w), s), __fdiv_rn(bf16_hi(w), s));
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
__device__ __forceinline__ uint2 codes8(const uint4& v, float s)
{
    uint2 o;
    o.x = codes2(v.x, s) | (codes2(v.y, s) << 16);
    o.y = codes2(v.z, s) | (codes2(v.w, s) << 16);
    return o;
}

// ---------------------------------------------------------------------------
// 1x128 activation tiles along the columns of x [R][C] (C a multiple of 128).
// 16 threads own one tile (8 values each); a warp covers two neighbouring
// tiles, i.e. 512 contiguous bytes of a row. Each thread handles UNROLL tiles
// (loads issued first for memory-level parallelism).
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
        float a = amax_v4(v[u]);
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        const int64_t t = first + u * 16;
        if (t < ntiles) {
            const int64_t r = t / nchunks, c = t - r * nchunks;
            const float sc = tile_scale(a);
            *reinterpret_cast<uint2*>(q + r * ldq + c * 128 + sub * 8) = codes8(v[u], sc);
            if (sub == 0)
                s[c * lds + r] = sc;
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
    const float sc = tile_scale(a);
    uint8_t* qb = q + (bi * 128 + r0) * ldq + bj * 128 + cg * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        *reinterpret_cast<uint2*>(qb + (int64_t)(16 * i) * ldq) = codes8(v[i], sc);
    if (tid == 0)
        s[bi * kblocks + bj] = sc;
}

// ---------------------------------------------------------------------------
// Transposed 1x128 tiles: tiles run down the columns of x [R][C] (along R, the
// contraction axis of the weight-gradient GEMM); codes are written transposed,
// qt [C][R128] (ldqt), scales st [R128/128][C] (ldst). One CTA per 128x128
// input block: the block is staged row-major in shared memory (coalesced
// 16-byte loads, zero rows past R), then warp w takes rows 32 (w%4) .. +31 of
// the column pairs 64 (w/4) + 2 lane, +1 (conflict-free 4-byte reads). The
// four row quarters combine their partial amax through shared memory. Pad
// rows R <= r < R128 hold +0 and so get code 0x00.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_transpose_kernel(const uint16_t* __restrict__ x, int64_t R,
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

    const int warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    const int col = (warp >> 2) * 64 + 2 * lane;  // first of the thread's two columns
    uint32_t wv[32];
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        wv[i] = tile[quarter * 32 + i][col >> 1];
        a0 = fmaxf(a0, fabsf(bf16_lo(wv[i])));
        a1 = fmaxf(a1, fabsf(bf16_hi(wv[i])));
    }
    *reinterpret_cast<float2*>(&part[quarter][col]) = make_float2(a0, a1);
    __syncthreads();
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
        const float2 p = *reinterpret_cast<const float2*>(&part[qq][col]);
        a0 = fmaxf(a0, p.x);
        a1 = fmaxf(a1, p.y);
    }
    const float s0 = tile_scale(a0), s1 = tile_scale(a1);

    // column col: low halves; column col+1: high halves. 32 rows -> 32 codes each.
    uint32_t c0[8], c1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t lo01 = codes2(__byte_perm(wv[4 * j], wv[4 * j + 1], 0x5410), s0);
        const uint32_t lo23 = codes2(__byte_perm(wv[4 * j + 2], wv[4 * j + 3], 0x5410), s0);
        const uint32_t hi01 = codes2(__byte_perm(wv[4 * j], wv[4 * j + 1], 0x7632), s1);
        const uint32_t hi23 = codes2(__byte_perm(wv[4 * j + 2], wv[4 * j + 3], 0x7632), s1);
        c0[j] = lo01 | (lo23 << 16);
        c1[j] = hi01 | (hi23 << 16);
    }
    uint8_t* out0 = qt + (cb * 128 + col) * ldqt + rb * 128 + quarter * 32;
    uint8_t* out1 = out0 + ldqt;
    reinterpret_cast<uint4*>(out0)[0] = make_uint4(c0[0], c0[1], c0[2], c0[3]);
    reinterpret_cast<uint4*>(out0)[1] = make_uint4(c0[4], c0[5], c0[6], c0[7]);
    reinterpret_cast<uint4*>(out1)[0] = make_uint4(c1[0], c1[1], c1[2], c1[3]);
    reinterpret_cast<uint4*>(out1)[1] = make_uint4(c1[4], c1[5], c1[6], c1[7]);
    if (quarter == 0)
        *reinterpret_cast<float2*>(st + rb * ldst + cb * 128 + col) = make_float2(s0, s1);
}

}  // namespace bfp8
