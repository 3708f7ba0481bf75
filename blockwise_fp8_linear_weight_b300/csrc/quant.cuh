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
// neither the quotient nor any rounding. The steps are odd in a (every
// rounding is to nearest-even), so the quotient of a signed x carries x's
// sign. They run on -x and -y, with the remainder's sign flipped:
//   q0 = (-x)(-y),  r' = fma(q, s, -x) = -(x - q s),  q = fma(r', -y, q),
// which gives the same values as the textbook form but keeps the sign of a
// zero: for x = -0 the remainder is +0 and q = (+0)(-y) + (-0) = -0, where the
// textbook fma(r, y, q) would give +0. So q = RN(x / s) bit for bit, signed
// zeros included, and the E4M3 conversion (which keeps the sign of values that
// round to zero) gives 0x80 for -0 and for negative quotients below the
// smallest code. An all-zero tile (s = 0) runs the same instructions with y = 0
// and yields the inputs' signed zeros. Where a is so small against s that a
// remainder still underflows, the quotient is below 2^-40 and its code is a
// signed zero either way.
//
// The kernels are meant to be HBM-bound (2 B read + 1 B written per element and
// per code layout): blocks arrive by TMA, shared-memory reads are 16-byte vector
// loads (4-byte column reads for the transposed layout), amax reductions use warp
// shuffles and a shared-memory combine across warps.
#pragma once

#include <cstdint>
#include <type_traits>

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

// Tile scales without a division: for a BF16 amax = (1 + i/128) * 2^(E - 127)
// (biased exponent E, 7-bit mantissa i) and 448 = 1.75 * 2^8,
//   amax / 448 = ((1 + i/128) / 1.75) * 2^(E - 135),
// and rounding commutes with the power-of-two factor whenever the result is a
// normal binary32 number, which holds for E >= 10. So s = T1[i] * 2^(E - 135)
// with T1[i] = RN((1 + i/128) / 1.75), and y = RN(1 / sp) = T2[i] * 2^-(E - 135 + P)
// with T2[i] = RN(1 / T1[i]) and P = 64 for pre-scaled tiles: two table reads
// and integer additions to the exponent field. Each CTA fills the 128-entry
// tables with IEEE divisions when it starts; zero and tiny maxima (E < 10,
// scales that are zero or subnormal) take tile_scale's divisions.
struct ScaleTables {
    uint32_t t1[128];  // bits of RN((1 + i/128) / 1.75)
    uint32_t t2[128];  // bits of RN(1 / T1[i])
};

__device__ __forceinline__ void init_scale_tables(ScaleTables& t)
{
    for (int i = threadIdx.x; i < 128; i += blockDim.x) {
        const float q = __fdiv_rn(1.0f + static_cast<float>(i) * 0.0078125f, 1.75f);
        t.t1[i] = __float_as_uint(q);
        t.t2[i] = __float_as_uint(__frcp_rn(q));
    }
}

__device__ __forceinline__ TileScale tile_scale_tab(float amax, const ScaleTables& t)
{
    const uint32_t ab = __float_as_uint(amax);
    const int E = static_cast<int>(ab >> 23);
    if (E < 10)
        return tile_scale(amax);
    const uint32_t i = (ab >> 16) & 0x7Fu;
    const uint32_t t1 = t.t1[i];
    const uint32_t k = static_cast<uint32_t>(E - 135) << 23;  // exponent offset (wraps for E < 135)
    const uint32_t sbits = t1 + k;
    const bool scaled = (sbits >> 23) < 67u;  // s < 2^-60
    const uint32_t kp = scaled ? k + (64u << 23) : k;
    TileScale r;
    r.s = __uint_as_float(sbits);
    r.pre = scaled ? 0x1p64f : 1.0f;
    r.sp = __uint_as_float(t1 + kp);
    r.y = __uint_as_float(t.t2[i] - kp);
    return r;
}

// ---------------------------------------------------------------------------
// Packed form used by the kernels: two values per 64-bit register pair, so the
// five quotient steps (one product, two Markstein corrections) are five packed
// FP32 instructions per pair (six for tiles that need the 2^64 pre-scaling,
// which take a separate code path). Lane i of every operand belongs to value i.
// ---------------------------------------------------------------------------
struct PairScale {
    uint64_t sp;   // {sp_lo, sp_hi}
    uint64_t ny;   // {-y_lo, -y_hi}
    uint64_t pre;  // {pre_lo, pre_hi}
    bool scaled;   // some lane has pre != 1
};

// One scale for both lanes, from a broadcast (y, signed sp): sp > 0 marks a
// pre-scaled tile, and the FMA operand is |sp| either way.
__device__ __forceinline__ PairScale pair_scale_bcast(float y, float sp_signed)
{
    PairScale p;
    const float sp = fabsf(sp_signed);
    p.sp = pack_f32x2(sp, sp);
    p.ny = pack_f32x2(-y, -y);
    p.pre = pack_f32x2(0x1p64f, 0x1p64f);
    p.scaled = sp_signed > 0.0f;
    return p;
}

__device__ __forceinline__ PairScale pair_scale(const TileScale& lo, const TileScale& hi)
{
    PairScale p;
    p.sp = pack_f32x2(lo.sp, hi.sp);
    p.ny = pack_f32x2(-lo.y, -hi.y);
    p.pre = pack_f32x2(lo.pre, hi.pre);
    p.scaled = lo.pre != 1.0f || hi.pre != 1.0f;
    return p;
}

// a packed BF16 pair as a packed FP32 pair, negated (exact; -0 for +0)
__device__ __forceinline__ uint64_t unpack2_neg(uint32_t w)
{
    return pack_f32x2(__uint_as_float((w << 16) ^ 0x80000000u), __uint_as_float((w & 0xFFFF0000u) ^ 0x80000000u));
}

// RN(a / s) lane-wise for a packed pair, from na = -a (SCALED: the tile pair has
// a 2^64 pre-scaling factor; the kernels branch on PairScale::scaled)
template <bool SCALED>
__device__ __forceinline__ uint64_t quotient2(uint64_t na, const PairScale& ps)
{
    if (SCALED)
        na = fmul2(na, ps.pre);
    uint64_t q = fmul2(na, ps.ny);  // q = a y
    uint64_t r = na;
    ffma2(r, q, ps.sp);  // r' = q s - a
    ffma2(q, r, ps.ny);  // q = q - r' y = q + (a - q s) y
    r = na;
    ffma2(r, q, ps.sp);
    ffma2(q, r, ps.ny);
    return q;
}

// E4M3 codes of a packed FP32 pair: low value in bits 0-7, high in bits 8-15
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint64_t q)
{
    uint16_t r;
    asm("{\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 {lo, hi}, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 %0, hi, lo;\n\t}"
        : "=h"(r)
        : "l"(q));
    return r;
}

// E4M3 codes of two packed FP32 pairs as one word: bytes q01.lo, q01.hi, q23.lo, q23.hi
__device__ __forceinline__ uint32_t cvt_e4m3x4(uint64_t q01, uint64_t q23)
{
    uint32_t r;
    asm("{\n\t.reg .f32 a0, a1, b0, b1;\n\t.reg .b16 c0, c1;\n\t"
        "mov.b64 {a0, a1}, %1;\n\tmov.b64 {b0, b1}, %2;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 c0, a1, a0;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 c1, b1, b0;\n\t"
        "mov.b32 %0, {c0, c1};\n\t}"
        : "=r"(r)
        : "l"(q01), "l"(q23));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// lane-wise max(|a|, |b|) of two BF16 pairs, each lane's sign bit the XOR of
// the inputs' (callers clear the sign bits once, after the last step)
__device__ __forceinline__ uint32_t bf16x2_maxabs(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// lane-wise max of |values| over the 4 BF16 pairs of a 16-byte vector
__device__ __forceinline__ uint32_t absmax_pairs(const uint4& v)
{
    return bf16x2_maxabs(bf16x2_maxabs(v.x, v.y), bf16x2_maxabs(v.z, v.w)) & 0x7FFF7FFFu;
}

// 8 BF16 values sharing one tile scale -> 8 codes (first value in the low byte)
template <bool SCALED>
__device__ __forceinline__ uint2 codes8_packed(const uint4& v, const PairScale& ps)
{
    const uint32_t lo =
        cvt_e4m3x4(quotient2<SCALED>(unpack2_neg(v.x), ps), quotient2<SCALED>(unpack2_neg(v.y), ps));
    const uint32_t hi =
        cvt_e4m3x4(quotient2<SCALED>(unpack2_neg(v.z), ps), quotient2<SCALED>(unpack2_neg(v.w), ps));
    return make_uint2(lo, hi);
}

__device__ __forceinline__ uint2 codes8(const uint4& v, const PairScale& ps)
{
    return ps.scaled ? codes8_packed<true>(v, ps) : codes8_packed<false>(v, ps);
}

// ---------------------------------------------------------------------------
// Column pass (transposed tiles). The 128x128 BF16 block sits row-major in
// shared memory (rows past R hold +0). Warp w takes rows 32 (w%4) .. +31 of
// the column pair 64 (w/4) + 2 lane, +1 (conflict-free 4-byte reads, one BF16
// pair per read: the two columns travel as the two lanes of every packed
// operation, each with its own scale); the four row quarters combine their
// amax through shared memory. Codes go to qt [C][R128] (row = input column),
// scales to st [R128/128][C]. Pad rows hold +0 and so get code 0x00.
// ---------------------------------------------------------------------------
template <bool SCALED>
__device__ __forceinline__ void column_encode(const uint32_t (*tile)[64], int quarter, int cw, const PairScale& ps,
                                              uint32_t (&c0)[8], uint32_t (&c1)[8])
{
    // rows in groups of 4: the row pair words w0..w3 give the codes of (row, col)
    // and (row, col + 1); cvt_e4m3x4 packs rows 0-1 and rows 2-3, byte_perm
    // regroups them by column
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int r = quarter * 32 + 4 * j;
        const uint32_t w0 = tile[r][cw], w1 = tile[r + 1][cw], w2 = tile[r + 2][cw], w3 = tile[r + 3][cw];
        const uint32_t a =
            cvt_e4m3x4(quotient2<SCALED>(unpack2_neg(w0), ps), quotient2<SCALED>(unpack2_neg(w1), ps));
        const uint32_t b =
            cvt_e4m3x4(quotient2<SCALED>(unpack2_neg(w2), ps), quotient2<SCALED>(unpack2_neg(w3), ps));
        c0[j] = __byte_perm(a, b, 0x6420);
        c1[j] = __byte_perm(a, b, 0x7531);
    }
}

__device__ __forceinline__ void column_pass(const uint32_t (*tile)[64], uint32_t (*part)[64], const ScaleTables& tab,
                                            int64_t cb, int64_t rb, uint8_t* __restrict__ qt, int64_t ldqt,
                                            float* __restrict__ st, int64_t ldst)
{
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;
    const int cw = (warp >> 2) * 32 + lane;  // the thread's column pair (word index in a row)
    const int col = 2 * cw;                  // first of the thread's two columns
    // lane-wise |max| of the pair over this quarter's 32 rows, combined across quarters
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        m = bf16x2_maxabs(m, tile[quarter * 32 + i][cw]);
    part[quarter][cw] = m & 0x7FFF7FFFu;
    __syncthreads();
    m = bf16x2_max(bf16x2_max(part[0][cw], part[1][cw]), bf16x2_max(part[2][cw], part[3][cw]));
    const TileScale s0 = tile_scale_tab(bf16_lo(m), tab), s1 = tile_scale_tab(bf16_hi(m), tab);
    const PairScale ps = pair_scale(s0, s1);

    uint32_t c0[8], c1[8];
    if (ps.scaled)
        column_encode<true>(tile, quarter, cw, ps, c0, c1);
    else
        column_encode<false>(tile, quarter, cw, ps, c0, c1);
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
// Persistent, TMA-fed quantiser over 128x128 blocks of a BF16 matrix x [R][C]
// (C a multiple of 128; rows past R read as +0 through the tensor map). Each
// CTA walks the blocks blockIdx.x, blockIdx.x + gridDim.x, ...; one thread
// keeps two blocks in flight (double-buffered 32 KB shared-memory tiles filled
// by cp.async.bulk.tensor, completion on an mbarrier) while all 256 threads
// encode the current one, so HBM reads overlap the arithmetic.
//   MODE_ROWS:   1x128 tiles along the columns -> q [R][C], s [C/128][R]
//   MODE_COLS:   1x128 tiles down the rows     -> qt [C][R128], st [R128/128][C]
// (both activation layouts from one read: quant_dual_kernel below)
// ---------------------------------------------------------------------------
enum QuantMode { MODE_ROWS = 1, MODE_COLS = 2 };

struct QuantArgs {
    int64_t R, nblk_c, nblocks;
    uint8_t* q;
    int64_t ldq;
    float* s;
    int64_t lds;
    uint8_t* qt;
    int64_t ldqt;
    float* st;
    int64_t ldst;
    unsigned* status;
    unsigned long long wait_ns;  // limit of one mbarrier wait
    int stall;                   // test switch: no block is loaded
};

// Row pass over 8 row tiles per half-warp (1x128 tiles along the columns):
// codes to q [R][C], scales to s [C/128][R].
__device__ __forceinline__ void row_tiles8(const uint32_t (*tile)[64], const ScaleTables& stab, const QuantArgs& a,
                                           int64_t rb, int64_t cb, int r_local, int rstep)
{
    const int tid = threadIdx.x;
    const int sub = tid & 15;
    // The thread covers rows r_local + rstep j (j = 0..7) of the block, columns
    // 8 (t%16) .. +7; a half-warp owns one row tile per j. The half-warp
    // reduces its 8 tiles at once with a butterfly that halves the number of
    // tiles each lane carries per step (lane bit 3 picks 4 of the 8, bit 2 two
    // of those, bit 1 one), so that lanes 2j and 2j+1 end with tile j's amax;
    // each lane computes that tile's scale, and the encoding pass fetches a
    // tile's scale by shuffle.
    uint32_t m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        m[j] = absmax_pairs(*reinterpret_cast<const uint4*>(&tile[r_local + rstep * j][sub * 4]));
    {
        const bool b3 = sub & 8, b2 = sub & 4, b1 = sub & 2;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t send = b3 ? m[i] : m[i + 4], keep = b3 ? m[i + 4] : m[i];
            m[i] = bf16x2_max(keep, __shfl_xor_sync(0xffffffffu, send, 8));
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t send = b2 ? m[i] : m[i + 2], keep = b2 ? m[i + 2] : m[i];
            m[i] = bf16x2_max(keep, __shfl_xor_sync(0xffffffffu, send, 4));
        }
        const uint32_t send = b1 ? m[0] : m[1], keep = b1 ? m[1] : m[0];
        m[0] = bf16x2_max(keep, __shfl_xor_sync(0xffffffffu, send, 2));
        m[0] = bf16x2_max(m[0], __shfl_xor_sync(0xffffffffu, m[0], 1));
    }
    const TileScale mine = tile_scale_tab(fmaxf(bf16_lo(m[0]), bf16_hi(m[0])), stab);  // tile sub >> 1
    const int lane = tid & 31;
    const int64_t r0 = rb * 128 + r_local;  // the thread's row for j = 0
    // lanes 2j store tile j's scale (row r0 + rstep j of their half-warp)
    if ((sub & 1) == 0 && r0 + rstep * (sub >> 1) < a.R)
        a.s[cb * a.lds + r0 + rstep * (sub >> 1)] = mine.s;
    const float bc_sp = mine.pre != 1.0f ? mine.sp : -mine.sp;  // sign carries the pre-scaling flag
    const int rows_left = static_cast<int>(a.R - r0 > 128 ? 128 : a.R - r0);
    uint8_t* qrow = a.q + r0 * a.ldq + cb * 128 + sub * 8;
    const int64_t qstep = rstep * a.ldq;
#pragma unroll 2
    for (int j = 0; j < 8; ++j) {
        const int src = (lane & 16) | (2 * j);
        const PairScale ps = pair_scale_bcast(__shfl_sync(0xffffffffu, mine.y, src),
                                              __shfl_sync(0xffffffffu, bc_sp, src));
        if (rstep * j < rows_left) {
            const uint4 v = *reinterpret_cast<const uint4*>(&tile[r_local + rstep * j][sub * 4]);
            *reinterpret_cast<uint2*>(qrow) = codes8(v, ps);
        }
        qrow += qstep;
    }
}

// 32 codes (one column of 32 rows) as one 32-byte store: a whole sector per lane.
// dst must be 32-byte aligned.
__device__ __forceinline__ void store_codes32(uint8_t* dst, const uint32_t (&c)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(c[0]), "r"(c[1]),
                 "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(c[5]), "r"(c[6]), "r"(c[7])
                 : "memory");
}

// Column pass by warps 4-7 only (while warps 0-3 do the row pass, in
// quant_dual_kernel): thread
// t' = t - 128 takes the column pair 32 ((t'/32) % 2) + lane over rows
// 64 (t'/64) .. +63; the two row halves combine their amax through shared
// memory behind a barrier of these 128 threads only, which is also their vote
// on whether the block's copy arrived.
// With ST32 every column's 32 codes go out as one 32-byte store (qt and ldqt 32-byte
// aligned), else as two 16-byte stores.
template <bool ST32>
__device__ __forceinline__ bool column_pass_4w(bool ok, const uint32_t (*tile)[64], uint32_t (*part)[64],
                                               const ScaleTables& tab, int64_t cb, int64_t rb,
                                               uint8_t* __restrict__ qt, int64_t ldqt, float* __restrict__ st,
                                               int64_t ldst)
{
    const int t = threadIdx.x - 128;
    const int w = t >> 5, lane = t & 31;
    const int half = w >> 1;
    const int cw = (w & 1) * 32 + lane;
    const int col = 2 * cw;
    if (ok) {
        uint32_t m = 0;
#pragma unroll 16
        for (int i = 0; i < 64; ++i)
            m = bf16x2_maxabs(m, tile[half * 64 + i][cw]);
        part[half][cw] = m & 0x7FFF7FFFu;
    }
    // the four warps combine their halves here, and take one decision on whether the
    // block's copy arrived (a warp whose wait gave up reads nothing and votes no), so
    // that none of them can be left waiting at this barrier for the others
    if (!bar_red_and(1, 128, ok))
        return false;
    const uint32_t m = bf16x2_max(part[0][cw], part[1][cw]);
    const TileScale s0 = tile_scale_tab(bf16_lo(m), tab), s1 = tile_scale_tab(bf16_hi(m), tab);
    const PairScale ps = pair_scale(s0, s1);
    uint8_t* out0 = qt + (cb * 128 + col) * ldqt + rb * 128 + half * 64;
    uint8_t* out1 = out0 + ldqt;
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // rows half*64 + 32 q .. +31
        uint32_t c0[8], c1[8];
        if (ps.scaled)
            column_encode<true>(tile, 2 * half + q, cw, ps, c0, c1);
        else
            column_encode<false>(tile, 2 * half + q, cw, ps, c0, c1);
        if constexpr (ST32) {
            store_codes32(out0 + 32 * q, c0);
            store_codes32(out1 + 32 * q, c1);
        } else {
            reinterpret_cast<uint4*>(out0 + 32 * q)[0] = make_uint4(c0[0], c0[1], c0[2], c0[3]);
            reinterpret_cast<uint4*>(out0 + 32 * q)[1] = make_uint4(c0[4], c0[5], c0[6], c0[7]);
            reinterpret_cast<uint4*>(out1 + 32 * q)[0] = make_uint4(c1[0], c1[1], c1[2], c1[3]);
            reinterpret_cast<uint4*>(out1 + 32 * q)[1] = make_uint4(c1[4], c1[5], c1[6], c1[7]);
        }
    }
    if (half == 0)
        *reinterpret_cast<float2*>(st + rb * ldst + cb * 128 + col) = make_float2(s0.s, s1.s);
    return true;
}

constexpr int kQuantTileBytes = 128 * 128 * 2;
constexpr int kQuantSmemBytes = 2 * kQuantTileBytes + 1024;  // two tiles + alignment slack

template <int MODE>
__global__ void __launch_bounds__(256, 3) quant_blocks_kernel(const __grid_constant__ CUtensorMap tmX, const QuantArgs a)
{
    extern __shared__ uint8_t qsmem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsmem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[2];
    __shared__ __align__(16) uint32_t part[4][64];
    __shared__ ScaleTables stab;
    __shared__ int abort_flag;
    const int tid = threadIdx.x;

    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    const int my_blocks = a.nblocks > first ? static_cast<int>((a.nblocks - 1 - first) / stride + 1) : 0;

    int issued = 0;            // thread 0: blocks whose copy was started
    auto issue = [&](int i) {  // thread 0: load my i-th block into buffer i & 1
        if (a.stall)           // test switch: nothing is loaded, so the first wait runs out
            return;
        ++issued;
        const int64_t b = first + static_cast<int64_t>(i) * stride;
        const int64_t rb = b / a.nblk_c, cb = b - rb * a.nblk_c;
        uint64_t* bar = &full[i & 1];
        mbar_arrive_expect_tx(bar, kQuantTileBytes);
        tma_load_2d(tiles + (i & 1) * kQuantTileBytes, &tmX, bar, static_cast<int32_t>(cb * 128),
                    static_cast<int32_t>(rb * 128));
    };
    init_scale_tables(stab);
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmX);
    }
    __syncthreads();
    if (tid == 0) {
        if (my_blocks > 0)
            issue(0);
        if (my_blocks > 1)
            issue(1);
    }

    int i = 0;
    for (; i < my_blocks; ++i) {
        const int64_t b = first + static_cast<int64_t>(i) * stride;
        const int64_t rb = b / a.nblk_c, cb = b - rb * a.nblk_c;
        // every thread takes the same decision, so no thread can be left at a barrier
        if (!__syncthreads_and(mbar_wait(&full[i & 1], (i >> 1) & 1, &abort_flag, a.status, a.wait_ns)))
            break;
        const uint32_t(*tile)[64] = reinterpret_cast<const uint32_t(*)[64]>(tiles + (i & 1) * kQuantTileBytes);

        if (MODE == MODE_ROWS) {
            row_tiles8(tile, stab, a, rb, cb, tid >> 4, 16);
        }
        if (MODE == MODE_COLS)
            column_pass(tile, part, stab, cb, rb, a.qt, a.ldqt, a.st, a.ldst);
        __syncthreads();  // everyone is done with this buffer (and with part / red)
        if (tid == 0 && i + 2 < my_blocks)
            issue(i + 2);
    }
    // an aborted CTA must not exit while a copy may still land in its shared memory
    if (tid == 0 && i < my_blocks) {
        volatile int never = 0;
        for (int k = i; k < issued && k < i + 2; ++k)
            mbar_wait(&full[k & 1], (k >> 1) & 1, &never, a.status, a.wait_ns);
    }
}

// ---------------------------------------------------------------------------
// Both activation layouts from one read of x (the outputs of MODE_ROWS and
// MODE_COLS together), without block-wide
// barriers: a producer warp (warp 8) keeps NB buffers in flight, each with a
// "full" mbarrier (TMA landed) and an "empty" one (all eight worker warps done
// with it); warps 0-3 run the row pass and warps 4-7 the transposed pass at the
// same time, each warp moving on to the next buffer as soon
// as it is done with the current one. The transposed pass combines its two row
// halves through a scratch array indexed by the block's parity, so a fast warp
// can write the next block's partial maxima while a slow one still reads this
// block's.
// ---------------------------------------------------------------------------
constexpr int kDualWorkers = 8;
constexpr int kDualThreads = 32 * (kDualWorkers + 1);

// The producer warp of the barrier-free block kernels: lane 0 loads this CTA's
// blocks (first = blockIdx.x, stride = gridDim.x) into NB buffers, each refilled
// once all kDualWorkers worker warps have arrived on its "empty" barrier.
template <int NB>
__device__ __forceinline__ void block_producer(const CUtensorMap& tmX, const QuantArgs& a, uint8_t* tiles,
                                               uint64_t* full, uint64_t* empty, volatile int* abort_flag,
                                               int my_blocks)
{
    if ((threadIdx.x & 31) != 0)
        return;
    const int64_t first = blockIdx.x, stride = gridDim.x;
    int issued = 0;
    const int to_issue = a.stall ? 0 : my_blocks;
    for (int i = 0; i < to_issue; ++i) {
        const int b = i % NB;
        // the buffer's previous block (i - NB) has been consumed by every worker
        if (i >= NB && !mbar_wait(&empty[b], ((i / NB) - 1) & 1, abort_flag, a.status, a.wait_ns))
            break;
        const int64_t blk = first + static_cast<int64_t>(i) * stride;
        const int64_t rb = blk / a.nblk_c, cb = blk - rb * a.nblk_c;
        mbar_arrive_expect_tx(&full[b], kQuantTileBytes);
        tma_load_2d(tiles + b * kQuantTileBytes, &tmX, &full[b], static_cast<int32_t>(cb * 128),
                    static_cast<int32_t>(rb * 128));
        ++issued;
    }
    // no copy may still be landing in shared memory at exit
    volatile int never = 0;
    for (int i = issued - NB < 0 ? 0 : issued - NB; i < issued; ++i)
        mbar_wait(&full[i % NB], (i / NB) & 1, &never, a.status, a.wait_ns);
}

template <int NB>
constexpr int dual_smem_bytes()
{
    return NB * kQuantTileBytes + 1024;
}

template <int NB, int MIN_CTAS, bool ST32>
__global__ void __launch_bounds__(kDualThreads, MIN_CTAS)
    quant_dual_kernel(const __grid_constant__ CUtensorMap tmX, const QuantArgs a)
{
    extern __shared__ uint8_t qsmem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsmem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[NB];
    __shared__ __align__(8) uint64_t empty[NB];
    __shared__ __align__(16) uint32_t part[2][2][64];
    __shared__ ScaleTables stab;
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    const int my_blocks = a.nblocks > first ? static_cast<int>((a.nblocks - 1 - first) / stride + 1) : 0;

    init_scale_tables(stab);
    if (tid == 0) {
        for (int b = 0; b < NB; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&empty[b], kDualWorkers);
        }
        abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmX);
    }
    __syncthreads();

    if (warp == kDualWorkers) {
        block_producer<NB>(tmX, a, tiles, full, empty, &abort_flag, my_blocks);
        return;
    }

    for (int i = 0; i < my_blocks; ++i) {
        const int b = i % NB;
        const int64_t blk = first + static_cast<int64_t>(i) * stride;
        const int64_t rb = blk / a.nblk_c, cb = blk - rb * a.nblk_c;
        // every worker waits on the same phase; a wait that gives up sets the abort
        // flag, which ends the others' waits too
        const bool ok = mbar_wait(&full[b], (i / NB) & 1, &abort_flag, a.status, a.wait_ns);
        const uint32_t(*tile)[64] = reinterpret_cast<const uint32_t(*)[64]>(tiles + b * kQuantTileBytes);
        if (warp < 4) {
            if (!ok)
                break;
            row_tiles8(tile, stab, a, rb, cb, tid >> 4, 8);
            row_tiles8(tile, stab, a, rb, cb, (tid >> 4) + 64, 8);
        } else if (!column_pass_4w<ST32>(ok, tile, part[i & 1], stab, cb, rb, a.qt, a.ldqt, a.st, a.ldst)) {
            break;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[b]);
    }
}


// ---------------------------------------------------------------------------
// Weight blocks (128x128, one scale per block) without block-wide barriers on
// the copies: a producer warp (warp 8) keeps NB buffers in flight with full and
// empty mbarriers, as in quant_dual_kernel. Each of the eight worker warps reads
// 16 rows of the block into registers (rows r0 + 16 j, 8 columns per thread),
// hands the buffer back, and votes on one 256-thread named barrier that also
// combines the warps' maxima (scratch indexed by the block's parity, so a fast
// warp can write the next block's maximum while a slow one still reads this
// block's); then it encodes its 16 rows from the registers.
// ---------------------------------------------------------------------------
template <int NB, int MIN_CTAS>
__global__ void __launch_bounds__(kDualThreads, MIN_CTAS)
    quant_weight_kernel(const __grid_constant__ CUtensorMap tmX, const QuantArgs a)
{
    extern __shared__ uint8_t qsmem_raw[];
    uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsmem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[NB];
    __shared__ __align__(8) uint64_t empty[NB];
    __shared__ uint32_t red[2][kDualWorkers];
    __shared__ ScaleTables stab;
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    const int my_blocks = a.nblocks > first ? static_cast<int>((a.nblocks - 1 - first) / stride + 1) : 0;

    init_scale_tables(stab);
    if (tid == 0) {
        for (int b = 0; b < NB; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&empty[b], kDualWorkers);
        }
        abort_flag = 0;
        fence_mbarrier_init();
        tma_prefetch_desc(&tmX);
    }
    __syncthreads();

    if (warp == kDualWorkers) {
        block_producer<NB>(tmX, a, tiles, full, empty, &abort_flag, my_blocks);
        return;
    }

    const int sub = tid & 15, r0 = tid >> 4;  // rows r0 + 16 j, columns 8 sub .. 8 sub + 7
    for (int i = 0; i < my_blocks; ++i) {
        const int b = i % NB;
        const int64_t blk = first + static_cast<int64_t>(i) * stride;
        const int64_t rb = blk / a.nblk_c, cb = blk - rb * a.nblk_c;
        const bool ok = mbar_wait(&full[b], (i / NB) & 1, &abort_flag, a.status, a.wait_ns);
        const uint32_t(*tile)[64] = reinterpret_cast<const uint32_t(*)[64]>(tiles + b * kQuantTileBytes);
        uint4 v[8];
        if (ok) {
            uint32_t m = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[j] = *reinterpret_cast<const uint4*>(&tile[r0 + 16 * j][sub * 4]);
                m = bf16x2_max(m, absmax_pairs(v[j]));
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
                m = bf16x2_max(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (lane == 0)
                red[i & 1][warp] = m;
        }
        // one decision for all workers on whether the copy arrived, and the warps' maxima
        if (!bar_red_and(1, 32 * kDualWorkers, ok))
            break;
        // the block is in registers: the buffer can be refilled while it is encoded
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[b]);
        uint32_t m = red[i & 1][0];
#pragma unroll
        for (int k = 1; k < kDualWorkers; ++k)
            m = bf16x2_max(m, red[i & 1][k]);
        const TileScale ts = tile_scale_tab(fmaxf(bf16_lo(m), bf16_hi(m)), stab);
        const PairScale ps = pair_scale(ts, ts);
        uint8_t* out = a.q + (rb * 128 + r0) * a.ldq + cb * 128 + sub * 8;
        auto encode = [&](auto scaled) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint2*>(out + 16 * j * a.ldq) = codes8_packed<decltype(scaled)::value>(v[j], ps);
        };
        if (ps.scaled)
            encode(std::true_type{});
        else
            encode(std::false_type{});
        if (tid == 0)
            a.s[rb * a.lds + cb] = ts.s;
    }
}

}  // namespace bfp8
