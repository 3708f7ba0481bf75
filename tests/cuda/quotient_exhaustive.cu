// Exhaustive check of the quantisers' division-free quotient (quant.cuh) against
// the IEEE binary32 division, over the whole input domain the kernels can see:
// every finite BF16 tile maximum `amax` >= 0 (s = RN(amax/448)) and every finite
// BF16 value x with |x| <= amax, each in the low lane of a packed pair (with
// another admissible value in the high lane, checked as well), exactly as the
// kernels compute it. Two counts, both must be zero:
//   code mismatches: E4M3 code of the quotient differs from that of x / s;
//   quotient mismatches: the quotient's bits (sign included) differ from
//     x / s, counted where |x / s| >= 2^-12 (below 2^-10 every code is a
//     signed zero).
// For an all-zero tile (amax = 0) the definition's quotient is x itself.
// The tile scale comes from the kernels' table path (tile_scale_tab), which is
// also compared field by field with the division-based tile_scale for every
// amax (a mismatch there counts once per value).
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#include "quant.cuh"

__global__ void check(unsigned long long* pairs, unsigned long long* bad, unsigned* first)
{
    __shared__ bfp8::ScaleTables tab;
    bfp8::init_scale_tables(tab);
    __syncthreads();
    const unsigned ab = blockIdx.y;  // amax bit pattern (0 .. largest finite)
    const float amax = __uint_as_float(ab << 16);
    const bfp8::TileScale ts = bfp8::tile_scale_tab(amax, tab);
    const bfp8::TileScale td = bfp8::tile_scale(amax);
    if (blockIdx.x == 0 && threadIdx.x == 0 &&
        (__float_as_uint(ts.s) != __float_as_uint(td.s) || __float_as_uint(ts.sp) != __float_as_uint(td.sp) ||
         __float_as_uint(ts.y) != __float_as_uint(td.y) || ts.pre != td.pre)) {
        const unsigned long long k = atomicAdd(bad, 1ull);
        if (k < 4) {
            first[3 * k] = 0xFFFFFFFFu;  // marks a scale mismatch
            first[3 * k + 1] = ab;
            first[3 * k + 2] = __float_as_uint(ts.s);
        }
    }
    const bfp8::PairScale ps = bfp8::pair_scale(ts, ts);
    unsigned long long n = 0;
    for (unsigned xb = blockIdx.x * blockDim.x + threadIdx.x; xb < 65536u; xb += gridDim.x * blockDim.x) {
        if ((xb & 0x7FFFu) > ab)
            continue;  // |x| > amax never occurs in a tile
        // the value travels in the low lane; a second value (any other admissible one) in the high lane
        unsigned xb2 = (xb * 40503u + 7u) & 0xFFFFu;
        if ((xb2 & 0x7FFFu) > ab)
            xb2 &= 0x8000u;
        const uint32_t w = xb | (xb2 << 16);
        // the kernels' sequence: the negated pair, the signed quotient, its codes
        const uint64_t na = bfp8::unpack2_neg(w);
        const uint64_t q = ps.scaled ? bfp8::quotient2<true>(na, ps) : bfp8::quotient2<false>(na, ps);
        const uint32_t code = bfp8::cvt_e4m3x4(q, 0);
        const unsigned vals[2] = {xb, xb2};
#pragma unroll
        for (int lane = 0; lane < 2; ++lane) {
            const float x = __uint_as_float(vals[lane] << 16);
            const float ql = __uint_as_float(static_cast<uint32_t>(q >> (32 * lane)));  // x / s
            const float d = ts.s == 0.0f ? x : __fdiv_rn(x, ts.s);                    // the definition
            ++n;
            const uint32_t want = bfp8::cvt_e4m3x2(d, 0.0f) & 0xFFu;
            const bool code_differs = ((code >> (8 * lane)) & 0xFFu) != want;
            const bool quot_differs = fabsf(d) >= 0x1p-12f && __float_as_uint(ql) != __float_as_uint(d);
            if (code_differs || quot_differs) {
                const unsigned long long k = atomicAdd(bad, 1ull);
                if (k < 4) {
                    first[3 * k] = vals[lane];
                    first[3 * k + 1] = ab;
                    first[3 * k + 2] = __float_as_uint(ql);
                }
            }
        }
    }
    atomicAdd(pairs, n);
}

int main()
{
    unsigned long long *dpairs = nullptr, *dbad = nullptr;
    unsigned* dfirst = nullptr;
    if (cudaMalloc(&dpairs, 8) != cudaSuccess || cudaMalloc(&dbad, 8) != cudaSuccess ||
        cudaMalloc(&dfirst, 12 * sizeof(unsigned)) != cudaSuccess)
        return 3;
    cudaMemset(dpairs, 0, 8);
    cudaMemset(dbad, 0, 8);
    const dim3 grid(32, 0x7F80);  // x blocks, every finite amax pattern 0x0000 .. 0x7F7F
    check<<<grid, 256>>>(dpairs, dbad, dfirst);
    unsigned long long pairs = 0, bad = 0;
    unsigned first[12] = {};
    cudaError_t err = cudaMemcpy(&pairs, dpairs, 8, cudaMemcpyDeviceToHost);
    if (err == cudaSuccess)
        err = cudaMemcpy(&bad, dbad, 8, cudaMemcpyDeviceToHost);
    if (err == cudaSuccess)
        err = cudaMemcpy(first, dfirst, sizeof first, cudaMemcpyDeviceToHost);
    printf("pairs %llu mismatches %llu status %s\n", pairs, bad, cudaGetErrorString(err));
    for (unsigned i = 0; i < bad && i < 4; ++i)
        printf("  x=%04x amax=%04x quotient=%08x\n", first[3 * i], first[3 * i + 1], first[3 * i + 2]);
    cudaFree(dpairs);
    cudaFree(dbad);
    cudaFree(dfirst);
    return (err == cudaSuccess && bad == 0 && pairs > 0) ? 0 : 2;
}
