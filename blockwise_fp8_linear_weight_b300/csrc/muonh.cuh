// MuonH update kernels: the reductions and element-wise passes around the
// Newton-Schulz orthogonalisation of a gradient.
//
// The Puro-2B recipe trains with MuonH (Puro-2B article on en.roboind.com,
// section "From ordinary learning to effective learning"): the size of each
// weight update is standardised on top of Muon, and after the update the
// weight is projected back to a fixed radius; the relative update size is a
// preset quantity rather than a drift of the weight norm. Read plainly, with
// U the Newton-Schulz orthogonalisation of the gradient G, a learning rate lr
// and the radius R (Frobenius norms):
//   X0    = G / (|G| + eps)                      (muonh_normalize, BF16 out)
//   U     = Newton-Schulz iterations on X0       (plain BF16 GEMMs)
//   W'    = W - lr R U / |U|                     (relative update size lr)
//   W_new = R W' / |W'|                          (back onto the sphere |W| = R)
// Three passes: |U|^2 (reads U), then |W'|^2 of the FP32 W' = fma(-a, U, W)
// that the last pass writes (reads W and U), then W_new (reads W and U, writes
// W). Summing the squares of W' itself, rather than expanding |W'|^2 as
// |W|^2 - 2 a <W,U> + a^2 |U|^2, keeps the norm free of cancellation: when W'
// is exactly zero the sum is zero and W is left unchanged.
//
// Sums are deterministic: each CTA reduces a fixed set of rows (FP32 within a
// row segment of a thread, FP64 beyond), warps by a fixed butterfly, CTAs by
// a fixed loop over the partials; every launch uses the same grid.
#pragma once

#include <cstdint>

namespace bfp8 {

constexpr int kMuonThreads = 256;

// Sum of three FP64 values over the CTA, in a fixed order; thread 0 returns them.
__device__ __forceinline__ void block_sum3(double& x, double& y, double& z, double (*sh)[3])
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        x += __shfl_xor_sync(0xffffffffu, x, o);
        y += __shfl_xor_sync(0xffffffffu, y, o);
        z += __shfl_xor_sync(0xffffffffu, z, o);
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        sh[warp][0] = x;
        sh[warp][1] = y;
        sh[warp][2] = z;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        x = y = z = 0.0;
        for (int w = 0; w < kMuonThreads / 32; ++w) {
            x += sh[w][0];
            y += sh[w][1];
            z += sh[w][2];
        }
    }
}

// Fixed-order total of component k of the CTA partials [nparts][3].
__device__ __forceinline__ double sum_partials(const double* partials, int nparts, int k)
{
    double s = 0.0;
    for (int i = 0; i < nparts; ++i)
        s += partials[3 * i + k];
    return s;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h)
{
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// partials[blockIdx.x] = (sum of a^2 over the CTA's rows, 0, 0); a FP32 [rows][lda], cols % 4 == 0.
__global__ void __launch_bounds__(kMuonThreads) muonh_sumsq_kernel(const float* __restrict__ a, int64_t rows,
                                                                   int64_t cols, int64_t lda,
                                                                   double* __restrict__ partials)
{
    __shared__ double sh[kMuonThreads / 32][3];
    double acc = 0.0, zero1 = 0.0, zero2 = 0.0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float4* row = reinterpret_cast<const float4*>(a + r * lda);
        float s = 0.0f;
        for (int64_t j = threadIdx.x; j < cols / 4; j += kMuonThreads) {
            const float4 v = row[j];
            s = fmaf(v.x, v.x, s);
            s = fmaf(v.y, v.y, s);
            s = fmaf(v.z, v.z, s);
            s = fmaf(v.w, v.w, s);
        }
        acc += static_cast<double>(s);
    }
    block_sum3(acc, zero1, zero2, sh);
    if (threadIdx.x == 0) {
        partials[3 * blockIdx.x + 0] = acc;
        partials[3 * blockIdx.x + 1] = 0.0;
        partials[3 * blockIdx.x + 2] = 0.0;
    }
}

// x = bf16_rn(a / (sqrt(sum of the partials) + eps)); x BF16 [rows][ldx].
__global__ void __launch_bounds__(kMuonThreads) muonh_scale_bf16_kernel(const float* __restrict__ a, int64_t rows,
                                                                        int64_t cols, int64_t lda,
                                                                        const double* __restrict__ partials,
                                                                        int nparts, float eps,
                                                                        uint16_t* __restrict__ x, int64_t ldx)
{
    __shared__ float inv;
    if (threadIdx.x == 0)
        inv = static_cast<float>(1.0 / (sqrt(sum_partials(partials, nparts, 0)) + static_cast<double>(eps)));
    __syncthreads();
    const float s = inv;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float4* src = reinterpret_cast<const float4*>(a + r * lda);
        uint2* dst = reinterpret_cast<uint2*>(x + r * ldx);
        for (int64_t j = threadIdx.x; j < cols / 4; j += kMuonThreads) {
            const float4 v = src[j];
            dst[j] = make_uint2(f32x2_to_bf16x2(v.x * s, v.y * s), f32x2_to_bf16x2(v.z * s, v.w * s));
        }
    }
}

// partials[blockIdx.x] = (0, 0, sum u^2) over the CTA's rows; u BF16 [rows][ldu].
__global__ void __launch_bounds__(kMuonThreads) muonh_sumsq_u_kernel(const uint16_t* __restrict__ u, int64_t ldu,
                                                                     int64_t rows, int64_t cols,
                                                                     double* __restrict__ partials)
{
    __shared__ double sh[kMuonThreads / 32][3];
    double uu = 0.0, zero1 = 0.0, zero2 = 0.0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint2* ur = reinterpret_cast<const uint2*>(u + r * ldu);
        float suu = 0.0f;
        for (int64_t j = threadIdx.x; j < cols / 4; j += kMuonThreads) {
            const uint2 b = ur[j];
            const float u0 = bf16_to_f32(static_cast<uint16_t>(b.x)), u1 = bf16_to_f32(static_cast<uint16_t>(b.x >> 16));
            const float u2 = bf16_to_f32(static_cast<uint16_t>(b.y)), u3 = bf16_to_f32(static_cast<uint16_t>(b.y >> 16));
            suu = fmaf(u0, u0, fmaf(u1, u1, fmaf(u2, u2, fmaf(u3, u3, suu))));
        }
        uu += static_cast<double>(suu);
    }
    block_sum3(uu, zero1, zero2, sh);
    if (threadIdx.x == 0) {
        partials[3 * blockIdx.x + 0] = 0.0;
        partials[3 * blockIdx.x + 1] = 0.0;
        partials[3 * blockIdx.x + 2] = uu;
    }
}

// Step coefficient a = lr R / |U| from the |U|^2 partials (component 2), 0 if |U| = 0.
__device__ __forceinline__ float muonh_step_coef(const double* partials, int nparts, float lr, float radius)
{
    const double nu = sqrt(sum_partials(partials, nparts, 2));
    return nu > 0.0 ? static_cast<float>(static_cast<double>(lr) * static_cast<double>(radius) / nu) : 0.0f;
}

// partials[blockIdx.x].0 = sum of W'^2 over the CTA's rows, W' = fma(-a, u, w) in FP32
// exactly as muonh_apply_kernel forms it; components 1 and 2 are left as they are.
__global__ void __launch_bounds__(kMuonThreads) muonh_wprime_sumsq_kernel(const float* __restrict__ w, int64_t ldw,
                                                                          const uint16_t* __restrict__ u, int64_t ldu,
                                                                          int64_t rows, int64_t cols,
                                                                          double* __restrict__ partials, int nparts,
                                                                          float lr, float radius)
{
    __shared__ double sh[kMuonThreads / 32][3];
    __shared__ float coef;
    if (threadIdx.x == 0)
        coef = muonh_step_coef(partials, nparts, lr, radius);
    __syncthreads();
    const float a = coef;
    double pp = 0.0, zero1 = 0.0, zero2 = 0.0;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const float4* wr = reinterpret_cast<const float4*>(w + r * ldw);
        const uint2* ur = reinterpret_cast<const uint2*>(u + r * ldu);
        float spp = 0.0f;
        for (int64_t j = threadIdx.x; j < cols / 4; j += kMuonThreads) {
            const float4 v = wr[j];
            const uint2 b = ur[j];
            const float p0 = fmaf(-a, bf16_to_f32(static_cast<uint16_t>(b.x)), v.x);
            const float p1 = fmaf(-a, bf16_to_f32(static_cast<uint16_t>(b.x >> 16)), v.y);
            const float p2 = fmaf(-a, bf16_to_f32(static_cast<uint16_t>(b.y)), v.z);
            const float p3 = fmaf(-a, bf16_to_f32(static_cast<uint16_t>(b.y >> 16)), v.w);
            spp = fmaf(p0, p0, fmaf(p1, p1, fmaf(p2, p2, fmaf(p3, p3, spp))));
        }
        pp += static_cast<double>(spp);
    }
    // every CTA has read the |U|^2 partials before any CTA writes its own component 0
    // (they live in different words, so there is no overlap to order)
    block_sum3(pp, zero1, zero2, sh);
    if (threadIdx.x == 0)
        partials[3 * blockIdx.x + 0] = pp;
}

// w = R W' / |W'| in place, W' = fma(-a, u, w), from the |U|^2 (component 2) and
// |W'|^2 (component 0) partials. |U| = 0 gives a = 0 (w is only projected); if
// W' is exactly zero (|W'|^2 = 0), w is left unchanged. The factor R / |W'| is
// applied as a power of two times an FP32 value, so that it cannot overflow
// even when |W'| is tiny; in the normal range this gives the bits of a single
// multiplication by fl32(R / |W'|).
__global__ void __launch_bounds__(kMuonThreads) muonh_apply_kernel(float* __restrict__ w, int64_t ldw,
                                                                   const uint16_t* __restrict__ u, int64_t ldu,
                                                                   int64_t rows, int64_t cols,
                                                                   const double* __restrict__ partials, int nparts,
                                                                   float lr, float radius)
{
    __shared__ float coef[3];  // a, 2^e, fl32(R / |W'| / 2^e)
    __shared__ int keep;
    if (threadIdx.x == 0) {
        coef[0] = muonh_step_coef(partials, nparts, lr, radius);
        const double n2 = sum_partials(partials, nparts, 0);
        keep = !(n2 > 0.0);
        const double scale = keep ? 1.0 : static_cast<double>(radius) / sqrt(n2);
        int e = 0;
        frexp(scale, &e);
        const double p2 = ldexp(1.0, e / 2);
        coef[1] = static_cast<float>(p2);
        coef[2] = static_cast<float>(scale / p2);
    }
    __syncthreads();
    if (keep)
        return;
    const float a = coef[0], f1 = coef[1], f2 = coef[2];
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        float4* wr = reinterpret_cast<float4*>(w + r * ldw);
        const uint2* ur = reinterpret_cast<const uint2*>(u + r * ldu);
        for (int64_t j = threadIdx.x; j < cols / 4; j += kMuonThreads) {
            float4 v = wr[j];
            const uint2 b = ur[j];
            v.x = fmaf(-a, bf16_to_f32(static_cast<uint16_t>(b.x)), v.x) * f1 * f2;
            v.y = fmaf(-a, bf16_to_f32(static_cast<uint16_t>(b.x >> 16)), v.y) * f1 * f2;
            v.z = fmaf(-a, bf16_to_f32(static_cast<uint16_t>(b.y)), v.z) * f1 * f2;
            v.w = fmaf(-a, bf16_to_f32(static_cast<uint16_t>(b.y >> 16)), v.w) * f1 * f2;
            wr[j] = v;
        }
    }
}

// dst[j][i] = src[i][j] for BF16 src [rows][cols] (transpose), or dst[i][j] = src[i][j]
// (copy), through 32 x 32 shared-memory tiles. grid (ceil(cols/32), ceil(rows/32)), 32 x 8.
template <bool TRANSPOSE>
__global__ void __launch_bounds__(256) bf16_copy_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t cols,
                                                         int64_t lds, uint16_t* __restrict__ dst, int64_t ldd)
{
    __shared__ uint16_t tile[32][33];
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32, c0 = static_cast<int64_t>(blockIdx.x) * 32;
    for (int i = threadIdx.y; i < 32; i += 8) {
        const int64_t r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols)
            tile[i][threadIdx.x] = src[r * lds + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
        if (TRANSPOSE) {
            const int64_t r = c0 + i, c = r0 + threadIdx.x;  // dst row = src column
            if (r < cols && c < rows)
                dst[r * ldd + c] = tile[threadIdx.x][i];
        } else {
            const int64_t r = r0 + i, c = c0 + threadIdx.x;
            if (r < rows && c < cols)
                dst[r * ldd + c] = tile[i][threadIdx.x];
        }
    }
}

}  // namespace bfp8
