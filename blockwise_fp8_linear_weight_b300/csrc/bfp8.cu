// C ABI of the blockwise-FP8 linear-layer library (declared in include/bfp8.h):
// host-side argument checks, TMA tensor-map encoding and kernel launches.
// Everything the path computes runs in the kernels of quant.cuh and gemm.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "bf16_gemm.cuh"
#include "bfp8.h"
#include "gemm.cuh"
#include "muonh.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace bfp8 {

// Set (OR-ed) by a kernel that gives up on a bounded wait.
__device__ unsigned g_device_status;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 256;  // TMA coordinates are int32
constexpr int64_t kMaxGridY = 65535;

std::atomic<int> g_tile_n{0};
std::atomic<unsigned long long> g_wait_ns{kWaitLimitNs};
std::atomic<int> g_stall{0};

// ----------------------------------------------------------------- helpers
bool aligned(const void* p, uintptr_t a)
{
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Compute capability 10.3 check, cached per device.
int check_arch(int* dev_out)
{
    static std::atomic<int> cache[kMaxDevices];  // 0 unknown, 1 ok, 2 wrong arch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return BFP8_ELAUNCH;
    if (dev_out)
        *dev_out = dev;
    int c = cache[dev].load(std::memory_order_relaxed);
    if (c == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return BFP8_ELAUNCH;
        c = (major == 10 && minor == 3) ? 1 : 2;
        cache[dev].store(c, std::memory_order_relaxed);
    }
    return c == 1 ? BFP8_OK : BFP8_EARCH;
}

unsigned* device_status_ptr(int dev)
{
    static std::atomic<unsigned*> cache[kMaxDevices];
    unsigned* p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        void* q = nullptr;
        if (cudaGetSymbolAddress(&q, g_device_status) != cudaSuccess)
            return nullptr;
        p = static_cast<unsigned*>(q);
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

// Number of SMs of a device, cached (the persistent GEMM launches one CTA per SM).
int sm_count(int dev)
{
    static std::atomic<int> cache[kMaxDevices];
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D tensor map over a row-major [outer][inner] array with the given row stride.
bool make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz)
{
    auto fn = encode_fn();
    if (!fn)
        return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_status()
{
    return cudaGetLastError() == cudaSuccess ? BFP8_OK : BFP8_ELAUNCH;
}

// Kernels launched by the library in this process (bfp8_kernel_launches).
std::atomic<int64_t> g_launches{0};

void note_launch()
{
    g_launches.fetch_add(1, std::memory_order_relaxed);
}

// ----------------------------------------------------------------- GEMM launch
struct GemmProblem {
    // A: codes [gm][ld_a] with the contraction axis (gk) contiguous
    const uint8_t* a;
    int64_t lda;
    // B: codes; K-major [gn][ld_b] (contraction contiguous) or MN-major [gk][ld_b]
    const uint8_t* b;
    int64_t ldb;
    bool b_mn;
    // A scales [gk/128][ld_sa]
    const float* sa;
    int64_t ld_sa;
    // B scales: vector [gk/128][ld_sb], or scalar table with strides
    const float* sb;
    int64_t ld_sb;
    bool sb_vec;
    int64_t sb_col_stride, sb_chunk_stride;
    void* d;
    int64_t ldd;
    int64_t gm, gn, gk;
    // caller workspace for the split tail (NULL: no split)
    float* ws;
    int64_t ws_bytes;
};

// A tail is split along the contraction axis only when it would leave at least a
// quarter of the grid idle and the split shortens the longest CTA's tail by at
// least this many chunks. Measured on the MLP GEMMs of a B300 (20 launches in a
// CUDA graph): the piece-mode launch runs its chunks at 1.3-2x the whole-tile
// time per chunk (its own start-up and the partial-tile stores) and the reduce
// adds about 6 us, so a split that saves 25 chunks lost up to 4 %, one that
// saves 51 chunks of the weight gradient gained 9 %.
constexpr int64_t kTailMinSaved = 40;

// Workspace of the split tail: two FP32 partial tiles of 128 x 256 per CTA.
int64_t tail_ws_bytes(int ctas)
{
    return 2LL * ctas * 128 * 256 * 4;
}

template <class Cfg>
int run_gemm(const GemmProblem& p, unsigned* status, cudaStream_t stream, int dev)
{
    CUtensorMap tmA, tmB, tmSA, tmD;
    const int64_t nc = p.gk / 128;
    bool ok = make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.a, p.gk, p.gm, p.lda, 128, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (Cfg::B_MN)
        ok = ok && make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, p.gn, p.gk, p.ldb, 128, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    else
        ok = ok && make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, p.b, p.gk, p.gn, p.ldb, 128, Cfg::BN,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    // A scales: one box holds SGROUP chunks (rows) of 128 scales (B scales are read
    // by the scale-producer warp with plain loads)
    ok = ok && make_map(&tmSA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.sa, p.gm, nc, p.ld_sa * 4, 128, Cfg::SGROUP,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    if (Cfg::EPI == EPI_F32_ADD)
        ok = ok && make_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.d, p.gn, p.gm, p.ldd * 4, 32, 32,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    else
        ok = ok && make_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.d, p.gn, p.gm, p.ldd * 2, 64, 32,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok)
        return BFP8_ELAUNCH;

    static std::atomic<bool> attr_set[kMaxDevices];
    auto kern = bfp8_gemm_kernel<Cfg, false>;
    auto kern_pieces = bfp8_gemm_kernel<Cfg, true>;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        for (auto k : {kern, kern_pieces}) {
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
                cudaSuccess)
                return BFP8_ELAUNCH;
            // The register split (setmaxnreg) only balances if the kernel was built
            // with the full per-thread budget; with fewer registers the promotion
            // warpgroups' setmaxnreg.inc could never be satisfied. Refuse to launch.
            cudaFuncAttributes fa;
            if (cudaFuncGetAttributes(&fa, k) != cudaSuccess)
                return BFP8_ELAUNCH;
            if (Cfg::REG_SPLIT && fa.numRegs < Cfg::LAUNCH_REGS)
                return BFP8_ELAUNCH;
        }
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    GemmArgs args;
    args.gm = static_cast<int>(p.gm);
    args.gn = static_cast<int>(p.gn);
    args.num_chunks = static_cast<int>(nc);
    args.tiles_m = static_cast<int>((p.gm + Cfg::BM - 1) / Cfg::BM);
    args.tiles_n = static_cast<int>((p.gn + Cfg::BN - 1) / Cfg::BN);
    // sweep along N first when B is the smaller operand (it then stays in L2
    // while the larger A is streamed once), along M otherwise
    args.n_fastest = p.gn < p.gm ? 1 : 0;
    args.sb_scalar = p.sb;
    args.sb_col_stride = p.sb_col_stride;
    args.sb_chunk_stride = p.sb_chunk_stride;
    args.sb_vec = p.sb;
    args.ld_sb = p.ld_sb;
    args.status = status;
    args.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    args.stall = g_stall.load(std::memory_order_relaxed);
    // persistent grid: one CTA per SM, or one per tile if there are fewer tiles
    const int sms = sm_count(dev);
    const int64_t tiles = static_cast<int64_t>(args.tiles_m) * args.tiles_n;
    int ctas = static_cast<int>(std::min<int64_t>(tiles, sms));
    int64_t tail_tile0 = tiles, units = 0;
    if (Cfg::EPI != EPI_F32_ADD && p.ws && nc > kTailMinSaved) {
        // whole rounds of the grid, then a tail split along the contraction axis
        const int64_t rounds = tiles / sms, rest = tiles - rounds * sms;
        if (rest > 0 && rest * 4 <= static_cast<int64_t>(sms) * 3) {
            const int64_t g = rounds > 0 ? sms : std::min<int64_t>(rest * nc, sms);
            const int64_t longest = (rest * nc + g - 1) / g;  // chunks of the longest tail range
            // (the reduce kernel lists at most 256 pieces per tile: one per CTA)
            if (nc - longest >= kTailMinSaved && g <= 256 && p.ws_bytes >= tail_ws_bytes(static_cast<int>(g))) {
                tail_tile0 = rounds * sms;
                units = rest * nc;
                ctas = static_cast<int>(g);
            }
        }
    }
    args.tail_tile0 = static_cast<int>(tail_tile0);
    args.tail_units = units;
    // a launch that may start before the one before it on the stream has finished
    // (programmatic dependent launch); the kernels wait inside where they need to
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    if (units == 0) {
        CUtensorMap unused = tmD;
        kern<<<ctas, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(tmA, tmB, tmSA, tmD, unused, args);
        note_launch();
        return launch_status();
    }
    // the whole rounds (if any), then the tail's pieces on the SMs that they free,
    // then the sum of the partial tiles
    if (tail_tile0 > 0) {
        CUtensorMap unused = tmD;
        kern<<<sms, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(tmA, tmB, tmSA, tmD, unused, args);
        note_launch();
    }
    // partial tiles: FP32 [2 ctas x 128 rows][BN], 32 x 32 boxes
    CUtensorMap tmW;
    if (!make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.ws, Cfg::BN, 2 * static_cast<uint64_t>(ctas) * Cfg::BM,
                  Cfg::BN * 4, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return BFP8_ELAUNCH;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(ctas));
    lc.blockDim = dim3(Cfg::THREADS);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = stream;
    lc.attrs = pdl;
    lc.numAttrs = tail_tile0 > 0 ? 1 : 0;
    if (cudaLaunchKernelEx(&lc, kern_pieces, tmA, tmB, tmSA, tmD, tmW, args) != cudaSuccess)
        return BFP8_ELAUNCH;
    note_launch();
    TailReduceArgs ra;
    ra.ws = p.ws;
    ra.d = static_cast<uint16_t*>(p.d);
    ra.ldd = p.ldd;
    ra.gm = args.gm;
    ra.gn = args.gn;
    ra.num_chunks = args.num_chunks;
    ra.tail_tile0 = args.tail_tile0;
    ra.grid = ctas;
    ra.tail_units = units;
    ra.tiles_m = args.tiles_m;
    ra.tiles_n = args.tiles_n;
    ra.n_fastest = args.n_fastest;
    cudaLaunchConfig_t lr = {};
    lr.gridDim = dim3(static_cast<unsigned>(tiles - tail_tile0), Cfg::BM / 8);
    lr.blockDim = dim3(256);
    lr.dynamicSmemBytes = 0;
    lr.stream = stream;
    lr.attrs = pdl;
    lr.numAttrs = 1;
    if (cudaLaunchKernelEx(&lr, gemm_tail_reduce_kernel<Cfg::BN>, ra) != cudaSuccess)
        return BFP8_ELAUNCH;
    note_launch();
    return launch_status();
}

template <bool B_MN, bool SB_VEC, int EPI = EPI_BF16_TMA>
int dispatch_gemm(const GemmProblem& p, cudaStream_t stream)
{
    int dev = 0;
    int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    unsigned* status = device_status_ptr(dev);
    if (!status)
        return BFP8_ELAUNCH;
    if constexpr (EPI == EPI_F32_ADD) {  // one configuration: 256-wide tiles, 8 promotion warps
        return run_gemm<GemmConfig<256, 3, B_MN, SB_VEC, EPI_F32_ADD>>(p, status, stream, dev);
    } else {
        int tn = g_tile_n.load(std::memory_order_relaxed);
        if (tn == 0)
            tn = 256;
        if (tn == 128)
            return run_gemm<GemmConfig<128, 5, B_MN, SB_VEC>>(p, status, stream, dev);
        if constexpr (!B_MN) {
            // 192-wide tiles: 12 promotion warps of 64 columns
            if (tn == 192)
                return run_gemm<GemmConfig<192, 4, B_MN, SB_VEC, EPI_BF16_TMA, 12>>(p, status, stream, dev);
        }
        return run_gemm<GemmConfig<256, 3, B_MN, SB_VEC>>(p, status, stream, dev);
    }
}

bool gemm_dims_ok(int64_t gm, int64_t gn, int64_t gk)
{
    return gm >= 1 && gn >= 128 && gk >= 128 && gn % 128 == 0 && gk % 128 == 0 && gm <= kMaxDim && gn <= kMaxDim &&
           gk <= kMaxDim && (gm + 127) / 128 <= kMaxGridY;
}

}  // namespace
}  // namespace bfp8

using namespace bfp8;

namespace bfp8 {
namespace {

// Launches the persistent block quantiser over x [R][C] (C % 128 == 0, R >= 1).
template <int MODE>
int run_quant_blocks(const void* x, int64_t R, int64_t C, int64_t ldx, const QuantArgs& base, cudaStream_t stream)
{
    int dev = 0;
    int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    unsigned* status = device_status_ptr(dev);
    if (!status)
        return BFP8_ELAUNCH;
    CUtensorMap tm;
    if (!make_map(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(C), static_cast<uint64_t>(R),
                  static_cast<uint64_t>(ldx) * 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
        return BFP8_ELAUNCH;
    static std::atomic<bool> attr_set[kMaxDevices];
    auto kern = quant_blocks_kernel<MODE>;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kQuantSmemBytes) != cudaSuccess)
            return BFP8_ELAUNCH;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    QuantArgs a = base;
    a.R = R;
    a.nblk_c = C / 128;
    a.nblocks = ((R + 127) / 128) * a.nblk_c;
    a.status = status;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    a.stall = g_stall.load(std::memory_order_relaxed);
    const int64_t ctas = std::min<int64_t>(a.nblocks, static_cast<int64_t>(sm_count(dev)) * 3);
    kern<<<static_cast<unsigned>(ctas), 256, kQuantSmemBytes, stream>>>(tm, a);
    note_launch();
    return launch_status();
}

// Launches the two-layout quantiser without block-wide barriers (quant_dual_kernel):
// kDualBuffers shared-memory buffers per CTA, kDualCtasPerSm CTAs per SM (measured
// best of 2 x 3, 3 x 2 and 4 x 1 on the MLP tensors).
constexpr int kDualBuffers = 2;
constexpr int kDualCtasPerSm = 3;

int run_quant_dual(const void* x, int64_t R, int64_t C, int64_t ldx, const QuantArgs& base, cudaStream_t stream)
{
    int dev = 0;
    int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    unsigned* status = device_status_ptr(dev);
    if (!status)
        return BFP8_ELAUNCH;
    CUtensorMap tm;
    if (!make_map(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(C), static_cast<uint64_t>(R),
                  static_cast<uint64_t>(ldx) * 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
        return BFP8_ELAUNCH;
    constexpr int smem = dual_smem_bytes<kDualBuffers>();
    static std::atomic<bool> attr_set[kMaxDevices];
    // 32-byte stores of the transposed codes when every code row starts on a 32-byte boundary
    const bool st32 = aligned(base.qt, 32) && base.ldqt % 32 == 0;
    auto kern = st32 ? quant_dual_kernel<kDualBuffers, kDualCtasPerSm, true>
                     : quant_dual_kernel<kDualBuffers, kDualCtasPerSm, false>;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(quant_dual_kernel<kDualBuffers, kDualCtasPerSm, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
            cudaFuncSetAttribute(quant_dual_kernel<kDualBuffers, kDualCtasPerSm, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BFP8_ELAUNCH;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    QuantArgs a = base;
    a.R = R;
    a.nblk_c = C / 128;
    a.nblocks = ((R + 127) / 128) * a.nblk_c;
    a.status = status;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    a.stall = g_stall.load(std::memory_order_relaxed);
    const int64_t ctas = std::min<int64_t>(a.nblocks, static_cast<int64_t>(sm_count(dev)) * kDualCtasPerSm);
    kern<<<static_cast<unsigned>(ctas), kDualThreads, smem, stream>>>(tm, a);
    note_launch();
    return launch_status();
}

// Launches the weight quantiser (quant_weight_kernel): the same buffers and CTAs per
// SM as the two-layout kernel.
int run_quant_weight(const void* w, int64_t N, int64_t K, int64_t ldw, const QuantArgs& base, cudaStream_t stream)
{
    int dev = 0;
    int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    unsigned* status = device_status_ptr(dev);
    if (!status)
        return BFP8_ELAUNCH;
    CUtensorMap tm;
    if (!make_map(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w, static_cast<uint64_t>(K), static_cast<uint64_t>(N),
                  static_cast<uint64_t>(ldw) * 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
        return BFP8_ELAUNCH;
    constexpr int smem = dual_smem_bytes<kDualBuffers>();
    static std::atomic<bool> attr_set[kMaxDevices];
    auto kern = quant_weight_kernel<kDualBuffers, kDualCtasPerSm>;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return BFP8_ELAUNCH;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    QuantArgs a = base;
    a.R = N;
    a.nblk_c = K / 128;
    a.nblocks = (N / 128) * a.nblk_c;
    a.status = status;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    a.stall = g_stall.load(std::memory_order_relaxed);
    const int64_t ctas = std::min<int64_t>(a.nblocks, static_cast<int64_t>(sm_count(dev)) * kDualCtasPerSm);
    kern<<<static_cast<unsigned>(ctas), kDualThreads, smem, stream>>>(tm, a);
    note_launch();
    return launch_status();
}

}  // namespace
}  // namespace bfp8

// =================================================================== quantisers
extern "C" int fp8_quantize_act(const void* x, int64_t R, int64_t C, int64_t ldx, uint8_t* q, int64_t ldq,
                                float* s, int64_t lds, void* stream)
{
    if (R < 0 || C < 0)
        return BFP8_EINVAL;
    if (C % 128 != 0 || R > kMaxDim || C > kMaxDim)
        return BFP8_ESHAPE;
    if (R == 0 || C == 0)
        return BFP8_OK;
    if (!x || !q || !s || ldx < C || ldq < C || lds < R)
        return BFP8_EINVAL;
    if (!aligned(x, 16) || ldx % 8 || !aligned(q, 8) || ldq % 8 || !aligned(s, 4))
        return BFP8_EALIGN;
    int rc = check_arch(nullptr);
    if (rc != BFP8_OK)
        return rc;
    QuantArgs qa{};
    qa.q = q;
    qa.ldq = ldq;
    qa.s = s;
    qa.lds = lds;
    return run_quant_blocks<MODE_ROWS>(x, R, C, ldx, qa, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_quantize_weight(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, int64_t ldq,
                                   float* s, void* stream)
{
    if (N < 0 || K < 0)
        return BFP8_EINVAL;
    if (N % 128 || K % 128 || N > kMaxDim || K > kMaxDim || N / 128 > kMaxGridY)
        return BFP8_ESHAPE;
    if (N == 0 || K == 0)
        return BFP8_OK;
    if (!w || !q || !s || ldw < K || ldq < K)
        return BFP8_EINVAL;
    if (!aligned(w, 16) || ldw % 8 || !aligned(q, 8) || ldq % 8 || !aligned(s, 4))
        return BFP8_EALIGN;
    int rc = check_arch(nullptr);
    if (rc != BFP8_OK)
        return rc;
    QuantArgs qa{};
    qa.q = q;
    qa.ldq = ldq;
    qa.s = s;
    qa.lds = K / 128;
    return run_quant_weight(w, N, K, ldw, qa, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_quantize_transpose(const void* x, int64_t R, int64_t C, int64_t ldx, uint8_t* qt,
                                      int64_t ldqt, float* st, int64_t ldst, void* stream)
{
    if (R < 0 || C < 0)
        return BFP8_EINVAL;
    if (C % 128 || R > kMaxDim || C > kMaxDim || (R + 127) / 128 > kMaxGridY)
        return BFP8_ESHAPE;
    if (R == 0 || C == 0)
        return BFP8_OK;
    const int64_t R128 = (R + 127) / 128 * 128;
    if (!x || !qt || !st || ldx < C || ldqt < R128 || ldst < C)
        return BFP8_EINVAL;
    if (!aligned(x, 16) || ldx % 8 || !aligned(qt, 16) || ldqt % 16 || !aligned(st, 8) || ldst % 2)
        return BFP8_EALIGN;
    int rc = check_arch(nullptr);
    if (rc != BFP8_OK)
        return rc;
    QuantArgs qa{};
    qa.qt = qt;
    qa.ldqt = ldqt;
    qa.st = st;
    qa.ldst = ldst;
    return run_quant_blocks<MODE_COLS>(x, R, C, ldx, qa, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_quantize_act_transpose(const void* x, int64_t R, int64_t C, int64_t ldx, uint8_t* q,
                                          int64_t ldq, float* s, int64_t lds, uint8_t* qt, int64_t ldqt,
                                          float* st, int64_t ldst, void* stream)
{
    if (R < 0 || C < 0)
        return BFP8_EINVAL;
    if (C % 128 || R > kMaxDim || C > kMaxDim || (R + 127) / 128 > kMaxGridY)
        return BFP8_ESHAPE;
    if (R == 0 || C == 0)
        return BFP8_OK;
    const int64_t R128 = (R + 127) / 128 * 128;
    if (!x || !q || !s || !qt || !st || ldx < C || ldq < C || lds < R || ldqt < R128 || ldst < C)
        return BFP8_EINVAL;
    if (!aligned(x, 16) || ldx % 8 || !aligned(q, 8) || ldq % 8 || !aligned(s, 4) || !aligned(qt, 16) ||
        ldqt % 16 || !aligned(st, 8) || ldst % 2)
        return BFP8_EALIGN;
    int rc = check_arch(nullptr);
    if (rc != BFP8_OK)
        return rc;
    QuantArgs qa{};
    qa.q = q;
    qa.ldq = ldq;
    qa.s = s;
    qa.lds = lds;
    qa.qt = qt;
    qa.ldqt = ldqt;
    qa.st = st;
    qa.ldst = ldst;
    return run_quant_dual(x, R, C, ldx, qa, static_cast<cudaStream_t>(stream));
}

// =================================================================== GEMMs
extern "C" int fp8_block_gemm_fwd(const uint8_t* qx, int64_t ldqx, const float* sx, int64_t ldsx,
                                  const uint8_t* qw, int64_t ldqw, const float* sw, void* y, int64_t ldy,
                                  int64_t M, int64_t N, int64_t K, void* workspace, int64_t workspace_bytes,
                                  void* stream)
{
    if (M < 0 || N < 0 || K < 0)
        return BFP8_EINVAL;
    if (M == 0)
        return (N % 128 || K % 128) ? BFP8_ESHAPE : BFP8_OK;
    if (!gemm_dims_ok(M, N, K))
        return BFP8_ESHAPE;
    if (!qx || !sx || !qw || !sw || !y || ldqx < K || ldqw < K || ldsx < M || ldy < N)
        return BFP8_EINVAL;
    if (!aligned(qx, 16) || !aligned(qw, 16) || !aligned(sx, 16) || !aligned(y, 16) || !aligned(sw, 4) ||
        ldqx % 16 || ldqw % 16 || ldsx % 4 || ldy % 8)
        return BFP8_EALIGN;
    if (workspace_bytes < 0 || (workspace && !aligned(workspace, 16)))
        return workspace_bytes < 0 ? BFP8_EINVAL : BFP8_EALIGN;
    GemmProblem p{};
    p.ws = static_cast<float*>(workspace);
    p.ws_bytes = workspace ? workspace_bytes : 0;
    p.a = qx;
    p.lda = ldqx;
    p.b = qw;
    p.ldb = ldqw;
    p.b_mn = false;
    p.sa = sx;
    p.ld_sa = ldsx;
    p.sb = sw;
    p.sb_vec = false;
    p.sb_col_stride = K / 128;  // sw[n/128][kb]
    p.sb_chunk_stride = 1;
    p.d = y;
    p.ldd = ldy;
    p.gm = M;
    p.gn = N;
    p.gk = K;
    return dispatch_gemm<false, false>(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_block_gemm_dgrad(const uint8_t* qdy, int64_t ldqdy, const float* sdy, int64_t ldsdy,
                                    const uint8_t* qw, int64_t ldqw, const float* sw, void* dx, int64_t lddx,
                                    int64_t M, int64_t N, int64_t K, void* workspace, int64_t workspace_bytes,
                                    void* stream)
{
    if (M < 0 || N < 0 || K < 0)
        return BFP8_EINVAL;
    if (M == 0)
        return (N % 128 || K % 128) ? BFP8_ESHAPE : BFP8_OK;
    if (!gemm_dims_ok(M, K, N))
        return BFP8_ESHAPE;
    if (!qdy || !sdy || !qw || !sw || !dx || ldqdy < N || ldqw < K || ldsdy < M || lddx < K)
        return BFP8_EINVAL;
    if (!aligned(qdy, 16) || !aligned(qw, 16) || !aligned(sdy, 16) || !aligned(dx, 16) || !aligned(sw, 4) ||
        ldqdy % 16 || ldqw % 16 || ldsdy % 4 || lddx % 8)
        return BFP8_EALIGN;
    if (workspace_bytes < 0 || (workspace && !aligned(workspace, 16)))
        return workspace_bytes < 0 ? BFP8_EINVAL : BFP8_EALIGN;
    GemmProblem p{};
    p.ws = static_cast<float*>(workspace);
    p.ws_bytes = workspace ? workspace_bytes : 0;
    p.a = qdy;
    p.lda = ldqdy;
    p.b = qw;  // [N][K]: contraction (N) strided, output columns (K) contiguous
    p.ldb = ldqw;
    p.b_mn = true;
    p.sa = sdy;
    p.ld_sa = ldsdy;
    p.sb = sw;
    p.sb_vec = false;
    p.sb_col_stride = 1;  // sw[nb][k/128]
    p.sb_chunk_stride = K / 128;
    p.d = dx;
    p.ldd = lddx;
    p.gm = M;
    p.gn = K;
    p.gk = N;
    return dispatch_gemm<true, false>(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_block_gemm_wgrad(const uint8_t* qdyt, int64_t ldqdyt, const float* sdyt, int64_t ldsdyt,
                                    const uint8_t* qxt, int64_t ldqxt, const float* sxt, int64_t ldsxt, void* dw,
                                    int64_t lddw, int64_t M, int64_t N, int64_t K, void* workspace,
                                    int64_t workspace_bytes, void* stream)
{
    if (M < 0 || N < 0 || K < 0)
        return BFP8_EINVAL;
    const int64_t M128 = (M + 127) / 128 * 128;
    if (M < 1 || !gemm_dims_ok(N, K, M128))
        return BFP8_ESHAPE;
    if (!qdyt || !sdyt || !qxt || !sxt || !dw || ldqdyt < M128 || ldqxt < M128 || ldsdyt < N || ldsxt < K ||
        lddw < K)
        return BFP8_EINVAL;
    if (!aligned(qdyt, 16) || !aligned(qxt, 16) || !aligned(sdyt, 16) || !aligned(sxt, 16) || !aligned(dw, 16) ||
        ldqdyt % 16 || ldqxt % 16 || ldsdyt % 4 || ldsxt % 4 || lddw % 8)
        return BFP8_EALIGN;
    if (workspace_bytes < 0 || (workspace && !aligned(workspace, 16)))
        return workspace_bytes < 0 ? BFP8_EINVAL : BFP8_EALIGN;
    GemmProblem p{};
    p.ws = static_cast<float*>(workspace);
    p.ws_bytes = workspace ? workspace_bytes : 0;
    p.a = qdyt;
    p.lda = ldqdyt;
    p.b = qxt;
    p.ldb = ldqxt;
    p.b_mn = false;
    p.sa = sdyt;
    p.ld_sa = ldsdyt;
    p.sb = sxt;
    p.ld_sb = ldsxt;
    p.sb_vec = true;
    p.d = dw;
    p.ldd = lddw;
    p.gm = N;
    p.gn = K;
    p.gk = M128;
    return dispatch_gemm<false, true>(p, static_cast<cudaStream_t>(stream));
}

extern "C" int fp8_block_gemm_wgrad_acc(const uint8_t* qdyt, int64_t ldqdyt, const float* sdyt, int64_t ldsdyt,
                                        const uint8_t* qxt, int64_t ldqxt, const float* sxt, int64_t ldsxt,
                                        float* main_grad, int64_t ldmg, int64_t M, int64_t N, int64_t K,
                                        void* stream)
{
    if (M < 0 || N < 0 || K < 0)
        return BFP8_EINVAL;
    const int64_t M128 = (M + 127) / 128 * 128;
    if (M < 1 || !gemm_dims_ok(N, K, M128))
        return BFP8_ESHAPE;
    if (!qdyt || !sdyt || !qxt || !sxt || !main_grad || ldqdyt < M128 || ldqxt < M128 || ldsdyt < N ||
        ldsxt < K || ldmg < K)
        return BFP8_EINVAL;
    if (!aligned(qdyt, 16) || !aligned(qxt, 16) || !aligned(sdyt, 16) || !aligned(sxt, 16) ||
        !aligned(main_grad, 16) || ldqdyt % 16 || ldqxt % 16 || ldsdyt % 4 || ldsxt % 4 || ldmg % 4)
        return BFP8_EALIGN;
    GemmProblem p{};
    p.a = qdyt;
    p.lda = ldqdyt;
    p.b = qxt;
    p.ldb = ldqxt;
    p.b_mn = false;
    p.sa = sdyt;
    p.ld_sa = ldsdyt;
    p.sb = sxt;
    p.ld_sb = ldsxt;
    p.sb_vec = true;
    p.d = main_grad;
    p.ldd = ldmg;
    p.gm = N;
    p.gn = K;
    p.gk = M128;
    return dispatch_gemm<false, true, EPI_F32_ADD>(p, static_cast<cudaStream_t>(stream));
}

extern "C" int bfp8_kernel_launches(int64_t* count)
{
    if (!count)
        return BFP8_EINVAL;
    *count = g_launches.load(std::memory_order_relaxed);
    return BFP8_OK;
}

extern "C" int fp8_block_gemm_workspace_bytes(int64_t* bytes)
{
    if (!bytes)
        return BFP8_EINVAL;
    int dev = 0;
    const int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    *bytes = tail_ws_bytes(sm_count(dev));
    return BFP8_OK;
}

// =================================================================== MuonH
namespace bfp8 {
namespace {
// One reduction grid for every MuonH call on a device, so that partial sums
// written by one kernel are read back by the next one in the same layout.
int muonh_grid(int dev)
{
    return 2 * sm_count(dev);
}

// Device-wide partial sums for muonh_apply_static (room for grids of up to 512 CTAs).
constexpr int64_t kStaticPartials = 3 * 512;
__device__ __align__(256) double g_muonh_partials[kStaticPartials];
}  // namespace
}  // namespace bfp8

extern "C" int muonh_partials_len(int* n)
{
    if (!n)
        return BFP8_EINVAL;
    int dev = 0;
    int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    *n = 3 * muonh_grid(dev);
    return BFP8_OK;
}

extern "C" int muonh_normalize(const float* g, int64_t rows, int64_t cols, int64_t ldg, void* x, int64_t ldx,
                               double* partials, int64_t partials_len, float eps, void* stream)
{
    if (rows < 1 || cols < 1)
        return BFP8_EINVAL;
    if (cols % 4 || rows > kMaxDim || cols > kMaxDim)
        return BFP8_ESHAPE;
    if (!g || !x || !partials || ldg < cols || ldx < cols || !(eps >= 0.0f))
        return BFP8_EINVAL;
    if (!aligned(g, 16) || ldg % 4 || !aligned(x, 8) || ldx % 4 || !aligned(partials, 8))
        return BFP8_EALIGN;
    int dev = 0;
    int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    const int grid = muonh_grid(dev);
    if (partials_len < 3 * static_cast<int64_t>(grid))
        return BFP8_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    muonh_sumsq_kernel<<<grid, kMuonThreads, 0, st>>>(g, rows, cols, ldg, partials);
    note_launch();
    muonh_scale_bf16_kernel<<<grid, kMuonThreads, 0, st>>>(g, rows, cols, ldg, partials, grid, eps,
                                                          static_cast<uint16_t*>(x), ldx);
    note_launch();
    return launch_status();
}

static int muonh_apply_impl(float* w, int64_t ldw, const void* u, int64_t ldu, int64_t rows, int64_t cols,
                            double* partials, int64_t partials_len, bool static_partials, float lr, float radius,
                            void* stream)
{
    if (rows < 1 || cols < 1)
        return BFP8_EINVAL;
    if (cols % 4 || rows > kMaxDim || cols > kMaxDim)
        return BFP8_ESHAPE;
    if (!w || !u || (!static_partials && !partials) || ldw < cols || ldu < cols || !(lr >= 0.0f) ||
        !(radius > 0.0f))
        return BFP8_EINVAL;
    if (!aligned(w, 16) || ldw % 4 || !aligned(u, 8) || ldu % 4 || !aligned(partials, 8))
        return BFP8_EALIGN;
    int dev = 0;
    int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    if (static_partials) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_muonh_partials) != cudaSuccess)
            return BFP8_ELAUNCH;
        partials = static_cast<double*>(p);
        partials_len = kStaticPartials;
    }
    const int grid = muonh_grid(dev);
    if (partials_len < 3 * static_cast<int64_t>(grid))
        return BFP8_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint16_t* ub = static_cast<const uint16_t*>(u);
    muonh_sumsq_u_kernel<<<grid, kMuonThreads, 0, st>>>(ub, ldu, rows, cols, partials);
    note_launch();
    muonh_wprime_sumsq_kernel<<<grid, kMuonThreads, 0, st>>>(w, ldw, ub, ldu, rows, cols, partials, grid, lr, radius);
    note_launch();
    muonh_apply_kernel<<<grid, kMuonThreads, 0, st>>>(w, ldw, ub, ldu, rows, cols, partials, grid, lr, radius);
    note_launch();
    return launch_status();
}

extern "C" int muonh_apply(float* w, int64_t ldw, const void* u, int64_t ldu, int64_t rows, int64_t cols,
                           double* partials, int64_t partials_len, float lr, float radius, void* stream)
{
    return muonh_apply_impl(w, ldw, u, ldu, rows, cols, partials, partials_len, false, lr, radius, stream);
}

extern "C" int muonh_apply_static(float* w, int64_t ldw, const void* u, int64_t ldu, int64_t rows, int64_t cols,
                                  float lr, float radius, void* stream)
{
    return muonh_apply_impl(w, ldw, u, ldu, rows, cols, nullptr, 0, true, lr, radius, stream);
}

// =================================================================== misc
extern "C" const char* bfp8_status_string(int status)
{
    switch (status) {
    case BFP8_OK:
        return "BFP8_OK";
    case BFP8_EINVAL:
        return "BFP8_EINVAL: null pointer, negative size or leading dimension too small";
    case BFP8_EALIGN:
        return "BFP8_EALIGN: pointer or leading dimension breaks a 16-byte alignment rule";
    case BFP8_ESHAPE:
        return "BFP8_ESHAPE: dimension not a multiple of 128, or too large";
    case BFP8_ELAUNCH:
        return "BFP8_ELAUNCH: CUDA launch or tensor-map encoding failed";
    case BFP8_ETIMEOUT:
        return "BFP8_ETIMEOUT: a kernel gave up on a bounded wait";
    case BFP8_EARCH:
        return "BFP8_EARCH: device is not compute capability 10.3 (sm_103)";
    default:
        return "unknown bfp8 status";
    }
}

extern "C" int bfp8_last_device_status(void* stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return BFP8_ELAUNCH;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned host = 0, zero = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return BFP8_ELAUNCH;
    if (cudaMemcpyFromSymbolAsync(&host, g_device_status, sizeof host, 0, cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return BFP8_ELAUNCH;
    return (host & kDevTimeout) ? BFP8_ETIMEOUT : BFP8_OK;
}


extern "C" int bfp8_set_wait_limit_ns(int64_t ns)
{
    if (ns == 0)
        ns = static_cast<int64_t>(kWaitLimitNs);
    if (ns < 1000 || ns > 60000000000ll)
        return BFP8_EINVAL;
    g_wait_ns.store(static_cast<unsigned long long>(ns), std::memory_order_relaxed);
    return BFP8_OK;
}

extern "C" int bfp8_test_stall_producers(int on)
{
    if (on != 0 && on != 1)
        return BFP8_EINVAL;
    return g_stall.exchange(on);
}

extern "C" int bfp8_set_gemm_tile_n(int tile_n)
{
    if (tile_n != 0 && tile_n != 128 && tile_n != 192 && tile_n != 256)
        return BFP8_EINVAL;
    return g_tile_n.exchange(tile_n);
}

// =================================================================== BF16 GEMM (Newton-Schulz)
namespace bfp8 {
namespace {

template <bool B_MN>
int run_bf16_gemm(const void* a, int64_t lda, const void* b, int64_t ldb, const void* c, int64_t ldc, void* d,
                  int64_t ldd, int64_t M, int64_t N, int64_t K, float alpha, float beta, cudaStream_t stream, int dev,
                  unsigned* status)
{
    using Cfg = Bf16GemmConfig<B_MN>;
    CUtensorMap tmA, tmB, tmD;
    bool ok = make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a, K, M, lda * 2, Cfg::BK, Cfg::BM,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (B_MN)
        ok = ok && make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b, N, K, ldb * 2, 64, Cfg::BK,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    else
        ok = ok && make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b, K, N, ldb * 2, Cfg::BK, Cfg::BN,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d, N, M, ldd * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok)
        return BFP8_ELAUNCH;
    static std::atomic<bool> attr_set[kMaxDevices];
    auto kern = bf16_gemm_kernel<Cfg>;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
            return BFP8_ELAUNCH;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    Bf16GemmArgs args;
    args.gm = static_cast<int>(M);
    args.gn = static_cast<int>(N);
    args.gk = static_cast<int>(K);
    args.tiles_m = static_cast<int>((M + Cfg::BM - 1) / Cfg::BM);
    args.tiles_n = static_cast<int>((N + Cfg::BN - 1) / Cfg::BN);
    args.kblocks = static_cast<int>((K + Cfg::BK - 1) / Cfg::BK);
    args.alpha = alpha;
    args.beta = beta;
    args.c = beta != 0.0f ? static_cast<const uint16_t*>(c) : nullptr;
    args.ldc = ldc;
    args.status = status;
    args.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    args.stall = g_stall.load(std::memory_order_relaxed);
    const int64_t tiles = static_cast<int64_t>(args.tiles_m) * args.tiles_n;
    const int ctas = static_cast<int>(std::min<int64_t>(tiles, sm_count(dev)));
    kern<<<ctas, Cfg::THREADS, Cfg::SMEM_BYTES, stream>>>(tmA, tmB, tmD, args);
    note_launch();
    return launch_status();
}

int bf16_gemm_checked(const void* a, int64_t lda, const void* b, int64_t ldb, int b_mn_major, const void* c,
                      int64_t ldc, void* d, int64_t ldd, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                      cudaStream_t stream)
{
    if (M < 1 || N < 1 || K < 1 || (b_mn_major != 0 && b_mn_major != 1))
        return BFP8_EINVAL;
    if (N % 8 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return BFP8_ESHAPE;
    if (!a || !b || !d || (beta != 0.0f && !c) || !(alpha == alpha) || !(beta == beta))
        return BFP8_EINVAL;
    if (lda < K || ldb < (b_mn_major ? N : K) || ldd < N || (beta != 0.0f && ldc < N))
        return BFP8_EINVAL;
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(d, 16) || (beta != 0.0f && !aligned(c, 16)) || lda % 8 ||
        ldb % 8 || ldd % 8 || (beta != 0.0f && ldc % 8))
        return BFP8_EALIGN;
    int dev = 0;
    int rc = check_arch(&dev);
    if (rc != BFP8_OK)
        return rc;
    unsigned* status = device_status_ptr(dev);
    if (!status)
        return BFP8_ELAUNCH;
    if (b_mn_major)
        return run_bf16_gemm<true>(a, lda, b, ldb, c, ldc, d, ldd, M, N, K, alpha, beta, stream, dev, status);
    return run_bf16_gemm<false>(a, lda, b, ldb, c, ldc, d, ldd, M, N, K, alpha, beta, stream, dev, status);
}

int64_t round8(int64_t x)
{
    return (x + 7) / 8 * 8;
}

// Workspace of muonh_newton_schulz: A and B [r][r8], Y0 and Y1 [r][c8] (BF16),
// r = min(rows, cols), c = max(rows, cols), row strides rounded up to 8 elements.
int64_t ns_work_bytes(int64_t rows, int64_t cols)
{
    const int64_t r = std::min(rows, cols), c = std::max(rows, cols);
    return 2 * (2 * r * round8(r) + 2 * r * round8(c));
}

}  // namespace
}  // namespace bfp8

extern "C" int bf16_gemm_axpby(const void* a, int64_t lda, const void* b, int64_t ldb, int b_mn_major, const void* c,
                               int64_t ldc, void* d, int64_t ldd, int64_t M, int64_t N, int64_t K, float alpha,
                               float beta, void* stream)
{
    return bf16_gemm_checked(a, lda, b, ldb, b_mn_major, c, ldc, d, ldd, M, N, K, alpha, beta,
                             static_cast<cudaStream_t>(stream));
}

extern "C" int muonh_newton_schulz_work_bytes(int64_t rows, int64_t cols, int64_t* bytes)
{
    if (!bytes || rows < 1 || cols < 1)
        return BFP8_EINVAL;
    *bytes = ns_work_bytes(rows, cols);
    return BFP8_OK;
}

extern "C" int muonh_newton_schulz(void* x, int64_t rows, int64_t cols, int64_t ldx, void* work, int64_t work_bytes,
                                   int steps, float a, float b, float c, void* stream)
{
    if (rows < 1 || cols < 1 || steps < 0 || !x || !work || ldx < cols)
        return BFP8_EINVAL;
    if (rows % 8 || cols % 8 || rows > kMaxDim || cols > kMaxDim || (rows + 31) / 32 > kMaxGridY)
        return BFP8_ESHAPE;
    if (work_bytes < ns_work_bytes(rows, cols))
        return BFP8_EINVAL;
    if (!aligned(x, 16) || ldx % 8 || !aligned(work, 16))
        return BFP8_EALIGN;
    int rc = check_arch(nullptr);
    if (rc != BFP8_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool tr = rows > cols;  // iterate on the orientation with fewer rows
    const int64_t r = tr ? cols : rows, cc = tr ? rows : cols;
    const int64_t ldr = round8(r), ldc = round8(cc);
    uint16_t* A = static_cast<uint16_t*>(work);
    uint16_t* B = A + r * ldr;
    uint16_t* Y[2] = {B + r * ldr, B + r * ldr + r * ldc};
    uint16_t* xs = static_cast<uint16_t*>(x);
    const dim3 blk(32, 8);
    const dim3 grid_in(static_cast<unsigned>((cols + 31) / 32), static_cast<unsigned>((rows + 31) / 32));
    if (tr)
        bf16_copy_kernel<true><<<grid_in, blk, 0, st>>>(xs, rows, cols, ldx, Y[0], ldc);
    else
        bf16_copy_kernel<false><<<grid_in, blk, 0, st>>>(xs, rows, cols, ldx, Y[0], ldc);
    note_launch();
    if ((rc = launch_status()) != BFP8_OK)
        return rc;
    int cur = 0;
    for (int i = 0; i < steps; ++i) {
        const uint16_t* y = Y[cur];
        // A = Y Y^T (contraction over the long side)
        rc = bf16_gemm_checked(y, ldc, y, ldc, 0, nullptr, 0, A, ldr, r, r, cc, 1.0f, 0.0f, st);
        // B = b A + c A A (A read as [K][N] for the second factor)
        if (rc == BFP8_OK)
            rc = bf16_gemm_checked(A, ldr, A, ldr, 1, A, ldr, B, ldr, r, r, r, c, b, st);
        // Y' = a Y + B Y (Y read as [K][N])
        if (rc == BFP8_OK)
            rc = bf16_gemm_checked(B, ldr, y, ldc, 1, y, ldc, Y[cur ^ 1], ldc, r, cc, r, 1.0f, a, st);
        if (rc != BFP8_OK)
            return rc;
        cur ^= 1;
    }
    const dim3 grid_out(static_cast<unsigned>((cc + 31) / 32), static_cast<unsigned>((r + 31) / 32));
    if (tr)
        bf16_copy_kernel<true><<<grid_out, blk, 0, st>>>(Y[cur], r, cc, ldc, xs, ldx);
    else
        bf16_copy_kernel<false><<<grid_out, blk, 0, st>>>(Y[cur], r, cc, ldc, xs, ldx);
    note_launch();
    return launch_status();
}
