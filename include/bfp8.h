/*
 * bfp8.h — C ABI of the blockwise-FP8 linear-layer library for B300 (sm_103a).
 *
 * What the library computes. The Puro-2B pretraining recipe runs the matrix
 * multiplications of its main linear layers in FP8, "following DeepSeek-V3's
 * fine-grained block quantisation", and keeps numerically sensitive work and
 * training state in BF16/FP32 (Puro-2B article on en.roboind.com, section
 * "FP8 takes advantage of the RTX 5090's low precision efficiency"; the
 * ainews.surl.tw article "Puro-2B Publishes a Consumer-Grade GPU Pretraining
 * Recipe ..." names it "blockwise FP8"). The pages fix no further detail; this
 * library adopts the DeepSeek-V3 convention:
 *   - activation tiles of 1x128 along the contraction axis, weight blocks of
 *     128x128;
 *   - codes in OCP E4M3FN (largest finite value 448);
 *   - one FP32 scale per tile: s = fl32(amax / 448), IEEE division;
 *   - code = e4m3_rn_satfinite(fl32(x / s)), IEEE division, then round to
 *     nearest-even with saturation to +-448; an all-zero tile has s = 0 and
 *     signed-zero codes (0x00 / 0x80 by the input's sign);
 *   - GEMMs: FP8 tensor-core products summed in FP32 per 128-wide chunk of the
 *     contraction axis, each chunk promoted into an FP32 accumulator with the
 *     product of its two scales; BF16 output, rounded to nearest-even.
 * A linear layer y = x W^T (x [M,K], W [N,K]) uses six calls per training
 * step: fp8_quantize_act(x), fp8_quantize_weight(W), fp8_block_gemm_fwd;
 * fp8_quantize_act(dy), fp8_block_gemm_dgrad; fp8_quantize_transpose(dy),
 * fp8_quantize_transpose(x), fp8_block_gemm_wgrad.
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers on the current CUDA device, owned and
 *     allocated by the caller. The library allocates nothing, frees nothing
 *     and never synchronises (except bfp8_last_device_status).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Calls are asynchronous on that stream.
 *   - Matrices are row-major; ld* arguments are row strides in ELEMENTS.
 *   - BF16 arrays are passed as void* holding IEEE bfloat16 bit patterns.
 *   - Arguments are checked on the host before any launch. Return value:
 *     BFP8_OK, or a negative bfp8_status; nothing is launched on error.
 *   - Inputs must be finite; NaN/Inf inputs give unspecified codes.
 *   - Outputs must not overlap inputs or each other.
 */
#ifndef BFP8_H
#define BFP8_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BFP8_OK = 0,
    BFP8_EINVAL = -1,   /* null pointer, negative size, leading dimension too small */
    BFP8_EALIGN = -2,   /* pointer or leading dimension breaks a 16-byte (TMA / vector) rule */
    BFP8_ESHAPE = -3,   /* a dimension that must be a multiple of 128 is not, or is too large */
    BFP8_ELAUNCH = -4,  /* the CUDA launch (or tensor-map encoding) failed */
    BFP8_ETIMEOUT = -5, /* a kernel gave up on a bounded wait (from bfp8_last_device_status) */
    BFP8_EARCH = -6     /* the current device is not compute capability 10.3 (sm_103) */
} bfp8_status;

/* Activation quantiser: 1x128 tiles along the columns.
 *   x [R][C] bf16 (ldx), C a multiple of 128, R >= 0 (R = 0 is a no-op).
 *   q [R][C] E4M3 codes (ldq), s [C/128][R] FP32 scales, chunk-major (lds >= R).
 * Used for x in the forward pass (tiles along K) and for dy in the input-
 * gradient pass (tiles along N).
 * Alignment: x 16 B and ldx % 8 == 0; q 8 B and ldq % 8 == 0; s 4 B. */
int fp8_quantize_act(const void* x, int64_t R, int64_t C, int64_t ldx,
                     uint8_t* q, int64_t ldq, float* s, int64_t lds, void* stream);

/* Weight quantiser: 128x128 blocks.
 *   w [N][K] bf16 (ldw), N and K multiples of 128.
 *   q [N][K] E4M3 codes (ldq), s [N/128][K/128] FP32 scales, dense.
 * The same codes and scales serve the forward and the input-gradient GEMM.
 * Alignment: w 16 B and ldw % 8 == 0; q 8 B and ldq % 8 == 0; s 4 B. */
int fp8_quantize_weight(const void* w, int64_t N, int64_t K, int64_t ldw,
                        uint8_t* q, int64_t ldq, float* s, void* stream);

/* Transposed activation quantiser (operands of the weight-gradient GEMM):
 * 1x128 tiles run down the columns of x, i.e. along the R rows (tokens), and
 * the codes are written transposed.
 *   x [R][C] bf16 (ldx), C a multiple of 128, R >= 0; R128 = R rounded up to 128.
 *   qt [C][R128] E4M3 codes (ldqt >= R128); pad columns R..R128-1 get 0x00.
 *   st [R128/128][C] FP32 scales (ldst >= C); a chunk's scale covers its valid rows.
 * Alignment: x 16 B and ldx % 8 == 0; qt 16 B and ldqt % 16 == 0;
 * st 8 B and ldst % 2 == 0. */
int fp8_quantize_transpose(const void* x, int64_t R, int64_t C, int64_t ldx,
                           uint8_t* qt, int64_t ldqt, float* st, int64_t ldst, void* stream);

/* Both activation layouts in one pass over x: exactly the outputs of
 * fp8_quantize_act(x, R, C, ldx, q, ldq, s, lds) and of
 * fp8_quantize_transpose(x, R, C, ldx, qt, ldqt, st, ldst), reading x once.
 * A training step needs both layouts of x (forward and weight-gradient GEMMs)
 * and of dy (input- and weight-gradient GEMMs); this call saves one read of
 * the BF16 tensor. Arguments, alignment rules and errors are the union of the
 * two calls'. */
int fp8_quantize_act_transpose(const void* x, int64_t R, int64_t C, int64_t ldx,
                               uint8_t* q, int64_t ldq, float* s, int64_t lds,
                               uint8_t* qt, int64_t ldqt, float* st, int64_t ldst, void* stream);

/* Workspace of the three BF16 GEMMs below (fwd, dgrad, wgrad), all optional.
 * The GEMMs run one persistent CTA per SM over 128-row output tiles. When the
 * tiles do not fill the grid's last round, that partial round (the tail) can
 * be split along the contraction axis: the whole rounds run in one launch; a
 * second launch, which starts on the SMs that the first one frees, gives
 * every CTA an equal contiguous share of the tail tiles' 128-wide chunks and
 * writes pieces that are not a whole tile to the workspace as FP32 partial
 * tiles; a third kernel adds the pieces of each tile in a fixed order and
 * stores it in BF16 (all on `stream`). The tail then costs about (tail tiles / SMs) of a round instead of
 * a whole round, and results stay deterministic (the same inputs give the
 * same bits on every call); they differ from the unsplit GEMM's only in the
 * FP32 summation order of the split tiles. The split is used when
 * `workspace` is non-NULL, `workspace_bytes` is at least the size below, the
 * tail leaves at least a quarter of the SMs idle, and splitting shortens the
 * longest CTA's share of the tail by at least 40 chunks of 128 (below that,
 * the extra launches and the partial tiles cost about what they save).
 *   workspace: caller-owned device memory, 16-byte aligned, used as scratch
 *   for the duration of the call (stream-ordered); calls that share one
 *   workspace must be ordered on the device (one stream, or events).
 *   NULL (or fewer bytes) = no split, the same results as before the split
 *   existed, bit for bit.
 * fp8_block_gemm_workspace_bytes: the size that enables the split on the
 * current device (two FP32 partial tiles of 128 x 256 per SM: 37.9 MB on a
 * 148-SM B300). */
int fp8_block_gemm_workspace_bytes(int64_t* bytes);

/* Forward GEMM, y = x W^T:
 *   y[m][n] = bf16( sum_kb sx[kb][m] * sw[n/128][kb] * sum_{k in kb} qx[m][k] qw[n][k] )
 *   qx [M][K] (ldqx), sx [K/128][M] (ldsx), qw [N][K] (ldqw), sw [N/128][K/128] dense,
 *   y [M][N] bf16 (ldy). K, N multiples of 128; M >= 0 any (M = 0 is a no-op).
 *   workspace, workspace_bytes: see fp8_block_gemm_workspace_bytes (NULL, 0: none).
 * Alignment: qx, qw, sx, y, workspace 16 B; ldqx, ldqw % 16 == 0; ldsx % 4 == 0;
 * ldy % 8 == 0. */
int fp8_block_gemm_fwd(const uint8_t* qx, int64_t ldqx, const float* sx, int64_t ldsx,
                       const uint8_t* qw, int64_t ldqw, const float* sw,
                       void* y, int64_t ldy, int64_t M, int64_t N, int64_t K,
                       void* workspace, int64_t workspace_bytes, void* stream);

/* Input-gradient GEMM, dx = dy W (contraction over the layer's N outputs):
 *   dx[m][k] = bf16( sum_nb sdy[nb][m] * sw[nb][k/128] * sum_{n in nb} qdy[m][n] qw[n][k] )
 *   qdy [M][N] (ldqdy), sdy [N/128][M] (ldsdy), qw/sw exactly as produced for the
 *   forward pass (qw is read with the contraction axis strided), dx [M][K] bf16 (lddx).
 *   workspace, workspace_bytes: as fp8_block_gemm_fwd.
 * Alignment: as fp8_block_gemm_fwd. */
int fp8_block_gemm_dgrad(const uint8_t* qdy, int64_t ldqdy, const float* sdy, int64_t ldsdy,
                         const uint8_t* qw, int64_t ldqw, const float* sw,
                         void* dx, int64_t lddx, int64_t M, int64_t N, int64_t K,
                         void* workspace, int64_t workspace_bytes, void* stream);

/* Weight-gradient GEMM, dW = dy^T x (contraction over the M tokens, padded
 * with zero codes to M128):
 *   dw[n][k] = bf16( sum_mb sdyt[mb][n] * sxt[mb][k] * sum_{m in mb} qdyt[n][m] qxt[k][m] )
 *   qdyt [N][M128] (ldqdyt), sdyt [M128/128][N] (ldsdyt), qxt [K][M128] (ldqxt),
 *   sxt [M128/128][K] (ldsxt), all from fp8_quantize_transpose; dw [N][K] bf16 (lddw).
 *   M >= 1 any; N, K multiples of 128.
 *   workspace, workspace_bytes: as fp8_block_gemm_fwd.
 * Alignment: qdyt, qxt, sdyt, sxt, dw, workspace 16 B; ldqdyt, ldqxt % 16 == 0;
 * ldsdyt, ldsxt % 4 == 0; lddw % 8 == 0. */
int fp8_block_gemm_wgrad(const uint8_t* qdyt, int64_t ldqdyt, const float* sdyt, int64_t ldsdyt,
                         const uint8_t* qxt, int64_t ldqxt, const float* sxt, int64_t ldsxt,
                         void* dw, int64_t lddw, int64_t M, int64_t N, int64_t K,
                         void* workspace, int64_t workspace_bytes, void* stream);

/* Weight-gradient GEMM accumulated into an FP32 main gradient (the recipe
 * keeps training state in FP32; same article and section as above):
 *   main_grad[n][k] += sum_mb sdyt[mb][n] * sxt[mb][k] * sum_{m in mb} qdyt[n][m] qxt[k][m]
 * The sum is formed exactly as in fp8_block_gemm_wgrad, in FP32, and is not
 * rounded to BF16: the TMA unit adds each FP32 element into main_grad (one
 * FP32 add per element and call, round to nearest-even; subnormal sums may be
 * flushed to zero). Operands as fp8_block_gemm_wgrad; main_grad [N][K] FP32
 * (ldmg) is read and written in place. Each element is updated atomically, so
 * calls that target the same buffer add up in either order.
 * Alignment: as fp8_block_gemm_wgrad, with main_grad 16 B and ldmg % 4 == 0. */
int fp8_block_gemm_wgrad_acc(const uint8_t* qdyt, int64_t ldqdyt, const float* sdyt, int64_t ldsdyt,
                             const uint8_t* qxt, int64_t ldqxt, const float* sxt, int64_t ldsxt,
                             float* main_grad, int64_t ldmg, int64_t M, int64_t N, int64_t K, void* stream);

/* MuonH update (Puro-2B article on en.roboind.com, section "From ordinary
 * learning to effective learning": the update size is standardised on top of
 * Muon and the weight is projected back to a fixed radius afterwards). Read
 * plainly, with Frobenius norms |.|, U the Newton-Schulz orthogonalisation of
 * the gradient G, learning rate lr and radius R:
 *   X0 = G / (|G| + eps);  W' = W - lr R U / |U|;  W_new = R W' / |W'|.
 * The Newton-Schulz iterations between the two calls run in the library's BF16
 * GEMM (muonh_newton_schulz, below). Sums are deterministic
 * (fixed grid, fixed order). Matrices are row-major; cols a multiple of 4.
 *   partials, partials_len: caller-owned scratch of at least
 *     muonh_partials_len() doubles, 8-byte aligned (BFP8_EINVAL if shorter);
 *     overwritten by each call; calls that share it must be ordered.
 * muonh_partials_len: writes the number of doubles; BFP8_EINVAL for NULL. */
int muonh_partials_len(int* n);

/* x[r][c] = bf16_rn(g[r][c] / (|g| + eps)).
 *   g FP32 [rows][ldg] (16-byte aligned, ldg % 4 == 0), x BF16 [rows][ldx]
 *   (8-byte aligned, ldx % 4 == 0), eps >= 0.
 * Errors: BFP8_EINVAL (null, sizes, eps), BFP8_ESHAPE (cols % 4), BFP8_EALIGN. */
int muonh_normalize(const float* g, int64_t rows, int64_t cols, int64_t ldg, void* x, int64_t ldx,
                    double* partials, int64_t partials_len, float eps, void* stream);

/* w = R (w - a u) / |w - a u| in place, a = lr R / |u| (a = 0 if |u| = 0).
 * w - a u is formed in FP32 as fma(-a, u, w), and its norm is the sum of the
 * squares of exactly those values (FP32 within a row segment, FP64 beyond); if
 * that sum is zero, w is left unchanged. Three passes: u is read three times,
 * w twice, and w written once.
 *   w FP32 [rows][ldw] (16-byte aligned, ldw % 4 == 0), u BF16 [rows][ldu]
 *   (8-byte aligned, ldu % 4 == 0), lr >= 0, radius > 0.
 * Errors: as muonh_normalize (lr, radius checked as BFP8_EINVAL). */
int muonh_apply(float* w, int64_t ldw, const void* u, int64_t ldu, int64_t rows, int64_t cols,
                double* partials, int64_t partials_len, float lr, float radius, void* stream);

/* muonh_apply without caller scratch: the partial sums live in one
 * library-owned device array per device (grids of up to 512 CTAs; BFP8_EINVAL
 * on a device that would need more). Calls on a device share that array, so
 * they must be ordered (one stream, or synchronised); results are bit-identical
 * to muonh_apply. Arguments and errors otherwise as muonh_apply. */
int muonh_apply_static(float* w, int64_t ldw, const void* u, int64_t ldu, int64_t rows, int64_t cols,
                       float lr, float radius, void* stream);

/* BF16 GEMM with a scaled sum, the product of the Newton-Schulz iterations below:
 *   d[m][n] = bf16_rn( alpha * sum_k a[m][k] * B(k, n) + beta * c[m][n] )
 *   a BF16 [M][K] (lda); b BF16 [N][K] with B(k, n) = b[n][k] (b_mn_major = 0) or
 *   [K][N] with B(k, n) = b[k][n] (b_mn_major = 1), ldb; c BF16 [M][N] (ldc), read only
 *   if beta != 0 (may be NULL otherwise); d BF16 [M][N] (ldd). The tensor core sums the
 *   exact BF16 products in FP32 over the whole contraction; alpha and beta are applied
 *   in FP32, then one rounding to BF16. M, N, K >= 1, N a multiple of 8 (K and M any).
 * Alignment: every pointer 16 B, every leading dimension % 8 == 0. d must not overlap
 * a, b or c. */
int bf16_gemm_axpby(const void* a, int64_t lda, const void* b, int64_t ldb, int b_mn_major,
                    const void* c, int64_t ldc, void* d, int64_t ldd, int64_t M, int64_t N, int64_t K,
                    float alpha, float beta, void* stream);

/* Newton-Schulz orthogonalisation of the MuonH update (the Muon part of MuonH; same
 * article and section as muonh_normalize), in place on x, BF16 [rows][cols] (ldx):
 * `steps` quintic iterations X <- a X + (b A + c A A) X with A = X X^T, run on the
 * orientation with fewer rows (x^T when rows > cols). Each product is one
 * bf16_gemm_axpby (A and the B = b A + c A A matrix are rounded to BF16, as is X after
 * each step). rows and cols multiples of 8; x 16-byte aligned, ldx % 8 == 0.
 *   work, work_bytes: caller scratch of at least muonh_newton_schulz_work_bytes(rows,
 *     cols) bytes, 16-byte aligned (BFP8_EINVAL if shorter); overwritten by every call,
 *     so calls that share it must be ordered.
 * muonh_newton_schulz_work_bytes: writes the scratch size; BFP8_EINVAL for NULL or
 * sizes < 1. */
int muonh_newton_schulz_work_bytes(int64_t rows, int64_t cols, int64_t* bytes);
int muonh_newton_schulz(void* x, int64_t rows, int64_t cols, int64_t ldx, void* work, int64_t work_bytes,
                        int steps, float a, float b, float c, void* stream);

/* Human-readable name of a bfp8_status value (static string, never NULL). */
const char* bfp8_status_string(int status);

/* Synchronises `stream`, then reads and clears the device status word that a
 * kernel sets when it gives up on a bounded wait. Returns BFP8_OK,
 * BFP8_ETIMEOUT, or BFP8_ELAUNCH if the synchronisation itself failed. */
int bfp8_last_device_status(void* stream);

/* Limit of a single wait of a kernel on one of its own pipeline barriers, in
 * nanoseconds of the GPU's global timer: 0 restores the default (2 s);
 * otherwise 1000 <= ns <= 6e10. A kernel whose wait runs out records
 * BFP8_ETIMEOUT in the device status word (read by bfp8_last_device_status),
 * waits for its own copies in flight, releases its tensor memory and returns;
 * its outputs are then unspecified. Applies to later launches from every
 * thread. Returns BFP8_OK, or BFP8_EINVAL for a value out of range. */
int bfp8_set_wait_limit_ns(int64_t ns);

/* Test switch for the timeout path: with on = 1, later launches of the
 * quantisers and GEMMs start no operand copies, so their first pipeline wait
 * runs out (after the limit above) and the kernels unwind as described there.
 * Meant for tests of the error path only; on = 0 (default) restores normal
 * operation. Returns the previous setting (0 or 1), or BFP8_EINVAL. */
int bfp8_test_stall_producers(int on);

/* Number of kernels the library has launched in this process so far, on every
 * device and stream (host-side count of successful launch calls; a call that
 * is captured into a CUDA graph counts once, at capture). Returns BFP8_OK, or
 * BFP8_EINVAL for a NULL pointer. */
int bfp8_kernel_launches(int64_t* count);

/* Tuning knob for the GEMMs' output tile width: 0 = automatic (default),
 * 128, 192 or 256 columns (192 applies to the forward and weight-gradient
 * GEMMs, whose B operand is K-major; the input-gradient GEMM then uses 256).
 * Returns the previous setting, or BFP8_EINVAL. Applies to later calls from
 * every thread. */
int bfp8_set_gemm_tile_n(int tile_n);


#ifdef __cplusplus
}
#endif

#endif /* BFP8_H */
