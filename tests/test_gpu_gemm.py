"""GPU parity of the three blockwise-FP8 GEMMs against the FP64 oracle.

Every input comes from the seeded generators or from the oracle's own
quantisers (never from the CUDA path). Bar, on every compared element:
    |y - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref)
with y_ref the oracle's FP64 result from the same codes and scales and rms over
the compared output (the whole matrix for small shapes, the sampled rows at
full size). Small shapes are compared in full and span several tiles and a
ragged tail; the Puro-2B workload shapes are compared, in the launch
configuration the benchmark uses, on one random row of every 128-row output
tile (plus the first and last rows and a few more at random) over all columns,
so that every output tile of every pass is checked.

Every GEMM runs with and without the optional workspace: with it, a grid whose
last round of tiles is partial splits that round along the contraction axis
(FP32 partial tiles summed by a second kernel), so the small shapes below take
that path with many pieces per tile; the full-size shapes run with it, as the
benchmark does."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import from_dev_bf16, gemm_tolerance_ok, scales_to_dev, tile_rows, to_dev

import blockwise_fp8_linear_weight_b300 as bfp8

pytestmark = pytest.mark.gpu
TILE = 128


@pytest.fixture(params=[128, 192, 256], ids=lambda t: f"tileN{t}")
def tile_n(request):
    """Every tile configuration: 128-wide tiles, 192-wide tiles with 12 promotion warps
    (forward and weight gradient; the input gradient then runs 256-wide), and 256-wide
    tiles (the default)."""
    prev_t = bfp8.set_gemm_tile_n(request.param)
    yield request.param
    bfp8.set_gemm_tile_n(prev_t)


@pytest.fixture(scope="module")
def workspace():
    return bfp8.gemm_workspace()


@pytest.fixture(params=["plain", "split"])
def ws(request, workspace):
    """No workspace (whole tiles only), or the workspace (tail split along the contraction)."""
    return workspace if request.param == "split" else None


def _check(y_gpu, y_ref, what):
    ok, ratio = gemm_tolerance_ok(y_gpu, y_ref)
    assert ok, f"{what}: worst error/allowance = {ratio:.3g}"


# ------------------------------------------------------------------ per-pass runners
def run_fwd(qx, sx, qw, sw, rows=None, ws=None):
    y = bfp8.fp8_block_gemm_fwd(to_dev(qx), scales_to_dev(sx), to_dev(qw), to_dev(sw), workspace=ws)
    torch.cuda.synchronize()
    y = from_dev_bf16(y)
    ref = oracle.gemm_fwd(qx, sx, qw, sw, rows=rows)
    return (y if rows is None else y[rows]), ref


def run_dgrad(qdy, sdy, qw, sw, rows=None, ws=None):
    dx = bfp8.fp8_block_gemm_dgrad(to_dev(qdy), scales_to_dev(sdy), to_dev(qw), to_dev(sw), workspace=ws)
    torch.cuda.synchronize()
    dx = from_dev_bf16(dx)
    ref = oracle.gemm_dgrad(qdy, sdy, qw, sw, rows=rows)
    return (dx if rows is None else dx[rows]), ref


def run_wgrad(qdyt, sdyt, qxt, sxt, M, rows=None, ws=None):
    dw = bfp8.fp8_block_gemm_wgrad(to_dev(qdyt), scales_to_dev(sdyt), to_dev(qxt), scales_to_dev(sxt), M,
                                   workspace=ws)
    torch.cuda.synchronize()
    dw = from_dev_bf16(dw)
    ref = oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, M, rows=rows)
    return (dw if rows is None else dw[rows]), ref


# ------------------------------------------------------------------ random codes and scales
SMALL = [(1, 128, 128), (5, 256, 128), (128, 128, 256), (200, 384, 640), (256, 256, 256), (300, 512, 384),
         (129, 640, 1024), (600, 384, 512)]


@pytest.mark.parametrize("M,N,K", SMALL)
def test_fwd_random_codes(tile_n, ws, M, N, K):
    qx = wl.random_codes((M, K), 1)
    sx = wl.random_scales((K // TILE, M), 2)
    qw = wl.random_codes((N, K), 3)
    sw = wl.random_scales((N // TILE, K // TILE), 4)
    _check(*run_fwd(qx, sx, qw, sw, ws=ws), "fwd")


@pytest.mark.parametrize("M,N,K", SMALL)
def test_dgrad_random_codes(tile_n, ws, M, N, K):
    qdy = wl.random_codes((M, N), 5)
    sdy = wl.random_scales((N // TILE, M), 6)
    qw = wl.random_codes((N, K), 7)
    sw = wl.random_scales((N // TILE, K // TILE), 8)
    _check(*run_dgrad(qdy, sdy, qw, sw, ws=ws), "dgrad")


@pytest.mark.parametrize("M,N,K", SMALL)
def test_wgrad_random_codes(tile_n, ws, M, N, K):
    M128 = (M + TILE - 1) // TILE * TILE
    qdyt = wl.random_codes((N, M128), 9)
    qxt = wl.random_codes((K, M128), 10)
    qdyt[:, M:] = 0
    qxt[:, M:] = 0
    sdyt = wl.random_scales((M128 // TILE, N), 11)
    sxt = wl.random_scales((M128 // TILE, K), 12)
    _check(*run_wgrad(qdyt, sdyt, qxt, sxt, M, ws=ws), "wgrad")


def test_zero_scale_chunks_and_single_chunk(tile_n, ws):
    """All-zero tiles (scale 0) contribute nothing; a lone non-zero chunk is one dot product."""
    M, N, K = 130, 256, 512
    qx = wl.random_codes((M, K), 21)
    sx = wl.random_scales((K // TILE, M), 22)
    sx[1, :] = 0.0
    qx[:, 2 * TILE:3 * TILE] = 0
    qw = wl.random_codes((N, K), 23)
    sw = wl.random_scales((N // TILE, K // TILE), 24)
    _check(*run_fwd(qx, sx, qw, sw, ws=ws), "fwd with zero chunks")


# ------------------------------------------------------------------ quantise (oracle) then GEMM
def _linear_case(lin, rows_m=None, rows_n=None, ws=None):
    x, w, dy = wl.make_linear(lin)
    qx, sx = oracle.quantize_act(x)
    qw, sw = oracle.quantize_weight(w)
    qdy, sdy = oracle.quantize_act(dy)
    qdyt, sdyt = oracle.quantize_transpose(dy)
    qxt, sxt = oracle.quantize_transpose(x)
    _check(*run_fwd(qx, sx, qw, sw, rows_m, ws=ws), f"{lin.name} fwd")
    _check(*run_dgrad(qdy, sdy, qw, sw, rows_m, ws=ws), f"{lin.name} dgrad")
    _check(*run_wgrad(qdyt, sdyt, qxt, sxt, lin.M, rows_n, ws=ws), f"{lin.name} wgrad")


@pytest.mark.parametrize("M,K,N", [(256, 256, 256), (1000, 512, 384), (333, 256, 640)])
def test_quantised_linear_small_full_compare(tile_n, ws, M, K, N):
    _linear_case(wl.Linear("small", M, K, N, "student_t3", M), ws=ws)


def test_single_linear_256_config(tile_n):
    """One linear, forward only: X [256,256] ~ N(0,1), W [256,256] ~ N(0, 0.02^2), seed 0; full compare."""
    lin = wl.single_linear_256().linears[0]
    x, w, _ = wl.make_linear(lin)
    qx, sx = oracle.quantize_act(x)
    qw, sw = oracle.quantize_weight(w)
    _check(*run_fwd(qx, sx, qw, sw), "single linear fwd")


def _full_size_cases():
    cases = list(wl.attention_projections().linears) + list(wl.mlp_projections().linears)
    cases += list(wl.full_stack(layers=1).linears)
    return cases


@pytest.mark.parametrize("lin", _full_size_cases(), ids=lambda l: f"{l.name}-M{l.M}-K{l.K}-N{l.N}")
def test_workload_shapes_every_tile(lin, workspace):
    _linear_case(lin, tile_rows(lin.M, lin.M + lin.N), tile_rows(lin.N, lin.K), ws=workspace)


@pytest.mark.parametrize("lin", wl.shape_sweep(), ids=lambda l: l.name)
def test_shape_sweep_every_tile(lin, workspace):
    _linear_case(lin, tile_rows(lin.M, lin.M + lin.N, extra=0), tile_rows(lin.N, lin.K, extra=0), ws=workspace)


# ------------------------------------------------------------------ guard bands around the outputs
CANARY = 0x7FA5  # a BF16 NaN pattern no GEMM writes


def _guarded(rows, cols, dev="cuda"):
    """A BF16 output view of rows x cols inside a larger buffer filled with a canary: two rows
    above and below, 8 columns to the left and 56 to the right (row stride cols + 64, so the
    view keeps 16-byte alignment)."""
    ld = cols + 64
    buf = torch.full((rows + 4, ld), CANARY, dtype=torch.int16, device=dev)
    return buf, buf[2:2 + rows, 8:8 + cols].view(torch.bfloat16)


def _untouched(buf, rows, cols):
    b = buf.cpu().numpy().view(np.uint16)
    mask = np.ones(b.shape, bool)
    mask[2:2 + rows, 8:8 + cols] = False
    return bool(np.all(b[mask] == CANARY))


@pytest.mark.parametrize("M,N,K", [(200, 384, 256), (129, 256, 640), (700, 384, 640)])
def test_outputs_leave_their_guard_bands_untouched(tile_n, ws, M, N, K):
    """Each pass writes exactly its M x N (or M x K, N x K) output through a strided view:
    nothing outside it changes, and the view itself matches the oracle."""
    M128 = (M + TILE - 1) // TILE * TILE
    qx, sx = wl.random_codes((M, K), 51), wl.random_scales((K // TILE, M), 52)
    qw, sw = wl.random_codes((N, K), 53), wl.random_scales((N // TILE, K // TILE), 54)
    qdy, sdy = wl.random_codes((M, N), 55), wl.random_scales((N // TILE, M), 56)
    qdyt, qxt = wl.random_codes((N, M128), 57), wl.random_codes((K, M128), 58)
    qdyt[:, M:] = 0
    qxt[:, M:] = 0
    sdyt, sxt = wl.random_scales((M128 // TILE, N), 59), wl.random_scales((M128 // TILE, K), 60)
    buf, y = _guarded(M, N)
    bfp8.fp8_block_gemm_fwd(to_dev(qx), scales_to_dev(sx), to_dev(qw), to_dev(sw), y, workspace=ws)
    buf2, dx = _guarded(M, K)
    bfp8.fp8_block_gemm_dgrad(to_dev(qdy), scales_to_dev(sdy), to_dev(qw), to_dev(sw), dx, workspace=ws)
    buf3, dw = _guarded(N, K)
    bfp8.fp8_block_gemm_wgrad(to_dev(qdyt), scales_to_dev(sdyt), to_dev(qxt), scales_to_dev(sxt), M, dw,
                              workspace=ws)
    torch.cuda.synchronize()
    assert _untouched(buf, M, N) and _untouched(buf2, M, K) and _untouched(buf3, N, K)
    _check(from_dev_bf16(y), oracle.gemm_fwd(qx, sx, qw, sw), "fwd")
    _check(from_dev_bf16(dx), oracle.gemm_dgrad(qdy, sdy, qw, sw), "dgrad")
    _check(from_dev_bf16(dw), oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, M), "wgrad")


# ------------------------------------------------------------------ the tail split itself
def _launches(fn):
    n0 = bfp8.kernel_launches()
    out = fn()
    torch.cuda.synchronize()
    return bfp8.kernel_launches() - n0, out


def _expect_split(tiles, nc, sms):
    """The library's rule: a partial last round leaving a quarter of the SMs idle, and a split
    that shortens the longest CTA's tail by at least 40 chunks."""
    rounds, rest = divmod(tiles, sms)
    if rest == 0 or 4 * rest > 3 * sms:
        return False
    g = sms if rounds else min(rest * nc, sms)
    return nc - (-(-(rest * nc) // g)) >= 40


@pytest.mark.parametrize("M,N,K", [(8192, 12288, 2048), (8192, 2048, 12288), (4000, 384, 12288)])
def test_tail_split_is_taken_and_deterministic(workspace, M, N, K):
    """With the workspace, a grid whose last round is partial launches the whole rounds, the
    tail's pieces and the tail reduce, gives the same bits on every call, and stays within the
    oracle's bar on rows of the split tiles; without it, one launch. Shapes: the MLP forward GEMM
    (3072 output tiles of 128 x 256 on 148 SMs: no split), the MLP input-gradient GEMM's shape
    (512 tiles, 96 chunks) and a small ragged one (64 tiles, 96 chunks)."""
    qx, sx = wl.random_codes((M, K), 71), wl.random_scales((K // TILE, M), 72)
    qw, sw = wl.random_codes((N, K), 73), wl.random_scales((N // TILE, K // TILE), 74)
    dqx, dsx, dqw, dsw = to_dev(qx), scales_to_dev(sx), to_dev(qw), to_dev(sw)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = ((M + TILE - 1) // TILE) * ((N + 255) // 256)
    expect_split = _expect_split(tiles, K // TILE, sms)
    if (M, N, K) != (8192, 12288, 2048):
        assert expect_split
    n1, y1 = _launches(lambda: bfp8.fp8_block_gemm_fwd(dqx, dsx, dqw, dsw, workspace=workspace))
    n2, y2 = _launches(lambda: bfp8.fp8_block_gemm_fwd(dqx, dsx, dqw, dsw, workspace=workspace))
    n0, y0 = _launches(lambda: bfp8.fp8_block_gemm_fwd(dqx, dsx, dqw, dsw))
    assert n0 == 1
    # split: the whole rounds (if any), the tail's pieces, the reduce of the partial tiles
    assert n1 == n2 == ((3 if tiles >= sms else 2) if expect_split else 1)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # rows of the last tiles (the tail, in the N-fastest or M-fastest tile order) and of the first
    rows = np.unique(np.concatenate([tile_rows(M, 5, extra=0)[-8:], tile_rows(M, 6, extra=0)[:2]]))
    ref = oracle.gemm_fwd(qx, sx, qw, sw, rows=rows)
    _check(from_dev_bf16(y1)[rows], ref, "fwd with the tail split")
    _check(from_dev_bf16(y0)[rows], ref, "fwd without the split")


def test_tail_with_fewer_chunks_than_ctas(workspace):
    """One whole round of 148 tiles plus one tail tile of 42 chunks: 42 tail chunks over 148 CTAs,
    so most CTAs have an empty tail range and each chunk of the tail tile is its own piece. All
    three passes, compared on a row of every tile (the tail tile's included) and its last row."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    R, C, X = TILE * (sms + 1), 256, 5376  # R rows of output, C columns, contraction X (42 chunks)
    qa, sa = wl.random_codes((R, X), 81), wl.random_scales((X // TILE, R), 82)
    qb, sb = wl.random_codes((C, X), 83), wl.random_scales((C // TILE, X // TILE), 84)
    rows = tile_rows(R, 85, extra=0)
    for ws_ in (workspace, None):
        _check(*run_fwd(qa, sa, qb, sb, rows, ws=ws_), "fwd")
    # dgrad: dx [R][C] = dy [R][X] W [X][C]
    qw, sw = wl.random_codes((X, C), 86), wl.random_scales((X // TILE, C // TILE), 87)
    _check(*run_dgrad(qa, sa, qw, sw, rows, ws=workspace), "dgrad")
    # wgrad: dW [R][C] from dy^T [R][X] and x^T [C][X] (contraction X = tokens)
    qdyt, sdyt = wl.random_codes((R, X), 88), wl.random_scales((X // TILE, R), 89)
    qxt, sxt = wl.random_codes((C, X), 90), wl.random_scales((X // TILE, C), 91)
    _check(*run_wgrad(qdyt, sdyt, qxt, sxt, X, rows, ws=workspace), "wgrad")


@pytest.mark.parametrize("M,N,K,Mw", [(200, 384, 5376, 5300), (129, 640, 5504, 5400)])
def test_small_shapes_with_split_tail(tile_n, workspace, M, N, K, Mw):
    """Few tiles with a long contraction: every tile is cut into pieces of one or two chunks over
    many CTAs (the ragged last row and column tiles included); full compare of all three passes
    in every tile width. Forward and input gradient contract over K and N; the weight gradient
    over Mw tokens (M128 = 5376 or 5504) into a [N][384] dW."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bn = 256 if tile_n == 256 else tile_n
    assert _expect_split(-(-M // TILE) * -(-N // bn), K // TILE, sms)
    qx, sx = wl.random_codes((M, K), 61), wl.random_scales((K // TILE, M), 62)
    qw, sw = wl.random_codes((N, K), 63), wl.random_scales((N // TILE, K // TILE), 64)
    _check(*run_fwd(qx, sx, qw, sw, ws=workspace), "fwd")
    # dgrad contracts over its N: a [M][K] x [K][N] problem with the roles of N and K swapped
    qdy, sdy = wl.random_codes((M, K), 65), wl.random_scales((K // TILE, M), 66)
    qw2, sw2 = wl.random_codes((K, N), 67), wl.random_scales((K // TILE, N // TILE), 68)
    _check(*run_dgrad(qdy, sdy, qw2, sw2, ws=workspace), "dgrad")
    M128 = (Mw + TILE - 1) // TILE * TILE
    qdyt, qxt = wl.random_codes((N, M128), 69), wl.random_codes((384, M128), 70)
    qdyt[:, Mw:] = 0
    qxt[:, Mw:] = 0
    sdyt, sxt = wl.random_scales((M128 // TILE, N), 71), wl.random_scales((M128 // TILE, 384), 72)
    _check(*run_wgrad(qdyt, sdyt, qxt, sxt, Mw, ws=workspace), "wgrad")


@pytest.mark.parametrize("M,N,K", [(1, 256, 8192), (3, 640, 6144)])
def test_split_tail_with_a_single_row_tile(workspace, M, N, K):
    """A handful of output rows and a long contraction: one or three tiles, each cut into one-chunk
    pieces over 64-144 CTAs; the partial tiles' rows past M are zero and must not be written."""
    qx, sx = wl.random_codes((M, K), 95), wl.random_scales((K // TILE, M), 96)
    qw, sw = wl.random_codes((N, K), 97), wl.random_scales((N // TILE, K // TILE), 98)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _expect_split(-(-N // 256), K // TILE, sms)
    buf, y = _guarded(M, N)
    bfp8.fp8_block_gemm_fwd(to_dev(qx), scales_to_dev(sx), to_dev(qw), to_dev(sw), y, workspace=workspace)
    torch.cuda.synchronize()
    assert _untouched(buf, M, N)
    _check(from_dev_bf16(y), oracle.gemm_fwd(qx, sx, qw, sw), "fwd, split single row tile")


def test_split_gemm_replays_from_a_cuda_graph(workspace):
    """The split launches (whole rounds, pieces as a programmatic dependent, tail reduce) captured in
    a CUDA graph replay to the eager call's bits, also after new operands are copied in."""
    M, N, K = 8192, 2048, 12288  # 512 output tiles, 96 chunks: the rounds, the pieces and the reduce
    qx, sx = wl.random_codes((M, K), 101), wl.random_scales((K // TILE, M), 102)
    qw, sw = wl.random_codes((N, K), 103), wl.random_scales((N // TILE, K // TILE), 104)
    dqx, dsx, dqw, dsw = to_dev(qx), scales_to_dev(sx), to_dev(qw), to_dev(sw)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    n, _ = _launches(lambda: bfp8.fp8_block_gemm_fwd(dqx, dsx, dqw, dsw, y, workspace=workspace))
    assert n == 3
    want = y.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        bfp8.fp8_block_gemm_fwd(dqx, dsx, dqw, dsw, y, workspace=workspace)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bfp8.fp8_block_gemm_fwd(dqx, dsx, dqw, dsw, y, workspace=workspace)
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), want.view(torch.int16))
    # doubled activation scales double every output exactly (a power of two)
    dsx.mul_(2.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y.float(), 2.0 * want.float())
