"""GPU parity of the weight-gradient GEMM that accumulates into an FP32 main
gradient (main_grad += dW, no BF16 rounding), against the FP64 oracle.

Bar, per element, with y_ref the oracle's dW and want = main + y_ref:
    |got - want| <= 1e-2 |y_ref| + 1e-3 rms(y_ref) + 2^-23 |want|
The first two terms are the GEMM tolerance on the added part; the last is one
FP32 rounding of the final add into the main gradient, which the plain BF16
wgrad does not have (there the BF16 rounding sits inside the first term)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import scales_to_dev, tile_rows, to_dev

import blockwise_fp8_linear_weight_b300 as bfp8

pytestmark = pytest.mark.gpu
TILE = 128


def _ok(got, main, y_ref):
    want = main.astype(np.float64) + y_ref
    rms = float(np.sqrt(np.mean(y_ref ** 2))) if y_ref.size else 0.0
    allow = 1e-2 * np.abs(y_ref) + 1e-3 * rms + 2.0 ** -23 * np.abs(want)
    err = np.abs(got.astype(np.float64) - want)
    return bool(np.all(err <= allow)), float(np.max(err / np.maximum(allow, 1e-300)))


def _operands(M, N, K, seed):
    M128 = (M + TILE - 1) // TILE * TILE
    qdyt = wl.random_codes((N, M128), seed)
    qxt = wl.random_codes((K, M128), seed + 1)
    qdyt[:, M:] = 0
    qxt[:, M:] = 0
    sdyt = wl.random_scales((M128 // TILE, N), seed + 2)
    sxt = wl.random_scales((M128 // TILE, K), seed + 3)
    return qdyt, sdyt, qxt, sxt


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (130, 256, 384), (300, 512, 640), (1000, 384, 256)])
def test_wgrad_acc_random_codes(M, N, K):
    qdyt, sdyt, qxt, sxt = _operands(M, N, K, seed=M + N)
    main = np.random.default_rng(K).standard_normal((N, K)).astype(np.float32)
    mg = torch.from_numpy(main.copy()).cuda()
    bfp8.fp8_block_gemm_wgrad_acc(to_dev(qdyt), scales_to_dev(sdyt), to_dev(qxt), scales_to_dev(sxt), M, mg)
    torch.cuda.synchronize()
    ref = oracle.gemm_wgrad_accumulate(main, qdyt, sdyt, qxt, sxt, M) - main.astype(np.float64)
    ok, ratio = _ok(mg.cpu().numpy(), main, ref)
    assert ok, f"worst error/allowance = {ratio:.3g}"


def test_wgrad_acc_twice_adds_twice_and_padded_stride():
    """Two calls add dW twice; the main gradient may have a padded row stride,
    and the padding columns are left untouched."""
    M, N, K = 200, 256, 256
    qdyt, sdyt, qxt, sxt = _operands(M, N, K, seed=9)
    buf = torch.full((N, K + 4), 7.0, dtype=torch.float32, device="cuda")
    mg = buf[:, :K]
    mg.zero_()
    args = (to_dev(qdyt), scales_to_dev(sdyt), to_dev(qxt), scales_to_dev(sxt), M)
    bfp8.fp8_block_gemm_wgrad_acc(*args, mg)
    bfp8.fp8_block_gemm_wgrad_acc(*args, mg)
    torch.cuda.synchronize()
    y_ref = oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, M)
    ok, ratio = _ok(mg.cpu().numpy(), np.zeros((N, K), np.float32), 2.0 * y_ref)
    assert ok, f"worst error/allowance = {ratio:.3g}"
    assert torch.all(buf[:, K:] == 7.0)


def test_wgrad_acc_matches_bf16_wgrad_before_rounding():
    """From a zero main gradient the FP32 result rounds to the BF16 wgrad's output
    within one BF16 rounding (both come from the same FP32 sums)."""
    M, N, K = 384, 256, 512
    qdyt, sdyt, qxt, sxt = _operands(M, N, K, seed=31)
    args = (to_dev(qdyt), scales_to_dev(sdyt), to_dev(qxt), scales_to_dev(sxt), M)
    mg = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    bfp8.fp8_block_gemm_wgrad_acc(*args, mg)
    dw = bfp8.fp8_block_gemm_wgrad(*args)
    torch.cuda.synchronize()
    assert torch.equal(mg.to(torch.bfloat16), dw)


@pytest.mark.parametrize("lin", list(wl.mlp_projections().linears), ids=lambda l: f"{l.name}-M{l.M}")
def test_wgrad_acc_mlp_shapes_every_tile(lin):
    x, _, dy = wl.make_linear(lin)
    qdyt, sdyt = oracle.quantize_transpose(dy)
    qxt, sxt = oracle.quantize_transpose(x)
    rows = tile_rows(lin.N, lin.K)
    main = np.random.default_rng(5).standard_normal((lin.N, lin.K)).astype(np.float32)
    mg = torch.from_numpy(main).cuda()
    bfp8.fp8_block_gemm_wgrad_acc(to_dev(qdyt), scales_to_dev(sdyt), to_dev(qxt), scales_to_dev(sxt), lin.M, mg)
    torch.cuda.synchronize()
    ref = oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, lin.M, rows=rows)
    ok, ratio = _ok(mg.cpu().numpy()[rows], main[rows], ref)
    assert ok, f"worst error/allowance = {ratio:.3g}"
