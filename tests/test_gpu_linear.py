"""The one-layer call sequence (BlockwiseFP8Linear) on the GPU: its outputs
against the oracle, the weight-quantisation reuse across micro-batches, and
the FP32 main-gradient mode.

Bars: codes and scales bit-exact; GEMM outputs within
|y - y_ref| <= 1e-2 |y_ref| + 1e-3 rms(y_ref) of the oracle's FP64 result from
the oracle's own codes and scales."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import from_dev_bf16, gemm_tolerance_ok, to_dev_bf16

import blockwise_fp8_linear_weight_b300 as bfp8

pytestmark = pytest.mark.gpu


def _case(M=300, K=256, N=384):
    lin = wl.Linear("small", M, K, N, "student_t3", 11)
    x, w, dy = wl.make_linear(lin)
    return lin, x, w, dy


def _check(got, ref, what):
    ok, ratio = gemm_tolerance_ok(got, ref)
    assert ok, f"{what}: worst error/allowance = {ratio:.3g}"


def test_layer_step_matches_oracle():
    lin, x, w, dy = _case()
    layer = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N)
    y = layer.forward(to_dev_bf16(x), to_dev_bf16(w))
    dx, dw = layer.backward(to_dev_bf16(dy))
    torch.cuda.synchronize()
    qx, sx = oracle.quantize_act(x)
    qw, sw = oracle.quantize_weight(w)
    qdy, sdy = oracle.quantize_act(dy)
    qdyt, sdyt = oracle.quantize_transpose(dy)
    qxt, sxt = oracle.quantize_transpose(x)
    assert np.array_equal(layer.qw.cpu().numpy(), qw)
    assert np.array_equal(layer.sw.cpu().numpy().view(np.uint32), sw.view(np.uint32))
    _check(from_dev_bf16(y), oracle.gemm_fwd(qx, sx, qw, sw), "fwd")
    _check(from_dev_bf16(dx), oracle.gemm_dgrad(qdy, sdy, qw, sw), "dgrad")
    _check(from_dev_bf16(dw), oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, lin.M), "wgrad")


def test_weight_quantisation_is_reused_until_the_weight_changes():
    lin, x, w, _ = _case()
    layer = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N, reuse_weight_quant=True)
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    y1 = layer.forward(xd, wd).clone()
    y2 = layer.forward(xd, wd).clone()
    assert layer.weight_quant_calls == 1
    assert torch.equal(y1, y2)
    sw1 = layer.sw.clone()
    # an in-place update (what an optimizer step does) bumps the version: re-quantised;
    # a power-of-two factor keeps every code and doubles every scale and output exactly
    wd.mul_(2.0)
    y3 = layer.forward(xd, wd).clone()
    assert layer.weight_quant_calls == 2
    assert torch.equal(layer.sw, 2.0 * sw1)
    assert torch.equal(y3, 2.0 * y1)
    # a different tensor with the same contents is quantised too
    layer.forward(xd, wd.clone())
    assert layer.weight_quant_calls == 3
    # without reuse every forward quantises
    plain = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N)
    plain.forward(xd, wd)
    plain.forward(xd, wd)
    assert plain.weight_quant_calls == 2


def _oracle_step(x, w, dy, M):
    """y, dx, dW of one step from the oracle's codes and scales of (x, w, dy)."""
    qx, sx = oracle.quantize_act(x)
    qw, sw = oracle.quantize_weight(w)
    qdy, sdy = oracle.quantize_act(dy)
    qdyt, sdyt = oracle.quantize_transpose(dy)
    qxt, sxt = oracle.quantize_transpose(x)
    return (oracle.gemm_fwd(qx, sx, qw, sw), oracle.gemm_dgrad(qdy, sdy, qw, sw),
            oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, M), qw, sw)


def _check_step(layer, y, dx, dw, x, w, dy, M, what):
    ry, rdx, rdw, qw, sw = _oracle_step(x, w, dy, M)
    assert np.array_equal(layer.qw.cpu().numpy(), qw), f"{what}: weight codes"
    assert np.array_equal(layer.sw.cpu().numpy().view(np.uint32), sw.view(np.uint32)), f"{what}: weight scales"
    _check(from_dev_bf16(y), ry, f"{what} fwd")
    _check(from_dev_bf16(dx), rdx, f"{what} dgrad")
    _check(from_dev_bf16(dw), rdw, f"{what} wgrad")


def test_weight_reuse_steps_match_the_oracle():
    """Micro-batches that reuse W's codes, an optimizer-style in-place update of W (new
    version: re-quantised), and a change made behind torch's version counter followed by
    invalidate_weight_quant(): every step's y, dx and dW against the oracle's codes and
    scales of the weight as it is at that step."""
    lin, x, w, dy = _case(M=300, K=384, N=256)
    x2 = wl.random_bits((lin.M, lin.K), 77)
    dy2 = wl.random_bits((lin.M, lin.N), 78)
    xd, wd, dyd = to_dev_bf16(x), to_dev_bf16(w), to_dev_bf16(dy)
    layer = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N, reuse_weight_quant=True)
    # micro-batch 1 quantises W; micro-batch 2 (other x, dy) reuses its codes
    y = layer.forward(xd, wd).clone()
    dx, dw = (t.clone() for t in layer.backward(dyd))
    _check_step(layer, y, dx, dw, x, w, dy, lin.M, "micro-batch 1")
    y = layer.forward(to_dev_bf16(x2), wd).clone()
    dx, dw = (t.clone() for t in layer.backward(to_dev_bf16(dy2)))
    assert layer.weight_quant_calls == 1
    _check_step(layer, y, dx, dw, x2, w, dy2, lin.M, "micro-batch 2 (reused codes)")
    # an in-place update of W (what an optimizer step does): new codes and scales
    step = wl.random_bits((lin.N, lin.K), 79, std=0.01)
    wd.add_(to_dev_bf16(step))
    w_new = wd.cpu().view(torch.int16).numpy().view(np.uint16).copy()
    y = layer.forward(xd, wd).clone()
    dx, dw = (t.clone() for t in layer.backward(dyd))
    assert layer.weight_quant_calls == 2
    _check_step(layer, y, dx, dw, x, w_new, dy, lin.M, "after an in-place update")
    # a change the version counter does not see, then an explicit invalidation
    wd.data.mul_(0.75)
    w_3 = wd.cpu().view(torch.int16).numpy().view(np.uint16).copy()
    layer.invalidate_weight_quant()
    y = layer.forward(xd, wd).clone()
    dx, dw = (t.clone() for t in layer.backward(dyd))
    assert layer.weight_quant_calls == 3
    _check_step(layer, y, dx, dw, x, w_3, dy, lin.M, "after invalidation")


def test_main_gradient_mode_accumulates_micro_batches():
    lin, x, w, dy = _case(M=257, K=384, N=256)
    xd, wd, dyd = to_dev_bf16(x), to_dev_bf16(w), to_dev_bf16(dy)
    ref_layer = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N)
    ref_layer.forward(xd, wd)
    _, dw_bf16 = ref_layer.backward(dyd)
    layer = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N, reuse_weight_quant=True, main_grad=True)
    assert layer.dw is None
    layer.forward(xd, wd)
    _, mg = layer.backward(dyd)
    torch.cuda.synchronize()
    # one micro-batch from zero: the FP32 sums round to the BF16 wgrad's output
    assert torch.equal(mg.to(torch.bfloat16), dw_bf16)
    once = mg.clone()
    layer.forward(xd, wd)
    layer.backward(dyd)
    torch.cuda.synchronize()
    assert layer.weight_quant_calls == 1
    # second micro-batch: once + once, one FP32 rounding per element
    assert torch.allclose(layer.main_grad, 2.0 * once, rtol=2.0 ** -23, atol=0.0)
    layer.zero_main_grad()
    assert torch.count_nonzero(layer.main_grad) == 0


def test_training_step_replays_from_a_cuda_graph():
    """The six calls of a step can be captured in a CUDA graph (after one eager step sets the
    library's lazily initialised state) and replayed: the replay gives the eager step's bits,
    and a replay after new inputs are copied into the captured buffers gives their results."""
    lin, x, w, dy = _case(M=640, K=512, N=768)
    xd, wd, dyd = to_dev_bf16(x), to_dev_bf16(w), to_dev_bf16(dy)
    layer = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N)
    layer.forward(xd, wd)
    layer.backward(dyd)
    torch.cuda.synchronize()
    want = [t.clone() for t in (layer.y, layer.dx, layer.dw)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(xd, wd)
        layer.backward(dyd)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(xd, wd)
        layer.backward(dyd)
    for t in (layer.y, layer.dx, layer.dw):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for got, ref in zip((layer.y, layer.dx, layer.dw), want):
        assert torch.equal(got, ref)
    # new inputs in the captured buffers: the replay computes them (2x on x scales y and dW by 2)
    xd.mul_(2.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.y, 2.0 * want[0])
    assert torch.equal(layer.dw, 2.0 * want[2])
    assert torch.equal(layer.dx, want[1])
