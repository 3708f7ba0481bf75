"""The kernels' bounded-wait error path on the GPU, made to run out on purpose.

Every pipeline wait in the quantisers and GEMMs gives up after a limit,
records BFP8_ETIMEOUT in the device status word and unwinds: it waits for its
own copies in flight, frees its tensor memory and returns. Here the limit is
set to 1 ms and a test switch makes the operand producers start no copies, so
the first wait of every CTA runs out; nothing faults or hangs, and the context
stays usable. Afterwards a normal call on the same device must match the
oracle again."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import from_dev_bf16, gemm_tolerance_ok, to_dev_bf16

import blockwise_fp8_linear_weight_b300 as bfp8

pytestmark = pytest.mark.gpu
ETIMEOUT = -5


@pytest.fixture
def stalled():
    assert bfp8.last_device_status() == 0
    bfp8.set_wait_limit_ns(1_000_000)
    prev = bfp8.test_stall_producers(True)
    try:
        yield
    finally:
        bfp8.test_stall_producers(prev)
        bfp8.set_wait_limit_ns(0)


def _case():
    lin = wl.Linear("timeout", 300, 256, 384, "normal", 41)
    return lin, *wl.make_linear(lin)


def test_every_kernel_reports_a_timeout(stalled):
    lin, x, w, dy = _case()
    xd, wd, dyd = to_dev_bf16(x), to_dev_bf16(w), to_dev_bf16(dy)
    calls = [
        ("quantize_act", lambda: bfp8.fp8_quantize_act(xd)),
        ("quantize_weight", lambda: bfp8.fp8_quantize_weight(wd)),
        ("quantize_transpose", lambda: bfp8.fp8_quantize_transpose(xd)),
        ("quantize_act_transpose", lambda: bfp8.fp8_quantize_act_transpose(dyd)),
    ]
    layer = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N)
    calls += [
        ("gemm_fwd", lambda: bfp8.fp8_block_gemm_fwd(layer.qx, layer.sx, layer.qw, layer.sw, layer.y)),
        ("gemm_dgrad", lambda: bfp8.fp8_block_gemm_dgrad(layer.qdy, layer.sdy, layer.qw, layer.sw, layer.dx)),
        ("gemm_wgrad", lambda: bfp8.fp8_block_gemm_wgrad(layer.qdyt, layer.sdyt, layer.qxt, layer.sxt, lin.M,
                                                         layer.dw)),
        ("gemm_wgrad_acc", lambda: bfp8.fp8_block_gemm_wgrad_acc(
            layer.qdyt, layer.sdyt, layer.qxt, layer.sxt, lin.M,
            torch.zeros((lin.N, lin.K), dtype=torch.float32, device="cuda"))),
        ("bf16_gemm", lambda: bfp8.bf16_gemm_axpby(xd, wd, None, 1.0, 0.0)),
    ]
    for name, call in calls:
        call()
        assert bfp8.last_device_status() == ETIMEOUT, name
        # reading the word clears it
        assert bfp8.last_device_status() == 0, name


def test_device_is_usable_after_timeouts(stalled):
    lin, x, w, dy = _case()
    xd, wd = to_dev_bf16(x), to_dev_bf16(w)
    layer = bfp8.BlockwiseFP8Linear(lin.M, lin.K, lin.N)
    layer.forward(xd, wd)
    assert bfp8.last_device_status() == ETIMEOUT
    # back to normal operation: the same layer computes the oracle's result
    bfp8.test_stall_producers(False)
    bfp8.set_wait_limit_ns(0)
    layer.forward(xd, wd)
    torch.cuda.synchronize()
    assert bfp8.last_device_status() == 0
    qx, sx = oracle.quantize_act(x)
    qw, sw = oracle.quantize_weight(w)
    assert np.array_equal(layer.qx.cpu().numpy(), qx)
    ok, ratio = gemm_tolerance_ok(from_dev_bf16(layer.y), oracle.gemm_fwd(qx, sx, qw, sw))
    assert ok, f"worst error/allowance = {ratio:.3g}"
