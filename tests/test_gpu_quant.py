"""GPU parity of the three quantisers: E4M3 codes and FP32 scales must equal the
oracle's bit for bit, on edge cases (ragged rows, zero tiles, signed zeros,
subnormal scales, huge values) and on the full-size Puro-2B workload tensors."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import to_dev_bf16

import blockwise_fp8_linear_weight_b300 as bfp8

pytestmark = pytest.mark.gpu


def _gpu_act(bits):
    q, s = bfp8.fp8_quantize_act(to_dev_bf16(bits))
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _gpu_weight(bits):
    q, s = bfp8.fp8_quantize_weight(to_dev_bf16(bits))
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def _gpu_transpose(bits):
    qt, st = bfp8.fp8_quantize_transpose(to_dev_bf16(bits))
    torch.cuda.synchronize()
    return qt.cpu().numpy(), st.cpu().numpy()


def _same(a, b):
    assert a.shape == b.shape
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    bad = np.argwhere(a != b)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


def _special_input(R, C, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((R, C)).astype(np.float32)
    if R >= 6:
        x[0, :] = 0.0                                    # all-zero tiles
        x[1, :] = -0.0                                   # signed zeros
        x[2, :] *= 1e-39                                 # bf16 subnormals -> tiny scales
        x[3, :] *= 3e38 / np.abs(x[3]).max()             # near the top of the range
        x[4, ::7] = 0.0
        x[5, :] = np.where(rng.random(C) < 0.5, -1.0, 1.0) * np.ldexp(1.0, rng.integers(-20, 20, C))
    return wl.bf16_bits(x)


@pytest.mark.parametrize("R,C", [(1, 128), (6, 256), (37, 384), (128, 128), (300, 640), (1000, 2048)])
def test_act_edge_shapes(R, C):
    x = _special_input(R, C, R + C)
    q, s = _gpu_act(x)
    qo, so = oracle.quantize_act(x)
    _same(q, qo)
    _same(s, so)


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (384, 256)])
def test_weight_edge_shapes(N, K):
    w = _special_input(N, K, N * K)
    q, s = _gpu_weight(w)
    qo, so = oracle.quantize_weight(w)
    _same(q, qo)
    _same(s, so)


@pytest.mark.parametrize("R,C", [(1, 128), (6, 256), (127, 128), (128, 256), (129, 128), (300, 384), (1000, 2048)])
def test_transpose_edge_shapes(R, C):
    x = _special_input(R, C, 7 * R + C)
    qt, st = _gpu_transpose(x)
    qo, so = oracle.quantize_transpose(x)
    _same(qt, qo)
    _same(st, so)


def test_zero_rows_and_student_t():
    rng = np.random.default_rng(3)
    x = wl.bf16_bits(rng.standard_t(3, size=(257, 1024)).astype(np.float32))
    for f in (_gpu_act, _gpu_transpose):
        a = f(x)
        b = oracle.quantize_act(x) if f is _gpu_act else oracle.quantize_transpose(x)
        _same(a[0], b[0])
        _same(a[1], b[1])


def _workload_tensors():
    out = []
    for lin in wl.attention_projections().linears + wl.mlp_projections().linears:
        out.append(lin)
    # one layer of the full stack (every layer has the same shapes), outlier-channel inputs
    out.extend(wl.full_stack(layers=1).linears)
    return out


@pytest.mark.parametrize("lin", _workload_tensors(), ids=lambda l: f"{l.name}-M{l.M}-K{l.K}-N{l.N}")
def test_full_size_workload_tensors(lin):
    x, w, dy = wl.make_linear(lin)
    for bits in (x, dy):
        q, s = _gpu_act(bits)
        qo, so = oracle.quantize_act(bits)
        _same(q, qo)
        _same(s, so)
        qt, st = _gpu_transpose(bits)
        qo, so = oracle.quantize_transpose(bits)
        _same(qt, qo)
        _same(st, so)
    q, s = _gpu_weight(w)
    qo, so = oracle.quantize_weight(w)
    _same(q, qo)
    _same(s, so)
    # both layouts from one read (what a training step calls)
    for bits in (x, dy):
        q, s, qt, st = _gpu_dual(bits)
        qo, so = oracle.quantize_act(bits)
        qto, sto = oracle.quantize_transpose(bits)
        _same(q, qo)
        _same(s, so)
        _same(qt, qto)
        _same(st, sto)


def test_strided_inputs_and_outputs():
    """Leading dimensions larger than the row length on every argument."""
    x = wl.random_bits((100, 384), seed=9)
    xd = torch.zeros((100, 512), dtype=torch.bfloat16, device="cuda")
    xd[:, :384] = to_dev_bf16(x)
    q = torch.full((100, 400), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((3, 104), -1.0, dtype=torch.float32, device="cuda")
    bfp8.fp8_quantize_act(xd[:, :384], q[:, :384], s[:, :100])
    qo, so = oracle.quantize_act(x)
    _same(q[:, :384].cpu().numpy(), qo)
    _same(s[:, :100].cpu().numpy(), so)
    assert (q[:, 384:].cpu().numpy() == 0xAB).all() and (s[:, 100:].cpu().numpy() == -1.0).all()
    qt = torch.full((384, 160), 0xCD, dtype=torch.uint8, device="cuda")
    st = torch.full((1, 390), -1.0, dtype=torch.float32, device="cuda")
    bfp8.fp8_quantize_transpose(xd[:, :384], qt[:, :128], st[:, :384])
    qo, so = oracle.quantize_transpose(x)
    _same(qt[:, :128].cpu().numpy(), qo)
    _same(st[:, :384].cpu().numpy(), so)
    assert (qt[:, 128:].cpu().numpy() == 0xCD).all()


# ------------------------------------------------------------------ both layouts in one pass
def _gpu_dual(bits):
    q, s, qt, st = bfp8.fp8_quantize_act_transpose(to_dev_bf16(bits))
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy(), qt.cpu().numpy(), st.cpu().numpy()


@pytest.mark.parametrize("R,C", [(1, 128), (6, 256), (127, 128), (129, 384), (300, 640), (1000, 2048)])
def test_dual_layouts_edge_shapes(R, C):
    x = _special_input(R, C, 11 * R + C)
    q, s, qt, st = _gpu_dual(x)
    qo, so = oracle.quantize_act(x)
    qto, sto = oracle.quantize_transpose(x)
    _same(q, qo)
    _same(s, so)
    _same(qt, qto)
    _same(st, sto)


def test_dual_layouts_into_strided_outputs():
    """The two-layout call into views with padded row strides; a transposed stride that is an odd
    multiple of 16 bytes takes the 16-byte-store path, a multiple of 32 the 32-byte one. Padding is
    left untouched."""
    R, C = 300, 384
    x = _special_input(R, C, 23)
    for pad in (16, 32):
        q = torch.full((R, C + 64), 0xAB, dtype=torch.uint8, device="cuda")
        s = torch.full((C // 128, R + 4), -1.0, dtype=torch.float32, device="cuda")
        qt = torch.full((C, 384 + pad), 0xCD, dtype=torch.uint8, device="cuda")
        st = torch.full((3, C + 4), -1.0, dtype=torch.float32, device="cuda")
        bfp8.fp8_quantize_act_transpose(to_dev_bf16(x), q[:, :C], s[:, :R], qt[:, :384], st[:, :C])
        torch.cuda.synchronize()
        qo, so = oracle.quantize_act(x)
        qto, sto = oracle.quantize_transpose(x)
        _same(q[:, :C].cpu().numpy(), qo)
        _same(s[:, :R].cpu().numpy(), so)
        _same(qt[:, :384].cpu().numpy(), qto)
        _same(st[:, :C].cpu().numpy(), sto)
        assert (q[:, C:].cpu().numpy() == 0xAB).all() and (qt[:, 384:].cpu().numpy() == 0xCD).all()
        assert (s[:, R:].cpu().numpy() == -1.0).all() and (st[:, C:].cpu().numpy() == -1.0).all()


def test_dual_layouts_tiny_and_zero_columns():
    """Column tiles that are all tiny (scales below 2^-60, the pre-scaled quotient path) or all
    zero, next to row tiles of each kind, through the two-layout call."""
    rng = np.random.default_rng(17)
    x = rng.standard_normal((300, 384)).astype(np.float32)
    x[:, 5] *= 1e-39      # BF16 subnormals all down the column
    x[:, 130] *= 1e-30    # tiny normals
    x[:, 200] = 0.0
    x[:, 201] = -0.0
    x[7, :] *= 1e-39      # a tiny row as well
    bits = wl.bf16_bits(x)
    q, s, qt, st = _gpu_dual(bits)
    qo, so = oracle.quantize_act(bits)
    qto, sto = oracle.quantize_transpose(bits)
    _same(q, qo)
    _same(s, so)
    _same(qt, qto)
    _same(st, sto)


def _sweep_rows(seed):
    """Rows of 1x128 tiles whose first element is the tile maximum and whose other 127 elements walk
    through every positive BF16 value below it (random signs). The maxima include 448 * 2^k, where
    the scale is a power of two and every quotient is exact (ties on the E4M3 grid are hit exactly),
    and random BF16 values, where quotients land anywhere between grid points."""
    rng = np.random.default_rng(seed)
    all_pos = np.arange(1, 0x7F80, dtype=np.uint16)            # every positive finite BF16 pattern
    maxima = [wl.bf16_bits(np.float32(448.0 * 2.0 ** k)).item() for k in (-20, -3, 0, 5)]
    maxima += list(rng.integers(0x3000, 0x4A00, size=12).astype(np.uint16))
    rows = []
    for m in maxima:
        vals = all_pos[all_pos < m]
        vals = np.concatenate([vals, vals[:(-len(vals)) % 127]])  # pad to whole rows
        body = vals.reshape(-1, 127)
        signs = (rng.random(body.shape) < 0.5).astype(np.uint16) << 15
        body = body | signs
        head = np.full((body.shape[0], 1), m, dtype=np.uint16)
        rows.append(np.concatenate([head, body], axis=1))
    return np.concatenate(rows, axis=0)


def test_codes_bit_exact_over_every_bf16_value():
    """The kernels compute fl32(x * fl32(1/s)) and fall back to the IEEE quotient near E4M3 rounding
    boundaries; every BF16 value below each tile maximum must still give the definition's code."""
    x = _sweep_rows(5)
    q, s = _gpu_act(x)
    qo, so = oracle.quantize_act(x)
    _same(q, qo)
    _same(s, so)
    # the same values down the columns (transposed tiles, and both layouts at once)
    R = x.shape[0] // 128 * 128
    xt = np.ascontiguousarray(x[:R].T)  # column i of xt is row i of x
    qt, st = _gpu_transpose(xt)
    qto, sto = oracle.quantize_transpose(xt)
    _same(qt, qto)
    _same(st, sto)
    q, s, qt, st = _gpu_dual(xt)
    _same(qt, qto)
    _same(st, sto)
    qo, so = oracle.quantize_act(xt)
    _same(q, qo)
    _same(s, so)
