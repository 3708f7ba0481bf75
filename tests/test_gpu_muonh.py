"""GPU parity of the MuonH update against the FP64 oracle (oracle/muonh.py), stage by stage.

Bars:
  * muonh_normalize: every BF16 output within one BF16 unit in the last place of
    the exact quotient, 2^-7 |x_ref| (the FP32 product is rounded once more to BF16);
  * bf16_gemm_axpby (one Newton-Schulz product) against alpha A B + beta C in FP64 from
    the same BF16 inputs, per element:
        |d - d_ref| <= 2^-8 |d_ref| + (K 2^-24 + 2^-22) (|alpha| (|A| |B|) + |beta| |C|)
    (one rounding to BF16, at most half a BF16 unit, 2^-8 relative; an FP32 sum of K exact
    products, at most K 2^-24 of the sum of magnitudes; the FP32 epilogue's own roundings);
  * muonh_newton_schulz (five iterations, every product rounded to BF16) against the FP64
    iteration from the same BF16 input: |U - U_ref|_F <= 3 % of |U_ref|_F (each step rounds
    A, b A + c A A and X to BF16, 2^-9 relative per element; measured about 1 %);
  * muonh_apply (given U): FP32 element-wise arithmetic on FP64 sums,
    |w - w_ref| <= 4e-6 |w_ref| + 4e-6 rms(w_ref), and |w|_F = R within 1e-5;
  * full update: the step is lr R U / |U|, so the Newton-Schulz bar carries over as
    |W - W_ref|_F <= 0.03 lr R.
"""
import numpy as np
import pytest
import torch

from oracle import muonh as ref

import blockwise_fp8_linear_weight_b300 as bfp8

pytestmark = pytest.mark.gpu


def _rand(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


@pytest.mark.parametrize("shape", [(4, 4), (256, 512), (300, 1028), (2048, 6144)])
def test_normalize_parity(shape):
    G = _rand(shape, 1)
    x = bfp8.muonh_normalize(torch.from_numpy(G).cuda())
    torch.cuda.synchronize()
    got = x.float().cpu().numpy().astype(np.float64)
    want = ref.normalize(G)
    assert np.all(np.abs(got - want) <= 2.0 ** -7 * np.abs(want) + 1e-30)


@pytest.mark.parametrize("shape", [(8, 16), (512, 256), (2048, 6144)])
def test_apply_parity_and_radius(shape):
    W = _rand(shape, 2, 0.02)
    U = torch.from_numpy(_rand(shape, 3)).to(torch.bfloat16)
    R, lr = 1.7, 0.05
    w = torch.from_numpy(W.copy()).cuda()
    bfp8.muonh_apply(w, U.cuda(), lr, R)
    torch.cuda.synchronize()
    got = w.cpu().numpy().astype(np.float64)
    want = ref.apply(W, U.float().numpy(), lr, R)
    rms = np.sqrt(np.mean(want ** 2))
    assert np.all(np.abs(got - want) <= 4e-6 * np.abs(want) + 4e-6 * rms)
    assert abs(np.linalg.norm(got) - R) <= 1e-5 * R


@pytest.mark.parametrize("shape", [(256, 512), (512, 256), (2048, 6144)])
def test_full_update_against_fp64_oracle(shape):
    W = _rand(shape, 4, 0.02)
    G = _rand(shape, 5)
    R, lr = float(np.linalg.norm(W.astype(np.float64))), 0.02
    w = torch.from_numpy(W.copy()).cuda()
    bfp8.muonh_update(w, torch.from_numpy(G).cuda(), lr, R)
    torch.cuda.synchronize()
    got = w.cpu().numpy().astype(np.float64)
    want = ref.update(W, G, lr, R)
    assert np.linalg.norm(got - want) <= 0.03 * lr * R
    assert abs(np.linalg.norm(got) - R) <= 1e-5 * R


def _bf16(shape, seed, scale=1.0):
    return torch.from_numpy(_rand(shape, seed, scale)).to(torch.bfloat16)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _dev_padded(t):
    """t on the GPU as a view whose row stride is rounded up to 8 elements (the 16-byte rule)."""
    rows, cols = t.shape
    buf = torch.zeros((rows, (cols + 7) // 8 * 8), dtype=t.dtype, device="cuda")
    buf[:, :cols] = t.cuda()
    return buf[:, :cols]


@pytest.mark.parametrize("M,N,K,mn", [(1, 8, 1, False), (200, 264, 100, False), (200, 264, 100, True),
                                      (256, 512, 256, True), (130, 2048, 2048, False),
                                      (2048, 2048, 6144, False), (2048, 6144, 2048, True)])
def test_bf16_gemm_axpby_parity(M, N, K, mn):
    a = _bf16((M, K), M + 1)
    b = _bf16((K, N) if mn else (N, K), N + 2, 0.1)
    c = _bf16((M, N), K + 3)
    alpha, beta = -1.25, 0.75
    d = bfp8.bf16_gemm_axpby(_dev_padded(a), _dev_padded(b), c.cuda(), alpha, beta, b_mn_major=mn)
    torch.cuda.synchronize()
    A, C = _f64(a), _f64(c)
    B = _f64(b) if mn else _f64(b).T
    want = ref.gemm_axpby(A, B, C, alpha, beta)
    allow = 2.0 ** -8 * np.abs(want) + (K * 2.0 ** -24 + 2.0 ** -22) * (
        abs(alpha) * (np.abs(A) @ np.abs(B)) + abs(beta) * np.abs(C))
    err = np.abs(_f64(d) - want)
    assert np.all(err <= allow), f"worst error/allowance {np.max(err / allow):.3g}"


def test_bf16_gemm_without_c_and_into_a_strided_view():
    """beta = 0 reads no C; the output may be a view with a padded row stride, whose padding
    is left untouched."""
    M, N, K = 300, 256, 384
    a, b = _bf16((M, K), 5), _bf16((N, K), 6)
    buf = torch.full((M, N + 16), 7.0, dtype=torch.bfloat16, device="cuda")
    d = buf[:, :N]
    bfp8.bf16_gemm_axpby(a.cuda(), b.cuda(), None, 0.5, 0.0, d=d)
    torch.cuda.synchronize()
    A, B = _f64(a), _f64(b).T
    want = 0.5 * (A @ B)
    allow = 2.0 ** -8 * np.abs(want) + (K * 2.0 ** -24 + 2.0 ** -22) * 0.5 * (np.abs(A) @ np.abs(B))
    assert np.all(np.abs(_f64(d) - want) <= allow)
    assert torch.all(buf[:, N:] == 7.0)


@pytest.mark.parametrize("shape", [(256, 512), (512, 256), (2048, 6144), (6144, 2048)])
def test_newton_schulz_parity(shape):
    """The library's five BF16 iterations against the FP64 oracle's from the same BF16 input,
    in both orientations (the iteration runs on x^T when rows > cols)."""
    x = bfp8.muonh_normalize(torch.from_numpy(_rand(shape, 8)).cuda())
    torch.cuda.synchronize()
    X0 = _f64(x)
    bfp8.muonh_newton_schulz(x)
    torch.cuda.synchronize()
    U, U_ref = _f64(x), ref.newton_schulz(X0)
    assert np.linalg.norm(U - U_ref) <= 0.03 * np.linalg.norm(U_ref)


def test_newton_schulz_zero_steps_is_identity():
    x = _bf16((64, 128), 9).cuda()
    y = x.clone()
    bfp8.muonh_newton_schulz(y, steps=0)
    torch.cuda.synchronize()
    assert torch.equal(x, y)


def test_update_is_deterministic():
    W = torch.from_numpy(_rand((1024, 2048), 6, 0.02)).cuda()
    G = torch.from_numpy(_rand((1024, 2048), 7)).cuda()
    w1, w2 = W.clone(), W.clone()
    bfp8.muonh_update(w1, G, 0.02, 1.0)
    bfp8.muonh_update(w2, G, 0.02, 1.0)
    torch.cuda.synchronize()
    assert torch.equal(w1, w2)


def test_short_partials_buffer_is_refused():
    g = torch.zeros((8, 16), dtype=torch.float32, device="cuda")
    short = torch.zeros(3, dtype=torch.float64, device="cuda")
    with pytest.raises(bfp8.Bfp8Error) as e:
        bfp8.muonh_normalize(g, partials=short)
    assert e.value.code == -1


@pytest.mark.parametrize("shape", [(8, 16), (2048, 6144)])
def test_apply_static_scratch_matches_caller_scratch(shape):
    W = _rand(shape, 12, 0.02)
    U = torch.from_numpy(_rand(shape, 13)).to(torch.bfloat16).cuda()
    R, lr = 2.0, 0.03
    w1 = torch.from_numpy(W.copy()).cuda()
    w2 = w1.clone()
    bfp8.muonh_apply(w1, U, lr, R)
    bfp8.muonh_apply_static(w2, U, lr, R)
    torch.cuda.synchronize()
    assert torch.equal(w1, w2)
    want = ref.apply(W, U.float().cpu().numpy(), lr, R)
    got = w2.cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(want ** 2))
    assert np.all(np.abs(got - want) <= 4e-6 * np.abs(want) + 4e-6 * rms)


def _degenerate(delta):
    """U = +-1 on 64 x 64 (|U| = 64), lr = 1/4, R = 2, so a = lr R / |U| = 2^-7 exactly, and
    W = a U + delta a V with V ~ N(0, 1): W - a U is delta a V (exactly zero for delta = 0)."""
    rng = np.random.default_rng(21)
    U = np.where(rng.standard_normal((64, 64)) < 0, -1.0, 1.0).astype(np.float32)
    V = rng.standard_normal((64, 64)).astype(np.float32)
    W = (np.float32(2.0 ** -7) * U + np.float32(delta * 2.0 ** -7) * V).astype(np.float32)
    return W, U, V


@pytest.mark.parametrize("static", [False, True], ids=["caller-scratch", "static-scratch"])
def test_apply_leaves_w_unchanged_when_the_step_cancels_it(static):
    W, U, _ = _degenerate(0.0)
    w = torch.from_numpy(W.copy()).cuda()
    u = torch.from_numpy(U).to(torch.bfloat16).cuda()
    (bfp8.muonh_apply_static if static else bfp8.muonh_apply)(w, u, 0.25, 2.0)
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy(), W)
    assert np.array_equal(ref.apply(W, U, 0.25, 2.0), W)


def test_apply_projects_onto_the_sphere_under_near_cancellation():
    """W - a U is 1e-3 of W: the norm of W' comes from W' itself, so the result lies on the
    sphere |w| = R and points along V (FP32 forms W' with an error of about 2^-24 |a U|,
    i.e. 6e-5 of |W'| here)."""
    W, U, V = _degenerate(1e-3)
    w = torch.from_numpy(W.copy()).cuda()
    bfp8.muonh_apply(w, torch.from_numpy(U).to(torch.bfloat16).cuda(), 0.25, 2.0)
    torch.cuda.synchronize()
    got = w.cpu().numpy().astype(np.float64)
    assert abs(np.linalg.norm(got) - 2.0) <= 1e-5 * 2.0
    want = 2.0 * V / np.linalg.norm(V.astype(np.float64))
    assert np.linalg.norm(got - want) <= 1e-3 * 2.0
