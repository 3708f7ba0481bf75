"""Pins for the MuonH oracle (oracle/muonh.py), from facts outside its own loops:
  * closed form of the Newton-Schulz iteration: with X = U S V^T (SVD), one step
    maps X to U (a S + b S^3 + c S^5) V^T, so after n steps the singular values
    are the scalar polynomial iterated n times; checked against numpy's SVD;
  * the iteration commutes with transposition (it runs on the shorter side);
  * normalising makes the update independent of the gradient's scale;
  * the step before projection has norm exactly lr R, and the result has norm R;
  * lr = 0 is a pure projection of W onto the sphere of radius R."""
import numpy as np
import pytest

from oracle import muonh

a, b, c = muonh.MUON_NS_COEFFS


def _poly_n(s, n):
    for _ in range(n):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


@pytest.mark.parametrize("shape", [(64, 96), (96, 64), (50, 50), (1, 32)])
@pytest.mark.parametrize("steps", [1, 5])
def test_newton_schulz_is_the_singular_value_polynomial(shape, steps):
    G = np.random.default_rng(shape[0] + steps).standard_normal(shape)
    X0 = muonh.normalize(G)
    U, S, Vt = np.linalg.svd(X0, full_matrices=False)
    want = (U * _poly_n(S, steps)) @ Vt
    got = muonh.newton_schulz(X0, steps)
    assert np.allclose(got, want, rtol=0, atol=1e-10 * max(1.0, np.abs(want).max()))


def test_newton_schulz_commutes_with_transpose_and_brings_singular_values_near_one():
    G = np.random.default_rng(3).standard_normal((48, 80))
    X = muonh.normalize(G)
    assert np.allclose(muonh.newton_schulz(X.T), muonh.newton_schulz(X).T, atol=1e-12)
    s = np.linalg.svd(muonh.newton_schulz(X), compute_uv=False)
    # the quintic pulls every singular value of a normalised random matrix into a band around 1
    assert s.min() > 0.5 and s.max() < 1.3


def test_update_scale_invariance_step_size_and_radius():
    rng = np.random.default_rng(7)
    W = rng.standard_normal((40, 64)) * 0.02
    G = rng.standard_normal((40, 64))
    R, lr = float(np.linalg.norm(W)), 0.03
    W1 = muonh.update(W, G, lr, R, eps=0.0)
    W2 = muonh.update(W, 1e3 * G, lr, R, eps=0.0)
    assert np.allclose(W1, W2, rtol=0, atol=1e-12)
    assert abs(np.linalg.norm(W1) - R) <= 1e-12 * R
    U = muonh.newton_schulz(muonh.normalize(G))
    step = (lr * R / np.linalg.norm(U)) * U
    assert abs(np.linalg.norm(step) - lr * R) <= 1e-12 * R
    # the result is the projection of W - step
    Wp = W - step
    assert np.allclose(W1, R * Wp / np.linalg.norm(Wp), atol=1e-12)


def test_zero_learning_rate_is_a_projection():
    rng = np.random.default_rng(9)
    W = rng.standard_normal((16, 32))
    G = rng.standard_normal((16, 32))
    got = muonh.update(W, G, 0.0, 2.5)
    assert np.allclose(got, 2.5 * W / np.linalg.norm(W), atol=1e-13)


def test_normalize():
    G = np.random.default_rng(1).standard_normal((8, 12))
    assert abs(np.linalg.norm(muonh.normalize(G, eps=0.0)) - 1.0) < 1e-14


def test_zero_step_result_leaves_w_unchanged():
    """W = a U exactly (a = lr R / |U|): W - a U is zero, which has no direction to project;
    the update leaves W as it is. U = +-1 on 64 x 64 has |U| = 64, so with lr = 1/4 and R = 2,
    a = 2^-7 and every product is exact."""
    U = np.where(np.random.default_rng(4).standard_normal((64, 64)) < 0, -1.0, 1.0)
    W = 2.0 ** -7 * U
    assert np.linalg.norm(W - (0.25 * 2.0 / np.linalg.norm(U)) * U) == 0.0
    got = muonh.apply(W, U, 0.25, 2.0)
    assert np.array_equal(got, W)


def test_gemm_axpby_matches_brute_force():
    """The oracle's plain product alpha A B + beta C against a triple loop on small inputs."""
    rng = np.random.default_rng(11)
    A, B, C = rng.standard_normal((5, 7)), rng.standard_normal((7, 3)), rng.standard_normal((5, 3))
    want = np.zeros((5, 3))
    for i in range(5):
        for j in range(3):
            want[i, j] = -0.5 * sum(A[i, k] * B[k, j] for k in range(7)) + 2.0 * C[i, j]
    assert np.allclose(muonh.gemm_axpby(A, B, C, -0.5, 2.0), want, rtol=0, atol=1e-13)
    assert np.allclose(muonh.gemm_axpby(A, B, None, 1.0, 0.0), A @ B, rtol=0, atol=1e-13)


def test_newton_schulz_step_is_three_products():
    """One iteration written as the three gemm_axpby products the library runs
    (A = X X^T, B = b A + c A A, X' = a X + B X) equals the oracle's iteration."""
    X = muonh.normalize(np.random.default_rng(12).standard_normal((24, 40)))
    A = muonh.gemm_axpby(X, X.T, None, 1.0, 0.0)
    Bm = muonh.gemm_axpby(A, A, A, c, b)
    Xn = muonh.gemm_axpby(Bm, X, X, 1.0, a)
    assert np.allclose(Xn, muonh.newton_schulz(X, 1), rtol=0, atol=1e-13)
