"""MuonH update, plain FP64 numpy. TEST INFRASTRUCTURE (tests, smoke, bench CPU legs only).

The Puro-2B recipe trains with MuonH (Puro-2B article on en.roboind.com, section
"From ordinary learning to effective learning"): on top of Muon the size of each
weight update is standardised, and after the update the weight is projected back
to a fixed radius, the relative update size being a preset quantity. Read plainly
(Frobenius norms):
  X0    = G / (|G| + eps)
  U     = Newton-Schulz iterations on X0:  X <- a X + (b A + c A^2) X,  A = X X^T,
          run on the orientation with fewer rows
  W'    = W - lr R U / |U|
  W_new = R W' / |W'|
The pages give neither the iteration coefficients nor the radius. The quintic
coefficients are those of the public Muon optimizer (K. Jordan et al., 2024).
Parity with the Puro-2B implementation is unpinned for that reason; the pins in
tests/test_oracle_muonh.py fix this reading (closed form of the iteration through
the SVD, invariants of the projection).
"""
from __future__ import annotations

import numpy as np

MUON_NS_COEFFS = (3.4445, -4.7750, 2.0315)


def normalize(G, eps: float = 1e-7):
    G = np.asarray(G, dtype=np.float64)
    return G / (np.linalg.norm(G) + eps)


def newton_schulz(X0, steps: int = 5, coeffs=MUON_NS_COEFFS):
    a, b, c = coeffs
    X = np.asarray(X0, dtype=np.float64)
    t = X.shape[0] > X.shape[1]
    if t:
        X = X.T
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if t else X


def gemm_axpby(A, B, C, alpha: float, beta: float):
    """alpha * A @ B + beta * C in FP64: one product of the Newton-Schulz iteration (A X^T,
    b A + c A A, a X + B X are all of this form)."""
    out = alpha * (np.asarray(A, dtype=np.float64) @ np.asarray(B, dtype=np.float64))
    if C is not None:
        out = out + beta * np.asarray(C, dtype=np.float64)
    return out


def apply(W, U, lr: float, radius: float):
    W = np.asarray(W, dtype=np.float64)
    U = np.asarray(U, dtype=np.float64)
    nu = np.linalg.norm(U)
    Wp = W - (lr * radius / nu) * U if nu > 0 else W.copy()
    n = np.linalg.norm(Wp)
    return radius * Wp / n if n > 0 else W.copy()


def update(W, G, lr: float, radius: float, steps: int = 5, coeffs=MUON_NS_COEFFS, eps: float = 1e-7):
    return apply(W, newton_schulz(normalize(G, eps), steps, coeffs), lr, radius)
