"""Closed-form twin of the Newton-Schulz oracle, through LAPACK's SVD.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Each Newton-Schulz step X <- a X + (b X X^T + c (X X^T)^2) X equals
X <- a X + b X X^T X + c X X^T X X^T X, an odd polynomial in X. Written with
the thin SVD X = U diag(s) V^T, it is U diag(f(s)) V^T with
f(s) = a s + b s^3 + c s^5, so the singular vectors never change and each
singular value follows the scalar recurrence alone. After the normalisation
X/(||X||_F + eps) and ``steps`` steps the exact result is
U diag(f^steps(s_i / (||X||_F + eps))) V^T. This is a different computation
from the step-by-step iteration (no matrix products, one SVD), so agreement
between the two pins the oracle.
"""
from __future__ import annotations

import numpy as np


def quintic(s, coeffs):
    """One step of the scalar map f(s) = a s + b s^3 + c s^5."""
    a, b, c = coeffs
    s = np.asarray(s, dtype=np.float64)
    s2 = s * s
    return s * (a + s2 * (b + c * s2))


def quintic_iterate(s, steps, coeffs):
    """f applied ``steps`` times; ``coeffs`` is one (a, b, c) triple or a
    (steps, 3) table whose row k is the triple of step k."""
    out = np.asarray(s, dtype=np.float64)
    table = np.asarray(coeffs, dtype=np.float64)
    for k in range(int(steps)):
        out = quintic(out, table[k] if table.ndim == 2 else table)
    return out


def closed_form(X: np.ndarray, steps: int, coeffs, eps: float) -> np.ndarray:
    """U diag(f^steps(s / (||X||_F + eps))) V^T for a 2-D fp64 array."""
    X = np.asarray(X, dtype=np.float64)
    if X.size == 0:
        return X.copy()
    fro = np.sqrt(np.sum(X * X))
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    g = quintic_iterate(s / (fro + eps), steps, coeffs)
    return (U * g) @ Vt


def polar(X: np.ndarray) -> np.ndarray:
    """Orthogonal polar factor U V^T (all singular values set to one)."""
    U, _, Vt = np.linalg.svd(np.asarray(X, dtype=np.float64), full_matrices=False)
    return U @ Vt


def singular_values(X: np.ndarray) -> np.ndarray:
    return np.linalg.svd(np.asarray(X, dtype=np.float64), compute_uv=False)


def closed_form_eigh(X: np.ndarray, steps: int, coeffs, eps: float) -> np.ndarray:
    """The same closed form through the eigen-decomposition of the smaller
    Gram matrix, for large inputs. With M >= N: X^T X = V diag(s^2) V^T and
    the result is X V diag(g(s)/s) V^T; with M < N: X X^T = U diag(s^2) U^T
    and the result is U diag(g(s)/s) U^T X, where g(s) = f^steps(s/(||X||+eps)).
    Directions with s == 0 contribute nothing (g(0) = 0)."""
    X = np.asarray(X, dtype=np.float64)
    if X.size == 0:
        return X.copy()
    fro = np.sqrt(np.sum(X * X))
    tall = X.shape[0] >= X.shape[1]
    G = X.T @ X if tall else X @ X.T
    lam, Q = np.linalg.eigh(G)
    s = np.sqrt(np.clip(lam, 0.0, None))
    g = quintic_iterate(s / (fro + eps), steps, coeffs)
    ratio = np.where(s > 0, g / np.where(s > 0, s, 1.0), 0.0)
    core = (Q * ratio) @ Q.T
    return X @ core if tall else core @ X
