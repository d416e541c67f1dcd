"""Symmetric GEMM by its definition (oracle; test infrastructure only).

Source: Dion3 paper summary, prerequisite "symmetric GEMM kernels" and the
page's "technical novelty" (the Gram form needs fused symmetric products of
the form alpha A B + beta C): the result D = alpha A B^T + beta C + gamma I is
symmetric, so a kernel may compute its lower triangle and mirror it.  The
oracle computes the whole product in float64; the triangle-and-mirror is the
GPU's business, checked there by exact bitwise symmetry.
"""

from __future__ import annotations

import numpy as np


def sym_gemm(A, C=None, alpha: float = 1.0, beta: float = 0.0, gamma: float = 0.0, B=None) -> np.ndarray:
    """D = alpha * A @ B^T + beta * C + gamma * I  (B defaults to A)."""
    A = np.asarray(A, dtype=np.float64)
    Bm = A if B is None else np.asarray(B, dtype=np.float64)
    D = alpha * (A @ Bm.T)
    if beta != 0.0:
        D = D + beta * np.asarray(C, dtype=np.float64)
    if gamma != 0.0:
        D = D + gamma * np.eye(D.shape[0])
    return D
