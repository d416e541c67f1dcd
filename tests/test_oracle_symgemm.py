"""sym_gemm against brute-force sums on tiny inputs."""

import numpy as np
import pytest

import oracle


def _brute(A, B, C, alpha, beta, gamma):
    n, k = len(A), len(A[0])
    D = [[0.0] * n for _ in range(n)]
    for i in range(n):
        for j in range(n):
            acc = 0.0
            for p in range(k):
                acc += A[i][p] * B[j][p]
            D[i][j] = alpha * acc + (beta * C[i][j] if beta else 0.0) + (gamma if i == j else 0.0)
    return np.array(D)


@pytest.mark.parametrize("alpha,beta,gamma", [(1.0, 0.0, 0.0), (0.5, 1.0, 0.0), (2.0, -0.3, 1.7)])
@pytest.mark.parametrize("with_b", [False, True])
def test_sym_gemm_brute_force(alpha, beta, gamma, with_b):
    rng = np.random.default_rng(0)
    n, k = 5, 3
    A = rng.standard_normal((n, k))
    B = rng.standard_normal((n, k)) if with_b else None
    C = rng.standard_normal((n, n))
    got = oracle.sym_gemm(A, C, alpha, beta, gamma, B=B)
    exp = _brute(A.tolist(), (A if B is None else B).tolist(), C.tolist(), alpha, beta, gamma)
    np.testing.assert_allclose(got, exp, rtol=1e-14, atol=1e-14)


def test_syrk_is_symmetric():
    A = np.random.default_rng(1).standard_normal((7, 11))
    D = oracle.sym_gemm(A, alpha=0.7, gamma=2.0)
    assert np.array_equal(D, D.T)
