"""Symmetric GEMM through the C ABI against the float64 oracle.

Tolerance: relative Frobenius error <= 5e-3 for 16-bit inputs with fp32 accumulation
(one bf16 rounding of the output is 2^-9 ~ 2e-3 relative); <= 1e-5 for the fp32 path.
Every stored result must be exactly symmetric, bit for bit.
"""

import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import oracle
import synthetic
from gpu_util import aligned_copy, exactly_symmetric, rel_frob, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = {torch.bfloat16: 5e-3, torch.float16: 5e-3, torch.float32: 1e-5}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


@pytest.mark.parametrize("n", [1, 17, 128, 130, 300, 513])
@pytest.mark.parametrize("k", [1, 64, 100, 1000])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_syrk_small(n, k, dtype):
    A = aligned_copy(synthetic.gaussian((n, k), seed=n * 7 + k, std=k ** -0.5, dtype=dtype, device=DEV))
    D = d3.sym_gemm(A)
    torch.cuda.synchronize()
    assert exactly_symmetric(D)
    ref = oracle.sym_gemm(to64(A))
    assert rel_frob(to64(D), ref) <= TOL[dtype]


@pytest.mark.parametrize("n,k", [(300, 200), (513, 64), (1024, 1024)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("alpha,beta,gamma", [(1.0, 1.0, 0.0), (2.0315, -4.775, 3.4445), (0.5, 0.0, 1.0)])
def test_epilogue_beta_gamma(n, k, dtype, alpha, beta, gamma):
    A = synthetic.gaussian((n, k), seed=11, std=k ** -0.5, dtype=dtype, device=DEV)
    C = aligned_copy(synthetic.symmetric_gaussian(n, seed=12, dtype=dtype, device=DEV))
    D = d3.sym_gemm(A, C=C, alpha=alpha, beta=beta, gamma=gamma)
    torch.cuda.synchronize()
    assert exactly_symmetric(D)
    ref = oracle.sym_gemm(to64(A), to64(C), alpha, beta, gamma)
    assert rel_frob(to64(D), ref) <= TOL[dtype]


def test_in_place_c_equals_d():
    n, k = 384, 256
    A = synthetic.gaussian((n, k), seed=13, std=k ** -0.5, dtype=torch.bfloat16, device=DEV)
    C = aligned_copy(synthetic.symmetric_gaussian(n, seed=14, dtype=torch.bfloat16, device=DEV))
    ref = oracle.sym_gemm(to64(A), to64(C), 1.0, 1.0, 0.5)
    d3.sym_gemm(A, C=C, beta=1.0, gamma=0.5, out=C)
    torch.cuda.synchronize()
    assert exactly_symmetric(C)
    assert rel_frob(to64(C), ref) <= 5e-3


def test_general_b_with_symmetric_product():
    """A B^T with B != A whose product is symmetric (two polynomials in the same R)."""
    n = 520
    X = synthetic.gaussian((n, 700), seed=15, std=700 ** -0.5, device=DEV)
    R = X @ X.T
    P = (0.3 * R + R @ R).to(torch.bfloat16)
    S = (1.5 * torch.eye(n, device=DEV) - 0.7 * R).to(torch.bfloat16)
    D = d3.sym_gemm(P, B=S)
    torch.cuda.synchronize()
    assert exactly_symmetric(D)
    ref = to64(P) @ to64(S).T
    ref_lower = np.tril(ref) + np.tril(ref, -1).T     # the kernel computes the lower triangle
    assert rel_frob(to64(D), ref_lower) <= 5e-3


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_batched_strided_and_fp32_out(dtype):
    batch, n, k = 5, 200, 136
    big = synthetic.gaussian((batch, n, k + 8), seed=16, std=k ** -0.5, dtype=dtype, device=DEV)
    A = big[:, :, :k]                                  # ld = k + 8, batch stride = n (k + 8)
    D = d3.sym_gemm(A, out_dtype=torch.float32)
    torch.cuda.synchronize()
    for b in range(batch):
        assert exactly_symmetric(D[b])
        assert rel_frob(to64(D[b]), oracle.sym_gemm(to64(A[b]))) <= (1e-5 if dtype == torch.float32 else 5e-3)


def test_k_zero():
    n = 130
    A = torch.empty((n, 0), dtype=torch.bfloat16, device=DEV)
    C = aligned_copy(synthetic.symmetric_gaussian(n, seed=17, dtype=torch.bfloat16, device=DEV))
    D = d3.sym_gemm(A, C=C, beta=2.0, gamma=1.0, out=aligned_copy(torch.empty_like(C)))
    torch.cuda.synchronize()
    assert exactly_symmetric(D)
    ref = 2.0 * to64(C) + np.eye(n)
    assert rel_frob(to64(D), ref) <= 5e-3


@pytest.mark.parametrize("n,kmul", [(1024, 1), (1024, 4), (2048, 1), (2048, 4), (4096, 1), (4096, 4),
                                    (8192, 1), (8192, 4)])
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_full_size_sampled(n, kmul, beta):
    """The symmetric-GEMM sweep at full size; entries checked on a sample the oracle computes one by one."""
    k = n * kmul
    A = synthetic.gaussian((n, k), seed=2000 + n + k, std=k ** -0.5, dtype=torch.bfloat16, device=DEV)
    C = synthetic.symmetric_gaussian(n, seed=2100 + n, dtype=torch.bfloat16, device=DEV) if beta else None
    D = d3.sym_gemm(A, C=C, beta=beta)
    torch.cuda.synchronize()
    # symmetry checked on whole row/column bands
    rng = np.random.default_rng(n + k)
    rows = torch.as_tensor(np.unique(np.concatenate([rng.integers(0, n, 48), [0, n - 1, n // 2]])), device=DEV)
    Dr = D[rows].cpu()
    Dc = D[:, rows].T.cpu()
    assert torch.equal(Dr.view(torch.int16), Dc.view(torch.int16))
    cols = torch.as_tensor(rng.integers(0, n, 64), device=DEV)
    Ar = to64(A[rows])
    Ac = to64(A[cols])
    ref = oracle.sym_gemm(Ar, B=Ac)          # the sampled entries D[rows, cols] = A[rows] A[cols]^T
    if beta:
        ref = ref + to64(C[rows][:, cols])
    got = to64(D[rows][:, cols])
    assert rel_frob(got, ref) <= 5e-3
