"""Standard Newton-Schulz (the square-matrix fallback) through the C ABI against the float64
oracle's plain definition of the iteration.

Tolerances (relative Frobenius): <= 3e-2 with 16-bit iterates, <= 1e-4 in fp32 compute mode.
"""

import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import oracle
import synthetic
from gpu_util import rel_frob, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
JORDAN = (3.4445, -4.7750, 2.0315)
ABC = [JORDAN] * 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


def _oracle(X):
    return np.stack([oracle.ns_standard(x, ABC) for x in to64(X)]) if X.dim() == 3 else oracle.ns_standard(to64(X), ABC)


SHAPES = [(1, 8), (17, 40), (64, 64), (130, 130), (130, 300), (256, 256), (200, 1000)]


@pytest.mark.parametrize("n,m", SHAPES)
@pytest.mark.parametrize("compute", [torch.float16, torch.bfloat16])
def test_16bit_iterates(n, m, compute):
    X = synthetic.lowrank_plus_noise(n, m, seed=3 * n + m, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    O = d3.ns_standard(X, ABC, compute=compute, status=status)
    torch.cuda.synchronize()
    assert O.dtype == torch.bfloat16
    assert rel_frob(to64(O), _oracle(X)) <= 3e-2
    assert int(status.item()) == 0



@pytest.mark.parametrize("n,m", [(1, 1), (2, 3), (3, 3), (3, 5), (5, 7)])
@pytest.mark.parametrize("compute,tol", [(torch.float16, 3e-2), (torch.float32, 1e-4)])
def test_rows_narrower_than_16_bytes(n, m, compute, tol):
    """m < 8: unaligned input rows and ragged tiles everywhere; a batch of three."""
    X = torch.stack([synthetic.lowrank_plus_noise(n, m, seed=60 + i, dtype=torch.bfloat16, device=DEV)
                     for i in range(3)])
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    O = d3.ns_standard(X, ABC, compute=compute, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rel_frob(to64(O), _oracle(X)) <= tol


@pytest.mark.parametrize("n,m", [(64, 64), (256, 256), (100, 333), (256, 1024)])
def test_fp32_mode(n, m):
    X = synthetic.gaussian((n, m), seed=n * m, device=DEV)
    O = d3.ns_standard(X, ABC, compute=torch.float32)
    torch.cuda.synchronize()
    assert O.dtype == torch.float32
    assert rel_frob(to64(O), _oracle(X)) <= 1e-4


def test_batched_square_and_fp32_output():
    """A batch of square matrices (alpha = 1), 16-bit iterates, fp32 output through the final cast."""
    X = synthetic.lowrank_batch(3, 192, 192, base_seed=40, dtype=torch.bfloat16, device=DEV)
    O = d3.ns_standard(X, ABC, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert O.dtype == torch.float32
    ref = _oracle(X)
    for i in range(3):
        assert rel_frob(to64(O[i]), ref[i]) <= 3e-2


def test_agrees_with_gram_ns_on_square_input():
    """Theorem 2: on a square input both iterations compute the same polynomial of X."""
    X = synthetic.lowrank_plus_noise(256, 256, seed=77, dtype=torch.bfloat16, device=DEV)
    a = to64(d3.ns_standard(X, ABC, compute=torch.float32, out_dtype=torch.float32))
    b = to64(d3.gram_ns(X.float(), ABC, (2, 4), compute=torch.float32))
    torch.cuda.synchronize()
    assert rel_frob(a, b) <= 1e-4


def test_strided_batch_input_not_modified():
    base = synthetic.lowrank_batch(2, 96, 264, base_seed=90, dtype=torch.bfloat16, device=DEV)
    X = torch.zeros((2, 96, 272), dtype=torch.bfloat16, device=DEV)
    X[:, :, :264] = base
    Xv = X[:, :, :264]
    before = X.clone()
    O = d3.ns_standard(Xv, ABC)
    torch.cuda.synchronize()
    assert torch.equal(X, before)
    ref = _oracle(base)
    for i in range(2):
        assert rel_frob(to64(O[i]), ref[i]) <= 3e-2


def test_T1_single_iteration():
    X = synthetic.gaussian((48, 96), seed=5, device=DEV)
    O = d3.ns_standard(X, [JORDAN], compute=torch.float32)
    torch.cuda.synchronize()
    ref = oracle.ns_standard(to64(X), [JORDAN])
    assert rel_frob(to64(O), ref) <= 1e-5
