"""Device status word: bounded waits give up cleanly and the context stays usable."""

import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import oracle
import synthetic
from gpu_util import exactly_symmetric, rel_frob, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


def test_watchdog_times_out_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    d3.selftest_watchdog(200_000, status)      # a barrier nothing completes; ~0.1 ms of spinning
    torch.cuda.synchronize()
    assert int(status.item()) & d3.DEV_TIMEOUT
    # the GPU context still works
    A = synthetic.gaussian((200, 96), seed=1, std=96 ** -0.5, dtype=torch.bfloat16, device=DEV)
    D = d3.sym_gemm(A)
    torch.cuda.synchronize()
    assert exactly_symmetric(D)
    assert rel_frob(to64(D), oracle.sym_gemm(to64(A))) <= 5e-3


def test_nonfinite_input_norm_sets_status():
    X = synthetic.gaussian((64, 128), seed=2, dtype=torch.bfloat16, device=DEV)
    X[3, 4] = float("inf")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    d3.gram_ns(X, [(3.4445, -4.7750, 2.0315)] * 5, (2,), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & d3.DEV_NONFINITE


def test_host_errors_raise_without_launching():
    X = torch.zeros((64, 32), dtype=torch.bfloat16, device=DEV)     # n > m
    with pytest.raises(d3.Dion3Error) as e:
        d3.gram_ns(X, [(1.5, -0.5, 0.0)] * 3, ())
    assert e.value.code == 1
    with pytest.raises(TypeError):
        d3.gram_ns(X.cpu(), [(1.5, -0.5, 0.0)] * 3, ())
