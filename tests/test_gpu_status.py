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


# A coefficient table that makes the iteration blow up without any restart: Z_t = a_t I with
# a_t = 1e4, so Q_t = 1e4^t I leaves the 16-bit range after two iterations (and R with it).  The
# inputs are finite and normal; only the iteration diverges -- the failure the pages describe
# under "half precision and numerical stability", forced here so that it happens for sure.
DIVERGING = [(1.0e4, 0.0, 0.0)] * 5


@pytest.mark.parametrize("n,m,compute", [(200, 640, torch.float16), (96, 2048, torch.float16),
                                         (96, 2048, torch.bfloat16), (130, 300, torch.float16)])
def test_diverging_iteration_sets_nonfinite(n, m, compute):
    """The last product's epilogue flags the non-finite output (separate products for n > 128,
    the fused segment kernel for n <= 128); the same finite input with the Jordan table does not."""
    X = synthetic.lowrank_plus_noise(n, m, seed=30 + n, dtype=torch.bfloat16, device=DEV)
    table = DIVERGING if compute == torch.float16 else [(1.0e9, 0.0, 0.0)] * 5   # bf16 reaches 3e38
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    O = d3.gram_ns(X, table, (), compute=compute, status=status)
    torch.cuda.synchronize()
    assert not bool(torch.isfinite(O.float()).all())
    assert int(status.item()) & d3.DEV_NONFINITE
    status.zero_()
    O = d3.gram_ns(X, [(3.4445, -4.7750, 2.0315)] * 5, (), compute=compute, status=status)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(O.float()).all()) and int(status.item()) == 0


def test_diverging_iteration_fp32_mode_sets_nonfinite():
    X = synthetic.gaussian((64, 256), seed=33, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    O = d3.gram_ns(X, [(1.0e20, 0.0, 0.0)] * 3, (), compute=torch.float32, status=status)
    torch.cuda.synchronize()
    assert not bool(torch.isfinite(O).all())
    assert int(status.item()) & d3.DEV_NONFINITE


def test_diverging_iteration_fp32_output_of_16_bit_iterates():
    """fp16 iterates, fp32 output: the fp32 store path of the last product flags it too."""
    X = synthetic.lowrank_plus_noise(160, 520, seed=34, dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    O = d3.gram_ns(X, DIVERGING, (), compute=torch.float16, out_dtype=torch.float32, status=status)
    torch.cuda.synchronize()
    assert not bool(torch.isfinite(O).all())
    assert int(status.item()) & d3.DEV_NONFINITE


@pytest.mark.parametrize("n,m,f", [(512, 1024, (1, 2)), (768, 2048, (1, 8))])
def test_diverging_step_flags_the_w_update(n, m, f):
    """In a Dion3 step the last product is fused into the W row update: a diverged iteration writes
    non-finite values into W[S,:] and raises the flag (k = 256 runs the separate products, k = 96
    the fused segments); rows outside S stay untouched."""
    W = synthetic.gaussian((2, n, m), seed=35, std=0.02, device=DEV)
    M = torch.zeros((2, n, m), device=DEV)
    G = synthetic.lowrank_batch(2, n, m, base_seed=36, device=DEV)
    W0 = W.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel = d3.step(W, M, G, f=f, abc=DIVERGING, restart_after=(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & d3.DEV_NONFINITE
    for b in range(2):
        rows = sel[b].long()
        assert not bool(torch.isfinite(W[b, rows]).all())
        keep = torch.ones(n, dtype=torch.bool, device=DEV)
        keep[rows] = False
        assert torch.equal(W[b, keep], W0[b, keep])


def test_diverging_standard_ns_sets_nonfinite():
    X = synthetic.lowrank_plus_noise(256, 256, seed=37, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    O = d3.ns_standard(X, [(1.0e4, 0.0, 0.0)] * 5, compute=torch.float16, status=status)
    torch.cuda.synchronize()
    assert not bool(torch.isfinite(O.float()).all())
    assert int(status.item()) & d3.DEV_NONFINITE
