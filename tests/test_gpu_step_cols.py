"""Dion3 step with column selection (matrices stored m x n, short side n as columns) through the
C ABI against the oracle's dion3_step_cols.

Bars as for rows: selected columns bit-exact, M bit-exact, Delta W within 3e-2 relative Frobenius
(1e-4 in fp32 compute mode)."""

import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import oracle
import synthetic
from gpu_util import bits32, rel_frob

pytestmark = pytest.mark.gpu
DEV = "cuda"
ABC = [(3.4445, -4.7750, 2.0315)] * 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


def _check(W, M, G, f, mu=0.95, eta=0.01, wd=0.0, norm_p=1, restarts=(2, 4), compute=torch.float16, cols=None,
           tol=3e-2, check_w=True):
    batch = M.shape[0]
    W0, M0, Gc = W.cpu().numpy().copy(), M.cpu().numpy().copy(), G.float().cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel = d3.step_cols(W, M, G, f=f, mu=mu, eta=eta, wd=wd, norm_p=norm_p, abc=ABC, restart_after=restarts,
                       compute=compute, status=status,
                       cols=None if cols is None else torch.from_numpy(cols).to(DEV))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(batch):
        W1, M1, S, _ = oracle.dion3_step_cols(W0[i], M0[i], Gc[i], *f, mu=mu, eta=eta, wd=wd, norm_p=norm_p, abc=ABC,
                                              restart_after=restarts, cols=None if cols is None else cols[i])
        assert np.array_equal(sel[i].cpu().numpy().astype(np.int64), S), f"matrix {i}: selection differs"
        assert np.array_equal(bits32(M[i]), bits32(M1)), f"matrix {i}: momentum differs"
        if check_w:
            assert rel_frob(W[i].double().cpu().numpy() - W0[i], W1 - W0[i]) <= tol, f"matrix {i}: update off"
    return sel


@pytest.mark.parametrize("m,n,f", [(256, 64, (1, 4)), (1000, 130, (1, 8)), (300, 300, (3, 5)), (1004, 96, (1, 1))])
@pytest.mark.parametrize("norm_p", [1, 2])
def test_two_steps(m, n, f, norm_p):
    batch = 3
    W = synthetic.gaussian((batch, m, n), seed=51, std=0.02, device=DEV)
    M = torch.zeros((batch, m, n), dtype=torch.float32, device=DEV)
    for step in range(2):
        G = synthetic.lowrank_batch(batch, m, n, base_seed=600 + 10 ** 6 * step + m, dtype=torch.bfloat16, device=DEV)
        _check(W, M, G, f, norm_p=norm_p)



@pytest.mark.parametrize("m,n,f", [(1, 1, (1, 1)), (3, 2, (1, 2)), (17, 3, (1, 8)), (40, 17, (1, 4))])
@pytest.mark.parametrize("norm_p", [1, 2])
def test_tiny_shapes(m, n, f, norm_p):
    """Degenerate sizes for column selection: one column, k = 1, rows of 1 to 3 elements."""
    batch = 3
    W = synthetic.gaussian((batch, m, n), seed=52, std=0.02, device=DEV)
    M = torch.zeros((batch, m, n), dtype=torch.float32, device=DEV)
    for step in range(2):
        G = synthetic.lowrank_batch(batch, m, n, base_seed=900 + 100 * step + 10 * m + n, dtype=torch.bfloat16,
                                    device=DEV)
        _check(W, M, G, f, norm_p=norm_p)


def test_moe_w2_shape():
    """The MoE w2 matrices as stored (2048 x 768): columns are the short side; f = 1/8, k = 96."""
    batch = 2
    W = synthetic.gaussian((batch, 2048, 768), seed=52, std=0.02, device=DEV)
    M = synthetic.gaussian((batch, 2048, 768), seed=53, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(batch, 2048, 768, base_seed=700, dtype=torch.bfloat16, device=DEV)
    _check(W, M, G, (1, 8))


def test_given_columns_weight_decay_and_fp32():
    m, n, f = 512, 80, (1, 4)
    k = d3.k_of(n, *f)
    rng = np.random.default_rng(3)
    cols = np.stack([np.sort(rng.choice(n, size=k, replace=False)) for _ in range(2)]).astype(np.int32)
    W = synthetic.gaussian((2, m, n), seed=54, std=0.02, device=DEV)
    M = synthetic.gaussian((2, m, n), seed=55, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(2, m, n, base_seed=710, dtype=torch.bfloat16, device=DEV)
    _check(W, M, G, f, wd=0.1, cols=cols)
    _check(W, M, G, f, compute=torch.float32, tol=1e-4)


def test_column_ties_and_near_ties():
    """Repeated columns tie exactly (lower index wins); columns one fp32 ulp apart force the exact
    integer re-ranking, which here walks a column with stride n."""
    m, n = 512, 64
    M = synthetic.gaussian((1, m, n), seed=56, std=0.05, device=DEV)
    src = torch.arange(0, n, 2, device=DEV)
    M[0][:, src + 1] = M[0][:, src]
    Mi = M.view(torch.int32)
    Mi[0, 7, src + 1] += torch.where(src % 4 == 0, 1, -1).to(torch.int32)
    G = torch.zeros((1, m, n), dtype=torch.bfloat16, device=DEV)
    W = torch.zeros((1, m, n), device=DEV)
    for norm_p in (1, 2):
        for f in ((1, 2), (1, 4), (3, 8)):
            _check(W.clone(), M.clone(), G, f, norm_p=norm_p, check_w=False)
    base = synthetic.gaussian((m, 5), seed=57, std=0.05, dtype=torch.bfloat16, device=DEV)
    G2 = base[:, torch.arange(40, device=DEV) % 5].unsqueeze(0).contiguous()   # columns repeat with period 5
    for norm_p in (1, 2):
        _check(torch.zeros((1, m, 40), device=DEV), torch.zeros((1, m, 40), device=DEV), G2, (1, 4), norm_p=norm_p,
               check_w=False)


@pytest.mark.parametrize("norm_p", [1, 2])
def test_tied_columns(norm_p):
    """Every column of M + G the same permutation of one column (equal exact keys, fp32 sums that
    differ with the order): more ambiguous columns than the selection block has threads, so the
    radix-select ranking reads the strided column vectors; ties take the lower column index."""
    m, n = 2048, 512
    rng = np.random.default_rng(91)
    perm = torch.from_numpy(np.stack([rng.permutation(m) for _ in range(n)])).to(DEV)
    vm = synthetic.gaussian((m,), seed=92, std=0.05, device=DEV)
    vg = synthetic.gaussian((m,), seed=93, std=0.01, dtype=torch.bfloat16, device=DEV)
    M = vm[perm].T.contiguous().unsqueeze(0)
    G = vg[perm].T.contiguous().unsqueeze(0)
    W = synthetic.gaussian((1, m, n), seed=94, std=0.02, device=DEV)
    sel = _check(W, M, G, (1, 4), norm_p=norm_p)
    assert np.array_equal(sel[0].cpu().numpy(), np.arange(d3.k_of(n, 1, 4)))
