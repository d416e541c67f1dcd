"""The carried error-feedback decay (dion3_step_carry, dion3_decay_rows) through the C ABI.

Moving the decay M[S,:] <- mu M[S,:] of one step into the next step's momentum pass rounds
exactly as the plain step does (mu M rounded to fp32, then + G rounded), so the bar is
bit-identity with the plain steps: the selected rows, W and (once the pending decay is applied)
M, at every step.  One chain is also compared with the float64 oracle's plain steps directly.
"""

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
MUS = [0.95, 0.9, 0.97, 0.8]  # a different mu each step: the carried factor is the earlier step's


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


def _random_rows(batch, n, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([np.sort(rng.choice(n, size=k, replace=False)) for _ in range(batch)]).astype(np.int32)


def _applied(M, sel, mu):
    """M with a pending decay applied, through the library (a copy; M is left as it is)."""
    out = M.clone()
    d3.decay_rows(out, sel, mu)
    return out


@pytest.mark.parametrize("n,m", [(64, 256), (96, 1004), (50, 333), (130, 1000)])
@pytest.mark.parametrize("f,norm_p", [((1, 4), 1), ((1, 8), 2), ((3, 5), 1), ((1, 1), 1)])
def test_carried_chain_is_bitwise_the_plain_chain(n, m, f, norm_p):
    batch = 3
    W = synthetic.gaussian((batch, n, m), seed=31, std=0.02, device=DEV)
    M = synthetic.gaussian((batch, n, m), seed=32, std=0.01, device=DEV)
    Wp, Mp = W.clone(), M.clone()      # plain steps
    Wc, Mc = W.clone(), M.clone()      # carried decay
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel_c = torch.empty((batch, d3.k_of(n, *f)), dtype=torch.int32, device=DEV)
    carry = None
    for t, mu in enumerate(MUS):
        G = synthetic.lowrank_batch(batch, n, m, base_seed=700 + 1000 * t + n, dtype=torch.bfloat16, device=DEV)
        sel_p = d3.step(Wp, Mp, G, f=f, mu=mu, eta=0.01, norm_p=norm_p, abc=ABC, restart_after=(2, 4),
                        status=status)
        # sel_c is both the carried list (read first) and the new selection (written after).
        d3.step(Wc, Mc, G, f=f, mu=mu, eta=0.01, norm_p=norm_p, abc=ABC, restart_after=(2, 4), status=status,
                sel_out=sel_c, carry=carry, defer=True)
        carry = (sel_c, mu)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(sel_p, sel_c), f"step {t}: selection differs"
        assert torch.equal(Wp, Wc), f"step {t}: W differs"
        assert torch.equal(Mp, _applied(Mc, sel_c, mu)), f"step {t}: M differs once the decay is applied"
        if f != (1, 1):
            rest = torch.ones((batch, n), dtype=torch.bool, device=DEV)
            rest.scatter_(1, sel_c.long(), False)
            assert torch.equal(Mp[rest], Mc[rest]), f"step {t}: an unselected row differs"
    d3.decay_rows(Mc, sel_c, MUS[-1])
    torch.cuda.synchronize()
    assert torch.equal(Mp, Mc)


@pytest.mark.parametrize("n,m,f", [(64, 256, (1, 4)), (96, 1004, (1, 8))])
def test_carried_chain_against_the_oracle(n, m, f):
    batch = 2
    W = synthetic.gaussian((batch, n, m), seed=33, std=0.02, device=DEV)
    M = torch.zeros((batch, n, m), dtype=torch.float32, device=DEV)
    Mo = [np.zeros((n, m), dtype=np.float32) for _ in range(batch)]
    sel = torch.empty((batch, d3.k_of(n, *f)), dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    carry = None
    for t, mu in enumerate(MUS[:3]):
        G = synthetic.lowrank_batch(batch, n, m, base_seed=800 + 1000 * t + n, dtype=torch.bfloat16, device=DEV)
        W_before = W.cpu().numpy().astype(np.float64)
        d3.step(W, M, G, f=f, mu=mu, eta=0.01, abc=ABC, restart_after=(2, 4), status=status, sel_out=sel,
                carry=carry, defer=True)
        carry = (sel, mu)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        Gc = G.float().cpu().numpy()
        Mnow = _applied(M, sel, mu)
        for i in range(batch):
            W1, M1, S, _ = oracle.dion3_step(W_before[i], Mo[i], Gc[i], *f, mu=mu, eta=0.01, abc=ABC,
                                             restart_after=(2, 4))
            Mo[i] = M1
            assert np.array_equal(sel[i].cpu().numpy().astype(np.int64), S), f"step {t}, matrix {i}: selection"
            assert np.array_equal(bits32(Mnow[i]), bits32(M1)), f"step {t}, matrix {i}: momentum"
            dW = W[i].double().cpu().numpy() - W_before[i]
            assert rel_frob(dW, W1 - W_before[i]) <= 3e-2, f"step {t}, matrix {i}: weight update"


def test_carry_with_given_rows_and_a_failed_selection():
    """A caller-chosen S (the carried list in its own buffer), with matrix 1's S invalid at the
    second step: that matrix is left unselected (sel -1) in both chains, so no decay is
    carried for it, exactly as the plain step applies none."""
    batch, n, m, f = 3, 64, 256, (1, 4)
    k = d3.k_of(n, *f)
    W = synthetic.gaussian((batch, n, m), seed=34, std=0.02, device=DEV)
    M = synthetic.gaussian((batch, n, m), seed=35, std=0.01, device=DEV)
    Wp, Mp, Wc, Mc = W.clone(), M.clone(), W.clone(), M.clone()
    status_p = torch.zeros(1, dtype=torch.int32, device=DEV)
    status_c = torch.zeros(1, dtype=torch.int32, device=DEV)
    carried = torch.empty((batch, k), dtype=torch.int32, device=DEV)
    carry = None
    for t, mu in enumerate(MUS[:3]):
        rows = _random_rows(batch, n, k, seed=60 + t)
        if t == 1:
            rows[1, 1] = rows[1, 0]
        rows_d = torch.from_numpy(rows).to(DEV)
        G = synthetic.lowrank_batch(batch, n, m, base_seed=900 + 1000 * t, dtype=torch.bfloat16, device=DEV)
        sel_p = d3.step(Wp, Mp, G, f=f, mu=mu, abc=ABC, restart_after=(2,), rows=rows_d, status=status_p)
        sel_c = d3.step(Wc, Mc, G, f=f, mu=mu, abc=ABC, restart_after=(2,), rows=rows_d, status=status_c,
                        carry=carry, defer=True)
        carried.copy_(sel_c)
        carry = (carried, mu)
        torch.cuda.synchronize()
        assert torch.equal(sel_p, sel_c)
        assert torch.equal(Wp, Wc)
        assert torch.equal(Mp, _applied(Mc, sel_c, mu))
        if t == 1:
            assert (sel_c[1] == -1).all()
    assert int(status_p.item()) == int(status_c.item()) == d3.DEV_SELECT


def test_given_rows_cannot_alias_the_carried_list():
    batch, n, m, f = 1, 64, 256, (1, 4)
    k = d3.k_of(n, *f)
    W = torch.zeros((batch, n, m), device=DEV)
    M = torch.zeros((batch, n, m), device=DEV)
    G = torch.zeros((batch, n, m), dtype=torch.bfloat16, device=DEV)
    rows = torch.from_numpy(_random_rows(batch, n, k, seed=1)).to(DEV)
    sel = torch.empty_like(rows)
    with pytest.raises(d3.Dion3Error):
        d3.step(W, M, G, f=f, abc=ABC, rows=rows, sel_out=sel, carry=(sel, 0.9), defer=True)


def test_decay_rows_matches_fp32_products():
    """M[b, r] *= mu for the listed rows, one fp32 rounding (numpy's float32 product rounds the
    same way); entries outside [0, n) are skipped; the ragged m takes the unvectorised path."""
    for batch, n, m in [(3, 40, 128), (2, 33, 97)]:
        M = synthetic.gaussian((batch, n, m), seed=36, std=1.0, device=DEV)
        rows = _random_rows(batch, n, 7, seed=n).astype(np.int32)
        rows[0, 0] = -1
        rows[1, -1] = n
        mu = np.float32(0.9)
        ref = M.cpu().numpy().copy()
        for b in range(batch):
            for r in rows[b]:
                if 0 <= r < n:
                    ref[b, r] = ref[b, r] * mu
        d3.decay_rows(M, torch.from_numpy(rows).to(DEV), float(mu))
        torch.cuda.synchronize()
        assert np.array_equal(bits32(M), bits32(ref))


def test_carried_decay_at_megabatch_size():
    """16 x 4096 x 4096 (k = 1024), two steps: the carried chain equals the plain chain."""
    batch, n, m, f = 16, 4096, 4096, (1, 4)
    W = synthetic.gaussian((batch, n, m), seed=37, std=0.02, device=DEV)
    M = synthetic.gaussian((batch, n, m), seed=38, std=0.01, device=DEV)
    Wp, Mp = W, M
    Wc, Mc = W.clone(), M.clone()
    sel = torch.empty((batch, d3.k_of(n, *f)), dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    carry = None
    for t, mu in enumerate(MUS[:2]):
        G = synthetic.gaussian((batch, n, m), seed=39 + t, std=1e-3, device=DEV).to(torch.bfloat16)
        sel_p = d3.step(Wp, Mp, G, f=f, mu=mu, abc=ABC, restart_after=(2, 4), status=status)
        d3.step(Wc, Mc, G, f=f, mu=mu, abc=ABC, restart_after=(2, 4), status=status, sel_out=sel, carry=carry,
                defer=True)
        carry = (sel, mu)
        del G
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(sel_p, sel)
        assert torch.equal(Wp, Wc)
    d3.decay_rows(Mc, sel, MUS[1])
    torch.cuda.synchronize()
    assert torch.equal(Mp, Mc)


def test_last_step_without_defer_needs_no_flush():
    """A carried chain whose last call takes the carry but does not defer (defer=False) ends with
    M exactly as after plain steps, with no dion3_decay_rows call."""
    batch, n, m, f = 2, 96, 512, (1, 4)
    W = synthetic.gaussian((batch, n, m), seed=40, std=0.02, device=DEV)
    M = synthetic.gaussian((batch, n, m), seed=41, std=0.01, device=DEV)
    Wp, Mp, Wc, Mc = W.clone(), M.clone(), W.clone(), M.clone()
    sel = torch.empty((batch, d3.k_of(n, *f)), dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    carry = None
    for t, mu in enumerate(MUS[:3]):
        G = synthetic.lowrank_batch(batch, n, m, base_seed=950 + 1000 * t, dtype=torch.bfloat16, device=DEV)
        d3.step(Wp, Mp, G, f=f, mu=mu, abc=ABC, restart_after=(2,), status=status)
        last = t == 2
        d3.step(Wc, Mc, G, f=f, mu=mu, abc=ABC, restart_after=(2,), status=status, sel_out=sel, carry=carry,
                defer=not last)
        carry = (sel, mu)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(Wp, Wc) and torch.equal(Mp, Mc)
