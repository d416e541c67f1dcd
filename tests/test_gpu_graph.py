"""A Dion3 step captured once in a CUDA graph and replayed, with the hyperparameters read from
device memory (dion3_step_dev): every replay must give exactly what eager calls give with the
same values, including a learning rate and weight decay that change between replays."""

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


SCHEDULE = [(0.95, 0.01, 0.1), (0.9, 0.02, 0.1), (0.95, 0.005, 0.0)]


@pytest.mark.parametrize("n,m,f,compute", [(128, 512, (1, 4), torch.float16), (96, 1004, (1, 8), torch.float16),
                                           (64, 256, (1, 2), torch.float32)])
def test_graph_replay_matches_eager(n, m, f, compute):
    batch = 3
    W0 = synthetic.gaussian((batch, n, m), seed=11, std=0.02, device=DEV)
    M0 = synthetic.gaussian((batch, n, m), seed=12, std=0.01, device=DEV)
    Gs = [synthetic.lowrank_batch(batch, n, m, base_seed=700 + 10 ** 6 * t, dtype=torch.bfloat16, device=DEV)
          for t in range(len(SCHEDULE))]
    k = d3.k_of(n, *f)
    ws_bytes = d3.workspace_bytes_step(batch, n, m, f[0], f[1], 1, compute, 2)

    # eager, host hyperparameters
    We, Me = W0.clone(), M0.clone()
    sel_e = []
    for t, (mu, eta, wd) in enumerate(SCHEDULE):
        sel_e.append(d3.step(We, Me, Gs[t], f=f, mu=mu, eta=eta, wd=wd, abc=ABC, restart_after=(2, 4),
                             compute=compute).clone())

    # captured once, replayed with new values in device memory
    Wg, Mg = W0.clone(), M0.clone()
    G = torch.empty_like(Gs[0])
    hyper = torch.tensor(SCHEDULE[0], dtype=torch.float32, device=DEV)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    sel = torch.empty((batch, k), dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # one eager call on scratch copies first: it fills the library's per-device caches
    d3.step(W0.clone(), M0.clone(), Gs[0], f=f, abc=ABC, restart_after=(2, 4), compute=compute, hyper=hyper,
            decay=True, workspace=ws, sel_out=sel, status=status)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        d3.step(Wg, Mg, G, f=f, abc=ABC, restart_after=(2, 4), compute=compute, hyper=hyper, decay=True,
                workspace=ws, sel_out=sel, status=status)
    for t, vals in enumerate(SCHEDULE):
        G.copy_(Gs[t])
        hyper.copy_(torch.tensor(vals, dtype=torch.float32))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(sel, sel_e[t]), f"replay {t}: selection differs"
    assert int(status.item()) == 0
    assert np.array_equal(bits32(Mg), bits32(Me))
    assert np.array_equal(bits32(Wg), bits32(We))


def test_device_hyper_matches_oracle_with_decay():
    n, m, f = 80, 320, (1, 4)
    W = synthetic.gaussian((2, n, m), seed=21, std=0.02, device=DEV)
    M = synthetic.gaussian((2, n, m), seed=22, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(2, n, m, base_seed=90, device=DEV)
    W0, M0, Gc = W.cpu().numpy().copy(), M.cpu().numpy().copy(), G.float().cpu().numpy()
    hyper = torch.tensor([0.9, 0.02, 0.05], dtype=torch.float32, device=DEV)
    sel = d3.step(W, M, G, f=f, abc=ABC, restart_after=(2,), hyper=hyper, decay=True)
    torch.cuda.synchronize()
    for i in range(2):
        W1, M1, S, _ = oracle.dion3_step(W0[i], M0[i], Gc[i], *f, mu=0.9, eta=0.02, wd=0.05, norm_p=1, abc=ABC,
                                         restart_after=(2,))
        assert np.array_equal(sel[i].cpu().numpy().astype(np.int64), S)
        assert np.array_equal(bits32(M[i]), bits32(M1))
        dW = W[i].double().cpu().numpy() - W0[i]
        assert rel_frob(dW, W1 - W0[i]) <= 3e-2


def test_decay_off_ignores_wd():
    n, m = 64, 256
    W = synthetic.gaussian((1, n, m), seed=31, std=0.02, device=DEV)
    M = synthetic.gaussian((1, n, m), seed=32, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(1, n, m, base_seed=95, device=DEV)
    Wa, Ma = W.clone(), M.clone()
    d3.step(Wa, Ma, G, f=(1, 4), abc=ABC, restart_after=(2,), hyper=torch.tensor([0.95, 0.01, 0.3], device=DEV),
            decay=False)
    Wb, Mb = W.clone(), M.clone()
    d3.step(Wb, Mb, G, f=(1, 4), mu=0.95, eta=0.01, wd=0.0, abc=ABC, restart_after=(2,))
    torch.cuda.synchronize()
    assert torch.equal(Wa, Wb) and torch.equal(Ma, Mb)


@pytest.mark.parametrize("n,m,f,compute", [(128, 512, (1, 4), torch.float16), (96, 1004, (1, 8), torch.float16)])
def test_graph_replay_with_carried_decay(n, m, f, compute):
    """dion3_step_dev_carry captured once: each replay applies the previous replay's decay (its mu
    kept in a device word that starts at 1.0) and leaves its own pending.  After the last replay
    and dion3_decay_rows, W, M and every selection equal eager plain steps bit for bit."""
    batch = 3
    W0 = synthetic.gaussian((batch, n, m), seed=13, std=0.02, device=DEV)
    M0 = synthetic.gaussian((batch, n, m), seed=14, std=0.01, device=DEV)
    Gs = [synthetic.lowrank_batch(batch, n, m, base_seed=750 + 10 ** 6 * t, dtype=torch.bfloat16, device=DEV)
          for t in range(len(SCHEDULE))]
    k = d3.k_of(n, *f)
    ws_bytes = d3.workspace_bytes_step(batch, n, m, f[0], f[1], 1, compute, 2)

    We, Me = W0.clone(), M0.clone()
    sel_e = []
    for t, (mu, eta, wd) in enumerate(SCHEDULE):
        sel_e.append(d3.step(We, Me, Gs[t], f=f, mu=mu, eta=eta, wd=wd, abc=ABC, restart_after=(2, 4),
                             compute=compute).clone())

    Wg, Mg = W0.clone(), M0.clone()
    G = torch.empty_like(Gs[0])
    hyper = torch.tensor(SCHEDULE[0], dtype=torch.float32, device=DEV)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=DEV)
    sel = torch.full((batch, k), -1, dtype=torch.int32, device=DEV)   # nothing pending yet
    mu_word = torch.ones(1, dtype=torch.float32, device=DEV)          # a factor of 1 changes nothing
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # warm the library's per-device caches on scratch state
    d3.step(W0.clone(), M0.clone(), Gs[0], f=f, abc=ABC, restart_after=(2, 4), compute=compute, hyper=hyper,
            decay=True, workspace=ws, sel_out=sel.clone(), status=status,
            carry=(None, torch.ones(1, dtype=torch.float32, device=DEV)), defer=True)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        d3.step(Wg, Mg, G, f=f, abc=ABC, restart_after=(2, 4), compute=compute, hyper=hyper, decay=True,
                workspace=ws, sel_out=sel, status=status, carry=(sel, mu_word), defer=True)
    for t, vals in enumerate(SCHEDULE):
        G.copy_(Gs[t])
        hyper.copy_(torch.tensor(vals, dtype=torch.float32))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(sel, sel_e[t]), f"replay {t}: selection differs"
        assert float(mu_word.item()) == float(np.float32(vals[0])), f"replay {t}: carried mu not stored"
    assert int(status.item()) == 0
    assert np.array_equal(bits32(Wg), bits32(We))
    d3.decay_rows(Mg, sel, float(mu_word.item()))
    torch.cuda.synchronize()
    assert np.array_equal(bits32(Mg), bits32(Me))
