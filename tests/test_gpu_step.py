"""One Dion3 step through the C ABI against the float64 oracle.

Bars: selected row indices bit-exact; the fp32 momentum M bit-exact (one rounding after
+G, one after *mu); the weight update Delta W within 3e-2 relative Frobenius error of the
oracle's (float16 Gram Newton-Schulz, the paper's precision); 1e-4 in fp32 compute mode.
"""

import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import oracle
import synthetic
from gpu_util import bits32, rel_frob, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
ABC = [(3.4445, -4.7750, 2.0315)] * 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


def _run_and_check(W, M, G, f, mu, eta, norm_p, restarts, compute=torch.float16, wd=0.0, idx=None, tol=3e-2,
                   check_w=True):
    """One step on the GPU (whole batch) and on the oracle (matrices in idx); compare."""
    batch = M.shape[0]
    idx = range(batch) if idx is None else idx
    W0 = {i: W[i].cpu().numpy().copy() for i in idx}
    M0 = {i: M[i].cpu().numpy().copy() for i in idx}
    Gc = {i: G[i].float().cpu().numpy() for i in idx}
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel = d3.step(W, M, G, f=f, mu=mu, eta=eta, wd=wd, norm_p=norm_p, abc=ABC, restart_after=restarts,
                  compute=compute, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in idx:
        W1, M1, S, _ = oracle.dion3_step(W0[i], M0[i], Gc[i], *f, mu=mu, eta=eta, wd=wd, norm_p=norm_p, abc=ABC,
                                         restart_after=restarts)
        assert np.array_equal(sel[i].cpu().numpy().astype(np.int64), S), f"matrix {i}: selection differs"
        assert np.array_equal(bits32(M[i]), bits32(M1)), f"matrix {i}: momentum differs"
        if check_w:
            dW = W[i].double().cpu().numpy() - W0[i]
            assert rel_frob(dW, W1 - W0[i]) <= tol, f"matrix {i}: weight update off"
    return sel


@pytest.mark.parametrize("n,m", [(64, 256), (130, 1000), (96, 1004)])
@pytest.mark.parametrize("f", [(1, 4), (1, 8), (3, 5), (1, 1)])
@pytest.mark.parametrize("norm_p", [1, 2])
def test_three_steps(n, m, f, norm_p):
    batch = 3
    W = synthetic.gaussian((batch, n, m), seed=1, std=0.02, device=DEV)
    M = torch.zeros((batch, n, m), dtype=torch.float32, device=DEV)
    for step in range(3):
        G = synthetic.lowrank_batch(batch, n, m, base_seed=400 + 10 ** 6 * step + n, dtype=torch.bfloat16,
                                    device=DEV)
        _run_and_check(W, M, G, f, 0.95, 0.01, norm_p, (2, 4))


def test_f1_selects_every_row():
    n, m = 48, 200
    W = synthetic.gaussian((2, n, m), seed=2, std=0.02, device=DEV)
    M = synthetic.gaussian((2, n, m), seed=3, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(2, n, m, base_seed=50, device=DEV)
    sel = _run_and_check(W, M, G, (1, 1), 0.9, 0.02, 1, (2,))
    assert torch.equal(sel.cpu(), torch.arange(n, dtype=torch.int32).expand(2, n))


def test_exact_ties_go_to_lower_index():
    """Duplicated rows have exactly equal keys: the lower row index must win.  (The selected rows
    repeat, so M[S,:] is rank-deficient and its orthogonalization is ill-posed in half precision;
    only the selection and the momentum are compared.)"""
    n, m = 40, 128
    base = synthetic.gaussian((5, m), seed=4, std=0.05, dtype=torch.bfloat16, device=DEV)
    G = base[torch.arange(n, device=DEV) % 5].unsqueeze(0).contiguous()   # rows repeat with period 5
    M = torch.zeros((1, n, m), device=DEV)
    W = torch.zeros((1, n, m), device=DEV)
    for norm_p in (1, 2):
        _run_and_check(W.clone(), M.clone(), G, (1, 4), 0.95, 0.01, norm_p, (2,), check_w=False)


def test_near_ties_resolved_exactly():
    """Rows that differ from a twin by one fp32 ulp in one entry: the fp32 key intervals overlap
    and the device must fall back to exact integer sums."""
    n, m = 64, 512
    M = synthetic.gaussian((1, n, m), seed=5, std=0.05, device=DEV)
    src = torch.arange(0, n, 2, device=DEV)
    M[0, src + 1] = M[0, src]
    Mi = M.view(torch.int32)
    Mi[0, src + 1, 7] += torch.where(src % 4 == 0, 1, -1).to(torch.int32)   # +/- one ulp
    G = torch.zeros((1, n, m), dtype=torch.bfloat16, device=DEV)
    W = torch.zeros((1, n, m), device=DEV)
    for norm_p in (1, 2):
        for f in ((1, 2), (1, 4), (3, 8)):
            _run_and_check(W.clone(), M.clone(), G, f, 0.95, 0.01, norm_p, (2,), check_w=False)



@pytest.mark.parametrize("n,m,f", [(1, 1, (1, 1)), (1, 8, (1, 4)), (2, 3, (1, 2)), (3, 17, (1, 8)), (8, 8, (1, 1)),
                                   (17, 40, (1, 4))])
@pytest.mark.parametrize("norm_p", [1, 2])
def test_tiny_shapes(n, m, f, norm_p):
    """Degenerate sizes: one row, k = 1 of 3 rows, square matrices, rows of 1 to 3 elements
    (no vector path; rows inside the batch not 16-byte aligned).  Two chained steps on a batch
    of three against the oracle."""
    batch = 3
    W = synthetic.gaussian((batch, n, m), seed=5, std=0.02, device=DEV)
    M = torch.zeros((batch, n, m), dtype=torch.float32, device=DEV)
    for step in range(2):
        G = synthetic.lowrank_batch(batch, n, m, base_seed=700 + 100 * step + 10 * n + m, dtype=torch.bfloat16,
                                    device=DEV)
        _run_and_check(W, M, G, f, 0.95, 0.01, norm_p, (2, 4))


def test_empty_batch_is_a_no_op():
    """batch = 0: nothing to select or update; the call succeeds and returns no rows."""
    W = torch.zeros((0, 64, 256), dtype=torch.float32, device=DEV)
    M = torch.zeros_like(W)
    G = torch.zeros((0, 64, 256), dtype=torch.bfloat16, device=DEV)
    sel = d3.step(W, M, G, f=(1, 4), abc=ABC, restart_after=(2, 4))
    torch.cuda.synchronize()
    assert tuple(sel.shape) == (0, d3.k_of(64, 1, 4))


@pytest.mark.parametrize("gdt", [torch.float32, torch.float16])
def test_gradient_dtypes_and_weight_decay(gdt):
    n, m = 80, 320
    W = synthetic.gaussian((2, n, m), seed=6, std=0.02, device=DEV)
    M = synthetic.gaussian((2, n, m), seed=7, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(2, n, m, base_seed=60, dtype=gdt, device=DEV)
    _run_and_check(W, M, G, (1, 4), 0.95, 0.01, 1, (2,), wd=0.1)


def test_fp32_compute_mode():
    n, m = 64, 256
    W = synthetic.gaussian((2, n, m), seed=8, std=0.02, device=DEV)
    M = synthetic.gaussian((2, n, m), seed=9, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(2, n, m, base_seed=80, device=DEV)
    _run_and_check(W, M, G, (1, 2), 0.95, 0.01, 1, (2,), compute=torch.float32, tol=1e-4)


def test_nonfinite_gradient_sets_status():
    n, m = 32, 64
    W = torch.zeros((1, n, m), device=DEV)
    M = torch.zeros((1, n, m), device=DEV)
    G = synthetic.lowrank_batch(1, n, m, base_seed=90, device=DEV)
    G[0, 3, 5] = float("nan")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    d3.step(W, M, G, f=(1, 4), abc=ABC, restart_after=(2,), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & d3.DEV_NONFINITE


@pytest.mark.parametrize("shape,count,f,norm_p,computes", [
    ((768, 2048), 3072, (1, 8), 1, (torch.float16, torch.bfloat16)),
    ((4096, 4096), 128, (1, 4), 1, (torch.float16, torch.bfloat16)),
    ((4096, 11008), 96, (1, 4), 1, (torch.float16, torch.bfloat16)),
    ((4096, 11008), 96, (1, 4), 2, (torch.float16,)),
])
def test_megabatch_full_size_two_steps(shape, count, f, norm_p, computes):
    """Full-size megabatches (MoE experts at f = 1/8 and 7B dense shapes at f = 1/4, each with float16
    and bfloat16 Gram iterates; the 4096 x 11008 batch also with row L2 selection, where the exact
    re-rank sums 11008 squares per row): matrices 0, B/2 and B-1 against the oracle over two
    steps (the second starts from error-feedback state).  Rows and M bit-exact, Delta W <= 3e-2.

    The oracle runs once per matrix and step: its M trajectory does not depend on O, and with
    wd = 0 its Delta W = -eta' O does not depend on W, so one float64 chain serves every
    compute type on the device."""
    n, m = shape
    W = torch.empty((count, n, m), dtype=torch.float32, device=DEV)
    for i in range(count):
        W[i] = synthetic.gaussian((n, m), seed=5000 + i, std=0.02, device=DEV)
    M = torch.zeros((count, n, m), dtype=torch.float32, device=DEV)
    runs = {c: ((W, M) if j == 0 else (W.clone(), M.clone())) for j, c in enumerate(computes)}
    idx = (0, count // 2, count - 1)
    Wo = {i: W[i].double().cpu().numpy() for i in idx}
    Mo = {i: np.zeros((n, m), np.float32) for i in idx}
    worst = {str(c): 0.0 for c in computes}
    for step in range(2):
        G = torch.empty((count, n, m), dtype=torch.bfloat16, device=DEV)
        for i in range(count):
            synthetic.lowrank_plus_noise(n, m, 4000 + i + 10 ** 6 * step, dtype=torch.bfloat16, device=DEV, out=G[i])
        ref = {}
        for i in idx:
            W1, M1, S, _ = oracle.dion3_step(Wo[i], Mo[i], G[i].float().cpu().numpy(), *f, mu=0.95, eta=0.01,
                                             norm_p=norm_p, abc=ABC, restart_after=(2, 4))
            ref[i] = (W1 - Wo[i], M1, S)
            Wo[i], Mo[i] = W1, M1
        for c, (Wc, Mc) in runs.items():
            before = {i: Wc[i].double().cpu().numpy() for i in idx}
            status = torch.zeros(1, dtype=torch.int32, device=DEV)
            sel = d3.step(Wc, Mc, G, f=f, mu=0.95, eta=0.01, norm_p=norm_p, abc=ABC, restart_after=(2, 4),
                          compute=c, status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            for i in idx:
                dW_ref, M1, S = ref[i]
                assert np.array_equal(sel[i].cpu().numpy().astype(np.int64), S), f"step {step} matrix {i}: rows"
                assert np.array_equal(bits32(Mc[i]), bits32(M1)), f"step {step} matrix {i}: momentum"
                err = rel_frob(Wc[i].double().cpu().numpy() - before[i], dW_ref)
                worst[str(c)] = max(worst[str(c)], err)
        del G
    print(f"{count}x{n}x{m} f={f} norm_p={norm_p}: worst Delta W rel. Frobenius error per iterate type:", worst)
    for c, err in worst.items():
        assert err <= 3e-2, f"{c}: {err:.4g}"


def _random_rows(batch, n, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([np.sort(rng.choice(n, size=k, replace=False)) for _ in range(batch)]).astype(np.int32)


@pytest.mark.parametrize("n,m,f", [(64, 256, (1, 4)), (130, 1000, (1, 8)), (96, 1004, (3, 5))])
def test_given_random_rows(n, m, f):
    """A caller-chosen S (random selection): the same rows are used, M bit-exact, Delta W in 3e-2."""
    batch = 3
    k = d3.k_of(n, *f)
    W = synthetic.gaussian((batch, n, m), seed=13, std=0.02, device=DEV)
    M = synthetic.gaussian((batch, n, m), seed=14, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(batch, n, m, base_seed=500 + n, dtype=torch.bfloat16, device=DEV)
    rows = _random_rows(batch, n, k, seed=n)
    W0, M0, Gc = W.cpu().numpy().copy(), M.cpu().numpy().copy(), G.float().cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel = d3.step(W, M, G, f=f, mu=0.9, eta=0.01, abc=ABC, restart_after=(2, 4),
                  rows=torch.from_numpy(rows).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(sel.cpu().numpy(), rows)
    for i in range(batch):
        W1, M1, S, _ = oracle.dion3_step(W0[i], M0[i], Gc[i], *f, mu=0.9, eta=0.01, abc=ABC, restart_after=(2, 4),
                                         rows=rows[i])
        assert np.array_equal(bits32(M[i]), bits32(M1))
        dW = W[i].double().cpu().numpy() - W0[i]
        assert rel_frob(dW, W1 - W0[i]) <= 3e-2


def test_given_rows_equal_to_topk_match_default_bitwise():
    n, m = 128, 512
    W = synthetic.gaussian((2, n, m), seed=15, std=0.02, device=DEV)
    M = synthetic.gaussian((2, n, m), seed=16, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(2, n, m, base_seed=520, dtype=torch.bfloat16, device=DEV)
    Wa, Ma = W.clone(), M.clone()
    sel = d3.step(Wa, Ma, G, f=(1, 4), abc=ABC, restart_after=(2,))
    Wb, Mb = W.clone(), M.clone()
    sel_b = d3.step(Wb, Mb, G, f=(1, 4), abc=ABC, restart_after=(2,), rows=sel.clone())
    torch.cuda.synchronize()
    assert torch.equal(sel, sel_b)
    assert torch.equal(Ma, Mb) and torch.equal(Wa, Wb)


def test_invalid_given_rows_leave_that_matrix_unselected():
    """Matrix 1 gets a repeated row, matrix 2 an out-of-range one: both are flagged and left
    alone (W unchanged, M only + G); matrix 0 is stepped normally."""
    n, m, f = 64, 256, (1, 4)
    k = d3.k_of(n, *f)
    W = synthetic.gaussian((3, n, m), seed=17, std=0.02, device=DEV)
    M = synthetic.gaussian((3, n, m), seed=18, std=0.01, device=DEV)
    G = synthetic.lowrank_batch(3, n, m, base_seed=540, dtype=torch.bfloat16, device=DEV)
    rows = _random_rows(3, n, k, seed=3)
    rows[1, 1] = rows[1, 0]
    rows[2, -1] = n
    W0, M0, Gc = W.cpu().numpy().copy(), M.cpu().numpy().copy(), G.float().cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel = d3.step(W, M, G, f=f, mu=0.9, eta=0.01, abc=ABC, restart_after=(2,),
                  rows=torch.from_numpy(rows).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 0x4
    assert (sel[1:] == -1).all()
    for i in (1, 2):
        assert np.array_equal(W[i].cpu().numpy(), W0[i])
        assert np.array_equal(bits32(M[i]), bits32(M0[i] + Gc[i].astype(np.float32)))
    W1, M1, S, _ = oracle.dion3_step(W0[0], M0[0], Gc[0], *f, mu=0.9, eta=0.01, abc=ABC, restart_after=(2,),
                                     rows=rows[0])
    assert np.array_equal(bits32(M[0]), bits32(M1))
    assert rel_frob(W[0].double().cpu().numpy() - W0[0], W1 - W0[0]) <= 3e-2




def _permuted_rows(n: int, m: int, seed: int):
    """fp32 M and bf16 G, [n, m], whose row i is the same column permutation p_i of one fp32 and
    one bf16 vector, so that every row of M + G is a permutation of one row."""
    rng = np.random.default_rng(seed)
    perm = torch.from_numpy(np.stack([rng.permutation(m) for _ in range(n)])).to(DEV)
    vm = synthetic.gaussian((m,), seed=seed + 1, std=0.05, device=DEV)
    vg = synthetic.gaussian((m,), seed=seed + 2, std=0.01, dtype=torch.bfloat16, device=DEV)
    return vm[perm], vg[perm]


@pytest.mark.parametrize("norm_p", [1, 2])
def test_tied_rows_more_ambiguous_than_threads(norm_p):
    """Selection when most rows tie exactly, so that more rows straddle the boundary than the
    selection block has threads and the exact ranking takes its radix-select route.  Matrix 0:
    rows that are permutations of one row, 64 of them (G zero there) one ulp smaller or larger in
    their largest entry.  Matrix 1: all zero, every key 0, S = {0, ..., k-1} and no update.
    Full oracle parity: rows bit-exact, M bit-exact, Delta W within 3e-2."""
    n = m = 2048
    M = torch.zeros((2, n, m), dtype=torch.float32, device=DEV)
    G = torch.zeros((2, n, m), dtype=torch.bfloat16, device=DEV)
    M[0], G[0] = _permuted_rows(n, m, 81)
    rng = np.random.default_rng(84)
    rows = np.sort(rng.choice(n, 64, replace=False))
    ri = torch.from_numpy(rows).to(DEV)
    P = (M[0, ri].cpu().numpy().astype(np.float64) + G[0, ri].float().cpu().numpy()).astype(np.float32)
    P.view(np.int32)[np.arange(64), np.argmax(np.abs(P), axis=1)] += np.where(rng.random(64) < 0.5, -1, 1).astype(np.int32)
    M[0, ri] = torch.from_numpy(P).to(DEV)
    G[0, ri] = 0
    W = synthetic.gaussian((2, n, m), seed=85, std=0.02, device=DEV)
    W1_zero = W[1].clone()
    sel = _run_and_check(W, M, G, (1, 4), 0.95, 0.01, norm_p, (2, 4))
    k = d3.k_of(n, 1, 4)
    assert np.array_equal(sel[1].cpu().numpy(), np.arange(k))
    assert torch.equal(W[1], W1_zero)


def _approx_keys(M1: np.ndarray, norm_p: int) -> np.ndarray:
    """float64 sums of |x| (or x^2) per row: every term is exact in float64 and numpy's pairwise
    sum of at most 65536 nonnegative terms is within 1e-14 relative of the exact key."""
    x = np.abs(M1.astype(np.float64))
    return x.sum(axis=1) if norm_p == 1 else (x * x).sum(axis=1)


def _expected_rows(M1: np.ndarray, k: int, norm_p: int) -> np.ndarray:
    """The k rows of largest exact key, ties to the lower index, ascending -- without exact keys
    for every row: the float64 sums settle each row more than 1e-9 relative away from the k-th
    sum, and the oracle's exact integer keys rank the rows inside that margin."""
    approx = _approx_keys(M1, norm_p)
    kth = np.sort(approx)[::-1][k - 1]
    sure = np.where(approx > kth * (1 + 1e-9))[0]
    amb = np.where(np.abs(approx - kth) <= kth * 1e-9)[0]
    assert len(sure) <= k <= len(sure) + len(amb)
    exact = oracle.exact_row_keys(np.ascontiguousarray(M1[amb]), norm_p)
    ranked = sorted(range(len(amb)), key=lambda i: (-exact[i], amb[i]))
    return np.sort(np.concatenate([sure, amb[ranked[:k - len(sure)]]]))


@pytest.mark.parametrize("n,m,f", [(16384, 16384, (1, 4)), (1024, 65536, (1, 8))])
@pytest.mark.parametrize("norm_p", [1, 2])
def test_boundary_ties_at_the_maximum_sizes(n, m, f, norm_p):
    """The step's size limits (n = 16384 rows, m = 65536 columns) with the k-th largest key inside
    a group of tied rows: the 64 rows of smallest key are rewritten (G = 0 there) as column
    permutations of the row ranked k - 32 -- equal exact keys, unequal fp32 sums -- and then the
    lowest-indexed of them loses one ulp in its largest entry and the highest-indexed gains one.
    The fp32 key intervals cannot order the group, so the exact integer re-rank runs on rows of
    full width.  Rows bit-exact against exact keys, M bit-exact, W changed on exactly the selected
    rows, and (where the oracle's float64 Gram Newton-Schulz of the k selected rows is quick)
    Delta W within 3e-2 of the oracle's.  Gradients are Gaussian here: the selection sees only M + G."""
    k = d3.k_of(n, *f)
    g = 64
    rng = np.random.default_rng(1000 * norm_p + m // n)
    M = synthetic.gaussian((1, n, m), seed=71, std=0.05, device=DEV)
    G = synthetic.gaussian((1, n, m), seed=72, std=0.01, dtype=torch.bfloat16, device=DEV)
    W = synthetic.gaussian((1, n, m), seed=73, std=0.02, device=DEV)
    M1 = (M[0].cpu().numpy().astype(np.float64) + G[0].float().cpu().numpy()).astype(np.float32)
    order = np.argsort(-_approx_keys(M1, norm_p), kind="stable")
    base = int(order[k - g // 2 - 1])
    group = np.sort(order[-g:])
    row = M1[base].copy()
    for r in group:
        M1[r] = row[rng.permutation(m)]
    bits = M1.view(np.int32)
    bits[group[0], int(np.argmax(np.abs(M1[group[0]])))] -= 1   # |x| one ulp smaller
    bits[group[-1], int(np.argmax(np.abs(M1[group[-1]])))] += 1  # |x| one ulp larger
    gi = torch.from_numpy(group).to(DEV)
    M[0, gi] = torch.from_numpy(M1[group]).to(DEV)
    G[0, gi] = 0
    W0 = W[0].cpu().numpy().copy()
    S = _expected_rows(M1, k, norm_p)
    assert group[-1] in S and group[0] not in S

    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel = d3.step(W, M, G, f=f, mu=0.95, eta=0.01, norm_p=norm_p, abc=ABC, restart_after=(2, 4), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(sel[0].cpu().numpy().astype(np.int64), S)
    Mexp = M1.copy()
    Mexp[S] = (np.float64(np.float32(0.95)) * M1[S].astype(np.float64)).astype(np.float32)
    assert np.array_equal(bits32(M[0]), Mexp.view(np.uint32))
    W1 = W[0].cpu().numpy()
    keep = np.ones(n, dtype=bool)
    keep[S] = False
    assert np.array_equal(W1[keep].view(np.uint32), W0[keep].view(np.uint32))
    assert np.isfinite(W1[S]).all()
    if k * k * m <= 2**30:
        O = oracle.gram_ns(M1[S].astype(np.float64), ABC, (2, 4))
        eta_p = 0.01 * np.sqrt(f[1] / f[0])
        assert rel_frob(W1[S].astype(np.float64) - W0[S], -eta_p * O) <= 3e-2


@pytest.mark.parametrize("norm_p", [1, 2])
def test_all_rows_tied_at_the_maximum_n(norm_p):
    """n = m = 16384 with every row of M and of G the same column permutation of one row, so
    every row of M + G is a permutation of one row: equal exact keys, fp32 sums that differ with
    the order.  Every row straddles the boundary, the exact re-rank runs on all 16384 rows, and
    ties to the lower index make S = {0, ..., k-1}.  M bit-exact, W changed on rows < k only."""
    n = m = 16384
    k = d3.k_of(n, 1, 4)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(76 + norm_p)
    perm = torch.argsort(torch.rand((n, m), generator=gen, device=DEV), dim=1)
    vm = synthetic.gaussian((m,), seed=74, std=0.05, device=DEV)
    vg = synthetic.gaussian((m,), seed=75, std=0.01, dtype=torch.bfloat16, device=DEV)
    M = vm[perm].unsqueeze(0).contiguous()
    G = vg[perm].unsqueeze(0).contiguous()
    W = synthetic.gaussian((1, n, m), seed=77, std=0.02, device=DEV)
    W0 = W[0].cpu().numpy().copy()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sel = d3.step(W, M, G, f=(1, 4), mu=0.95, eta=0.01, norm_p=norm_p, abc=ABC, restart_after=(2, 4),
                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(sel[0].cpu().numpy(), np.arange(k))
    v1 = (vm.double().cpu().numpy() + vg.double().cpu().numpy()).astype(np.float32)
    v2 = (np.float64(np.float32(0.95)) * v1.astype(np.float64)).astype(np.float32)
    p = perm.cpu().numpy()
    del perm
    Mh = bits32(M[0])
    assert np.array_equal(Mh[:k], v2.view(np.uint32)[p[:k]])
    assert np.array_equal(Mh[k:], v1.view(np.uint32)[p[k:]])
    W1 = W[0].cpu().numpy()
    assert np.array_equal(W1[k:].view(np.uint32), W0[k:].view(np.uint32))
    assert np.isfinite(W1[:k]).all() and not np.array_equal(W1[:k], W0[:k])
