"""Pins for the oracle's Dion3 step, selection and exact keys.

Checked against: brute force with exact fractions, the pairwise definition
of "top k with ties to the lower index", an independent fp32-state Muon
(f = 1 must be Muon), numpy fp32 arithmetic for the stored momentum, and the
learning-rate transfer identity ||eta' O||_F = eta sqrt(n).
"""

import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _fp32_matrix(n, m, seed, specials=False):
    rng = np.random.default_rng(seed)
    M = (rng.standard_normal((n, m)) * 0.05).astype(np.float32)
    if specials:
        M[0, :3] = [np.float32(1e-45), np.float32(-1.2e-38), np.float32(0.0)]   # subnormals and zero
        M[1, :2] = [np.float32(3.0e38), np.float32(-2.5e37)]                      # near the top of fp32
        M[2, 0] = np.float32(-0.0)
    return M


@pytest.mark.parametrize("norm_p", [1, 2])
def test_exact_keys_equal_fraction_sums(norm_p):
    M = _fp32_matrix(6, 13, seed=1, specials=True)
    keys = oracle.exact_row_keys(M, norm_p)
    scale = Fraction(2) ** (149 if norm_p == 1 else 298)
    for i in range(M.shape[0]):
        if norm_p == 1:
            exact = sum(abs(Fraction(float(v))) for v in M[i])
        else:
            exact = sum(Fraction(float(v)) ** 2 for v in M[i])
        assert Fraction(keys[i]) == exact * scale


def test_exact_keys_reject_nonfinite():
    M = _fp32_matrix(3, 4, 0)
    M[1, 2] = np.nan
    with pytest.raises(ValueError):
        oracle.exact_row_keys(M)


def _is_valid_topk(keys, S, k):
    S = set(int(i) for i in S)
    if len(S) != k:
        return False
    for i in S:
        for j in range(len(keys)):
            if j in S:
                continue
            if not (keys[i] > keys[j] or (keys[i] == keys[j] and i < j)):
                return False
    return True


@pytest.mark.parametrize("seed", range(6))
def test_top_k_matches_pairwise_definition(seed):
    rng = np.random.default_rng(seed)
    n = 23
    keys = [int(v) for v in rng.integers(0, 6, size=n)]   # many ties on purpose
    for k in [0, 1, 5, 11, 22, 23]:
        S = oracle.top_k_rows(keys, k)
        assert list(S) == sorted(S)
        assert _is_valid_topk(keys, S, k)


def test_ties_go_to_lower_index():
    M = np.tile(np.float32([0.5, -0.25, 0.125]), (6, 1))     # six identical rows
    M[4] *= np.float32(2.0)                                   # row 4 strictly largest
    keys = oracle.exact_row_keys(M, 1)
    assert list(oracle.top_k_rows(keys, 3)) == [0, 1, 4]


def test_ceil_k():
    assert oracle.ceil_k(4096, 1, 4) == 1024
    assert oracle.ceil_k(768, 1, 8) == 96
    assert oracle.ceil_k(10, 1, 3) == 4
    assert oracle.ceil_k(7, 1, 1) == 7
    assert oracle.ceil_k(1, 1, 8) == 1
    with pytest.raises(ValueError):
        oracle.ceil_k(5, 0, 1)


def _step_inputs(n, m, seed):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((n, m)) * 0.02).astype(np.float32)
    M = (rng.standard_normal((n, m)) * 0.1).astype(np.float32)
    # G holds bf16 values: fp32 with the low 16 bits cleared
    G = (rng.standard_normal((n, m)) * 0.05).astype(np.float32)
    G = (G.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    return W, M, G


@pytest.mark.parametrize("f", [(1, 4), (1, 8), (3, 5)])
@pytest.mark.parametrize("norm_p", [1, 2])
def test_error_feedback_state_is_fp32_exact(f, norm_p, jordan):
    """Error feedback: unselected rows change by exactly +G, selected rows become mu*(M+G) in fp32."""
    n, m = 24, 40
    W, M, G = _step_inputs(n, m, seed=3)
    mu = 0.95
    W1, M1, S, O = oracle.dion3_step(W, M, G, *f, mu=mu, eta=0.01, norm_p=norm_p,
                                     abc=[jordan] * 5, restart_after=(2,))
    summed = M + G                                   # numpy fp32 add: one correctly rounded op
    decayed = np.float32(mu) * summed                # numpy fp32 multiply
    sel = np.zeros(n, bool)
    sel[S] = True
    assert len(S) == oracle.ceil_k(n, *f)
    assert np.array_equal(M1[~sel].view(np.uint32), summed[~sel].view(np.uint32))
    assert np.array_equal(M1[sel].view(np.uint32), decayed[sel].view(np.uint32))
    # unselected rows of W untouched (wd = 0); the selection is the exact top k of the summed state
    assert np.array_equal(W1[~sel], W[~sel].astype(np.float64))
    keys = oracle.exact_row_keys(summed, norm_p)
    assert _is_valid_topk(keys, S, len(S))


def _muon_fp32_state(W, Ms, Gs, mu, eta, abc):
    """Muon with an fp32 momentum buffer: M <- fl32(fl32(mu M) + G); W <- W - eta NS(M)."""
    W = W.astype(np.float64)
    M = Ms
    for G in Gs:
        M = (np.float32(mu) * M) + G
        W = W - eta * oracle.ns_standard(M.astype(np.float64), abc)
    return W


def test_f1_is_muon_over_three_steps(jordan):
    """f = 1 selects every row, and Dion3 reduces to Muon (montaan summary, update-rule paragraph)."""
    n, m = 12, 30
    W0, _, _ = _step_inputs(n, m, seed=4)
    Gs = [_step_inputs(n, m, seed=40 + t)[2] for t in range(3)]
    mu, eta = 0.95, 0.01
    abc = [jordan] * 5
    W = W0
    M = np.zeros((n, m), np.float32)
    for G in Gs:
        W, M, S, _ = oracle.dion3_step(W, M, G, 1, 1, mu=mu, eta=eta, abc=abc, restart_after=(2,))
        assert list(S) == list(range(n))
    ref = _muon_fp32_state(W0, np.zeros((n, m), np.float32), Gs, mu, eta, abc)
    assert np.linalg.norm(W - ref) / np.linalg.norm(ref - W0) <= 1e-12


def test_learning_rate_transfer_keeps_update_norm():
    """Prerequisite 'spectral-norm steepest descent': with exact polar, ||eta' O||_F = eta sqrt(n)."""
    n, m = 16, 40
    W, M, G = _step_inputs(n, m, seed=6)
    eta = 0.01
    cubic = [(1.5, -0.5, 0.0)] * 60
    for f_num, f_den in [(1, 1), (1, 4), (1, 2)]:
        W1, _, S, O = oracle.dion3_step(W, M, G, f_num, f_den, mu=0.9, eta=eta, abc=cubic)
        dW = W1 - W.astype(np.float64)
        assert abs(np.linalg.norm(dW) - eta * math.sqrt(n)) <= 1e-9


def test_weight_decay_uses_eta_prime(jordan):
    n, m = 8, 16
    W, M, G = _step_inputs(n, m, seed=8)
    wd = 0.1
    W1, _, S, _ = oracle.dion3_step(W, M, G, 1, 4, mu=0.9, eta=0.01, wd=wd, abc=[jordan] * 5)
    sel = np.zeros(n, bool)
    sel[S] = True
    np.testing.assert_allclose(W1[~sel], W[~sel].astype(np.float64) * (1 - 0.02 * wd), rtol=0, atol=0)


@pytest.mark.parametrize("f", [(1, 4), (3, 8)])
def test_given_rows_follow_error_feedback(f, jordan):
    """A caller-chosen S ('limitations': random selection): M[S] = fl32(mu (M+G)), the other rows
    are M+G bit for bit, W changes only on S, and the update on S is eta' times the polar factor
    of M[S] (checked against an SVD with the classic cubic run to convergence)."""
    n, m = 20, 48
    W, M, G = _step_inputs(n, m, seed=11)
    k = oracle.ceil_k(n, *f)
    rows = np.random.default_rng(5).choice(n, size=k, replace=False)
    mu, eta = 0.9, 0.01
    cubic = [(1.5, -0.5, 0.0)] * 60
    W1, M1, S, O = oracle.dion3_step(W, M, G, *f, mu=mu, eta=eta, abc=cubic, rows=rows)
    assert list(S) == sorted(rows.tolist())
    summed = M + G
    sel = np.zeros(n, bool)
    sel[S] = True
    assert np.array_equal(M1[~sel].view(np.uint32), summed[~sel].view(np.uint32))
    assert np.array_equal(M1[sel].view(np.uint32), (np.float32(mu) * summed)[sel].view(np.uint32))
    assert np.array_equal(W1[~sel], W[~sel].astype(np.float64))
    U, _, Vt = np.linalg.svd(summed[S].astype(np.float64), full_matrices=False)
    eta_p = eta * math.sqrt(f[1] / f[0])
    np.testing.assert_allclose(W1[S] - W[S].astype(np.float64), -eta_p * (U @ Vt), rtol=0, atol=1e-10)


def test_given_rows_equal_to_topk_reproduce_default(jordan):
    n, m = 24, 40
    W, M, G = _step_inputs(n, m, seed=12)
    a = oracle.dion3_step(W, M, G, 1, 4, mu=0.95, eta=0.01, abc=[jordan] * 5, restart_after=(2,))
    b = oracle.dion3_step(W, M, G, 1, 4, mu=0.95, eta=0.01, abc=[jordan] * 5, restart_after=(2,),
                          rows=a[2][::-1].copy())
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("rows", [[0, 0, 1, 2, 3, 4], [0, 1, 2, 3, 4, 24], [0, 1, 2], [-1, 1, 2, 3, 4, 5]])
def test_given_rows_validated(rows, jordan):
    W, M, G = _step_inputs(24, 40, seed=13)
    with pytest.raises(ValueError):
        oracle.dion3_step(W, M, G, 1, 4, mu=0.95, eta=0.01, abc=[jordan] * 5, rows=rows)


def test_column_step_error_feedback_and_polar(jordan):
    """Column selection on a matrix stored m x n: the k columns of largest exact l1 norm (checked
    with exact fractions), M[:, S] = fl32(mu (M+G)), other columns M+G bit for bit, W changes only
    on S, by eta' times the SVD polar factor of M[:, S] (cubic iteration run to convergence)."""
    m, n = 30, 12
    rng = np.random.default_rng(21)
    W = (rng.standard_normal((m, n)) * 0.02).astype(np.float32)
    M = (rng.standard_normal((m, n)) * 0.05).astype(np.float32)
    G = rng.standard_normal((m, n)).astype(np.float32)
    G = (G.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
    mu, eta, f = 0.9, 0.01, (1, 3)
    cubic = [(1.5, -0.5, 0.0)] * 60
    W1, M1, S, _ = oracle.dion3_step_cols(W, M, G, *f, mu=mu, eta=eta, abc=cubic)
    summed = M + G
    keys = [sum(Fraction(float(abs(x))) for x in summed[:, j]) for j in range(n)]
    k = oracle.ceil_k(n, *f)
    order = sorted(range(n), key=lambda j: (-keys[j], j))
    assert list(S) == sorted(order[:k])
    sel = np.zeros(n, bool)
    sel[S] = True
    assert np.array_equal(M1[:, ~sel].view(np.uint32), summed[:, ~sel].view(np.uint32))
    assert np.array_equal(M1[:, sel].view(np.uint32), (np.float32(mu) * summed)[:, sel].view(np.uint32))
    assert np.array_equal(W1[:, ~sel], W[:, ~sel].astype(np.float64))
    U, _, Vt = np.linalg.svd(summed[:, S].T.astype(np.float64), full_matrices=False)
    eta_p = eta * math.sqrt(f[1] / f[0])
    np.testing.assert_allclose((W1 - W.astype(np.float64))[:, S], (-eta_p * (U @ Vt)).T, rtol=0, atol=1e-10)


def test_column_step_given_columns(jordan):
    m, n = 20, 8
    rng = np.random.default_rng(22)
    W = (rng.standard_normal((m, n)) * 0.02).astype(np.float32)
    M = np.zeros((m, n), np.float32)
    G = rng.standard_normal((m, n)).astype(np.float32)
    W1, M1, S, _ = oracle.dion3_step_cols(W, M, G, 1, 4, mu=0.95, eta=0.01, abc=[jordan] * 5, cols=[6, 1])
    assert list(S) == [1, 6]
    assert np.array_equal(W1[:, [0, 2, 3, 4, 5, 7]], W[:, [0, 2, 3, 4, 5, 7]].astype(np.float64))
