"""Pins for the oracle's Newton-Schulz functions against SVD, closed forms and the pages' values.

Each test checks the oracle against something other than itself:
numpy's SVD, the scalar polynomial written out here, the exact polar
factor U V^T, Theorem 2's equivalence, and numbers printed on the pages
(tests/golden/pages_values.json).
"""

import numpy as np
import pytest

import oracle


def _rand(n, m, seed):
    return np.random.default_rng(seed).standard_normal((n, m))


def _with_singular_values(n, m, sig, seed):
    rng = np.random.default_rng(seed)
    U, _ = np.linalg.qr(rng.standard_normal((n, n)))
    V, _ = np.linalg.qr(rng.standard_normal((m, n)))
    return (U * np.asarray(sig)) @ V.T, U, V


def _quintic_chain(x, abc):
    # p(x) = a x + b x^3 + c x^5, applied T times (written out here, not taken from the oracle)
    for a, b, c in abc:
        x = a * x + b * x ** 3 + c * x ** 5
    return x


@pytest.mark.parametrize("shape", [(5, 8), (8, 5), (3, 3), (1, 7), (6, 20)])
def test_ns_standard_acts_on_singular_values(shape, jordan):
    """Muon blog, 'Doing an SVD without an SVD': the odd polynomial maps each sigma_i and keeps U, V."""
    n, m = shape
    X = _rand(n, m, seed=11 * n + m)
    abc = [jordan] * 5
    eps = 1e-7
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    expect = (U * _quintic_chain(s / (np.linalg.norm(X) + eps), abc)) @ Vt
    got = oracle.ns_standard(X, abc, eps)
    assert got.shape == X.shape
    assert np.max(np.abs(got - expect)) <= 1e-12 * max(1.0, np.max(np.abs(expect)))


def test_ns_standard_per_iteration_coefficients():
    """Different (a,b,c) per iteration are applied in order (p_T o ... o p_1)."""
    X = _rand(4, 9, seed=3)
    abc = [(1.9, -1.1, 0.2), (1.5, -0.5, 0.0), (2.0, -1.5, 0.5)]
    U, s, Vt = np.linalg.svd(X, full_matrices=False)
    expect = (U * _quintic_chain(s / (np.linalg.norm(X) + 1e-7), abc)) @ Vt
    got = oracle.ns_standard(X, abc)
    np.testing.assert_allclose(got, expect, rtol=0, atol=1e-12)
    # the reversed order gives a different map, so order is really pinned
    assert np.max(np.abs(oracle.ns_standard(X, abc[::-1]) - expect)) > 1e-4


@pytest.mark.parametrize("shape", [(6, 6), (4, 11), (11, 4)])
def test_cubic_iteration_reaches_polar_factor(shape):
    """Dion3 summary, prerequisite 'polar decomposition': polar(X) = U V^T."""
    n, m = shape
    r = min(n, m)
    sig = np.linspace(0.5, 1.0, r)
    if n <= m:
        X, U, V = _with_singular_values(n, m, sig, seed=5)
        polar = U @ V.T
    else:
        Xt, U, V = _with_singular_values(m, n, sig, seed=5)
        X = Xt.T
        polar = (U @ V.T).T
    got = oracle.ns_standard(X, [(1.5, -0.5, 0.0)] * 60)
    np.testing.assert_allclose(got, polar, rtol=0, atol=1e-10)


def test_jordan_band_matches_printed_band(jordan, pages):
    """Muon blog: with the tuned triple the output singular values sit roughly in [0.7, 1.3]."""
    lo, hi = pages["output_singular_band"]["value"]
    n, m = 48, 96
    rest = np.logspace(-2, np.log10(0.12), n - 1)          # normalized sigma in [0.01, 0.12]
    s = np.concatenate([[np.sqrt(1.0 - np.sum(rest ** 2))], rest])   # ||s|| = 1, top value ~0.86
    X, U, V = _with_singular_values(n, m, s, seed=7)
    out = oracle.ns_standard(X, [jordan] * 5, eps=0.0)
    sv = np.linalg.svd(out, compute_uv=False)
    assert sv.min() >= lo - 0.05 and sv.max() <= hi


@pytest.mark.parametrize("n,alpha_num,alpha_den", [(4, 1, 1), (4, 4, 1), (64, 43, 16), (64, 4, 1), (16, 64, 3), (256, 1, 1), (96, 64, 3)])
@pytest.mark.parametrize("restarts", [(), (2,), (2, 4), (1, 2, 3, 4)])
def test_gram_ns_equals_standard(n, alpha_num, alpha_den, restarts, jordan):
    """Theorem 2 + Algorithm 3: Gram NS (with any restart schedule) equals standard NS."""
    m = n * alpha_num // alpha_den
    X = _rand(n, m, seed=1000 + n + m + len(restarts))
    abc = [jordan] * 5
    std = oracle.ns_standard(X, abc)
    gram = oracle.gram_ns(X, abc, restarts)
    err = np.linalg.norm(gram - std) / np.linalg.norm(std)
    assert err <= 1e-10


def test_theorem2_scalar_recurrence_equals_composite(jordan):
    """Theorem 2: (p_T o ... o p_1)(x) = q_T x, with and without restarts."""
    x = np.linspace(0.0, 1.0, 2001)
    abc = [jordan] * 5
    expect = _quintic_chain(x.copy(), abc)
    for rs in [(), (2,), (2, 4), (1, 3)]:
        got = oracle.theorem2_scalar(x, abc, rs)
        np.testing.assert_allclose(got, expect, rtol=1e-12, atol=1e-14)


def test_gram_ns_singular_values_follow_theorem2(jordan):
    """The matrix output's singular values equal the scalar recurrence on sigma / ||X||_F."""
    X = _rand(6, 15, seed=21)
    abc = [jordan] * 5
    s = np.linalg.svd(X, compute_uv=False)
    expect = np.sort(_quintic_chain(s / (np.linalg.norm(X) + 1e-7), abc))
    got = np.sort(np.linalg.svd(oracle.gram_ns(X, abc, (2,)), compute_uv=False))
    np.testing.assert_allclose(got, expect, rtol=1e-11)


def test_negative_eigenvalue_diverges_and_restart_cures_it(jordan, pages):
    """Dion3 summary, 'half precision and numerical stability': a spurious eigenvalue of R as low
    as -4e-4 makes the inverse-square-root iteration diverge; the restart removes it."""
    lam = pages["spurious_negative_eigenvalue"]["value"]
    abc = [jordan] * pages["ns_steps"]["value"]
    restart_after = pages["restart_iteration"]["value"] - 1
    # scalar recurrence from r0 = lam: |r| explodes
    r = lam
    for a, b, c in abc:
        z = a + b * r + c * r * r
        r = r * z * z
    assert r < -1e8
    # matrix: one tiny singular direction whose Gram eigenvalue is pushed to lam
    n, m = 8, 32
    sig = np.concatenate([np.linspace(1.0, 0.2, n - 1), [1e-3]])
    X, U, V = _with_singular_values(n, m, sig, seed=9)
    Xn = X / (np.linalg.norm(X) + 1e-7)
    u = U[:, -1]
    s_min2 = (1e-3 / (np.linalg.norm(X) + 1e-7)) ** 2
    E = -(s_min2 - lam) * np.outer(u, u)          # eigenvalue of R0 + E along u becomes lam
    assert abs(np.linalg.eigvalsh(Xn @ Xn.T + E).min() - lam) < 1e-12
    bad = oracle.gram_ns(X, abc, (), r0_add=E)
    good_trace = []
    good = oracle.gram_ns(X, abc, (restart_after,), r0_add=E, trace=good_trace)
    assert np.linalg.svd(bad, compute_uv=False).max() > 1e2
    sv = np.linalg.svd(good, compute_uv=False)
    assert sv.max() < 1.5
    # after the restart R is rebuilt as X X^T: positive semidefinite again
    R_after = [R for (t, R, Q) in good_trace if t == restart_after][0]
    assert np.linalg.eigvalsh(R_after).min() > -1e-12


def test_restart_schedule_validation(jordan):
    X = _rand(3, 5, 0)
    for bad in [(0,), (5,), (3, 2), (2, 2)]:
        with pytest.raises(ValueError):
            oracle.gram_ns(X, [jordan] * 5, bad)
    with pytest.raises(ValueError):
        oracle.gram_ns(_rand(5, 3, 0), [jordan] * 5)


def test_odd_poly_matches_library_polynomial_evaluation(jordan):
    """Muon blog, 'Doing an SVD without an SVD': each step applies the odd quintic
    p(x) = a x + b x^3 + c x^5 to the singular values.  numpy's polynomial evaluator, given the
    coefficient vector (0, a, 0, b, 0, c), is the independent definition."""
    x = np.linspace(-1.5, 1.5, 601)
    for a, b, c in [jordan, (1.5, -0.5, 0.0), (2.0, -1.5, 0.5)]:
        ref = np.polynomial.polynomial.polyval(x, [0.0, a, 0.0, b, 0.0, c])
        np.testing.assert_allclose(oracle.odd_poly(x, a, b, c), ref, rtol=1e-13, atol=1e-14)
        # odd: p(-x) = -p(x), and p(0) = 0
        xp = np.linspace(0.0, 1.5, 301)
        np.testing.assert_allclose(oracle.odd_poly(-xp, a, b, c), -oracle.odd_poly(xp, a, b, c), rtol=1e-14, atol=0)
        assert oracle.odd_poly(0.0, a, b, c) == 0.0


def test_composite_scalar_is_the_iterated_polynomial_and_the_svd_map(jordan):
    """(p_T o ... o p_1) in the order given: against the library evaluator applied T times, and
    against the singular values that numpy's SVD finds in the oracle's standard NS output."""
    abc = [(1.9, -1.1, 0.2), jordan, (1.5, -0.5, 0.0)]
    x = np.linspace(0.0, 1.0, 1001)
    ref = x.copy()
    for a, b, c in abc:
        ref = np.polynomial.polynomial.polyval(ref, [0.0, a, 0.0, b, 0.0, c])
    np.testing.assert_allclose(oracle.composite_scalar(x, abc), ref, rtol=1e-12, atol=1e-14)
    # the order matters: reversing the table gives a different map
    assert np.max(np.abs(oracle.composite_scalar(x, abc[::-1]) - ref)) > 1e-3
    # a matrix with known singular values: SVD of the standard-NS output
    sig = np.array([0.9, 0.5, 0.3, 0.1, 0.02])
    X, _, _ = _with_singular_values(5, 12, sig, seed=31)
    got = np.sort(np.linalg.svd(oracle.ns_standard(X, abc, eps=0.0), compute_uv=False))
    expect = np.sort(oracle.composite_scalar(sig / np.linalg.norm(sig), abc))
    np.testing.assert_allclose(got, expect, rtol=1e-11)


def test_composite_scalar_cubic_converges_to_sign():
    """Dion3 summary, prerequisite 'polar decomposition': iterating the cubic
    (1.5, -0.5, 0) drives every x in (0, sqrt(3)) to 1 (and -x to -1): the scalar polar factor."""
    x = np.concatenate([np.linspace(0.05, 1.7, 200), -np.linspace(0.05, 1.7, 200)])
    np.testing.assert_allclose(oracle.composite_scalar(x, [(1.5, -0.5, 0.0)] * 80), np.sign(x), rtol=0, atol=1e-12)
