"""The oracle's executed-FLOP counts against the pages' closed forms and printed savings."""

from fractions import Fraction

import pytest

import oracle


def _gram_formula(n, m, T, r):
    # (4T + 3a - 3) n^3 + r * 3 (a - 1) n^3 with a = m / n, in exact integers
    return (4 * T - 3) * n ** 3 + 3 * m * n * n + r * 3 * (m * n * n - n ** 3)


@pytest.mark.parametrize("n,m", [(8, 8), (8, 32), (16, 43), (12, 256), (96, 2048)])
@pytest.mark.parametrize("T", [1, 3, 5])
def test_standard_counts(n, m, T):
    assert oracle.flop_count(n, m, T, variant="standard") == 2 * T * (2 * m * n * n + n ** 3)   # 2T(2a+1)n^3
    assert oracle.flop_count(n, m, T, variant="standard_sym") == T * (3 * m * n * n + n ** 3)  # T(3a+1)n^3


@pytest.mark.parametrize("n,m", [(8, 8), (8, 32), (16, 43), (12, 256), (96, 2048)])
@pytest.mark.parametrize("T,restarts", [(1, ()), (5, ()), (5, (2,)), (5, (2, 4)), (6, (1, 3, 5))])
def test_gram_counts(n, m, T, restarts):
    assert oracle.flop_count(n, m, T, restarts, variant="gram") == _gram_formula(n, m, T, len(restarts))


def test_printed_savings(pages):
    ex = pages["flop_example"]
    T, a = ex["T"], ex["alpha"]
    n = 8
    m = a * n
    gram = oracle.flop_count(n, m, T, variant="gram")
    sym = oracle.flop_count(n, m, T, variant="standard_sym")
    plain = oracle.flop_count(n, m, T, variant="standard")
    save_sym = 1 - Fraction(gram, sym)
    save_plain = 1 - Fraction(gram, plain)
    assert save_sym == 1 - Fraction(29, 65)
    assert save_plain == 1 - Fraction(29, 90)
    assert round(float(save_sym), 2) == ex["saving_vs_symmetric_standard"]
    assert round(float(save_plain), 2) == ex["saving_vs_plain_standard"]
    # the plain count is the table's (20a + 10) n^3 at T = 5
    assert plain == (20 * a + 10) * n ** 3


def test_square_matrices_gain_nothing():
    # montaan summary: at alpha = 1 standard NS on symmetric kernels and Gram NS cost the same
    n = 16
    assert oracle.flop_count(n, n, 5, variant="gram") == oracle.flop_count(n, n, 5, variant="standard_sym")
