"""The Dion3 update rule (Algorithm 4) with error feedback (oracle; test infrastructure only).

Sources (page title, section):

* Dion3 paper summary, section "method details", Algorithm 4:
  M <- M + G; S = indices of the k = ceil(f n) rows of largest l1 norm;
  O = GramNS(M[S, :]); optional NorMuon (not built); W <- (1 - eta wd) W;
  W[S, :] <- W[S, :] - eta O; M[S, :] <- mu M[S, :].
* Same page, prerequisite "error feedback": M <- mu M_hat + (M - M_hat) --
  only the selected rows decay, unselected rows keep accumulating G.
* Same page, prerequisite "spectral-norm steepest descent": the learning
  rate transfers as eta' = eta / sqrt(f), keeping ||eta' O||_F = eta sqrt(n).
  The step takes the Muon-equivalent eta and applies eta' itself; the weight
  decay factor uses eta' as well.
* Same page, "existing work": k = ceil(f n), rows taken as they are.
* "Dion3" summary (m.montaan.com), update-rule paragraph: f is the fraction of rows (or columns)
  selected.  ``dion3_step_cols`` takes a matrix stored m x n with the short side n as its
  columns and selects columns: by definition the row step applied to the transpose.
* Same page, "limitations" and "future directions": choosing S at random
  works about as well as the l1 rule, and a set S that does not depend on M
  is what lets a data-parallel run synchronise only M[S, :].  ``rows``
  passes such a caller-chosen S (e.g. drawn at random by the caller); the
  step is otherwise unchanged.

Readings where the pages are silent:

* Keys.  key_i is the exact real l1 norm (norm_p = 1) or the exact real
  sum of squares (norm_p = 2, same order as the row L2 norm) of row i of the
  stored fp32 momentum.  Every fp32 value x is an integer multiple of 2^-149
  and x^2 one of 2^-298, so the keys are computed exactly as Python integers
  (key * 2^149, resp. key * 2^298) -- no rounding anywhere.
* Order.  Larger key first; equal keys go to the lower row index.  S is
  returned sorted ascending (polar is permutation-equivariant, so the
  order of the rows of M[S, :] changes nothing but determinism).
* State precision.  M and W are fp32, G is 16-bit.  M is rounded to fp32
  exactly where a device stores it: after + G and after * mu (mu taken at
  its fp32 value).  float64 has more than 2*24+2 bits, so rounding the
  float64 result once more to fp32 equals one correctly rounded fp32
  operation.  W is returned in float64 (only its update is compared).
"""

from __future__ import annotations

import math

import numpy as np

from .newton_schulz import gram_ns

_TWO_149 = 2.0 ** 149
_TWO_298 = 2.0 ** 298


def ceil_k(n: int, f_num: int, f_den: int) -> int:
    """k = ceil(n f) for a rational f = f_num / f_den, in exact integers."""
    if f_num <= 0 or f_den <= 0 or f_num > f_den:
        raise ValueError("need 0 < f <= 1")
    return -((-n * f_num) // f_den)


def exact_row_keys(M32, norm_p: int = 1):
    """Exact per-row keys of an fp32 matrix, as Python ints.

    norm_p = 1: sum_j |x_ij| * 2^149.   norm_p = 2: sum_j x_ij^2 * 2^298.
    Each term is an exact integer held exactly by a float64 (a power-of-two
    scaling of an fp32 value or of its exact float64 square), converted with
    int() and summed in Python's unbounded integers.
    """
    M32 = np.asarray(M32)
    if M32.dtype != np.float32:
        raise TypeError("keys are defined on the stored fp32 values")
    if not np.all(np.isfinite(M32)):
        raise ValueError("non-finite momentum")
    x = np.abs(M32.astype(np.float64))
    if norm_p == 1:
        scaled = x * _TWO_149
    elif norm_p == 2:
        scaled = (x * x) * _TWO_298
    else:
        raise ValueError("norm_p must be 1 or 2")
    return [sum(int(v) for v in row.tolist()) for row in scaled]


def top_k_rows(keys, k: int) -> np.ndarray:
    """Indices of the k largest keys (ties -> lower index), sorted ascending."""
    order = sorted(range(len(keys)), key=lambda i: (-keys[i], i))
    return np.array(sorted(order[:k]), dtype=np.int64)


def given_rows(rows, n: int, k: int) -> np.ndarray:
    """A caller-chosen S: k distinct row indices in [0, n), returned sorted ascending."""
    S = np.asarray(rows, dtype=np.int64).reshape(-1)
    if S.size != k or np.unique(S).size != k or (k and (S.min() < 0 or S.max() >= n)):
        raise ValueError("rows must be k distinct indices in [0, n)")
    return np.sort(S)


def dion3_step(W, M, G, f_num: int, f_den: int, mu: float, eta: float, wd: float = 0.0,
               norm_p: int = 1, abc=None, restart_after=(), eps: float = 1e-7, rows=None):
    """One Dion3 step on one n x m matrix (n <= m).

    ``rows``: optional caller-chosen S (k distinct indices); then no keys are computed.
    Returns (W_new float64, M_new fp32, S int64 ascending, O float64 k x m).
    """
    M = np.asarray(M, dtype=np.float32)
    n, m = M.shape
    if n > m:
        raise ValueError("orient the matrix so that n <= m")
    M1 = (M.astype(np.float64) + np.asarray(G, dtype=np.float64)).astype(np.float32)
    k = ceil_k(n, f_num, f_den)
    if rows is None:
        S = top_k_rows(exact_row_keys(M1, norm_p), k)
    else:
        S = given_rows(rows, n, k)
    O = gram_ns(M1[S].astype(np.float64), abc, restart_after, eps)
    eta_p = eta * math.sqrt(f_den / f_num)
    W1 = np.asarray(W, dtype=np.float64) * (1.0 - eta_p * wd)
    W1[S] -= eta_p * O
    M2 = M1.copy()
    mu32 = np.float64(np.float32(mu))
    M2[S] = (mu32 * M1[S].astype(np.float64)).astype(np.float32)
    return W1, M2, S, O


def dion3_step_cols(W, M, G, f_num: int, f_den: int, mu: float, eta: float, wd: float = 0.0,
                    norm_p: int = 1, abc=None, restart_after=(), eps: float = 1e-7, cols=None):
    """One Dion3 step on a matrix stored m x n (n <= m) that selects columns.

    ``cols``: optional caller-chosen column set.  Returns (W_new float64 m x n, M_new fp32 m x n,
    S int64 ascending column indices, O float64 k x m).  The row step of the transposed matrix,
    transposed back.
    """
    W = np.asarray(W)
    M = np.asarray(M, dtype=np.float32)
    G = np.asarray(G)
    W1t, M1t, S, O = dion3_step(W.T, M.T, G.T, f_num, f_den, mu=mu, eta=eta, wd=wd, norm_p=norm_p, abc=abc,
                                restart_after=restart_after, eps=eps, rows=cols)
    return W1t.T, np.ascontiguousarray(M1t.T), S, O

