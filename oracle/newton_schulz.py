"""Standard and Gram Newton-Schulz in float64 (oracle; test infrastructure only).

Sources (page title, section):

* Dion3 paper summary, prerequisite "Newton-Schulz iteration": one step is
  X <- a_t X + b_t (X X^T) X + c_t (X X^T)^2 X, usually T = 5 steps.
* "Muon: Orthogonalized Momentum ...", section "Doing an SVD without an
  SVD": X is divided by (||X||_F + eps) first; the iteration runs on the
  short side (transpose when rows > columns); the odd polynomial acts on each
  singular value as x -> a x + b x^3 + c x^5 and leaves U, V alone.
* Dion3 paper summary, section "core method", Theorem 2: write each odd p_t
  as p_t(x) = x h_t(x^2) with h_t(r) = a_t + b_t r + c_t r^2.  With
  r_0 = x^2, q_0 = 1, z_t = h_t(r_{t-1}), r_t = r_{t-1} z_t^2,
  q_t = q_{t-1} z_t, the composite is (p_T o ... o p_1)(x) = q_T x.  Lifted
  to matrices: R_0 = X X^T, Q_0 = I, Z_t = h_t(R_{t-1}), R_t = Z_t R_{t-1} Z_t,
  Q_t = Q_{t-1} Z_t, output Q_T X.
* Dion3 paper summary, section "method details", Algorithm 3 (stabilised
  Gram Newton-Schulz): prescale by the Frobenius norm; restart "at t = 3",
  read here as: after iteration 2 completes, X <- Q_2 X, R <- X X^T,
  Q <- I; output Q_T X.  (The garbled "R_t = Z_t R_{t-1} Z_t + a_t(.)" on
  that page is read as Theorem 2's R_t = Z_t R_{t-1} Z_t, with
  Z_t = a_t I + b_t R + c_t R^2 -- the page's "Z = bR + cR^2, Q = QZ + aQ"
  is the same Z split as a_t I + (b_t R + c_t R^2).)
* Dion3 paper summary, table "structured data" and "limitations": FLOP
  costs 2T(2a+1)n^3 (plain standard NS), T(3a+1)n^3 (standard NS on
  symmetric kernels), (4T+3a-3)n^3 (Gram NS), +3(a-1)n^3 per restart.

The FLOP counter charges each product the way those formulas do: a product
whose output is symmetric costs n^2 k on symmetric kernels (2 n^2 k plain);
a general product costs 2 m n k.  Work that is mathematically dead is not
executed: the product with Q = I (Q <- Z instead), the R update after the
last iteration, and the R update that a restart overwrites.  Skipping it
changes no value.
"""

from __future__ import annotations

import numpy as np


class FlopCounter:
    """Accumulates matrix-product FLOPs as the pages' cost formulas count them."""

    def __init__(self, symmetric_kernels: bool):
        self.symmetric_kernels = bool(symmetric_kernels)
        self.flops = 0

    def gram(self, n: int, k: int) -> None:
        """X X^T for X of n x k (symmetric n x n output)."""
        self.flops += n * n * k if self.symmetric_kernels else 2 * n * n * k

    def sym_product(self, n: int) -> None:
        """n x n times n x n whose result is symmetric (R^2, Q Z, R Z, (RZ) Z)."""
        self.flops += n ** 3 if self.symmetric_kernels else 2 * n ** 3

    def general(self, m: int, n: int, k: int) -> None:
        """(m x k) times (k x n), no symmetry in the output."""
        self.flops += 2 * m * n * k


def _as_triples(abc):
    trip = [tuple(float(v) for v in t) for t in abc]
    for t in trip:
        if len(t) != 3:
            raise ValueError("each iteration needs one (a, b, c) triple")
    if not trip:
        raise ValueError("need at least one iteration")
    return trip


def _frobenius_prescale(X: np.ndarray, eps: float) -> np.ndarray:
    return X / (np.linalg.norm(X) + eps)


def ns_standard(X, abc, eps: float = 1e-7, counter: FlopCounter | None = None) -> np.ndarray:
    """Standard Newton-Schulz: T quintic steps on the short-side orientation.

    ``abc`` is a sequence of T triples (a_t, b_t, c_t).
    """
    trip = _as_triples(abc)
    X = _frobenius_prescale(np.asarray(X, dtype=np.float64), eps)
    transposed = X.shape[0] > X.shape[1]
    if transposed:
        X = X.T
    n, m = X.shape
    for a, b, c in trip:
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
        if counter is not None:
            counter.gram(n, m)
            counter.sym_product(n)
            counter.general(n, m, n)
    return X.T if transposed else X


def _check_restarts(restart_after, T):
    rs = [int(r) for r in restart_after]
    for i, r in enumerate(rs):
        if not 1 <= r <= T - 1:
            raise ValueError("restart positions must lie in [1, T-1]")
        if i and r <= rs[i - 1]:
            raise ValueError("restart positions must be strictly increasing")
    return set(rs)


def gram_ns(X, abc, restart_after=(), eps: float = 1e-7, counter: FlopCounter | None = None,
            r0_add=None, trace=None) -> np.ndarray:
    """Gram Newton-Schulz (Theorem 2 lifted to matrices) with restarts (Algorithm 3).

    ``X`` is n x m with n <= m.  ``restart_after`` lists the iterations t
    after which X <- Q_t X, R <- X X^T, Q <- I.  ``r0_add`` (n x n) is added
    to R_0 -- it stands for the rounding error a half-precision X X^T carries
    (the spurious negative eigenvalues of the "half precision and numerical
    stability" prerequisite); ``trace`` (a list) receives (t, R, Q) after each
    iteration.  Both are for the restart-stability pins only.
    """
    trip = _as_triples(abc)
    T = len(trip)
    restarts = _check_restarts(restart_after, T)
    X = _frobenius_prescale(np.asarray(X, dtype=np.float64), eps)
    n, m = X.shape
    if n > m:
        raise ValueError("gram_ns expects the short side first (n <= m)")
    I = np.eye(n)
    R = X @ X.T
    if counter is not None:
        counter.gram(n, m)
    if r0_add is not None:
        R = R + np.asarray(r0_add, dtype=np.float64)
    Q = None  # None stands for the identity
    for t, (a, b, c) in enumerate(trip, start=1):
        Z = a * I + b * R + c * (R @ R)
        if counter is not None:
            counter.sym_product(n)
        if Q is None:
            Q = Z
        else:
            Q = Q @ Z
            if counter is not None:
                counter.sym_product(n)
        if t in restarts:
            X = Q @ X
            R = X @ X.T
            Q = None
            if counter is not None:
                counter.general(n, m, n)
                counter.gram(n, m)
        elif t < T:
            R = Z @ R @ Z
            if counter is not None:
                counter.sym_product(n)
                counter.sym_product(n)
        if trace is not None:
            trace.append((t, R.copy(), None if Q is None else Q.copy()))
    out = Q @ X
    if counter is not None:
        counter.general(n, m, n)
    return out


def odd_poly(x, a, b, c):
    """The scalar quintic p(x) = a x + b x^3 + c x^5."""
    return a * x + b * x ** 3 + c * x ** 5


def composite_scalar(x, abc):
    """(p_T o ... o p_1)(x) applied elementwise."""
    y = np.asarray(x, dtype=np.float64)
    for a, b, c in _as_triples(abc):
        y = odd_poly(y, a, b, c)
    return y


def theorem2_scalar(x, abc, restart_after=()):
    """Theorem 2's scalar recurrence, with the same restarts as ``gram_ns``.

    r_0 = x^2, q_0 = 1; z_t = a_t + b_t r + c_t r^2; r <- r z_t^2; q <- q z_t;
    a restart after t sets x <- q x, r <- x^2, q <- 1.  Returns q_T x.
    """
    trip = _as_triples(abc)
    restarts = _check_restarts(restart_after, len(trip))
    x = np.asarray(x, dtype=np.float64)
    r = x * x
    q = np.ones_like(x)
    for t, (a, b, c) in enumerate(trip, start=1):
        z = a + b * r + c * r * r
        r = r * z * z
        q = q * z
        if t in restarts:
            x = q * x
            r = x * x
            q = np.ones_like(x)
    return q * x


def flop_count(n: int, m: int, T: int, restart_after=(), variant: str = "gram", seed: int = 0) -> int:
    """FLOPs the oracle executes on a seeded n x m input.

    variant: "gram" (Gram NS on symmetric kernels), "standard_sym" (standard
    NS on symmetric kernels) or "standard" (standard NS, plain GEMMs).  The
    coefficients do not affect the count, so a fixed triple is used.
    """
    X = np.random.default_rng(seed).standard_normal((n, m))
    abc = [(1.5, -0.5, 0.0)] * T
    if variant == "gram":
        ctr = FlopCounter(symmetric_kernels=True)
        gram_ns(X, abc, restart_after, counter=ctr)
    elif variant in ("standard_sym", "standard"):
        if restart_after:
            raise ValueError("standard NS has no restarts")
        ctr = FlopCounter(symmetric_kernels=(variant == "standard_sym"))
        ns_standard(X, abc, counter=ctr)
    else:
        raise ValueError(variant)
    return ctr.flops
