"""Plain float64 CPU oracle for the Dion3 / Gram Newton-Schulz hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
link this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``matrix_orthogonalizing_optimizer_syrk_gb300``)
and imports nothing from it; the only module both sides use is the seeded
input generator package ``synthetic``, which holds none of the method's
arithmetic.

Every function follows a passage of the pages it restates, cited as
"<page title>, <section / equation / table>":

* Dion3 paper summary (paper.rainbus.top, "Dion3: Full-Stack Orthogonal
  Updates"), prerequisites "Newton-Schulz iteration", "polar decomposition",
  "spectral-norm steepest descent", "half precision and numerical
  stability", "error feedback"; section "core method" (Theorem 2);
  section "method details" (Algorithm 3 = stabilised Gram Newton-Schulz,
  Algorithm 4 = the Dion3 update rule); table "structured data"
  (FLOP formulas); "limitations" (restart cost).
* "Muon: Orthogonalized Momentum and Why It Trains LLMs 2x Cheaper",
  section "Doing an SVD without an SVD" (odd polynomial acting on singular
  values, Frobenius prescale with eps, short-side orientation).

Parity status: every public function here is pinned by ``-m "not gpu"``
tests against closed forms, SVD, brute force or the pages' printed values
(see tests/test_oracle_*.py).  No function is "parity unpinned".
"""

from .newton_schulz import (
    FlopCounter,
    composite_scalar,
    flop_count,
    gram_ns,
    ns_standard,
    odd_poly,
    theorem2_scalar,
)
from .dion3 import ceil_k, dion3_step, dion3_step_cols, exact_row_keys, top_k_rows
from .sym_gemm import sym_gemm

__all__ = [
    "FlopCounter",
    "ceil_k",
    "composite_scalar",
    "dion3_step",
    "dion3_step_cols",
    "exact_row_keys",
    "flop_count",
    "gram_ns",
    "ns_standard",
    "odd_poly",
    "sym_gemm",
    "theorem2_scalar",
    "top_k_rows",
]
