"""The range-checked build (libdion3_checked.so) on a GPU, in a child process.

The checked build compiles the same kernels with in-kernel index checks that set DION3_DEV_RANGE
in the status word (the library's stand-in for a memory checker, which is not available on the
GPUs it is tested on).  On valid inputs it must produce bit-identical results to the default
build and leave the status word at 0; an out-of-range row in a carried-decay list (device data
the host cannot check) must set DION3_DEV_RANGE in the checked build only, while both builds skip
the row.
"""

import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import synthetic
if {checked!r}:
    d3.use_checked_build()
assert d3.lib().dion3_range_checks() == int({checked!r})
dev = "cuda"
ABC = [(3.4445, -4.7750, 2.0315)] * 5
out = {{}}
status = torch.zeros(1, dtype=torch.int32, device=dev)
# symmetric GEMM (pair tiles and a ragged single-tile product), Gram NS (separate products and
# fused segments), standard NS
A = synthetic.gaussian((2, 700, 320), seed=1, std=320 ** -0.5, dtype=torch.bfloat16, device=dev)
out["sym"] = d3.sym_gemm(A, status=status).float()
X = synthetic.lowrank_batch(3, 200, 640, base_seed=2, dtype=torch.bfloat16, device=dev)
out["gram"] = d3.gram_ns(X, ABC, (2, 4), status=status).float()
Xs = synthetic.lowrank_batch(4, 96, 500, base_seed=3, dtype=torch.bfloat16, device=dev)
out["gram_small"] = d3.gram_ns(Xs, ABC, (2,), status=status).float()
Xq = synthetic.lowrank_batch(2, 256, 256, base_seed=4, dtype=torch.bfloat16, device=dev)
out["ns"] = d3.ns_standard(Xq, ABC, status=status).float()
# two carried Dion3 steps (top-k rows), then the pending decay applied
n, m = 160, 512
W = synthetic.gaussian((3, n, m), seed=5, std=0.02, device=dev)
M = torch.zeros((3, n, m), device=dev)
sel = torch.empty((3, 40), dtype=torch.int32, device=dev)
for s in range(2):
    G = synthetic.lowrank_batch(3, n, m, base_seed=10 + s, dtype=torch.bfloat16, device=dev)
    d3.step(W, M, G, f=(1, 4), abc=ABC, restart_after=(2, 4), sel_out=sel, status=status,
            carry=(sel, 0.95) if s else None, defer=True)
d3.decay_rows(M, sel, 0.95)
out["W"], out["M"], out["sel"] = W, M, sel.clone()
# column selection
Wc = synthetic.gaussian((2, 512, 96), seed=6, std=0.02, device=dev)
Mc = torch.zeros_like(Wc)
Gc = synthetic.lowrank_batch(2, 512, 96, base_seed=7, dtype=torch.bfloat16, device=dev)
out["sel_cols"] = d3.step_cols(Wc, Mc, Gc, f=(1, 8), abc=ABC, restart_after=(2,), status=status).clone()
out["Wc"] = Wc
torch.cuda.synchronize()
out["status_valid"] = torch.tensor([int(status.item())])
# a carried list with one row outside [-1, n): both builds skip it, the checked one flags it
status.zero_()
bad = sel.clone()
bad[1, 3] = n + 3
G = synthetic.lowrank_batch(3, n, m, base_seed=20, dtype=torch.bfloat16, device=dev)
d3.step(W, M, G, f=(1, 4), abc=ABC, restart_after=(2, 4), sel_out=sel, status=status, carry=(bad, 0.95),
        defer=True)
torch.cuda.synchronize()
out["M_bad"] = M
out["status_bad"] = torch.tensor([int(status.item())])
np.savez({path!r}, **{{k: v.detach().cpu().numpy() for k, v in out.items()}})
'''


def _run(tmp_path, checked: bool):
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build(checked=checked)
    path = str(tmp_path / f"out_{int(checked)}.npz")
    code = CHILD.format(root=ROOT, checked=checked, path=path)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return dict(np.load(path))


def test_checked_build_matches_default_and_flags_out_of_range_rows(tmp_path):
    plain = _run(tmp_path, checked=False)
    chk = _run(tmp_path, checked=True)
    for key in ("sym", "gram", "gram_small", "ns", "W", "M", "sel", "sel_cols", "Wc", "M_bad"):
        a, b = plain[key], chk[key]
        assert a.shape == b.shape, key
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"{key}: checked build differs"
    assert int(plain["status_valid"][0]) == 0 and int(chk["status_valid"][0]) == 0
    assert int(plain["status_bad"][0]) & d3.DEV_RANGE == 0
    assert int(chk["status_bad"][0]) & d3.DEV_RANGE
