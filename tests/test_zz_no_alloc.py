"""dion3_gram_ns_noalloc: Gram Newton-Schulz for callers that may not allocate device memory.

Such callers (embedded runtimes whose device memory is carved up at start-up, plug-ins handed
raw buffers by a host application that owns every allocation, code inside allocator
callbacks) cannot supply dion3_gram_ns's workspace, so this entry point uses a scratch array
compiled into the library.  Its results must match dion3_gram_ns, the workspace entry point,
within the Gram Newton-Schulz test tolerance -- on two calls in a row, the second running on
whatever the first left in the shared scratch.
"""

import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import synthetic
from gpu_util import rel_frob, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
ABC = [(3.4445, -4.7750, 2.0315)] * 5
TOL = 3e-2   # the 16-bit Gram Newton-Schulz bar used by the other parity tests


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


def test_two_calls_match_workspace_entry_point():
    X1 = synthetic.lowrank_batch(3, 200, 800, base_seed=900, dtype=torch.bfloat16, device=DEV)
    X2 = synthetic.lowrank_batch(2, 130, 300, base_seed=950, dtype=torch.float32, device=DEV)  # copied path
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got1 = d3.gram_ns_noalloc(X1, ABC, (2, 4), status=status)
    got2 = d3.gram_ns_noalloc(X2, ABC, (2,), status=status)
    torch.cuda.synchronize()
    ref1 = d3.gram_ns(X1, ABC, (2, 4))
    ref2 = d3.gram_ns(X2, ABC, (2,))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in range(X1.shape[0]):
        assert rel_frob(to64(got1[b]), to64(ref1[b])) <= TOL
    for b in range(X2.shape[0]):
        assert rel_frob(to64(got2[b]), to64(ref2[b])) <= TOL


def test_rejects_problems_beyond_the_scratch_size():
    n, m, batch = 1024, 4096, 8
    need = d3.workspace_bytes_gram_ns(batch, n, m, torch.bfloat16, torch.float16, 2)
    assert need > d3.NOALLOC_SCRATCH_BYTES
    X = torch.zeros((batch, n, m), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(d3.Dion3Error) as e:
        d3.gram_ns_noalloc(X, ABC, (2, 4))
    assert e.value.code == 3   # DION3_EWORKSPACE
