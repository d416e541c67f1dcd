"""dion3_gram_ns_noalloc: Gram Newton-Schulz for callers that may not allocate device memory.

Such callers (embedded runtimes whose device memory is carved up at start-up, plug-ins handed
raw buffers by a host application that owns every allocation, code inside allocator
callbacks) cannot supply dion3_gram_ns's workspace, so this entry point uses a scratch array
compiled into the library.  It runs the very kernels dion3_gram_ns runs, on the same inputs,
so its output must be bit-identical to the workspace entry point's -- on several calls in a
row, each running on whatever the previous one left in the shared scratch -- and within the
Gram Newton-Schulz tolerances of the float64 oracle.

This file is collected last, so a run that stops at the first failure has run every other
test before it; it also passes when run on its own in a fresh process.
"""

import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import oracle
import synthetic
from gpu_util import rel_frob, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"
ABC = [(3.4445, -4.7750, 2.0315)] * 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def test_calls_in_a_row_equal_the_workspace_entry_point():
    """Three calls in a row (X read in place, X copied and cast, the first again): each output is
    bit-identical to dion3_gram_ns on the same input, and within 3e-2 (16-bit iterates) or 1e-4
    (fp32 mode) of the oracle."""
    X1 = synthetic.lowrank_batch(3, 200, 800, base_seed=900, dtype=torch.float16, device=DEV)   # in place
    X2 = synthetic.lowrank_batch(2, 130, 300, base_seed=950, dtype=torch.float32, device=DEV)   # copied
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got1 = d3.gram_ns_noalloc(X1, ABC, (2, 4), compute=torch.float16, status=status)
    got2 = d3.gram_ns_noalloc(X2, ABC, (2,), compute=torch.float16, out_dtype=torch.float32, status=status)
    got3 = d3.gram_ns_noalloc(X1, ABC, (2, 4), compute=torch.float16, status=status)
    got4 = d3.gram_ns_noalloc(X2, ABC, (2,), compute=torch.float32, status=status)
    torch.cuda.synchronize()
    ref1 = d3.gram_ns(X1, ABC, (2, 4), compute=torch.float16)
    ref2 = d3.gram_ns(X2, ABC, (2,), compute=torch.float16, out_dtype=torch.float32)
    ref4 = d3.gram_ns(X2, ABC, (2,), compute=torch.float32)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(_bits(got1), _bits(ref1))
    assert torch.equal(_bits(got2), _bits(ref2))
    assert torch.equal(_bits(got3), _bits(ref1))
    assert torch.equal(_bits(got4), _bits(ref4))
    for b in range(X1.shape[0]):
        assert rel_frob(to64(got1[b]), oracle.gram_ns(to64(X1[b]), ABC, (2, 4))) <= 3e-2
    for b in range(X2.shape[0]):
        ref = oracle.gram_ns(to64(X2[b]), ABC, (2,))
        assert rel_frob(to64(got2[b]), ref) <= 3e-2
        assert rel_frob(to64(got4[b]), ref) <= 1e-4


def test_workspace_just_under_the_limit():
    """The largest batch of 512 x 4096 fp16 matrices whose workspace fits the scratch array."""
    n, m = 512, 4096
    cap = d3.NOALLOC_SCRATCH_BYTES
    batch = 1
    while d3.workspace_bytes_gram_ns(batch + 1, n, m, torch.float16, torch.float16, 2) <= cap:
        batch += 1
    need = d3.workspace_bytes_gram_ns(batch, n, m, torch.float16, torch.float16, 2)
    assert cap - need < need // batch + 4096
    X = synthetic.lowrank_batch(batch, n, m, base_seed=1200, dtype=torch.float16, device=DEV)
    for _ in range(2):
        got = d3.gram_ns_noalloc(X, ABC, (2, 4), compute=torch.float16)
        ref = d3.gram_ns(X, ABC, (2, 4), compute=torch.float16)
        torch.cuda.synchronize()
        assert torch.equal(_bits(got), _bits(ref))
    assert rel_frob(to64(got[batch - 1]), oracle.gram_ns(to64(X[batch - 1]), ABC, (2, 4))) <= 3e-2


def test_rejects_problems_beyond_the_scratch_size():
    n, m, batch = 1024, 4096, 8
    need = d3.workspace_bytes_gram_ns(batch, n, m, torch.bfloat16, torch.float16, 2)
    assert need > d3.NOALLOC_SCRATCH_BYTES
    X = torch.zeros((batch, n, m), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(d3.Dion3Error) as e:
        d3.gram_ns_noalloc(X, ABC, (2, 4))
    assert e.value.code == 3   # DION3_EWORKSPACE


def test_misaligned_x_over_the_limit_is_rejected_and_writes_nothing():
    """An X that fits when read in place, but whose rows do not start on 16 bytes: its copy does
    not fit, so the call fails with DION3_EWORKSPACE and Out keeps its contents."""
    n, m = 512, 4096
    cap = d3.NOALLOC_SCRATCH_BYTES
    batch = 1
    while d3.workspace_bytes_gram_ns(batch + 1, n, m, torch.float16, torch.float16, 1) <= cap:
        batch += 1
    assert d3.workspace_bytes_gram_ns(batch, n, m, torch.float32, torch.float16, 1) > cap
    flat = synthetic.gaussian((batch * n * m + 1,), seed=1300, dtype=torch.float16, device=DEV)
    X = flat[1:].view(batch, n, m)   # 2 bytes past a 16-byte boundary
    assert X.data_ptr() % 16 != 0
    out = torch.full((batch, n, m), 7.0, dtype=torch.float16, device=DEV)
    with pytest.raises(d3.Dion3Error) as e:
        d3.gram_ns_noalloc(X, ABC, (2,), compute=torch.float16, out=out)
    assert e.value.code == 3
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


@pytest.mark.parametrize("xdt,odt", [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32)])
def test_guard_band_around_out(xdt, odt):
    """Out is a window (padded rows, a margin before and after) into a pattern-filled buffer:
    nothing outside the window may change.  bf16 X with bf16 iterates is read in place; fp32 X
    is copied and cast."""
    batch, n, m = 3, 72, 300
    pad, margin = 20, 4096
    ldo = m + pad
    X = synthetic.lowrank_batch(batch, n, m, base_seed=1400, dtype=xdt, device=DEV)
    X = X.contiguous() if xdt == torch.float32 else X
    if xdt == torch.bfloat16:
        Xa = torch.zeros((batch, n, 304), dtype=xdt, device=DEV)   # 608-byte rows: read in place
        Xa[:, :, :m] = X
        X = Xa[:, :, :m]
    es = torch.tensor([], dtype=odt).element_size()
    total = margin + batch * n * ldo + margin
    buf = torch.empty(total * es, dtype=torch.uint8, device=DEV)
    buf.fill_(0xA5)
    before = buf.clone()
    out = buf.view(odt)[margin:margin + batch * n * ldo].view(batch, n, ldo)[:, :, :m]
    compute = torch.bfloat16 if xdt == torch.bfloat16 else torch.float16
    d3.gram_ns_noalloc(X, ABC, (2, 4), compute=compute, out=out)
    torch.cuda.synchronize()
    mask = torch.ones(total, dtype=torch.bool, device=DEV)
    mask[margin:margin + batch * n * ldo].view(batch, n, ldo)[:, :, :m] = False
    mask_b = mask.repeat_interleave(es)
    assert torch.equal(buf[mask_b], before[mask_b])
    ref = d3.gram_ns(X, ABC, (2, 4), compute=compute, out_dtype=odt)
    torch.cuda.synchronize()
    assert torch.equal(_bits(out.contiguous()), _bits(ref.contiguous()))
