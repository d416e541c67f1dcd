"""Guard bands: every entry point writes only inside the buffers it was given.

Each output, state tensor and workspace is a window into a larger buffer whose surrounding
bytes (and, for padded leading dimensions, the padding columns) hold a fixed pattern; after
the call the pattern must be intact.  Covers the fused small-n and the product-by-product
Gram-NS paths, fp32 compute, standard NS, the Dion3 step (top-k and caller-given rows) and the
symmetric GEMM."""

import pytest
import torch

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
import synthetic
from gpu_util import aligned_copy

pytestmark = pytest.mark.gpu
DEV = "cuda"
ABC = [(3.4445, -4.7750, 2.0315)] * 5
GUARD = 4096  # bytes on each side
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

    _build.build()
    d3.lib()


class Guarded:
    """A byte buffer with GUARD pattern bytes on both sides of an inner window."""

    def __init__(self, nbytes):
        self.n = nbytes
        self.raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=DEV)

    def inner(self):
        return self.raw[GUARD:GUARD + self.n]

    def intact(self):
        return bool((self.raw[:GUARD] == PATTERN).all()) and bool((self.raw[GUARD + self.n:] == PATTERN).all())


def guarded_tensor(shape, dtype, fill=None):
    es = torch.empty((), dtype=dtype).element_size()
    numel = 1
    for s in shape:
        numel *= s
    g = Guarded(numel * es)
    t = g.inner().view(dtype).view(shape)
    if fill is not None:
        t.copy_(fill)
    return g, t


def padded_matrix(batch, rows, cols, ld, dtype):
    """[batch, rows, cols] view with leading dimension ld, inside a guarded buffer whose padding
    columns keep the pattern."""
    es = torch.empty((), dtype=dtype).element_size()
    g = Guarded(batch * rows * ld * es)
    full = g.inner().view(dtype).view(batch, rows, ld)
    return g, full, full[:, :, :cols]


def pad_intact(full, cols):
    pad = full[:, :, cols:].contiguous().view(torch.uint8)
    return bool((pad == PATTERN).all())


@pytest.mark.parametrize("n,m,compute", [(96, 2048, torch.float16), (200, 520, torch.float16),
                                         (64, 300, torch.bfloat16), (130, 264, torch.float32)])
def test_gram_ns_writes_stay_inside(n, m, compute):
    B = 3
    X = synthetic.lowrank_batch(B, n, m, base_seed=1300, dtype=torch.bfloat16 if compute != torch.float32 else torch.float32,
                                device=DEV)
    odt = torch.float32 if compute == torch.float32 else torch.bfloat16
    ld = (m + 7) // 8 * 8 + 8  # 16-byte rows for every dtype, plus one padding unit
    go, full, O = padded_matrix(B, n, m, ld, odt)
    need = d3.workspace_bytes_gram_ns(B, n, m, X.dtype, compute, 2)
    gw = Guarded(need)
    d3.gram_ns(X, ABC, (2, 4), compute=compute, out=O, workspace=gw.inner())
    torch.cuda.synchronize()
    assert go.intact() and gw.intact()
    assert pad_intact(full, m)
    assert torch.isfinite(O.float()).all()


@pytest.mark.parametrize("n,m", [(64, 64), (150, 400)])
def test_ns_standard_writes_stay_inside(n, m):
    B = 2
    X = synthetic.lowrank_batch(B, n, m, base_seed=1400, dtype=torch.bfloat16, device=DEV)
    ld = (m + 7) // 8 * 8 + 8
    go, full, O = padded_matrix(B, n, m, ld, torch.bfloat16)
    gw = Guarded(d3.workspace_bytes_ns_standard(B, n, m, torch.float16))
    d3.ns_standard(X, ABC, out=O, workspace=gw.inner())
    torch.cuda.synchronize()
    assert go.intact() and gw.intact() and pad_intact(full, m)


@pytest.mark.parametrize("n,m,f,given", [(96, 512, (1, 4), False), (256, 1000, (1, 8), False), (128, 640, (1, 2), True)])
def test_step_writes_stay_inside(n, m, f, given):
    B = 3
    k = d3.k_of(n, *f)
    gW, W = guarded_tensor((B, n, m), torch.float32, synthetic.gaussian((B, n, m), seed=21, std=0.02, device=DEV))
    gM, M = guarded_tensor((B, n, m), torch.float32, synthetic.gaussian((B, n, m), seed=22, std=0.01, device=DEV))
    G = synthetic.lowrank_batch(B, n, m, base_seed=1500, dtype=torch.bfloat16, device=DEV)
    gS, sel = guarded_tensor((B, k), torch.int32)
    gws = Guarded(d3.workspace_bytes_step(B, n, m, f[0], f[1], 0 if given else 1, torch.float16, 2))
    rows = None
    if given:
        rows = torch.stack([torch.randperm(n, generator=torch.Generator().manual_seed(i))[:k].sort().values
                            for i in range(B)]).to(torch.int32).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    d3.step(W, M, G, f=f, abc=ABC, restart_after=(2, 4), sel_out=sel, workspace=gws.inner(), rows=rows,
            status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert gW.intact() and gM.intact() and gS.intact() and gws.intact()


@pytest.mark.parametrize("n,k,beta", [(300, 100, 0.0), (513, 64, 1.0), (1024, 256, 1.0)])
def test_sym_gemm_writes_stay_inside(n, k, beta):
    A = aligned_copy(synthetic.gaussian((n, k), seed=31, std=k ** -0.5, dtype=torch.bfloat16, device=DEV))
    C = aligned_copy(synthetic.symmetric_gaussian(n, seed=32, dtype=torch.bfloat16, device=DEV))
    ld = (n + 7) // 8 * 8 + 8
    go, full, D = padded_matrix(1, n, n, ld, torch.bfloat16)
    d3.sym_gemm(A, C=C if beta else None, beta=beta, out=D[0])
    torch.cuda.synchronize()
    assert go.intact() and pad_intact(full, n)


def test_step_cols_writes_stay_inside():
    B, m, n, f = 2, 600, 72, (1, 4)
    k = d3.k_of(n, *f)
    gW, W = guarded_tensor((B, m, n), torch.float32, synthetic.gaussian((B, m, n), seed=41, std=0.02, device=DEV))
    gM, M = guarded_tensor((B, m, n), torch.float32, synthetic.gaussian((B, m, n), seed=42, std=0.01, device=DEV))
    G = synthetic.lowrank_batch(B, m, n, base_seed=1600, dtype=torch.bfloat16, device=DEV)
    gS, sel = guarded_tensor((B, k), torch.int32)
    gws = Guarded(d3.workspace_bytes_step_cols(B, m, n, f[0], f[1], 1, torch.float16, 2))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    d3.step_cols(W, M, G, f=f, abc=ABC, restart_after=(2, 4), sel_out=sel, workspace=gws.inner(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert gW.intact() and gM.intact() and gS.intact() and gws.intact()
