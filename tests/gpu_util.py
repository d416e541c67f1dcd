"""Helpers shared by the GPU parity tests (comparison metrics only; no method arithmetic)."""

import numpy as np
import torch


def rel_frob(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def bits32(t) -> np.ndarray:
    a = t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return a.astype(np.float32, copy=False).view(np.uint32)


def exactly_symmetric(t: torch.Tensor) -> bool:
    a = t.detach().cpu()
    if a.dtype == torch.bfloat16 or a.dtype == torch.float16:
        a = a.view(torch.int16)
    else:
        a = a.view(torch.int32)
    return bool(torch.equal(a, a.transpose(-1, -2)))


def aligned_copy(t: torch.Tensor) -> torch.Tensor:
    """Same values, leading dimension rounded up so that each row starts on 16 bytes
    (the documented layout rule of the symmetric GEMM's inputs)."""
    es = t.element_size()
    q = 16 // es
    cols = t.shape[-1]
    ld = max(q, (cols + q - 1) // q * q)
    buf = torch.zeros(t.shape[:-1] + (ld,), dtype=t.dtype, device=t.device)
    view = buf[..., :cols]
    view.copy_(t)
    return view
