"""Seeded synthetic inputs shaped like the Dion3 paper's workloads.

This module only draws random numbers and assembles test matrices; it holds
none of the method's arithmetic.  It is the one module that both the oracle
side (tests, CPU baseline) and the CUDA side (tests, bench) use, so that both
see the very same tensors.

Recipes (the paper measures isolated optimizer steps on synthetic data):

* ``gaussian``: i.i.d. N(0, std^2).
* ``symmetric_gaussian``: N(0, 1) lower triangle mirrored to the upper one,
  so the stored matrix is exactly symmetric in every dtype.
* ``lowrank_plus_noise``: M = U diag(sigma) V^T + noise * N(0, 1) with U, V
  orthonormal (QR of Gaussian n x r and m x r, float64 on the host),
  sigma_i = 1 / i over rank r = 64, noise = 0.01 -- a momentum-like matrix
  whose rows are noise-dominated (many near-equal row norms).

Seeds: the caller picks them; the bench and the tests use
``1000 * workload + matrix_index (+ 10**6 * step)`` for the batched
workloads so that each matrix can be regenerated on its own.
"""

from __future__ import annotations

import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian(shape, seed: int, std: float = 1.0, dtype=torch.float32, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def symmetric_gaussian(n: int, seed: int, dtype=torch.float32, device="cpu", batch: int | None = None) -> torch.Tensor:
    shape = (n, n) if batch is None else (batch, n, n)
    x = gaussian(shape, seed, dtype=torch.float32, device=device)
    low = torch.tril(x)
    sym = low + torch.tril(x, diagonal=-1).transpose(-1, -2)
    return sym.to(dtype)


def _orthonormal_columns(rows: int, rank: int, seed: int) -> torch.Tensor:
    g = _gen(seed, "cpu")
    a = torch.randn((rows, rank), generator=g, dtype=torch.float64)
    q, _ = torch.linalg.qr(a)
    return q


def lowrank_plus_noise(n: int, m: int, seed: int, rank: int = 64, noise: float = 0.01,
                       dtype=torch.bfloat16, device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
    """One n x m low-rank-plus-noise matrix (see module docstring).

    If ``out`` is given (an n x m tensor on ``device``), the matrix is written
    into it and ``out`` is returned.
    """
    r = min(rank, n, m)
    U = _orthonormal_columns(n, r, 2 * seed + 1)
    V = _orthonormal_columns(m, r, 2 * seed + 2)
    sig = 1.0 / torch.arange(1, r + 1, dtype=torch.float64)
    low = ((U * sig) @ V.T).to(device=device, dtype=torch.float32)
    g = _gen(seed, device)
    z = torch.randn((n, m), generator=g, device=device, dtype=torch.float32)
    z.mul_(noise).add_(low)
    if out is None:
        return z.to(dtype)
    out.copy_(z)
    return out


def lowrank_batch(batch: int, n: int, m: int, base_seed: int, rank: int = 64, noise: float = 0.01,
                  dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """[batch, n, m] stack; matrix i uses seed base_seed + i."""
    out = torch.empty((batch, n, m), dtype=dtype, device=device)
    for i in range(batch):
        lowrank_plus_noise(n, m, base_seed + i, rank, noise, dtype, device, out=out[i])
    return out
