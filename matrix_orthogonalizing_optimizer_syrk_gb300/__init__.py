"""GB300 (sm_103a) Dion3 / Gram Newton-Schulz hot path: Python binding of libdion3.so.

This module only marshals arguments: it turns torch CUDA tensors into device pointers,
leading dimensions and strides, and calls the C ABI declared in ``include/dion3.h``.
Every step of the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and a missing library raises at first use.

Entry points (same names as the C ABI, without the prefix):

* ``sym_gemm``  -- D = alpha A B^T + beta C + gamma I for symmetric results, lower
  triangle computed and mirrored ("Dion3: Full-Stack Orthogonal Updates", prerequisite
  "symmetric GEMM kernels").
* ``gram_ns``   -- batched Gram Newton-Schulz with restarts (same page, Theorem 2 and
  Algorithm 3).
* ``step``      -- one Dion3 step on a megabatch (same page, Algorithm 4 with error
  feedback).
* ``k_of``, ``status_str``, ``workspace_bytes_gram_ns``, ``workspace_bytes_step``.
"""

from __future__ import annotations

import ctypes
import os

import torch

_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_DIR, "libdion3.so")
# The same library built with in-kernel range checks (DION3_DEV_RANGE); see use_checked_build().
CHECKED_LIB_PATH = os.path.join(_DIR, "libdion3_checked.so")

BF16, FP16, FP32 = 0, 1, 2
DEV_NONFINITE, DEV_TIMEOUT, DEV_SELECT, DEV_RANGE = 0x1, 0x2, 0x4, 0x8
_DT = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}

_c_int, _c_i64, _c_f, _c_p, _c_sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/dion3.h
SIGNATURES = {
    "dion3_sym_gemm": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64,
                                _c_p, _c_i64, _c_i64, _c_p, _c_i64, _c_i64, _c_f, _c_f, _c_f, _c_int, _c_int,
                                _c_p, _c_p]),
    "dion3_gram_ns_workspace_bytes": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "dion3_gram_ns": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_i64, _c_i64, _c_int, _c_p, _c_i64, _c_i64, _c_int,
                               _c_int, ctypes.POINTER(_c_f), ctypes.POINTER(_c_int), _c_int, _c_f, _c_int,
                               _c_p, _c_sz, _c_p, _c_p]),
    "dion3_ns_standard_workspace_bytes": (_c_sz, [_c_int, _c_int, _c_int, _c_int]),
    "dion3_ns_standard": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_i64, _c_i64, _c_int, _c_p, _c_i64, _c_i64,
                                   _c_int, _c_int, ctypes.POINTER(_c_f), _c_f, _c_int, _c_p, _c_sz, _c_p, _c_p]),
    "dion3_k": (_c_int, [_c_int, _c_int, _c_int]),
    "dion3_step_workspace_bytes": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "dion3_step": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_f, _c_f, _c_f,
                            _c_int, _c_int, ctypes.POINTER(_c_f), ctypes.POINTER(_c_int), _c_int, _c_f, _c_int,
                            _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "dion3_step_timed": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_f, _c_f,
                                  _c_f, _c_int, _c_int, ctypes.POINTER(_c_f), ctypes.POINTER(_c_int), _c_int, _c_f,
                                  _c_int, _c_p, _c_p, _c_sz, _c_p, _c_p, ctypes.POINTER(_c_p), _c_int]),
    "dion3_step_cols_workspace_bytes": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "dion3_step_cols": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_f, _c_f, _c_f,
                                 _c_int, _c_int, ctypes.POINTER(_c_f), ctypes.POINTER(_c_int), _c_int, _c_f, _c_int,
                                 _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "dion3_step_dev": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_p, _c_int,
                                _c_int, _c_int, ctypes.POINTER(_c_f), ctypes.POINTER(_c_int), _c_int, _c_f, _c_int,
                                _c_p, _c_p, _c_sz, _c_p, _c_p]),
    "dion3_step_carry": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_f, _c_f,
                                  _c_f, _c_int, _c_int, ctypes.POINTER(_c_f), ctypes.POINTER(_c_int), _c_int, _c_f,
                                  _c_int, _c_p, _c_p, _c_f, _c_int, _c_p, _c_sz, _c_p, _c_p, ctypes.POINTER(_c_p),
                                  _c_int]),
    "dion3_decay_rows": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p, _c_int, _c_f, _c_p]),
    "dion3_step_dev_carry": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_p,
                                      _c_int, _c_int, _c_int, ctypes.POINTER(_c_f), ctypes.POINTER(_c_int), _c_int,
                                      _c_f, _c_int, _c_p, _c_p, _c_p, _c_int, _c_p, _c_sz, _c_p, _c_p]),
    "dion3_gram_ns_noalloc": (_c_int, [_c_int, _c_int, _c_int, _c_p, _c_i64, _c_i64, _c_int, _c_p, _c_i64, _c_i64,
                                       _c_int, _c_int, ctypes.POINTER(_c_f), ctypes.POINTER(_c_int), _c_int, _c_f,
                                       _c_int, _c_p, _c_p]),
    "dion3_status_str": (ctypes.c_char_p, [_c_int]),
    "dion3_abi_version": (_c_int, []),
    "dion3_range_checks": (_c_int, []),
    "dion3_selftest_watchdog": (_c_int, [ctypes.c_longlong, _c_p, _c_p]),
}

SELECT_GIVEN = 0  # norm_p of a caller-chosen row set (DION3_SELECT_GIVEN)

_lib = None
_lib_path = LIB_PATH


class Dion3Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_str(code)} ({code})")


def use_checked_build() -> None:
    """Load libdion3_checked.so instead of libdion3.so (call before the first entry point).

    The checked build runs the same kernels with in-kernel range checks that set DEV_RANGE in
    the status word; it is built by ``_build.build(checked=True)``.
    """
    global _lib_path
    if _lib is not None and _lib_path != CHECKED_LIB_PATH:
        raise RuntimeError("the default library is already loaded in this process")
    _lib_path = CHECKED_LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_lib_path):
            raise RuntimeError(f"{_lib_path} is missing; build it with "
                               "`python -m matrix_orthogonalizing_optimizer_syrk_gb300._build`")
        L = ctypes.CDLL(_lib_path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().dion3_status_str(int(code)).decode()


def k_of(n: int, f_num: int, f_den: int) -> int:
    return int(lib().dion3_k(int(n), int(f_num), int(f_den)))


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise Dion3Error(rc, where)


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _dtype_code(d) -> int:
    return d if isinstance(d, int) else _DT[d]


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (there is no CPU path)")
    return t


def _layout(t: torch.Tensor):
    """(batch, rows, cols, ld, stride) of a 2-D or 3-D tensor with unit column stride."""
    if t.dim() == 2:
        rows, cols = t.shape
        if t.stride(1) != 1 and cols > 1:
            raise ValueError("columns must be contiguous")
        ld = t.stride(0) if t.stride(0) >= max(cols, 1) else max(cols, 1)
        return 1, rows, cols, ld, rows * ld
    if t.dim() == 3:
        batch, rows, cols = t.shape
        if t.stride(2) != 1 and cols > 1:
            raise ValueError("columns must be contiguous")
        ld = t.stride(1) if t.stride(1) >= max(cols, 1) else max(cols, 1)
        return batch, rows, cols, ld, t.stride(0)
    raise ValueError("expected a 2-D or 3-D tensor")


def _stream_ptr(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _empty_aligned(shape, dtype, device) -> torch.Tensor:
    """Uninitialised tensor whose rows start on 16-byte boundaries (padded leading dim)."""
    es = torch.tensor([], dtype=dtype).element_size()
    q = 16 // es
    cols = shape[-1]
    ld = max(q, (cols + q - 1) // q * q)
    return torch.empty(tuple(shape[:-1]) + (ld,), dtype=dtype, device=device)[..., :cols]


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _abc_arrays(abc, restart_after):
    trip = [tuple(float(v) for v in t) for t in abc]
    T = len(trip)
    flat = (_c_f * (3 * T))(*[v for t in trip for v in t])
    rs = list(int(r) for r in restart_after)
    rarr = (_c_int * max(1, len(rs)))(*rs) if rs else (_c_int * 1)(0)
    return T, flat, rarr, len(rs)


def sym_gemm(A: torch.Tensor, C: torch.Tensor | None = None, B: torch.Tensor | None = None, alpha: float = 1.0,
             beta: float = 0.0, gamma: float = 0.0, out: torch.Tensor | None = None, out_dtype=None,
             status: torch.Tensor | None = None) -> torch.Tensor:
    """D = alpha A B^T + beta C + gamma I (B defaults to A); lower triangle computed, upper mirrored."""
    _cuda(A, "A")
    batch, n, k, lda, sa = _layout(A)
    odt = A.dtype if out_dtype is None else out_dtype
    if out is None:
        shape = (n, n) if A.dim() == 2 else (batch, n, n)
        out = _empty_aligned(shape, odt, A.device)
    _, _, _, ldd, sd = _layout(_cuda(out, "out"))
    ldb = sb = 0
    if B is not None:
        _, _, _, ldb, sb = _layout(_cuda(B, "B"))
    ldc = sc = 0
    if C is not None:
        _, _, _, ldc, sc = _layout(_cuda(C, "C"))
    rc = lib().dion3_sym_gemm(batch, n, k, _ptr(A), lda, sa, _ptr(B), ldb, sb, _ptr(C), ldc, sc, _ptr(out), ldd, sd,
                              float(alpha), float(beta), float(gamma), _dt(A), _dt(out), _ptr(status),
                              _stream_ptr(A.device))
    _check(rc, "dion3_sym_gemm")
    return out


def workspace_bytes_gram_ns(batch: int, n: int, m: int, x_dtype, compute, n_restart: int) -> int:
    return int(lib().dion3_gram_ns_workspace_bytes(batch, n, m, _dtype_code(x_dtype), _dtype_code(compute),
                                                   n_restart))


def gram_ns(X: torch.Tensor, abc, restart_after=(), eps: float = 1e-7, compute=torch.float16,
            out: torch.Tensor | None = None, out_dtype=None, workspace: torch.Tensor | None = None,
            status: torch.Tensor | None = None) -> torch.Tensor:
    """Gram Newton-Schulz of each n x m matrix of X (n <= m).

    ``compute`` is the storage type of the iterates R, Z, Q and the restarted X (fp32
    accumulation throughout).  The default is float16, the precision the Dion3 paper runs
    Gram Newton-Schulz in (method details, Algorithm 3: normalise, then convert to float16);
    bfloat16 is supported but its 8-bit mantissa costs roughly an order of magnitude in
    accuracy on the iterates.  The output defaults to X's dtype (fp32 for fp32 compute).
    """
    _cuda(X, "X")
    batch, n, m, ldx, sx = _layout(X)
    odt = (torch.float32 if compute == torch.float32 else X.dtype) if out_dtype is None else out_dtype
    if out is None:
        out = _empty_aligned(tuple(X.shape), odt, X.device)
    _, _, _, ldo, so = _layout(_cuda(out, "out"))
    T, flat, rarr, nr = _abc_arrays(abc, restart_after)
    need = workspace_bytes_gram_ns(batch, n, m, X.dtype, compute, nr)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=X.device)
    rc = lib().dion3_gram_ns(batch, n, m, _ptr(X), ldx, sx, _dt(X), _ptr(out), ldo, so, _dt(out), T, flat, rarr, nr,
                             float(eps), _dtype_code(compute), _ptr(workspace), workspace.numel(), _ptr(status),
                             _stream_ptr(X.device))
    _check(rc, "dion3_gram_ns")
    return out


def workspace_bytes_ns_standard(batch: int, n: int, m: int, compute) -> int:
    return int(lib().dion3_ns_standard_workspace_bytes(batch, n, m, _dtype_code(compute)))


def ns_standard(X: torch.Tensor, abc, eps: float = 1e-7, compute=torch.float16, out: torch.Tensor | None = None,
                out_dtype=None, workspace: torch.Tensor | None = None,
                status: torch.Tensor | None = None) -> torch.Tensor:
    """Standard quintic Newton-Schulz of each n x m matrix of X (n <= m): the fallback for
    square matrices, where Gram Newton-Schulz saves nothing (Dion3 paper, limitations)."""
    _cuda(X, "X")
    batch, n, m, ldx, sx = _layout(X)
    odt = (torch.float32 if compute == torch.float32 else X.dtype) if out_dtype is None else out_dtype
    if out is None:
        out = _empty_aligned(tuple(X.shape), odt, X.device)
    _, _, _, ldo, so = _layout(_cuda(out, "out"))
    T, flat, _, _ = _abc_arrays(abc, ())
    need = workspace_bytes_ns_standard(batch, n, m, compute)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=X.device)
    rc = lib().dion3_ns_standard(batch, n, m, _ptr(X), ldx, sx, _dt(X), _ptr(out), ldo, so, _dt(out), T, flat,
                                 float(eps), _dtype_code(compute), _ptr(workspace), workspace.numel(), _ptr(status),
                                 _stream_ptr(X.device))
    _check(rc, "dion3_ns_standard")
    return out


def ns_standard_launch_count(T: int) -> int:
    """Kernel launches of one dion3_ns_standard call: sum of squares, scale, cast, then three
    products per iteration (plus a final cast when the output dtype differs)."""
    return 3 + 3 * T


def workspace_bytes_step(batch: int, n: int, m: int, f_num: int, f_den: int, norm_p: int, compute,
                         n_restart: int) -> int:
    return int(lib().dion3_step_workspace_bytes(batch, n, m, f_num, f_den, norm_p, _dtype_code(compute), n_restart))


def step(W: torch.Tensor, M: torch.Tensor, G: torch.Tensor, f=(1, 4), mu: float = 0.95, eta: float = 0.01,
         wd: float = 0.0, norm_p: int = 1, abc=None, restart_after=(2,), eps: float = 1e-7, compute=torch.float16,
         sel_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
         status: torch.Tensor | None = None, events=None, hyper: torch.Tensor | None = None,
         decay: bool = False, rows: torch.Tensor | None = None, carry=None, defer: bool = False) -> torch.Tensor:
    """One Dion3 step on [batch, n, m] (or [n, m]) contiguous W, M (fp32) and G; returns the selected rows.

    ``events``: optional list of up to five recorded-once ``torch.cuda.Event`` objects, recorded
    by the library at the phase boundaries (see dion3_step_timed in include/dion3.h).
    ``hyper``: optional fp32 device tensor {mu, eta, wd}; the kernels read it when they run
    (``mu``, ``eta``, ``wd`` are then ignored and ``decay`` turns the W decay pass on), so the
    call can be captured in a CUDA graph once and replayed with new values.
    ``rows``: optional caller-chosen row set S, int32 [batch, k] (or [k]) with strictly ascending
    rows per matrix (e.g. a sorted random subset); no keys are computed (``norm_p`` is ignored).
    A matrix whose rows break the rule is left unselected and flags DION3_DEV_SELECT.
    ``defer``: leave this step's decay of M[S,:] by ``mu`` pending (M[S,:] keeps M + G) and
    pass ``carry=(sel, mu)`` -- the returned rows and this mu -- to the next call, whose momentum
    pass applies it (dion3_step_carry in include/dion3.h); ``decay_rows`` applies it on its own.
    The state that results is bit-identical to that of plain steps.  With ``hyper`` the carried
    mu is a one-element fp32 device tensor, read as the pending factor and, with ``defer``,
    overwritten with this step's mu (dion3_step_dev_carry): ``carry=(sel, mu_word)`` every call,
    mu_word set to 1.0 before the first (``carry=(None, mu_word)`` carries nothing in).
    """
    carrying = carry is not None or defer
    mu_word = None
    if carrying and hyper is not None:
        if carry is None or not isinstance(carry[1], torch.Tensor):
            raise ValueError("with hyper, carry=(rows or None, mu_word) with mu_word a device fp32 tensor")
        mu_word = carry[1]
        _cuda(mu_word, "carried mu")
        if mu_word.dtype != torch.float32 or mu_word.numel() < 1:
            raise ValueError("the carried mu word must be an fp32 device tensor")
    elif carry is not None and isinstance(carry[1], torch.Tensor):
        raise ValueError("a device carried mu needs hyper (device hyperparameters)")
    for t, name in ((W, "W"), (M, "M"), (G, "G")):
        _cuda(t, name)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if W.dtype != torch.float32 or M.dtype != torch.float32:
        raise TypeError("W and M are fp32 state")
    if W.shape != M.shape or G.shape != M.shape:
        raise ValueError("W, M, G must have the same shape")
    batch, n, m, _, _ = _layout(M)
    f_num, f_den = f
    k = k_of(n, f_num, f_den)
    if k < 0:
        raise ValueError("need 0 < f <= 1")
    shape = (k,) if M.dim() == 2 else (batch, k)
    if sel_out is None:
        sel_out = torch.empty(shape, dtype=torch.int32, device=M.device)
    if rows is not None:
        _cuda(rows, "rows")
        if rows.dtype != torch.int32 or tuple(rows.shape) != shape:
            raise ValueError(f"rows must be int32 of shape {shape}")
        if rows.data_ptr() != sel_out.data_ptr():
            sel_out.copy_(rows)
        norm_p = SELECT_GIVEN
    carry_rows, carry_mu = None, 1.0
    if carry is not None:
        carry_rows, carry_mu = carry
    if carry_rows is not None:
        _cuda(carry_rows, "carry rows")
        if carry_rows.dtype != torch.int32 or tuple(carry_rows.shape) != shape or not carry_rows.is_contiguous():
            raise ValueError(f"carry rows must be contiguous int32 of shape {shape}")
    T, flat, rarr, nr = _abc_arrays(abc, restart_after)
    need = workspace_bytes_step(batch, n, m, f_num, f_den, norm_p, compute, nr)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=M.device)
    if hyper is not None:
        _cuda(hyper, "hyper")
        if hyper.dtype != torch.float32 or hyper.numel() < 3 or not hyper.is_contiguous():
            raise ValueError("hyper must be a contiguous fp32 device tensor {mu, eta, wd}")
        if events is not None:
            raise ValueError("events and hyper cannot be combined")
        if carrying:
            rc = lib().dion3_step_dev_carry(batch, n, m, _ptr(W), _ptr(M), _ptr(G), _dt(G), f_num, f_den,
                                            _ptr(hyper), int(bool(decay)), norm_p, T, flat, rarr, nr, float(eps),
                                            _dtype_code(compute), _ptr(sel_out), _ptr(carry_rows), _ptr(mu_word),
                                            int(bool(defer)), _ptr(workspace), workspace.numel(), _ptr(status),
                                            _stream_ptr(M.device))
            _check(rc, "dion3_step_dev_carry")
            return sel_out
        rc = lib().dion3_step_dev(batch, n, m, _ptr(W), _ptr(M), _ptr(G), _dt(G), f_num, f_den, _ptr(hyper),
                                  int(bool(decay)), norm_p, T, flat, rarr, nr, float(eps), _dtype_code(compute),
                                  _ptr(sel_out), _ptr(workspace), workspace.numel(), _ptr(status),
                                  _stream_ptr(M.device))
        _check(rc, "dion3_step_dev")
    elif carrying:
        evs = list(events) if events is not None else []
        handles = (_c_p * max(len(evs), 1))(*[ctypes.c_void_p(e.cuda_event) for e in evs])
        rc = lib().dion3_step_carry(batch, n, m, _ptr(W), _ptr(M), _ptr(G), _dt(G), f_num, f_den, float(mu),
                                    float(eta), float(wd), norm_p, T, flat, rarr, nr, float(eps),
                                    _dtype_code(compute), _ptr(sel_out), _ptr(carry_rows), float(carry_mu),
                                    int(bool(defer)), _ptr(workspace), workspace.numel(), _ptr(status),
                                    _stream_ptr(M.device), handles, len(evs))
        _check(rc, "dion3_step_carry")
    elif events is None:
        rc = lib().dion3_step(batch, n, m, _ptr(W), _ptr(M), _ptr(G), _dt(G), f_num, f_den, float(mu), float(eta),
                              float(wd), norm_p, T, flat, rarr, nr, float(eps), _dtype_code(compute), _ptr(sel_out),
                              _ptr(workspace), workspace.numel(), _ptr(status), _stream_ptr(M.device))
        _check(rc, "dion3_step")
    else:
        handles = (_c_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        rc = lib().dion3_step_timed(batch, n, m, _ptr(W), _ptr(M), _ptr(G), _dt(G), f_num, f_den, float(mu),
                                    float(eta), float(wd), norm_p, T, flat, rarr, nr, float(eps),
                                    _dtype_code(compute), _ptr(sel_out), _ptr(workspace), workspace.numel(),
                                    _ptr(status), _stream_ptr(M.device), handles, len(events))
        _check(rc, "dion3_step_timed")
    return sel_out


def decay_rows(M: torch.Tensor, rows: torch.Tensor, mu: float) -> None:
    """M[b, rows[b, j], :] *= mu (fp32, one rounding): applies a decay that ``step(defer=True)``
    left pending.  M is [batch, n, m] (or [n, m]) contiguous fp32, rows int32 [batch, k] (or [k])."""
    _cuda(M, "M")
    _cuda(rows, "rows")
    if M.dtype != torch.float32 or not M.is_contiguous():
        raise ValueError("M must be contiguous fp32")
    if rows.dtype != torch.int32 or not rows.is_contiguous() or rows.dim() != M.dim() - 1:
        raise ValueError("rows must be contiguous int32 with one dimension fewer than M")
    batch, n, m, _, _ = _layout(M)
    k = rows.shape[-1]
    if M.dim() == 3 and rows.shape[0] != batch:
        raise ValueError("rows must have one row list per matrix")
    rc = lib().dion3_decay_rows(batch, n, m, _ptr(M), _ptr(rows), k, float(mu), _stream_ptr(M.device))
    _check(rc, "dion3_decay_rows")


def workspace_bytes_step_cols(batch: int, m: int, n: int, f_num: int, f_den: int, norm_p: int, compute,
                              n_restart: int) -> int:
    return int(lib().dion3_step_cols_workspace_bytes(batch, m, n, f_num, f_den, norm_p, _dtype_code(compute),
                                                     n_restart))


def step_cols(W: torch.Tensor, M: torch.Tensor, G: torch.Tensor, f=(1, 4), mu: float = 0.95, eta: float = 0.01,
              wd: float = 0.0, norm_p: int = 1, abc=None, restart_after=(2,), eps: float = 1e-7,
              compute=torch.float16, sel_out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
              status: torch.Tensor | None = None, cols: torch.Tensor | None = None) -> torch.Tensor:
    """One Dion3 step on [batch, m, n] (or [m, n]) contiguous W, M (fp32) and G stored with the
    short side n as columns (n <= m); selects k = ceil(f n) columns and returns them.  ``cols``:
    optional caller-chosen columns, int32 [batch, k] ascending."""
    for t, name in ((W, "W"), (M, "M"), (G, "G")):
        _cuda(t, name)
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if W.dtype != torch.float32 or M.dtype != torch.float32:
        raise TypeError("W and M are fp32 state")
    if W.shape != M.shape or G.shape != M.shape:
        raise ValueError("W, M, G must have the same shape")
    batch = 1 if M.dim() == 2 else M.shape[0]
    m, n = M.shape[-2], M.shape[-1]
    f_num, f_den = f
    k = k_of(n, f_num, f_den)
    if k < 0:
        raise ValueError("need 0 < f <= 1")
    shape = (k,) if M.dim() == 2 else (batch, k)
    if sel_out is None:
        sel_out = torch.empty(shape, dtype=torch.int32, device=M.device)
    if cols is not None:
        _cuda(cols, "cols")
        if cols.dtype != torch.int32 or tuple(cols.shape) != shape:
            raise ValueError(f"cols must be int32 of shape {shape}")
        if cols.data_ptr() != sel_out.data_ptr():
            sel_out.copy_(cols)
        norm_p = SELECT_GIVEN
    T, flat, rarr, nr = _abc_arrays(abc, restart_after)
    need = workspace_bytes_step_cols(batch, m, n, f_num, f_den, norm_p, compute, nr)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=M.device)
    rc = lib().dion3_step_cols(batch, m, n, _ptr(W), _ptr(M), _ptr(G), _dt(G), f_num, f_den, float(mu), float(eta),
                               float(wd), norm_p, T, flat, rarr, nr, float(eps), _dtype_code(compute), _ptr(sel_out),
                               _ptr(workspace), workspace.numel(), _ptr(status), _stream_ptr(M.device))
    _check(rc, "dion3_step_cols")
    return sel_out


def selftest_watchdog(spin_limit_cycles: int, status: torch.Tensor) -> None:
    _cuda(status, "status")
    rc = lib().dion3_selftest_watchdog(int(spin_limit_cycles), _ptr(status), _stream_ptr(status.device))
    _check(rc, "dion3_selftest_watchdog")


def gram_core_launch_count(T: int, restart_after=(), n: int | None = None, compute=torch.float16) -> int:
    """Kernel launches of the Gram Newton-Schulz product chain (mirrors the library's driver).

    n x n Gram matrices with n <= 128 and 16-bit iterates: R_0, one fused launch per restart
    segment, the restart's Q X and X X^T, and the final Q X.  Otherwise: R_0; per iteration Z,
    Q Z (not right after a (re)start), then either the restart's Q X and X X^T or, before the
    last iteration, the two R-update products; finally Q X."""
    rs = sorted(set(int(r) for r in restart_after))
    if n is not None and n <= 128 and compute != torch.float32 and \
            all(b - a <= 32 for a, b in zip([0] + rs, rs + [T])):
        return 1 + (len(rs) + 1) + 2 * len(rs) + 1
    count, q_identity = 1, True
    for t in range(1, T + 1):
        count += 1
        if q_identity:
            q_identity = False
        else:
            count += 1
        if t in rs:
            count += 2
            q_identity = True
        elif t < T:
            count += 2
    return count + 1


def step_launch_count(T: int, restart_after=(), k: int | None = None, compute=torch.float16,
                      carry: bool = False) -> int:
    """Kernel launches of one dion3_step call (k selected rows): momentum pass, selection, gather,
    product chain; with a carried decay, the per-row flag pass before the momentum pass."""
    return 3 + int(bool(carry)) + gram_core_launch_count(T, restart_after, k, compute)


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024  # DION3_NOALLOC_SCRATCH_BYTES in include/dion3.h


def gram_ns_noalloc(X: torch.Tensor, abc, restart_after=(), eps: float = 1e-7, compute=torch.float16,
                    out: torch.Tensor | None = None, out_dtype=None, status: torch.Tensor | None = None) -> torch.Tensor:
    """Gram Newton-Schulz without a caller workspace, for callers that may not allocate device
    memory: the library uses its own fixed scratch array (NOALLOC_SCRATCH_BYTES per GPU).  The
    output tensor must be provided when the caller cannot allocate; when ``out`` is None this
    wrapper allocates it (for convenience in tests and scripts).  Calls share the scratch array,
    so calls whose work overlaps on the GPU must be serialised."""
    _cuda(X, "X")
    batch, n, m, ldx, sx = _layout(X)
    odt = (torch.float32 if compute == torch.float32 else X.dtype) if out_dtype is None else out_dtype
    if out is None:
        out = _empty_aligned(tuple(X.shape), odt, X.device)
    _, _, _, ldo, so = _layout(_cuda(out, "out"))
    T, flat, rarr, nr = _abc_arrays(abc, restart_after)
    rc = lib().dion3_gram_ns_noalloc(batch, n, m, _ptr(X), ldx, sx, _dt(X), _ptr(out), ldo, so, _dt(out), T, flat,
                                     rarr, nr, float(eps), _dtype_code(compute), _ptr(status), _stream_ptr(X.device))
    _check(rc, "dion3_gram_ns_noalloc")
    return out
