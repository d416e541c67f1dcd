"""Host-only checks of the C ABI: the library loads, exports every symbol the header
declares, and rejects bad arguments synchronously (before touching the GPU)."""

import ctypes
import os
import re

import pytest

import matrix_orthogonalizing_optimizer_syrk_gb300 as d3
from matrix_orthogonalizing_optimizer_syrk_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dion3.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return d3.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dion3_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for required in ["dion3_sym_gemm", "dion3_gram_ns", "dion3_step", "dion3_k", "dion3_status_str",
                     "dion3_gram_ns_workspace_bytes", "dion3_step_workspace_bytes"]:
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), f"libdion3.so does not export {name}"
        assert name in d3.SIGNATURES, f"binding does not declare {name}"


def test_abi_version(L):
    assert L.dion3_abi_version() == 1


@pytest.mark.parametrize("n,fn,fd,k", [(4096, 1, 4, 1024), (768, 1, 8, 96), (10, 1, 3, 4), (7, 1, 1, 7),
                                        (0, 1, 4, 0), (5, 0, 1, -1), (5, 2, 1, -1), (5, 1, 0, -1), (-1, 1, 2, -1)])
def test_k(L, n, fn, fd, k):
    assert d3.k_of(n, fn, fd) == k


def test_status_strings(L):
    for code in range(6):
        assert d3.status_str(code).startswith("DION3_")


NULL = ctypes.c_void_p(0)
FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: validation fails first
FAKE_ODD = ctypes.c_void_p(0x10008)   # 8-byte aligned only


def _sym(L, batch=1, n=64, k=64, A=FAKE, lda=64, B=NULL, C=NULL, D=FAKE, ldd=64, beta=0.0, it=0, ot=0):
    return L.dion3_sym_gemm(batch, n, k, A, lda, n * lda, B, lda, n * lda, C, ldd, n * ldd, D, ldd, n * ldd,
                            1.0, beta, 0.0, it, ot, NULL, NULL)


def test_sym_gemm_validation(L):
    assert _sym(L, n=-1) == 1
    assert _sym(L, A=NULL) == 1
    assert _sym(L, D=NULL) == 1
    assert _sym(L, beta=1.0) == 1               # C missing
    assert _sym(L, lda=32) == 1                 # lda < k
    assert _sym(L, ldd=32) == 1                 # ldd < n
    assert _sym(L, it=2, ot=0) == 2             # fp32 in, bf16 out
    assert _sym(L, it=0, ot=1) == 2             # bf16 in, fp16 out
    assert _sym(L, it=7) == 1
    assert _sym(L, A=FAKE_ODD) == 5
    assert _sym(L, lda=68) == 5                 # 136 bytes: not a multiple of 16
    assert _sym(L, n=0) == 0                    # empty: nothing to do
    assert _sym(L, batch=0) == 0


def _abc(T=5):
    return (ctypes.c_float * (3 * T))(*([3.4445, -4.7750, 2.0315] * T))


def _gram(L, n=64, m=128, X=FAKE, ldx=128, Out=FAKE, ldo=128, T=5, abc=None, rs=(2,), ws=FAKE, wsb=1 << 40,
          xt=0, ot=0, ct=0, eps=1e-7):
    abc = _abc(T) if abc is None else abc
    r = (ctypes.c_int * max(1, len(rs)))(*rs)
    return L.dion3_gram_ns(1, n, m, X, ldx, n * ldx, xt, Out, ldo, n * ldo, ot, T, abc, r, len(rs), eps, ct,
                           ws, wsb, NULL, NULL)


def test_gram_ns_validation(L):
    assert _gram(L, n=200, m=100, ldx=100, ldo=104) == 1     # n > m
    assert _gram(L, T=0) == 1
    assert _gram(L, rs=(0,)) == 1
    assert _gram(L, rs=(5,)) == 1
    assert _gram(L, rs=(3, 2)) == 1
    assert _gram(L, rs=(2, 2)) == 1
    assert _gram(L, X=NULL) == 1
    assert _gram(L, eps=-1.0) == 1
    assert _gram(L, ws=NULL) == 3
    assert _gram(L, wsb=16) == 3
    assert _gram(L, Out=FAKE_ODD) == 5
    # a misaligned X of the compute dtype needs the copy buffer the query did not reserve
    no_copy = d3.workspace_bytes_gram_ns(1, 64, 128, 0, 0, 1)
    assert _gram(L, X=FAKE_ODD, wsb=no_copy) == 3
    assert _gram(L, ldx=132, wsb=no_copy) == 3              # 264-byte rows: copied, too
    assert _gram(L, ct=2, ot=0) == 2                         # fp32 compute needs fp32 output
    nan_abc = (ctypes.c_float * 15)(*([float("nan")] * 15))
    assert _gram(L, abc=nan_abc) == 1


def _gram_pair(L, batch=1, n=64, m=128, X=FAKE, ldx=128, Out=FAKE, ldo=128, T=5, abc=None, rs=(2,), xt=0, ot=0,
               ct=0, eps=1e-7, wsb=1 << 40):
    """The same call through dion3_gram_ns (ample fake workspace) and dion3_gram_ns_noalloc."""
    abc = _abc(T) if abc is None else abc
    r = (ctypes.c_int * max(1, len(rs)))(*rs)
    a = L.dion3_gram_ns(batch, n, m, X, ldx, n * ldx, xt, Out, ldo, n * ldo, ot, T, abc, r, len(rs), eps, ct,
                        FAKE, wsb, NULL, NULL)
    b = L.dion3_gram_ns_noalloc(batch, n, m, X, ldx, n * ldx, xt, Out, ldo, n * ldo, ot, T, abc, r, len(rs), eps,
                                ct, NULL, NULL)
    return a, b


def test_noalloc_returns_the_same_codes_as_the_workspace_entry_point(L):
    """Bad and empty calls get the same code from both Gram NS entry points (nothing reaches the
    GPU: every case fails or finishes in the argument checks)."""
    nan_abc = (ctypes.c_float * 15)(*([float("nan")] * 15))
    cases = [dict(n=200, m=100, ldx=100, ldo=104), dict(T=0), dict(rs=(0,)), dict(rs=(5,)), dict(rs=(3, 2)),
             dict(X=NULL), dict(Out=NULL), dict(eps=-1.0), dict(Out=FAKE_ODD), dict(ct=2, ot=0), dict(abc=nan_abc),
             dict(xt=7), dict(ct=9), dict(ldx=100), dict(batch=-1),
             # empty problems: OK from both, even with a bad schedule or dtype left unchecked by neither
             dict(batch=0), dict(n=0), dict(batch=0, n=200, m=100), dict(batch=0, T=0), dict(batch=0, ct=2, ot=0)]
    for kw in cases:
        a, b = _gram_pair(L, **kw)
        assert a == b, f"{kw}: dion3_gram_ns -> {a}, dion3_gram_ns_noalloc -> {b}"
        assert a != 3, kw


def test_noalloc_rejects_oversized_problems_on_the_host(L):
    """Beyond DION3_NOALLOC_SCRATCH_BYTES: DION3_EWORKSPACE before the GPU is touched -- also when
    only the copy that a misaligned X needs pushes the workspace over the limit."""
    cap = d3.NOALLOC_SCRATCH_BYTES
    assert _gram_pair(L, batch=8, n=1024, m=4096, ldx=4096, ldo=4096, rs=(2, 4))[1] == 3
    # find an aligned problem that fits, whose copied (misaligned-X) variant does not
    n, m = 512, 4096
    batch = 1
    while d3.workspace_bytes_gram_ns(batch + 1, n, m, 0, 0, 1) <= cap:
        batch += 1
    fits = d3.workspace_bytes_gram_ns(batch, n, m, 0, 0, 1)
    copied = d3.workspace_bytes_gram_ns(batch, n, m, 0, 1, 1)   # bf16 X, fp16 compute: copied
    assert fits <= cap < copied
    assert _gram_pair(L, batch=batch, n=n, m=m, ldx=m, ldo=m, X=FAKE_ODD, rs=(2,))[1] == 3
    assert _gram_pair(L, batch=batch, n=n, m=m, ldx=m, ldo=m, xt=0, ct=1, rs=(2,))[1] == 3


def test_workspace_queries(L):
    small = d3.workspace_bytes_gram_ns(1, 64, 128, 0, 0, 1)
    big = d3.workspace_bytes_gram_ns(2, 64, 128, 0, 0, 1)
    more_r = d3.workspace_bytes_gram_ns(1, 64, 128, 0, 0, 2)
    copy = d3.workspace_bytes_gram_ns(1, 64, 128, 2, 0, 1)
    assert 0 < small < big and small < more_r and small < copy
    assert small % 256 == 0
    assert d3.workspace_bytes_gram_ns(1, 65, 64, 0, 0, 1) == 0   # n > m
    s1 = d3.workspace_bytes_step(2, 64, 128, 1, 4, 1, 0, 2)
    s2 = d3.workspace_bytes_step(2, 64, 128, 1, 2, 1, 0, 2)
    s3 = d3.workspace_bytes_step(2, 64, 128, 1, 4, 2, 0, 2)
    assert 0 < s1 < s2 and s1 < s3
    assert d3.workspace_bytes_step(2, 64, 128, 0, 4, 1, 0, 2) == 0


def _step(L, n=64, m=128, W=FAKE, M=FAKE, G=FAKE, sel=FAKE, fn=1, fd=4, p=1, T=5, rs=(2,), ws=FAKE,
          wsb=1 << 40, mu=0.95):
    r = (ctypes.c_int * max(1, len(rs)))(*rs)
    return L.dion3_step(1, n, m, W, M, G, 0, fn, fd, mu, 0.01, 0.0, p, T, _abc(T), r, len(rs), 1e-7, 0, sel, ws,
                        wsb, NULL, NULL)


def test_step_validation(L):
    assert _step(L, fn=0) == 1
    assert _step(L, fn=5, fd=4) == 1
    assert _step(L, p=3) == 1
    assert _step(L, W=NULL) == 1
    assert _step(L, sel=NULL) == 1
    assert _step(L, n=129, m=128) == 1
    assert _step(L, n=20000, m=20000) == 2
    assert _step(L, M=FAKE_ODD) == 5
    assert _step(L, ws=NULL) == 3
    assert _step(L, mu=float("nan")) == 1
    assert _step(L, rs=(9,)) == 1


def _ns(L, n=64, m=128, X=FAKE, ldx=128, Out=FAKE, ldo=128, T=5, abc=None, ws=FAKE, wsb=1 << 40, xt=0, ot=0, ct=0,
        eps=1e-7, batch=1):
    abc = _abc(T) if abc is None else abc
    return L.dion3_ns_standard(batch, n, m, X, ldx, n * ldx, xt, Out, ldo, n * ldo, ot, T, abc, eps, ct, ws, wsb,
                               NULL, NULL)


def test_ns_standard_validation(L):
    assert _ns(L, n=200, m=100, ldx=100, ldo=104) == 1     # n > m
    assert _ns(L, T=0) == 1
    assert _ns(L, X=NULL) == 1
    assert _ns(L, Out=NULL) == 1
    assert _ns(L, ldo=64) == 1                              # ldo < m
    assert _ns(L, eps=float("nan")) == 1
    assert _ns(L, ws=NULL) == 3
    assert _ns(L, wsb=16) == 3
    assert _ns(L, Out=FAKE_ODD) == 5
    assert _ns(L, ldo=132) == 5                             # 264-byte rows of bf16
    assert _ns(L, ct=2, ot=0) == 2                          # fp32 compute needs fp32 output
    assert _ns(L, xt=9) == 1
    nan_abc = (ctypes.c_float * 15)(*([float("nan")] * 15))
    assert _ns(L, abc=nan_abc) == 1
    assert _ns(L, n=0) == 0
    assert _ns(L, batch=0) == 0


def test_ns_standard_workspace_query(L):
    a = d3.workspace_bytes_ns_standard(1, 64, 128, 0)
    b = d3.workspace_bytes_ns_standard(2, 64, 128, 0)
    c = d3.workspace_bytes_ns_standard(1, 64, 128, 2)
    assert 0 < a < b and a < c and a % 256 == 0
    assert d3.workspace_bytes_ns_standard(1, 65, 64, 0) == 0


def test_step_dev_validation(L):
    hyper = FAKE
    r = (ctypes.c_int * 1)(2)

    def call(hyper=hyper, **kw):
        args = dict(n=64, m=128, W=FAKE, M=FAKE, G=FAKE, sel=FAKE, fn=1, fd=4, ws=FAKE, wsb=1 << 40)
        args.update(kw)
        return L.dion3_step_dev(1, args["n"], args["m"], args["W"], args["M"], args["G"], 0, args["fn"], args["fd"],
                                hyper, 1, 1, 5, _abc(5), r, 1, 1e-7, 0, args["sel"], args["ws"], args["wsb"],
                                NULL, NULL)

    assert call(hyper=NULL) == 1
    assert call(hyper=ctypes.c_void_p(0x10002)) == 5      # not 4-byte aligned
    assert call(fn=0) == 1
    assert call(W=NULL) == 1
    assert call(ws=NULL) == 3
    assert call(n=0) == 0


def test_given_selection_mode_accepted(L):
    """norm_p = DION3_SELECT_GIVEN passes validation (nothing launched: workspace too small)."""
    assert _step(L, p=0, wsb=16) == 3
    assert _step(L, p=3) == 1
    assert d3.workspace_bytes_step(2, 64, 128, 1, 4, 0, 0, 2) > 0
    assert d3.workspace_bytes_step(2, 64, 128, 1, 4, 0, 0, 2) < d3.workspace_bytes_step(2, 64, 128, 1, 4, 1, 0, 2)


def test_step_cols_validation(L):
    r = (ctypes.c_int * 1)(2)

    def call(batch=1, m=128, n=64, W=FAKE, ws=FAKE, wsb=1 << 40, p=1):
        return L.dion3_step_cols(batch, m, n, W, FAKE, FAKE, 0, 1, 4, 0.95, 0.01, 0.0, p, 5, _abc(5), r, 1, 1e-7, 0,
                                 FAKE, ws, wsb, NULL, NULL)

    assert call(m=32, n=64) == 1          # n > m
    assert call(W=NULL) == 1
    assert call(ws=NULL) == 3
    assert call(p=3) == 1
    assert call(batch=70000, wsb=16) == 2
    assert d3.workspace_bytes_step_cols(2, 128, 64, 1, 4, 1, 0, 2) > d3.workspace_bytes_step(2, 64, 128, 1, 4, 1, 0, 2)


def test_step_carry_validation(L):
    """dion3_step_carry rejects a bad carried decay before any launch."""
    r = (ctypes.c_int * 1)(2)
    SEL = ctypes.c_void_p(0x20000)

    def call(carry=FAKE, cmu=0.95, defer=1, p=1, sel=SEL, ws=FAKE, wsb=1 << 40, n_events=0):
        return L.dion3_step_carry(1, 64, 128, FAKE, FAKE, FAKE, 0, 1, 4, 0.95, 0.01, 0.0, p, 5, _abc(5), r, 1,
                                  1e-7, 0, sel, carry, cmu, defer, ws, wsb, NULL, NULL, None, n_events)

    assert call(cmu=float("nan")) == 1
    assert call(cmu=float("inf")) == 1
    assert call(carry=ctypes.c_void_p(0x10002)) == 5      # int32 list not 4-byte aligned
    assert call(p=0, carry=SEL) == 1                       # S given in sel_out: cannot also be the carried list
    assert call(p=0, carry=FAKE, ws=NULL) == 3             # a separate carried list is fine with a given S
    assert call(carry=SEL, ws=NULL) == 3                   # aliasing sel_out is fine with computed keys
    assert call(carry=NULL, defer=0, ws=NULL) == 3
    assert call(n_events=-1) == 1
    assert call(carry=NULL, cmu=float("nan"), wsb=16) == 3  # carry_mu is unused without a list


def test_decay_rows_validation(L):
    assert L.dion3_decay_rows(-1, 8, 8, FAKE, FAKE, 2, 0.9, NULL) == 1
    assert L.dion3_decay_rows(1, 8, 8, FAKE, FAKE, 9, 0.9, NULL) == 1        # k > n
    assert L.dion3_decay_rows(1, 8, 8, FAKE, FAKE, 2, float("nan"), NULL) == 1
    assert L.dion3_decay_rows(1, 8, 8, NULL, FAKE, 2, 0.9, NULL) == 1
    assert L.dion3_decay_rows(1, 8, 8, FAKE, NULL, 2, 0.9, NULL) == 1
    assert L.dion3_decay_rows(1, 8, 8, ctypes.c_void_p(0x10002), FAKE, 2, 0.9, NULL) == 5
    assert L.dion3_decay_rows(1, 8, 8, FAKE, ctypes.c_void_p(0x10001), 2, 0.9, NULL) == 5
    assert L.dion3_decay_rows(0, 8, 8, NULL, NULL, 2, 0.9, NULL) == 0        # nothing to do
    assert L.dion3_decay_rows(1, 8, 8, NULL, NULL, 0, 0.9, NULL) == 0


def test_carry_adds_one_launch():
    base = d3.step_launch_count(5, (2, 4), 1024)
    assert d3.step_launch_count(5, (2, 4), 1024, carry=True) == base + 1


def test_step_dev_carry_validation(L):
    r = (ctypes.c_int * 1)(2)
    SEL = ctypes.c_void_p(0x20000)
    MU = ctypes.c_void_p(0x30000)

    def call(hyper=FAKE, carry=SEL, mu=MU, defer=1, p=1, ws=FAKE, wsb=1 << 40):
        return L.dion3_step_dev_carry(1, 64, 128, FAKE, FAKE, FAKE, 0, 1, 4, hyper, 0, p, 5, _abc(5), r, 1, 1e-7, 0,
                                      SEL, carry, mu, defer, ws, wsb, NULL, NULL)

    assert call(hyper=NULL) == 1
    assert call(mu=NULL) == 1                              # a carried list needs the mu word
    assert call(carry=NULL, mu=NULL) == 1                  # so does defer
    assert call(carry=NULL, mu=NULL, defer=0, ws=NULL) == 3  # neither: the plain device step
    assert call(mu=ctypes.c_void_p(0x30002)) == 5
    assert call(p=0) == 1                                  # given S in sel_out cannot be the carried list
    assert call(ws=NULL) == 3


def _declared_signatures():
    """name -> list of parameter type strings, from the header's prototypes."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"\b[\w\s\*]+?\b(dion3_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = " ".join(m.group(2).split())
        if params in ("", "void"):
            out[m.group(1)] = []
        else:
            out[m.group(1)] = [p.strip() for p in params.split(",")]
    return out


def _ctype_kind(t):
    if t in (ctypes.c_float,):
        return "float"
    if t in (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_longlong):
        return "int"
    return "ptr"


def _decl_kind(p):
    if "*" in p:
        return "ptr"
    if p.startswith("float"):
        return "float"
    return "int"


def test_binding_signatures_match_header():
    """Every prototype in the header has the binding's argument count and kinds (pointer, integer,
    float), so a change on one side cannot silently shift the other's arguments."""
    decl = _declared_signatures()
    assert set(decl) == set(_declared_functions())
    for name, params in decl.items():
        _, args = d3.SIGNATURES[name]
        assert len(args) == len(params), f"{name}: header has {len(params)} parameters, binding {len(args)}"
        for i, (p, a) in enumerate(zip(params, args)):
            assert _decl_kind(p) == _ctype_kind(a), f"{name} argument {i} ({p}): binding declares {a}"


def test_checked_build_loads_and_reports_itself():
    """The range-checked variant (DION3_RANGE_CHECKS=1) exports the same symbols and reports 1 from
    dion3_range_checks; the default build reports 0."""
    path = _build.build(checked=True)
    assert path.endswith("libdion3_checked.so")
    Lc = ctypes.CDLL(path)
    for name in _declared_functions():
        assert hasattr(Lc, name), f"libdion3_checked.so does not export {name}"
    Lc.dion3_range_checks.restype = ctypes.c_int
    assert Lc.dion3_range_checks() == 1
    assert d3.lib().dion3_range_checks() == 0
    # argument validation is the same code in both builds
    Lc.dion3_k.restype = ctypes.c_int
    assert Lc.dion3_k(4096, 1, 4) == 1024
