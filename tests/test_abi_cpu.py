"""C-ABI checks that need no GPU: the library loads, exports every entry point
that include/muon.h declares, and rejects bad arguments before any CUDA call.
(Pointers here are fake addresses: validation never dereferences them.)"""
import ctypes
import os
import re

import pytest

import muon_newton_schulz_step_gb300 as mg
from muon_newton_schulz_step_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, CUDA, OOM, TIMEOUT, CORRUPT = range(7)


@pytest.fixture(scope="module")
def L():
    cuda_build.build()
    return mg.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "muon.h")) as f:
        text = f.read()
    return set(re.findall(r"MUON_API\s+[\w\s\*]+?\b(muon_\w+)\s*\(", text))


def test_library_exports_every_declared_symbol(L):
    declared = _declared()
    assert declared == set(mg.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def _arr(ctype, vals):
    return (ctype * max(1, len(vals)))(*vals)


def _step(L, W, G, M, rows, cols, count=None, lr=0.02, mu=0.95, wd=0.1):
    n = len(rows) if count is None else count
    vp = ctypes.c_void_p
    return L.muon_step(_arr(vp, W), _arr(vp, G), _arr(vp, M), _arr(ctypes.c_int, rows),
                       _arr(ctypes.c_int, cols), n, lr, mu, wd, None)


def _ns(L, P, rows, cols, steps=5, count=None):
    n = len(rows) if count is None else count
    return L.muon_ns5_batched(_arr(ctypes.c_void_p, P), _arr(ctypes.c_int, rows),
                              _arr(ctypes.c_int, cols), n, steps, None, None)


def test_count_zero_is_a_noop(L):
    assert _step(L, [], [], [], [], [], count=0) == OK
    assert _ns(L, [], [], [], count=0) == OK


def test_invalid_arguments_are_rejected(L):
    A = 1 << 20
    good = dict(W=[A], G=[2 * A], M=[3 * A], rows=[64], cols=[256])
    assert _step(L, **good, count=-1) == INVALID
    assert _step(L, [A], [2 * A], [3 * A], [0], [256]) == INVALID
    assert _step(L, [A], [2 * A], [3 * A], [64], [40000]) == INVALID
    assert _step(L, [A + 8], [2 * A], [3 * A], [64], [256]) == INVALID      # misaligned W
    assert _step(L, [A], [0], [3 * A], [64], [256]) == INVALID              # NULL G
    assert _step(L, [A], [A], [3 * A], [64], [256]) == INVALID              # W aliases G
    assert _step(L, [A], [2 * A], [A + 4096], [64], [256]) == INVALID       # M overlaps W
    assert _step(L, **good, lr=float("nan")) == INVALID
    assert _step(L, **good, wd=float("inf")) == INVALID
    # two matrices whose buffers overlap (each is 64 * 256 * 2 bytes)
    assert _ns(L, [A, A + 64 * 256], [64, 64], [256, 256]) == INVALID
    assert b"overlap" in L.muon_last_error()
    assert _ns(L, [A], [64], [256], steps=-1) == INVALID
    assert _ns(L, [A], [64], [256], steps=65) == INVALID
    assert L.muon_ns5_batched(None, _arr(ctypes.c_int, [1]), _arr(ctypes.c_int, [1]), 1, 5, None,
                              None) == INVALID


def test_step_ex_option_validation(L):
    A = 1 << 20
    vp = ctypes.c_void_p
    o = mg._Opts()
    L.muon_step_opts_init(ctypes.byref(o))
    assert (o.w_dtype, o.g_dtype, o.steps, o.nesterov) == (0, 0, 5, 1)
    assert abs(o.eps - 1e-7) < 1e-12 and not o.workspace and not o.o_out
    args = (_arr(vp, [A]), _arr(vp, [2 * A]), _arr(vp, [3 * A]), _arr(ctypes.c_int, [8]),
            _arr(ctypes.c_int, [8]), 1, 0.02, 0.95, 0.1)
    for field, val in [("w_dtype", 7), ("g_dtype", -1), ("steps", 100), ("nesterov", 2)]:
        bad = mg._Opts()
        L.muon_step_opts_init(ctypes.byref(bad))
        setattr(bad, field, val)
        assert L.muon_step_ex(*args, ctypes.byref(bad), None) == INVALID, field
    bad = mg._Opts()
    L.muon_step_opts_init(ctypes.byref(bad))
    bad.eps = -1.0
    assert L.muon_step_ex(*args, ctypes.byref(bad), None) == INVALID
    bad = mg._Opts()
    L.muon_step_opts_init(ctypes.byref(bad))
    bad.workspace = ctypes.c_void_p(A + 16)
    bad.workspace_bytes = 1 << 30
    assert L.muon_step_ex(*args, ctypes.byref(bad), None) == INVALID   # not 256-byte aligned


def test_caller_workspace_too_small_for_one_matrix(L):
    # a caller workspace smaller than the batch is used group by group; one that
    # cannot hold a single matrix is rejected before any CUDA call
    A = 1 << 28                       # fake, non-overlapping 2048 x 6144 buffers
    vp = ctypes.c_void_p
    args = (_arr(vp, [A, 5 * A]), _arr(vp, [2 * A, 6 * A]), _arr(vp, [3 * A, 7 * A]),
            _arr(ctypes.c_int, [2048, 2048]), _arr(ctypes.c_int, [6144, 6144]), 2, 0.02, 0.95, 0.1)
    o = mg._Opts()
    L.muon_step_opts_init(ctypes.byref(o))
    o.workspace = ctypes.c_void_p(1 << 34)
    o.workspace_bytes = 1 << 20
    assert L.muon_step_ex(*args, ctypes.byref(o), None) == OOM
    assert b"matrix 0 alone" in L.muon_last_error()


def test_status_strings_and_last_error(L):
    for s in range(7):
        assert L.muon_status_string(s).decode().startswith("MUON_")
    assert b"unknown" in L.muon_status_string(99)
    A = 1 << 20
    assert _step(L, [A + 8], [2 * A], [3 * A], [64], [256]) == INVALID
    assert b"W[0]" in L.muon_last_error()


def test_debug_guards_enlarge_the_workspace(monkeypatch):
    shapes = [(2048, 6144), (6144, 2048), (64, 256), (300, 700)]
    monkeypatch.delenv("MUON_DEBUG_GUARD", raising=False)
    plain = mg.muon_workspace_bytes(shapes)
    monkeypatch.setenv("MUON_DEBUG_GUARD", "1")
    guarded = mg.muon_workspace_bytes(shapes)
    # partials, sigma, small region and X0, X1, A, B of two buckets: 11 regions + 1 leading guard
    assert guarded >= plain + 12 * 4096


def test_workspace_bytes_grows_with_the_batch(L):
    one = mg.muon_workspace_bytes([(2048, 6144)])
    two = mg.muon_workspace_bytes([(2048, 6144), (6144, 2048)])
    assert one > 0 and two > one
    # X0, X1 (2048 x 6144) and A, B (2048 x 2048) in bf16 at least
    assert one >= 2 * (2 * 2048 * 6144 + 2 * 2048 * 2048)
    assert mg.muon_workspace_bytes([]) == 0
    assert mg.muon_workspace_bytes([(0, 5)]) == 0


def test_fp8_gram_flag_is_validated_before_any_work():
    import ctypes
    import muon_newton_schulz_step_gb300 as mg
    L = mg.lib()
    o = mg._Opts()
    L.muon_step_opts_init(ctypes.byref(o))
    assert o.ns_fp8_gram == 0
    o.ns_fp8_gram = 2
    one = (ctypes.c_int * 1)(4)
    ptr = (ctypes.c_void_p * 1)(16)
    rc = L.muon_step_ex(ptr, ptr, ptr, one, one, 1, 0.02, 0.95, 0.1, ctypes.byref(o), None)
    assert rc == 1 and b"ns_fp8_gram" in L.muon_last_error()
