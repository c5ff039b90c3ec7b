"""The C-ABI library builds for sm_103a, loads, and exports every entry point that
include/g3h.h declares; argument validation that happens before any CUDA call works on a
machine without a GPU. No compute calls here."""
import ctypes
import os
import re

import numpy as np
import pytest

from bn254_scalar_field_gb300 import build, g3h, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return g3h.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "g3h.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(g3h_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_entry_points():
    assert set(_declared()) == set(g3h.ENTRY_POINTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_no_compute_symbols_missing_and_no_cpu_fallback():
    # the binding has no path that computes without the library
    src = open(os.path.join(ROOT, "bn254_scalar_field_gb300", "g3h.py")).read()
    assert "oracle" not in src


def test_strerror(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert g3h.strerror(code) != "unknown error"
    assert g3h.strerror(-99) == "unknown error"


def test_header_constants_match_the_binding():
    text = open(os.path.join(ROOT, "include", "g3h.h")).read()
    consts = dict(re.findall(r"#define (G3H_\w+) \(?(-?(?:0x)?[0-9a-f]+)u?\)?", text))
    for name, value in consts.items():
        assert getattr(g3h, name) == int(value, 0), name
    assert "G3H_E_POINT" in consts and "G3H_MSM_MAX_LOG" in consts


def _rc(L, log_n, n_wires, A, B):
    keep = []

    def csr(m):
        if m is None:
            return None
        rp, col, val = (np.ascontiguousarray(x, dtype=np.uint32) for x in m)
        s = g3h.g3h_csr(rp.shape[0] - 1, rp.ctypes.data, col.ctypes.data if col.size else None,
                        val.ctypes.data if val.size else None)
        keep.extend([rp, col, val, s])
        return ctypes.byref(s)

    out = ctypes.c_void_p()
    return L.g3h_prepare(log_n, n_wires, csr(A), csr(B), 0, None, ctypes.byref(out))


def test_prepare_validation_before_cuda(L):
    A, B, w = synth.problem(4, seed=3)
    assert _rc(L, 28, 16, A, B) == g3h.G3H_E_RANGE
    assert _rc(L, 4, 16, A, None) == g3h.G3H_E_INVAL
    assert L.g3h_prepare(4, 16, None, None, 0, None, None) == g3h.G3H_E_INVAL
    # row_ptr not starting at 0
    bad = (A[0] + 1, A[1], A[2])
    assert _rc(L, 4, 16, bad, B) == g3h.G3H_E_RANGE
    # non-monotone row_ptr
    rp = A[0].copy()
    i = int(np.argmax(np.diff(rp.astype(np.int64)) > 0))
    rp[i + 1] = rp[i] - 1 if rp[i] > 0 else rp[i]
    if rp[i + 1] < rp[i]:
        assert _rc(L, 4, 16, (rp, A[1], A[2]), B) == g3h.G3H_E_RANGE
    # column index out of range
    col = A[1].copy()
    col[0] = 16
    assert _rc(L, 4, 16, (A[0], col, A[2]), B) == g3h.G3H_E_RANGE
    # coefficient >= r
    val = A[2].copy()
    val[0] = synth.MODULUS_LIMBS
    assert _rc(L, 4, 16, (A[0], A[1], val), B) == g3h.G3H_E_NONCANON
    # more rows than the domain
    big = synth.problem(5, seed=1)[0]
    assert _rc(L, 4, 32, big, big) == g3h.G3H_E_INVAL


def test_null_context_calls(L):
    assert L.g3h_sync(None) == g3h.G3H_E_INVAL
    assert L.g3h_compute_h(None, None, None, None, 0) == g3h.G3H_E_INVAL
    assert L.g3h_ntt(None, None, 0, 0, 0) == g3h.G3H_E_INVAL
    assert L.g3h_info(None, None, None) == g3h.G3H_E_INVAL
    assert L.g3h_mont_to_std(None, None, None, 0, 0) == g3h.G3H_E_INVAL
    assert L.g3h_msm_prepare(None, None, 0, 0) == g3h.G3H_E_INVAL
    assert L.g3h_msm(None, None, 0, None, 0) == g3h.G3H_E_INVAL
    L.g3h_destroy(None)
