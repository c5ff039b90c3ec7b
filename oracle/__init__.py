"""CPU oracle for the Groth16 quotient-evaluation path over BN254 Fr.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package. The library (``bn254_scalar_field_gb300``) never
does, and shares no code with it.

Two independent implementations live here:
  * ``fr_int``: pure-Python ints in standard form (small domains only);
  * ``g3h_oracle.c``: plain C with four 64-bit limbs, built by :func:`build` into
    ``oracle/_build/liboracle.so`` and called through ctypes by the wrappers below.
Array arguments are numpy uint32 arrays of shape (m, 8): eight little-endian limbs per
element, Montgomery form (R = 2^256), as the library's boundary uses.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "g3h_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force=False):
    """Compile the C oracle with gcc (-O2, portable: no -march flags). Returns the path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if force or not fresh:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        U = ctypes.c_uint
        S = ctypes.c_size_t
        L.orc_fr_mul.argtypes = [P, P, P]
        L.orc_fr_add.argtypes = [P, P, P]
        L.orc_fr_sub.argtypes = [P, P, P]
        L.orc_fr_mul_vec.argtypes = [P, P, P, S]
        L.orc_from_mont.argtypes = [P, P, S]
        L.orc_to_mont.argtypes = [P, P, S]
        L.orc_domain.argtypes = [U, P, P]
        L.orc_domain.restype = ctypes.c_int
        L.orc_ntt.argtypes = [U, P, ctypes.c_int, ctypes.c_int]
        L.orc_ntt.restype = ctypes.c_int
        L.orc_gather.argtypes = [U, S, P, P, P, P, P, P, P, P, P, P]
        L.orc_gather.restype = ctypes.c_int
        L.orc_compute_h.argtypes = [U, S, P, P, P, P, P, P, P, P, P]
        L.orc_compute_h.restype = ctypes.c_int
        L.orc_compute_h_abc.argtypes = [U, P, P, P, P, P]
        L.orc_compute_h_abc.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _fr(a):
    a = np.ascontiguousarray(a, dtype=np.uint32)
    if a.ndim != 2 or a.shape[1] != 8:
        a = a.reshape(-1, 8)
    return a


def _u32(a):
    return np.ascontiguousarray(a, dtype=np.uint32)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("oracle %s failed with %d" % (what, rc))


def fr_mul(a, b):
    a, b = _fr(a), _fr(b)
    out = np.empty_like(a)
    for i in range(a.shape[0]):
        lib().orc_fr_mul(_p(a[i]), _p(b[i]), _p(out[i]))
    return out


def fr_add(a, b):
    a, b = _fr(a), _fr(b)
    out = np.empty_like(a)
    for i in range(a.shape[0]):
        lib().orc_fr_add(_p(a[i]), _p(b[i]), _p(out[i]))
    return out


def fr_sub(a, b):
    a, b = _fr(a), _fr(b)
    out = np.empty_like(a)
    for i in range(a.shape[0]):
        lib().orc_fr_sub(_p(a[i]), _p(b[i]), _p(out[i]))
    return out


def fr_mul_vec(a, b):
    """Elementwise Montgomery product of two (m, 8) arrays."""
    a, b = _fr(a), _fr(b)
    assert a.shape == b.shape
    out = np.empty_like(a)
    lib().orc_fr_mul_vec(_p(a), _p(b), _p(out), a.shape[0])
    return out


def from_mont(a):
    a = _fr(a)
    out = np.empty_like(a)
    lib().orc_from_mont(_p(a), _p(out), a.shape[0])
    return out


def to_mont(a):
    a = _fr(a)
    out = np.empty_like(a)
    lib().orc_to_mont(_p(a), _p(out), a.shape[0])
    return out


def domain(log_n):
    """(omega_n, g) as eight-limb standard-form arrays."""
    w = np.zeros(8, np.uint32)
    g = np.zeros(8, np.uint32)
    _check(lib().orc_domain(log_n, _p(w), _p(g)), "domain")
    return w, g


def ntt(data, log_n, inverse=False, coset=False):
    """Forward: DFT_omega(x) (x_j g^j first if coset). Inverse: n^-1 DFT_omega^-1, then
    x_j g^-j if coset. Returns a new array."""
    x = _fr(data).copy()
    assert x.shape[0] == 1 << log_n
    _check(lib().orc_ntt(log_n, _p(x), int(inverse), int(coset)), "ntt")
    return x


def gather(log_n, A, B, w):
    """A, B: (row_ptr, col, val) triples. Returns a, b, c as (n, 8) arrays."""
    n = 1 << log_n
    ra, ca, va = _u32(A[0]), _u32(A[1]), _fr(A[2])
    rb, cb, vb = _u32(B[0]), _u32(B[1]), _fr(B[2])
    assert ra.shape[0] == rb.shape[0]
    w = _fr(w)
    a = np.zeros((n, 8), np.uint32)
    b = np.zeros((n, 8), np.uint32)
    c = np.zeros((n, 8), np.uint32)
    _check(lib().orc_gather(log_n, ra.shape[0] - 1, _p(ra), _p(ca), _p(va), _p(rb), _p(cb),
                            _p(vb), _p(w), _p(a), _p(b), _p(c)), "gather")
    return a, b, c


def compute_h(log_n, A, B, w):
    """The whole path. Returns (h_mont, h_std) as (n, 8) arrays."""
    n = 1 << log_n
    ra, ca, va = _u32(A[0]), _u32(A[1]), _fr(A[2])
    rb, cb, vb = _u32(B[0]), _u32(B[1]), _fr(B[2])
    assert ra.shape[0] == rb.shape[0]
    w = _fr(w)
    hm = np.zeros((n, 8), np.uint32)
    hs = np.zeros((n, 8), np.uint32)
    _check(lib().orc_compute_h(log_n, ra.shape[0] - 1, _p(ra), _p(ca), _p(va), _p(rb), _p(cb),
                               _p(vb), _p(w), _p(hm), _p(hs)), "compute_h")
    return hm, hs


def compute_h_abc(log_n, a, b, c):
    """Steps after the gather on given evaluation vectors a, b, c (Montgomery)."""
    n = 1 << log_n
    a, b, c = _fr(a), _fr(b), _fr(c)
    hm = np.zeros((n, 8), np.uint32)
    hs = np.zeros((n, 8), np.uint32)
    _check(lib().orc_compute_h_abc(log_n, _p(a), _p(b), _p(c), _p(hm), _p(hs)), "compute_h_abc")
    return hm, hs
