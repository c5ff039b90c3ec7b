"""CPU oracle for the Groth16 quotient-evaluation path over BN254 Fr.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this package. The library (``bn254_scalar_field_gb300``) never
does, and shares no code with it.

Two independent implementations live here for each part:
  * ``fr_int`` (quotient path) and ``g1_int`` (G1 multi-scalar multiplication): pure-Python
    ints in standard form (small sizes only);
  * ``g3h_oracle.c`` and ``g1_oracle.c``: plain C with four 64-bit limbs, built by
    :func:`build` into ``oracle/_build/liboracle.so`` and called through ctypes by the
    wrappers below.
Array arguments are numpy uint32 arrays of shape (m, 8): eight little-endian limbs per
element, Montgomery form (R = 2^256), as the library's boundary uses; G1 points are
(m, 16) (affine x then y, infinity all zero), MSM scalars (m, 8) in standard form.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "g3h_oracle.c"), os.path.join(_HERE, "g1_oracle.c")]
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force=False):
    """Compile the C oracle with gcc (-O2, portable: no -march flags). Returns the path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and all(
        os.path.getmtime(_LIB_PATH) >= os.path.getmtime(s) for s in _SRCS)
    if force or not fresh:
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-Wall", "-o", tmp] + _SRCS)
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
        L.orc_poly_eval.argtypes = [S, P, P, P]
        L.orc_fq_mul.argtypes = [P, P, P]
        L.orc_fq_inv.argtypes = [P, P]
        for name, args in (("orc_g1_on_curve", [P]), ("orc_g1_add", [P, P, P]),
                           ("orc_g1_mul", [P, P, P]), ("orc_g1_msm", [S, P, P, P]),
                           ("orc_g1_jacobian_to_affine", [P, P]),
                           ("orc_g2_on_curve", [P]), ("orc_g2_add", [P, P, P]),
                           ("orc_g2_mul", [P, P, P]), ("orc_g2_msm", [S, P, P, P]),
                           ("orc_g2_jacobian_to_affine", [P, P])):
            getattr(L, name).argtypes = args
            getattr(L, name).restype = ctypes.c_int
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


def poly_eval(coeffs, z):
    """sum_j coeffs[j] z^j (Montgomery in and out), one point."""
    c = _fr(coeffs)
    zz = _fr(z).reshape(8)
    out = np.zeros(8, np.uint32)
    lib().orc_poly_eval(c.shape[0], _p(c), _p(zz), _p(out))
    return out


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


# ------------------------------------------------------------------------- G1 ----

def _pts(a):
    a = np.ascontiguousarray(a, dtype=np.uint32)
    return a.reshape(-1, 16)


def fq_mul(a, b):
    """Montgomery product over F_q, elementwise on (m, 8) arrays."""
    a, b = _fr(a), _fr(b)
    out = np.empty_like(a)
    for i in range(a.shape[0]):
        lib().orc_fq_mul(_p(a[i]), _p(b[i]), _p(out[i]))
    return out


def fq_inv(a):
    a = _fr(a)
    out = np.empty_like(a)
    for i in range(a.shape[0]):
        lib().orc_fq_inv(_p(a[i]), _p(out[i]))
    return out


def g1_on_curve(points):
    """Per point: on y^2 = x^3 + 3 with canonical coordinates, or the all-zero infinity."""
    pts = _pts(points)
    return np.array([bool(lib().orc_g1_on_curve(_p(pts[i]))) for i in range(pts.shape[0])])


def g1_add(p, q):
    p, q = _pts(p), _pts(q)
    out = np.empty_like(p)
    for i in range(p.shape[0]):
        lib().orc_g1_add(_p(p[i]), _p(q[i]), _p(out[i]))
    return out


def g1_mul(points, scalars):
    """scalars[i] * points[i] (scalars in standard form), affine."""
    pts, k = _pts(points), _fr(scalars)
    out = np.empty_like(pts)
    for i in range(pts.shape[0]):
        lib().orc_g1_mul(_p(pts[i]), _p(k[i]), _p(out[i]))
    return out


def g1_msm(points, scalars):
    """sum_i scalars[i] * points[i] as one affine point, shape (16,)."""
    pts, k = _pts(points), _fr(scalars)
    if pts.shape[0] != k.shape[0]:
        raise ValueError("points and scalars differ in length")
    out = np.zeros(16, np.uint32)
    lib().orc_g1_msm(pts.shape[0], _p(pts), _p(k), _p(out))
    return out


def g1_jacobian_to_affine(jac):
    """The affine point (16 limbs) of a Jacobian point (24 limbs X, Y, Z)."""
    j = np.ascontiguousarray(jac, dtype=np.uint32).reshape(24)
    out = np.zeros(16, np.uint32)
    lib().orc_g1_jacobian_to_affine(_p(j), _p(out))
    return out


# ------------------------------------------------------------------------- G2 ----

def _pts2(a):
    return np.ascontiguousarray(a, dtype=np.uint32).reshape(-1, 32)


def g2_on_curve(points):
    pts = _pts2(points)
    return np.array([bool(lib().orc_g2_on_curve(_p(pts[i]))) for i in range(pts.shape[0])])


def g2_add(p, q):
    p, q = _pts2(p), _pts2(q)
    out = np.empty_like(p)
    for i in range(p.shape[0]):
        lib().orc_g2_add(_p(p[i]), _p(q[i]), _p(out[i]))
    return out


def g2_mul(points, scalars):
    pts, k = _pts2(points), _fr(scalars)
    out = np.empty_like(pts)
    for i in range(pts.shape[0]):
        lib().orc_g2_mul(_p(pts[i]), _p(k[i]), _p(out[i]))
    return out


def g2_msm(points, scalars):
    """sum_i scalars[i] * points[i] over the twist, one affine point, shape (32,)."""
    pts, k = _pts2(points), _fr(scalars)
    if pts.shape[0] != k.shape[0]:
        raise ValueError("points and scalars differ in length")
    out = np.zeros(32, np.uint32)
    lib().orc_g2_msm(pts.shape[0], _p(pts), _p(k), _p(out))
    return out


def g2_jacobian_to_affine(jac):
    j = np.ascontiguousarray(jac, dtype=np.uint32).reshape(48)
    out = np.zeros(32, np.uint32)
    lib().orc_g2_jacobian_to_affine(_p(j), _p(out))
    return out
