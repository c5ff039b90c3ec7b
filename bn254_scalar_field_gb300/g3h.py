"""Thin ctypes binding of include/g3h.h: the same entry points, argument marshalling only.

Every step of the path runs in the CUDA library libg3h.so; there is no fallback. Loading
fails loudly (G3HError) when the library has not been built (``build.build()``).

Buffers are passed either as numpy arrays (host memory; the call copies to the device
and back and returns when done) or as torch CUDA tensors (device memory; the call only
enqueues work on the context's stream, which defaults to torch's current stream, and
``g3h_sync`` waits). A field element is eight little-endian uint32 limbs: arrays of shape
(m, 8), dtype uint32 (numpy) or int32/uint32 (torch).
"""
import ctypes
import os

import numpy as np

from . import build as _build

G3H_OK = 0
G3H_E_INVAL = -1
G3H_E_NONCANON = -2
G3H_E_RANGE = -3
G3H_E_NOMEM = -4
G3H_E_CUDA = -5
G3H_E_POINT = -6

G3H_DEVICE_PTRS = 0x1
G3H_NOCHECK = 0x2
G3H_FUSED_JOIN = 0x4
G3H_SERIALIZE = 0x8
G3H_NO_GRAPH = 0x10

G3H_MUL_LO = 0
G3H_MUL_HI = 1
G3H_MUL_WIDE = 2

G3H_MAX_LOG_N = 27
G3H_MSM_MAX_LOG = 24

# cudaStreamLegacy: the runtime's handle for the legacy default stream.
CUDA_STREAM_LEGACY = 0x1

ENTRY_POINTS = ("g3h_prepare", "g3h_compute_h", "g3h_compute_h_abc", "g3h_gather", "g3h_ntt",
                "g3h_join", "g3h_mul", "g3h_sync", "g3h_destroy", "g3h_strerror", "g3h_info",
                "g3h_timing_enable", "g3h_timing_read", "g3h_compute_h_abc_static",
                "g3h_compute_h_batch", "g3h_mont_to_std", "g3h_msm_prepare", "g3h_msm",
                "g3h_msm_g2_prepare", "g3h_msm_g2", "g3h_measure_imad",
                "g3h_measure_int_mul")


class G3HError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s: %s (%d)" % (what, strerror(code), code))


class g3h_csr(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_uint32), ("row_ptr", ctypes.c_void_p),
                ("col", ctypes.c_void_p), ("val", ctypes.c_void_p)]


class g3h_kernel_time(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_uint32),
                ("ms", ctypes.c_double)]


_lib = None


def lib():
    """The loaded libg3h.so. Raises G3HError if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise G3HError(G3H_E_CUDA, "libg3h.so not built at %s; run "
                           "bn254_scalar_field_gb300.build.build()" % path)
        L = ctypes.CDLL(path)
        P, U, I, S = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_int, ctypes.c_size_t
        L.g3h_prepare.argtypes = [U, U, P, P, I, P, ctypes.POINTER(P)]
        L.g3h_compute_h.argtypes = [P, P, P, P, U]
        L.g3h_compute_h_abc.argtypes = [P, P, P, P, P, P, U]
        L.g3h_gather.argtypes = [P, P, P, P, P, U]
        L.g3h_ntt.argtypes = [P, P, I, I, U]
        L.g3h_join.argtypes = [P, P, P, P, P, P, U]
        L.g3h_mul.argtypes = [P, P, P, P, S, U]
        L.g3h_mont_to_std.argtypes = [P, P, P, S, U]
        L.g3h_msm_prepare.argtypes = [P, P, U, U]
        L.g3h_msm.argtypes = [P, P, U, P, U]
        L.g3h_msm_g2_prepare.argtypes = [P, P, U, U]
        L.g3h_msm_g2.argtypes = [P, P, U, P, U]
        L.g3h_sync.argtypes = [P]
        L.g3h_destroy.argtypes = [P]
        L.g3h_destroy.restype = None
        L.g3h_strerror.argtypes = [I]
        L.g3h_strerror.restype = ctypes.c_char_p
        L.g3h_info.argtypes = [P, ctypes.POINTER(U), ctypes.POINTER(U)]
        L.g3h_timing_enable.argtypes = [P, I]
        L.g3h_timing_read.argtypes = [P, ctypes.POINTER(g3h_kernel_time), I,
                                      ctypes.POINTER(I)]
        L.g3h_compute_h_abc_static.argtypes = [U, P, P, P, P, P, P]
        L.g3h_compute_h_batch.argtypes = [P, U, P, P, P, U]
        L.g3h_measure_imad.argtypes = [P, ctypes.POINTER(ctypes.c_double)]
        L.g3h_measure_int_mul.argtypes = [P, I, ctypes.POINTER(ctypes.c_double)]
        for name in ENTRY_POINTS:
            if name not in ("g3h_destroy", "g3h_strerror"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def strerror(code):
    try:
        return lib().g3h_strerror(int(code)).decode()
    except G3HError:
        return "error %d" % code


def _check(rc, what):
    if rc != G3H_OK:
        raise G3HError(rc, what)


def _is_torch(x):
    return type(x).__module__.startswith("torch")


def _ptr(x, device):
    """(pointer, is_device) of a numpy array or torch tensor, checked for layout."""
    if x is None:
        return None, None
    if _is_torch(x):
        if not x.is_contiguous():
            raise ValueError("tensor must be contiguous")
        if x.element_size() != 4 or x.dtype.is_floating_point or x.dtype.is_complex:
            raise ValueError("tensors must hold 32-bit integer limbs (int32 or uint32)")
        if x.is_cuda and x.data_ptr() % 16:
            raise ValueError("device tensors must start on a 16-byte boundary")
        return ctypes.c_void_p(x.data_ptr()), x.is_cuda
    if not isinstance(x, np.ndarray) or x.dtype != np.uint32 or not x.flags.c_contiguous:
        raise ValueError("host arrays must be C-contiguous numpy uint32")
    return ctypes.c_void_p(x.ctypes.data), False


def _flags(bufs, flags):
    kinds = {d for _, d in bufs if d is not None}
    if len(kinds) > 1:
        raise ValueError("mix of host arrays and device tensors in one call")
    if kinds == {True}:
        flags |= G3H_DEVICE_PTRS
    return flags


def _elems(x):
    return (x.numel() if _is_torch(x) else x.size) // 8


# ---------------------------------------------------------------- entry points ----

def g3h_prepare(log_n, n_wires, A=None, B=None, device=0, stream=None):
    """A, B: (row_ptr, col, val) numpy triples or None. stream: a cudaStream_t handle
    (int), None for torch's current stream on `device` if torch is loaded, else a stream
    the context owns. Returns an opaque context handle (ctypes.c_void_p)."""
    keep = []

    def csr(m):
        if m is None:
            return None
        rp, col, val = (np.ascontiguousarray(x, dtype=np.uint32) for x in m)
        keep.extend([rp, col, val])
        s = g3h_csr(rp.shape[0] - 1, rp.ctypes.data, col.ctypes.data if col.size else None,
                    val.ctypes.data if val.size else None)
        keep.append(s)
        return ctypes.byref(s)

    if stream is None:
        try:
            import torch

            if torch.cuda.is_available():
                stream = torch.cuda.current_stream(device).cuda_stream
                if stream == 0:
                    # torch's default stream is the legacy default stream: name it by the
                    # runtime's handle for it (cudaStreamLegacy), since NULL asks the
                    # library for a stream of its own.
                    stream = CUDA_STREAM_LEGACY
        except ImportError:
            pass
    out = ctypes.c_void_p()
    rc = lib().g3h_prepare(log_n, n_wires, csr(A), csr(B), device,
                           ctypes.c_void_p(stream) if stream else None, ctypes.byref(out))
    _check(rc, "g3h_prepare")
    return out


def g3h_compute_h(ctx, witness, h_mont, h_std, flags=0):
    bufs = [_ptr(witness, None), _ptr(h_mont, None), _ptr(h_std, None)]
    f = _flags(bufs, flags)
    _check(lib().g3h_compute_h(ctx, bufs[0][0], bufs[1][0], bufs[2][0], f), "g3h_compute_h")


def g3h_compute_h_batch(ctx, witnesses, h_mont, h_std, flags=0):
    """witnesses: (count, n_wires, 8); h_mont, h_std: (count, n, 8)."""
    count = witnesses.shape[0] if witnesses.ndim == 3 else 1
    bufs = [_ptr(witnesses, None), _ptr(h_mont, None), _ptr(h_std, None)]
    f = _flags(bufs, flags)
    _check(lib().g3h_compute_h_batch(ctx, count, bufs[0][0], bufs[1][0], bufs[2][0], f),
           "g3h_compute_h_batch")


def g3h_compute_h_abc(ctx, a, b, c, h_mont, h_std, flags=0):
    bufs = [_ptr(x, None) for x in (a, b, c, h_mont, h_std)]
    f = _flags(bufs, flags)
    _check(lib().g3h_compute_h_abc(ctx, *[p for p, _ in bufs], f), "g3h_compute_h_abc")


def g3h_gather(ctx, witness, a, b, c, flags=0):
    bufs = [_ptr(x, None) for x in (witness, a, b, c)]
    f = _flags(bufs, flags)
    _check(lib().g3h_gather(ctx, *[p for p, _ in bufs], f), "g3h_gather")


def g3h_ntt(ctx, data, inverse=False, coset=False, flags=0):
    bufs = [_ptr(data, None)]
    f = _flags(bufs, flags)
    _check(lib().g3h_ntt(ctx, bufs[0][0], int(inverse), int(coset), f), "g3h_ntt")


def g3h_join(ctx, ea, eb, ec, h_mont, h_std, flags=0):
    bufs = [_ptr(x, None) for x in (ea, eb, ec, h_mont, h_std)]
    f = _flags(bufs, flags)
    _check(lib().g3h_join(ctx, *[p for p, _ in bufs], f), "g3h_join")


def g3h_mul(ctx, a, b, out, flags=0):
    bufs = [_ptr(x, None) for x in (a, b, out)]
    f = _flags(bufs, flags)
    _check(lib().g3h_mul(ctx, bufs[0][0], bufs[1][0], bufs[2][0], _elems(out), f), "g3h_mul")


def g3h_mont_to_std(ctx, x, out, flags=0):
    """out = x in standard form (x Montgomery); out may be x itself."""
    if _elems(x) != _elems(out):
        raise ValueError("x and out differ in length")
    bufs = [_ptr(v, None) for v in (x, out)]
    f = _flags(bufs, flags)
    _check(lib().g3h_mont_to_std(ctx, bufs[0][0], bufs[1][0], _elems(out), f),
           "g3h_mont_to_std")


def _words(x):
    return x.numel() if _is_torch(x) else x.size


def g3h_msm_prepare(ctx, bases, flags=0):
    """Loads the G1 bases (n, 16) limbs: affine x, y in Montgomery form over F_q."""
    if _words(bases) % 16:
        raise ValueError("bases must hold 16 limbs per point")
    bufs = [_ptr(bases, None)]
    f = _flags(bufs, flags)
    _check(lib().g3h_msm_prepare(ctx, bufs[0][0], _words(bases) // 16, f), "g3h_msm_prepare")


def g3h_msm(ctx, scalars, result, flags=0):
    """result (24 limbs: Jacobian X, Y, Z over F_q) = sum scalars[i] * base[i]; scalars
    (count, 8) in standard form."""
    if _words(result) != 24:
        raise ValueError("result must hold 24 limbs")
    bufs = [_ptr(v, None) for v in (scalars, result)]
    f = _flags(bufs, flags)
    _check(lib().g3h_msm(ctx, bufs[0][0], _elems(scalars), bufs[1][0], f), "g3h_msm")


def g3h_msm_g2_prepare(ctx, bases, flags=0):
    """Loads the G2 bases (n, 32) limbs: affine x, y over F_q2, Montgomery over F_q."""
    if _words(bases) % 32:
        raise ValueError("bases must hold 32 limbs per point")
    bufs = [_ptr(bases, None)]
    f = _flags(bufs, flags)
    _check(lib().g3h_msm_g2_prepare(ctx, bufs[0][0], _words(bases) // 32, f),
           "g3h_msm_g2_prepare")


def g3h_msm_g2(ctx, scalars, result, flags=0):
    """result (48 limbs: Jacobian X, Y, Z over F_q2) = sum scalars[i] * base[i]."""
    if _words(result) != 48:
        raise ValueError("result must hold 48 limbs")
    bufs = [_ptr(v, None) for v in (scalars, result)]
    f = _flags(bufs, flags)
    _check(lib().g3h_msm_g2(ctx, bufs[0][0], _elems(scalars), bufs[1][0], f), "g3h_msm_g2")


def g3h_measure_imad(ctx):
    """The device's measured 32-bit IMAD results per second (the roofline's unit)."""
    v = ctypes.c_double()
    _check(lib().g3h_measure_imad(ctx, ctypes.byref(v)), "g3h_measure_imad")
    return v.value


def g3h_measure_int_mul(ctx, kind):
    """Thread-level instructions per second of independent mad.lo / mad.hi / mad.wide
    chains (kind G3H_MUL_LO, G3H_MUL_HI, G3H_MUL_WIDE)."""
    v = ctypes.c_double()
    _check(lib().g3h_measure_int_mul(ctx, int(kind), ctypes.byref(v)), "g3h_measure_int_mul")
    return v.value


def g3h_sync(ctx):
    _check(lib().g3h_sync(ctx), "g3h_sync")


def g3h_destroy(ctx):
    lib().g3h_destroy(ctx)


def g3h_strerror(code):
    return strerror(code)


def g3h_info(ctx):
    log_n, n_wires = ctypes.c_uint32(), ctypes.c_uint32()
    _check(lib().g3h_info(ctx, ctypes.byref(log_n), ctypes.byref(n_wires)), "g3h_info")
    return log_n.value, n_wires.value


def g3h_timing_enable(ctx, enable=True):
    _check(lib().g3h_timing_enable(ctx, int(bool(enable))), "g3h_timing_enable")


def g3h_timing_read(ctx):
    """{kernel name: (launches, total device ms)} of the launches recorded since
    g3h_timing_enable."""
    buf = (g3h_kernel_time * 64)()
    count = ctypes.c_int()
    _check(lib().g3h_timing_read(ctx, buf, 64, ctypes.byref(count)), "g3h_timing_read")
    return {buf[i].name.decode(): (buf[i].launches, buf[i].ms)
            for i in range(min(count.value, 64))}


def g3h_compute_h_abc_static(log_n, a, b, c, h_mont, h_std, stream=None):
    """Steps 2-5 with no allocation (library-internal fixed array, log_n <= 16). Device
    tensors on the current device only; `stream` defaults to torch's current stream."""
    bufs = [_ptr(x, None) for x in (a, b, c, h_mont, h_std)]
    if any(d is not True for _, d in bufs):
        raise ValueError("g3h_compute_h_abc_static takes device tensors only")
    if stream is None:
        import torch

        stream = torch.cuda.current_stream().cuda_stream
    _check(lib().g3h_compute_h_abc_static(log_n, *[p for p, _ in bufs],
                                          ctypes.c_void_p(stream) if stream else None),
           "g3h_compute_h_abc_static")


class Context:
    """A prepared domain (and optionally the CSR matrices) with its resident tables."""

    def __init__(self, log_n, n_wires=0, A=None, B=None, device=0, stream=None):
        self.log_n = log_n
        self.n = 1 << log_n
        self.n_wires = n_wires
        self.device = device
        self.handle = g3h_prepare(log_n, n_wires, A, B, device, stream)

    def compute_h(self, witness, h_mont, h_std, flags=0):
        g3h_compute_h(self.handle, witness, h_mont, h_std, flags)

    def compute_h_batch(self, witnesses, h_mont, h_std, flags=0):
        g3h_compute_h_batch(self.handle, witnesses, h_mont, h_std, flags)

    def compute_h_abc(self, a, b, c, h_mont, h_std, flags=0):
        g3h_compute_h_abc(self.handle, a, b, c, h_mont, h_std, flags)

    def gather(self, witness, a, b, c, flags=0):
        g3h_gather(self.handle, witness, a, b, c, flags)

    def ntt(self, data, inverse=False, coset=False, flags=0):
        g3h_ntt(self.handle, data, inverse, coset, flags)

    def join(self, ea, eb, ec, h_mont, h_std, flags=0):
        g3h_join(self.handle, ea, eb, ec, h_mont, h_std, flags)

    def mul(self, a, b, out, flags=0):
        g3h_mul(self.handle, a, b, out, flags)

    def mont_to_std(self, x, out, flags=0):
        g3h_mont_to_std(self.handle, x, out, flags)

    def msm_prepare(self, bases, flags=0):
        g3h_msm_prepare(self.handle, bases, flags)

    def msm(self, scalars, result, flags=0):
        g3h_msm(self.handle, scalars, result, flags)

    def msm_g2_prepare(self, bases, flags=0):
        g3h_msm_g2_prepare(self.handle, bases, flags)

    def msm_g2(self, scalars, result, flags=0):
        g3h_msm_g2(self.handle, scalars, result, flags)

    def measure_imad(self):
        return g3h_measure_imad(self.handle)

    def measure_int_mul(self, kind):
        return g3h_measure_int_mul(self.handle, kind)

    def sync(self):
        g3h_sync(self.handle)

    def timing_enable(self, enable=True):
        g3h_timing_enable(self.handle, enable)

    def timing_read(self):
        return g3h_timing_read(self.handle)

    def close(self):
        if self.handle:
            g3h_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
