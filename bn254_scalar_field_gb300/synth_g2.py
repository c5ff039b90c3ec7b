"""Seeded synthetic bases for the multi-scalar multiplication over the BN254 twist (G2).

The proving key's B-query points are not available; the generator stands in with points
drawn uniformly at random on E': y^2 = x^3 + b2 over F_q2 = F_q[u]/(u^2 + 1),
b2 = 3 / (9 + u). The multiexp is defined on every point of E'(F_q2); these points are
not reduced into the order-r subgroup G2 (that would take point arithmetic), which does
not change what is computed or how.

Sampling takes field arithmetic, none of the multiexp's point arithmetic: x uniform in
F_q2, y a square root of x^3 + b2 when one exists, by the complex method (for q = 3 mod 4
and u^2 = -1: with t = sqrt(a0^2 + a1^2) in F_q, y0 = sqrt((a0 +- t) / 2),
y1 = a1 / (2 y0)). Each accepted x gives six points (beta^j x, +-y), beta a primitive cube
root of unity in F_q. Coordinates are written x.c0, x.c1, y.c0, y.c1, eight little-endian
uint32 limbs each, Montgomery form over F_q.
"""
import numpy as np

from .synth import SplitMix64
from .synth_g1 import Q_MOD, _BETA, _BETA2, _limbs

_SQRT_EXP = (Q_MOD + 1) // 4


def _fsqrt(v):
    r = pow(v, _SQRT_EXP, Q_MOD)
    return r if r * r % Q_MOD == v % Q_MOD else None


def _f2mul(a, b):
    return ((a[0] * b[0] - a[1] * b[1]) % Q_MOD, (a[0] * b[1] + a[1] * b[0]) % Q_MOD)


_NINE_U_INV = (9 * pow(82, Q_MOD - 2, Q_MOD) % Q_MOD, (-1) * pow(82, Q_MOD - 2, Q_MOD) % Q_MOD)
CURVE_B = _f2mul((3, 0), _NINE_U_INV)  # 3 / (9 + u); 1/(9 + u) = (9 - u) / 82


def _f2sqrt(a):
    a0, a1 = a
    if a1 == 0:
        r = _fsqrt(a0)
        if r is not None:
            return (r, 0)
        r = _fsqrt((-a0) % Q_MOD)
        return None if r is None else (0, r)
    t = _fsqrt((a0 * a0 + a1 * a1) % Q_MOD)
    if t is None:
        return None
    half = (Q_MOD + 1) // 2
    for tt in (t, (-t) % Q_MOD):
        y0 = _fsqrt((a0 + tt) * half % Q_MOD)
        if y0:
            y1 = a1 * pow(2 * y0, Q_MOD - 2, Q_MOD) % Q_MOD
            if _f2mul((y0, y1), (y0, y1)) == (a0 % Q_MOD, a1 % Q_MOD):
                return (y0, y1)
    return None


def points(count, seed):
    """count points of E'(F_q2), shape (count, 32) uint32, Montgomery form, none at infinity."""
    rng = SplitMix64(seed)
    out = np.zeros((count, 32), np.uint32)
    r256 = (1 << 256) % Q_MOD
    filled = 0
    while filled < count:
        w = rng.u32(16)
        x0 = sum(int(w[k]) << (32 * k) for k in range(8)) & ((1 << 254) - 1)
        x1 = sum(int(w[8 + k]) << (32 * k) for k in range(8)) & ((1 << 254) - 1)
        if x0 >= Q_MOD or x1 >= Q_MOD:
            continue
        x = (x0, x1)
        rhs = _f2mul(_f2mul(x, x), x)
        rhs = ((rhs[0] + CURVE_B[0]) % Q_MOD, (rhs[1] + CURVE_B[1]) % Q_MOD)
        y = _f2sqrt(rhs)
        if y is None:
            continue
        ny = ((-y[0]) % Q_MOD, (-y[1]) % Q_MOD)
        for b in (1, _BETA, _BETA2):
            xx = (x[0] * b % Q_MOD, x[1] * b % Q_MOD)
            for yy in (y, ny):
                if filled == count:
                    break
                for k, v in enumerate(xx + yy):
                    out[filled, 8 * k:8 * k + 8] = _limbs(v * r256 % Q_MOD)
                filled += 1
    return out


def default_seed(log_n):
    return 0x67350000 + log_n
