"""Pure-Python integer reference for the multi-scalar multiplication over BN254 G1.

TEST INFRASTRUCTURE ONLY: the library never imports this module; the tests, the package
entry's smoke check and the benchmark's CPU-baseline leg may.

What is computed (MSM_CU, header "stages 5-9": Pippenger over G1, the H multiexp of
stage 9 taking the standard-form h as scalars; POINTWISE_CU "two output buffers": a
window digit of a Montgomery representative would be a digit of h*R, so the scalars are
the integers in [0, r)):

    Q = sum_i s_i * P_i

over the curve E: y^2 = x^3 + 3 on F_q. Here it is the plain definition: every s_i * P_i
by double-and-add on affine points with the chord-and-tangent group law, then summed.
Points are tuples (x, y) of ints in [0, q), the point at infinity is ``None``. The
Montgomery encoding (x * 2^256 mod q) appears only in the array conversions at the
boundary.

Curve data (the pages name the curve, BN254, but print none of its constants; these are
the ones of the Ethereum precompiles EIP-196/197, which define this curve as alt_bn128):
q the base-field prime, b = 3, generator (1, 2), group order r (the scalar field of the
quotient path, so every point except infinity has order r: the cofactor is 1).
"""
from . import fr_int

Q_MOD = 21888242871839275222246405745257275088696311157297823662689037894645226208583
R_ORDER = fr_int.R_MOD
CURVE_B = 3
GENERATOR = (1, 2)
MONT_R = 1 << 256


def inv(x):
    """x^-1 mod q by Fermat (q is prime)."""
    return pow(x % Q_MOD, Q_MOD - 2, Q_MOD)


def on_curve(P):
    if P is None:
        return True
    x, y = P
    return 0 <= x < Q_MOD and 0 <= y < Q_MOD and (y * y - x * x * x - CURVE_B) % Q_MOD == 0


def neg(P):
    return None if P is None else (P[0], (-P[1]) % Q_MOD)


def add(P, Q):
    """The chord-and-tangent law: the third intersection of the line through P and Q (the
    tangent when P = Q) with the curve, reflected in the x-axis."""
    if P is None:
        return Q
    if Q is None:
        return P
    x1, y1 = P
    x2, y2 = Q
    if x1 == x2:
        if (y1 + y2) % Q_MOD == 0:
            return None  # Q = -P (this includes doubling a point with y = 0)
        lam = 3 * x1 * x1 * inv(2 * y1) % Q_MOD  # tangent slope, a = 0
    else:
        lam = (y2 - y1) * inv(x2 - x1) % Q_MOD
    x3 = (lam * lam - x1 - x2) % Q_MOD
    y3 = (lam * (x1 - x3) - y1) % Q_MOD
    return (x3, y3)


def double(P):
    return add(P, P)


def mul(k, P):
    """k * P by left-to-right double-and-add over the bits of the integer k >= 0."""
    acc = None
    for bit in bin(k)[2:] if k > 0 else "":
        acc = double(acc)
        if bit == "1":
            acc = add(acc, P)
    return acc


def msm(scalars, points):
    """sum_i scalars[i] * points[i], by the definition."""
    acc = None
    for s, P in zip(scalars, points):
        acc = add(acc, mul(s, P))
    return acc


def sqrt(a):
    """A square root mod q of a quadratic residue a (q = 3 mod 4), or None."""
    y = pow(a % Q_MOD, (Q_MOD + 1) // 4, Q_MOD)
    return y if y * y % Q_MOD == a % Q_MOD else None


# -------------------------------------------------------------- array boundary ----

def to_mont(x):
    return x * MONT_R % Q_MOD


def from_mont(x):
    return x * pow(MONT_R, -1, Q_MOD) % Q_MOD


def points_to_array(points):
    """(n, 16) uint32: x then y, each eight little-endian limbs in Montgomery form;
    infinity is all zero."""
    import numpy as np

    out = np.zeros((len(points), 16), np.uint32)
    for i, P in enumerate(points):
        if P is not None:
            out[i, :8] = fr_int.int_to_limbs(to_mont(P[0]))
            out[i, 8:] = fr_int.int_to_limbs(to_mont(P[1]))
    return out


def array_to_points(arr):
    pts = []
    for row in arr.reshape(-1, 16):
        x = fr_int.limbs_to_int(row[:8])
        y = fr_int.limbs_to_int(row[8:])
        pts.append(None if x == 0 and y == 0 else (from_mont(x), from_mont(y)))
    return pts


def jacobian_array_to_point(row):
    """A point given as 24 limbs (X, Y, Z, Montgomery form) of Jacobian coordinates,
    x = X/Z^2, y = Y/Z^3, Z = 0 the point at infinity."""
    X, Y, Z = (from_mont(fr_int.limbs_to_int(row[8 * k:8 * k + 8])) for k in range(3))
    if Z % Q_MOD == 0:
        return None
    zi = inv(Z)
    return (X * zi * zi % Q_MOD, Y * zi * zi * zi % Q_MOD)
