"""Pure-Python integer reference for the multi-scalar multiplication over BN254 G2.

TEST INFRASTRUCTURE ONLY: the library never imports this module; the tests, the package
entry's smoke check and the benchmark's CPU-baseline leg may.

What is computed (MSM_CU, header "stages 5-9": Pippenger over G1 and G2; the G2 one is
stage 7, the witness multiexp of the B query): Q = sum_i s_i * P_i on the twist
E': y^2 = x^3 + 3/(9 + u) over F_q2 = F_q[u]/(u^2 + 1), by the definition (each s_i P_i by
double-and-add on affine points, chord-and-tangent). Elements of F_q2 are pairs (c0, c1)
of ints in [0, q) meaning c0 + c1 u; points are pairs (x, y) of those, infinity ``None``.

Curve data (printed on none of the pages; those of Ethereum's EIP-197 pairing check, which
defines this twist and its group G2 of order r): the twist's b = 3 / (9 + u) and the
generator of G2. The multiexp itself is defined on every point of E'(F_q2), also those
outside G2 (the twist has a large cofactor), which is what the synthetic bases are.
"""
from . import fr_int
from .g1_int import Q_MOD

R_ORDER = fr_int.R_MOD
MONT_R = 1 << 256


def f2_add(a, b):
    return ((a[0] + b[0]) % Q_MOD, (a[1] + b[1]) % Q_MOD)


def f2_sub(a, b):
    return ((a[0] - b[0]) % Q_MOD, (a[1] - b[1]) % Q_MOD)


def f2_mul(a, b):
    # (a0 + a1 u)(b0 + b1 u) with u^2 = -1
    return ((a[0] * b[0] - a[1] * b[1]) % Q_MOD, (a[0] * b[1] + a[1] * b[0]) % Q_MOD)


def f2_inv(a):
    # 1 / (a0 + a1 u) = (a0 - a1 u) / (a0^2 + a1^2)
    n = pow((a[0] * a[0] + a[1] * a[1]) % Q_MOD, Q_MOD - 2, Q_MOD)
    return (a[0] * n % Q_MOD, (-a[1]) * n % Q_MOD)


def f2_neg(a):
    return ((-a[0]) % Q_MOD, (-a[1]) % Q_MOD)


ZERO = (0, 0)
CURVE_B = f2_mul((3, 0), f2_inv((9, 1)))
GENERATOR = (
    (10857046999023057135944570762232829481370756359578518086990519993285655852781,
     11559732032986387107991004021392285783925812861821192530917403151452391805634),
    (8495653923123431417604973247489272438418190587263600148770280649306958101930,
     4082367875863433681332203403145435568316851327593401208105741076214120093531))


def on_curve(P):
    if P is None:
        return True
    x, y = P
    ok = all(0 <= c < Q_MOD for c in x + y)
    return ok and f2_mul(y, y) == f2_add(f2_mul(f2_mul(x, x), x), CURVE_B)


def neg(P):
    return None if P is None else (P[0], f2_neg(P[1]))


def add(P, Q):
    """Chord and tangent on y^2 = x^3 + b (a = 0)."""
    if P is None:
        return Q
    if Q is None:
        return P
    (x1, y1), (x2, y2) = P, Q
    if x1 == x2:
        if f2_add(y1, y2) == ZERO:
            return None
        lam = f2_mul(f2_mul((3, 0), f2_mul(x1, x1)), f2_inv(f2_add(y1, y1)))
    else:
        lam = f2_mul(f2_sub(y2, y1), f2_inv(f2_sub(x2, x1)))
    x3 = f2_sub(f2_sub(f2_mul(lam, lam), x1), x2)
    y3 = f2_sub(f2_mul(lam, f2_sub(x1, x3)), y1)
    return (x3, y3)


def mul(k, P):
    acc = None
    for bit in bin(k)[2:] if k > 0 else "":
        acc = add(acc, acc)
        if bit == "1":
            acc = add(acc, P)
    return acc


def msm(scalars, points):
    acc = None
    for s, P in zip(scalars, points):
        acc = add(acc, mul(s, P))
    return acc


# -------------------------------------------------------------- array boundary ----

def _mont(v):
    return v * MONT_R % Q_MOD


def _unmont(v):
    return v * pow(MONT_R, -1, Q_MOD) % Q_MOD


def points_to_array(points):
    """(n, 32) uint32: x.c0, x.c1, y.c0, y.c1, eight limbs each, Montgomery over F_q;
    infinity all zero."""
    import numpy as np

    out = np.zeros((len(points), 32), np.uint32)
    for i, P in enumerate(points):
        if P is not None:
            for k, v in enumerate(P[0] + P[1]):
                out[i, 8 * k:8 * k + 8] = fr_int.int_to_limbs(_mont(v))
    return out


def array_to_points(arr):
    pts = []
    for row in arr.reshape(-1, 32):
        v = [_unmont(fr_int.limbs_to_int(row[8 * k:8 * k + 8])) for k in range(4)]
        raw = [fr_int.limbs_to_int(row[8 * k:8 * k + 8]) for k in range(4)]
        pts.append(None if not any(raw) else ((v[0], v[1]), (v[2], v[3])))
    return pts


def jacobian_array_to_point(row):
    """48 limbs X.c0, X.c1, Y.c0, Y.c1, Z.c0, Z.c1 (Montgomery), x = X/Z^2, y = Y/Z^3."""
    v = [_unmont(fr_int.limbs_to_int(row[8 * k:8 * k + 8])) for k in range(6)]
    X, Y, Z = (v[0], v[1]), (v[2], v[3]), (v[4], v[5])
    if Z == ZERO:
        return None
    zi = f2_inv(Z)
    zi2 = f2_mul(zi, zi)
    return (f2_mul(X, zi2), f2_mul(Y, f2_mul(zi2, zi)))
