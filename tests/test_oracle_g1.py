"""Pins of the G1 multi-scalar-multiplication oracle against what the mathematics fixes.

Neither oracle implementation (pure Python affine, C Jacobian) is trusted by itself:
  * the curve data against the published constants (tests/golden/g1_constants.txt);
  * the Python group law against group axioms and the group order (r * P = O for every
    point, the cofactor being 1): a wrong slope, sign or coordinate formula breaks them;
  * the C field and point arithmetic against Python ints and the Python group law, on
    edge cases (doubling through the addition, opposite points, infinity, scalars 0, 1,
    r - 1, r and above);
  * the MSM against the closed form: with bases P_i = t_i G, sum s_i P_i = (sum s_i t_i) G,
    the right side computed through the scalar field alone;
  * planted mistakes in a copy of the Python group law, each caught.
"""
import os
import random

import numpy as np
import pytest

import oracle
from oracle import fr_int as F
from oracle import g1_int as G
from bn254_scalar_field_gb300 import synth_g1

Q = G.Q_MOD
R = G.R_ORDER
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()
    yield


def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "g1_constants.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v, 0)
    return vals


def _is_probable_prime(n, rounds=48):
    d, s = n - 1, 0
    while d % 2 == 0:
        d //= 2
        s += 1
    rnd = random.Random(777)
    for _ in range(rounds):
        x = pow(rnd.randrange(2, n - 2), d, n)
        if x in (1, n - 1):
            continue
        for _ in range(s - 1):
            x = x * x % n
            if x == n - 1:
                break
        else:
            return False
    return True


def _random_points(k, seed=3):
    return G.array_to_points(synth_g1.points(k, seed))


# ---------------------------------------------------------------------- constants ----

def test_curve_constants():
    g = _golden()
    assert g["q"] == Q and g["b"] == G.CURVE_B and (g["gx"], g["gy"]) == G.GENERATOR
    assert g["order"] == R == F.R_MOD
    assert _is_probable_prime(Q) and Q % 4 == 3 and Q < (1 << 254)
    assert 4 * Q < (1 << 256)  # lazy reduction in [0, 2q) needs this
    assert g["mont_r_q"] == (1 << 256) % Q
    assert (g["np32_q"] * Q) % (1 << 32) == (1 << 32) - 1
    assert G.on_curve(G.GENERATOR)
    # Hasse bound: |q + 1 - #E| <= 2 sqrt(q), with #E = r
    assert (Q + 1 - R) ** 2 <= 4 * Q


# -------------------------------------------------------------- Python group law ----

def test_python_group_order_and_axioms():
    Gp = G.GENERATOR
    assert G.mul(R, Gp) is None
    assert G.mul(R + 1, Gp) == Gp
    assert G.mul(R - 1, Gp) == G.neg(Gp)
    P, Qp, S = _random_points(3)
    for X in (P, Qp, S):
        assert G.on_curve(X)
        assert G.mul(R, X) is None  # cofactor 1: every point has order r
    assert G.add(G.add(P, Qp), S) == G.add(P, G.add(Qp, S))
    assert G.add(P, Qp) == G.add(Qp, P)
    assert G.add(P, G.neg(P)) is None
    assert G.add(P, None) == P and G.add(None, P) == P
    assert G.double(P) == G.mul(2, P)
    assert G.mul(5, P) == G.add(G.double(G.double(P)), P)


def test_python_mul_is_linear():
    P = _random_points(1, seed=11)[0]
    rnd = random.Random(5)
    a, b = rnd.randrange(R), rnd.randrange(R)
    assert G.add(G.mul(a, P), G.mul(b, P)) == G.mul((a + b) % R, P)
    assert G.mul(a, G.mul(b, P)) == G.mul(a * b % R, P)


def _planted(kind):
    """A copy of the chord-and-tangent addition with one mistake."""
    def add(P, Qp):
        if P is None:
            return Qp
        if Qp is None:
            return P
        x1, y1 = P
        x2, y2 = Qp
        if x1 == x2:
            if (y1 + y2) % Q == 0:
                return None
            num = (2 if kind == "slope" else 3) * x1 * x1
            lam = num * G.inv(2 * y1) % Q
        else:
            lam = (y2 - y1) * G.inv(x2 - x1) % Q
        x3 = (lam * lam - x1 - (x2 if kind != "x3" else -x2)) % Q
        y3 = (lam * (x1 - x3) + (y1 if kind == "y3" else -y1)) % Q
        return (x3, y3)

    def mul(k, P):
        acc = None
        for bit in bin(k)[2:]:
            acc = add(acc, acc)
            if bit == "1":
                acc = add(acc, P)
        return acc
    return mul


@pytest.mark.parametrize("kind", ["slope", "x3", "y3"])
def test_planted_group_law_mistakes_are_caught(kind):
    mul = _planted(kind)
    P = _random_points(1, seed=17)[0]
    Rp = mul(R, P)
    assert not (Rp is None), kind


# ------------------------------------------------------------------- C vs Python ----

def test_c_field_against_python():
    rnd = random.Random(8)
    vals = [0, 1, 2, Q - 1, Q - 2, (1 << 253), (1 << 256) % Q] + [rnd.randrange(Q) for _ in range(200)]
    a = F.ints_to_array(vals)
    b = F.ints_to_array(vals[::-1])
    got = [F.limbs_to_int(r) for r in oracle.fq_mul(a, b)]
    rinv = pow(1 << 256, -1, Q)
    assert got == [x * y * rinv % Q for x, y in zip(vals, vals[::-1])]
    nz = [v for v in vals if v]
    inv = [F.limbs_to_int(r) for r in oracle.fq_inv(F.ints_to_array(nz))]
    # the Montgomery form of the inverse of the element whose Montgomery form is v = xR is
    # x^-1 R = R^2 / v
    assert inv == [pow(v, -1, Q) * (1 << 512) % Q for v in nz]


def test_c_on_curve():
    pts = synth_g1.points(12, seed=21)
    assert oracle.g1_on_curve(pts).all()
    bad = pts.copy()
    bad[0, 8] ^= 1  # y changed
    bad[1, :8] = F.int_to_limbs(Q)  # x not canonical
    bad[2, 8:] = F.int_to_limbs(Q + 1)
    assert list(oracle.g1_on_curve(bad)[:3]) == [False, False, False]
    assert oracle.g1_on_curve(np.zeros((1, 16), np.uint32)).all()  # infinity


def test_c_add_against_python():
    pts = _random_points(6, seed=23)
    P, Qp = pts[:3], pts[3:]
    cases = [(P[0], Qp[0]), (P[1], Qp[1]), (P[0], P[0]), (P[1], G.neg(P[1])), (P[2], None),
             (None, Qp[2]), (None, None)]
    a = G.points_to_array([c[0] for c in cases])
    b = G.points_to_array([c[1] for c in cases])
    got = G.array_to_points(oracle.g1_add(a, b))
    assert got == [G.add(x, y) for x, y in cases]


def test_c_mul_against_python():
    rnd = random.Random(31)
    pts = _random_points(3, seed=29) + [G.GENERATOR]
    ks = [0, 1, 2, 3, R - 1, R, R + 5, (1 << 256) - 1, rnd.randrange(R), rnd.randrange(R)]
    cases = [(P, k) for P in pts for k in ks]
    got = G.array_to_points(oracle.g1_mul(G.points_to_array([c[0] for c in cases]),
                                          F.ints_to_array([c[1] for c in cases])))
    assert got == [G.mul(k, P) for P, k in cases]


def test_c_jacobian_to_affine():
    rnd = random.Random(37)
    for P in _random_points(4, seed=41):
        z = rnd.randrange(1, Q)
        X, Y, Z = P[0] * z * z % Q, P[1] * z * z * z % Q, z
        row = np.array(F.int_to_limbs(G.to_mont(X)) + F.int_to_limbs(G.to_mont(Y)) +
                       F.int_to_limbs(G.to_mont(Z)), np.uint32)
        assert G.array_to_points(oracle.g1_jacobian_to_affine(row))[0] == P
        assert G.jacobian_array_to_point(row) == P
    inf = np.zeros(24, np.uint32)
    inf[:8] = F.int_to_limbs(G.to_mont(1))
    assert G.array_to_points(oracle.g1_jacobian_to_affine(inf))[0] is None


# --------------------------------------------------------------------------- MSM ----

@pytest.mark.parametrize("n", [0, 1, 2, 7, 16])
def test_c_msm_against_python(n):
    pts = synth_g1.points(n, seed=43)
    s = synth_g1.scalars(n, seed=47)
    want = G.msm(F.array_to_ints(s), G.array_to_points(pts)) if n else None
    got = G.array_to_points(oracle.g1_msm(pts, s))[0]
    assert got == want


def test_c_msm_closed_form():
    """Bases t_i G with known t_i: sum s_i t_i G = (sum s_i t_i mod r) G."""
    n = 40
    rnd = random.Random(53)
    t = [rnd.randrange(R) for _ in range(n)]
    s = [rnd.randrange(R) for _ in range(n)]
    s[:5] = [0, 1, R - 1, 2, 1]  # special scalars
    bases = G.points_to_array([G.mul(ti, G.GENERATOR) for ti in t])
    got = G.array_to_points(oracle.g1_msm(bases, F.ints_to_array(s)))[0]
    assert got == G.mul(sum(a * b for a, b in zip(s, t)) % R, G.GENERATOR)


def test_c_msm_special_inputs():
    P = _random_points(2, seed=59)
    # P and -P with equal scalars cancel; a base at infinity contributes nothing
    bases = G.points_to_array([P[0], G.neg(P[0]), None, P[1]])
    s = F.ints_to_array([12345, 12345, 999, 0])
    assert G.array_to_points(oracle.g1_msm(bases, s))[0] is None
    s = F.ints_to_array([R - 1, R - 1, 1, 3])
    assert G.array_to_points(oracle.g1_msm(bases, s))[0] == G.mul(3, P[1])


def test_point_sampler():
    pts = synth_g1.points(60, seed=61)
    assert oracle.g1_on_curve(pts).all()
    py = G.array_to_points(pts)
    assert all(G.on_curve(P) for P in py)
    assert len(set(py)) == 60  # distinct
    # the six points of one draw: (beta^j x, +-y)
    assert py[1] == G.neg(py[0]) and py[2][1] == py[0][1] and py[2][0] != py[0][0]
