"""Pins of the G2 (twist) multiexp oracle against what the mathematics fixes.

  * the twist's b and the generator against EIP-197 (the generator on the curve, of order
    r); F_q2 arithmetic against its defining identities;
  * the Python group law on random twist points: axioms and linearity of the scalar
    multiplication (these points lie outside G2, where r * P need not vanish);
  * the C oracle against Python: field, addition edge cases, scalar multiplication,
    the multiexp on small sizes, the Jacobian-to-affine map;
  * the multiexp's closed form on G2: sum s_i (t_i G) = (sum s_i t_i) G;
  * planted mistakes in a copy of the Python law (tangent slope, wrong twist) caught.
"""
import random

import numpy as np
import pytest

import oracle
from oracle import fr_int as F
from oracle import g2_int as G
from bn254_scalar_field_gb300 import synth_g2

Q = G.Q_MOD
R = G.R_ORDER


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()
    yield


def _pts(k, seed):
    return G.array_to_points(synth_g2.points(k, seed))


def test_twist_constants():
    # b2 (9 + u) = 3
    assert G.f2_mul(G.CURVE_B, (9, 1)) == (3, 0)
    assert synth_g2.CURVE_B == G.CURVE_B
    assert G.on_curve(G.GENERATOR)
    assert G.mul(R, G.GENERATOR) is None
    assert G.mul(R - 1, G.GENERATOR) == G.neg(G.GENERATOR)


def test_fq2_identities():
    rnd = random.Random(3)
    for _ in range(20):
        a = (rnd.randrange(Q), rnd.randrange(Q))
        b = (rnd.randrange(Q), rnd.randrange(Q))
        c = (rnd.randrange(Q), rnd.randrange(Q))
        assert G.f2_mul(a, G.f2_add(b, c)) == G.f2_add(G.f2_mul(a, b), G.f2_mul(a, c))
        if a != G.ZERO:
            assert G.f2_mul(a, G.f2_inv(a)) == (1, 0)
    assert G.f2_mul((0, 1), (0, 1)) == (Q - 1, 0)  # u^2 = -1


def test_python_law_on_random_twist_points():
    P, Qp, S = _pts(3, 5)
    for X in (P, Qp, S):
        assert G.on_curve(X)
    assert G.add(G.add(P, Qp), S) == G.add(P, G.add(Qp, S))
    assert G.add(P, Qp) == G.add(Qp, P)
    assert G.add(P, G.neg(P)) is None
    rnd = random.Random(7)
    a, b = rnd.randrange(1 << 64), rnd.randrange(1 << 64)
    assert G.add(G.mul(a, P), G.mul(b, P)) == G.mul(a + b, P)


@pytest.mark.parametrize("kind", ["slope", "twist"])
def test_planted_mistakes_are_caught(kind):
    if kind == "twist":
        wrong_b = G.f2_mul((3, 0), G.f2_inv((9, Q - 1)))  # 3 / (9 - u)
        x, y = G.GENERATOR
        assert G.f2_mul(y, y) != G.f2_add(G.f2_mul(G.f2_mul(x, x), x), wrong_b)
        return

    def add(P, Qp):
        if P is None:
            return Qp
        if Qp is None:
            return P
        (x1, y1), (x2, y2) = P, Qp
        if x1 == x2:
            if G.f2_add(y1, y2) == G.ZERO:
                return None
            lam = G.f2_mul(G.f2_mul((2, 0), G.f2_mul(x1, x1)), G.f2_inv(G.f2_add(y1, y1)))
        else:
            lam = G.f2_mul(G.f2_sub(y2, y1), G.f2_inv(G.f2_sub(x2, x1)))
        x3 = G.f2_sub(G.f2_sub(G.f2_mul(lam, lam), x1), x2)
        return (x3, G.f2_sub(G.f2_mul(lam, G.f2_sub(x1, x3)), y1))

    acc = None
    for bit in bin(R)[2:]:
        acc = add(acc, acc)
        if bit == "1":
            acc = add(acc, G.GENERATOR)
    assert acc is not None


def test_c_against_python():
    pts = _pts(4, 11)
    P = G.points_to_array(pts)
    assert oracle.g2_on_curve(P).all()
    bad = P.copy()
    bad[0, 16] ^= 1
    assert not oracle.g2_on_curve(bad)[0]
    cases = [(pts[0], pts[1]), (pts[2], pts[2]), (pts[3], G.neg(pts[3])), (pts[0], None)]
    got = G.array_to_points(oracle.g2_add(G.points_to_array([c[0] for c in cases]),
                                          G.points_to_array([c[1] for c in cases])))
    assert got == [G.add(a, b) for a, b in cases]
    rnd = random.Random(13)
    ks = [0, 1, 2, R - 1, rnd.randrange(R)]
    got = G.array_to_points(oracle.g2_mul(np.repeat(P[:1], len(ks), axis=0), F.ints_to_array(ks)))
    assert got == [G.mul(k, pts[0]) for k in ks]


@pytest.mark.parametrize("n", [0, 1, 5])
def test_c_msm_against_python(n):
    pts = synth_g2.points(n, seed=17)
    s = synth_g2_scalars(n, 19)
    want = G.msm(F.array_to_ints(s), G.array_to_points(pts)) if n else None
    assert G.array_to_points(oracle.g2_msm(pts, s))[0] == want


def synth_g2_scalars(n, seed):
    from bn254_scalar_field_gb300 import synth_g1

    return synth_g1.scalars(n, seed)


def test_c_msm_closed_form_on_g2():
    rnd = random.Random(23)
    n = 6
    t = [rnd.randrange(R) for _ in range(n)]
    s = [rnd.randrange(R) for _ in range(n)]
    s[0] = 1
    bases = G.points_to_array([G.mul(ti, G.GENERATOR) for ti in t])
    got = G.array_to_points(oracle.g2_msm(bases, F.ints_to_array(s)))[0]
    assert got == G.mul(sum(a * b for a, b in zip(s, t)) % R, G.GENERATOR)


def test_c_jacobian_to_affine():
    rnd = random.Random(29)
    P = _pts(1, 31)[0]
    z = (rnd.randrange(Q), rnd.randrange(Q))
    z2 = G.f2_mul(z, z)
    X, Y = G.f2_mul(P[0], z2), G.f2_mul(P[1], G.f2_mul(z2, z))
    row = np.concatenate([np.array(F.int_to_limbs(G._mont(v)), np.uint32) for v in X + Y + z])
    assert G.jacobian_array_to_point(row) == P
    assert G.array_to_points(oracle.g2_jacobian_to_affine(row))[0] == P


def test_point_sampler():
    pts = synth_g2.points(24, seed=37)
    assert oracle.g2_on_curve(pts).all()
    py = G.array_to_points(pts)
    assert all(G.on_curve(P) for P in py) and len(set(py)) == 24
