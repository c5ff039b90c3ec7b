"""Pins for the CPU oracle: each check ties it to something other than itself.

* constants: primality and 2-adicity of r, the Montgomery constants, the order of the
  roots of unity (closed forms);
* field operations of the C oracle (4 x 64-bit limbs) against Python ints;
* transforms against the O(n^2) definition of the DFT, special inputs with closed-form
  transforms (delta, constant), the inverse round trip, linearity, and the coset transform
  against Horner evaluation at g*omega^i;
* the gather against a dense matrix-vector product;
* the whole path against the pure-Python path, and against the mathematics of the method:
  P = A*B - C vanishes on the domain, so P = H*(x^n - 1) with deg H <= n - 2 and
  h_i = P(g*omega^i) = -2*H(g*omega^i) (POINTWISE_CU page, "no division by Z(coset)");
  H is recomputed by schoolbook product and long division on small domains;
* planted mistakes in a copy of the Python path (dropped 1/n, wrong join sign, wrong
  coset element, transposed root) each fail at least one of the pins.
"""
import os
import random

import numpy as np
import pytest

import oracle
from oracle import fr_int as F
from bn254_scalar_field_gb300 import synth

R = F.R_MOD
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_constants():
    vals = {}
    with open(os.path.join(GOLDEN, "fr_constants.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            vals[k] = int(v, 0)
    return vals


def _is_probable_prime(n, rounds=48):
    if n < 4:
        return n in (2, 3)
    d, s = n - 1, 0
    while d % 2 == 0:
        d //= 2
        s += 1
    rnd = random.Random(12345)
    for _ in range(rounds):
        a = rnd.randrange(2, n - 2)
        x = pow(a, d, n)
        if x in (1, n - 1):
            continue
        for _ in range(s - 1):
            x = x * x % n
            if x == n - 1:
                break
        else:
            return False
    return True


# ------------------------------------------------------------------------ constants ----

def test_modulus_and_constants():
    g = _golden_constants()
    assert g["r"] == R
    assert _is_probable_prime(R)
    assert (R - 1) % (1 << 28) == 0 and ((R - 1) >> 28) % 2 == 1
    assert g["two_adicity"] == F.TWO_ADICITY == 28
    assert g["mont_r"] == (1 << 256) % R
    assert (g["np32"] * R) % (1 << 32) == (1 << 32) - 1
    assert F.limbs_to_int(synth.MODULUS_LIMBS) == R
    assert F.limbs_to_int(synth.MONT_ONE_LIMBS) == (1 << 256) % R
    assert 4 * R < (1 << 256)  # lazy reduction in [0, 2r) needs this


def test_two_adic_root_has_order_2_28():
    w = F.two_adic_root()
    assert w == _golden_constants()["root_2_28"]
    assert pow(F.NON_RESIDUE, (R - 1) // 2, R) == R - 1
    assert pow(w, 1 << 27, R) == R - 1
    assert pow(w, 1 << 28, R) == 1


@pytest.mark.parametrize("log_n", list(range(0, 28)))
def test_domain_roots(log_n, oracle_lib):
    n = 1 << log_n
    omega, g = F.domain(log_n)
    assert pow(omega, n, R) == 1
    if n > 1:
        assert pow(omega, n // 2, R) != 1
    assert pow(g, n, R) == R - 1  # primitive 2n-th root: g^n = -1
    assert g * g % R == omega
    w_c, g_c = oracle.domain(log_n)
    assert F.limbs_to_int(w_c) == omega and F.limbs_to_int(g_c) == g


# --------------------------------------------------------------------- field (C) ----

def _edge_values():
    mr = (1 << 256) % R
    return [0, 1, 2, R - 1, R - 2, mr, R - mr, (1 << 253), (1 << 254) - 1 - ((1 << 254) - R),
            (R - 1) // 2, (R + 1) // 2, 0xFFFFFFFF, 1 << 32, (1 << 224) - 1]


def _rand_vals(k, seed):
    rnd = random.Random(seed)
    return [rnd.randrange(R) for _ in range(k)]


def test_c_field_ops_against_python_ints(oracle_lib):
    vals = [v % R for v in _edge_values()] + _rand_vals(400, 1)
    xs = vals
    ys = list(reversed(vals))
    a = F.ints_to_array(xs)
    b = F.ints_to_array(ys)
    rinv = pow(1 << 256, -1, R)
    got_mul = F.array_to_ints(oracle.fr_mul(a, b))
    got_add = F.array_to_ints(oracle.fr_add(a, b))
    got_sub = F.array_to_ints(oracle.fr_sub(a, b))
    for x, y, m, s, d in zip(xs, ys, got_mul, got_add, got_sub):
        assert m == x * y * rinv % R
        assert s == (x + y) % R
        assert d == (x - y) % R
    std = F.array_to_ints(oracle.from_mont(a))
    assert std == [x * rinv % R for x in xs]
    back = F.array_to_ints(oracle.to_mont(oracle.from_mont(a)))
    assert back == xs


# -------------------------------------------------------------------- transforms ----

@pytest.mark.parametrize("log_n", [0, 1, 2, 3, 4, 5, 6])
def test_python_dft_recursive_matches_definition(log_n):
    omega, _ = F.domain(log_n)
    x = _rand_vals(1 << log_n, 10 + log_n)
    assert F.dft_recursive(x, omega) == F.dft_naive(x, omega)


@pytest.mark.parametrize("log_n", [0, 1, 2, 3, 5, 7, 8])
def test_c_ntt_matches_definition(log_n, oracle_lib):
    n = 1 << log_n
    omega, g = F.domain(log_n)
    x = _rand_vals(n, 20 + log_n)
    xm = F.ints_to_array([F.to_mont(v) for v in x])
    # forward: X_i = sum_j x_j omega^ij
    got = [F.from_mont(v) for v in F.array_to_ints(oracle.ntt(xm, log_n))]
    assert got == F.dft_naive(x, omega)
    # inverse: n^-1 sum_j x_j omega^-ij
    got = [F.from_mont(v) for v in F.array_to_ints(oracle.ntt(xm, log_n, inverse=True))]
    ninv = F.inv(n)
    assert got == [v * ninv % R for v in F.dft_naive(x, F.inv(omega))]
    # coset forward: sum_j x_j (g omega^i)^j, i.e. Horner at g omega^i
    got = [F.from_mont(v) for v in F.array_to_ints(oracle.ntt(xm, log_n, coset=True))]
    assert got == [F.poly_eval(x, g * pow(omega, i, R) % R) for i in range(n)]


def test_c_poly_eval_matches_python_horner(oracle_lib):
    """The C single-point evaluation (used to sample outputs of transforms too large for
    the whole oracle) against Python ints, at edge points and random ones."""
    for n, seed in ((1, 1), (2, 2), (37, 3), (300, 4)):
        x = _rand_vals(n, 700 + seed)
        xm = F.ints_to_array([F.to_mont(v) for v in x])
        for z in (0, 1, R - 1, _rand_vals(1, 800 + seed)[0]):
            got = F.from_mont(F.limbs_to_int(oracle.poly_eval(xm, F.ints_to_array([F.to_mont(z)]))))
            assert got == F.poly_eval(x, z)


@pytest.mark.parametrize("log_n", [1, 4, 9])
def test_ntt_special_inputs_and_round_trip(log_n, oracle_lib):
    n = 1 << log_n
    one = F.to_mont(1)
    delta = F.ints_to_array([one] + [0] * (n - 1))
    assert F.array_to_ints(oracle.ntt(delta, log_n)) == [one] * n
    ones = F.ints_to_array([one] * n)
    assert F.array_to_ints(oracle.ntt(ones, log_n)) == [F.to_mont(n)] + [0] * (n - 1)
    x = F.ints_to_array(_rand_vals(n, 30 + log_n))
    y = F.ints_to_array(_rand_vals(n, 40 + log_n))
    for coset in (False, True):
        fx = oracle.ntt(x, log_n, coset=coset)
        assert np.array_equal(oracle.ntt(fx, log_n, inverse=True, coset=coset), x)
        # linearity: NTT(x + y) = NTT(x) + NTT(y)
        fxy = oracle.ntt(oracle.fr_add(x, y), log_n, coset=coset)
        assert np.array_equal(fxy, oracle.fr_add(fx, oracle.ntt(y, log_n, coset=coset)))


# ------------------------------------------------------------------------ gather ----

def _ints_problem(A, B, w):
    def dec(arr):
        return [F.from_mont(v) for v in F.array_to_ints(arr)]

    return ([int(v) for v in A[0]], [int(v) for v in A[1]], dec(A[2]),
            [int(v) for v in B[0]], [int(v) for v in B[1]], dec(B[2]), dec(w))


@pytest.mark.parametrize("log_n", [3, 6, 8])
def test_gather_against_dense_product(log_n, oracle_lib):
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=99 + log_n)
    ra, ca, va, rb, cb, vb, wi = _ints_problem(A, B, w)
    n_wires = len(wi)
    dense_a = [[0] * n_wires for _ in range(n)]
    dense_b = [[0] * n_wires for _ in range(n)]
    for i in range(n):
        for k in range(ra[i], ra[i + 1]):
            dense_a[i][ca[k]] = (dense_a[i][ca[k]] + va[k]) % R
        for k in range(rb[i], rb[i + 1]):
            dense_b[i][cb[k]] = (dense_b[i][cb[k]] + vb[k]) % R
    a_ref = [sum(x * y for x, y in zip(row, wi)) % R for row in dense_a]
    b_ref = [sum(x * y for x, y in zip(row, wi)) % R for row in dense_b]
    c_ref = [x * y % R for x, y in zip(a_ref, b_ref)]
    a, b, c = oracle.gather(log_n, A, B, w)
    assert [F.from_mont(v) for v in F.array_to_ints(a)] == a_ref
    assert [F.from_mont(v) for v in F.array_to_ints(b)] == b_ref
    assert [F.from_mont(v) for v in F.array_to_ints(c)] == c_ref
    pa, pb, pc = F.gather(n, ra, ca, va, rb, cb, vb, wi)
    assert (pa, pb, pc) == (a_ref, b_ref, c_ref)


# ---------------------------------------------------------------------- pipeline ----

def _poly_mul(p, q):
    out = [0] * (len(p) + len(q) - 1)
    for i, x in enumerate(p):
        if x:
            for j, y in enumerate(q):
                out[i + j] = (out[i + j] + x * y) % R
    return out


def _divide_by_vanishing(p, n):
    """Long division of p by x^n - 1: returns (quotient, remainder)."""
    p = list(p)
    q = [0] * max(1, len(p) - n)
    for d in range(len(p) - 1, n - 1, -1):
        coef = p[d]
        if coef:
            q[d - n] = coef
            p[d] = 0
            p[d - n] = (p[d - n] + coef) % R
    return q, p[:n]


def _check_method_invariants(log_n, a, b, c, h, schoolbook):
    """h against the mathematics: the vanishing of P on the domain and its quotient."""
    n = 1 << log_n
    omega, g = F.domain(log_n)
    # interpolants by the O(n^2) definition, independent of the radix-2 code
    ninv, winv = F.inv(n), F.inv(omega)
    A = [v * ninv % R for v in F.dft_naive(a, winv)]
    Bc = [v * ninv % R for v in F.dft_naive(b, winv)]
    C = [v * ninv % R for v in F.dft_naive(c, winv)]
    # Q: interpolant of h on the coset, by the definition
    ginv = F.inv(g)
    Q = [v * ninv % R * pow(ginv, j, R) % R for j, v in enumerate(F.dft_naive(h, winv))]
    # deg(-2H) <= n - 2
    if n >= 2:
        assert Q[n - 1] == 0
    H = [v * F.inv(R - 2) % R for v in Q]
    rnd = random.Random(log_n)
    for _ in range(8):
        z = rnd.randrange(R)
        lhs = (F.poly_eval(A, z) * F.poly_eval(Bc, z) - F.poly_eval(C, z)) % R
        assert lhs == F.poly_eval(H, z) * (pow(z, n, R) - 1) % R
    if schoolbook:
        P = _poly_mul(A, Bc)
        for i, v in enumerate(C):
            P[i] = (P[i] - v) % R
        Hs, rem = _divide_by_vanishing(P, n)
        assert all(v == 0 for v in rem)
        Hs = Hs + [0] * (n - len(Hs))
        assert Hs[:n] == H[:n]


@pytest.mark.parametrize("log_n", [0, 1, 2, 3, 4, 5, 6, 7])
def test_pipeline_c_vs_python_and_invariants(log_n, oracle_lib):
    A, B, w = synth.problem(log_n, seed=7 + log_n)
    hm, hs = oracle.compute_h(log_n, A, B, w)
    ra, ca, va, rb, cb, vb, wi = _ints_problem(A, B, w)
    h_py = F.compute_h(log_n, ra, ca, va, rb, cb, vb, wi)
    assert [F.from_mont(v) for v in F.array_to_ints(hm)] == h_py
    assert F.array_to_ints(hs) == h_py
    assert all(v < R for v in F.array_to_ints(hm))
    a, b, c = F.gather(1 << log_n, ra, ca, va, rb, cb, vb, wi)
    _check_method_invariants(log_n, a, b, c, h_py, schoolbook=log_n <= 6)


@pytest.mark.parametrize("log_n", [9, 10])
def test_pipeline_invariants_larger(log_n, oracle_lib):
    A, B, w = synth.problem(log_n, seed=3 + log_n)
    hm, hs = oracle.compute_h(log_n, A, B, w)
    ra, ca, va, rb, cb, vb, wi = _ints_problem(A, B, w)
    h = F.array_to_ints(hs)
    assert h == [F.from_mont(v) for v in F.array_to_ints(hm)]
    a, b, c = F.gather(1 << log_n, ra, ca, va, rb, cb, vb, wi)
    n = 1 << log_n
    omega, g = F.domain(log_n)
    # coset interpolant of h has zero top coefficient (radix-2 path, then checked at z)
    Q = F.interpolate(h, log_n)
    ginv = F.inv(g)
    Q = [v * pow(ginv, j, R) % R for j, v in enumerate(Q)]
    assert Q[n - 1] == 0
    Acoef, Bcoef, Ccoef = (F.interpolate(v, log_n) for v in (a, b, c))
    H = [v * F.inv(R - 2) % R for v in Q]
    rnd = random.Random(100 + log_n)
    for _ in range(4):
        z = rnd.randrange(R)
        lhs = (F.poly_eval(Acoef, z) * F.poly_eval(Bcoef, z) - F.poly_eval(Ccoef, z)) % R
        assert lhs == F.poly_eval(H, z) * (pow(z, n, R) - 1) % R


def test_compute_h_abc_matches_compute_h(oracle_lib):
    log_n = 8
    A, B, w = synth.problem(log_n, seed=5)
    a, b, c = oracle.gather(log_n, A, B, w)
    hm1, hs1 = oracle.compute_h(log_n, A, B, w)
    hm2, hs2 = oracle.compute_h_abc(log_n, a, b, c)
    assert np.array_equal(hm1, hm2) and np.array_equal(hs1, hs2)


def test_golden_tiny_h(oracle_lib):
    """The stored 2^3 example, written by tests/golden/make_golden.py from the oracle."""
    path = os.path.join(GOLDEN, "h_k3_seed1.txt")
    want = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, i, v = line.split()
            want[(k, int(i))] = int(v, 16)
    A, B, w = synth.problem(3, seed=1)
    hm, hs = oracle.compute_h(3, A, B, w)
    for i, v in enumerate(F.array_to_ints(hm)):
        assert want[("h_mont", i)] == v
    for i, v in enumerate(F.array_to_ints(hs)):
        assert want[("h_std", i)] == v


# -------------------------------------------------------------- planted mistakes ----

def _mutant_quotient(log_n, a, b, c, mutation):
    n = 1 << log_n
    omega, g = F.domain(log_n)
    if mutation == "coset_is_domain":
        g = omega
    root_inv = omega if mutation == "transposed_root" else F.inv(omega)
    ninv = 1 if mutation == "dropped_1_over_n" else F.inv(n)

    def ev(v):
        coeffs = [x * ninv % R for x in F.dft_recursive(v, root_inv)]
        coeffs = [x * pow(g, j, R) % R for j, x in enumerate(coeffs)]
        return F.dft_recursive(coeffs, omega)

    ea, eb, ec = ev(a), ev(b), ev(c)
    if mutation == "join_sign":
        return [(x * y + z) % R for x, y, z in zip(ea, eb, ec)]
    return [(x * y - z) % R for x, y, z in zip(ea, eb, ec)]


@pytest.mark.parametrize("mutation", ["dropped_1_over_n", "join_sign", "coset_is_domain",
                                      "transposed_root"])
def test_planted_mistakes_are_caught(mutation):
    log_n = 4
    A, B, w = synth.problem(log_n, seed=21)
    ra, ca, va, rb, cb, vb, wi = _ints_problem(A, B, w)
    a, b, c = F.gather(1 << log_n, ra, ca, va, rb, cb, vb, wi)
    good = F.quotient_evals(log_n, a, b, c)
    bad = _mutant_quotient(log_n, a, b, c, mutation)
    assert bad != good
    with pytest.raises(AssertionError):
        _check_method_invariants(log_n, a, b, c, bad, schoolbook=True)
