"""GPU parity on inputs random vectors do not reach, against the CPU oracle, bit for bit.

1. The constant multiply's short quotient. The library forms Shoup's quotient from the
   upper limb columns only, so about one product in 2^29 comes out with the quotient one
   short and its result in [r, 2r) rather than [0, r) (tests/shoup_model.py). Inputs are
   planted where the first multiply of a transform sees them directly, and each planted
   value is checked on the CPU to produce the short quotient with that constant:
     * compute_h_abc: the first inverse pass multiplies (v[p] - v[p + n/2]) by omega^-p,
       so v[p] = x, v[p + n/2] = 0;
     * g3h_ntt, forward or inverse without coset: the first multiply of the bit-reversed
       load's passes is (y[4g+2] - y[4g+3]) * omega^(+-n/4), y[i] = data[brev(i)];
     * g3h_ntt, forward coset: the load multiplies data[j] by g^j.
   Slices of 2^6 (radix-2 build), 2^9 (radix-4, 128 threads) and 2^11 elements (radix-4,
   256 threads) are covered by the domains 2^12, 2^18 and 2^22.
2. Edge-valued vectors: all r - 1 (sums reach 2r - 2 before any reduction), alternating
   0 and r - 1, the Montgomery form of 1 everywhere, all zero, through every transform
   mode and the quotient path.
"""
import random

import numpy as np
import pytest

import oracle
from oracle import fr_int as F
from bn254_scalar_field_gb300 import build, g3h, synth
from shoup_model import R, shoup_model, short_quotient_input

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()
    yield


def _zeros(n):
    return np.zeros((n, 8), np.uint32)


def _brev(i, bits):
    return int(format(i, "0%db" % bits)[::-1], 2) if bits else 0


def _plant(vec, idx, x, w):
    """vec[idx] = x after checking that x * w takes the short quotient."""
    y, short = shoup_model(x, w)
    assert short and x < R, (idx, hex(x))
    vec[idx] = F.int_to_limbs(x)


@pytest.mark.parametrize("log_n", [12, 18, 22])
def test_short_quotient_in_the_quotient_path(log_n):
    n = 1 << log_n
    omega, _ = F.domain(log_n)
    omega_inv = F.inv(omega)
    rng = random.Random(1000 + log_n)
    srng = synth.SplitMix64(1100 + log_n)
    vecs = [synth.uniform_fr(srng, n) for _ in range(3)]
    planted = []
    for v in range(3):
        for p in (1 + v, 5 + 7 * v, n // 2 - 1 - v, rng.randrange(8, n // 2 - 8)):
            x = short_quotient_input(pow(omega_inv, p, R), rng)
            _plant(vecs[v], p, x, pow(omega_inv, p, R))
            vecs[v][p + n // 2] = 0
            planted.append((v, p, hex(x)))
    a, b, c = vecs
    want_m, want_s = oracle.compute_h_abc(log_n, a, b, c)
    with g3h.Context(log_n) as ctx:
        hm, hs = _zeros(n), _zeros(n)
        ctx.compute_h_abc(a, b, c, hm, hs)
    assert np.array_equal(hm, want_m), planted
    assert np.array_equal(hs, want_s), planted


@pytest.mark.parametrize("log_n", [12, 18, 22])
def test_short_quotient_in_standalone_transforms(log_n):
    n = 1 << log_n
    omega, g = F.domain(log_n)
    rng = random.Random(2000 + log_n)
    groups = (0, 1, n // 4 - 1, rng.randrange(2, n // 4 - 2))
    with g3h.Context(log_n) as ctx:
        for inverse in (False, True):
            w = pow(omega, n // 4, R) if not inverse else pow(F.inv(omega), n // 4, R)
            x = synth.uniform_fr(synth.SplitMix64(2100 + log_n + inverse), n)
            planted = []
            for grp in groups:
                xv = short_quotient_input(w, rng)
                _plant(x, _brev(4 * grp + 2, log_n), xv, w)
                x[_brev(4 * grp + 3, log_n)] = 0
                planted.append((grp, hex(xv)))
            for coset in (False, True):
                got = x.copy()
                ctx.ntt(got, inverse=inverse, coset=coset)
                want = oracle.ntt(x, log_n, inverse=inverse, coset=coset)
                assert np.array_equal(got, want), (inverse, coset, planted)
        # the coset load: data[j] * g^j
        x = synth.uniform_fr(synth.SplitMix64(2200 + log_n), n)
        planted = []
        for j in (1, 2, n - 1, rng.randrange(3, n - 3)):
            wj = pow(g, j, R)
            xv = short_quotient_input(wj, rng)
            _plant(x, j, xv, wj)
            planted.append((j, hex(xv)))
        got = x.copy()
        ctx.ntt(got, coset=True)
        assert np.array_equal(got, oracle.ntt(x, log_n, coset=True)), planted


def _edge_vectors(n):
    one_mont = (1 << 256) % R
    out = {
        "all r-1": F.ints_to_array([R - 1] * n),
        "alternating 0, r-1": F.ints_to_array([0 if i % 2 == 0 else R - 1 for i in range(n)]),
        "all Montgomery one": F.ints_to_array([one_mont] * n),
        "all zero": _zeros(n),
        "r-1 at the ends": F.ints_to_array([R - 1 if i in (0, n - 1) else 0 for i in range(n)]),
    }
    return out


@pytest.mark.parametrize("log_n", [6, 12, 18])
def test_edge_valued_vectors(log_n):
    n = 1 << log_n
    vecs = _edge_vectors(n)
    with g3h.Context(log_n) as ctx:
        for name, x in vecs.items():
            for inverse in (False, True):
                for coset in (False, True):
                    got = x.copy()
                    ctx.ntt(got, inverse=inverse, coset=coset)
                    want = oracle.ntt(x, log_n, inverse=inverse, coset=coset)
                    assert np.array_equal(got, want), (name, inverse, coset)
        names = list(vecs)
        for i, name in enumerate(names):
            a = vecs[name]
            b = vecs[names[(i + 1) % len(names)]]
            c = vecs[names[(i + 2) % len(names)]]
            want_m, want_s = oracle.compute_h_abc(log_n, a, b, c)
            hm, hs = _zeros(n), _zeros(n)
            ctx.compute_h_abc(a, b, c, hm, hs)
            assert np.array_equal(hm, want_m) and np.array_equal(hs, want_s), name
