"""Seeded synthetic inputs for the multi-scalar multiplication over BN254 G1.

The H multiexp takes the proving key's H bases, which are not available; the generator
stands in with points drawn uniformly at random on the curve y^2 = x^3 + 3 over F_q (the
curve has cofactor 1, so every such point is in G1), and with scalars uniform in [0, r)
in standard form (the distribution of h, a vector of evaluations of a random-looking
polynomial).

Sampling a point takes field arithmetic, but none of the multi-scalar multiplication's
point arithmetic (no point additions or doublings): draw x uniform in [0, q), take
y = (x^3 + 3)^((q+1)/4) (a square root, q = 3 mod 4) and keep (x, y) when y^2 = x^3 + 3.
Each accepted x gives six points at no further exponentiation, through the curve's
automorphisms (x, y) -> (beta^j x, +-y), beta a primitive cube root of unity mod q; the
six are consecutive in the output. Coordinates are then written in Montgomery form
(x * 2^256 mod q), eight little-endian uint32 limbs each, x then y.

Random numbers come from the same splitmix64 streams as the quotient-path inputs.
"""
import numpy as np

from .synth import SplitMix64, uniform_fr

Q_MOD = 21888242871839275222246405745257275088696311157297823662689037894645226208583
_SQRT_EXP = (Q_MOD + 1) // 4


def _cube_root_of_unity():
    for g in range(2, 100):
        beta = pow(g, (Q_MOD - 1) // 3, Q_MOD)
        if beta != 1:
            return beta
    raise AssertionError("no cubic non-residue below 100")


_BETA = _cube_root_of_unity()
_BETA2 = _BETA * _BETA % Q_MOD


def _limbs(v):
    return [(v >> (32 * k)) & 0xFFFFFFFF for k in range(8)]


def points(count, seed):
    """count affine points, shape (count, 16) uint32, Montgomery form, none at infinity."""
    rng = SplitMix64(seed)
    out = np.zeros((count, 16), np.uint32)
    filled = 0
    r256 = (1 << 256) % Q_MOD
    while filled < count:
        words = rng.u32(8)
        x = sum(int(words[k]) << (32 * k) for k in range(8)) & ((1 << 254) - 1)
        if x >= Q_MOD:
            continue
        rhs = (x * x * x + 3) % Q_MOD
        y = pow(rhs, _SQRT_EXP, Q_MOD)
        if y * y % Q_MOD != rhs:
            continue
        for xx in (x, _BETA * x % Q_MOD, _BETA2 * x % Q_MOD):
            for yy in (y, (Q_MOD - y) % Q_MOD):
                if filled == count:
                    break
                out[filled, :8] = _limbs(xx * r256 % Q_MOD)
                out[filled, 8:] = _limbs(yy * r256 % Q_MOD)
                filled += 1
    return out


def scalars(count, seed):
    """count scalars uniform in [0, r), standard form, shape (count, 8) uint32."""
    return uniform_fr(SplitMix64(seed), count)


def default_seed(log_n):
    return 0x67340000 + log_n
