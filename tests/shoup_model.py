"""Inputs that drive the library's constant multiply through its rare short quotient.

Test infrastructure. The library multiplies data by table constants (twiddles, the coset
shift, scales) with Shoup's method at beta = 2^256: for a constant w < r it keeps
w' = floor(w * 2^256 / r), forms the quotient q from the columns i + j >= 6 of the limb
product x * w' only (eight 32-bit limbs each), and returns y = x*w - q*r. Dropping the low
columns makes q one short of floor(x * w' / 2^256) when those columns would have carried
into bit 256, which puts y in [r, 2r) instead of [0, r): about once in 2^29 random
products, so random test vectors essentially never reach it.

`shoup_model` restates that computation on Python ints (exactly the set of products the
library sums) and reports whether the quotient came out short; `short_quotient_input`
constructs an x < r for a given constant w whose quotient does, by choosing x with
x * w' = t (mod 2^256) for a small odd t, so that the dropped columns carry. Expected
values never come from here: the tests compare the library with the oracle on vectors that
contain these x.
"""
R = 21888242871839275222246405745257275088548364400416034343698204186575808495617
BETA = 1 << 256
MASK32 = 0xFFFFFFFF


def limbs(x):
    return [(x >> (32 * i)) & MASK32 for i in range(8)]


def w_prime(w):
    return (w * BETA) // R


def dropped_columns(x, w):
    """The sum of the limb products x_i w'_j 2^(32(i+j)) with i + j < 6."""
    xl, wl = limbs(x), limbs(w_prime(w))
    return sum((xl[i] * wl[j]) << (32 * (i + j)) for i in range(8) for j in range(8) if i + j < 6)


def shoup_model(x, w):
    """(y, short) of the library's constant multiply of x by the constant w < r: y = x*w -
    q*r with q from the columns i + j >= 6, and whether q fell one short of
    floor(x * w' / 2^256)."""
    wp = w_prime(w)
    xl, wl = limbs(x), limbs(wp)
    s = sum((xl[i] * wl[j]) << (32 * (i + j)) for i in range(8) for j in range(8) if i + j >= 6)
    q = s >> 256
    q_full = (x * wp) >> 256
    assert q_full - q in (0, 1)
    return x * w - q * R, q != q_full


def short_quotient_input(w, rng, tries=10000):
    """An x in [0, r) whose product with the constant w has the short quotient.
    rng: a random.Random."""
    wp = w_prime(w)
    v = (wp & -wp).bit_length() - 1 if wp else 0
    u = wp >> v
    bits = 256 - v
    uinv = pow(u, -1, 1 << bits)
    for _ in range(tries):
        t = (rng.getrandbits(160) | 1) << v
        x = ((t >> v) * uinv) % (1 << bits)
        if v:
            x |= rng.getrandbits(v) << bits
        if x < R and shoup_model(x, w)[1]:
            return x
    raise RuntimeError("no input found")
