"""The constant multiply's quotient truncation, on the CPU (no GPU): the model of the
library's computation agrees with x * w mod r, its result stays below 2r for every operand
the library can pass (values below 2r) even at the extremes of the bound, and inputs that
make the quotient come out one short can be constructed for real table constants (the GPU
tests run them through the transforms)."""
import random

from oracle import fr_int as F
from shoup_model import BETA, R, dropped_columns, shoup_model, short_quotient_input, w_prime


def test_model_is_a_product_mod_r_below_2r():
    rng = random.Random(7)
    for _ in range(3000):
        x, w = rng.randrange(2 * R), rng.randrange(R)
        y, _ = shoup_model(x, w)
        assert 0 <= y < 2 * R and y % R == x * w % R


def test_dropped_columns_bound():
    # six columns of at most k + 1 products of 32-bit limbs: below 6.01 * 2^224 < 2^227
    worst = (1 << 256) - 1
    for w in (R - 1, (1 << 253) + 12345, 1):
        assert dropped_columns(worst, w) < (1 << 227)
    d_max = sum((k + 1) * (2**32 - 1) ** 2 << (32 * k) for k in range(6))
    assert d_max < 6.01 * 2**224 < 2**227


def _constant_with_remainder(delta):
    """w < r with w * 2^256 = r - delta (mod r): the largest remainder e = r - delta."""
    return (-delta * pow(BETA, -1, R)) % R


def test_result_below_2r_at_the_extremes():
    # y = (rho r + x e) / 2^256 + (r if the quotient is short): largest with x near 2r, the
    # remainder e near r, and the quotient short; still below 2r.
    rng = random.Random(11)
    for delta in (1, 2, 3, 1 << 20, 1 << 200):
        w = _constant_with_remainder(delta)
        assert (w * BETA) % R == R - delta
        for x in (2 * R - 1, 2 * R - 2, 2 * R - (1 << 64), (1 << 255) + (1 << 254)):
            if x >= 2 * R:
                continue
            y, _ = shoup_model(x, w)
            assert 0 <= y < 2 * R
        # short quotient with the largest remainder: x * w' = t (mod 2^256), t just below the
        # dropped columns' sum
        wp = w_prime(w)
        v = (wp & -wp).bit_length() - 1
        uinv = pow(wp >> v, -1, 1 << (256 - v))
        found = 0
        for _ in range(400):
            t = rng.getrandbits(200) | 1
            x = (t * uinv) % (1 << (256 - v))
            if x >= 2 * R:
                continue
            y, short = shoup_model(x, w)
            assert 0 <= y < 2 * R
            found += short
        assert found > 0


def test_short_quotient_inputs_for_table_constants():
    rng = random.Random(3)
    for log_n in (12, 18, 22):
        omega, g = F.domain(log_n)
        n = 1 << log_n
        for w in (pow(F.inv(omega), 1, R), pow(omega, n // 4, R), pow(g, n - 1, R)):
            x = short_quotient_input(w, rng)
            y, short = shoup_model(x, w)
            assert short and x < R and R <= y < 2 * R and y % R == x * w % R


def test_random_products_almost_never_short():
    rng = random.Random(5)
    assert sum(shoup_model(rng.randrange(R), rng.randrange(R))[1] for _ in range(5000)) == 0
