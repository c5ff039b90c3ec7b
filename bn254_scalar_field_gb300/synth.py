"""Seeded synthetic inputs for the Groth16 quotient-evaluation path (BN254 Fr).

This module holds no field arithmetic: it draws integers, compares them with the modulus
and lays them out. Both the CUDA path's tests and the oracle's tests take their inputs
from here, so neither side generates data the other consumes.

Random numbers come from splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), one counter-based stream per seed.

Field elements are eight little-endian uint32 limbs. A uniform integer in [0, r) is a
uniform field element whatever encoding it is read in, so the uniform draws below are
used directly as Montgomery-form values; the only other values placed are 0 and the
Montgomery form of 1 (2^256 mod r), which is stored here as data.

Workloads ("snarkrs_gpu_kernels" GATHER_CU page, table of the real proving keys
js_1x1_d8 ... js_16x16_d32: mean row length, empty rows and longest row of A and B):
the proving keys themselves are not available, so the generator reproduces those
statistics and nothing else:
  * rows [m, n) are empty (the domain rounds up past the constraint count m); B has a
    few extra empty rows chosen uniformly among the constraint rows;
  * non-empty row lengths are 1 + geometric, fitted to the mean, capped at the longest
    row; one row has exactly the longest length, and the total equals the page's
    mean x n exactly;
  * column indices are uniform over the wires, distinct and sorted within a row (the
    CSR sort the pages rely on); coefficients are uniform field elements;
  * the witness has w[0] = 1 and a fraction of wires in {0, 1} (half each), the rest
    uniform.
"""
import numpy as np

# r, little-endian 32-bit limbs.
MODULUS_LIMBS = np.array([0xF0000001, 0x43E1F593, 0x79B97091, 0x2833E848, 0x8181585D,
                          0xB85045B6, 0xE131A029, 0x30644E72], dtype=np.uint32)
# 2^256 mod r: the Montgomery representative of 1.
MONT_ONE_LIMBS = np.array([0x4FFFFFFB, 0xAC96341C, 0x9F60CD29, 0x36FC7695, 0x7879462E,
                           0x666EA36F, 0x9A07DF2F, 0x0E0A77C1], dtype=np.uint32)

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


class SplitMix64:
    """Counter-based splitmix64: output i is mix(seed + (i + 1) * golden)."""

    def __init__(self, seed):
        self.seed = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        self.counter = 0

    def u64(self, count):
        idx = np.arange(self.counter + 1, self.counter + 1 + count, dtype=np.uint64)
        self.counter += count
        with np.errstate(over="ignore"):
            z = self.seed + idx * _GOLDEN
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))

    def u32(self, count):
        return self.u64((count + 1) // 2).view(np.uint32)[:count].copy()

    def uniform(self, count):
        """Doubles in [0, 1) from the top 53 bits."""
        return (self.u64(count) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))

    def below(self, bound, count):
        """Integers in [0, bound) (bound <= 2^32; exact when bound is a power of two)."""
        return (self.u64(count) % np.uint64(bound)).astype(np.int64)


def _less_than_modulus(x):
    less = np.zeros(x.shape[0], dtype=bool)
    eq = np.ones(x.shape[0], dtype=bool)
    for w in range(7, -1, -1):
        less |= eq & (x[:, w] < MODULUS_LIMBS[w])
        eq &= x[:, w] == MODULUS_LIMBS[w]
    return less


def uniform_fr(rng, count):
    """count uniform elements of [0, r) by rejection sampling 254-bit integers."""
    out = np.empty((count, 8), dtype=np.uint32)
    filled = 0
    while filled < count:
        want = count - filled
        draw = int(want * 1.35) + 16
        x = rng.u32(draw * 8).reshape(draw, 8)
        x[:, 7] &= np.uint32(0x3FFFFFFF)
        x = x[_less_than_modulus(x)][:want]
        out[filled:filled + x.shape[0]] = x
        filled += x.shape[0]
    return out


def witness(rng, n_wires, frac01):
    """w[0] = 1; a fraction frac01 of the other wires in {0, 1}, half each; rest uniform."""
    w = uniform_fr(rng, n_wires)
    u = rng.uniform(n_wires)
    small = u < frac01
    one = u < frac01 / 2
    w[small] = 0
    w[one] = MONT_ONE_LIMBS
    if n_wires:
        w[0] = MONT_ONE_LIMBS
    return w


def _row_lengths(rng, n_nonempty, nnz, max_len):
    if n_nonempty == 0:
        return np.zeros(0, np.int64)
    mean_extra = nnz / n_nonempty - 1.0
    if mean_extra <= 0:
        lens = np.ones(n_nonempty, np.int64)
    else:
        q = 1.0 / (1.0 + mean_extra)
        u = rng.uniform(n_nonempty)
        lens = 1 + np.floor(np.log1p(-u) / np.log1p(-q)).astype(np.int64)
    lens = np.minimum(lens, max_len)
    forced = int(rng.below(n_nonempty, 1)[0])
    lens[forced] = max_len
    # Move the total onto nnz exactly, one term at a time on random rows.
    diff = int(lens.sum()) - nnz
    while diff != 0:
        picks = rng.below(n_nonempty, max(64, 2 * abs(diff)))
        for p in picks:
            if diff == 0:
                break
            if p == forced:
                continue
            if diff > 0 and lens[p] > 1:
                lens[p] -= 1
                diff -= 1
            elif diff < 0 and lens[p] < max_len:
                lens[p] += 1
                diff += 1
    return lens


def _columns(rng, row_of_term, n_wires):
    """Distinct, sorted column indices per row."""
    nnz = row_of_term.shape[0]
    cols = rng.below(n_wires, nnz)
    while True:
        order = np.lexsort((cols, row_of_term))
        cols = cols[order]  # row_of_term is already sorted, so only cols move
        dup = np.zeros(nnz, dtype=bool)
        if nnz > 1:
            dup[1:] = (row_of_term[1:] == row_of_term[:-1]) & (cols[1:] == cols[:-1])
        k = int(dup.sum())
        if k == 0:
            return cols
        cols[dup] = rng.below(n_wires, k)


def csr(rng, n, nonempty_rows, nnz, max_len, n_wires):
    """A CSR matrix with n rows (row_ptr has n + 1 entries), non-empty exactly on the rows
    listed in nonempty_rows, nnz terms, longest row max_len."""
    nonempty_rows = np.asarray(nonempty_rows, dtype=np.int64)
    lens_ne = _row_lengths(rng, nonempty_rows.shape[0], nnz, max_len)
    lens = np.zeros(n, np.int64)
    lens[nonempty_rows] = lens_ne
    row_ptr = np.zeros(n + 1, np.int64)
    np.cumsum(lens, out=row_ptr[1:])
    row_of_term = np.repeat(np.arange(n, dtype=np.int64), lens)
    cols = _columns(rng, row_of_term, n_wires)
    vals = uniform_fr(rng, nnz)
    return row_ptr.astype(np.uint32), cols.astype(np.uint32), vals


# Row statistics of the proving keys on the GATHER_CU page, with nnz = mean x n.
CONFIGS = {
    12: dict(n_wires=4096, m=3364, extra_b_empty=5, nnz_a=9462, nnz_b=15155,
             max_a=65, max_b=64, frac01=0.90),
    14: dict(n_wires=16384, m=10160, extra_b_empty=7, nnz_a=24740, nnz_b=38339,
             max_a=67, max_b=66, frac01=0.95),
    17: dict(n_wires=131072, m=70376, extra_b_empty=19, nnz_a=148111, nnz_b=222822,
             max_a=79, max_b=78, frac01=0.99),
    18: dict(n_wires=262144, m=140296, extra_b_empty=35, nnz_a=296223, nnz_b=443023,
             max_a=95, max_b=94, frac01=0.99),
}
STRESS_LOG_N = 22


def default_seed(log_n):
    return 0x67330000 + log_n


def problem(log_n, seed=None, **overrides):
    """A (row_ptr, col, val), B (row_ptr, col, val) and witness w for a proving-key-shaped
    domain of 2^log_n. log_n in CONFIGS uses the page's statistics; other sizes scale the
    2^12 shape (constraint fraction, row means, caps) down or up."""
    n = 1 << log_n
    if log_n in CONFIGS:
        cfg = dict(CONFIGS[log_n])
    else:
        base = CONFIGS[12]
        scale = n / 4096.0
        cfg = dict(n_wires=max(1, n), m=max(0, int(round(base["m"] * scale))),
                   extra_b_empty=int(round(base["extra_b_empty"] * scale)),
                   nnz_a=int(round(base["nnz_a"] * scale)),
                   nnz_b=int(round(base["nnz_b"] * scale)),
                   max_a=min(base["max_a"], max(1, n)), max_b=min(base["max_b"], max(1, n)),
                   frac01=base["frac01"])
    cfg.update(overrides)
    rng = SplitMix64(default_seed(log_n) if seed is None else seed)
    m = min(cfg["m"], n)
    rows_a = np.arange(m, dtype=np.int64)
    extra = min(cfg["extra_b_empty"], m)
    drop = np.unique(rng.below(max(m, 1), extra)) if extra else np.zeros(0, np.int64)
    rows_b = np.setdiff1d(rows_a, drop)
    nnz_a = min(cfg["nnz_a"], rows_a.shape[0] * min(cfg["max_a"], cfg["n_wires"]))
    nnz_b = min(cfg["nnz_b"], rows_b.shape[0] * min(cfg["max_b"], cfg["n_wires"]))
    nnz_a = max(nnz_a, rows_a.shape[0])
    nnz_b = max(nnz_b, rows_b.shape[0])
    max_a = min(cfg["max_a"], cfg["n_wires"])
    max_b = min(cfg["max_b"], cfg["n_wires"])
    A = csr(rng, n, rows_a, nnz_a, max_a, cfg["n_wires"])
    B = csr(rng, n, rows_b, nnz_b, max_b, cfg["n_wires"])
    w = witness(rng, cfg["n_wires"], cfg["frac01"])
    return A, B, w


def stress_ab(log_n=STRESS_LOG_N, seed=None):
    """The NTT stress workload's a and b: uniform field elements. Its c is a*b (pointwise),
    which the caller forms with field arithmetic this module does not hold."""
    rng = SplitMix64(default_seed(log_n) if seed is None else seed)
    n = 1 << log_n
    return uniform_fr(rng, n), uniform_fr(rng, n)
