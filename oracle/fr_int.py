"""Pure-Python integer reference for the Groth16 quotient-evaluation path over BN254 Fr.

TEST INFRASTRUCTURE ONLY: the library never imports this module; the tests, the package
entry's smoke check and the benchmark's CPU-baseline leg may.

Everything is plain modular arithmetic on Python ints in STANDARD form (the integer in
[0, r)); the Montgomery encoding (x * 2^256 mod r) appears only in ``to_mont`` /
``from_mont`` at the boundary. Pure-Python loops, so only for small domains.

Sources (snarkrs_gpu_kernels pages):
  * NTT_CU, header "the algorithm is the CPU backend's, exactly": the transform pair, the
    1/n of the inverse, and the coset shift x[j] *= g^j with g a primitive 2n-th root of
    unity that is not the field generator;
  * POINTWISE_CU, "no division by Z(coset)": h = a*b - c with no division, the points being
    the odd powers of the 2n-th root; "two output buffers": the Montgomery and standard
    encodings of h;
  * GATHER_CU, g16_gather_abc: a_i = sum_j A[i,j] w_j, b_i likewise, c_i = a_i * b_i.

Reading taken where the pages are silent: the 2^28-th root of unity is
5^((r-1)/2^28) (5 is a quadratic non-residue mod r, so this has order exactly 2^28), and
omega_n = w^(2^(28-k)), g = w^(2^(27-k)) come from that one tower, so g^2 = omega_n.
"""

R_MOD = 21888242871839275222246405745257275088548364400416034343698204186575808495617
TWO_ADICITY = 28
MONT_R = 1 << 256
NON_RESIDUE = 5


def two_adic_root():
    """A primitive 2^28-th root of unity: 5^((r-1)/2^28)."""
    return pow(NON_RESIDUE, (R_MOD - 1) >> TWO_ADICITY, R_MOD)


def domain(log_n):
    """(omega_n, g) for n = 2^log_n: omega_n generates the order-n subgroup, g^2 = omega_n."""
    if not 0 <= log_n <= TWO_ADICITY - 1:
        raise ValueError("log_n must be in [0, 27]")
    w = two_adic_root()
    g = pow(w, 1 << (TWO_ADICITY - 1 - log_n), R_MOD)
    return g * g % R_MOD, g


def inv(x):
    return pow(x, R_MOD - 2, R_MOD)


def to_mont(x):
    return x * MONT_R % R_MOD


def from_mont(x):
    return x * inv(MONT_R % R_MOD) % R_MOD


# ---------------------------------------------------------------- limb conversion ----

def limbs_to_int(row):
    """Eight little-endian u32 limbs -> int."""
    v = 0
    for i in range(7, -1, -1):
        v = (v << 32) | int(row[i])
    return v


def int_to_limbs(x):
    return [(x >> (32 * i)) & 0xFFFFFFFF for i in range(8)]


def array_to_ints(arr):
    """(m, 8) uint32 array -> list of ints."""
    return [limbs_to_int(r) for r in arr.reshape(-1, 8)]


def ints_to_array(vals):
    import numpy as np

    out = np.zeros((len(vals), 8), dtype=np.uint32)
    for i, v in enumerate(vals):
        out[i] = int_to_limbs(v)
    return out


# --------------------------------------------------------------------- transforms ----

def dft_naive(x, w):
    """X_i = sum_j x_j w^(ij): the definition, O(n^2)."""
    n = len(x)
    out = []
    for i in range(n):
        wi = pow(w, i, R_MOD)
        acc, p = 0, 1
        for j in range(n):
            acc = (acc + x[j] * p) % R_MOD
            p = p * wi % R_MOD
        out.append(acc)
    return out


def dft_recursive(x, w):
    """The same DFT by the textbook radix-2 split into even and odd halves."""
    n = len(x)
    if n == 1:
        return [x[0] % R_MOD]
    w2 = w * w % R_MOD
    even = dft_recursive(x[0::2], w2)
    odd = dft_recursive(x[1::2], w2)
    out = [0] * n
    p = 1
    for i in range(n // 2):
        t = odd[i] * p % R_MOD
        out[i] = (even[i] + t) % R_MOD
        out[i + n // 2] = (even[i] - t) % R_MOD
        p = p * w % R_MOD
    return out


def interpolate(evals, log_n):
    """Coefficients of the degree < n polynomial with P(omega^i) = evals[i]."""
    omega, _ = domain(log_n)
    n = 1 << log_n
    coeffs = dft_recursive(evals, inv(omega))
    ninv = inv(n)
    return [c * ninv % R_MOD for c in coeffs]


def coset_evaluate(coeffs, log_n):
    """P(g * omega^i) for i < n from the coefficients: shift by g^j, then the DFT."""
    omega, g = domain(log_n)
    shifted = []
    p = 1
    for c in coeffs:
        shifted.append(c * p % R_MOD)
        p = p * g % R_MOD
    return dft_recursive(shifted, omega)


def poly_eval(coeffs, z):
    acc = 0
    for c in reversed(coeffs):
        acc = (acc * z + c) % R_MOD
    return acc


# ----------------------------------------------------------------------- pipeline ----

def gather(n, row_ptr_a, col_a, val_a, row_ptr_b, col_b, val_b, w):
    """a_i = sum_j A[i,j] w_j, b_i likewise, c_i = a_i b_i, for i < n (standard-form ints).

    row_ptr has n_rows + 1 entries; rows from n_rows to n - 1 are empty.
    """
    n_rows = len(row_ptr_a) - 1
    a, b, c = [0] * n, [0] * n, [0] * n
    for i in range(min(n, n_rows)):
        sa = 0
        for k in range(row_ptr_a[i], row_ptr_a[i + 1]):
            sa = (sa + val_a[k] * w[col_a[k]]) % R_MOD
        sb = 0
        for k in range(row_ptr_b[i], row_ptr_b[i + 1]):
            sb = (sb + val_b[k] * w[col_b[k]]) % R_MOD
        a[i], b[i] = sa, sb
    for i in range(n):
        c[i] = a[i] * b[i] % R_MOD
    return a, b, c


def quotient_evals(log_n, a, b, c):
    """h_i = A(g w^i) B(g w^i) - C(g w^i), A, B, C the interpolants of a, b, c on <w>."""
    ea = coset_evaluate(interpolate(a, log_n), log_n)
    eb = coset_evaluate(interpolate(b, log_n), log_n)
    ec = coset_evaluate(interpolate(c, log_n), log_n)
    return [(x * y - z) % R_MOD for x, y, z in zip(ea, eb, ec)]


def compute_h(log_n, row_ptr_a, col_a, val_a, row_ptr_b, col_b, val_b, w):
    """The whole path on standard-form ints; returns h as standard-form ints."""
    n = 1 << log_n
    a, b, c = gather(n, row_ptr_a, col_a, val_a, row_ptr_b, col_b, val_b, w)
    return quotient_evals(log_n, a, b, c)
