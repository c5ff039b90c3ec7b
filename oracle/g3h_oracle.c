/*
 * CPU oracle for the Groth16 quotient-evaluation path over BN254 Fr.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library or its Python binding may call this;
 * only the tests, the package entry's smoke check and the benchmark's CPU-baseline leg do.
 *
 * Plain, slow and obviously correct: four 64-bit limbs with unsigned __int128 products
 * (the GPU path uses eight 32-bit limbs and shares no code with this file), textbook
 * Montgomery multiplication in CIOS form (Koc, Acar & Kaliski, IEEE Micro 1996), and a
 * textbook iterative radix-2 decimation-in-time NTT (bit-reverse, then passes of length
 * 2, 4, ..., n), as the snarkrs_gpu_kernels NTT_CU page describes its CPU backend
 * ("the algorithm is the CPU backend's": bit-reverse the input, then log n passes).
 *
 * What it computes (pages: NTT_CU header, POINTWISE_CU "no division by Z(coset)",
 * GATHER_CU g16_gather_abc):
 *   a_i = sum_j A[i,j] w_j,  b_i = sum_j B[i,j] w_j,  c_i = a_i b_i          (gather)
 *   x = n^-1 DFT_{omega^-1}(v) for v in {a, b, c}                            (iNTT)
 *   x_j <- x_j g^j, g a primitive 2n-th root with g^2 = omega                (coset shift)
 *   e = DFT_omega(x)                                                         (forward NTT)
 *   h_i = e_a[i] e_b[i] - e_c[i], written as h*R mod r and as h in [0, r)   (join)
 * The 1/n factor is applied after the inverse DFT, as the pages say their CPU backend
 * does; the GPU folds it elsewhere, which is the same linear map.
 *
 * Roots of unity (the pages name the element but do not print it): omega_{2^28} =
 * 5^((r-1)/2^28), 5 being a quadratic non-residue mod r; omega_n = omega_{2^28}^(2^(28-k))
 * and g = omega_{2^28}^(2^(27-k)), so g^2 = omega_n and g^n = -1.
 *
 * All field elements cross this file's interface as eight little-endian 32-bit limbs in
 * Montgomery form (R = 2^256) unless a function says otherwise, and every output is
 * canonical (< r).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef unsigned __int128 u128;
typedef struct {
  uint64_t l[4]; /* little-endian 64-bit limbs */
} fe;

/* r = 21888242871839275222246405745257275088548364400416034343698204186575808495617 */
static const fe P = {{0x43e1f593f0000001ULL, 0x2833e84879b97091ULL, 0xb85045b68181585dULL,
                      0x30644e72e131a029ULL}};

static uint64_t NP;   /* -r^-1 mod 2^64 */
static fe R1;         /* 2^256 mod r: the Montgomery form of 1 */
static fe R2;         /* 2^512 mod r */
static int inited = 0;

static int fe_geq(const fe* a, const fe* b) {
  for (int i = 3; i >= 0; i--) {
    if (a->l[i] > b->l[i]) return 1;
    if (a->l[i] < b->l[i]) return 0;
  }
  return 1;
}

/* a - b over 256 bits, returns the borrow */
static uint64_t raw_sub(fe* d, const fe* a, const fe* b) {
  uint64_t borrow = 0;
  for (int i = 0; i < 4; i++) {
    u128 t = (u128)a->l[i] - b->l[i] - borrow;
    d->l[i] = (uint64_t)t;
    borrow = (uint64_t)(t >> 64) & 1;
  }
  return borrow;
}

static uint64_t raw_add(fe* s, const fe* a, const fe* b) {
  uint64_t carry = 0;
  for (int i = 0; i < 4; i++) {
    u128 t = (u128)a->l[i] + b->l[i] + carry;
    s->l[i] = (uint64_t)t;
    carry = (uint64_t)(t >> 64);
  }
  return carry;
}

static fe fe_add(fe a, fe b) {
  fe s;
  uint64_t carry = raw_add(&s, &a, &b);
  if (carry || fe_geq(&s, &P)) raw_sub(&s, &s, &P);
  return s;
}

static fe fe_sub(fe a, fe b) {
  fe d;
  if (raw_sub(&d, &a, &b)) raw_add(&d, &d, &P);
  return d;
}

/* CIOS Montgomery product a*b*2^-256 mod r for canonical a, b. */
static fe fe_mont_mul(fe a, fe b) {
  uint64_t t[6] = {0, 0, 0, 0, 0, 0};
  for (int i = 0; i < 4; i++) {
    uint64_t C = 0;
    for (int j = 0; j < 4; j++) {
      u128 s = (u128)a.l[j] * b.l[i] + t[j] + C;
      t[j] = (uint64_t)s;
      C = (uint64_t)(s >> 64);
    }
    u128 s = (u128)t[4] + C;
    t[4] = (uint64_t)s;
    t[5] = (uint64_t)(s >> 64);
    uint64_t m = t[0] * NP;
    s = (u128)m * P.l[0] + t[0];
    C = (uint64_t)(s >> 64);
    for (int j = 1; j < 4; j++) {
      s = (u128)m * P.l[j] + t[j] + C;
      t[j - 1] = (uint64_t)s;
      C = (uint64_t)(s >> 64);
    }
    s = (u128)t[4] + C;
    t[3] = (uint64_t)s;
    C = (uint64_t)(s >> 64);
    t[4] = t[5] + C;
  }
  fe r;
  memcpy(r.l, t, sizeof(r.l));
  if (t[4] != 0 || fe_geq(&r, &P)) raw_sub(&r, &r, &P);
  return r;
}

static void init(void) {
  if (inited) return;
  /* Newton iteration for r^-1 mod 2^64: each step doubles the number of correct bits. */
  uint64_t inv = 1;
  for (int i = 0; i < 7; i++) inv *= 2 - P.l[0] * inv;
  NP = (uint64_t)0 - inv;
  /* 2^256 and 2^512 mod r by doubling 1 modulo r. */
  fe x = {{1, 0, 0, 0}};
  for (int i = 0; i < 512; i++) {
    x = fe_add(x, x);
    if (i == 255) R1 = x;
  }
  R2 = x;
  inited = 1;
}

static fe to_mont(fe a) { return fe_mont_mul(a, R2); }
static fe from_mont(fe a) {
  fe one = {{1, 0, 0, 0}};
  return fe_mont_mul(a, one);
}

static fe fe_pow(fe base_mont, fe e) {
  fe acc = R1;
  for (int i = 255; i >= 0; i--) {
    acc = fe_mont_mul(acc, acc);
    if ((e.l[i / 64] >> (i % 64)) & 1) acc = fe_mont_mul(acc, base_mont);
  }
  return acc;
}

static fe fe_inv(fe a_mont) {
  fe e = P;
  fe two = {{2, 0, 0, 0}};
  raw_sub(&e, &e, &two);
  return fe_pow(a_mont, e);
}

static fe load32(const uint32_t* p) {
  fe a;
  for (int i = 0; i < 4; i++) a.l[i] = (uint64_t)p[2 * i] | ((uint64_t)p[2 * i + 1] << 32);
  return a;
}

static void store32(uint32_t* p, fe a) {
  for (int i = 0; i < 4; i++) {
    p[2 * i] = (uint32_t)a.l[i];
    p[2 * i + 1] = (uint32_t)(a.l[i] >> 32);
  }
}

/* omega_{2^28} = 5^((r-1)/2^28), Montgomery form. */
static fe two_adic_root(void) {
  fe e = P;
  fe one = {{1, 0, 0, 0}};
  raw_sub(&e, &e, &one);
  for (int i = 0; i < 28; i++) { /* shift right by one bit, 28 times */
    for (int j = 0; j < 4; j++) e.l[j] = (e.l[j] >> 1) | (j < 3 ? (e.l[j + 1] << 63) : 0);
  }
  fe five = {{5, 0, 0, 0}};
  return fe_pow(to_mont(five), e);
}

/* omega_n (k squarings short of the 2^28-th root) and g with g^2 = omega_n. */
static void domain(unsigned log_n, fe* omega, fe* g) {
  fe w = two_adic_root();
  /* g = w^(2^(27-k)), omega = g^2 */
  for (unsigned i = 0; i < 27 - log_n; i++) w = fe_mont_mul(w, w);
  *g = w;
  *omega = fe_mont_mul(w, w);
}

static unsigned bitrev(unsigned x, unsigned bits) {
  unsigned y = 0;
  for (unsigned i = 0; i < bits; i++) y |= ((x >> i) & 1u) << (bits - 1 - i);
  return y;
}

/* In place: x <- DFT_w(x), i.e. x'_i = sum_j x_j w^(ij), w a primitive n-th root. */
static int dft_radix2(fe* x, unsigned log_n, fe w) {
  size_t n = (size_t)1 << log_n;
  for (size_t i = 0; i < n; i++) {
    size_t j = bitrev((unsigned)i, log_n);
    if (i < j) {
      fe t = x[i];
      x[i] = x[j];
      x[j] = t;
    }
  }
  fe* tw = (fe*)malloc(sizeof(fe) * (n / 2 + 1));
  if (!tw) return -1;
  for (unsigned s = 1; s <= log_n; s++) {
    size_t len = (size_t)1 << s, half = len / 2;
    /* wlen = w^(n/len), a primitive len-th root */
    fe wlen = w;
    for (unsigned i = 0; i < log_n - s; i++) wlen = fe_mont_mul(wlen, wlen);
    tw[0] = R1;
    for (size_t j = 1; j < half; j++) tw[j] = fe_mont_mul(tw[j - 1], wlen);
    for (size_t i = 0; i < n; i += len) {
      for (size_t j = 0; j < half; j++) {
        fe u = x[i + j];
        fe v = fe_mont_mul(x[i + j + half], tw[j]);
        x[i + j] = fe_add(u, v);
        x[i + j + half] = fe_sub(u, v);
      }
    }
  }
  free(tw);
  return 0;
}

/* ------------------------------------------------------------------ exported API ---- */

/* Field primitives on single elements (Montgomery in, Montgomery out). */
void orc_fr_mul(const uint32_t* a, const uint32_t* b, uint32_t* out) {
  init();
  store32(out, fe_mont_mul(load32(a), load32(b)));
}
void orc_fr_add(const uint32_t* a, const uint32_t* b, uint32_t* out) {
  init();
  store32(out, fe_add(load32(a), load32(b)));
}
void orc_fr_sub(const uint32_t* a, const uint32_t* b, uint32_t* out) {
  init();
  store32(out, fe_sub(load32(a), load32(b)));
}
/* out_i = a_i * b_i * 2^-256 for i < n (the product the gather forms for C). */
void orc_fr_mul_vec(const uint32_t* a, const uint32_t* b, uint32_t* out, size_t n) {
  init();
  for (size_t i = 0; i < n; i++)
    store32(out + 8 * i, fe_mont_mul(load32(a + 8 * i), load32(b + 8 * i)));
}

/* Montgomery -> standard and back, on n elements. */
void orc_from_mont(const uint32_t* in, uint32_t* out, size_t n) {
  init();
  for (size_t i = 0; i < n; i++) store32(out + 8 * i, from_mont(load32(in + 8 * i)));
}
void orc_to_mont(const uint32_t* in, uint32_t* out, size_t n) {
  init();
  for (size_t i = 0; i < n; i++) store32(out + 8 * i, to_mont(load32(in + 8 * i)));
}

/* omega_n and g in standard form (not Montgomery), for the pins. */
/* sum_j coeffs[j] z^j over j < n by Horner's rule; coeffs and z Montgomery, out Montgomery
 * (canonical). The definition of a forward transform's output e[i] = P(omega^i), or
 * P(g omega^i) on the coset, one point at a time. */
void orc_poly_eval(size_t n, const uint32_t* coeffs, const uint32_t* z, uint32_t* out) {
  init();
  const fe zz = load32(z);
  fe acc = {{0, 0, 0, 0}};
  for (size_t j = n; j-- > 0;) acc = fe_add(fe_mont_mul(acc, zz), load32(coeffs + 8 * j));
  store32(out, acc);
}

int orc_domain(unsigned log_n, uint32_t* omega_std, uint32_t* g_std) {
  init();
  if (log_n > 27) return -1;
  fe w, g;
  domain(log_n, &w, &g);
  store32(omega_std, from_mont(w));
  store32(g_std, from_mont(g));
  return 0;
}

/*
 * Transform of one vector of n = 2^log_n Montgomery elements, in place.
 *   inverse = 0: x <- DFT_omega(c), c = x, or c_j = x_j g^j when coset != 0
 *   inverse = 1: x <- n^-1 DFT_omega^-1(x), then x_j <- x_j g^-j when coset != 0
 * so the inverse undoes the forward for either coset setting.
 */
int orc_ntt(unsigned log_n, uint32_t* data, int inverse, int coset) {
  init();
  if (log_n > 27) return -1;
  size_t n = (size_t)1 << log_n;
  fe w, g;
  domain(log_n, &w, &g);
  fe* x = (fe*)malloc(sizeof(fe) * n);
  if (!x) return -2;
  for (size_t i = 0; i < n; i++) x[i] = load32(data + 8 * i);
  int rc = 0;
  if (!inverse) {
    if (coset) {
      fe gp = R1;
      for (size_t j = 0; j < n; j++) {
        x[j] = fe_mont_mul(x[j], gp);
        gp = fe_mont_mul(gp, g);
      }
    }
    rc = dft_radix2(x, log_n, w);
  } else {
    rc = dft_radix2(x, log_n, fe_inv(w));
    fe ninv = fe_inv(to_mont((fe){{(uint64_t)n, 0, 0, 0}}));
    for (size_t j = 0; j < n; j++) x[j] = fe_mont_mul(x[j], ninv);
    if (coset) {
      fe ginv = fe_inv(g), gp = R1;
      for (size_t j = 0; j < n; j++) {
        x[j] = fe_mont_mul(x[j], gp);
        gp = fe_mont_mul(gp, ginv);
      }
    }
  }
  for (size_t i = 0; i < n; i++) store32(data + 8 * i, x[i]);
  free(x);
  return rc;
}

/*
 * The gather (GATHER_CU, g16_gather_abc): for i < n,
 *   a_i = sum over CSR row i of A.val[k] * w[A.col[k]], likewise b_i, c_i = a_i * b_i;
 * rows at or beyond n_rows are empty. row_ptr has n_rows + 1 entries.
 */
static void gather(size_t n, size_t n_rows, const uint32_t* ra, const uint32_t* ca,
                   const uint32_t* va, const uint32_t* rb, const uint32_t* cb,
                   const uint32_t* vb, const uint32_t* w, fe* a, fe* b, fe* c) {
  fe zero = {{0, 0, 0, 0}};
  for (size_t i = 0; i < n; i++) {
    fe sa = zero, sb = zero;
    if (i < n_rows) {
      for (uint32_t k = ra[i]; k < ra[i + 1]; k++)
        sa = fe_add(sa, fe_mont_mul(load32(va + 8 * (size_t)k), load32(w + 8 * (size_t)ca[k])));
      for (uint32_t k = rb[i]; k < rb[i + 1]; k++)
        sb = fe_add(sb, fe_mont_mul(load32(vb + 8 * (size_t)k), load32(w + 8 * (size_t)cb[k])));
    }
    a[i] = sa;
    b[i] = sb;
    c[i] = fe_mont_mul(sa, sb);
  }
}

int orc_gather(unsigned log_n, size_t n_rows, const uint32_t* ra, const uint32_t* ca,
               const uint32_t* va, const uint32_t* rb, const uint32_t* cb, const uint32_t* vb,
               const uint32_t* w, uint32_t* a_out, uint32_t* b_out, uint32_t* c_out) {
  init();
  size_t n = (size_t)1 << log_n;
  fe* v = (fe*)malloc(sizeof(fe) * 3 * n);
  if (!v) return -2;
  gather(n, n_rows, ra, ca, va, rb, cb, vb, w, v, v + n, v + 2 * n);
  for (size_t i = 0; i < n; i++) {
    store32(a_out + 8 * i, v[i]);
    store32(b_out + 8 * i, v[n + i]);
    store32(c_out + 8 * i, v[2 * n + i]);
  }
  free(v);
  return 0;
}

/* Steps 2-5 on evaluation vectors a, b, c already in memory (fe, Montgomery). */
static int quotient_evals(unsigned log_n, fe* v /* 3n: a | b | c */, uint32_t* h_mont,
                          uint32_t* h_std) {
  size_t n = (size_t)1 << log_n;
  fe w, g;
  domain(log_n, &w, &g);
  fe winv = fe_inv(w);
  fe ninv = fe_inv(to_mont((fe){{(uint64_t)n, 0, 0, 0}}));
  for (int s = 0; s < 3; s++) {
    fe* x = v + (size_t)s * n;
    /* interpolate: coefficients of the degree < n polynomial through the evaluations */
    if (dft_radix2(x, log_n, winv)) return -2;
    for (size_t j = 0; j < n; j++) x[j] = fe_mont_mul(x[j], ninv);
    /* coset shift */
    fe gp = R1;
    for (size_t j = 0; j < n; j++) {
      x[j] = fe_mont_mul(x[j], gp);
      gp = fe_mont_mul(gp, g);
    }
    /* evaluate on g * <omega> */
    if (dft_radix2(x, log_n, w)) return -2;
  }
  for (size_t i = 0; i < n; i++) {
    fe h = fe_sub(fe_mont_mul(v[i], v[n + i]), v[2 * n + i]);
    store32(h_mont + 8 * i, h);
    store32(h_std + 8 * i, from_mont(h));
  }
  return 0;
}

int orc_compute_h(unsigned log_n, size_t n_rows, const uint32_t* ra, const uint32_t* ca,
                  const uint32_t* va, const uint32_t* rb, const uint32_t* cb,
                  const uint32_t* vb, const uint32_t* w, uint32_t* h_mont, uint32_t* h_std) {
  init();
  if (log_n > 27) return -1;
  size_t n = (size_t)1 << log_n;
  if (n_rows > n) return -1;
  fe* v = (fe*)malloc(sizeof(fe) * 3 * n);
  if (!v) return -2;
  gather(n, n_rows, ra, ca, va, rb, cb, vb, w, v, v + n, v + 2 * n);
  int rc = quotient_evals(log_n, v, h_mont, h_std);
  free(v);
  return rc;
}

int orc_compute_h_abc(unsigned log_n, const uint32_t* a, const uint32_t* b, const uint32_t* c,
                      uint32_t* h_mont, uint32_t* h_std) {
  init();
  if (log_n > 27) return -1;
  size_t n = (size_t)1 << log_n;
  fe* v = (fe*)malloc(sizeof(fe) * 3 * n);
  if (!v) return -2;
  for (size_t i = 0; i < n; i++) {
    v[i] = load32(a + 8 * i);
    v[n + i] = load32(b + 8 * i);
    v[2 * n + i] = load32(c + 8 * i);
  }
  int rc = quotient_evals(log_n, v, h_mont, h_std);
  free(v);
  return rc;
}
