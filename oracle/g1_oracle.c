/*
 * CPU oracle for the multi-scalar multiplication over BN254 G1 (the H multiexp).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library or its Python binding may call this;
 * only the tests, the package entry's smoke check and the benchmark's CPU-baseline leg do.
 *
 * What it computes (snarkrs_gpu_kernels pages, MSM_CU header "stages 5-9": Pippenger
 * over G1, stage 9 being the H multiexp on the standard-form h of POINTWISE_CU):
 *     Q = sum_i s_i * P_i   on E: y^2 = x^3 + 3 over F_q,
 * by the definition: each s_i * P_i by left-to-right double-and-add over the bits of the
 * integer s_i, summed in order. No buckets, no windows.
 *
 * Plain and slow: F_q in four 64-bit limbs with unsigned __int128 products and textbook
 * CIOS Montgomery multiplication (Koc, Acar & Kaliski, IEEE Micro 1996); points in
 * Jacobian coordinates (x = X/Z^2, y = Y/Z^3), with the doubling and addition formulas
 * obtained by substituting those into the affine tangent and chord formulas (as in
 * Cohen, Miyaji & Ono, "Efficient elliptic curve exponentiation using mixed coordinates",
 * ASIACRYPT 1998), the equal-x cases of the chord handled explicitly. The GPU path uses
 * eight 32-bit limbs and the (X, Y, ZZ, ZZZ) coordinates and shares no code with this
 * file.
 *
 * Interface: coordinates are eight little-endian 32-bit limbs in Montgomery form
 * (2^256 mod q); an affine point is x then y (16 limbs), the point at infinity written as
 * x = y = 0 (not on the curve, since 0 != 3); a Jacobian point is X, Y, Z (24 limbs).
 * Scalars are eight limbs in standard form (the integer), any 256-bit value.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef unsigned __int128 u128;
typedef struct {
  uint64_t l[4];
} fq;

/* q = 21888242871839275222246405745257275088696311157297823662689037894645226208583 */
static const fq Q = {{0x3c208c16d87cfd47ULL, 0x97816a916871ca8dULL, 0xb85045b68181585dULL,
                      0x30644e72e131a029ULL}};
static uint64_t QINV; /* -q^-1 mod 2^64 */
static fq ONE;        /* 2^256 mod q */
static fq R2Q;        /* 2^512 mod q */
static int ready = 0;

static int fq_geq(const fq* a, const fq* b) {
  for (int i = 3; i >= 0; i--) {
    if (a->l[i] != b->l[i]) return a->l[i] > b->l[i];
  }
  return 1;
}

static uint64_t fq_raw_sub(fq* d, const fq* a, const fq* b) {
  uint64_t borrow = 0;
  for (int i = 0; i < 4; i++) {
    u128 t = (u128)a->l[i] - b->l[i] - borrow;
    d->l[i] = (uint64_t)t;
    borrow = (uint64_t)(t >> 64) & 1;
  }
  return borrow;
}

static uint64_t fq_raw_add(fq* s, const fq* a, const fq* b) {
  uint64_t carry = 0;
  for (int i = 0; i < 4; i++) {
    u128 t = (u128)a->l[i] + b->l[i] + carry;
    s->l[i] = (uint64_t)t;
    carry = (uint64_t)(t >> 64);
  }
  return carry;
}

/* operands and results in [0, q) */
static fq fq_add(fq a, fq b) {
  fq s;
  uint64_t c = fq_raw_add(&s, &a, &b);
  if (c || fq_geq(&s, &Q)) fq_raw_sub(&s, &s, &Q);
  return s;
}

static fq fq_sub(fq a, fq b) {
  fq d;
  if (fq_raw_sub(&d, &a, &b)) fq_raw_add(&d, &d, &Q);
  return d;
}

/* a * b / 2^256 mod q, CIOS over 64-bit words */
static fq fq_mul(fq a, fq b) {
  uint64_t t[6] = {0, 0, 0, 0, 0, 0};
  for (int i = 0; i < 4; i++) {
    uint64_t c = 0;
    for (int j = 0; j < 4; j++) {
      u128 s = (u128)a.l[j] * b.l[i] + t[j] + c;
      t[j] = (uint64_t)s;
      c = (uint64_t)(s >> 64);
    }
    u128 s = (u128)t[4] + c;
    t[4] = (uint64_t)s;
    t[5] = (uint64_t)(s >> 64);
    uint64_t m = t[0] * QINV;
    s = (u128)m * Q.l[0] + t[0];
    c = (uint64_t)(s >> 64);
    for (int j = 1; j < 4; j++) {
      s = (u128)m * Q.l[j] + t[j] + c;
      t[j - 1] = (uint64_t)s;
      c = (uint64_t)(s >> 64);
    }
    s = (u128)t[4] + c;
    t[3] = (uint64_t)s;
    t[4] = t[5] + (uint64_t)(s >> 64);
  }
  fq r = {{t[0], t[1], t[2], t[3]}};
  if (t[4] || fq_geq(&r, &Q)) fq_raw_sub(&r, &r, &Q);
  return r;
}

static int fq_is_zero(fq a) { return (a.l[0] | a.l[1] | a.l[2] | a.l[3]) == 0; }
static int fq_eq(fq a, fq b) { return memcmp(&a, &b, sizeof(fq)) == 0; }

static void init(void) {
  if (ready) return;
  /* Newton iteration for q^-1 mod 2^64 (q odd): x <- x (2 - q x) doubles the bits */
  uint64_t x = 1;
  for (int i = 0; i < 7; i++) x *= 2 - Q.l[0] * x;
  QINV = (uint64_t)0 - x;
  /* 2^256 mod q and 2^512 mod q by repeated doubling of 1 */
  fq v = {{1, 0, 0, 0}};
  for (int i = 0; i < 512; i++) {
    v = fq_add(v, v);
    if (i == 255) ONE = v;
  }
  R2Q = v;
  ready = 1;
}

/* a^e mod q in Montgomery form, e given as four 64-bit limbs, square-and-multiply */
static fq fq_pow(fq a, const uint64_t* e) {
  fq acc = ONE;
  for (int i = 255; i >= 0; i--) {
    acc = fq_mul(acc, acc);
    if ((e[i / 64] >> (i % 64)) & 1) acc = fq_mul(acc, a);
  }
  return acc;
}

/* a^-1 = a^(q-2) (Fermat); 0 maps to 0 */
static fq fq_inv(fq a) {
  uint64_t e[4] = {Q.l[0] - 2, Q.l[1], Q.l[2], Q.l[3]};
  return fq_pow(a, e);
}

static fq load_fq(const uint32_t* p) {
  fq a;
  for (int i = 0; i < 4; i++) a.l[i] = (uint64_t)p[2 * i] | ((uint64_t)p[2 * i + 1] << 32);
  return a;
}

static void store_fq(uint32_t* p, fq a) {
  for (int i = 0; i < 4; i++) {
    p[2 * i] = (uint32_t)a.l[i];
    p[2 * i + 1] = (uint32_t)(a.l[i] >> 32);
  }
}

/* ------------------------------------------------------------------ the curve ---- */

typedef struct {
  fq X, Y, Z; /* Z = 0: the point at infinity */
} jac;

static jac jac_infinity(void) {
  jac r;
  memset(&r, 0, sizeof r);
  r.X = ONE;
  r.Y = ONE;
  return r;
}

static fq small(uint64_t k) { /* Montgomery form of a small integer */
  fq a = {{k, 0, 0, 0}};
  fq r2 = R2Q;
  return fq_mul(a, r2);
}

/* 2P. The tangent slope at (x, y) is 3x^2 / 2y; with x = X/Z^2, y = Y/Z^3:
 *   M = 3 X^2, S = 4 X Y^2,  X3 = M^2 - 2S,  Y3 = M (S - X3) - 8 Y^4,  Z3 = 2 Y Z. */
static jac jac_double(jac P) {
  if (fq_is_zero(P.Z) || fq_is_zero(P.Y)) return jac_infinity();
  fq XX = fq_mul(P.X, P.X);
  fq YY = fq_mul(P.Y, P.Y);
  fq M = fq_add(fq_add(XX, XX), XX);
  fq XYY = fq_mul(P.X, YY);
  fq S = fq_add(XYY, XYY);
  S = fq_add(S, S);
  fq Y4 = fq_mul(YY, YY);
  fq Y4x8 = fq_add(Y4, Y4);
  Y4x8 = fq_add(Y4x8, Y4x8);
  Y4x8 = fq_add(Y4x8, Y4x8);
  fq YZ = fq_mul(P.Y, P.Z);
  jac R;
  R.X = fq_sub(fq_mul(M, M), fq_add(S, S));
  R.Y = fq_sub(fq_mul(M, fq_sub(S, R.X)), Y4x8);
  R.Z = fq_add(YZ, YZ);
  return R;
}

/* P + Q. The chord through the two points, with U1 = X1 Z2^2, U2 = X2 Z1^2 (the x
 * coordinates over a common denominator) and S1 = Y1 Z2^3, S2 = Y2 Z1^3:
 *   H = U2 - U1, r = S2 - S1,  X3 = r^2 - H^3 - 2 U1 H^2,
 *   Y3 = r (U1 H^2 - X3) - S1 H^3,  Z3 = H Z1 Z2.
 * H = 0 means equal x: the same point (double it) or opposite points (infinity). */
static jac jac_add(jac P, jac Qp) {
  if (fq_is_zero(P.Z)) return Qp;
  if (fq_is_zero(Qp.Z)) return P;
  fq Z1Z1 = fq_mul(P.Z, P.Z), Z2Z2 = fq_mul(Qp.Z, Qp.Z);
  fq U1 = fq_mul(P.X, Z2Z2), U2 = fq_mul(Qp.X, Z1Z1);
  fq S1 = fq_mul(P.Y, fq_mul(Qp.Z, Z2Z2)), S2 = fq_mul(Qp.Y, fq_mul(P.Z, Z1Z1));
  if (fq_eq(U1, U2)) {
    if (fq_eq(S1, S2)) return jac_double(P);
    return jac_infinity();
  }
  fq H = fq_sub(U2, U1), r = fq_sub(S2, S1);
  fq HH = fq_mul(H, H), HHH = fq_mul(H, HH);
  fq V = fq_mul(U1, HH);
  jac R;
  R.X = fq_sub(fq_sub(fq_mul(r, r), HHH), fq_add(V, V));
  R.Y = fq_sub(fq_mul(r, fq_sub(V, R.X)), fq_mul(S1, HHH));
  R.Z = fq_mul(H, fq_mul(P.Z, Qp.Z));
  return R;
}

/* k P by left-to-right double-and-add over the 256 bits of k (eight 32-bit limbs) */
static jac jac_mul(jac P, const uint32_t* k) {
  jac acc = jac_infinity();
  for (int i = 255; i >= 0; i--) {
    acc = jac_double(acc);
    if ((k[i / 32] >> (i % 32)) & 1) acc = jac_add(acc, P);
  }
  return acc;
}

static jac load_affine(const uint32_t* p) {
  jac P;
  P.X = load_fq(p);
  P.Y = load_fq(p + 8);
  if (fq_is_zero(P.X) && fq_is_zero(P.Y)) return jac_infinity();
  P.Z = ONE;
  return P;
}

/* writes x, y (Montgomery) of P; infinity as zeros. Returns 1 for infinity. */
static int store_affine(uint32_t* out, jac P) {
  if (fq_is_zero(P.Z)) {
    memset(out, 0, 16 * sizeof(uint32_t));
    return 1;
  }
  fq zi = fq_inv(P.Z);
  fq zi2 = fq_mul(zi, zi);
  store_fq(out, fq_mul(P.X, zi2));
  store_fq(out + 8, fq_mul(P.Y, fq_mul(zi2, zi)));
  return 0;
}

/* ------------------------------------------------------------------ interface ---- */

void orc_fq_mul(const uint32_t* a, const uint32_t* b, uint32_t* out) {
  init();
  store_fq(out, fq_mul(load_fq(a), load_fq(b)));
}

void orc_fq_inv(const uint32_t* a, uint32_t* out) {
  init();
  store_fq(out, fq_inv(load_fq(a)));
}

/* 1 when the affine point (x, y) satisfies y^2 = x^3 + 3 with both coordinates < q, or is
 * the point at infinity (0, 0); 0 otherwise */
int orc_g1_on_curve(const uint32_t* p) {
  init();
  fq x = load_fq(p), y = load_fq(p + 8);
  if (fq_is_zero(x) && fq_is_zero(y)) return 1;
  if (fq_geq(&x, &Q) || fq_geq(&y, &Q)) return 0;
  fq lhs = fq_mul(y, y);
  fq rhs = fq_add(fq_mul(fq_mul(x, x), x), small(3));
  return fq_eq(lhs, rhs);
}

int orc_g1_add(const uint32_t* p, const uint32_t* q, uint32_t* out) {
  init();
  return store_affine(out, jac_add(load_affine(p), load_affine(q)));
}

int orc_g1_mul(const uint32_t* p, const uint32_t* k, uint32_t* out) {
  init();
  return store_affine(out, jac_mul(load_affine(p), k));
}

/* sum_i scalars[i] * bases[i] over i < n; result affine (Montgomery), returns 1 for
 * infinity */
int orc_g1_msm(size_t n, const uint32_t* bases, const uint32_t* scalars, uint32_t* out) {
  init();
  jac acc = jac_infinity();
  for (size_t i = 0; i < n; i++) acc = jac_add(acc, jac_mul(load_affine(bases + 16 * i), scalars + 8 * i));
  return store_affine(out, acc);
}

/* the affine point of Jacobian (X, Y, Z) (24 limbs, Montgomery); returns 1 for infinity */
int orc_g1_jacobian_to_affine(const uint32_t* p, uint32_t* out) {
  init();
  jac P;
  P.X = load_fq(p);
  P.Y = load_fq(p + 8);
  P.Z = load_fq(p + 16);
  return store_affine(out, P);
}

/* ================================================================= G2 over F_q2 ====
 *
 * The same definition over the twist E': y^2 = x^3 + b2 over F_q2 = F_q[u]/(u^2 + 1),
 * b2 = 3 / (9 + u) (EIP-197), the witness multiexp of the B query (MSM_CU stage 7). The
 * point formulas are the Jacobian ones above with F_q2 arithmetic; an affine point is
 * x.c0, x.c1, y.c0, y.c1 (32 limbs), a Jacobian one X, Y, Z (48 limbs), each coordinate
 * c0 + c1 u in Montgomery form over F_q. */

typedef struct {
  fq c0, c1;
} fq2;

static fq2 f2_add(fq2 a, fq2 b) { fq2 r = {fq_add(a.c0, b.c0), fq_add(a.c1, b.c1)}; return r; }
static fq2 f2_sub(fq2 a, fq2 b) { fq2 r = {fq_sub(a.c0, b.c0), fq_sub(a.c1, b.c1)}; return r; }

/* (a0 + a1 u)(b0 + b1 u) = (a0 b0 - a1 b1) + (a0 b1 + a1 b0) u, by the schoolbook formula */
static fq2 f2_mul(fq2 a, fq2 b) {
  fq2 r;
  r.c0 = fq_sub(fq_mul(a.c0, b.c0), fq_mul(a.c1, b.c1));
  r.c1 = fq_add(fq_mul(a.c0, b.c1), fq_mul(a.c1, b.c0));
  return r;
}

static int f2_is_zero(fq2 a) { return fq_is_zero(a.c0) && fq_is_zero(a.c1); }
static int f2_eq(fq2 a, fq2 b) { return fq_eq(a.c0, b.c0) && fq_eq(a.c1, b.c1); }

/* 1 / (a0 + a1 u) = (a0 - a1 u) / (a0^2 + a1^2) */
static fq2 f2_inv(fq2 a) {
  fq n = fq_inv(fq_add(fq_mul(a.c0, a.c0), fq_mul(a.c1, a.c1)));
  fq zero = {{0, 0, 0, 0}};
  fq2 r = {fq_mul(a.c0, n), fq_mul(fq_sub(zero, a.c1), n)};
  return r;
}

static fq2 load_fq2(const uint32_t* p) { fq2 a = {load_fq(p), load_fq(p + 8)}; return a; }
static void store_fq2(uint32_t* p, fq2 a) { store_fq(p, a.c0); store_fq(p + 8, a.c1); }

static fq2 twist_b(void) {
  fq2 three = {small(3), {{0, 0, 0, 0}}};
  fq2 nine_u = {small(9), ONE};
  return f2_mul(three, f2_inv(nine_u));
}

typedef struct {
  fq2 X, Y, Z; /* Z = 0: the point at infinity */
} jac2;

static jac2 jac2_infinity(void) {
  jac2 r;
  memset(&r, 0, sizeof r);
  r.X.c0 = ONE;
  r.Y.c0 = ONE;
  return r;
}

/* the tangent formula of jac_double, over F_q2 */
static jac2 jac2_double(jac2 P) {
  if (f2_is_zero(P.Z) || f2_is_zero(P.Y)) return jac2_infinity();
  fq2 XX = f2_mul(P.X, P.X), YY = f2_mul(P.Y, P.Y);
  fq2 M = f2_add(f2_add(XX, XX), XX);
  fq2 XYY = f2_mul(P.X, YY);
  fq2 S = f2_add(XYY, XYY);
  S = f2_add(S, S);
  fq2 Y4 = f2_mul(YY, YY);
  fq2 Y4x8 = f2_add(Y4, Y4);
  Y4x8 = f2_add(Y4x8, Y4x8);
  Y4x8 = f2_add(Y4x8, Y4x8);
  fq2 YZ = f2_mul(P.Y, P.Z);
  jac2 R;
  R.X = f2_sub(f2_mul(M, M), f2_add(S, S));
  R.Y = f2_sub(f2_mul(M, f2_sub(S, R.X)), Y4x8);
  R.Z = f2_add(YZ, YZ);
  return R;
}

/* the chord formula of jac_add, over F_q2 */
static jac2 jac2_add(jac2 P, jac2 Qp) {
  if (f2_is_zero(P.Z)) return Qp;
  if (f2_is_zero(Qp.Z)) return P;
  fq2 Z1Z1 = f2_mul(P.Z, P.Z), Z2Z2 = f2_mul(Qp.Z, Qp.Z);
  fq2 U1 = f2_mul(P.X, Z2Z2), U2 = f2_mul(Qp.X, Z1Z1);
  fq2 S1 = f2_mul(P.Y, f2_mul(Qp.Z, Z2Z2)), S2 = f2_mul(Qp.Y, f2_mul(P.Z, Z1Z1));
  if (f2_eq(U1, U2)) {
    if (f2_eq(S1, S2)) return jac2_double(P);
    return jac2_infinity();
  }
  fq2 H = f2_sub(U2, U1), r = f2_sub(S2, S1);
  fq2 HH = f2_mul(H, H), HHH = f2_mul(H, HH);
  fq2 V = f2_mul(U1, HH);
  jac2 R;
  R.X = f2_sub(f2_sub(f2_mul(r, r), HHH), f2_add(V, V));
  R.Y = f2_sub(f2_mul(r, f2_sub(V, R.X)), f2_mul(S1, HHH));
  R.Z = f2_mul(H, f2_mul(P.Z, Qp.Z));
  return R;
}

static jac2 jac2_mul(jac2 P, const uint32_t* k) {
  jac2 acc = jac2_infinity();
  for (int i = 255; i >= 0; i--) {
    acc = jac2_double(acc);
    if ((k[i / 32] >> (i % 32)) & 1) acc = jac2_add(acc, P);
  }
  return acc;
}

static jac2 load_affine2(const uint32_t* p) {
  jac2 P;
  P.X = load_fq2(p);
  P.Y = load_fq2(p + 16);
  if (f2_is_zero(P.X) && f2_is_zero(P.Y)) return jac2_infinity();
  memset(&P.Z, 0, sizeof P.Z);
  P.Z.c0 = ONE;
  return P;
}

static int store_affine2(uint32_t* out, jac2 P) {
  if (f2_is_zero(P.Z)) {
    memset(out, 0, 32 * sizeof(uint32_t));
    return 1;
  }
  fq2 zi = f2_inv(P.Z);
  fq2 zi2 = f2_mul(zi, zi);
  store_fq2(out, f2_mul(P.X, zi2));
  store_fq2(out + 16, f2_mul(P.Y, f2_mul(zi2, zi)));
  return 0;
}

int orc_g2_on_curve(const uint32_t* p) {
  init();
  fq2 x = load_fq2(p), y = load_fq2(p + 16);
  if (f2_is_zero(x) && f2_is_zero(y)) return 1;
  if (fq_geq(&x.c0, &Q) || fq_geq(&x.c1, &Q) || fq_geq(&y.c0, &Q) || fq_geq(&y.c1, &Q))
    return 0;
  return f2_eq(f2_mul(y, y), f2_add(f2_mul(f2_mul(x, x), x), twist_b()));
}

int orc_g2_add(const uint32_t* p, const uint32_t* q, uint32_t* out) {
  init();
  return store_affine2(out, jac2_add(load_affine2(p), load_affine2(q)));
}

int orc_g2_mul(const uint32_t* p, const uint32_t* k, uint32_t* out) {
  init();
  return store_affine2(out, jac2_mul(load_affine2(p), k));
}

int orc_g2_msm(size_t n, const uint32_t* bases, const uint32_t* scalars, uint32_t* out) {
  init();
  jac2 acc = jac2_infinity();
  for (size_t i = 0; i < n; i++)
    acc = jac2_add(acc, jac2_mul(load_affine2(bases + 32 * i), scalars + 8 * i));
  return store_affine2(out, acc);
}

int orc_g2_jacobian_to_affine(const uint32_t* p, uint32_t* out) {
  init();
  jac2 P;
  P.X = load_fq2(p);
  P.Y = load_fq2(p + 16);
  P.Z = load_fq2(p + 32);
  return store_affine2(out, P);
}
