// BN254 scalar field Fr on sm_103a: 8 x 32-bit little-endian limbs, Montgomery form
// with R = 2^256.
//
// The field is the one the "snarkrs_gpu_kernels" pages compute in (POINTWISE_CU, "two
// output buffers": Montgomery limbs vs the integer in [0, r)); its modulus is
//   r = 0x30644e72e131a029b85045b68181585d2833e84879b9709143e1f593f0000001.
// The arithmetic here is written from the mathematics, not from any header the pages
// mention: Montgomery multiplication in coarsely integrated operand scanning (CIOS) form
// (Koc, Acar & Kaliski, "Analyzing and Comparing Montgomery Multiplication Algorithms",
// IEEE Micro 1996) on 32-bit words, and additions and subtractions as PTX add-with-carry
// chains.
//
// Lazy reduction. 4r < 2^256, so every intermediate value is kept in [0, 2r):
//   * fr_mul with both inputs in [0, 2r) returns a value in [0, 2r) without the final
//     conditional subtraction, because (a*b + m*r) / R < (4r^2 + R*r) / R < 2r;
//   * fr_add / fr_sub fold their result back into [0, 2r) with one conditional 2r;
//   * fr_canon maps [0, 2r) to the canonical [0, r). Every value that leaves the library
//     goes through it.
#pragma once
#include <stdint.h>

namespace g3h {

struct __align__(16) fr_t {
  uint32_t v[8];
};

// r, 2r and -r^{-1} mod 2^32.
#define G3H_R0 0xf0000001u
#define G3H_R1 0x43e1f593u
#define G3H_R2 0x79b97091u
#define G3H_R3 0x2833e848u
#define G3H_R4 0x8181585du
#define G3H_R5 0xb85045b6u
#define G3H_R6 0xe131a029u
#define G3H_R7 0x30644e72u

#define G3H_2R0 0xe0000002u
#define G3H_2R1 0x87c3eb27u
#define G3H_2R2 0xf372e122u
#define G3H_2R3 0x5067d090u
#define G3H_2R4 0x0302b0bau
#define G3H_2R5 0x70a08b6du
#define G3H_2R6 0xc2634053u
#define G3H_2R7 0x60c89ce5u

#define G3H_NPRIME 0xefffffffu

__device__ __forceinline__ fr_t fr_zero() {
  fr_t z;
#pragma unroll
  for (int i = 0; i < 8; i++) z.v[i] = 0u;
  return z;
}

// One CIOS row on words t0..t7 (t < 3r < 2^256 on entry): t <- (t + a*bi + m*r) / 2^32,
// m = (t + a*bi) * (-r^{-1}) mod 2^32. The products of a*bi are added as two carry
// chains, one over the even limbs a0, a2, a4, a6 (whose low and high words land on word
// pairs (0,1), (2,3), (4,5), (6,7)) and one over the odd limbs (pairs (1,2) ... (7,8)),
// so that the low and high word of each product are adjacent in one chain; m*r likewise,
// and its odd chain writes each word one position down, which is the division by 2^32.
// The sum before the division is below 3r + 2*2^32*2r < 2^288, so nothing carries out of
// the ninth word t8.
#define G3H_CIOS_ROW(t0, t1, t2, t3, t4, t5, t6, t7, bi)                                   \
  asm("{\n\t"                                                                             \
      ".reg .u32 m, t8;\n\t"                                                              \
      "mad.lo.cc.u32  %0, %8,  %16, %0;\n\t"                                              \
      "madc.hi.cc.u32 %1, %8,  %16, %1;\n\t"                                              \
      "madc.lo.cc.u32 %2, %10, %16, %2;\n\t"                                              \
      "madc.hi.cc.u32 %3, %10, %16, %3;\n\t"                                              \
      "madc.lo.cc.u32 %4, %12, %16, %4;\n\t"                                              \
      "madc.hi.cc.u32 %5, %12, %16, %5;\n\t"                                              \
      "madc.lo.cc.u32 %6, %14, %16, %6;\n\t"                                              \
      "madc.hi.cc.u32 %7, %14, %16, %7;\n\t"                                              \
      "addc.u32       t8, 0, 0;\n\t"                                                      \
      "mad.lo.cc.u32  %1, %9,  %16, %1;\n\t"                                              \
      "madc.hi.cc.u32 %2, %9,  %16, %2;\n\t"                                              \
      "madc.lo.cc.u32 %3, %11, %16, %3;\n\t"                                              \
      "madc.hi.cc.u32 %4, %11, %16, %4;\n\t"                                              \
      "madc.lo.cc.u32 %5, %13, %16, %5;\n\t"                                              \
      "madc.hi.cc.u32 %6, %13, %16, %6;\n\t"                                              \
      "madc.lo.cc.u32 %7, %15, %16, %7;\n\t"                                              \
      "madc.hi.u32    t8, %15, %16, t8;\n\t"                                              \
      "mul.lo.u32     m,  %0, 0xefffffff;\n\t"                                            \
      "mad.lo.cc.u32  %0, m, 0xf0000001, %0;\n\t"                                         \
      "madc.hi.cc.u32 %1, m, 0xf0000001, %1;\n\t"                                         \
      "madc.lo.cc.u32 %2, m, 0x79b97091, %2;\n\t"                                         \
      "madc.hi.cc.u32 %3, m, 0x79b97091, %3;\n\t"                                         \
      "madc.lo.cc.u32 %4, m, 0x8181585d, %4;\n\t"                                         \
      "madc.hi.cc.u32 %5, m, 0x8181585d, %5;\n\t"                                         \
      "madc.lo.cc.u32 %6, m, 0xe131a029, %6;\n\t"                                         \
      "madc.hi.cc.u32 %7, m, 0xe131a029, %7;\n\t"                                         \
      "addc.u32       t8, t8, 0;\n\t"                                                     \
      "mad.lo.cc.u32  %0, m, 0x43e1f593, %1;\n\t"                                         \
      "madc.hi.cc.u32 %1, m, 0x43e1f593, %2;\n\t"                                         \
      "madc.lo.cc.u32 %2, m, 0x2833e848, %3;\n\t"                                         \
      "madc.hi.cc.u32 %3, m, 0x2833e848, %4;\n\t"                                         \
      "madc.lo.cc.u32 %4, m, 0xb85045b6, %5;\n\t"                                         \
      "madc.hi.cc.u32 %5, m, 0xb85045b6, %6;\n\t"                                         \
      "madc.lo.cc.u32 %6, m, 0x30644e72, %7;\n\t"                                         \
      "madc.hi.u32    %7, m, 0x30644e72, t8;\n\t"                                         \
      "}"                                                                                 \
      : "+r"(t0), "+r"(t1), "+r"(t2), "+r"(t3), "+r"(t4), "+r"(t5), "+r"(t6), "+r"(t7)   \
      : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]),    \
        "r"(a.v[6]), "r"(a.v[7]), "r"(bi))

// a * b * 2^-256 mod r, inputs in [0, 2r), output in [0, 2r) (CIOS: one row per word of
// b; written with even/odd carry chains so that the low and high word of each product
// sit in one chain and the compiler can issue the product once. Measured on GB300: a full
// 32 x 32 -> 64-bit product costs about 2.7 of the 32-bit multiply-adds' issue slots on
// the integer multiply pipe (mad.wide.u32 23.7 and mad.lo.u32 63.8 per clock per SM).
__device__ __forceinline__ fr_t fr_mul(const fr_t& a, const fr_t& b) {
  uint32_t t0 = 0, t1 = 0, t2 = 0, t3 = 0, t4 = 0, t5 = 0, t6 = 0, t7 = 0;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    G3H_CIOS_ROW(t0, t1, t2, t3, t4, t5, t6, t7, b.v[i]);
  }
  fr_t c;
  c.v[0] = t0; c.v[1] = t1; c.v[2] = t2; c.v[3] = t3;
  c.v[4] = t4; c.v[5] = t5; c.v[6] = t6; c.v[7] = t7;
  return c;
}

// ---------------------------------------------------------------------------------------
// Multiplication by a constant (twiddles, shift, scale): Shoup's method (V. Shoup, NTL;
// D. Harvey, "Faster arithmetic for number-theoretic transforms", J. Symb. Comp. 2014)
// with beta = 2^256. For a constant w < r store w and w' = floor(w * beta / r), i.e.
// w * beta = w' * r + e with 0 <= e < r. For x < beta let P = x * w' = Q * beta + rho
// (0 <= rho < beta); then x * w = Q * r + (rho * r + x * e) / beta, so y = x*w - Q*r lies
// in [0, 2r). Here the quotient is computed from the columns i + j >= 6 of the limb
// product x * w' only; the dropped columns sum to D < 6.01 * 2^224 < 2^227, so the
// quotient q is Q or, when rho < D (the dropped columns would have carried into bit 256),
// Q - 1. In that case y = (rho * r + x * e) / beta + r, which is below 2r because
// rho * r + x * e < D * r + x * r <= beta * r whenever x <= beta - D. Every operand the
// library multiplies is a value in [0, 2r) (2r < beta - 2^227), so y = x*w - q*r lies in
// [0, 2r) and is exact mod 2^256: no correction step is needed. With x in Montgomery form
// (x = X*R) and w in standard form the product is the Montgomery form of X*w, so data
// never leaves the Montgomery domain. Cost: 43 + 2 * 28 full and 16 low-only 32x32
// products, against 128 full and 8 low-only for a Montgomery multiply.
struct __align__(16) fr_const_t {
  fr_t w;   // the constant, standard form, < r
  fr_t wp;  // floor(w * 2^256 / r)
};

// One product of a column sum (c0, c1, c2) += a*b.
#define G3H_MAC(c0, c1, c2, a, b)                                                          \
  asm("mad.lo.cc.u32  %0, %3, %4, %0;\n\t"                                                 \
      "madc.hi.cc.u32 %1, %3, %4, %1;\n\t"                                                 \
      "addc.u32       %2, %2, 0;"                                                          \
      : "+r"(c0), "+r"(c1), "+r"(c2)                                                       \
      : "r"(a), "r"(b))

// lo = (a * b) mod 2^256, by columns.
__device__ __forceinline__ void mul_low256(const uint32_t* a, const uint32_t* b, uint32_t* lo) {
  uint32_t c0 = 0, c1 = 0, c2 = 0;
#pragma unroll
  for (int k = 0; k < 7; k++) {
#pragma unroll
    for (int i = 0; i <= k; i++) G3H_MAC(c0, c1, c2, a[i], b[k - i]);
    lo[k] = c0;
    c0 = c1;
    c1 = c2;
    c2 = 0;
  }
#pragma unroll
  for (int i = 0; i <= 7; i++) c0 += a[i] * b[7 - i];
  lo[7] = c0;
}

// q = words 8..15 of the sum over i + j >= 6 of a_i * b_j * 2^(32(i+j)).
__device__ __forceinline__ void mul_high256_from6(const uint32_t* a, const uint32_t* b,
                                                  uint32_t* q) {
  uint32_t c0 = 0, c1 = 0, c2 = 0;
#pragma unroll
  for (int k = 6; k <= 14; k++) {
#pragma unroll
    for (int i = (k > 7 ? k - 7 : 0); i <= (k < 7 ? k : 7); i++) G3H_MAC(c0, c1, c2, a[i], b[k - i]);
    if (k >= 8) q[k - 8] = c0;
    c0 = c1;
    c1 = c2;
    c2 = 0;
  }
  q[7] = c0;
}

// x * w mod r in [0, 2r) for x < 2^256 - 2^227 (in the library: x < 2r) and a constant
// given as (w, w'). The bound on x is what makes the truncated quotient safe (above).
__device__ __forceinline__ fr_t fr_mul_const(const fr_t& x, const fr_t& w, const fr_t& wp) {
  const uint32_t R[8] = {G3H_R0, G3H_R1, G3H_R2, G3H_R3, G3H_R4, G3H_R5, G3H_R6, G3H_R7};
  uint32_t q[8], lxw[8], lqr[8];
  mul_high256_from6(x.v, wp.v, q);
  mul_low256(x.v, w.v, lxw);
  mul_low256(q, R, lqr);
  fr_t y;
  asm("sub.cc.u32  %0, %8,  %16;\n\t"
      "subc.cc.u32 %1, %9,  %17;\n\t"
      "subc.cc.u32 %2, %10, %18;\n\t"
      "subc.cc.u32 %3, %11, %19;\n\t"
      "subc.cc.u32 %4, %12, %20;\n\t"
      "subc.cc.u32 %5, %13, %21;\n\t"
      "subc.cc.u32 %6, %14, %22;\n\t"
      "subc.u32    %7, %15, %23;"
      : "=r"(y.v[0]), "=r"(y.v[1]), "=r"(y.v[2]), "=r"(y.v[3]), "=r"(y.v[4]), "=r"(y.v[5]),
        "=r"(y.v[6]), "=r"(y.v[7])
      : "r"(lxw[0]), "r"(lxw[1]), "r"(lxw[2]), "r"(lxw[3]), "r"(lxw[4]), "r"(lxw[5]),
        "r"(lxw[6]), "r"(lxw[7]), "r"(lqr[0]), "r"(lqr[1]), "r"(lqr[2]), "r"(lqr[3]),
        "r"(lqr[4]), "r"(lqr[5]), "r"(lqr[6]), "r"(lqr[7]));
  return y;
}

// -r^{-1} mod 2^256: w' = (w * 2^256 mod r) * (-r^{-1}) mod 2^256 for w < r, because
// w * 2^256 = w' * r + (w * 2^256 mod r) and w' < 2^256.
#define G3H_NINV256 {0xefffffffu, 0xc2e1f593u, 0x4c6911b3u, 0x6586864bu, \
                     0x99062391u, 0xe39a9828u, 0x0d8341b2u, 0x73f82f1du}

// a + b, inputs in [0, 2r), output in [0, 2r): the sum is below 4r < 2^256, and 2r is
// subtracted when the subtraction does not borrow.
__device__ __forceinline__ fr_t fr_add(const fr_t& a, const fr_t& b) {
  fr_t s, d;
  uint32_t borrow;
  asm("add.cc.u32  %0, %8,  %16;\n\t"
      "addc.cc.u32 %1, %9,  %17;\n\t"
      "addc.cc.u32 %2, %10, %18;\n\t"
      "addc.cc.u32 %3, %11, %19;\n\t"
      "addc.cc.u32 %4, %12, %20;\n\t"
      "addc.cc.u32 %5, %13, %21;\n\t"
      "addc.cc.u32 %6, %14, %22;\n\t"
      "addc.u32    %7, %15, %23;"
      : "=r"(s.v[0]), "=r"(s.v[1]), "=r"(s.v[2]), "=r"(s.v[3]), "=r"(s.v[4]), "=r"(s.v[5]),
        "=r"(s.v[6]), "=r"(s.v[7])
      : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]),
        "r"(a.v[6]), "r"(a.v[7]), "r"(b.v[0]), "r"(b.v[1]), "r"(b.v[2]), "r"(b.v[3]),
        "r"(b.v[4]), "r"(b.v[5]), "r"(b.v[6]), "r"(b.v[7]));
  asm("sub.cc.u32  %0, %9,  0xe0000002;\n\t"
      "subc.cc.u32 %1, %10, 0x87c3eb27;\n\t"
      "subc.cc.u32 %2, %11, 0xf372e122;\n\t"
      "subc.cc.u32 %3, %12, 0x5067d090;\n\t"
      "subc.cc.u32 %4, %13, 0x0302b0ba;\n\t"
      "subc.cc.u32 %5, %14, 0x70a08b6d;\n\t"
      "subc.cc.u32 %6, %15, 0xc2634053;\n\t"
      "subc.cc.u32 %7, %16, 0x60c89ce5;\n\t"
      "subc.u32    %8, 0, 0;"
      : "=r"(d.v[0]), "=r"(d.v[1]), "=r"(d.v[2]), "=r"(d.v[3]), "=r"(d.v[4]), "=r"(d.v[5]),
        "=r"(d.v[6]), "=r"(d.v[7]), "=r"(borrow)
      : "r"(s.v[0]), "r"(s.v[1]), "r"(s.v[2]), "r"(s.v[3]), "r"(s.v[4]), "r"(s.v[5]),
        "r"(s.v[6]), "r"(s.v[7]));
  // borrow is 0xffffffff when s < 2r, 0 otherwise.
#pragma unroll
  for (int i = 0; i < 8; i++) d.v[i] = borrow ? s.v[i] : d.v[i];
  return d;
}

// a - b, inputs in [0, 2r), output in [0, 2r): 2r is added back when the difference
// borrows.
__device__ __forceinline__ fr_t fr_sub(const fr_t& a, const fr_t& b) {
  fr_t d;
  uint32_t borrow;
  asm("sub.cc.u32  %0, %9,  %17;\n\t"
      "subc.cc.u32 %1, %10, %18;\n\t"
      "subc.cc.u32 %2, %11, %19;\n\t"
      "subc.cc.u32 %3, %12, %20;\n\t"
      "subc.cc.u32 %4, %13, %21;\n\t"
      "subc.cc.u32 %5, %14, %22;\n\t"
      "subc.cc.u32 %6, %15, %23;\n\t"
      "subc.cc.u32 %7, %16, %24;\n\t"
      "subc.u32    %8, 0, 0;"
      : "=r"(d.v[0]), "=r"(d.v[1]), "=r"(d.v[2]), "=r"(d.v[3]), "=r"(d.v[4]), "=r"(d.v[5]),
        "=r"(d.v[6]), "=r"(d.v[7]), "=r"(borrow)
      : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]),
        "r"(a.v[6]), "r"(a.v[7]), "r"(b.v[0]), "r"(b.v[1]), "r"(b.v[2]), "r"(b.v[3]),
        "r"(b.v[4]), "r"(b.v[5]), "r"(b.v[6]), "r"(b.v[7]));
  asm("add.cc.u32  %0, %0, %8;\n\t"
      "addc.cc.u32 %1, %1, %9;\n\t"
      "addc.cc.u32 %2, %2, %10;\n\t"
      "addc.cc.u32 %3, %3, %11;\n\t"
      "addc.cc.u32 %4, %4, %12;\n\t"
      "addc.cc.u32 %5, %5, %13;\n\t"
      "addc.cc.u32 %6, %6, %14;\n\t"
      "addc.u32    %7, %7, %15;"
      : "+r"(d.v[0]), "+r"(d.v[1]), "+r"(d.v[2]), "+r"(d.v[3]), "+r"(d.v[4]), "+r"(d.v[5]),
        "+r"(d.v[6]), "+r"(d.v[7])
      : "r"(borrow & G3H_2R0), "r"(borrow & G3H_2R1), "r"(borrow & G3H_2R2),
        "r"(borrow & G3H_2R3), "r"(borrow & G3H_2R4), "r"(borrow & G3H_2R5),
        "r"(borrow & G3H_2R6), "r"(borrow & G3H_2R7));
  return d;
}

// [0, 2r) -> [0, r).
__device__ __forceinline__ fr_t fr_canon(const fr_t& a) {
  fr_t d;
  uint32_t borrow;
  asm("sub.cc.u32  %0, %9,  0xf0000001;\n\t"
      "subc.cc.u32 %1, %10, 0x43e1f593;\n\t"
      "subc.cc.u32 %2, %11, 0x79b97091;\n\t"
      "subc.cc.u32 %3, %12, 0x2833e848;\n\t"
      "subc.cc.u32 %4, %13, 0x8181585d;\n\t"
      "subc.cc.u32 %5, %14, 0xb85045b6;\n\t"
      "subc.cc.u32 %6, %15, 0xe131a029;\n\t"
      "subc.cc.u32 %7, %16, 0x30644e72;\n\t"
      "subc.u32    %8, 0, 0;"
      : "=r"(d.v[0]), "=r"(d.v[1]), "=r"(d.v[2]), "=r"(d.v[3]), "=r"(d.v[4]), "=r"(d.v[5]),
        "=r"(d.v[6]), "=r"(d.v[7]), "=r"(borrow)
      : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]),
        "r"(a.v[6]), "r"(a.v[7]));
#pragma unroll
  for (int i = 0; i < 8; i++) d.v[i] = borrow ? a.v[i] : d.v[i];
  return d;
}

// Montgomery reduction of a canonical value: a * 2^-256 mod r, i.e. the standard-form
// integer of a Montgomery representative. For a < r the result (a + M*r) / R is below r,
// so it is canonical with no final subtraction.
__device__ __forceinline__ fr_t fr_from_mont(const fr_t& a) {
  const uint32_t R[8] = {G3H_R0, G3H_R1, G3H_R2, G3H_R3, G3H_R4, G3H_R5, G3H_R6, G3H_R7};
  uint32_t t[8];
#pragma unroll
  for (int j = 0; j < 8; j++) t[j] = a.v[j];
#pragma unroll
  for (int i = 0; i < 8; i++) {
    uint32_t m = t[0] * G3H_NPRIME;
    uint64_t s = (uint64_t)m * R[0] + t[0];
    uint64_t c = s >> 32;
#pragma unroll
    for (int j = 1; j < 8; j++) {
      s = (uint64_t)m * R[j] + t[j] + c;
      t[j - 1] = (uint32_t)s;
      c = s >> 32;
    }
    t[7] = (uint32_t)c;
  }
  fr_t r;
#pragma unroll
  for (int j = 0; j < 8; j++) r.v[j] = t[j];
  return r;
}

// True when a < r (the canonical range every input must be in).
__device__ __forceinline__ bool fr_is_canonical(const fr_t& a) {
  uint32_t borrow;
  asm("{\n\t"
      ".reg .u32 x;\n\t"
      "sub.cc.u32  x, %1, 0xf0000001;\n\t"
      "subc.cc.u32 x, %2, 0x43e1f593;\n\t"
      "subc.cc.u32 x, %3, 0x79b97091;\n\t"
      "subc.cc.u32 x, %4, 0x2833e848;\n\t"
      "subc.cc.u32 x, %5, 0x8181585d;\n\t"
      "subc.cc.u32 x, %6, 0xb85045b6;\n\t"
      "subc.cc.u32 x, %7, 0xe131a029;\n\t"
      "subc.cc.u32 x, %8, 0x30644e72;\n\t"
      "subc.u32    %0, 0, 0;\n\t"
      "}"
      : "=r"(borrow)
      : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]),
        "r"(a.v[6]), "r"(a.v[7]));
  return borrow != 0u;
}

__device__ __forceinline__ bool fr_is_zero(const fr_t& x) {
  return (x.v[0] | x.v[1] | x.v[2] | x.v[3] | x.v[4] | x.v[5] | x.v[6] | x.v[7]) == 0u;
}

// x == 2^256 mod r, the Montgomery form of 1.
__device__ __forceinline__ bool fr_is_mont_one(const fr_t& x) {
  return ((x.v[0] ^ 0x4ffffffbu) | (x.v[1] ^ 0xac96341cu) | (x.v[2] ^ 0x9f60cd29u) |
          (x.v[3] ^ 0x36fc7695u) | (x.v[4] ^ 0x7879462eu) | (x.v[5] ^ 0x666ea36fu) |
          (x.v[6] ^ 0x9a07df2fu) | (x.v[7] ^ 0x0e0a77c1u)) == 0u;
}

// 32-byte loads and stores as two 16-byte vector accesses.
__device__ __forceinline__ fr_t fr_load(const fr_t* p) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 x = q[0], y = q[1];
  fr_t a;
  a.v[0] = x.x; a.v[1] = x.y; a.v[2] = x.z; a.v[3] = x.w;
  a.v[4] = y.x; a.v[5] = y.y; a.v[6] = y.z; a.v[7] = y.w;
  return a;
}

__device__ __forceinline__ fr_t fr_ldg(const fr_t* p) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 x = __ldg(q), y = __ldg(q + 1);
  fr_t a;
  a.v[0] = x.x; a.v[1] = x.y; a.v[2] = x.z; a.v[3] = x.w;
  a.v[4] = y.x; a.v[5] = y.y; a.v[6] = y.z; a.v[7] = y.w;
  return a;
}

__device__ __forceinline__ fr_const_t fr_const_ldg(const fr_const_t* p) {
  fr_const_t c;
  c.w = fr_ldg(&p->w);
  c.wp = fr_ldg(&p->wp);
  return c;
}

__device__ __forceinline__ fr_t fr_mul_c(const fr_t& x, const fr_const_t& c) {
  return fr_mul_const(x, c.w, c.wp);
}

// Load through L2 only (not L1): for values other blocks wrote during this kernel.
__device__ __forceinline__ fr_t fr_ldcg(const fr_t* p) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  uint4 x = __ldcg(q), y = __ldcg(q + 1);
  fr_t a;
  a.v[0] = x.x; a.v[1] = x.y; a.v[2] = x.z; a.v[3] = x.w;
  a.v[4] = y.x; a.v[5] = y.y; a.v[6] = y.z; a.v[7] = y.w;
  return a;
}

__device__ __forceinline__ void fr_store(fr_t* p, const fr_t& a) {
  uint4* q = reinterpret_cast<uint4*>(p);
  q[0] = make_uint4(a.v[0], a.v[1], a.v[2], a.v[3]);
  q[1] = make_uint4(a.v[4], a.v[5], a.v[6], a.v[7]);
}

}  // namespace g3h
