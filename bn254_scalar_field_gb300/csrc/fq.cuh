// BN254 base field F_q on sm_103a: 8 x 32-bit little-endian limbs, Montgomery form with
// R = 2^256, for the G1 point arithmetic of the multi-scalar multiplication (MSM_CU:
// stage 9, the H multiexp over G1). Its modulus is
//   q = 0x30644e72e131a029b85045b68181585d97816a916871ca8d3c208c16d87cfd47
// (the alt_bn128 base field of Ethereum's EIP-196).
//
// The arithmetic is that of fr.cuh with q in place of r, written from the same
// mathematics: CIOS Montgomery multiplication (Koc, Acar & Kaliski, IEEE Micro 1996) with
// even/odd carry chains, additions as PTX add-with-carry chains, and lazy reduction:
// 4q < 2^256, so every intermediate value is kept in [0, 2q) and fq_canon maps to [0, q)
// only where a value is compared or leaves the library.
#pragma once
#include <stdint.h>

namespace g3h {

struct __align__(16) fq_t {
  uint32_t v[8];
};

#define G3H_Q0 0xd87cfd47u
#define G3H_Q1 0x3c208c16u
#define G3H_Q2 0x6871ca8du
#define G3H_Q3 0x97816a91u
#define G3H_Q4 0x8181585du
#define G3H_Q5 0xb85045b6u
#define G3H_Q6 0xe131a029u
#define G3H_Q7 0x30644e72u

// Montgomery form of 1 (2^256 mod q) and of 3 (the curve's b).
#define G3H_QONE {0xc58f0d9du, 0xd35d438du, 0xf5c70b3du, 0x0a78eb28u, \
                  0x7879462cu, 0x666ea36fu, 0x9a07df2fu, 0x0e0a77c1u}
#define G3H_QTHREE {0x50ad28d7u, 0x7a17caa9u, 0xe15521b9u, 0x1f6ac17au, \
                    0x696bd284u, 0x334bea4eu, 0xce179d8eu, 0x2a1f6744u}

__device__ __forceinline__ fq_t fq_zero() {
  fq_t z;
#pragma unroll
  for (int i = 0; i < 8; i++) z.v[i] = 0u;
  return z;
}

__device__ __forceinline__ fq_t fq_one() {
  const uint32_t o[8] = G3H_QONE;
  fq_t a;
#pragma unroll
  for (int i = 0; i < 8; i++) a.v[i] = o[i];
  return a;
}

// One CIOS row (see G3H_CIOS_ROW in fr.cuh for the layout of the two carry chains):
// t <- (t + a*bi + m*q) / 2^32 with m = (t + a*bi) * (-q^-1) mod 2^32, -q^-1 = 0xe4866389.
#define G3H_FQ_ROW(t0, t1, t2, t3, t4, t5, t6, t7, bi)                                    \
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
      "mul.lo.u32     m,  %0, 0xe4866389;\n\t"                                            \
      "mad.lo.cc.u32  %0, m, 0xd87cfd47, %0;\n\t"                                         \
      "madc.hi.cc.u32 %1, m, 0xd87cfd47, %1;\n\t"                                         \
      "madc.lo.cc.u32 %2, m, 0x6871ca8d, %2;\n\t"                                         \
      "madc.hi.cc.u32 %3, m, 0x6871ca8d, %3;\n\t"                                         \
      "madc.lo.cc.u32 %4, m, 0x8181585d, %4;\n\t"                                         \
      "madc.hi.cc.u32 %5, m, 0x8181585d, %5;\n\t"                                         \
      "madc.lo.cc.u32 %6, m, 0xe131a029, %6;\n\t"                                         \
      "madc.hi.cc.u32 %7, m, 0xe131a029, %7;\n\t"                                         \
      "addc.u32       t8, t8, 0;\n\t"                                                     \
      "mad.lo.cc.u32  %0, m, 0x3c208c16, %1;\n\t"                                         \
      "madc.hi.cc.u32 %1, m, 0x3c208c16, %2;\n\t"                                         \
      "madc.lo.cc.u32 %2, m, 0x97816a91, %3;\n\t"                                         \
      "madc.hi.cc.u32 %3, m, 0x97816a91, %4;\n\t"                                         \
      "madc.lo.cc.u32 %4, m, 0xb85045b6, %5;\n\t"                                         \
      "madc.hi.cc.u32 %5, m, 0xb85045b6, %6;\n\t"                                         \
      "madc.lo.cc.u32 %6, m, 0x30644e72, %7;\n\t"                                         \
      "madc.hi.u32    %7, m, 0x30644e72, t8;\n\t"                                         \
      "}"                                                                                 \
      : "+r"(t0), "+r"(t1), "+r"(t2), "+r"(t3), "+r"(t4), "+r"(t5), "+r"(t6), "+r"(t7)   \
      : "r"(a.v[0]), "r"(a.v[1]), "r"(a.v[2]), "r"(a.v[3]), "r"(a.v[4]), "r"(a.v[5]),    \
        "r"(a.v[6]), "r"(a.v[7]), "r"(bi))

// a * b * 2^-256 mod q, inputs in [0, 2q), output in [0, 2q).
__device__ __forceinline__ fq_t fq_mul(const fq_t& a, const fq_t& b) {
  uint32_t t0 = 0, t1 = 0, t2 = 0, t3 = 0, t4 = 0, t5 = 0, t6 = 0, t7 = 0;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    G3H_FQ_ROW(t0, t1, t2, t3, t4, t5, t6, t7, b.v[i]);
  }
  fq_t c;
  c.v[0] = t0; c.v[1] = t1; c.v[2] = t2; c.v[3] = t3;
  c.v[4] = t4; c.v[5] = t5; c.v[6] = t6; c.v[7] = t7;
  return c;
}

__device__ __forceinline__ fq_t fq_sqr(const fq_t& a) { return fq_mul(a, a); }

// x - 2q when that does not borrow, else x (x < 4q): the fold back into [0, 2q).
__device__ __forceinline__ fq_t fq_fold2q(const fq_t& s) {
  fq_t d;
  uint32_t borrow;
  asm("sub.cc.u32  %0, %9,  0xb0f9fa8e;\n\t"
      "subc.cc.u32 %1, %10, 0x7841182d;\n\t"
      "subc.cc.u32 %2, %11, 0xd0e3951a;\n\t"
      "subc.cc.u32 %3, %12, 0x2f02d522;\n\t"
      "subc.cc.u32 %4, %13, 0x0302b0bb;\n\t"
      "subc.cc.u32 %5, %14, 0x70a08b6d;\n\t"
      "subc.cc.u32 %6, %15, 0xc2634053;\n\t"
      "subc.cc.u32 %7, %16, 0x60c89ce5;\n\t"
      "subc.u32    %8, 0, 0;"
      : "=r"(d.v[0]), "=r"(d.v[1]), "=r"(d.v[2]), "=r"(d.v[3]), "=r"(d.v[4]), "=r"(d.v[5]),
        "=r"(d.v[6]), "=r"(d.v[7]), "=r"(borrow)
      : "r"(s.v[0]), "r"(s.v[1]), "r"(s.v[2]), "r"(s.v[3]), "r"(s.v[4]), "r"(s.v[5]),
        "r"(s.v[6]), "r"(s.v[7]));
#pragma unroll
  for (int i = 0; i < 8; i++) d.v[i] = borrow ? s.v[i] : d.v[i];
  return d;
}

// a + b, inputs and output in [0, 2q).
__device__ __forceinline__ fq_t fq_add(const fq_t& a, const fq_t& b) {
  fq_t s;
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
  return fq_fold2q(s);
}

__device__ __forceinline__ fq_t fq_dbl(const fq_t& a) { return fq_add(a, a); }

// a - b, inputs and output in [0, 2q): 2q is added back when the difference borrows.
__device__ __forceinline__ fq_t fq_sub(const fq_t& a, const fq_t& b) {
  fq_t d;
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
      : "r"(borrow & 0xb0f9fa8eu), "r"(borrow & 0x7841182du), "r"(borrow & 0xd0e3951au),
        "r"(borrow & 0x2f02d522u), "r"(borrow & 0x0302b0bbu), "r"(borrow & 0x70a08b6du),
        "r"(borrow & 0xc2634053u), "r"(borrow & 0x60c89ce5u));
  return d;
}

// -a for a in [0, 2q): 0 - a, folded into [0, 2q).
__device__ __forceinline__ fq_t fq_neg(const fq_t& a) { return fq_sub(fq_zero(), a); }

// [0, 2q) -> [0, q).
__device__ __forceinline__ fq_t fq_canon(const fq_t& a) {
  fq_t d;
  uint32_t borrow;
  asm("sub.cc.u32  %0, %9,  0xd87cfd47;\n\t"
      "subc.cc.u32 %1, %10, 0x3c208c16;\n\t"
      "subc.cc.u32 %2, %11, 0x6871ca8d;\n\t"
      "subc.cc.u32 %3, %12, 0x97816a91;\n\t"
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

__device__ __forceinline__ bool fq_is_zero_raw(const fq_t& a) {
  return (a.v[0] | a.v[1] | a.v[2] | a.v[3] | a.v[4] | a.v[5] | a.v[6] | a.v[7]) == 0u;
}

// a == 0 mod q, for a in [0, 2q) (0 or q).
__device__ __forceinline__ bool fq_is_zero(const fq_t& a) { return fq_is_zero_raw(fq_canon(a)); }

// a < q.
__device__ __forceinline__ bool fq_is_canonical(const fq_t& a) {
  uint32_t borrow;
  asm("{\n\t"
      ".reg .u32 x;\n\t"
      "sub.cc.u32  x, %1, 0xd87cfd47;\n\t"
      "subc.cc.u32 x, %2, 0x3c208c16;\n\t"
      "subc.cc.u32 x, %3, 0x6871ca8d;\n\t"
      "subc.cc.u32 x, %4, 0x97816a91;\n\t"
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

// a^(q-2) = a^-1 (Fermat; 0 maps to 0), by left-to-right square-and-multiply over the
// bits of q - 2. Used once per point where a point leaves projective coordinates.
__device__ __noinline__ fq_t fq_inv(const fq_t& a) {
  const uint32_t e[8] = {G3H_Q0 - 2u, G3H_Q1, G3H_Q2, G3H_Q3, G3H_Q4, G3H_Q5, G3H_Q6, G3H_Q7};
  fq_t acc = fq_one();
  for (int i = 253; i >= 0; i--) {
    acc = fq_sqr(acc);
    if ((e[i >> 5] >> (i & 31)) & 1u) acc = fq_mul(acc, a);
  }
  return acc;
}

}  // namespace g3h
