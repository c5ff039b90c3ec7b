// BN254 G1 point arithmetic for the multi-scalar multiplication (MSM_CU, "points
// accumulate in XYZZ, bases stay affine").
//
// Curve: y^2 = x^3 + 3 over F_q (fq.cuh). Bases are affine (x, y), Montgomery form, the
// point at infinity written as (0, 0) (not on the curve). Sums are kept in the extended
// Jacobian coordinates (X, Y, ZZ, ZZZ) with x = X/ZZ, y = Y/ZZZ and ZZ^3 = ZZZ^2; ZZ = 0
// is the point at infinity. The formulas are those published in the Explicit-Formulas
// Database for these coordinates (Bernstein & Lange; for a = 0): madd-2008-s (mixed
// addition, 8M + 2S), add-2008-s (12M + 2S), dbl-2008-s-1 and mdbl-2008-s-1, with the
// cases they exclude (an operand at infinity, equal x: the same point or opposite
// points) handled before them.
#pragma once
#include "fq.cuh"

namespace g3h {

struct __align__(16) g1_aff_t {
  fq_t x, y;
};

struct __align__(16) g1_xyzz_t {
  fq_t x, y, zz, zzz;
};

// Which field multiplication the point formulas use: fq_mul inlined at every call, or one
// out-of-line copy. A point addition inlines 14 multiplies (some 30 KB of code), more than
// the instruction cache keeps; where few warps run, as in the bucket sum, they stall on
// instruction fetch, and calling one compact multiply is faster.
//
// mul2 takes two independent products (x = a b, y = c d). FqPair computes them in one
// out-of-line call whose two inlined multiplies interleave, so that a lone warp waits on
// the latency of about one multiply for both.
struct FqInline {
  static __device__ __forceinline__ fq_t mul(const fq_t& a, const fq_t& b) { return fq_mul(a, b); }
  static __device__ __forceinline__ void mul2(const fq_t& a, const fq_t& b, const fq_t& c,
                                              const fq_t& d, fq_t& x, fq_t& y) {
    x = fq_mul(a, b);
    y = fq_mul(c, d);
  }
};
__device__ __noinline__ fq_t fq_mul_call(fq_t a, fq_t b) { return fq_mul(a, b); }
struct FqCall {
  static __device__ __forceinline__ fq_t mul(const fq_t& a, const fq_t& b) {
    return fq_mul_call(a, b);
  }
  static __device__ __forceinline__ void mul2(const fq_t& a, const fq_t& b, const fq_t& c,
                                              const fq_t& d, fq_t& x, fq_t& y) {
    x = fq_mul_call(a, b);
    y = fq_mul_call(c, d);
  }
};
struct fq_pair_t {
  fq_t x, y;
};
__device__ __noinline__ fq_pair_t fq_mul2_call(fq_t a, fq_t b, fq_t c, fq_t d) {
  return {fq_mul(a, b), fq_mul(c, d)};
}
struct FqPair {
  static __device__ __forceinline__ fq_t mul(const fq_t& a, const fq_t& b) {
    return fq_mul_call(a, b);
  }
  static __device__ __forceinline__ void mul2(const fq_t& a, const fq_t& b, const fq_t& c,
                                              const fq_t& d, fq_t& x, fq_t& y) {
    const fq_pair_t r = fq_mul2_call(a, b, c, d);
    x = r.x;
    y = r.y;
  }
};

__device__ __forceinline__ g1_xyzz_t xyzz_infinity() {
  g1_xyzz_t p;
  p.x = fq_zero();
  p.y = fq_zero();
  p.zz = fq_zero();
  p.zzz = fq_zero();
  return p;
}

__device__ __forceinline__ bool xyzz_is_inf(const g1_xyzz_t& p) { return fq_is_zero(p.zz); }

__device__ __forceinline__ bool aff_is_inf(const g1_aff_t& p) {
  return fq_is_zero_raw(p.x) && fq_is_zero_raw(p.y);
}

__device__ __forceinline__ g1_xyzz_t xyzz_from_aff(const g1_aff_t& a) {
  if (aff_is_inf(a)) return xyzz_infinity();
  g1_xyzz_t p;
  p.x = a.x;
  p.y = a.y;
  p.zz = fq_one();
  p.zzz = fq_one();
  return p;
}

// 2P for P in (X, Y, ZZ, ZZZ) (dbl-2008-s-1, a = 0):
//   U = 2Y, V = U^2, W = U V, S = X V, M = 3 X^2,
//   X3 = M^2 - 2S, Y3 = M (S - X3) - W Y, ZZ3 = V ZZ, ZZZ3 = W ZZZ.
// Infinity doubles to itself (V = W = 0 when ZZ = 0 keeps ZZ3 = 0); y = 0 does not occur
// (the group has odd order r) but would give ZZ3 = 0, the right answer, too.
template <class M>
__device__ __forceinline__ g1_xyzz_t xyzz_dbl_t(const g1_xyzz_t& p) {
  const fq_t u = fq_dbl(p.y);
  fq_t v, xx, w, s, mm, my, wy;
  M::mul2(u, u, p.x, p.x, v, xx);
  M::mul2(u, v, p.x, v, w, s);
  const fq_t m = fq_add(fq_dbl(xx), xx);
  g1_xyzz_t r;
  M::mul2(m, m, v, p.zz, mm, r.zz);
  r.x = fq_sub(mm, fq_dbl(s));
  M::mul2(m, fq_sub(s, r.x), w, p.y, my, wy);
  r.y = fq_sub(my, wy);
  r.zzz = M::mul(w, p.zzz);
  return r;
}

// 2P for an affine P (mdbl-2008-s-1: ZZ = ZZZ = 1, so ZZ3 = V, ZZZ3 = W).
template <class M>
__device__ __forceinline__ g1_xyzz_t xyzz_mdbl_t(const g1_aff_t& p) {
  const fq_t u = fq_dbl(p.y);
  const fq_t v = M::mul(u, u);
  const fq_t w = M::mul(u, v);
  const fq_t s = M::mul(p.x, v);
  const fq_t xx = M::mul(p.x, p.x);
  const fq_t m = fq_add(fq_dbl(xx), xx);
  g1_xyzz_t r;
  r.x = fq_sub(M::mul(m, m), fq_dbl(s));
  r.y = fq_sub(M::mul(m, fq_sub(s, r.x)), M::mul(w, p.y));
  r.zz = v;
  r.zzz = w;
  return r;
}

// acc + b, b affine and not at infinity (madd-2008-s):
//   U2 = x2 ZZ1, S2 = y2 ZZZ1, P = U2 - X1, R = S2 - Y1, PP = P^2, PPP = P PP, Q = X1 PP,
//   X3 = R^2 - PPP - 2Q, Y3 = R (Q - X3) - Y1 PPP, ZZ3 = ZZ1 PP, ZZZ3 = ZZZ1 PPP.
// P = 0 means the same x: R = 0 is the same point (double b), else opposite points
// (infinity).
template <class M>
__device__ __forceinline__ g1_xyzz_t xyzz_madd_t(const g1_xyzz_t& acc, const g1_aff_t& b) {
  if (xyzz_is_inf(acc)) return xyzz_from_aff(b);
  const fq_t u2 = M::mul(b.x, acc.zz);
  const fq_t s2 = M::mul(b.y, acc.zzz);
  const fq_t p = fq_sub(u2, acc.x);
  const fq_t r = fq_sub(s2, acc.y);
  if (fq_is_zero(p)) {
    if (fq_is_zero(r)) return xyzz_mdbl_t<M>(b);
    return xyzz_infinity();
  }
  const fq_t pp = M::mul(p, p);
  const fq_t ppp = M::mul(p, pp);
  const fq_t q = M::mul(acc.x, pp);
  g1_xyzz_t o;
  o.x = fq_sub(fq_sub(M::mul(r, r), ppp), fq_dbl(q));
  o.y = fq_sub(M::mul(r, fq_sub(q, o.x)), M::mul(acc.y, ppp));
  o.zz = M::mul(acc.zz, pp);
  o.zzz = M::mul(acc.zzz, ppp);
  return o;
}

// a + b, both in (X, Y, ZZ, ZZZ) (add-2008-s):
//   U1 = X1 ZZ2, U2 = X2 ZZ1, S1 = Y1 ZZZ2, S2 = Y2 ZZZ1, P = U2 - U1, R = S2 - S1,
//   PP = P^2, PPP = P PP, Q = U1 PP, X3 = R^2 - PPP - 2Q, Y3 = R (Q - X3) - S1 PPP,
//   ZZ3 = ZZ1 ZZ2 PP, ZZZ3 = ZZZ1 ZZZ2 PPP.
template <class M>
__device__ __forceinline__ g1_xyzz_t xyzz_add_t(const g1_xyzz_t& a, const g1_xyzz_t& b) {
  if (xyzz_is_inf(a)) return b;
  if (xyzz_is_inf(b)) return a;
  fq_t u1, u2, s1, s2;
  M::mul2(a.x, b.zz, b.x, a.zz, u1, u2);
  M::mul2(a.y, b.zzz, b.y, a.zzz, s1, s2);
  const fq_t p = fq_sub(u2, u1);
  const fq_t r = fq_sub(s2, s1);
  if (fq_is_zero(p)) {
    if (fq_is_zero(r)) return xyzz_dbl_t<M>(a);
    return xyzz_infinity();
  }
  fq_t pp, rr, ppp, q, zz12, zzz12, ry, sp;
  M::mul2(p, p, r, r, pp, rr);
  M::mul2(p, pp, u1, pp, ppp, q);
  M::mul2(a.zz, b.zz, a.zzz, b.zzz, zz12, zzz12);
  g1_xyzz_t o;
  o.x = fq_sub(fq_sub(rr, ppp), fq_dbl(q));
  M::mul2(r, fq_sub(q, o.x), s1, ppp, ry, sp);
  o.y = fq_sub(ry, sp);
  M::mul2(zz12, pp, zzz12, ppp, o.zz, o.zzz);
  return o;
}

__device__ __forceinline__ g1_xyzz_t xyzz_dbl(const g1_xyzz_t& p) { return xyzz_dbl_t<FqInline>(p); }
__device__ __forceinline__ g1_xyzz_t xyzz_madd(const g1_xyzz_t& acc, const g1_aff_t& b) {
  return xyzz_madd_t<FqInline>(acc, b);
}
__device__ __forceinline__ g1_xyzz_t xyzz_add(const g1_xyzz_t& a, const g1_xyzz_t& b) {
  return xyzz_add_t<FqInline>(a, b);
}

// The affine point of p, canonical coordinates; (0, 0) for infinity. One inversion:
// with i = 1/ZZZ, 1/ZZ = ZZ^2 i^2 (as ZZ^3 = ZZZ^2), so x = X ZZ^2 i^2 and y = Y i.
__device__ __forceinline__ g1_aff_t xyzz_to_aff(const g1_xyzz_t& p) {
  g1_aff_t a;
  if (xyzz_is_inf(p)) {
    a.x = fq_zero();
    a.y = fq_zero();
    return a;
  }
  const fq_t i = fq_inv(p.zzz);
  const fq_t zz_i = fq_mul(p.zz, i);  // ZZ / ZZZ
  a.x = fq_canon(fq_mul(p.x, fq_sqr(zz_i)));
  a.y = fq_canon(fq_mul(p.y, i));
  return a;
}

// Jacobian (X', Y', Z') of p with x = X'/Z'^2, y = Y'/Z'^3: Z' = ZZ ZZZ,
// X' = X ZZ ZZZ^2, Y' = Y ZZ^3 ZZZ^2 (no inversion); infinity as (0, 0, 0).
template <class M>
__device__ __forceinline__ void xyzz_to_jacobian_t(const g1_xyzz_t& p, fq_t& X, fq_t& Y,
                                                   fq_t& Z) {
  if (xyzz_is_inf(p)) {
    X = fq_zero();
    Y = fq_zero();
    Z = fq_zero();
    return;
  }
  const fq_t z = M::mul(p.zz, p.zzz);
  const fq_t zzz2 = M::mul(p.zzz, p.zzz);
  X = fq_canon(M::mul(M::mul(p.x, p.zz), zzz2));
  const fq_t zz3 = M::mul(M::mul(p.zz, p.zz), p.zz);
  Y = fq_canon(M::mul(M::mul(p.y, zz3), zzz2));
  Z = fq_canon(z);
}

__device__ __forceinline__ g1_aff_t aff_neg(const g1_aff_t& a) {
  g1_aff_t r;
  r.x = a.x;
  r.y = fq_canon(fq_neg(a.y));
  return r;
}

// y^2 == x^3 + 3 for canonical (x, y) not at infinity.
__device__ __forceinline__ bool aff_on_curve(const g1_aff_t& a) {
  const uint32_t three[8] = G3H_QTHREE;
  fq_t b;
#pragma unroll
  for (int i = 0; i < 8; i++) b.v[i] = three[i];
  const fq_t lhs = fq_canon(fq_sqr(a.y));
  const fq_t rhs = fq_canon(fq_add(fq_mul(fq_sqr(a.x), a.x), b));
  bool eq = true;
#pragma unroll
  for (int i = 0; i < 8; i++) eq = eq && lhs.v[i] == rhs.v[i];
  return eq;
}

}  // namespace g3h
