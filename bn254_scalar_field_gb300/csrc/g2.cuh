// BN254 G2 for the witness multiexp of the B query (MSM_CU stage 7): points of the twist
// E': y^2 = x^3 + b2 over F_q2 = F_q[u]/(u^2 + 1), b2 = 3 / (9 + u) (EIP-197).
//
// F_q2 elements are pairs (c0, c1) of fq_t meaning c0 + c1 u, each in Montgomery form and
// lazily reduced to [0, 2q) like fq_t. Multiplication by Karatsuba (3 F_q multiplies),
// squaring by (c0 + c1)(c0 - c1), 2 c0 c1 (2 multiplies), inverse through the norm
// c0^2 + c1^2 (one F_q inversion). The point formulas are those of g1.cuh for the same
// (X, Y, ZZ, ZZZ) coordinates (they do not depend on b), over F_q2.
#pragma once
#include "g1.cuh"

namespace g3h {

struct __align__(16) fq2_t {
  fq_t c0, c1;
};

__device__ __forceinline__ fq2_t fq2_zero() { return {fq_zero(), fq_zero()}; }
__device__ __forceinline__ fq2_t fq2_one() { return {fq_one(), fq_zero()}; }
__device__ __forceinline__ fq2_t fq2_add(const fq2_t& a, const fq2_t& b) {
  return {fq_add(a.c0, b.c0), fq_add(a.c1, b.c1)};
}
__device__ __forceinline__ fq2_t fq2_sub(const fq2_t& a, const fq2_t& b) {
  return {fq_sub(a.c0, b.c0), fq_sub(a.c1, b.c1)};
}
__device__ __forceinline__ fq2_t fq2_dbl(const fq2_t& a) { return fq2_add(a, a); }
__device__ __forceinline__ fq2_t fq2_neg(const fq2_t& a) { return {fq_neg(a.c0), fq_neg(a.c1)}; }
__device__ __forceinline__ fq2_t fq2_canon(const fq2_t& a) { return {fq_canon(a.c0), fq_canon(a.c1)}; }
__device__ __forceinline__ bool fq2_is_zero(const fq2_t& a) { return fq_is_zero(a.c0) && fq_is_zero(a.c1); }
__device__ __forceinline__ bool fq2_is_zero_raw(const fq2_t& a) {
  return fq_is_zero_raw(a.c0) && fq_is_zero_raw(a.c1);
}
__device__ __forceinline__ bool fq2_is_canonical(const fq2_t& a) {
  return fq_is_canonical(a.c0) && fq_is_canonical(a.c1);
}

// (a0 + a1 u)(b0 + b1 u): v0 = a0 b0, v1 = a1 b1, c0 = v0 - v1, c1 = (a0 + a1)(b0 + b1) - v0 - v1.
template <class M>
__device__ __forceinline__ fq2_t fq2_mul_t(const fq2_t& a, const fq2_t& b) {
  const fq_t v0 = M::mul(a.c0, b.c0), v1 = M::mul(a.c1, b.c1);
  const fq_t s = M::mul(fq_add(a.c0, a.c1), fq_add(b.c0, b.c1));
  return {fq_sub(v0, v1), fq_sub(fq_sub(s, v0), v1)};
}

// (a0 + a1 u)^2 = (a0 + a1)(a0 - a1) + 2 a0 a1 u.
template <class M>
__device__ __forceinline__ fq2_t fq2_sqr_t(const fq2_t& a) {
  const fq_t t = M::mul(a.c0, a.c1);
  return {M::mul(fq_add(a.c0, a.c1), fq_sub(a.c0, a.c1)), fq_dbl(t)};
}

// F_q2 products as out-of-line calls with their F_q multiplies inlined: one call per F_q2
// product, whose three (two for a square) independent F_q products interleave.
__device__ __noinline__ fq2_t fq2_mul_call(fq2_t a, fq2_t b) { return fq2_mul_t<FqInline>(a, b); }
__device__ __noinline__ fq2_t fq2_sqr_call(fq2_t a) { return fq2_sqr_t<FqInline>(a); }
struct Fq2Call {};
template <>
__device__ __forceinline__ fq2_t fq2_mul_t<Fq2Call>(const fq2_t& a, const fq2_t& b) {
  return fq2_mul_call(a, b);
}
template <>
__device__ __forceinline__ fq2_t fq2_sqr_t<Fq2Call>(const fq2_t& a) {
  return fq2_sqr_call(a);
}

// 1 / (a0 + a1 u) = (a0 - a1 u) / (a0^2 + a1^2); 0 maps to 0.
__device__ __forceinline__ fq2_t fq2_inv(const fq2_t& a) {
  const fq_t ni = fq_inv(fq_add(fq_mul(a.c0, a.c0), fq_mul(a.c1, a.c1)));
  return {fq_mul(a.c0, ni), fq_mul(fq_neg(a.c1), ni)};
}

struct __align__(16) g2_aff_t {
  fq2_t x, y;
};

struct __align__(16) g2_xyzz_t {
  fq2_t x, y, zz, zzz;
};

__device__ __forceinline__ g2_xyzz_t g2_infinity() {
  return {fq2_zero(), fq2_zero(), fq2_zero(), fq2_zero()};
}
__device__ __forceinline__ bool g2_is_inf(const g2_xyzz_t& p) { return fq2_is_zero(p.zz); }
__device__ __forceinline__ bool g2_aff_is_inf(const g2_aff_t& p) {
  return fq2_is_zero_raw(p.x) && fq2_is_zero_raw(p.y);
}
__device__ __forceinline__ g2_xyzz_t g2_from_aff(const g2_aff_t& a) {
  if (g2_aff_is_inf(a)) return g2_infinity();
  return {a.x, a.y, fq2_one(), fq2_one()};
}
__device__ __forceinline__ g2_aff_t g2_aff_neg(const g2_aff_t& a) {
  return {a.x, fq2_canon(fq2_neg(a.y))};
}

// dbl-2008-s-1 over F_q2 (see xyzz_dbl_t)
template <class M>
__device__ __forceinline__ g2_xyzz_t g2_dbl_t(const g2_xyzz_t& p) {
  const fq2_t u = fq2_dbl(p.y);
  const fq2_t v = fq2_sqr_t<M>(u);
  const fq2_t w = fq2_mul_t<M>(u, v);
  const fq2_t s = fq2_mul_t<M>(p.x, v);
  const fq2_t xx = fq2_sqr_t<M>(p.x);
  const fq2_t m = fq2_add(fq2_dbl(xx), xx);
  g2_xyzz_t r;
  r.x = fq2_sub(fq2_sqr_t<M>(m), fq2_dbl(s));
  r.y = fq2_sub(fq2_mul_t<M>(m, fq2_sub(s, r.x)), fq2_mul_t<M>(w, p.y));
  r.zz = fq2_mul_t<M>(v, p.zz);
  r.zzz = fq2_mul_t<M>(w, p.zzz);
  return r;
}

// mdbl-2008-s-1 over F_q2
template <class M>
__device__ __forceinline__ g2_xyzz_t g2_mdbl_t(const g2_aff_t& p) {
  const fq2_t u = fq2_dbl(p.y);
  const fq2_t v = fq2_sqr_t<M>(u);
  const fq2_t w = fq2_mul_t<M>(u, v);
  const fq2_t s = fq2_mul_t<M>(p.x, v);
  const fq2_t xx = fq2_sqr_t<M>(p.x);
  const fq2_t m = fq2_add(fq2_dbl(xx), xx);
  g2_xyzz_t r;
  r.x = fq2_sub(fq2_sqr_t<M>(m), fq2_dbl(s));
  r.y = fq2_sub(fq2_mul_t<M>(m, fq2_sub(s, r.x)), fq2_mul_t<M>(w, p.y));
  r.zz = v;
  r.zzz = w;
  return r;
}

// madd-2008-s over F_q2, b not at infinity (see xyzz_madd_t)
template <class M>
__device__ __forceinline__ g2_xyzz_t g2_madd_t(const g2_xyzz_t& acc, const g2_aff_t& b) {
  if (g2_is_inf(acc)) return g2_from_aff(b);
  const fq2_t u2 = fq2_mul_t<M>(b.x, acc.zz);
  const fq2_t s2 = fq2_mul_t<M>(b.y, acc.zzz);
  const fq2_t p = fq2_sub(u2, acc.x);
  const fq2_t r = fq2_sub(s2, acc.y);
  if (fq2_is_zero(p)) {
    if (fq2_is_zero(r)) return g2_mdbl_t<M>(b);
    return g2_infinity();
  }
  const fq2_t pp = fq2_sqr_t<M>(p);
  const fq2_t ppp = fq2_mul_t<M>(p, pp);
  const fq2_t q = fq2_mul_t<M>(acc.x, pp);
  g2_xyzz_t o;
  o.x = fq2_sub(fq2_sub(fq2_sqr_t<M>(r), ppp), fq2_dbl(q));
  o.y = fq2_sub(fq2_mul_t<M>(r, fq2_sub(q, o.x)), fq2_mul_t<M>(acc.y, ppp));
  o.zz = fq2_mul_t<M>(acc.zz, pp);
  o.zzz = fq2_mul_t<M>(acc.zzz, ppp);
  return o;
}

// add-2008-s over F_q2 (see xyzz_add_t)
template <class M>
__device__ __forceinline__ g2_xyzz_t g2_add_t(const g2_xyzz_t& a, const g2_xyzz_t& b) {
  if (g2_is_inf(a)) return b;
  if (g2_is_inf(b)) return a;
  const fq2_t u1 = fq2_mul_t<M>(a.x, b.zz);
  const fq2_t u2 = fq2_mul_t<M>(b.x, a.zz);
  const fq2_t s1 = fq2_mul_t<M>(a.y, b.zzz);
  const fq2_t s2 = fq2_mul_t<M>(b.y, a.zzz);
  const fq2_t p = fq2_sub(u2, u1);
  const fq2_t r = fq2_sub(s2, s1);
  if (fq2_is_zero(p)) {
    if (fq2_is_zero(r)) return g2_dbl_t<M>(a);
    return g2_infinity();
  }
  const fq2_t pp = fq2_sqr_t<M>(p);
  const fq2_t ppp = fq2_mul_t<M>(p, pp);
  const fq2_t q = fq2_mul_t<M>(u1, pp);
  g2_xyzz_t o;
  o.x = fq2_sub(fq2_sub(fq2_sqr_t<M>(r), ppp), fq2_dbl(q));
  o.y = fq2_sub(fq2_mul_t<M>(r, fq2_sub(q, o.x)), fq2_mul_t<M>(s1, ppp));
  o.zz = fq2_mul_t<M>(fq2_mul_t<M>(a.zz, b.zz), pp);
  o.zzz = fq2_mul_t<M>(fq2_mul_t<M>(a.zzz, b.zzz), ppp);
  return o;
}

// Affine, canonical; (0, 0) for infinity (one F_q2 inversion, as xyzz_to_aff).
__device__ __forceinline__ g2_aff_t g2_to_aff(const g2_xyzz_t& p) {
  if (g2_is_inf(p)) return {fq2_zero(), fq2_zero()};
  const fq2_t i = fq2_inv(p.zzz);
  const fq2_t zz_i = fq2_mul_t<FqInline>(p.zz, i);
  return {fq2_canon(fq2_mul_t<FqInline>(p.x, fq2_sqr_t<FqInline>(zz_i))),
          fq2_canon(fq2_mul_t<FqInline>(p.y, i))};
}

// Jacobian (X ZZ ZZZ^2, Y ZZ^3 ZZZ^2, ZZ ZZZ) as xyzz_to_jacobian_t, over F_q2; out[0..2]
// are X, Y, Z, canonical; infinity (0, 0, 0).
template <class M>
__device__ __forceinline__ void g2_to_jacobian_t(const g2_xyzz_t& p, fq2_t* out) {
  if (g2_is_inf(p)) {
    out[0] = out[1] = out[2] = fq2_zero();
    return;
  }
  const fq2_t zzz2 = fq2_sqr_t<M>(p.zzz);
  out[0] = fq2_canon(fq2_mul_t<M>(fq2_mul_t<M>(p.x, p.zz), zzz2));
  const fq2_t zz3 = fq2_mul_t<M>(fq2_sqr_t<M>(p.zz), p.zz);
  out[1] = fq2_canon(fq2_mul_t<M>(fq2_mul_t<M>(p.y, zz3), zzz2));
  out[2] = fq2_canon(fq2_mul_t<M>(p.zz, p.zzz));
}

// y^2 == x^3 + b2 for canonical (x, y) not at infinity; b2 = 3 / (9 + u), Montgomery.
__device__ __forceinline__ bool g2_aff_on_curve(const g2_aff_t& a) {
  const uint32_t b0[8] = {0x77b802a8u, 0x3bf938e3u, 0x3633535du, 0x020b1b27u,
                          0x49755260u, 0x26b7edf0u, 0x4384a86du, 0x2514c632u};
  const uint32_t b1[8] = {0xd1dcff67u, 0x38e7ecccu, 0x93ce0d3eu, 0x65f0b37du,
                          0x22ac00aau, 0xd749d0ddu, 0x4a688d4du, 0x0141b9ceu};
  fq2_t b;
#pragma unroll
  for (int i = 0; i < 8; i++) {
    b.c0.v[i] = b0[i];
    b.c1.v[i] = b1[i];
  }
  const fq2_t lhs = fq2_canon(fq2_sqr_t<FqInline>(a.y));
  const fq2_t rhs = fq2_canon(fq2_add(fq2_mul_t<FqInline>(fq2_sqr_t<FqInline>(a.x), a.x), b));
  bool eq = true;
#pragma unroll
  for (int i = 0; i < 8; i++)
    eq = eq && lhs.c0.v[i] == rhs.c0.v[i] && lhs.c1.v[i] == rhs.c1.v[i];
  return eq;
}

}  // namespace g3h
