// The H multiexp: Q = sum_i s_i P_i over BN254 G1 (MSM_CU, stage 9: Pippenger over G1
// with the standard-form h of POINTWISE_CU as scalars), by the bucket method.
//
// Scalars are split into 16 signed digits of 16 bits (s = sum_w d_w 2^(16 w),
// d_w in [-2^15, 2^15]; a digit above 2^15 becomes d - 2^16 with a carry into the next
// window, and since s < r < 2^254 the last window never carries out). The bases are
// fixed per proving key, so the context keeps, for every base P_i, the 16 affine points
// 2^(16 w) P_i (prepared once, 1 KiB per base). Then
//   Q = sum_i sum_w d_{i,w} 2^(16 w) P_i = sum_{j=1}^{2^15} j B_j,
//   B_j = sum over (i, w) with |d_{i,w}| = j of sign(d_{i,w}) 2^(16 w) P_i,
// one set of 2^15 buckets for all windows: no per-window bucket sums and no doubling
// chain between windows. Steps:
//   0. ones: the bases whose scalar is exactly 1 are summed apart (a tree per block, then
//      one block), so they do not pile into one bucket; on a second stream, from the end
//      of step 3 on;
//   1. count: per-bucket entry counts of each sort block (one per SM, counters in shared
//      memory), then per bucket the prefix over the blocks and the total;
//   2. scan: exclusive prefix sum of the totals (bucket offsets);
//   3. scatter: each (i, w) entry, as (16 i + w) << 1 | sign, into its bucket's run at its
//      block's place (a counting sort by bucket; order inside a run is arbitrary, the sum
//      commutes);
//   4. accumulate: the sorted entries in fixed-length slices, one thread per slice, so
//      that work per thread does not depend on how the digits spread over buckets; a run
//      that lies inside one slice is written to its bucket, a run cut by a slice boundary
//      leaves its part in that slice's head or tail slot (MSM_CU, "the load-balanced
//      form": segmented accumulation with boundary spills);
//   5. merge: a cut bucket sums its parts from the slices its run covers (one thread per
//      bucket; a block per bucket for runs over many slices);
//   6-8. the weighted sum sum_j j B_j: per pair of buckets (t = 0 .. 16383) U_t and V_t;
//      then Q = sum_t V_t + sum_b 2^(b+1) sum_{t : bit b of t} U_t, fourteen bit-sums and
//      one sum of V reduced by trees over all SMs, scaled by doublings (one SM per part)
//      and added in a last kernel, which writes Q in Jacobian coordinates.
#pragma once
#include "fr.cuh"
#include "g1.cuh"
#include "g2.cuh"

namespace g3h {

constexpr uint32_t kMsmWindows = 16;          // windows of 16 bits
constexpr uint32_t kMsmBuckets = 1u << 15;    // digit magnitudes 1 .. 2^15
constexpr uint32_t kMsmErrPoint = 2u;  // error word bit: a base is not on the curve

// The bucket sum's point operations (see the kernels below) call out-of-line copies built
// on one out-of-line multiply, so that the code their few warps loop over stays in the
// instruction cache.
using FqTail = FqCall;
__device__ __noinline__ g1_xyzz_t xyzz_add_nl(g1_xyzz_t a, g1_xyzz_t b) {
  return xyzz_add_t<FqTail>(a, b);
}
// The same for the kernels that run one warp per SM (the upper levels of the parts' and
// the last sum's trees): their time is the chain of multiplies, and pairs of independent
// ones overlap in part (between their carry chains, which share the one carry flag).
// Where many warps run, the pairs measured slower.
using FqLat = FqPair;
__device__ __noinline__ g1_xyzz_t xyzz_add_lat(g1_xyzz_t a, g1_xyzz_t b) {
  return xyzz_add_t<FqLat>(a, b);
}
__device__ __noinline__ g2_xyzz_t g2_add_nl(g2_xyzz_t a, g2_xyzz_t b) {
  return g2_add_t<Fq2Call>(a, b);
}

// Doublings by a whole warp, for the one-lane chain of doublings in the parts' kernel:
// every lane holds the point, the independent F_q products of each step of dbl-2008-s-1
// go to different lanes (one out-of-line multiply each) and come back by shuffles, so a
// doubling waits on four multiplies instead of nine (G1) or 27 (G2). The products and
// their operands are those of xyzz_dbl_t / g2_dbl_t, so the results are the same
// representatives. All 32 lanes must call it together.
__device__ __forceinline__ fq_t fq_shfl(const fq_t& x, uint32_t src) {
  fq_t o;
#pragma unroll
  for (int i = 0; i < 8; i++) o.v[i] = __shfl_sync(0xffffffffu, x.v[i], src);
  return o;
}

__device__ __forceinline__ fq_t fq_sel(bool c, const fq_t& a, const fq_t& b) {
  fq_t o;
#pragma unroll
  for (int i = 0; i < 8; i++) o.v[i] = c ? a.v[i] : b.v[i];
  return o;
}

__device__ __noinline__ g1_xyzz_t xyzz_dbl_coop(g1_xyzz_t p) {
  const uint32_t lane = threadIdx.x & 31u;
  const fq_t u = fq_dbl(p.y);
  // V = U U (lane 0), XX = X X (lane 1)
  const fq_t a1 = fq_sel(lane == 0, u, p.x);
  fq_t r = fq_mul_call(a1, a1);
  const fq_t v = fq_shfl(r, 0), xx = fq_shfl(r, 1);
  // W = U V (0), S = X V (1), ZZ3 = ZZ V (2; the Montgomery product is symmetric)
  r = fq_mul_call(fq_sel(lane == 0, u, fq_sel(lane == 1, p.x, p.zz)), v);
  const fq_t w = fq_shfl(r, 0), s = fq_shfl(r, 1), zz3 = fq_shfl(r, 2);
  const fq_t m = fq_add(fq_dbl(xx), xx);
  // M M (0), W Y (1), W ZZZ (2)
  r = fq_mul_call(fq_sel(lane == 0, m, w), fq_sel(lane == 0, m, fq_sel(lane == 1, p.y, p.zzz)));
  const fq_t mm = fq_shfl(r, 0), wy = fq_shfl(r, 1), zzz3 = fq_shfl(r, 2);
  g1_xyzz_t o;
  o.x = fq_sub(mm, fq_dbl(s));
  o.y = fq_sub(fq_mul_call(m, fq_sub(s, o.x)), wy);
  o.zz = zz3;
  o.zzz = zzz3;
  return o;
}

// The F_q products of an F_q2 product a b (Karatsuba, as fq2_mul_t): k = 0: a0 b0,
// 1: a1 b1, 2: (a0 + a1)(b0 + b1); and of a square (as fq2_sqr_t): 0: a0 a1,
// 1: (a0 + a1)(a0 - a1).
__device__ __forceinline__ void fq2_mul_operands(uint32_t k, const fq2_t& a, const fq2_t& b,
                                                 fq_t& x, fq_t& y) {
  x = k == 0 ? a.c0 : (k == 1 ? a.c1 : fq_add(a.c0, a.c1));
  y = k == 0 ? b.c0 : (k == 1 ? b.c1 : fq_add(b.c0, b.c1));
}
__device__ __forceinline__ void fq2_sqr_operands(uint32_t k, const fq2_t& a, fq_t& x, fq_t& y) {
  x = k == 0 ? a.c0 : fq_add(a.c0, a.c1);
  y = k == 0 ? a.c1 : fq_sub(a.c0, a.c1);
}
// The F_q2 product from its three F_q products on lanes l, l + 1, l + 2.
__device__ __forceinline__ fq2_t fq2_mul_gather(const fq_t& r, uint32_t l) {
  const fq_t v0 = fq_shfl(r, l), v1 = fq_shfl(r, l + 1), sm = fq_shfl(r, l + 2);
  return {fq_sub(v0, v1), fq_sub(fq_sub(sm, v0), v1)};
}
// The F_q2 square from its two F_q products on lanes l, l + 1.
__device__ __forceinline__ fq2_t fq2_sqr_gather(const fq_t& r, uint32_t l) {
  const fq_t t = fq_shfl(r, l), c0 = fq_shfl(r, l + 1);
  return {c0, fq_dbl(t)};
}

__device__ __noinline__ g2_xyzz_t g2_dbl_coop(g2_xyzz_t p) {
  const uint32_t lane = threadIdx.x & 31u;
  fq_t x, y;
  const fq2_t u = fq2_dbl(p.y);
  // V = U^2 (lanes 0-1), XX = X^2 (lanes 2-3)
  fq2_sqr_operands(lane & 1u, lane < 2 ? u : p.x, x, y);
  fq_t r = fq_mul_call(x, y);
  const fq2_t v = fq2_sqr_gather(r, 0), xx = fq2_sqr_gather(r, 2);
  // W = U V (0-2), S = X V (3-5), ZZ3 = V ZZ (6-8)
  {
    const uint32_t g = lane < 3 ? 0u : (lane < 6 ? 1u : 2u);
    const fq2_t a = g == 0 ? u : (g == 1 ? p.x : v);
    const fq2_t b = g == 2 ? p.zz : v;
    fq2_mul_operands(lane - 3u * g, a, b, x, y);
  }
  r = fq_mul_call(x, y);
  const fq2_t w = fq2_mul_gather(r, 0), s = fq2_mul_gather(r, 3), zz3 = fq2_mul_gather(r, 6);
  const fq2_t m = fq2_add(fq2_dbl(xx), xx);
  // M^2 (0-1), W Y (2-4), W ZZZ (5-7)
  if (lane < 2) {
    fq2_sqr_operands(lane, m, x, y);
  } else {
    const uint32_t g = lane < 5 ? 0u : 1u;
    fq2_mul_operands(lane - 2u - 3u * g, w, g == 0 ? p.y : p.zzz, x, y);
  }
  r = fq_mul_call(x, y);
  const fq2_t mm = fq2_sqr_gather(r, 0), wy = fq2_mul_gather(r, 2), zzz3 = fq2_mul_gather(r, 5);
  g2_xyzz_t o;
  o.x = fq2_sub(mm, fq2_dbl(s));
  // M (S - X3) (0-2)
  fq2_mul_operands(lane < 3 ? lane : 2u, m, fq2_sub(s, o.x), x, y);
  r = fq_mul_call(x, y);
  o.y = fq2_sub(fq2_mul_gather(r, 0), wy);
  o.zz = zz3;
  o.zzz = zzz3;
  return o;
}

// An addition by a whole warp (add-2008-s, as xyzz_add_t, the same products of the same
// operands): four steps of independent F_q products spread over the lanes. Every lane
// passes the same a and b; all 32 lanes must call it together. (Over G2 the same scheme,
// 18 lanes per step, measured slower than one thread per addition: 1.63 -> 1.65 ms.)
__device__ __noinline__ g1_xyzz_t xyzz_add_coop(g1_xyzz_t a, g1_xyzz_t b) {
  if (xyzz_is_inf(a)) return b;
  if (xyzz_is_inf(b)) return a;
  const uint32_t lane = threadIdx.x & 31u;
  // U1 = X1 ZZ2 (0), U2 = X2 ZZ1 (1), S1 = Y1 ZZZ2 (2), S2 = Y2 ZZZ1 (3), ZZ1 ZZ2 (4),
  // ZZZ1 ZZZ2 (5)
  const fq_t x = fq_sel(lane == 0, a.x, fq_sel(lane == 1, b.x, fq_sel(lane == 2, a.y,
                 fq_sel(lane == 3, b.y, fq_sel(lane == 4, a.zz, a.zzz)))));
  const fq_t y = fq_sel(lane == 0, b.zz, fq_sel(lane == 1, a.zz, fq_sel(lane == 2, b.zzz,
                 fq_sel(lane == 3, a.zzz, fq_sel(lane == 4, b.zz, b.zzz)))));
  fq_t r = fq_mul_call(x, y);
  const fq_t u1 = fq_shfl(r, 0), u2 = fq_shfl(r, 1), s1 = fq_shfl(r, 2), s2 = fq_shfl(r, 3);
  const fq_t zz12 = fq_shfl(r, 4), zzz12 = fq_shfl(r, 5);
  const fq_t p = fq_sub(u2, u1), rr0 = fq_sub(s2, s1);
  if (fq_is_zero(p)) {
    if (fq_is_zero(rr0)) return xyzz_dbl_coop(a);
    return xyzz_infinity();
  }
  // PP = P P (0), RR = R R (1)
  const fq_t pr = fq_sel(lane == 0, p, rr0);
  r = fq_mul_call(pr, pr);
  const fq_t pp = fq_shfl(r, 0), rr = fq_shfl(r, 1);
  // PPP = P PP (0), Q = U1 PP (1), ZZ3 = ZZ1 ZZ2 PP (2)
  r = fq_mul_call(fq_sel(lane == 0, p, fq_sel(lane == 1, u1, zz12)), pp);
  const fq_t ppp = fq_shfl(r, 0), q = fq_shfl(r, 1);
  g1_xyzz_t o;
  o.zz = fq_shfl(r, 2);
  o.x = fq_sub(fq_sub(rr, ppp), fq_dbl(q));
  // R (Q - X3) (0), S1 PPP (1), ZZZ1 ZZZ2 PPP (2)
  r = fq_mul_call(fq_sel(lane == 0, rr0, fq_sel(lane == 1, s1, zzz12)),
                  fq_sel(lane == 0, fq_sub(q, o.x), ppp));
  o.y = fq_sub(fq_shfl(r, 0), fq_shfl(r, 1));
  o.zzz = fq_shfl(r, 2);
  return o;
}

// One level of a shuffle tree by the whole warp: lanes j < d replace acc by acc + o, one
// addition after another, each by all lanes. All 32 lanes must call it together.
template <class G>
__device__ __forceinline__ void coop_level(typename G::Pt& acc, const typename G::Pt& o, uint32_t d) {
  const uint32_t lane = threadIdx.x & 31u;
  for (uint32_t j = 0; j < d; j++) {
    const typename G::Pt r = G::add_coop(pt_shfl(acc, j), pt_shfl(o, j));
    if (lane == j) acc = r;
  }
}

template <class P>
__device__ __forceinline__ P pt_shfl_down(const P& p, uint32_t d) {
  constexpr int words = sizeof(P) / 4;
  const uint32_t* src = reinterpret_cast<const uint32_t*>(&p);
  P o;
  uint32_t* dst = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int w = 0; w < words; w++) dst[w] = __shfl_down_sync(0xffffffffu, src[w], d);
  return o;
}

template <class P>
__device__ __forceinline__ P pt_shfl(const P& p, uint32_t src) {
  constexpr int words = sizeof(P) / 4;
  const uint32_t* in = reinterpret_cast<const uint32_t*>(&p);
  P o;
  uint32_t* out = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
  for (int w = 0; w < words; w++) out[w] = __shfl_sync(0xffffffffu, in[w], src);
  return o;
}

// The group of a multiexp: its point types and operations. G1: points of E over F_q, the
// bucket additions inlined (many warps keep the multiply pipe busy). G2: points of the
// twist over F_q2, every F_q2 product one out-of-line call whose three F_q products are
// inlined and interleave (an inlined F_q2 addition would be some 90 KB of code; a call per
// F_q product measured 0.73 -> 0.65 ms for the 2^16 accumulation, 2.00 -> 1.75 ms for the
// whole multiexp), trees of 128 threads (points of 256 bytes in shared memory).
struct G1 {
  using Aff = g1_aff_t;
  using Pt = g1_xyzz_t;
  using F = fq_t;
  static constexpr const char* kName = "g3h_msm";
  static constexpr uint32_t kTree = 256;
  static __device__ __forceinline__ Pt inf() { return xyzz_infinity(); }
  static __device__ __forceinline__ bool aff_inf(const Aff& a) { return aff_is_inf(a); }
  static __device__ __forceinline__ Aff neg(const Aff& a) { return aff_neg(a); }
  static __device__ __forceinline__ Pt madd(const Pt& acc, const Aff& a) { return xyzz_madd(acc, a); }
  static __device__ __forceinline__ Pt add(const Pt& a, const Pt& b) { return xyzz_add(a, b); }
  static __device__ __forceinline__ Pt add_nl(const Pt& a, const Pt& b) { return xyzz_add_nl(a, b); }
  static __device__ __forceinline__ Pt add_lat(const Pt& a, const Pt& b) { return xyzz_add_lat(a, b); }
  static __device__ __forceinline__ Pt dbl_coop(const Pt& a) { return xyzz_dbl_coop(a); }
  static __device__ __forceinline__ Pt add_coop(const Pt& a, const Pt& b) { return xyzz_add_coop(a, b); }
  // the one-warp trees' levels of at most this many additions go to coop_level (1 and 2
  // measured best: parts and last sum 111 -> 102 us)
  static constexpr uint32_t kCoopLevels = 2;
  static __device__ __forceinline__ void jacobian(const Pt& p, F* out) {
    xyzz_to_jacobian_t<FqTail>(p, out[0], out[1], out[2]);
  }
  static __device__ __forceinline__ bool canonical(const Aff& a) {
    return fq_is_canonical(a.x) && fq_is_canonical(a.y);
  }
  static __device__ __forceinline__ bool on_curve(const Aff& a) { return aff_on_curve(a); }
  static __device__ __forceinline__ Aff zero_aff() { return {fq_zero(), fq_zero()}; }
  static __device__ __forceinline__ Pt from_aff(const Aff& a) { return xyzz_from_aff(a); }
  static __device__ __forceinline__ Pt dbl(const Pt& p) { return xyzz_dbl(p); }
  static __device__ __forceinline__ Aff to_aff(const Pt& p) { return xyzz_to_aff(p); }
};

struct G2 {
  using Aff = g2_aff_t;
  using Pt = g2_xyzz_t;
  using F = fq2_t;
  static constexpr const char* kName = "g3h_msm_g2";
  static constexpr uint32_t kTree = 128;
  static __device__ __forceinline__ Pt inf() { return g2_infinity(); }
  static __device__ __forceinline__ bool aff_inf(const Aff& a) { return g2_aff_is_inf(a); }
  static __device__ __forceinline__ Aff neg(const Aff& a) { return g2_aff_neg(a); }
  static __device__ __forceinline__ Pt madd(const Pt& acc, const Aff& a) { return g2_madd_t<Fq2Call>(acc, a); }
  static __device__ __forceinline__ Pt add(const Pt& a, const Pt& b) { return g2_add_nl(a, b); }
  static __device__ __forceinline__ Pt add_nl(const Pt& a, const Pt& b) { return g2_add_nl(a, b); }
  static __device__ __forceinline__ Pt add_lat(const Pt& a, const Pt& b) { return g2_add_nl(a, b); }
  static __device__ __forceinline__ Pt dbl_coop(const Pt& a) { return g2_dbl_coop(a); }
  static constexpr uint32_t kCoopLevels = 0;
  static __device__ __forceinline__ void jacobian(const Pt& p, F* out) { g2_to_jacobian_t<Fq2Call>(p, out); }
  static __device__ __forceinline__ bool canonical(const Aff& a) {
    return fq2_is_canonical(a.x) && fq2_is_canonical(a.y);
  }
  static __device__ __forceinline__ bool on_curve(const Aff& a) { return g2_aff_on_curve(a); }
  static __device__ __forceinline__ Aff zero_aff() { return {fq2_zero(), fq2_zero()}; }
  static __device__ __forceinline__ Pt from_aff(const Aff& a) { return g2_from_aff(a); }
  static __device__ __forceinline__ Pt dbl(const Pt& p) { return g2_dbl_t<Fq2Call>(p); }
  static __device__ __forceinline__ Aff to_aff(const Pt& p) { return g2_to_aff(p); }
};

// Signed 16-bit digit w of the scalar s (eight 32-bit limbs), given the carry out of
// window w - 1; updates the carry.
__device__ __forceinline__ int msm_digit(const uint32_t* s, uint32_t w, uint32_t& carry) {
  const uint32_t v = ((s[w >> 1] >> ((w & 1u) * 16u)) & 0xffffu) + carry;
  if (v > 0x8000u) {
    carry = 1u;
    return (int)v - 0x10000;
  }
  carry = 0u;
  return (int)v;
}

// Scalars equal to 1 (half of a typical witness) would all be one entry of bucket 1 and
// make one bucket's run as long as the rest together (MSM_CU, "scalars 0 and 1 never reach
// a bucket"); they are summed apart, by k_msm_ones. Scalars 0 give no entries anyway.
__device__ __forceinline__ bool msm_is_one(const uint32_t* s) {
  return s[0] == 1u && (s[1] | s[2] | s[3] | s[4] | s[5] | s[6] | s[7]) == 0u;
}

__device__ __forceinline__ void msm_load_scalar(const fr_t* scalars, uint32_t i, uint32_t* s,
                                                uint32_t check, uint32_t* err) {
  const fr_t x = fr_load(scalars + i);
  if (check && !fr_is_canonical(x)) atomicOr(err, 1u);
#pragma unroll
  for (int k = 0; k < 8; k++) s[k] = x.v[k];
}

// Prepare: table[16 i + w] = 2^(16 w) P_i, affine, canonical; a base at infinity (0, 0)
// gives 16 points at infinity. Checks that each base is canonical and on the curve.
// Launch: ceil(n / 128) blocks of 128.
template <class G>
__global__ void __launch_bounds__(128) k_msm_precompute(const typename G::Aff* bases, uint32_t n,
                                                        typename G::Aff* table, uint32_t* err) {
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  typename G::Aff b = bases[i];
  typename G::Aff* out = table + (size_t)i * kMsmWindows;
  if (G::aff_inf(b)) {
    for (uint32_t w = 0; w < kMsmWindows; w++) out[w] = b;
    return;
  }
  if (!G::canonical(b)) {
    atomicOr(err, 1u);
    b = G::zero_aff();
    for (uint32_t w = 0; w < kMsmWindows; w++) out[w] = b;
    return;
  }
  if (!G::on_curve(b)) atomicOr(err, kMsmErrPoint);
  out[0] = b;
  typename G::Pt p = G::from_aff(b);
  for (uint32_t w = 1; w < kMsmWindows; w++) {
    for (int d = 0; d < 16; d++) p = G::dbl(p);
    out[w] = G::to_aff(p);
  }
}

// Steps 1-3 sort the entries by bucket in blocks: sort block b owns the scalars
// [b C, min(b C + C, n)) (C = ceil(n / B), B sort blocks of kMsmSortThreads threads, one per
// SM: a block keeps a counter per bucket, 128 KiB, in shared memory), so no entry needs an
// atomic in global memory. The order of the entries inside a bucket's run is arbitrary
// (the sum commutes).
constexpr uint32_t kMsmSortThreads = 1024;
constexpr uint32_t kMsmSortSmem = kMsmBuckets * sizeof(uint32_t);

__device__ __forceinline__ uint32_t msm_sort_end(uint32_t n, uint32_t chunk) {
  return (uint32_t)min((uint64_t)n, (uint64_t)(blockIdx.x + 1u) * chunk);
}

// Step 1: block_counts[b][j] = entries of sort block b in bucket j + 1. Launch: grid B,
// kMsmSortThreads threads, kMsmSortSmem bytes of dynamic shared memory.
__global__ void __launch_bounds__(kMsmSortThreads) k_msm_count(const fr_t* scalars, uint32_t n,
                                                               uint32_t chunk,
                                                               uint32_t* block_counts,
                                                               uint32_t check, uint32_t* err) {
  extern __shared__ uint32_t hist[];
  for (uint32_t j = threadIdx.x; j < kMsmBuckets; j += blockDim.x) hist[j] = 0u;
  __syncthreads();
  const uint32_t end = msm_sort_end(n, chunk);
  for (uint32_t i = blockIdx.x * chunk + threadIdx.x; i < end; i += blockDim.x) {
    uint32_t s[8];
    msm_load_scalar(scalars, i, s, check, err);
    if (msm_is_one(s)) continue;  // summed by k_msm_ones
    uint32_t carry = 0;
#pragma unroll
    for (uint32_t w = 0; w < kMsmWindows; w++) {
      const int d = msm_digit(s, w, carry);
      if (d != 0) atomicAdd(hist + (uint32_t)(d < 0 ? -d : d) - 1u, 1u);
    }
  }
  __syncthreads();
  uint4* out = reinterpret_cast<uint4*>(block_counts + (size_t)blockIdx.x * kMsmBuckets);
  const uint4* h4 = reinterpret_cast<const uint4*>(hist);
  for (uint32_t j = threadIdx.x; j < kMsmBuckets / 4; j += blockDim.x) out[j] = h4[j];
}

// Step 1b: per bucket j, block_counts[b][j] becomes the entries of blocks before b (an
// exclusive prefix over the sort blocks, in place) and counts[j] the total. A block takes
// 32 buckets (the lanes) and splits the sort blocks into 8 ranges (the warps).
// Launch: kMsmBuckets / 32 blocks of 256.
__global__ void __launch_bounds__(256) k_msm_count_cols(uint32_t* block_counts, uint32_t blocks,
                                                        uint32_t* counts) {
  __shared__ uint32_t part[8][32];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t j = blockIdx.x * 32u + lane;
  const uint32_t per = (blocks + 7u) / 8u;
  const uint32_t b0 = min(blocks, warp * per), b1 = min(blocks, b0 + per);
  uint32_t sum = 0;
#pragma unroll 8
  for (uint32_t b = b0; b < b1; b++) sum += block_counts[(size_t)b * kMsmBuckets + j];
  part[warp][lane] = sum;
  __syncthreads();
  uint32_t run = 0;
  for (uint32_t w = 0; w < warp; w++) run += part[w][lane];
  if (warp == 7) counts[j] = run + sum;
#pragma unroll 8
  for (uint32_t b = b0; b < b1; b++) {
    uint32_t* p = block_counts + (size_t)b * kMsmBuckets + j;
    const uint32_t c = *p;
    *p = run;
    run += c;
  }
}

// Step 2: offsets[j] = sum of counts[0 .. j), offsets[kMsmBuckets] = total.
// Warp w scans buckets [1024 w, 1024 w + 1024) as 32 rows of 32 (coalesced loads and
// stores), then the 32 warp totals are scanned. Launch: one block of 1024 threads.
__global__ void __launch_bounds__(1024) k_msm_scan(const uint32_t* counts, uint32_t* offsets) {
  constexpr uint32_t rows = kMsmBuckets / 1024;  // per warp: rows of 32 buckets
  __shared__ uint32_t warp_tot[32];
  const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
  const uint32_t base = warp * 1024u;
  uint32_t v[rows];
#pragma unroll
  for (uint32_t k = 0; k < rows; k++) v[k] = counts[base + k * 32u + lane];
  uint32_t run = 0;  // this warp's total before row k
#pragma unroll
  for (uint32_t k = 0; k < rows; k++) {
    uint32_t inc = v[k];
#pragma unroll
    for (uint32_t d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += o;
    }
    const uint32_t row_total = __shfl_sync(0xffffffffu, inc, 31);
    v[k] = run + inc - v[k];  // exclusive prefix within the warp's segment
    run += row_total;
  }
  if (lane == 0) warp_tot[warp] = run;
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = warp_tot[lane];
    uint32_t inc = t;
#pragma unroll
    for (uint32_t d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, inc, d);
      if (lane >= d) inc += o;
    }
    warp_tot[lane] = inc - t;  // exclusive over the warps
    if (lane == 31) offsets[kMsmBuckets] = inc;
  }
  __syncthreads();
  const uint32_t off = warp_tot[warp];
#pragma unroll
  for (uint32_t k = 0; k < rows; k++) {
    offsets[base + k * 32u + lane] = off + v[k];
  }
}

// Step 3: each (i, w) entry, as (16 i + w) << 1 | sign, to its place in its bucket's run:
// sort block b's cursor for bucket j starts at offsets[j] + block_counts[b][j] (the
// prefix of step 1b). Launch: as k_msm_count, with the same grid and chunk.
__global__ void __launch_bounds__(kMsmSortThreads) k_msm_scatter(const fr_t* scalars, uint32_t n,
                                                                 uint32_t chunk,
                                                                 const uint32_t* offsets,
                                                                 const uint32_t* block_counts,
                                                                 uint32_t* entries) {
  extern __shared__ uint32_t cur[];
  const uint32_t* pre = block_counts + (size_t)blockIdx.x * kMsmBuckets;
  for (uint32_t j = threadIdx.x; j < kMsmBuckets; j += blockDim.x) cur[j] = offsets[j] + pre[j];
  __syncthreads();
  const uint32_t end = msm_sort_end(n, chunk);
  for (uint32_t i = blockIdx.x * chunk + threadIdx.x; i < end; i += blockDim.x) {
    uint32_t s[8];
    msm_load_scalar(scalars, i, s, 0u, nullptr);
    if (msm_is_one(s)) continue;
    uint32_t carry = 0;
#pragma unroll
    for (uint32_t w = 0; w < kMsmWindows; w++) {
      const int d = msm_digit(s, w, carry);
      if (d == 0) continue;
      const uint32_t slot = atomicAdd(cur + (uint32_t)(d < 0 ? -d : d) - 1u, 1u);
      entries[slot] = ((i * kMsmWindows + w) << 1) | (d < 0 ? 1u : 0u);
    }
  }
}

// Slice length: the entries present (offsets[kMsmBuckets], known only here) spread over the
// n_slices threads launched for the most there can be, at least kMsmMinSlice per thread (a
// run cut into more slices costs its bucket more additions at the merge). The merge
// computes the same length.
constexpr uint32_t kMsmMinSlice = 16;

__device__ __forceinline__ uint32_t msm_slice_len(uint32_t total, uint32_t n_slices) {
  return max(kMsmMinSlice, (total + n_slices - 1u) / n_slices);
}

// Step 4: slice k = entries [k L, min(k L + L, total)). Launch: ceil(n_slices / T)
// blocks of T (256 for G1, 128 for G2); slices past the total exit.
template <class G>
__global__ void __launch_bounds__(G::kTree) k_msm_accumulate(
    const uint32_t* entries, const uint32_t* offsets, const typename G::Aff* table,
    typename G::Pt* buckets, typename G::Pt* head, typename G::Pt* tail, uint32_t n_slices) {
  using Pt = typename G::Pt;
  const uint32_t k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n_slices) return;
  const uint32_t total = offsets[kMsmBuckets];
  const uint32_t slice = msm_slice_len(total, n_slices);
  const uint32_t lo = k * slice;
  if (lo >= total) return;
  const uint32_t hi = min(lo + slice, total);
  // the bucket whose run holds entry lo: offsets[b] <= lo < offsets[b + 1]
  uint32_t a = 0, z = kMsmBuckets;
  while (z - a > 1u) {
    const uint32_t m = (a + z) >> 1;
    if (offsets[m] <= lo) a = m; else z = m;
  }
  uint32_t b = a;
  uint32_t run_end = offsets[b + 1];
  Pt acc = G::inf();
  auto emit = [&]() {
    if (offsets[b] < lo) head[k] = acc;
    else if (run_end > hi) tail[k] = acc;
    else buckets[b] = acc;
  };
  for (uint32_t i = lo; i < hi; i++) {
    if (i == run_end) {
      emit();
      acc = G::inf();
      do {
        b++;
        run_end = offsets[b + 1];
      } while (run_end <= i);
    }
    const uint32_t e = entries[i];
    typename G::Aff p = table[e >> 1];
    if (G::aff_inf(p)) continue;
    if (e & 1u) p = G::neg(p);
    acc = G::madd(acc, p);
  }
  emit();
}

// Step 5: one thread per bucket. A bucket with no entries is set to infinity; a run cut by
// slice boundaries is the tail part of its first slice plus the head parts of the rest.
// A run over more than kMsmMergeSerial slices (a value repeated in many scalars puts all
// its digits in one bucket) is left to k_msm_merge_long: its index goes to long_list.
// Launch: kMsmBuckets / 128 blocks of 128; long_list[0] (the count) zero beforehand.
constexpr uint32_t kMsmMergeSerial = 16;

template <class G>
__global__ void __launch_bounds__(128) k_msm_merge(const uint32_t* offsets, typename G::Pt* buckets,
                                                   const typename G::Pt* head,
                                                   const typename G::Pt* tail, uint32_t n_slices,
                                                   uint32_t* long_list) {
  const uint32_t j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= kMsmBuckets) return;
  const uint32_t slice = msm_slice_len(offsets[kMsmBuckets], n_slices);
  const uint32_t s = offsets[j], e = offsets[j + 1];
  if (s == e) {
    buckets[j] = G::inf();
    return;
  }
  const uint32_t k_lo = s / slice, k_hi = (e - 1u) / slice;
  if (k_lo == k_hi) return;
  if (k_hi - k_lo > kMsmMergeSerial) {
    long_list[1 + atomicAdd(long_list, 1u)] = j;
    return;
  }
  typename G::Pt acc = tail[k_lo];
  for (uint32_t k = k_lo + 1; k <= k_hi; k++) acc = G::add(acc, head[k]);
  buckets[j] = acc;
}

// Step 5 for the long runs: one block per listed bucket (grid-stride over the list), its
// threads sum the head parts by strides, a tree in shared memory adds them and the first
// slice's tail part. Launch: any grid of G::kTree threads.
template <class G>
__global__ void __launch_bounds__(G::kTree) k_msm_merge_long(const uint32_t* offsets,
                                                             typename G::Pt* buckets,
                                                             const typename G::Pt* head,
                                                             const typename G::Pt* tail,
                                                             uint32_t n_slices,
                                                             const uint32_t* long_list) {
  __shared__ typename G::Pt sm[G::kTree];
  const uint32_t tid = threadIdx.x, count = long_list[0];
  const uint32_t slice = msm_slice_len(offsets[kMsmBuckets], n_slices);
  for (uint32_t d = blockIdx.x; d < count; d += gridDim.x) {
    const uint32_t j = long_list[1 + d];
    const uint32_t k_lo = offsets[j] / slice, k_hi = (offsets[j + 1] - 1u) / slice;
    typename G::Pt acc = tid == 0 ? tail[k_lo] : G::inf();
    for (uint32_t k = k_lo + 1 + tid; k <= k_hi; k += blockDim.x) acc = G::add_nl(acc, head[k]);
    sm[tid] = acc;
    __syncthreads();
    for (uint32_t w = G::kTree / 2; w > 0; w >>= 1) {
      if (tid < w) sm[tid] = G::add_nl(sm[tid], sm[tid + w]);
      __syncthreads();
    }
    if (tid == 0) buckets[j] = sm[0];
    __syncthreads();  // sm is reused by the next listed bucket
  }
}

// The weighted sum Q = sum_j (j + 1) B_j. With pairs t = (B_2t, B_2t+1), digits 2t + 1 and
// 2t + 2: U_t = B_2t + B_2t+1 and V_t = U_t + B_2t+1 = B_2t + 2 B_2t+1, so
//   Q = sum_t (V_t + 2t U_t) = sum_t V_t + sum_{b < 14} 2^(b+1) sum_{t : bit b of t} U_t.
// Part p < 14 is the sum over U_t with bit p of t set; part 14 is the sum of V. The point
// operations of steps 6-9 are a chain of some thirty dependent ones on few warps: their
// time is latency, and they use the out-of-line copies (add_nl, add_lat) and, where one
// warp works on one point, the warp-cooperative dbl_coop and add_coop.
constexpr uint32_t kMsmPairs = kMsmBuckets / 2;          // 16384 = 2^14
constexpr uint32_t kMsmPairBits = 14;
constexpr uint32_t kMsmSumParts = kMsmPairBits + 1;      // 15

// items per block in step 7 (two per thread) and chunks of the V part (the bit parts have
// half as many)
template <class G>
__host__ __device__ constexpr uint32_t msm_chunk() { return 2 * G::kTree; }
template <class G>
__host__ __device__ constexpr uint32_t msm_chunks() { return kMsmPairs / msm_chunk<G>(); }

// Step 6: U_t, V_t. Launch: kMsmPairs / 128 blocks of 128.
template <class G>
__global__ void __launch_bounds__(128) k_msm_pairs(const typename G::Pt* buckets,
                                                   typename G::Pt* U, typename G::Pt* V) {
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= kMsmPairs) return;
  const typename G::Pt hi = buckets[2 * t + 1];
  const typename G::Pt u = G::add_nl(buckets[2 * t], hi);
  U[t] = u;
  V[t] = G::add_nl(u, hi);
}

// Step 7: partial sums of the parts, chunk c of part p = blockIdx (c, p): 2 T items, two per
// thread, then a tree in shared memory. The bit parts have 8192 items: item i is t with
// bit p set, i.e. bit p inserted into i. Launch: grid (msm_chunks<G>(), kMsmSumParts) of
// T = G::kTree threads.
template <class G>
__global__ void __launch_bounds__(G::kTree) k_msm_part_chunks(const typename G::Pt* U,
                                                               const typename G::Pt* V,
                                                               typename G::Pt* partial) {
  using Pt = typename G::Pt;
  __shared__ Pt sm_pts[G::kTree];
  constexpr uint32_t chunk = msm_chunk<G>(), chunks = msm_chunks<G>();
  const uint32_t c = blockIdx.x, p = blockIdx.y, tid = threadIdx.x;
  const bool bit_part = p < kMsmPairBits;
  if (bit_part && c >= chunks / 2) return;  // whole block exits together
  Pt x[2];
#pragma unroll
  for (int k = 0; k < 2; k++) {
    const uint32_t i = c * chunk + 2 * tid + (uint32_t)k;
    if (bit_part) {
      const uint32_t t = ((i >> p) << (p + 1)) | (1u << p) | (i & ((1u << p) - 1u));
      x[k] = U[t];
    } else {
      x[k] = V[i];
    }
  }
  sm_pts[tid] = G::add_nl(x[0], x[1]);
  __syncthreads();
  for (uint32_t s = G::kTree / 2; s > 0; s >>= 1) {
    if (tid < s) sm_pts[tid] = G::add_nl(sm_pts[tid], sm_pts[tid + s]);
    __syncthreads();
  }
  if (tid == 0) partial[p * chunks + c] = sm_pts[0];
}

// Step 8: block p (one warp, a block per part so that each runs on an SM of its own) sums
// part p's chunks (lane by lane, then shuffles) and scales the sum: part p < 14 by
// 2^(p+1), p + 1 doublings. Launch: kMsmSumParts blocks of 32.
template <class G>
__global__ void __launch_bounds__(32) k_msm_parts(const typename G::Pt* partial, typename G::Pt* parts) {
  constexpr uint32_t chunks = msm_chunks<G>();
  const uint32_t lane = threadIdx.x, p = blockIdx.x;
  const uint32_t n_chunks = p < kMsmPairBits ? chunks / 2 : chunks;
  typename G::Pt acc = G::inf();
  for (uint32_t c = lane; c < n_chunks; c += 32) acc = G::add_lat(acc, partial[p * chunks + c]);
  for (uint32_t d = 16; d > 0; d >>= 1) {
    const typename G::Pt o = pt_shfl_down(acc, d);
    if constexpr (G::kCoopLevels > 0) {
      if (d <= G::kCoopLevels) {
        coop_level<G>(acc, o, d);
        continue;
      }
    }
    if (lane < d) acc = G::add_lat(acc, o);
  }
  // the doublings by the whole warp, on lane 0's sum (106 -> 72 us for G1; G2 multiexp
  // 1.75 -> 1.63 ms)
  if (p < kMsmPairBits) {
    acc = pt_shfl(acc, 0u);
    for (uint32_t k = 0; k <= p; k++) acc = G::dbl_coop(acc);
  }
  if (lane == 0) parts[p] = acc;
}

// The sum of the bases whose scalar is 1, beside the bucket path: each thread adds its
// share (grid-stride, mixed additions of the bases, which are the window-0 table entries),
// then a tree per block leaves one point per block in partial[blockIdx.x].
// Launch: any grid of G::kTree threads.
template <class G>
__global__ void __launch_bounds__(G::kTree) k_msm_ones(const fr_t* scalars, uint32_t n,
                                                       const typename G::Aff* table,
                                                       typename G::Pt* partial) {
  __shared__ typename G::Pt sm[G::kTree];
  const uint32_t stride = gridDim.x * blockDim.x, tid = threadIdx.x;
  typename G::Pt acc = G::inf();
  for (uint32_t i = blockIdx.x * blockDim.x + tid; i < n; i += stride) {
    const fr_t x = fr_load(scalars + i);
    if (!msm_is_one(x.v)) continue;
    const typename G::Aff p = table[(size_t)i * kMsmWindows];
    if (!G::aff_inf(p)) acc = G::madd(acc, p);
  }
  sm[tid] = acc;
  __syncthreads();
  for (uint32_t d = G::kTree / 2; d > 0; d >>= 1) {
    if (tid < d) sm[tid] = G::add_nl(sm[tid], sm[tid + d]);
    __syncthreads();
  }
  if (tid == 0) partial[blockIdx.x] = sm[0];
}

// The block sums of k_msm_ones (count of them) into one point, parts[kMsmSumParts].
// Launch: one block of G::kTree.
template <class G>
__global__ void __launch_bounds__(G::kTree) k_msm_ones_sum(const typename G::Pt* partial,
                                                           uint32_t count, typename G::Pt* parts) {
  __shared__ typename G::Pt sm[G::kTree];
  const uint32_t tid = threadIdx.x;
  typename G::Pt acc = G::inf();
  for (uint32_t i = tid; i < count; i += blockDim.x) acc = G::add_nl(acc, partial[i]);
  sm[tid] = acc;
  __syncthreads();
  for (uint32_t d = G::kTree / 2; d > 0; d >>= 1) {
    if (tid < d) sm[tid] = G::add_nl(sm[tid], sm[tid + d]);
    __syncthreads();
  }
  if (tid == 0) parts[kMsmSumParts] = sm[0];
}

// Step 9: Q = the sum of the 15 parts and the ones' sum (shuffles), written in Jacobian
// coordinates (X, Y, Z), canonical Montgomery, infinity as (0, 0, 0). Launch: one warp.
template <class G>
__global__ void __launch_bounds__(32) k_msm_final(const typename G::Pt* parts, typename G::F* out) {
  const uint32_t lane = threadIdx.x;
  typename G::Pt acc = lane <= kMsmSumParts ? parts[lane] : G::inf();
  for (uint32_t d = 8; d > 0; d >>= 1) {
    const typename G::Pt o = pt_shfl_down(acc, d);
    if constexpr (G::kCoopLevels > 0) {
      if (d <= G::kCoopLevels) {
        coop_level<G>(acc, o, d);
        continue;
      }
    }
    if (lane < d) acc = G::add_lat(acc, o);
  }
  if (lane == 0) G::jacobian(acc, out);
}

}  // namespace g3h
