// Gather, join, pointwise product, the small-domain path and the table builders.
#pragma once
#include "fr.cuh"
#include "ntt.cuh"

namespace g3h {

// ---------------------------------------------------------------------------------------
// Step 1, the sums of one matrix: thread i forms row i of A (or of B) against the
// witness; the two matrices are launched separately, on separate streams, and c = a * b
// is formed by the first inverse kernel of c at its load (SL_C_FROM_AB). Outputs
// canonical. Launch: ceil(n / 256) x (batch) blocks of 256; grid row blockIdx.y reads the
// witness at w + blockIdx.y * w_stride and writes out + blockIdx.y * out_stride.
//
// The kernel lasts as long as its slowest warp, and a row is a chain of dependent loads
// (column, then witness value and coefficient) per term, so the longest row (95 terms in
// the 2^18 key) would set the time alone. Rows of at most kGatherLaneTerms terms are
// summed by their own lane; longer rows are summed by the whole warp, lanes striding over
// the terms, then combined with a shuffle reduction. Sums are mod r in any order, so the
// outputs are the same canonical values. At its start each block streams its share of the
// witness and its rows' columns and coefficients into L2 (bulk prefetches), so that the
// row loops' later loads find them there (measured at 2^18, with the lane loop below:
// 0.2790 -> 0.2780 ms per H).
constexpr uint32_t kGatherLaneTerms = 8;

// acc + coefficient * witness value: nothing for 0, the coefficient for the Montgomery form
// of 1, else the product. (The multiply out of line, to keep its temporaries out of the row
// loops' registers, measured slower where a tenth of the witness values are neither 0 nor
// 1: batched 2^12 H 263 k -> 253 k H/s; it also took more registers, 58 vs 54.)
__device__ __forceinline__ fr_t gather_add(const fr_t& acc, const fr_t& wv, const fr_t& cv) {
  if (fr_is_zero(wv)) return acc;
  return fr_add(acc, fr_is_mont_one(wv) ? cv : fr_mul(cv, wv));
}

// Streams [p, p + bytes) into L2 (bulk prefetch: no registers, no wait). p and bytes are
// multiples of 16; callers keep the range inside one buffer.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  if (bytes)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ fr_t fr_shfl_xor(const fr_t& x, int lane_mask) {
  fr_t y;
#pragma unroll
  for (int j = 0; j < 8; j++) y.v[j] = __shfl_xor_sync(0xffffffffu, x.v[j], lane_mask);
  return y;
}

__global__ void __launch_bounds__(256) k_gather_rows(const uint32_t* __restrict__ rp,
                                                     const uint32_t* __restrict__ col,
                                                     const fr_t* __restrict__ val,
                                                     const fr_t* __restrict__ w,
                                                     uint32_t n_rows, uint32_t n,
                                                     uint32_t n_wires, fr_t* out,
                                                     uint32_t check, uint32_t* err,
                                                     size_t w_stride, size_t out_stride) {
  // No early return: every lane takes part in the warp-wide loop below.
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  w += (size_t)blockIdx.y * w_stride;
  out += (size_t)blockIdx.y * out_stride;
  if (threadIdx.x == 0) {
    // this block's share of the witness, 16-byte granules
    const uint32_t granules = n_wires * 2u, per = (granules + gridDim.x - 1u) / gridDim.x;
    const uint32_t g0 = blockIdx.x * per, g1 = min(granules, g0 + per);
    if (g0 < g1) l2_prefetch(reinterpret_cast<const uint4*>(w) + g0, (g1 - g0) * 16u);
  }
  if (threadIdx.x == 32u) {
    // the coefficients and columns of this block's rows (at most 2^20 terms' worth)
    const uint32_t r0 = blockIdx.x * blockDim.x;
    if (r0 < n_rows) {
      const uint32_t r1 = min(n_rows, r0 + blockDim.x);
      const uint32_t t0 = rp[r0], t1 = t0 + min(rp[r1] - t0, 1u << 20);
      l2_prefetch(val + t0, (t1 - t0) * 32u);
      const uint32_t c0 = t0 & ~3u, c1 = t1 & ~3u;
      l2_prefetch(col + c0, (c1 - c0) * 4u);
    }
  }
  const uint32_t lane = threadIdx.x & 31u;
  uint32_t kx = 0, ke = 0;
  if (i < n && i < n_rows) {
    kx = rp[i];
    ke = rp[i + 1];
  }
  const bool lane_row = ke - kx <= kGatherLaneTerms;
  fr_t acc = fr_zero();
  if (lane_row && kx < ke) {
    // One term per iteration; the next term's column is loaded while this term's witness
    // value and coefficient are in flight (measured at 2^18 against two terms per
    // iteration: 0.2803 -> 0.2790 ms per H). The coefficient's load is issued beside the
    // witness value's, not after the zero test: one dependent load less per term for the
    // bytes of the zero terms' coefficients (2^12 H 0.069 -> 0.064 ms).
    uint32_t c = col[kx];
    for (uint32_t k = kx; k < ke; k++) {
      const fr_t wv = fr_ldg(w + c);
      const fr_t cv = fr_ldg(val + k);
      if (k + 1u < ke) c = col[k + 1u];
      if (check) check_canonical(wv, err);
      acc = gather_add(acc, wv, cv);
    }
  }
  // The warp's long rows, one at a time.
  uint32_t longs = __ballot_sync(0xffffffffu, !lane_row);
  while (longs) {
    const int src = __ffs(longs) - 1;
    longs &= longs - 1u;
    const uint32_t rb = __shfl_sync(0xffffffffu, kx, src);
    const uint32_t re = __shfl_sync(0xffffffffu, ke, src);
    fr_t part = fr_zero();
    for (uint32_t k = rb + lane; k < re; k += 32u) {
      const fr_t wv = fr_ldg(w + col[k]);
      const fr_t cv = fr_ldg(val + k);
      if (check) check_canonical(wv, err);
      part = gather_add(part, wv, cv);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part = fr_add(part, fr_shfl_xor(part, off));
    if ((int)lane == src) acc = part;
  }
  if (i < n) fr_store(out + i, fr_canon(acc));
}

// Step 1 alone (GATHER_CU, g16_gather_abc; gather_row in ntt.cuh). Outputs are canonical.
// Launch: ceil(n / 256) blocks of 256.
__global__ void __launch_bounds__(256) k_gather(const uint32_t* __restrict__ rpa,
                                                const uint32_t* __restrict__ cola,
                                                const fr_t* __restrict__ vala,
                                                const uint32_t* __restrict__ rpb,
                                                const uint32_t* __restrict__ colb,
                                                const fr_t* __restrict__ valb,
                                                const fr_t* __restrict__ w, uint32_t n_rows_a,
                                                uint32_t n_rows_b, uint32_t n, fr_t* a_out,
                                                fr_t* b_out, fr_t* c_out, uint32_t check,
                                                uint32_t* err) {
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const fr_t a = i < n_rows_a ? gather_row(rpa, cola, vala, w, i, check, err) : fr_zero();
  const fr_t b = i < n_rows_b ? gather_row(rpb, colb, valb, w, i, check, err) : fr_zero();
  fr_store(a_out + i, a);
  fr_store(b_out + i, b);
  fr_store(c_out + i, gather_c(a, b));
}

// Step 5 alone (POINTWISE_CU, g16_h_join): h = a*b - c in both encodings.
// Launch: ceil(n / 256) x (batch) blocks of 256; grid row blockIdx.y reads a, b, c +
// blockIdx.y * in_stride and writes h_mont, h_std + blockIdx.y * h_stride.
__global__ void __launch_bounds__(256) k_join(const fr_t* a, const fr_t* b, const fr_t* c,
                                              fr_t* h_mont, fr_t* h_std, size_t n,
                                              uint32_t check, uint32_t* err,
                                              size_t in_stride, size_t h_stride) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const size_t zi = (size_t)blockIdx.y * in_stride, zh = (size_t)blockIdx.y * h_stride;
  a += zi;
  b += zi;
  c += zi;
  h_mont += zh;
  h_std += zh;
  const fr_t x = fr_load(a + i), y = fr_load(b + i), z = fr_load(c + i);
  if (check) {
    check_canonical(x, err);
    check_canonical(y, err);
    check_canonical(z, err);
  }
  const fr_t h = fr_canon(fr_sub(fr_mul(x, y), z));
  fr_store(h_mont + i, h);
  fr_store(h_std + i, fr_from_mont(h));
}

// Step 5 in two parts on the single-problem path. k_join_product: p = a * b (Montgomery
// product, canonical), written over a (each thread reads its element of a before it
// writes it). k_join_reduce: h = p - c in Montgomery form and from_mont(h), the same
// values as k_join. Launch: ceil(n / 256) blocks of 256.
__global__ void __launch_bounds__(256) k_join_product(fr_t* a, const fr_t* b, size_t n) {
  wait_prior_grid();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  fr_store(a + i, fr_canon(fr_mul(fr_load(a + i), fr_load(b + i))));
}

__global__ void __launch_bounds__(256) k_join_reduce(const fr_t* p, const fr_t* c, fr_t* h_mont,
                                                     fr_t* h_std, size_t n) {
  wait_prior_grid();
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const fr_t h = fr_canon(fr_sub(fr_load(p + i), fr_load(c + i)));
  fr_store(h_mont + i, h);
  fr_store(h_std + i, fr_from_mont(h));
}

// out = a * b (Montgomery product), canonical. Launch: ceil(n / 256) blocks of 256.
__global__ void __launch_bounds__(256) k_mul(const fr_t* a, const fr_t* b, fr_t* out, size_t n,
                                             uint32_t check, uint32_t* err) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const fr_t x = fr_load(a + i), y = fr_load(b + i);
  if (check) {
    check_canonical(x, err);
    check_canonical(y, err);
  }
  fr_store(out + i, fr_canon(fr_mul(x, y)));
}

// Montgomery to standard form, elementwise (POINTWISE_CU, g16_mont_to_std: the witness is
// uploaded once in Montgomery form for the gather and its standard-form copy, which the
// MSM digit decomposition reads, is made on the device). out may equal in. A canonical
// input gives a canonical output (REDC of a < r is < r). HBM-bound: 64 bytes per element
// against 136 IMAD. Launch: a grid-stride loop, any grid (a multiple of the SM count).
__global__ void __launch_bounds__(256) k_mont_to_std(const fr_t* in, fr_t* out, size_t n,
                                                     uint32_t check, uint32_t* err) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const fr_t x = fr_load(in + i);
    if (check) check_canonical(x, err);
    fr_store(out + i, fr_from_mont(x));
  }
}

// ---------------------------------------------------------------------------------------
// Domains of at most 2^5 points: one block of 32 threads, every pass a loop over
// butterflies through shared memory (the plain radix-2 schedule; such domains are too
// small to fill slices of eight elements per thread).
constexpr uint32_t kSmallMaxLog = 5;

// Steps 2-5 on a, b, c: decimation-in-frequency inverse (tw_inv), shift by
// shift_br[p] = g^brev(p) / n, decimation-in-time forward (tw_fwd), join.
// Launch: 1 block of 32 threads.
__global__ void __launch_bounds__(32) k_small_quotient(const fr_t* a, const fr_t* b,
                                                       const fr_t* c, const fr_const_t* tw_inv,
                                                       const fr_const_t* tw_fwd,
                                                       const fr_const_t* shift_br, fr_t* h_mont,
                                                       fr_t* h_std, uint32_t k,
                                                       uint32_t check, uint32_t* err) {
  __shared__ fr_t s[3][1u << kSmallMaxLog];
  const uint32_t tid = threadIdx.x, n = 1u << k;
  const fr_t* in[3] = {a, b, c};
  for (uint32_t v = 0; v < 3; v++) {
    for (uint32_t i = tid; i < n; i += blockDim.x) {
      s[v][i] = fr_load(in[v] + i);
      if (check) check_canonical(s[v][i], err);
    }
  }
  __syncthreads();
  for (int bb = (int)k - 1; bb >= 0; bb--) {
    const uint32_t bit = (uint32_t)bb;
    for (uint32_t v = 0; v < 3; v++) {
      for (uint32_t f = tid; f < n / 2; f += blockDim.x) {
        const uint32_t j = f & ((1u << bit) - 1u);
        const uint32_t lo = ((f >> bit) << (bit + 1u)) | j, hi = lo + (1u << bit);
        const fr_t u = s[v][lo], w = s[v][hi];
        s[v][lo] = fr_add(u, w);
        s[v][hi] = fr_mul_c(fr_sub(u, w), tw_inv[j << (k - 1u - bit)]);
      }
    }
    __syncthreads();
  }
  for (uint32_t v = 0; v < 3; v++)
    for (uint32_t i = tid; i < n; i += blockDim.x) s[v][i] = fr_mul_c(s[v][i], shift_br[i]);
  __syncthreads();
  for (uint32_t bit = 0; bit < k; bit++) {
    for (uint32_t v = 0; v < 3; v++) {
      for (uint32_t f = tid; f < n / 2; f += blockDim.x) {
        const uint32_t j = f & ((1u << bit) - 1u);
        const uint32_t lo = ((f >> bit) << (bit + 1u)) | j, hi = lo + (1u << bit);
        const fr_t u = s[v][lo];
        const fr_t w = fr_mul_c(s[v][hi], tw_fwd[j << (k - 1u - bit)]);
        s[v][lo] = fr_add(u, w);
        s[v][hi] = fr_sub(u, w);
      }
    }
    __syncthreads();
  }
  for (uint32_t i = tid; i < n; i += blockDim.x) {
    const fr_t h = fr_canon(fr_sub(fr_mul(s[0][i], s[1][i]), s[2][i]));
    fr_store(h_mont + i, h);
    fr_store(h_std + i, fr_from_mont(h));
  }
}

// A natural-order transform of one small vector in place: position p loads
// data[brev(p)] (times scale_load[p] if given: a table in bit-reversed order),
// decimation-in-time passes with tw, stores times scale_store[p] if given, else times
// kscale if given.
// Launch: 1 block of 32 threads.
__global__ void __launch_bounds__(32) k_small_ntt(fr_t* data, const fr_const_t* tw,
                                                  const fr_const_t* scale_load,
                                                  const fr_const_t* scale_store, fr_const_t kscale,
                                                  uint32_t use_kscale, uint32_t k,
                                                  uint32_t check, uint32_t* err) {
  __shared__ fr_t s[1u << kSmallMaxLog];
  const uint32_t tid = threadIdx.x, n = 1u << k;
  for (uint32_t i = tid; i < n; i += blockDim.x) {
    const uint32_t j = bitrev(i, k);
    fr_t x = fr_load(data + j);
    if (check) check_canonical(x, err);
    if (scale_load) x = fr_mul_c(x, scale_load[i]);
    s[i] = x;
  }
  __syncthreads();
  for (uint32_t bit = 0; bit < k; bit++) {
    for (uint32_t f = tid; f < n / 2; f += blockDim.x) {
      const uint32_t j = f & ((1u << bit) - 1u);
      const uint32_t lo = ((f >> bit) << (bit + 1u)) | j, hi = lo + (1u << bit);
      const fr_t u = s[lo];
      const fr_t w = fr_mul_c(s[hi], tw[j << (k - 1u - bit)]);
      s[lo] = fr_add(u, w);
      s[hi] = fr_sub(u, w);
    }
    __syncthreads();
  }
  for (uint32_t i = tid; i < n; i += blockDim.x) {
    fr_t x = s[i];
    if (scale_store) x = fr_mul_c(x, scale_store[i]);
    else if (use_kscale) x = fr_mul_c(x, kscale);
    fr_store(data + i, fr_canon(x));
  }
}

// ---------------------------------------------------------------------------------------
// Tables, built on the device at prepare time and kept resident.

// 2^512 mod r (to enter Montgomery form: x * R^2 * R^-1 = x * R).
__constant__ uint32_t kR2[8] = {0xae216da7u, 0x1bb8e645u, 0xe35c59e3u, 0x53fe3ab1u,
                                0x53bb8085u, 0x8c49833du, 0x7f4e44a5u, 0x0216d0b1u};
// r - 2 (Fermat inversion exponent) and (r - 1) / 2^28.
__constant__ uint32_t kRm2[8] = {0xefffffffu, 0x43e1f593u, 0x79b97091u, 0x2833e848u,
                                 0x8181585du, 0xb85045b6u, 0xe131a029u, 0x30644e72u};
__constant__ uint32_t kOddPart[8] = {0x3e1f593fu, 0x9b970914u, 0x833e8487u, 0x181585d2u,
                                     0x85045b68u, 0x131a029bu, 0x0644e72eu, 0x00000003u};

__device__ __forceinline__ fr_t fr_one_mont() {
  fr_t x = fr_zero();
  x.v[0] = 1u;
  fr_t r2;
#pragma unroll
  for (int i = 0; i < 8; i++) r2.v[i] = kR2[i];
  return fr_canon(fr_mul(x, r2));
}

__device__ __forceinline__ fr_t fr_small_mont(uint32_t v) {
  fr_t x = fr_zero();
  x.v[0] = v;
  fr_t r2;
#pragma unroll
  for (int i = 0; i < 8; i++) r2.v[i] = kR2[i];
  return fr_canon(fr_mul(x, r2));
}

// base^e for a 256-bit exponent given as 8 limbs; Montgomery in and out, canonical.
__device__ fr_t fr_pow_limbs(const fr_t& base, const uint32_t* e) {
  fr_t acc = fr_one_mont();
  for (int i = 255; i >= 0; i--) {
    acc = fr_mul(acc, acc);
    if ((e[i >> 5] >> (i & 31)) & 1u) acc = fr_mul(acc, base);
  }
  return fr_canon(acc);
}

__device__ fr_t fr_pow_u32(const fr_t& base, uint32_t e) {
  fr_t acc = fr_one_mont();
  for (int i = 31; i >= 0; i--) {
    acc = fr_mul(acc, acc);
    if ((e >> i) & 1u) acc = fr_mul(acc, base);
  }
  return fr_canon(acc);
}

// Domain constants for 2^k, Montgomery form: out[0] = omega, out[1] = omega^-1, out[2] = g,
// out[3] = g^-1, out[4] = n^-1, out[5] = 1. The 2^28-th root of unity is 5^((r-1)/2^28)
// (5 is a quadratic non-residue mod r); g = that root to the 2^(27-k), omega = g^2.
__device__ void domain_constants(fr_t* out, uint32_t k) {
  fr_t w = fr_pow_limbs(fr_small_mont(5u), kOddPart);
  for (uint32_t i = 0; i < 27u - k; i++) w = fr_canon(fr_mul(w, w));
  const fr_t g = w;
  const fr_t omega = fr_canon(fr_mul(g, g));
  out[0] = omega;
  out[1] = fr_pow_limbs(omega, kRm2);
  out[2] = g;
  out[3] = fr_pow_limbs(g, kRm2);
  out[4] = fr_pow_limbs(fr_small_mont(1u << k), kRm2);
  out[5] = fr_one_mont();
}

// Launch: 1 block of 1 thread.
__global__ void k_domain(fr_t* out, uint32_t k) { domain_constants(out, k); }

// The constant scale * base^e in the (w, w') form of the constant multiply; base and scale
// are indices into the domain constants (scale < 0: none). The power is formed in
// Montgomery form x = w*R mod r, then w = from_mont(x) and w' = x * (-r^-1) mod 2^256.
__device__ __forceinline__ fr_const_t pow_table_entry(const fr_t* consts, int base_idx,
                                                      int scale_idx, uint32_t e) {
  fr_t x = fr_pow_u32(consts[base_idx], e);
  if (scale_idx >= 0) x = fr_canon(fr_mul(x, consts[scale_idx]));
  const uint32_t ninv[8] = G3H_NINV256;
  fr_const_t c;
  c.w = fr_from_mont(x);
  mul_low256(x.v, ninv, c.wp.v);
  return c;
}

// tab[i] = pow_table_entry(base^(bit-reversed i if brev_bits else i)), i < count.
// Launch: ceil(count/256) x 256.
__global__ void k_pow_table(fr_const_t* tab, size_t count, const fr_t* consts, int base_idx,
                            int scale_idx, uint32_t brev_bits) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const uint32_t e = brev_bits ? bitrev((uint32_t)i, brev_bits) : (uint32_t)i;
  tab[i] = pow_table_entry(consts, base_idx, scale_idx, e);
}

}  // namespace g3h
