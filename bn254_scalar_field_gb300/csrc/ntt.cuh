// Radix-2 NTT passes over slices of a vector, staged through shared memory.
//
// What is computed is the transform pair of the "snarkrs_gpu_kernels" NTT_CU page: the
// inverse DFT of the evaluation vectors, the coset shift x_j *= g^j, the forward DFT. The
// pages' own CUDA kernels run decimation in time on a bit-reversed load, two launches per
// transform. Here the arithmetic is exact, so any schedule that computes the same DFT
// gives identical bits, and the schedule is chosen for this GPU:
//
//  * The inverse is a decimation-in-frequency (Gentleman-Sande) transform: natural order
//    in, bit-reversed order out, pass on bit b pairs p and p + 2^b and multiplies the
//    difference by omega^-(j * n / 2^(b+1)), j = p mod 2^b.
//  * The forward is a decimation-in-time (Cooley-Tukey) transform on that bit-reversed
//    vector: bit-reversed in, natural out, the pass on bit b multiplies the upper input by
//    omega^(j * n / 2^(b+1)). No bit-reversal permutation is ever materialised.
//  * Between the two, position p holds the coefficient of index brev(p), so the coset
//    shift multiplies it by g^brev(p); the 1/n of the inverse is folded into the same
//    table (shift[p] = g^brev(p) / n), which is exact because the maps are linear.
//  * A pass on bit b only mixes elements that differ in bit b, so passes over a range of
//    bits [c0, c0 + kk) can run on the "slice" of 2^kk elements that agree on all other
//    bits (the six-step decomposition the NTT_CU page describes as (s0, k) batching).
//    The lowest slice (c0 = 0) is contiguous, and the inverse's last passes and the
//    forward's first passes both live there, so one kernel runs them back to back with
//    the shift in between (k_ntt_mid).
//
// Every multiplication here is by a table constant (twiddle, shift, scale), so it uses
// the constant multiply of fr.cuh (Shoup's method, tables of (w, w') pairs).
//
// Inside a block every pass is a loop over butterflies, one butterfly per iteration, with
// the slice in shared memory and a barrier between passes. The 256-bit multiply is the
// cost that matters; keeping one copy of it per loop body keeps each kernel's hot code
// within the instruction cache and the register count low enough for 32 warps per SM,
// which the measured profile of an eight-element-per-thread register variant (half of all
// issue slots lost to instruction fetch, two warps per scheduler) showed to be the limit.
//
// Shared memory holds each 32-byte element as two 16-byte halves in two planes, with the
// 16-byte slot index swizzled (swz below) so that every access pattern of the passes
// falls on distinct bank groups.
#pragma once
#include "fr.cuh"

namespace g3h {

enum : uint32_t {
  SL_CHECK = 1u,        // check loaded inputs are canonical, report through *err
  SL_SCALE_TABLE = 2u,  // scale by scale_tab (see each kernel)
  SL_SCALE_CONST = 4u,  // scale by kscale
  SL_JOIN = 8u,         // k_ntt_dit: vectors 0, 1, 2 are a, b, c; write h = a*b - c
  SL_C_FROM_AB = 16u,   // k_ntt_dif: vector 2 (c) is not loaded but formed as
                        // src[0][i] * src[1][i] (the gather's C = A o B) at load
  SL_JOIN_LAST = 32u,   // k_ntt_dit: vectors 0, 1, 2 (grid.y) are a, b, c; the last of a
                        // slice's three blocks to finish writes h for that slice (one
                        // problem per launch: the counters are per slice)
};

struct SliceArgs {
  const fr_t* src[3];
  fr_t* dst[3];
  const fr_const_t* tw;         // twiddles of the passes (forward or inverse, n/2 entries)
  const fr_const_t* tw2;        // k_ntt_mid: forward twiddles for its decimation-in-time half
  const fr_const_t* scale_tab;  // per-kernel scale table (n entries)
  fr_t* h_mont;
  fr_t* h_std;
  uint32_t* err;
  fr_const_t kscale;
  uint32_t log_n;  // k: the vector has 2^k elements
  uint32_t kk;     // slice bits: a block owns 2^kk elements
  uint32_t c0;     // the slice's bits are [c0, c0 + kk) of the element index
  uint32_t mode;   // SL_* flags
  uint32_t* counters;  // SL_JOIN_LAST: one zeroed counter per slice, left zeroed
  uint32_t vbase;      // vector of grid row blockIdx.y is vbase + blockIdx.y
  uint32_t vfast;      // nonzero: the three vectors of a slice are adjacent blocks (slice
                       // blockIdx.x / 3, vector vbase + blockIdx.x % 3; grid.y = 1), so that
                       // they read the slice's twiddles and scales close together in time
  // Batches: grid layer blockIdx.z works on an independent problem whose vectors are at
  // src[v] + blockIdx.z * zs_src, dst[v] + blockIdx.z * zs_dst and h_mont / h_std +
  // blockIdx.z * zs_h (elements; all zero for a single problem)
  uint64_t zs_src, zs_dst, zs_h;
};

// 16-byte slot of element m's half: the low three bits (the bank group of a 16-byte
// access) are XORed with a fold of the higher bits, so that eight lanes at element
// strides 1, 2, 4, ..., 128 land on eight distinct bank groups.
__device__ __forceinline__ uint32_t swz(uint32_t m) {
  return m ^ (((m >> 3) ^ (m >> 6) ^ (m >> 9)) & 7u);
}

__device__ __forceinline__ void sm_put(uint4* sm, uint32_t half, uint32_t m, const fr_t& x) {
  const uint32_t s = swz(m);
  sm[s] = make_uint4(x.v[0], x.v[1], x.v[2], x.v[3]);
  sm[half + s] = make_uint4(x.v[4], x.v[5], x.v[6], x.v[7]);
}

__device__ __forceinline__ fr_t sm_get(const uint4* sm, uint32_t half, uint32_t m) {
  const uint32_t s = swz(m);
  const uint4 x = sm[s], y = sm[half + s];
  fr_t a;
  a.v[0] = x.x; a.v[1] = x.y; a.v[2] = x.z; a.v[3] = x.w;
  a.v[4] = y.x; a.v[5] = y.y; a.v[6] = y.z; a.v[7] = y.w;
  return a;
}

// In a launch made with programmatic stream serialization: waits until the previous kernel
// on the stream has completed and its writes are visible (the grid may have been launched
// while that kernel's last blocks ran); in any other launch it returns at once.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint32_t bitrev(uint32_t x, uint32_t bits) {
  return bits == 0u ? 0u : (__brev(x) >> (32u - bits));
}

__device__ __forceinline__ void check_canonical(const fr_t& x, uint32_t* err) {
  if (!fr_is_canonical(x)) atomicOr(err, 1u);
}

// ---------------------------------------------------------------------------------------
// Step 1 (GATHER_CU, g16_gather_abc): a_i = sum over CSR row i of A.val[k] * w[A.col[k]],
// b_i likewise, c_i = a_i * b_i; one thread per row, as on the page (rows are short,
// ragged and half empty).
//
// Most witness values of a circuit are 0 or 1 (bits, flags, the constant wire), so a term
// whose wire value is 0 contributes nothing and one whose value is the Montgomery form of
// 1 contributes its coefficient unchanged; only the remaining terms take a multiply, and
// c is only multiplied out when both a and b are non-zero. These are identities of the
// field, so the outputs are the same canonical values.
__device__ __forceinline__ fr_t gather_row(const uint32_t* __restrict__ rp,
                                           const uint32_t* __restrict__ col,
                                           const fr_t* __restrict__ val,
                                           const fr_t* __restrict__ w, uint32_t i,
                                           uint32_t check, uint32_t* err) {
  fr_t acc = fr_zero();
  for (uint32_t kx = rp[i], ke = rp[i + 1]; kx < ke; kx++) {
    const fr_t wv = fr_ldg(w + col[kx]);
    if (check) check_canonical(wv, err);
    if (fr_is_zero(wv)) continue;
    const fr_t cv = fr_ldg(val + kx);
    acc = fr_add(acc, fr_is_mont_one(wv) ? cv : fr_mul(cv, wv));
  }
  return fr_canon(acc);
}

__device__ __forceinline__ fr_t gather_c(const fr_t& a, const fr_t& b) {
  return (fr_is_zero(a) || fr_is_zero(b)) ? fr_zero() : fr_canon(fr_mul(a, b));
}

// Butterfly of the pass on slice bit lb: index bf in [0, 2^(kk-1)) -> lower element lo,
// upper element lo + 2^lb, and the twiddle table index of the element bit c0 + lb:
// j = (element index of lo) mod 2^(c0+lb) = low + ((lo mod 2^lb) << c0), times
// 2^(k - 1 - c0 - lb).
struct Bfly {
  uint32_t lo, hi, tw;
};

// Butterfly order within a pass: for lb <= kk - 6 the index runs j-major (bf = j * Q + q,
// Q = 2^(kk-1-lb) >= 32), so the 32 lanes of a warp share one twiddle index; above
// that, q-major (bf = q * 2^lb + j). Both orders visit every butterfly once.
__device__ __forceinline__ Bfly bfly_at(uint32_t bf, uint32_t lb, uint32_t kk, uint32_t low,
                                        uint32_t c0, uint32_t k) {
  Bfly b;
  uint32_t j, q;
  if (lb + 6u <= kk) {
    j = bf >> (kk - 1u - lb);
    q = bf & ((1u << (kk - 1u - lb)) - 1u);
  } else {
    j = bf & ((1u << lb) - 1u);
    q = bf >> lb;
  }
  b.lo = (q << (lb + 1u)) | j;
  b.hi = b.lo + (1u << lb);
  b.tw = (low + (j << c0)) << (k - 1u - c0 - lb);
  return b;
}

// Twiddle index 0 is omega^0 = 1. In the warp-uniform (j-major) passes a whole warp
// shares it, so the multiply is skipped without divergence; in pass 0 of element bit 0
// every butterfly has it.

// One decimation-in-frequency pass over the slice in shared memory, then a barrier.
__device__ __forceinline__ void dif_pass(uint4* sm, uint32_t kk, const fr_const_t* __restrict__ tw,
                                         uint32_t lb, uint32_t low, uint32_t c0, uint32_t k) {
  const uint32_t size = 1u << kk;
#pragma unroll 1
  for (uint32_t bf = threadIdx.x; bf < (size >> 1); bf += blockDim.x) {
    const Bfly b = bfly_at(bf, lb, kk, low, c0, k);
    const fr_t u = sm_get(sm, size, b.lo), v = sm_get(sm, size, b.hi);
    fr_t d = fr_sub(u, v);
    sm_put(sm, size, b.lo, fr_add(u, v));
    if (b.tw != 0u) d = fr_mul_c(d, fr_const_ldg(tw + b.tw));
    sm_put(sm, size, b.hi, d);
  }
  __syncthreads();
}

// One decimation-in-time pass, then a barrier.
__device__ __forceinline__ void dit_pass(uint4* sm, uint32_t kk, const fr_const_t* __restrict__ tw,
                                         uint32_t lb, uint32_t low, uint32_t c0, uint32_t k) {
  const uint32_t size = 1u << kk;
#pragma unroll 1
  for (uint32_t bf = threadIdx.x; bf < (size >> 1); bf += blockDim.x) {
    const Bfly b = bfly_at(bf, lb, kk, low, c0, k);
    fr_t v = sm_get(sm, size, b.hi);
    if (b.tw != 0u) v = fr_mul_c(v, fr_const_ldg(tw + b.tw));
    const fr_t u = sm_get(sm, size, b.lo);
    sm_put(sm, size, b.lo, fr_add(u, v));
    sm_put(sm, size, b.hi, fr_sub(u, v));
  }
  __syncthreads();
}

// Two passes at once, on slice bits L and L + 1: a group of four elements e0 = base,
// e1 = base + 2^L, e2 = base + 2^(L+1), e3 = e2 + 2^L (base with both bits clear), one
// group per thread iteration, one barrier for the two passes. Groups run j-major (a warp
// shares g_lo, hence every twiddle) when there are at least 32 groups per g_lo.
struct Quad4 {
  uint32_t e0, e1, e2, e3, glo;
};

__device__ __forceinline__ Quad4 quad_at(uint32_t g, uint32_t L, uint32_t kk) {
  Quad4 q;
  uint32_t glo, ghi;
  const uint32_t hib = kk - L - 2u;  // log2 of the number of g_hi values
  if (hib >= 5u) {
    glo = g >> hib;
    ghi = g & ((1u << hib) - 1u);
  } else {
    glo = g & ((1u << L) - 1u);
    ghi = g >> L;
  }
  q.e0 = (ghi << (L + 2u)) | glo;
  q.e1 = q.e0 + (1u << L);
  q.e2 = q.e0 + (2u << L);
  q.e3 = q.e2 + (1u << L);
  q.glo = glo;
  return q;
}

__device__ __forceinline__ uint32_t tw_index(uint32_t j, uint32_t b, uint32_t low, uint32_t c0,
                                             uint32_t k) {
  return (low + (j << c0)) << (k - 1u - c0 - b);
}

// Decimation in frequency on bits L + 1 (first) and L, then a barrier. SKIP1: test the
// first product's twiddle index for 0 (twiddle 1) and skip the product. That index is 0
// only when low = 0 (the contiguous slices, whose first groups of a pass have it, often
// for a whole warp); in the strided slices the test is left out, so that the two
// independent products share a basic block and the compiler can interleave them
// (measured: 2^18 k_ntt_dif 82.0 -> 79.9 us, k_ntt_dit 78.0 -> 75.8 us; in k_ntt_mid
// the skipped products are worth more: 127.5 vs 128.4 us).
template <bool SKIP1>
__device__ __forceinline__ void dif_pass2(uint4* sm, uint32_t kk, const fr_const_t* __restrict__ tw,
                                          uint32_t L, uint32_t low, uint32_t c0, uint32_t k) {
  const uint32_t size = 1u << kk;
  for (uint32_t g = threadIdx.x; g < (size >> 2); g += blockDim.x) {
    const Quad4 q = quad_at(g, L, kk);
    fr_t x0 = sm_get(sm, size, q.e0), x1 = sm_get(sm, size, q.e1);
    fr_t x2 = sm_get(sm, size, q.e2), x3 = sm_get(sm, size, q.e3);
    const uint32_t ta = tw_index(q.glo, L + 1u, low, c0, k);
    const uint32_t tb = tw_index(q.glo + (1u << L), L + 1u, low, c0, k);
    const uint32_t tc = tw_index(q.glo, L, low, c0, k);
    fr_t d02 = fr_sub(x0, x2), d13 = fr_sub(x1, x3);
    x0 = fr_add(x0, x2);
    x1 = fr_add(x1, x3);
    if (!SKIP1 || ta != 0u) d02 = fr_mul_c(d02, fr_const_ldg(tw + ta));
    d13 = fr_mul_c(d13, fr_const_ldg(tw + tb));  // tb != 0: its j has bit L set
    // bit L: (x0, x1) and (d02, d13), both with twiddle tc
    fr_t d01 = fr_sub(x0, x1), d23 = fr_sub(d02, d13);
    sm_put(sm, size, q.e0, fr_add(x0, x1));
    sm_put(sm, size, q.e2, fr_add(d02, d13));
    if (tc != 0u) {
      const fr_const_t wc = fr_const_ldg(tw + tc);
      d01 = fr_mul_c(d01, wc);
      d23 = fr_mul_c(d23, wc);
    }
    sm_put(sm, size, q.e1, d01);
    sm_put(sm, size, q.e3, d23);
  }
  __syncthreads();
}

// Decimation in time on bits L (first) and L + 1, then a barrier. SKIP1 as dif_pass2.
template <bool SKIP1>
__device__ __forceinline__ void dit_pass2(uint4* sm, uint32_t kk, const fr_const_t* __restrict__ tw,
                                          uint32_t L, uint32_t low, uint32_t c0, uint32_t k) {
  const uint32_t size = 1u << kk;
  for (uint32_t g = threadIdx.x; g < (size >> 2); g += blockDim.x) {
    const Quad4 q = quad_at(g, L, kk);
    fr_t x0 = sm_get(sm, size, q.e0), x1 = sm_get(sm, size, q.e1);
    fr_t x2 = sm_get(sm, size, q.e2), x3 = sm_get(sm, size, q.e3);
    const uint32_t tc = tw_index(q.glo, L, low, c0, k);
    const uint32_t ta = tw_index(q.glo, L + 1u, low, c0, k);
    const uint32_t tb = tw_index(q.glo + (1u << L), L + 1u, low, c0, k);
    // bit L: (x0, x1) and (x2, x3), twiddle tc on the upper elements
    if (tc != 0u) {
      const fr_const_t wc = fr_const_ldg(tw + tc);
      x1 = fr_mul_c(x1, wc);
      x3 = fr_mul_c(x3, wc);
    }
    fr_t y0 = fr_add(x0, x1), y1 = fr_sub(x0, x1);
    fr_t y2 = fr_add(x2, x3), y3 = fr_sub(x2, x3);
    // bit L + 1: (y0, y2) with ta, (y1, y3) with tb
    if (!SKIP1 || ta != 0u) y2 = fr_mul_c(y2, fr_const_ldg(tw + ta));
    y3 = fr_mul_c(y3, fr_const_ldg(tw + tb));
    sm_put(sm, size, q.e0, fr_add(y0, y2));
    sm_put(sm, size, q.e2, fr_sub(y0, y2));
    sm_put(sm, size, q.e1, fr_add(y1, y3));
    sm_put(sm, size, q.e3, fr_sub(y1, y3));
  }
  __syncthreads();
}

// The decimation-in-frequency passes of a slice on bits kk-1 .. lo_bit, two at a time with
// R4; SKIP1 for contiguous slices (dif_pass2).
template <bool R4, bool SKIP1 = false>
__device__ __forceinline__ void dif_passes(uint4* sm, uint32_t kk, const fr_const_t* __restrict__ tw,
                                           uint32_t low, uint32_t c0, uint32_t k,
                                           uint32_t lo_bit = 0) {
  int lb = (int)kk - 1;
  if (R4)
    for (; lb >= (int)lo_bit + 1; lb -= 2)
      dif_pass2<SKIP1>(sm, kk, tw, (uint32_t)lb - 1u, low, c0, k);
  for (; lb >= (int)lo_bit; lb--) dif_pass(sm, kk, tw, (uint32_t)lb, low, c0, k);
}

// The decimation-in-time passes of a slice on bits first_bit .. kk-1, two at a time with R4.
template <bool R4, bool SKIP1 = false>
__device__ __forceinline__ void dit_passes(uint4* sm, uint32_t kk, const fr_const_t* __restrict__ tw,
                                           uint32_t low, uint32_t c0, uint32_t k,
                                           uint32_t first_bit = 0) {
  uint32_t lb = first_bit;
  if (R4)
    for (; lb + 1u < kk; lb += 2) dit_pass2<SKIP1>(sm, kk, tw, lb, low, c0, k);
  for (; lb < kk; lb++) dit_pass(sm, kk, tw, lb, low, c0, k);
}

// On a contiguous slice (c0 = 0): the inverse's pass on bit 0 (twiddle 1), the coset shift
// and the forward's pass on bit 0 (twiddle 1). All three work on the element pairs
// (2m, 2m + 1), so one thread holds each pair throughout: (u, v) -> (u + v, u - v), times
// the shift entries (s_2m, s_2m+1) -> (a, b) -> (a + b, a - b); then a barrier.
__device__ __forceinline__ void bit0_shift_bit0(uint4* sm, uint32_t kk,
                                                const fr_const_t* __restrict__ shift) {
  const uint32_t size = 1u << kk;
#pragma unroll 1
  for (uint32_t bf = threadIdx.x; bf < (size >> 1); bf += blockDim.x) {
    const uint32_t lo = 2u * bf, hi = lo + 1u;
    const fr_t u = sm_get(sm, size, lo), v = sm_get(sm, size, hi);
    const fr_t a = fr_mul_c(fr_add(u, v), fr_const_ldg(shift + lo));
    const fr_t b = fr_mul_c(fr_sub(u, v), fr_const_ldg(shift + hi));
    sm_put(sm, size, lo, fr_add(a, b));
    sm_put(sm, size, hi, fr_sub(a, b));
  }
  __syncthreads();
}

// Three builds of each slice kernel, chosen by slice size (measured on GB300):
//   0: radix-2 passes, 256 threads, four resident blocks per SM (64 registers): slices up
//      to 2^8 (2^12, 2^14: latency-bound, the pass pairs measured 0.069 -> 0.081 ms);
//   1: radix-4 pass pairs, 128 threads, five blocks (up to 102 registers): 2^9 and 2^10
//      slices (2^18 H: 0.310 -> 0.295 ms; 2^20: 1.146 -> 1.071 ms);
//   2: radix-4 pass pairs, 256 threads, three blocks (85 registers; three 64 KiB slices
//      fill the shared memory): 2^11 slices (2^22 H: 4.97 -> 4.81 ms; build 1 there: 5.18).
template <int C>
struct SliceCfg;
template <>
struct SliceCfg<0> {
  static constexpr bool r4 = false;
  static constexpr uint32_t threads = 256, min_blocks = 4;
};
template <>
struct SliceCfg<1> {
  static constexpr bool r4 = true;
  static constexpr uint32_t threads = 128, min_blocks = 5;
};
template <>
struct SliceCfg<2> {
  static constexpr bool r4 = true;
  static constexpr uint32_t threads = 256, min_blocks = 3;
};
constexpr uint32_t kRadix4MinSliceBits = 9, kRadix4MaxSliceBits = 10, kCfg2MinSliceBits = 11;

// Block s of a strided slice kernel owns low = s mod 2^c0, high = s >> c0 and the
// elements low + (m << c0) + (high << (c0 + kk)), m < 2^kk.
__device__ __forceinline__ size_t slice_base(uint32_t s, uint32_t c0, uint32_t kk) {
  return (size_t)(s & ((1u << c0) - 1u)) + ((size_t)(s >> c0) << (c0 + kk));
}

// The slice and the vector (grid row) of this block, in either block order (SliceArgs::vfast).
__device__ __forceinline__ uint32_t block_slice(const SliceArgs& p) {
  return p.vfast ? blockIdx.x / 3u : blockIdx.x;
}
__device__ __forceinline__ uint32_t block_vector(const SliceArgs& p) {
  return p.vbase + (p.vfast ? blockIdx.x % 3u : blockIdx.y);
}

// ---------------------------------------------------------------------------------------
// k_ntt_dif: decimation-in-frequency passes over slice bits [c0, c0 + kk) of vector
// vbase + blockIdx.y, src -> dst (in place when equal: every block reads its whole slice before
// it writes). With SL_C_FROM_AB vector 2 is formed as a * b from vectors 0 and 1 at load.
// Launch: grid (n >> kk, vectors), block min(2^(kk-1), 256), dynamic shared memory
// 2^kk * 32 bytes.
template <int C>
__global__ void __launch_bounds__(SliceCfg<C>::threads, SliceCfg<C>::min_blocks) k_ntt_dif(const __grid_constant__ SliceArgs p) {
  extern __shared__ uint4 sm[];
  wait_prior_grid();
  const uint32_t kk = p.kk, c0 = p.c0, k = p.log_n, size = 1u << kk;
  const uint32_t sl = block_slice(p);
  const uint32_t low = sl & ((1u << c0) - 1u);
  const size_t base = slice_base(sl, c0, kk);
  const uint32_t vec = block_vector(p);
  const size_t zsrc = (size_t)blockIdx.z * p.zs_src;
  const fr_t* src = p.src[vec] + zsrc;
  fr_t* dst = p.dst[vec] + (size_t)blockIdx.z * p.zs_dst;
  const uint32_t check = p.mode & SL_CHECK;
  if ((p.mode & SL_C_FROM_AB) && vec == 2u) {
    for (uint32_t m = threadIdx.x; m < size; m += blockDim.x) {
      const size_t i = zsrc + base + ((size_t)m << c0);
      sm_put(sm, size, m, gather_c(fr_load(p.src[0] + i), fr_load(p.src[1] + i)));
    }
  } else {
    for (uint32_t m = threadIdx.x; m < size; m += blockDim.x) {
      const fr_t x = fr_load(src + base + ((size_t)m << c0));
      if (check) check_canonical(x, p.err);
      sm_put(sm, size, m, x);
    }
  }
  __syncthreads();
  dif_passes<SliceCfg<C>::r4>(sm, kk, p.tw, low, c0, k);
  for (uint32_t m = threadIdx.x; m < size; m += blockDim.x)
    fr_store(dst + base + ((size_t)m << c0), sm_get(sm, size, m));
}

// ---------------------------------------------------------------------------------------
// k_ntt_mid: on the contiguous slice of 2^kk elements starting at blockIdx.x << kk of
// vector vbase + blockIdx.y: the inverse transform's decimation-in-frequency passes on bits
// kk-1 .. 0 (twiddles p.tw), the shift by scale_tab[position] (g^brev(position) / n),
// then the forward transform's decimation-in-time passes on bits 0 .. kk-1 (twiddles
// p.tw2). In place. With kk odd the two passes on bit 0 and the shift run as one step. Launch: grid (n >> kk, vectors), block min(2^(kk-1), 256), shared
// 2^kk * 32 bytes.
template <int C>
__global__ void __launch_bounds__(SliceCfg<C>::threads, SliceCfg<C>::min_blocks) k_ntt_mid(const __grid_constant__ SliceArgs p) {
  extern __shared__ uint4 sm[];
  wait_prior_grid();
  const uint32_t kk = p.kk, k = p.log_n, size = 1u << kk;
  const size_t base = (size_t)block_slice(p) << kk;
  fr_t* vec = p.dst[block_vector(p)] + (size_t)blockIdx.z * p.zs_dst;
  for (uint32_t m = threadIdx.x; m < size; m += blockDim.x)
    sm_put(sm, size, m, fr_load(vec + base + m));
  __syncthreads();
  if (kk & 1u) {
    // odd slice bits: the passes on bit 0 meet the shift in one step (two barriers and two
    // shared-memory round trips fewer); the forward's pairs then start at bit 1
    dif_passes<SliceCfg<C>::r4, true>(sm, kk, p.tw, 0u, 0u, k, 1u);
    bit0_shift_bit0(sm, kk, p.scale_tab + base);
    dit_passes<SliceCfg<C>::r4, true>(sm, kk, p.tw2, 0u, 0u, k, 1u);
  } else {
    dif_passes<SliceCfg<C>::r4, true>(sm, kk, p.tw, 0u, 0u, k);
    for (uint32_t m = threadIdx.x; m < size; m += blockDim.x)
      sm_put(sm, size, m, fr_mul_c(sm_get(sm, size, m), fr_const_ldg(p.scale_tab + base + m)));
    __syncthreads();
    dit_passes<SliceCfg<C>::r4, true>(sm, kk, p.tw2, 0u, 0u, k);
  }
  for (uint32_t m = threadIdx.x; m < size; m += blockDim.x)
    fr_store(vec + base + m, sm_get(sm, size, m));
}

// ---------------------------------------------------------------------------------------
// k_ntt_dit: decimation-in-time passes over slice bits [c0, c0 + kk) (geometry as
// k_ntt_dif), src -> dst. Store epilogues:
//   SL_SCALE_TABLE: dst[i] = x * scale_tab[i];  SL_SCALE_CONST: dst[i] = x * kscale;
//   SL_JOIN: one block runs vectors 0, 1, 2 (a, b, c) of its slice in turn; a and b are
//   stored to dst[0], dst[1], and at c's store every thread re-reads the a and b values
//   it stored itself and writes h = a*b - c to h_mont and from_mont(h) to h_std
//   (the POINTWISE_CU join fused into the last transform's store).
//   SL_JOIN_LAST: block (s, v) runs vector v of slice s and stores it to dst[v]; the
//   three blocks of a slice then count themselves in on counters[s] (each thread fences
//   its stores first), and the block that arrives third reads a, b, c of the slice from
//   L2 and writes h, then resets the counter. No block ever waits for another.
// Launch: grid (n >> kk, vectors; 1 with SL_JOIN), block min(2^(kk-1), 256), shared
// 2^kk * 32 bytes.
template <int C>
__global__ void __launch_bounds__(SliceCfg<C>::threads, SliceCfg<C>::min_blocks) k_ntt_dit(const __grid_constant__ SliceArgs p) {
  extern __shared__ uint4 sm[];
  wait_prior_grid();
  const uint32_t kk = p.kk, c0 = p.c0, k = p.log_n, size = 1u << kk;
  const uint32_t sl = block_slice(p);
  const uint32_t low = sl & ((1u << c0) - 1u);
  const size_t base = slice_base(sl, c0, kk);
  const bool join = (p.mode & SL_JOIN) != 0u;
  const uint32_t nvec = join ? 3u : 1u;
  const size_t zsrc = (size_t)blockIdx.z * p.zs_src, zdst = (size_t)blockIdx.z * p.zs_dst;
  const size_t zh = (size_t)blockIdx.z * p.zs_h;
  for (uint32_t vi = 0; vi < nvec; vi++) {
    const uint32_t v = join ? vi : block_vector(p);
    const fr_t* src = p.src[v] + zsrc;
    fr_t* dst = p.dst[v] + zdst;
    if (vi > 0) __syncthreads();  // the previous vector's last shared-memory reads
    for (uint32_t m = threadIdx.x; m < size; m += blockDim.x)
      sm_put(sm, size, m, fr_load(src + base + ((size_t)m << c0)));
    __syncthreads();
    dit_passes<SliceCfg<C>::r4>(sm, kk, p.tw, low, c0, k);
    for (uint32_t m = threadIdx.x; m < size; m += blockDim.x) {
      const size_t i = base + ((size_t)m << c0);
      const fr_t x = sm_get(sm, size, m);
      if (join && v == 2u) {
        const fr_t a = fr_load(p.dst[0] + zdst + i);
        const fr_t b = fr_load(p.dst[1] + zdst + i);
        const fr_t h = fr_canon(fr_sub(fr_mul(a, b), x));
        fr_store(p.h_mont + zh + i, h);
        fr_store(p.h_std + zh + i, fr_from_mont(h));
      } else if (join || (p.mode & SL_JOIN_LAST)) {
        fr_store(dst + i, x);
      } else {
        fr_t y = x;
        if (p.mode & SL_SCALE_TABLE) y = fr_mul_c(y, fr_const_ldg(p.scale_tab + i));
        if (p.mode & SL_SCALE_CONST) y = fr_mul_c(y, p.kscale);
        fr_store(dst + i, fr_canon(y));
      }
    }
  }
  if (p.mode & SL_JOIN_LAST) {
    __shared__ uint32_t arrived;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      arrived = atomicAdd(p.counters + sl, 1u);
      __threadfence();
    }
    __syncthreads();
    if (arrived == 2u) {
      for (uint32_t m = threadIdx.x; m < size; m += blockDim.x) {
        const size_t i = base + ((size_t)m << c0);
        const fr_t a = fr_ldcg(p.dst[0] + zdst + i), b = fr_ldcg(p.dst[1] + zdst + i);
        const fr_t c = fr_ldcg(p.dst[2] + zdst + i);
        const fr_t h = fr_canon(fr_sub(fr_mul(a, b), c));
        fr_store(p.h_mont + zh + i, h);
        fr_store(p.h_std + zh + i, fr_from_mont(h));
      }
      if (threadIdx.x == 0) p.counters[sl] = 0u;
    }
  }
}

// ---------------------------------------------------------------------------------------
// k_ntt_brev: the first decimation-in-time passes (bits 0 .. kk-1) of a natural-order
// transform, on the contiguous slice at blockIdx.x << kk: position i loads src[brev(i)]
// (the bit-reversal permutation absorbed into the load, as on the NTT_CU page), scaled by
// scale_tab[i] (SL_SCALE_TABLE: a table kept in bit-reversed order, so that its reads are
// contiguous) or kscale (SL_SCALE_CONST), and the result goes to
// dst (out of place: a block reads other blocks' elements). The passes are those of the
// slice build C (radix-4 pass pairs in builds 1 and 2). Every 32-byte element is one
// sector, so the scattered loads read no byte they do not use.
// Launch: grid (n >> kk), block as the build's other kernels, shared 2^kk * 32 bytes.
template <int C>
__global__ void __launch_bounds__(SliceCfg<C>::threads, SliceCfg<C>::min_blocks) k_ntt_brev(const __grid_constant__ SliceArgs p) {
  extern __shared__ uint4 sm[];
  const uint32_t kk = p.kk, k = p.log_n, size = 1u << kk;
  // Block b runs slice brev(b): slice s reads the elements whose low k - kk index bits are
  // brev(s), so consecutive blocks read neighbouring elements, which share cache lines
  // (measured at 2^22: 805 -> 403 MB of DRAM reads per launch, 439 -> 428 us)
  const size_t base = (size_t)bitrev(blockIdx.x, k - kk) << kk;
  for (uint32_t m = threadIdx.x; m < size; m += blockDim.x) {
    const uint32_t j = bitrev((uint32_t)base + m, k);
    fr_t x = fr_load(p.src[0] + j);
    if (p.mode & SL_CHECK) check_canonical(x, p.err);
    if (p.mode & SL_SCALE_TABLE) x = fr_mul_c(x, fr_const_ldg(p.scale_tab + base + m));
    if (p.mode & SL_SCALE_CONST) x = fr_mul_c(x, p.kscale);
    sm_put(sm, size, m, x);
  }
  __syncthreads();
  dit_passes<SliceCfg<C>::r4, true>(sm, kk, p.tw, 0u, 0u, k);
  for (uint32_t m = threadIdx.x; m < size; m += blockDim.x)
    fr_store(p.dst[0] + base + m, sm_get(sm, size, m));
}

}  // namespace g3h
