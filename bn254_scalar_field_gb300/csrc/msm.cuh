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
//   1. count: per-bucket entry counts (32-bit atomics on counters, never on points);
//   2. scan: exclusive prefix sum of the counts (bucket offsets);
//   3. scatter: each (i, w) entry, as (16 i + w) << 1 | sign, into its bucket's run
//      (a counting sort by bucket; order inside a run is arbitrary, the sum commutes);
//   4. accumulate: the sorted entries in fixed-length slices, one thread per slice, so
//      that work per thread does not depend on how the digits spread over buckets; a run
//      that lies inside one slice is written to its bucket, a run cut by a slice boundary
//      leaves its part in that slice's head or tail slot (MSM_CU, "the load-balanced
//      form": segmented accumulation with boundary spills);
//   5. merge: a cut bucket sums its parts from the slices its run covers;
//   6-8. the weighted sum sum_j j B_j: per group of 4 buckets (t = 0 .. 8191) the
//      running sums give U_t = sum B and V_t = sum (j - 4t) B_j; then
//      Q = sum_t V_t + sum_b 2^(b+2) sum_{t : bit b of t} U_t, thirteen bit-sums and one
//      sum of V reduced by trees, scaled by doublings, and added in a last kernel, which
//      writes Q in Jacobian coordinates.
#pragma once
#include "fr.cuh"
#include "g1.cuh"

namespace g3h {

constexpr uint32_t kMsmWindows = 16;          // windows of 16 bits
constexpr uint32_t kMsmBuckets = 1u << 15;    // digit magnitudes 1 .. 2^15
constexpr uint32_t kMsmGroup = 4;             // buckets per running-sum group
constexpr uint32_t kMsmGroups = kMsmBuckets / kMsmGroup;  // 8192 = 2^13
constexpr uint32_t kMsmGroupBits = 13;
constexpr uint32_t kMsmParts = kMsmGroupBits + 1;  // 13 bit-sums of U, one sum of V
constexpr uint32_t kMsmReduceThreads = 512;
constexpr uint32_t kMsmErrPoint = 2u;  // error word bit: a base is not on the curve

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
__global__ void __launch_bounds__(128) k_msm_precompute(const g1_aff_t* bases, uint32_t n,
                                                        g1_aff_t* table, uint32_t* err) {
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  g1_aff_t b = bases[i];
  g1_aff_t* out = table + (size_t)i * kMsmWindows;
  if (aff_is_inf(b)) {
    for (uint32_t w = 0; w < kMsmWindows; w++) out[w] = b;
    return;
  }
  if (!fq_is_canonical(b.x) || !fq_is_canonical(b.y)) {
    atomicOr(err, 1u);
    b.x = fq_zero();
    b.y = fq_zero();
    for (uint32_t w = 0; w < kMsmWindows; w++) out[w] = b;
    return;
  }
  if (!aff_on_curve(b)) atomicOr(err, kMsmErrPoint);
  out[0] = b;
  g1_xyzz_t p = xyzz_from_aff(b);
  for (uint32_t w = 1; w < kMsmWindows; w++) {
    for (int d = 0; d < 16; d++) p = xyzz_dbl(p);
    out[w] = xyzz_to_aff(p);
  }
}

// Step 1. Launch: any grid of 256-thread blocks (grid-stride over the scalars).
__global__ void __launch_bounds__(256) k_msm_count(const fr_t* scalars, uint32_t n,
                                                   uint32_t* counts, uint32_t check,
                                                   uint32_t* err) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint32_t s[8];
    msm_load_scalar(scalars, i, s, check, err);
    uint32_t carry = 0;
#pragma unroll
    for (uint32_t w = 0; w < kMsmWindows; w++) {
      const int d = msm_digit(s, w, carry);
      if (d != 0) atomicAdd(counts + (uint32_t)(d < 0 ? -d : d) - 1u, 1u);
    }
  }
}

// Step 2: offsets[j] = sum of counts[0 .. j), offsets[kMsmBuckets] = total; cursor = offsets.
// Launch: one block of 1024 threads (32 buckets per thread).
__global__ void __launch_bounds__(1024) k_msm_scan(const uint32_t* counts, uint32_t* offsets,
                                                   uint32_t* cursor) {
  constexpr uint32_t per = kMsmBuckets / 1024;
  __shared__ uint32_t warp_tot[32];
  const uint32_t t = threadIdx.x, lane = t & 31u, warp = t >> 5;
  uint32_t local[per];
  uint32_t sum = 0;
#pragma unroll
  for (uint32_t k = 0; k < per; k++) {
    local[k] = counts[t * per + k];
    sum += local[k];
  }
  // inclusive scan of the per-thread sums within the warp, then over the warps
  uint32_t inc = sum;
#pragma unroll
  for (uint32_t d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    uint32_t v = warp_tot[lane];
#pragma unroll
    for (uint32_t d = 1; d < 32; d <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += o;
    }
    warp_tot[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  uint32_t run = inc - sum + (warp ? warp_tot[warp - 1] : 0u);
#pragma unroll
  for (uint32_t k = 0; k < per; k++) {
    offsets[t * per + k] = run;
    cursor[t * per + k] = run;
    run += local[k];
  }
  if (t == 1023) offsets[kMsmBuckets] = run;
}

// Step 3. Launch: as k_msm_count.
__global__ void __launch_bounds__(256) k_msm_scatter(const fr_t* scalars, uint32_t n,
                                                     uint32_t* cursor, uint32_t* entries) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint32_t s[8];
    msm_load_scalar(scalars, i, s, 0u, nullptr);
    uint32_t carry = 0;
#pragma unroll
    for (uint32_t w = 0; w < kMsmWindows; w++) {
      const int d = msm_digit(s, w, carry);
      if (d == 0) continue;
      const uint32_t slot = atomicAdd(cursor + (uint32_t)(d < 0 ? -d : d) - 1u, 1u);
      entries[slot] = ((i * kMsmWindows + w) << 1) | (d < 0 ? 1u : 0u);
    }
  }
}

// Step 4: slice k = entries [k L, min(k L + L, total)). Launch: ceil(n_slices / 256)
// blocks of 256; slices past the total exit.
__global__ void __launch_bounds__(256) k_msm_accumulate(const uint32_t* entries,
                                                        const uint32_t* offsets,
                                                        const g1_aff_t* table,
                                                        g1_xyzz_t* buckets, g1_xyzz_t* head,
                                                        g1_xyzz_t* tail, uint32_t slice,
                                                        uint32_t n_slices) {
  const uint32_t k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n_slices) return;
  const uint32_t total = offsets[kMsmBuckets];
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
  g1_xyzz_t acc = xyzz_infinity();
  auto emit = [&]() {
    if (offsets[b] < lo) head[k] = acc;
    else if (run_end > hi) tail[k] = acc;
    else buckets[b] = acc;
  };
  for (uint32_t i = lo; i < hi; i++) {
    if (i == run_end) {
      emit();
      acc = xyzz_infinity();
      do {
        b++;
        run_end = offsets[b + 1];
      } while (run_end <= i);
    }
    const uint32_t e = entries[i];
    g1_aff_t p = table[e >> 1];
    if (aff_is_inf(p)) continue;
    if (e & 1u) p = aff_neg(p);
    acc = xyzz_madd(acc, p);
  }
  emit();
}

// Step 5: one thread per bucket. A bucket with no entries is set to infinity; a run cut by
// slice boundaries is the tail part of its first slice plus the head parts of the rest.
// Launch: kMsmBuckets / 256 blocks of 256.
__global__ void __launch_bounds__(256) k_msm_merge(const uint32_t* offsets, g1_xyzz_t* buckets,
                                                   const g1_xyzz_t* head, const g1_xyzz_t* tail,
                                                   uint32_t slice) {
  const uint32_t j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= kMsmBuckets) return;
  const uint32_t s = offsets[j], e = offsets[j + 1];
  if (s == e) {
    buckets[j] = xyzz_infinity();
    return;
  }
  const uint32_t k_lo = s / slice, k_hi = (e - 1u) / slice;
  if (k_lo == k_hi) return;
  g1_xyzz_t acc = tail[k_lo];
  for (uint32_t k = k_lo + 1; k <= k_hi; k++) acc = xyzz_add(acc, head[k]);
  buckets[j] = acc;
}

// Step 6: group t = buckets 4t .. 4t+3 (digits 4t+1 .. 4t+4): U_t = sum B,
// V_t = sum_u (u + 1) B_{4t+u}, by running sums from the top. Launch: kMsmGroups / 256
// blocks of 256.
__global__ void __launch_bounds__(256) k_msm_reduce_groups(const g1_xyzz_t* buckets,
                                                           g1_xyzz_t* U, g1_xyzz_t* V) {
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= kMsmGroups) return;
  g1_xyzz_t run = xyzz_infinity(), acc = xyzz_infinity();
  for (int u = (int)kMsmGroup - 1; u >= 0; u--) {
    run = xyzz_add(run, buckets[t * kMsmGroup + (uint32_t)u]);
    acc = xyzz_add(acc, run);
  }
  U[t] = run;
  V[t] = acc;
}

// Step 7: block b < 13 sums U_t over the t with bit b set and doubles the sum b + 2 times
// (the weight 4 t of U_t, bit by bit); block 13 sums V. Launch: kMsmParts blocks of
// kMsmReduceThreads, kMsmReduceThreads * 128 bytes of dynamic shared memory.
__global__ void __launch_bounds__(kMsmReduceThreads) k_msm_reduce_bits(const g1_xyzz_t* U,
                                                                       const g1_xyzz_t* V,
                                                                       g1_xyzz_t* parts) {
  extern __shared__ g1_xyzz_t sm_pts[];
  const uint32_t b = blockIdx.x, tid = threadIdx.x;
  g1_xyzz_t acc = xyzz_infinity();
  for (uint32_t t = tid; t < kMsmGroups; t += kMsmReduceThreads) {
    if (b < kMsmGroupBits) {
      if ((t >> b) & 1u) acc = xyzz_add(acc, U[t]);
    } else {
      acc = xyzz_add(acc, V[t]);
    }
  }
  sm_pts[tid] = acc;
  __syncthreads();
  for (uint32_t s = kMsmReduceThreads / 2; s > 0; s >>= 1) {
    if (tid < s) sm_pts[tid] = xyzz_add(sm_pts[tid], sm_pts[tid + s]);
    __syncthreads();
  }
  if (tid == 0) {
    g1_xyzz_t p = sm_pts[0];
    if (b < kMsmGroupBits)
      for (uint32_t d = 0; d < b + 2; d++) p = xyzz_dbl(p);
    parts[b] = p;
  }
}

// Step 8: Q = sum of the parts, written as Jacobian (X, Y, Z), canonical Montgomery
// coordinates, infinity as (0, 0, 0). Launch: one block of 32 (lane 0 works).
__global__ void __launch_bounds__(32) k_msm_final(const g1_xyzz_t* parts, fq_t* out) {
  if (threadIdx.x != 0) return;
  g1_xyzz_t acc = xyzz_infinity();
  for (uint32_t b = 0; b < kMsmParts; b++) acc = xyzz_add(acc, parts[b]);
  xyzz_to_jacobian(acc, out[0], out[1], out[2]);
}

}  // namespace g3h
