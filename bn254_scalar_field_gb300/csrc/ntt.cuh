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
//    bits [c0, c0 + KK) can run on the "slice" of 2^KK elements that agree on all other
//    bits (the six-step decomposition the NTT_CU page describes as (s0, k) batching).
//    The lowest slice (c0 = 0) is contiguous, and the inverse's last passes and the
//    forward's first passes both live there, so one kernel runs them back to back with
//    the shift in between (k_ntt_mid).
//
// Thread mapping. A slice of 2^KK elements has 2^(KK-3) threads; in each round a thread
// holds 8 elements in registers, those whose local indices differ only in three chosen
// bits [P, P+3), and runs up to three radix-2 passes on them before exchanging through
// shared memory. Local index of register e of thread t in a round at P:
//   m = (t mod 2^P) | (e << P) | ((t >> P) << (P + 3)).
//
// Shared memory holds each 32-byte element as two 16-byte halves in two planes, with the
// 16-byte slot index swizzled as m ^ ((m >> 3) & 7). Every round's access pattern then
// hits eight distinct 16-byte bank groups per quarter warp.
#pragma once
#include "fr.cuh"

namespace g3h {

enum : uint32_t {
  SL_CHECK = 1u,        // check loaded inputs are canonical, report through *err
  SL_SCALE_TABLE = 2u,  // scale by scale_tab (see each kernel)
  SL_SCALE_CONST = 4u,  // scale by kscale
  SL_JOIN = 8u,         // k_ntt_dit: vectors 0, 1, 2 are a, b, c; write h = a*b - c
};

struct SliceArgs {
  const fr_t* src[3];
  fr_t* dst[3];
  const fr_t* tw;         // twiddles of the passes (forward or inverse table, n/2 entries)
  const fr_t* tw2;        // k_ntt_mid: forward twiddles for its decimation-in-time half
  const fr_t* scale_tab;  // per-kernel scale table (n entries)
  fr_t* h_mont;
  fr_t* h_std;
  uint32_t* err;
  fr_t kscale;
  uint32_t log_n;  // k: the vector has 2^k elements
  uint32_t kk;     // slice bits
  uint32_t c0;     // the slice's bits are [c0, c0 + kk) of the element index
  uint32_t mode;   // SL_* flags
};

__device__ __forceinline__ uint32_t swz(uint32_t m) { return m ^ ((m >> 3) & 7u); }

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

__device__ __forceinline__ uint32_t local_index(uint32_t t, uint32_t e, uint32_t P) {
  return (t & ((1u << P) - 1u)) | (e << P) | ((t >> P) << (P + 3u));
}

__device__ __forceinline__ uint32_t bitrev(uint32_t x, uint32_t bits) {
  return bits == 0u ? 0u : (__brev(x) >> (32u - bits));
}

__device__ __forceinline__ void check_canonical(const fr_t& x, uint32_t* err) {
  if (!fr_is_canonical(x)) atomicOr(err, 1u);
}

// Twiddle table index of the butterfly whose lower element is register e, for the pass
// on slice bit lb = P + q (element bit b = c0 + lb): j = (element index) mod 2^b
// = low + ((m mod 2^lb) << c0), index j * 2^(k - 1 - b).
__device__ __forceinline__ uint32_t tw_index(uint32_t t, uint32_t e, uint32_t q, uint32_t P,
                                             uint32_t low, uint32_t c0, uint32_t k) {
  const uint32_t mmod = (t & ((1u << P) - 1u)) | ((e & ((1u << q) - 1u)) << P);
  const uint32_t j = low + (mmod << c0);
  return j << (k - 1u - c0 - P - q);
}

// Decimation-in-frequency passes on register bits q = qb, qb-1, ..., 0 of a round at P.
__device__ __forceinline__ void dif_round(fr_t (&x)[8], const fr_t* __restrict__ tw, uint32_t t,
                                          uint32_t P, int qb, uint32_t low, uint32_t c0,
                                          uint32_t k) {
#pragma unroll
  for (int q = 2; q >= 0; q--) {
    if (q > qb) continue;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      if (e & (1 << q)) continue;
      const int f = e | (1 << q);
      const fr_t w = fr_ldg(tw + tw_index(t, e, q, P, low, c0, k));
      const fr_t u = x[e];
      x[e] = fr_add(u, x[f]);
      x[f] = fr_mul(fr_sub(u, x[f]), w);
    }
  }
}

// Decimation-in-time passes on register bits q = qa, ..., 2 of a round at P.
__device__ __forceinline__ void dit_round(fr_t (&x)[8], const fr_t* __restrict__ tw, uint32_t t,
                                          uint32_t P, int qa, uint32_t low, uint32_t c0,
                                          uint32_t k) {
#pragma unroll
  for (int q = 0; q <= 2; q++) {
    if (q < qa) continue;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      if (e & (1 << q)) continue;
      const int f = e | (1 << q);
      const fr_t w = fr_ldg(tw + tw_index(t, e, q, P, low, c0, k));
      const fr_t v = fr_mul(x[f], w);
      const fr_t u = x[e];
      x[e] = fr_add(u, v);
      x[f] = fr_sub(u, v);
    }
  }
}

// The round at P = 0 of a contiguous slice (c0 = 0): the butterfly index j = e mod 2^q
// is known at compile time, and j = 0 means the twiddle is 1 and the multiply is skipped.
__device__ __forceinline__ void dif_round_p0(fr_t (&x)[8], const fr_t* __restrict__ tw, int qb,
                                             uint32_t k) {
#pragma unroll
  for (int q = 2; q >= 0; q--) {
    if (q > qb) continue;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      if (e & (1 << q)) continue;
      const int f = e | (1 << q);
      const int j = e & ((1 << q) - 1);
      const fr_t u = x[e];
      x[e] = fr_add(u, x[f]);
      if (j == 0) {
        x[f] = fr_sub(u, x[f]);
      } else {
        const fr_t w = fr_ldg(tw + ((uint32_t)j << (k - 1u - (uint32_t)q)));
        x[f] = fr_mul(fr_sub(u, x[f]), w);
      }
    }
  }
}

__device__ __forceinline__ void dit_round_p0(fr_t (&x)[8], const fr_t* __restrict__ tw, int qa,
                                             uint32_t k) {
#pragma unroll
  for (int q = 0; q <= 2; q++) {
    if (q < qa) continue;
#pragma unroll
    for (int e = 0; e < 8; e++) {
      if (e & (1 << q)) continue;
      const int f = e | (1 << q);
      const int j = e & ((1 << q) - 1);
      fr_t v = x[f];
      if (j != 0) v = fr_mul(v, fr_ldg(tw + ((uint32_t)j << (k - 1u - (uint32_t)q))));
      const fr_t u = x[e];
      x[e] = fr_add(u, v);
      x[f] = fr_sub(u, v);
    }
  }
}

// Rounds of a slice of kk bits. Decimation in frequency runs the bits from the top:
// full rounds at P = kk-3, kk-6, ..., then (kk mod 3 != 0) a partial round at P = 0 on
// bits kk mod 3 - 1 .. 0. Decimation in time runs from the bottom: full rounds at
// P = 0, 3, ..., then a partial round at P = kk - 3 on its top kk mod 3 bits.
__device__ __forceinline__ uint32_t dif_round_P(uint32_t r, uint32_t kk) {
  return (r < kk / 3u) ? kk - 3u * (r + 1u) : 0u;
}
__device__ __forceinline__ int dif_round_qb(uint32_t r, uint32_t kk) {
  return (r < kk / 3u) ? 2 : (int)(kk % 3u) - 1;
}
__device__ __forceinline__ uint32_t dit_round_P(uint32_t r, uint32_t kk) {
  return (r < kk / 3u) ? 3u * r : kk - 3u;
}
__device__ __forceinline__ int dit_round_qa(uint32_t r, uint32_t kk) {
  return (r < kk / 3u) ? 0 : 3 - (int)(kk % 3u);
}

// ---------------------------------------------------------------------------------------
// k_ntt_dif: decimation-in-frequency passes over slice bits [c0, c0 + kk) of vector
// blockIdx.y, src -> dst (in place when equal: every block reads its whole slice before
// it writes). Block s owns low = s mod 2^c0, high = s >> c0, elements
// low + (m << c0) + (high << (c0 + kk)). Launch: grid (n >> kk, vectors), block
// 2^(kk-3), dynamic shared memory 2^kk * 32 bytes.
__global__ void __launch_bounds__(256) k_ntt_dif(const __grid_constant__ SliceArgs p) {
  extern __shared__ uint4 sm[];
  const uint32_t t = threadIdx.x, kk = p.kk, c0 = p.c0, k = p.log_n;
  const uint32_t half = 1u << kk;
  const uint32_t s = blockIdx.x, v = blockIdx.y;
  const uint32_t low = s & ((1u << c0) - 1u);
  const size_t base = low + ((size_t)(s >> c0) << (c0 + kk));
  const fr_t* src = p.src[v];
  fr_t* dst = p.dst[v];
  const uint32_t rounds = (kk + 2u) / 3u;
  fr_t x[8];
  for (uint32_t r = 0; r < rounds; r++) {
    const uint32_t P = dif_round_P(r, kk);
    if (r == 0) {
#pragma unroll
      for (int e = 0; e < 8; e++) {
        x[e] = fr_load(src + base + ((size_t)local_index(t, e, P) << c0));
        if (p.mode & SL_CHECK) check_canonical(x[e], p.err);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; e++) x[e] = sm_get(sm, half, local_index(t, e, P));
    }
    dif_round(x, p.tw, t, P, dif_round_qb(r, kk), low, c0, k);
    if (r + 1 == rounds) {
#pragma unroll
      for (int e = 0; e < 8; e++) fr_store(dst + base + ((size_t)local_index(t, e, P) << c0), x[e]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; e++) sm_put(sm, half, local_index(t, e, P), x[e]);
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------------------------------
// k_ntt_mid: on the contiguous slice of 2^kk elements starting at blockIdx.x << kk of
// vector blockIdx.y, the inverse transform's decimation-in-frequency passes on bits
// kk-1 .. 0 (twiddles p.tw), the shift by scale_tab[position] (g^brev(position) / n),
// then the forward transform's decimation-in-time passes on bits 0 .. kk-1 (twiddles
// p.tw2). In place. Launch: grid (n >> kk, vectors), block 2^(kk-3), shared 2^kk * 32.
__global__ void __launch_bounds__(256) k_ntt_mid(const __grid_constant__ SliceArgs p) {
  extern __shared__ uint4 sm[];
  const uint32_t t = threadIdx.x, kk = p.kk, k = p.log_n;
  const uint32_t half = 1u << kk;
  const size_t base = (size_t)blockIdx.x << kk;
  fr_t* vec = p.dst[blockIdx.y];
  const uint32_t rounds = (kk + 2u) / 3u;
  fr_t x[8];
  for (uint32_t r = 0; r < rounds; r++) {
    const uint32_t P = dif_round_P(r, kk);
    if (r == 0) {
#pragma unroll
      for (int e = 0; e < 8; e++) x[e] = fr_load(vec + base + local_index(t, e, P));
    } else {
#pragma unroll
      for (int e = 0; e < 8; e++) x[e] = sm_get(sm, half, local_index(t, e, P));
    }
    if (r + 1 < rounds) {
      dif_round(x, p.tw, t, P, dif_round_qb(r, kk), 0u, 0u, k);
#pragma unroll
      for (int e = 0; e < 8; e++) sm_put(sm, half, local_index(t, e, P), x[e]);
      __syncthreads();
    } else {
      // P == 0: finish the inverse, shift, start the forward on the same registers.
      dif_round_p0(x, p.tw, dif_round_qb(r, kk), k);
#pragma unroll
      for (int e = 0; e < 8; e++) x[e] = fr_mul(x[e], fr_ldg(p.scale_tab + base + local_index(t, e, 0u)));
      dit_round_p0(x, p.tw2, 0, k);
    }
  }
  // decimation in time, rounds 1 .. rounds-1 (round 0 ran above)
  for (uint32_t r = 1; r < rounds; r++) {
    const uint32_t Pprev = dit_round_P(r - 1u, kk);
#pragma unroll
    for (int e = 0; e < 8; e++) sm_put(sm, half, local_index(t, e, Pprev), x[e]);
    __syncthreads();
    const uint32_t P = dit_round_P(r, kk);
#pragma unroll
    for (int e = 0; e < 8; e++) x[e] = sm_get(sm, half, local_index(t, e, P));
    dit_round(x, p.tw2, t, P, dit_round_qa(r, kk), 0u, 0u, k);
  }
  const uint32_t Plast = dit_round_P(rounds - 1u, kk);
#pragma unroll
  for (int e = 0; e < 8; e++) fr_store(vec + base + local_index(t, e, Plast), x[e]);
}

// ---------------------------------------------------------------------------------------
// k_ntt_dit: decimation-in-time passes over slice bits [c0, c0 + kk) (geometry as
// k_ntt_dif), src -> dst. Store epilogues:
//   SL_SCALE_TABLE: dst[i] = x * scale_tab[i];  SL_SCALE_CONST: dst[i] = x * kscale;
//   SL_JOIN: one block runs vectors 0, 1, 2 (a, b, c) of its slice in turn; a and b are
//   stored to dst[0], dst[1], and at c's store every thread re-reads the a and b values
//   it stored itself and writes h = a*b - c to h_mont and from_mont(h) to h_std
//   (the POINTWISE_CU join fused into the last transform's store).
// Launch: grid (n >> kk, vectors or 1 with SL_JOIN), block 2^(kk-3), shared 2^kk * 32.
__global__ void __launch_bounds__(256) k_ntt_dit(const __grid_constant__ SliceArgs p) {
  extern __shared__ uint4 sm[];
  const uint32_t t = threadIdx.x, kk = p.kk, c0 = p.c0, k = p.log_n;
  const uint32_t half = 1u << kk;
  const uint32_t s = blockIdx.x;
  const uint32_t low = s & ((1u << c0) - 1u);
  const size_t base = low + ((size_t)(s >> c0) << (c0 + kk));
  const uint32_t rounds = (kk + 2u) / 3u;
  const bool join = (p.mode & SL_JOIN) != 0u;
  const uint32_t nvec = join ? 3u : 1u;
  for (uint32_t vi = 0; vi < nvec; vi++) {
    const uint32_t v = join ? vi : blockIdx.y;
    const fr_t* src = p.src[v];
    fr_t* dst = p.dst[v];
    fr_t x[8];
    for (uint32_t r = 0; r < rounds; r++) {
      const uint32_t P = dit_round_P(r, kk);
      if (r == 0) {
        if (vi > 0) __syncthreads();  // the previous vector's last shared-memory reads
#pragma unroll
        for (int e = 0; e < 8; e++) x[e] = fr_load(src + base + ((size_t)local_index(t, e, P) << c0));
      } else {
#pragma unroll
        for (int e = 0; e < 8; e++) x[e] = sm_get(sm, half, local_index(t, e, P));
      }
      dit_round(x, p.tw, t, P, dit_round_qa(r, kk), low, c0, k);
      if (r + 1 < rounds) {
#pragma unroll
        for (int e = 0; e < 8; e++) sm_put(sm, half, local_index(t, e, P), x[e]);
        __syncthreads();
      } else {
#pragma unroll
        for (int e = 0; e < 8; e++) {
          const size_t i = base + ((size_t)local_index(t, e, P) << c0);
          if (join && v == 2u) {
            const fr_t a = fr_load(p.dst[0] + i);
            const fr_t b = fr_load(p.dst[1] + i);
            const fr_t h = fr_canon(fr_sub(fr_mul(a, b), x[e]));
            fr_store(p.h_mont + i, h);
            fr_store(p.h_std + i, fr_from_mont(h));
          } else {
            fr_t y = x[e];
            if (p.mode & SL_SCALE_TABLE) y = fr_mul(y, fr_ldg(p.scale_tab + i));
            if (p.mode & SL_SCALE_CONST) y = fr_mul(y, p.kscale);
            fr_store(dst + i, join ? y : fr_canon(y));
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// k_ntt_brev: the first decimation-in-time passes (bits 0 .. kk-1) of a natural-order
// forward transform, on the contiguous slice at blockIdx.x << kk: position i loads
// src[brev(i)] (the bit-reversal permutation absorbed into the load, as on the NTT_CU
// page), scaled by scale_tab[brev(i)] (SL_SCALE_TABLE) or kscale (SL_SCALE_CONST), and
// the result goes to dst (out of place: a block reads other blocks' elements).
// Launch: grid (n >> kk), block 2^(kk-3), shared 2^kk * 32.
__global__ void __launch_bounds__(256) k_ntt_brev(const __grid_constant__ SliceArgs p) {
  extern __shared__ uint4 sm[];
  const uint32_t t = threadIdx.x, kk = p.kk, k = p.log_n;
  const uint32_t half = 1u << kk;
  const size_t base = (size_t)blockIdx.x << kk;
  const uint32_t rounds = (kk + 2u) / 3u;
  fr_t x[8];
#pragma unroll
  for (int e = 0; e < 8; e++) {
    const uint32_t j = bitrev((uint32_t)base + local_index(t, e, 0u), k);
    x[e] = fr_load(p.src[0] + j);
    if (p.mode & SL_CHECK) check_canonical(x[e], p.err);
    if (p.mode & SL_SCALE_TABLE) x[e] = fr_mul(x[e], fr_ldg(p.scale_tab + j));
    if (p.mode & SL_SCALE_CONST) x[e] = fr_mul(x[e], p.kscale);
  }
  dit_round_p0(x, p.tw, dit_round_qa(0u, kk), k);
  for (uint32_t r = 1; r < rounds; r++) {
    const uint32_t Pprev = dit_round_P(r - 1u, kk);
#pragma unroll
    for (int e = 0; e < 8; e++) sm_put(sm, half, local_index(t, e, Pprev), x[e]);
    __syncthreads();
    const uint32_t P = dit_round_P(r, kk);
#pragma unroll
    for (int e = 0; e < 8; e++) x[e] = sm_get(sm, half, local_index(t, e, P));
    dit_round(x, p.tw, t, P, dit_round_qa(r, kk), 0u, 0u, k);
  }
  const uint32_t Plast = dit_round_P(rounds - 1u, kk);
#pragma unroll
  for (int e = 0; e < 8; e++) fr_store(p.dst[0] + base + local_index(t, e, Plast), x[e]);
}

}  // namespace g3h
