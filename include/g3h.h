/*
 * g3h: the Groth16 quotient-evaluation (H) path over the BN254 scalar field Fr, on one
 * NVIDIA GB300 (sm_103a).
 *
 * The operation ("snarkrs_gpu_kernels" pages: GATHER_CU, NTT_CU, POINTWISE_CU), for a
 * domain of n = 2^log_n points with generator omega and a primitive 2n-th root g, g^2 =
 * omega:
 *   1. gather   a_i = sum_j A[i,j] w_j,  b_i = sum_j B[i,j] w_j,  c_i = a_i * b_i
 *               (GATHER_CU, g16_gather_abc, and "why C is computed here")
 *   2. iNTT     x = n^-1 * DFT_{omega^-1}(v) for v in {a, b, c}   (NTT_CU header)
 *   3. shift    x_j <- x_j * g^j                                     (NTT_CU header)
 *   4. NTT      e = DFT_omega(x): the values on the odd coset g*<omega>
 *   5. join     h_i = e_a[i] * e_b[i] - e_c[i], no division by Z (POINTWISE_CU, "no
 *               division by Z(coset)"), written as h_mont (Montgomery) and h_std (the
 *               integer in [0, r)) in one pass (POINTWISE_CU, "two output buffers").
 * The 2^28-th root of unity is 5^((r-1)/2^28); omega = w^(2^(28-log_n)) and
 * g = w^(2^(27-log_n)).
 *
 * Also here: the H multiexp of the next stage (MSM_CU, stage 9: sum_i h_i P_i over the
 * BN254 curve group G1, with the standard-form h as scalars), g3h_msm_prepare / g3h_msm.
 *
 * Layout. A field element is 32 bytes: eight little-endian uint32 limbs, least
 * significant limb first, no padding. "Montgomery" means the limbs hold x * 2^256 mod r
 * (arkworks' internal form, POINTWISE_CU "two output buffers"). Every input element must
 * be canonical (< r); every output element is canonical. Vectors are contiguous arrays of
 * elements in natural index order.
 *
 * Pointers. By default every data pointer passed to a call is a HOST pointer: the call
 * copies inputs to the device, runs, copies outputs back and returns when they are in
 * place (pinned host memory makes the copies faster; pageable memory works). With
 * G3H_DEVICE_PTRS in `flags`, every data pointer of that call is a DEVICE pointer on the
 * context's device: the call only enqueues work on the context's stream and returns;
 * g3h_sync waits for it and reports errors found on the device. Device pointers must be
 * 16-byte aligned (elements move as 16-byte vectors; cudaMalloc and torch allocations
 * are); a call given one that is not returns G3H_E_INVAL and does nothing. The caller
 * owns every buffer it passes; the context owns its tables, its copy of the CSR matrices
 * and its scratch vectors.
 *
 * Errors. Every int-returning call returns G3H_OK (0) or a negative G3H_E_* code; no call
 * aborts or throws. A failed call leaves the context usable. Input elements that are not
 * canonical are reported as G3H_E_NONCANON: by the call itself for host pointers, by the
 * next g3h_sync for device pointers (outputs of that call are then unspecified).
 *
 * Threads. A context may be used by one host thread at a time; calls on one context run
 * in order on its stream. Separate contexts are independent.
 *
 * Failure injection, for tests of the failure paths (nothing is done to the GPU): with the
 * environment variable G3H_FAULT set to "alloc:N" the N-th device or pinned allocation the
 * library attempts fails as if out of memory (G3H_E_NOMEM); with "cuda:N" the N-th kernel
 * launch or copy is not issued and reports G3H_E_CUDA. N counts from 1 and restarts when
 * the value changes; unset, empty or malformed: no effect.
 */
#ifndef G3H_H
#define G3H_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define G3H_OK 0
#define G3H_E_INVAL (-1)    /* NULL pointer, device pointer not 16-byte aligned, bad size,
                               call not valid for this context */
#define G3H_E_NONCANON (-2) /* an input field element is >= r */
#define G3H_E_RANGE (-3)    /* log_n outside [0, 27]; CSR row pointers not monotone, not
                               starting at 0, or a column index >= n_wires */
#define G3H_E_NOMEM (-4)    /* device or pinned host allocation failed */
#define G3H_E_CUDA (-5)     /* a CUDA runtime call failed (no device, launch error, ...) */
#define G3H_E_POINT (-6)    /* a multiexp base point is not on its curve */

/* flags */
#define G3H_DEVICE_PTRS 0x1u  /* data pointers of this call are device pointers */
#define G3H_NOCHECK 0x2u      /* skip the canonical-input checks */
#define G3H_FUSED_JOIN 0x4u   /* compute_h / compute_h_abc: write h from the last forward
                                 kernel (the last of a slice's three blocks to finish
                                 joins that slice) instead of the join's own kernels after
                                 the forward transforms (POINTWISE_CU, g16_h_join): the
                                 product a * b once a and b are transformed, the reduction
                                 h = p - c once c is. The pages fuse to save a read of
                                 a, b, c; on GB300 these kernels are bound by the integer
                                 multiplier and the separate join measured faster, so it
                                 is the default. Same results. */

#define G3H_SERIALIZE 0x8u    /* compute_h / compute_h_abc: run the three vectors' transforms
                                 as one launch per phase on the context's stream instead
                                 of one stream per vector, so that every kernel runs alone
                                 (for per-kernel measurement). Same results. */

#define G3H_NO_GRAPH 0x10u    /* compute_h / compute_h_abc / compute_h_batch: issue the
                                 launches one by one instead of replaying the context's
                                 launch graph for these buffers and flags. Same results. */

#define G3H_MAX_LOG_N 27
#define G3H_MSM_MAX_LOG 24 /* at most 2^24 G1 bases per context */

typedef struct g3h_ctx g3h_ctx;

/* One R1CS coefficient matrix in CSR form (GATHER_CU, "why one thread per row": the CSR
 * sort). Row i holds the terms row_ptr[i] .. row_ptr[i+1]-1; term k has column col[k]
 * (a wire index < n_wires) and coefficient val[8k .. 8k+7] (Montgomery). Rows at or
 * beyond n_rows are empty. All three arrays are host memory, read only during
 * g3h_prepare. */
typedef struct {
  uint32_t n_rows;          /* <= 2^log_n */
  const uint32_t* row_ptr;  /* n_rows + 1 entries, row_ptr[0] = 0, non-decreasing */
  const uint32_t* col;      /* row_ptr[n_rows] entries */
  const uint32_t* val;      /* 8 * row_ptr[n_rows] limbs */
} g3h_csr;

/* Builds a context for the domain 2^log_n on CUDA device `device` (NTT_CU header: the
 * host builds the twiddle and shift tables once at prepare time and leaves them
 * resident). A and B are copied to the device. A and B may both be NULL: the context
 * then serves g3h_compute_h_abc, g3h_ntt, g3h_join and g3h_mul only. `stream` is a
 * cudaStream_t to run on (cudaStreamLegacy for the legacy default stream), or NULL for a
 * non-blocking stream the context creates and owns.
 * On success *out receives the context; on failure *out is NULL.
 * Errors: G3H_E_INVAL (out NULL, only one of A/B given, n_rows > 2^log_n, NULL array
 * with a non-zero size), G3H_E_RANGE, G3H_E_NONCANON (a coefficient >= r), G3H_E_NOMEM,
 * G3H_E_CUDA. */
int g3h_prepare(uint32_t log_n, uint32_t n_wires, const g3h_csr* A, const g3h_csr* B,
                int device, void* stream, g3h_ctx** out);

/* The whole path, steps 1-5: witness (n_wires elements, Montgomery) -> h_mont, h_std
 * (n elements each). Needs a context prepared with A and B. */
int g3h_compute_h(g3h_ctx* ctx, const uint32_t* witness, uint32_t* h_mont, uint32_t* h_std,
                  uint32_t flags);

/* Steps 2-5 on given evaluation vectors a, b, c (n elements each, Montgomery): the
 * pages' stages after the gather, for callers that already hold a, b and c. */
int g3h_compute_h_abc(g3h_ctx* ctx, const uint32_t* a, const uint32_t* b, const uint32_t* c,
                      uint32_t* h_mont, uint32_t* h_std, uint32_t flags);

/* Steps 1-5 for `count` witnesses over the same prepared matrices (batched H): witness i
 * is the n_wires elements at witnesses + 8*n_wires*i, its outputs the n elements at
 * h_mont + 8*n*i and h_std + 8*n*i. Consecutive witnesses run on up to three streams with
 * their own buffers (allocated by the first batched call and kept by the context), so
 * that one computation's gather and kernel tails overlap another's transforms and, with
 * host pointers, its copies (use pinned host memory for the copies to overlap). The batch
 * completes in the order of the context's stream. Results are those of count separate
 * g3h_compute_h calls. count = 0 does nothing. */
int g3h_compute_h_batch(g3h_ctx* ctx, uint32_t count, const uint32_t* witnesses,
                        uint32_t* h_mont, uint32_t* h_std, uint32_t flags);

/* Step 1 alone: a, b, c (n elements each, Montgomery) from the witness. */
int g3h_gather(g3h_ctx* ctx, const uint32_t* witness, uint32_t* a, uint32_t* b, uint32_t* c,
               uint32_t flags);

/* One transform of n elements in place (NTT_CU: the transform pair of the path):
 *   inverse = 0: x <- DFT_omega(y) where y = x, or y_j = x_j * g^j when coset != 0
 *   inverse = 1: x <- n^-1 DFT_omega^-1(x), then x_j <- x_j * g^-j when coset != 0
 * so an inverse call undoes the forward call with the same coset setting. */
int g3h_ntt(g3h_ctx* ctx, uint32_t* data, int inverse, int coset, uint32_t flags);

/* Step 5 alone (POINTWISE_CU g16_h_join): h = ea * eb - ec elementwise over n elements,
 * written in both encodings. */
int g3h_join(g3h_ctx* ctx, const uint32_t* ea, const uint32_t* eb, const uint32_t* ec,
             uint32_t* h_mont, uint32_t* h_std, uint32_t flags);

/* out_i = a_i * b_i (Montgomery product, canonical) for i < count: the product the gather
 * forms for C (GATHER_CU, "why C is computed here"), e.g. to build c = a * b for
 * g3h_compute_h_abc. */
int g3h_mul(g3h_ctx* ctx, const uint32_t* a, const uint32_t* b, uint32_t* out, size_t count,
            uint32_t flags);

/* out_i = in_i * R^-1 mod r for i < count: Montgomery form to standard form, the integer
 * in [0, r) (POINTWISE_CU g16_mont_to_std, the witness path's step before the MSMs: the
 * witness is uploaded once in Montgomery form for the gather, and its standard-form copy
 * for the MSM window digits is made on the device). in and out may be the same buffer
 * (converted in place); otherwise they must not overlap. Inputs must be canonical. Any
 * count; independent of the context's domain (count may exceed 2^log_n). With host
 * pointers the context's staging buffer grows to count elements. */
int g3h_mont_to_std(g3h_ctx* ctx, const uint32_t* in, uint32_t* out, size_t count,
                    uint32_t flags);

/* ---- The H multiexp over G1 (MSM_CU, stage 9: Pippenger over BN254 G1, taking the
 * standard-form h of g3h_compute_h as scalars) ----
 *
 * Curve y^2 = x^3 + 3 over F_q, q = 0x30644e72e131a029b85045b68181585d97816a916871ca8d3c
 * 208c16d87cfd47 (alt_bn128 of EIP-196). A base is an affine point of 16 limbs: x then y,
 * each eight little-endian 32-bit limbs in Montgomery form over F_q (x * 2^256 mod q),
 * canonical (< q); (0, 0) stands for the point at infinity. */

/* Loads n_bases G1 bases into the context (replacing any loaded before) and prepares them:
 * for each base P the 16 points 2^(16 w) P, w < 16, are computed on the device and kept
 * resident (1 KiB per base; 256 MiB for 2^18 bases), so that every later g3h_msm needs
 * one bucket pass for all its windows. Scratch for the multiexp is allocated here too:
 * 320 bytes per base (576 for G2) and about 30 MiB independent of n_bases (among it a
 * 128 KiB bucket-counter array per SM for the sort of the window digits). `bases`: 16 * n_bases limbs, host memory, or device
 * memory with G3H_DEVICE_PTRS (read only during the call). n_bases <= 2^G3H_MSM_MAX_LOG.
 * Synchronous. Returns G3H_E_NONCANON (a coordinate >= q), G3H_E_POINT (a base off the
 * curve), G3H_E_RANGE, G3H_E_NOMEM; on error no bases are loaded. n_bases = 0 unloads. */
int g3h_msm_prepare(g3h_ctx* ctx, const uint32_t* bases, uint32_t n_bases, uint32_t flags);

/* result = sum_{i < count} s_i * P_i, P_i the first count loaded bases (count <= n_bases).
 * scalars: 8 * count limbs, each scalar in standard form (the integer, < r; the h_std
 * output of g3h_compute_h, not h_mont: a window digit of a Montgomery representative is a
 * digit of s * R). result: 24 limbs, the sum in Jacobian coordinates (X, Y, Z),
 * x = X / Z^2, y = Y / Z^3, each canonical Montgomery over F_q; the point at infinity is
 * written as X = Y = Z = 0. Host pointers (synchronous) or, with G3H_DEVICE_PTRS, device
 * pointers (asynchronous on the context's stream; errors at g3h_sync). Scalars >= r give
 * G3H_E_NONCANON unless G3H_NOCHECK. count = 0 writes infinity. */
int g3h_msm(g3h_ctx* ctx, const uint32_t* scalars, uint32_t count, uint32_t* result,
            uint32_t flags);

/* The same over G2, the twist E': y^2 = x^3 + 3/(9 + u) over F_q2 = F_q[u]/(u^2 + 1)
 * (EIP-197; MSM_CU stage 7, the witness multiexp of the B query). An F_q2 element is
 * c0 + c1 u as two F_q elements (16 limbs, c0 first, each Montgomery, canonical); a base is
 * x then y (32 limbs), (0, 0) the point at infinity; the result is Jacobian (X, Y, Z),
 * 48 limbs, infinity as zeros. Bases are points of E'(F_q2) (not checked to lie in the
 * order-r subgroup); each is checked to be canonical and on the twist (G3H_E_POINT).
 * 2 KiB of prepared data per base. Otherwise as g3h_msm_prepare / g3h_msm. */
int g3h_msm_g2_prepare(g3h_ctx* ctx, const uint32_t* bases, uint32_t n_bases, uint32_t flags);
int g3h_msm_g2(g3h_ctx* ctx, const uint32_t* scalars, uint32_t count, uint32_t* result,
               uint32_t flags);

/* Steps 2-5 like g3h_compute_h_abc, for callers that cannot allocate device memory: a
 * framework whose caching allocator must own every device byte, or a latency-critical
 * path that cannot take cudaMalloc's device-wide synchronisation. It has no counterpart
 * on the pages; it is this library's own addition.
 *
 * It needs no context and allocates nothing: its working vectors and domain tables live in
 * one fixed device array of 14 MiB inside the library, reserved on every GPU that loads
 * the library until the process exits. Hence log_n <= 16 (domains up to 2^16 points);
 * larger domains return G3H_E_RANGE without doing anything.
 *
 * a, b, c (inputs, n elements each, Montgomery, canonical; NOT checked) and h_mont, h_std
 * (outputs, n elements each) are device pointers on the current CUDA device, each 16-byte
 * aligned; `stream` is the cudaStream_t to run on (NULL: the legacy default stream). The
 * call enqueues the work and returns; the outputs are ready when the stream reaches that
 * point.
 *
 * The first call on a device looks up the array's device address (a one-time set-up with
 * that device current); make that first call before any stream capture begins. Every call
 * first enqueues three small kernels that check, on the GPU, whether the array holds the
 * tables of this log_n, and rebuild them if it does not (the first call for a domain, or
 * the first after a call for another domain, takes about a millisecond more). All calls
 * on a device share the array and it keeps the last call's contents, so calls that overlap
 * on the GPU (on different streams, or from different threads without ordering) race and
 * give wrong results: order them on one stream.
 * Returns G3H_OK, G3H_E_INVAL (a NULL pointer, or one not 16-byte aligned), G3H_E_RANGE
 * (log_n > 16) or G3H_E_CUDA. */
int g3h_compute_h_abc_static(uint32_t log_n, const uint32_t* a, const uint32_t* b,
                             const uint32_t* c, uint32_t* h_mont, uint32_t* h_std,
                             void* stream);

/* Waits for all work enqueued on the context's stream; returns G3H_E_NONCANON (or
 * G3H_E_POINT) if a device-side input check failed since the last sync (and clears it),
 * G3H_E_CUDA on a CUDA error. */
int g3h_sync(g3h_ctx* ctx);

/* Frees the context and everything it owns (waits for its stream first). NULL is a
 * no-op. */
void g3h_destroy(g3h_ctx* ctx);

/* A static string describing an error code. */
const char* g3h_strerror(int code);

/* Domain of a context: log_n and n_wires, or G3H_E_INVAL for NULL. */
int g3h_info(const g3h_ctx* ctx, uint32_t* log_n, uint32_t* n_wires);

/* Per-kernel device timing, for measurement: with `enable` != 0 the context records a CUDA
 * event pair on its stream around every kernel it launches, until disabled. Enabling
 * clears the previous records. */
int g3h_timing_enable(g3h_ctx* ctx, int enable);

/* Aggregates the recorded launches per kernel name after waiting for the stream: up to
 * `max` entries (name, number of launches, summed device milliseconds); *count receives
 * the number of distinct kernels. Names are static strings; an H records "gather_a",
 * "gather_b", "ntt_dif", "ntt_mid", "ntt_dit", "prejoin" (the join's products) and "join"
 * (its reduction), or "ntt_dit_join" with G3H_FUSED_JOIN ("gather" and "small_quotient"
 * on domains of at most 2^5 points); g3h_ntt "ntt_brev" and "ntt_dit" (or "small_ntt"); a
 * multiexp its "msm_*" kernels. */
typedef struct {
  const char* name;
  uint32_t launches;
  double ms;
} g3h_kernel_time;
int g3h_timing_read(g3h_ctx* ctx, g3h_kernel_time* out, int max, int* count);

/* For measurement: the throughput of the device's integer multiply pipe in the unit of
 * the library's roofline, 32-bit IMAD results per second. A probe kernel runs independent
 * chains of 32-bit multiply-adds (mad.lo.u32) on every SM for a few milliseconds, timed
 * with CUDA events on the context's stream (best of three runs after a warm-up).
 * Synchronous. Returns G3H_E_INVAL (NULL), G3H_E_NOMEM or G3H_E_CUDA. */
int g3h_measure_imad(g3h_ctx* ctx, double* results_per_s);

/* The same probe for each kind of 32-bit integer multiply the field arithmetic issues:
 * *per_s receives the thread-level instructions per second of independent chains of
 *   G3H_MUL_LO:   mad.lo.u32   (the low word of a 32 x 32 product; = g3h_measure_imad)
 *   G3H_MUL_HI:   mad.hi.u32   (the high word)
 *   G3H_MUL_WIDE: mad.wide.u32 (the full 64-bit product, with a 64-bit addend)
 * so that the cost of a full product can be stated in units of the 32-bit rate (the
 * roofline's denominator) instead of assumed. Synchronous. Returns G3H_E_INVAL (NULL
 * argument or unknown kind), G3H_E_NOMEM or G3H_E_CUDA. */
#define G3H_MUL_LO 0
#define G3H_MUL_HI 1
#define G3H_MUL_WIDE 2
int g3h_measure_int_mul(g3h_ctx* ctx, int kind, double* per_s);

#ifdef __cplusplus
}
#endif

#endif /* G3H_H */
