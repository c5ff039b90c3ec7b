// The C ABI of include/g3h.h: context, resident tables, launch plans.
//
// Work per H computation on a domain of 2^k >= 2^6 points (two slice levels, k = lo + hi;
// three levels for k > 22; a slice is at most 2^11 elements), per vector a, b, c:
//   k_gather_rows  (a, b)    the CSR rows of A and of B against the witness
//   k_ntt_dif                inverse passes on the top bits, strided slices; for c the
//                            load forms c = a * b (compute_h_abc loads a, b, c)
//   k_ntt_mid                inverse passes on the low bits, shift g^brev(p)/n, forward
//                            passes on the low bits, contiguous slices
//   k_ntt_dit                forward passes on the top bits
//   k_join                   h = a*b - c in both encodings
// The three vectors' kernels run on three streams (fork/join events), the whole sequence
// captured once into a CUDA graph per set of pointers and replayed; G3H_SERIALIZE runs the
// three vectors as one launch per phase on one stream, G3H_FUSED_JOIN writes h from the last
// forward kernel instead of k_join. Slice kernels come in three builds (ntt.cuh, SliceCfg):
// radix-4 pass pairs for slices of 2^9 elements and more, radix-2 passes below. Batched
// calls on domains of 2^6 .. 2^16 points run a chunk of witnesses per launch (the witness
// index in the grid's z or y dimension) on two alternating "z lanes".
//
// The multiexps over G1 and G2 (msm.cuh) keep their prepared bases in the context.
// Every computing entry point and every stage of an H is an NVTX range; the environment
// variable G3H_FAULT injects allocation or launch failures on the host (inject_fault).
#include <cuda_runtime.h>

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/g3h.h"
#include "kernels.cuh"
#include "msm.cuh"

using namespace g3h;

namespace {

const uint32_t kModulus[8] = {G3H_R0, G3H_R1, G3H_R2, G3H_R3, G3H_R4, G3H_R5, G3H_R6, G3H_R7};

// The kernels move elements as 16-byte vectors, so a device pointer that is not 16-byte
// aligned would fault the device; such a call is refused instead (G3H_E_INVAL).
bool misaligned(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 15u) return true;
  return false;
}

bool host_canonical(const uint32_t* x) {
  for (int i = 7; i >= 0; i--) {
    if (x[i] < kModulus[i]) return true;
    if (x[i] > kModulus[i]) return false;
  }
  return false;  // equal to r
}

// Host-side fault injection, for tests of the failure paths (no GPU fault is ever made):
// with the environment variable G3H_FAULT set to "alloc:N", the N-th device or pinned
// allocation the library attempts fails as if the device were out of memory (the call
// returns G3H_E_NOMEM); with "cuda:N", the N-th kernel launch or copy it issues is not
// issued and reports a CUDA error (G3H_E_CUDA). N counts from 1 and the count restarts
// whenever the variable's value changes; unset, empty or malformed: nothing is injected.
enum class Fault { alloc, cuda };

bool inject_fault(Fault kind) {
  static std::mutex mu;
  static std::string spec;
  static unsigned long long seen[2] = {0, 0};
  const char* env = std::getenv("G3H_FAULT");
  if (!env || !*env) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (spec != env) {
    spec = env;
    seen[0] = seen[1] = 0;
  }
  const char* name = kind == Fault::alloc ? "alloc:" : "cuda:";
  const size_t len = std::strlen(name);
  if (spec.compare(0, len, name) != 0) return false;
  char* end = nullptr;
  const unsigned long long n = std::strtoull(spec.c_str() + len, &end, 10);
  if (!end || *end || n == 0) return false;
  return ++seen[kind == Fault::alloc ? 0 : 1] == n;
}

// An NVTX range for the duration of a scope (shown by profilers that record NVTX).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

struct TimedLaunch {
  const char* name;
  cudaEvent_t e0, e1;
};

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

// Slice levels of a transform of 2^k points: level 0 is the contiguous low slice.
struct Plan {
  int levels;
  uint32_t kk[3];
  uint32_t c0[3];
};

Plan plan_for(uint32_t k) {
  Plan p{};
  if (k <= 22) {
    const uint32_t lo = (k + 1) / 2;
    p.levels = 2;
    p.kk[0] = lo;
    p.kk[1] = k - lo;
    p.c0[0] = 0;
    p.c0[1] = lo;
  } else {
    const uint32_t lo = (k + 2) / 3, rest = k - lo, mid = (rest + 1) / 2;
    p.levels = 3;
    p.kk[0] = lo;
    p.kk[1] = mid;
    p.kk[2] = rest - mid;
    p.c0[0] = 0;
    p.c0[1] = lo;
    p.c0[2] = lo + mid;
  }
  return p;
}

}  // namespace

// One set of per-computation buffers and the stream that uses them. Lane 0 is the
// context's own stream and buffers; batched calls add lanes so that consecutive
// computations overlap (one lane's gather and kernel tails run beside another's NTTs).
struct Lane {
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  fr_t* abc = nullptr;        // 3n: a | b | c while they are transformed
  fr_t* ab_in = nullptr;      // 2n: the gather's a | b
  uint32_t* counters = nullptr;  // fused join: one per top-level slice, kept zero
  fr_t* stage = nullptr;      // host-pointer calls: witness | h_mont | h_std
  size_t stage_elems = 0;
  cudaEvent_t done = nullptr;
  // vectors b and c run on two more streams; events order them against the lane's stream
  cudaStream_t aux[2] = {nullptr, nullptr};
  cudaStream_t cap = nullptr;  // launch graphs are captured here (the caller's stream may
                               // be the legacy default stream, which cannot be captured)
  cudaEvent_t ev_fork = nullptr, ev_ga = nullptr, ev_gb = nullptr;
  cudaEvent_t ev_end[2] = {nullptr, nullptr};
  cudaEvent_t ev_a = nullptr, ev_p = nullptr;  // vector a transformed; the join's product formed
};

int make_lane_streams(Lane& l) {
  for (int i = 0; i < 2; i++)
    if (cudaStreamCreateWithFlags(&l.aux[i], cudaStreamNonBlocking) != cudaSuccess)
      return G3H_E_CUDA;
  if (cudaStreamCreateWithFlags(&l.cap, cudaStreamNonBlocking) != cudaSuccess) return G3H_E_CUDA;
  cudaEvent_t* evs[] = {&l.ev_fork, &l.ev_ga,     &l.ev_gb, &l.ev_end[0],
                        &l.ev_end[1], &l.ev_a, &l.ev_p};
  for (cudaEvent_t* e : evs)
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return G3H_E_CUDA;
  return G3H_OK;
}

void free_lane_streams(Lane& l) {
  for (int i = 0; i < 2; i++)
    if (l.aux[i]) cudaStreamDestroy(l.aux[i]);
  if (l.cap) cudaStreamDestroy(l.cap);
  cudaEvent_t evs[] = {l.ev_fork, l.ev_ga, l.ev_gb, l.ev_end[0], l.ev_end[1], l.ev_a, l.ev_p};
  for (cudaEvent_t e : evs)
    if (e) cudaEventDestroy(e);
}

// Frees a lane's buffers, streams and events (any of them may be missing).
void free_lane(Lane& l) {
  void* lb[] = {l.abc, l.ab_in, l.counters, l.stage};
  for (void* b : lb)
    if (b) cudaFree(b);
  if (l.done) cudaEventDestroy(l.done);
  free_lane_streams(l);
  if (l.own_stream && l.stream) cudaStreamDestroy(l.stream);
  l = Lane();
}

// Batched H on small and middle domains: a chunk of up to `z` witnesses runs as one
// launch per phase, the witness index in the grid's z dimension (slice kernels) or y
// dimension (gather, join), so that a few thousand-point domains fill the GPU. Two such
// lanes alternate between chunks, each with its own stream and buffers, so that one
// chunk's copies (host-pointer calls) overlap the other's kernels.
struct ZLane {
  cudaStream_t stream = nullptr;
  fr_t* ab_in = nullptr;  // z x 2n: the gathers' a | b per witness
  fr_t* abc = nullptr;    // z x 3n: a | b | c per witness while they are transformed
  fr_t* stage = nullptr;  // z x (n_wires + 2n): witnesses | h_mont | h_std (host pointers)
  cudaEvent_t done = nullptr;
};

void free_zlane(ZLane& l) {
  void* b[] = {l.ab_in, l.abc, l.stage};
  for (void* x : b)
    if (x) cudaFree(x);
  if (l.done) cudaEventDestroy(l.done);
  if (l.stream) cudaStreamDestroy(l.stream);
  l = ZLane();
}

// The buffers of one group's multiexp (bytes as raw device memory, typed at use).
struct MsmState {
  uint32_t n = 0;                    // bases prepared
  uint32_t slots = 0;                // resident threads of the accumulation kernel
  void* table = nullptr;             // 16 affine points per base: 2^(16 w) P_i
  uint32_t* entries = nullptr;       // 16 per base
  uint32_t* counts = nullptr;        // per bucket | long-run list (count, indices)
  uint32_t* offsets = nullptr;       // per bucket + 1
  uint32_t sort_blocks = 0;          // blocks of the counting sort (one per SM)
  uint32_t* block_counts = nullptr;  // per sort block and bucket
  void* buckets = nullptr;           // per bucket
  void* spill = nullptr;             // head | tail parts, (n + 1) each
  void* groups = nullptr;            // U | V, kMsmPairs each
  void* parts = nullptr;             // chunk sums | the parts and the ones' sum | ones' block sums
  void* result = nullptr;            // Jacobian X, Y, Z
};

struct g3h_ctx {
  int device = 0;
  int sm_count = 1;
  int smem_per_sm = 0, smem_reserved = 0;  // shared memory of an SM, reserved per block
  int8_t carveout[4][32] = {};             // slice launches' carveout (percent), 0: unset
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  uint32_t log_n = 0, n_wires = 0;
  size_t n = 0;
  bool has_csr = false;
  uint32_t n_rows_a = 0, n_rows_b = 0;
  uint32_t *d_rpa = nullptr, *d_cola = nullptr, *d_rpb = nullptr, *d_colb = nullptr;
  fr_t *d_vala = nullptr, *d_valb = nullptr;
  fr_t* d_consts = nullptr;  // omega, omega^-1, g, g^-1, n^-1, 1 (Montgomery)
  // constant tables in the (w, w') form of the constant multiply
  fr_const_t *d_tw_fwd = nullptr, *d_tw_inv = nullptr, *d_shift_br = nullptr;
  fr_const_t *d_coset_fwd = nullptr, *d_coset_inv = nullptr;
  bool coset_ready = false;  // both coset tables allocated and built
  fr_const_t* d_ninv = nullptr;  // n^-1
  fr_t* d_abc = nullptr;  // 3n scratch: a | b | c while they are transformed
  fr_t* d_ab_in = nullptr;  // 2n: the gather's a | b, read by the first inverse kernel
  uint32_t* d_counters = nullptr;  // per top-level slice, for the fused join (kept zero)
  fr_t* d_stage = nullptr;
  size_t stage_elems = 0;
  uint32_t* d_err = nullptr;
  fr_const_t h_ninv;  // host copy of n^-1, passed by value to kernels
  Lane own;  // the auxiliary streams and events of lane 0 (its buffers are the fields above)
  uint32_t* h_err = nullptr;  // pinned host copy of the device error word
  // Launch graphs of quotient(): the per-H launches of one lane with one set of pointers
  // and flags, captured once and replayed (fewer host calls per H, one graph launch).
  struct Graph {
    cudaStream_t stream;
    const void* ptr[6];
    uint32_t flags;
    cudaGraphExec_t exec;
  };
  std::vector<Graph> graphs;
  std::vector<Lane> extra_lanes;  // batched calls: lanes 1, 2, ...
  ZLane zl[2];                    // batched calls on small and middle domains
  uint32_t z_chunk = 0;           // witnesses per chunk the z lanes hold (0: none yet)
  bool z_staged = false;          // the z lanes hold staging buffers
  cudaEvent_t batch_start = nullptr;
  // multiexps over G1 and G2 (g3h_msm_prepare / g3h_msm and the _g2 pair)
  MsmState msm1, msm2;
  bool timing = false;
  std::vector<TimedLaunch> launches;
  std::vector<cudaEvent_t> event_pool;
  size_t events_used = 0;
};

namespace {

int raw_alloc(void** p, size_t bytes) {
  *p = nullptr;
  if (inject_fault(Fault::alloc)) return G3H_E_NOMEM;
  return cudaMalloc(p, std::max<size_t>(bytes, 1)) == cudaSuccess ? G3H_OK : G3H_E_NOMEM;
}

template <class T>
int dalloc(T** p, size_t count) {
  void* q = nullptr;
  const int rc = raw_alloc(&q, std::max<size_t>(count, 1) * sizeof(T));
  *p = (T*)q;
  return rc;
}

void msm_free(MsmState& m) {
  void* bufs[] = {m.table, m.entries, m.counts, m.offsets, m.block_counts,
                  m.buckets, m.spill, m.groups, m.parts, m.result};
  for (void* b : bufs)
    if (b) cudaFree(b);
  m = MsmState();
}

void release(g3h_ctx* c) {
  msm_free(c->msm1);
  msm_free(c->msm2);
  void* bufs[] = {c->d_rpa,      c->d_cola,     c->d_rpb,      c->d_colb,        c->d_vala,
                  c->d_valb,     c->d_consts,   c->d_tw_fwd,   c->d_tw_inv,      c->d_shift_br,
                  c->d_coset_fwd, c->d_coset_inv, c->d_abc,    c->d_stage,       c->d_err,
                  c->d_ab_in,    c->d_counters, c->d_ninv};
  for (void* b : bufs)
    if (b) cudaFree(b);
  for (cudaEvent_t e : c->event_pool) cudaEventDestroy(e);
  for (Lane& l : c->extra_lanes) free_lane(l);
  for (ZLane& l : c->zl) free_zlane(l);
  free_lane_streams(c->own);
  if (c->batch_start) cudaEventDestroy(c->batch_start);
  for (auto& g : c->graphs) cudaGraphExecDestroy(g.exec);
  if (c->h_err) cudaFreeHost(c->h_err);
  if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
}

cudaEvent_t take_event(g3h_ctx* c) {
  if (c->events_used == c->event_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    c->event_pool.push_back(e);
  }
  return c->event_pool[c->events_used++];
}

template <class F>
int run_on(g3h_ctx* c, cudaStream_t st, const char* name, F&& launch) {
  if (inject_fault(Fault::cuda)) return G3H_E_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (c->timing) {
    e0 = take_event(c);
    e1 = take_event(c);
    if (e0 && e1) cudaEventRecord(e0, st);
  }
  launch();
  const cudaError_t err = cudaGetLastError();
  if (c->timing && e0 && e1) {
    cudaEventRecord(e1, st);
    c->launches.push_back({name, e0, e1});
  }
  return err == cudaSuccess ? G3H_OK : G3H_E_CUDA;
}

template <class F>
int run(g3h_ctx* c, const char* name, F&& launch) {
  return run_on(c, c->stream, name, static_cast<F&&>(launch));
}

unsigned blocks_for(size_t count, unsigned per) { return (unsigned)((count + per - 1) / per); }

enum class Slice { dif, mid, dit, brev };

// The build of a slice kernel for slices of 2^kk elements, and its threads per block: one
// per butterfly of a radix-2 pass, one per group of four of a radix-4 pass pair, up to
// the build's block size.
void (*slice_kernel(Slice which, uint32_t kk, uint32_t* threads))(SliceArgs) {
  if (kk >= kCfg2MinSliceBits) {
    *threads = std::min(1u << (kk - 2u), SliceCfg<2>::threads);
    switch (which) {
      case Slice::dif: return k_ntt_dif<2>;
      case Slice::mid: return k_ntt_mid<2>;
      case Slice::dit: return k_ntt_dit<2>;
      default: return k_ntt_brev<2>;
    }
  }
  const bool r4 = kk >= kRadix4MinSliceBits && kk <= kRadix4MaxSliceBits && kk >= 2;
  *threads = r4 ? std::min(1u << (kk - 2u), SliceCfg<1>::threads)
                : std::min(1u << (kk - 1u), SliceCfg<0>::threads);
  switch (which) {
    case Slice::dif: return r4 ? k_ntt_dif<1> : k_ntt_dif<0>;
    case Slice::mid: return r4 ? k_ntt_mid<1> : k_ntt_mid<0>;
    case Slice::dit: return r4 ? k_ntt_dit<1> : k_ntt_dit<0>;
    default: return r4 ? k_ntt_brev<1> : k_ntt_brev<0>;
  }
}

// Launches a slice kernel over the n >> kk slices of nvec vectors (grid rows) and nz
// batch layers. With three vectors per launch, the three blocks of a slice are adjacent
// in launch order (SliceArgs::vfast): they read the same twiddles and scale entries, which
// then come from L2 for two of them.
//
// On domains whose slices are all of at most 2^9 elements (2^18 and below), each launch
// asks for the split of the SM's L1 / shared memory that holds just the shared memory of as
// many blocks as can be resident, the rest left to L1, where the twiddle and shift loads
// hit: 2^18 H 0.2783 -> 0.2775 ms (one fixed 40 % of the maximum for all slice kernels:
// 0.2811 -> 0.2798; all of it: 0.2870). With larger slices the same rule measured slower
// (2^22 H 4.63 -> 4.87 ms), and so did asking it only for a domain's 2^9 slices while its
// 2^10 slices ran beside them with the driver's split (2^19 H 0.504 -> 0.513 ms): such
// domains keep the driver's choice for every launch. Every launch but the bit-reversed
// load's may also begin while the previous kernel on its stream finishes (launch_pdl).
constexpr uint32_t kCarveoutMaxSliceBits = 9;

int launch_slice_on(g3h_ctx* c, cudaStream_t st, const char* name, Slice which,
                    const SliceArgs& a_in, unsigned nvec, unsigned nz = 1) {
  uint32_t threads = 0;
  void (*kern)(SliceArgs) = slice_kernel(which, a_in.kk, &threads);
  SliceArgs a = a_in;
  const unsigned slices = (unsigned)(c->n >> a.kk);
  a.vfast = (nvec == 3u && !(a.mode & SL_JOIN)) ? 1u : 0u;
  const dim3 grid(a.vfast ? 3u * slices : slices, a.vfast ? 1u : nvec, nz);
  const size_t smem = (size_t)32 << a.kk;
  const Plan pl = plan_for(c->log_n);
  bool carve = true;
  for (int l = 0; l < pl.levels; l++) carve = carve && pl.kk[l] <= kCarveoutMaxSliceBits;
  int8_t& pct = c->carveout[(int)which][a.kk & 31u];
  if (carve && pct == 0) {
    int resident = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kern, (int)threads, smem) !=
            cudaSuccess ||
        resident < 1 || c->smem_per_sm <= 0)
      return G3H_E_CUDA;
    const size_t need = (size_t)resident * (smem + (size_t)c->smem_reserved);
    pct = (int8_t)std::min<size_t>(100, (need * 100 + c->smem_per_sm - 1) / c->smem_per_sm);
    if (pct < 1) pct = 1;
  }
  return run_on(c, st, name, [&] {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    unsigned na = 0;
    if (carve) {
      at[na].id = cudaLaunchAttributePreferredSharedMemoryCarveout;
      at[na++].val.sharedMemCarveout = (unsigned)pct;
    }
    if (which != Slice::brev) {  // brev reads what a copy or the caller's work wrote
      at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[na++].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = at;
    cfg.numAttrs = na;
    cudaLaunchKernelEx(&cfg, kern, a);
  });
}

int launch_slice(g3h_ctx* c, const char* name, Slice which, const SliceArgs& a, unsigned nvec) {
  return launch_slice_on(c, c->stream, name, which, a, nvec);
}

int set_smem_limits() {
  const int bytes = 32 << 11;  // the largest slice, 2^11 elements
  void (*kerns[])(SliceArgs) = {k_ntt_dif<0>,  k_ntt_mid<0>, k_ntt_dit<0>, k_ntt_brev<0>,
                                k_ntt_dif<1>,  k_ntt_mid<1>, k_ntt_dit<1>, k_ntt_brev<1>,
                                k_ntt_dif<2>,  k_ntt_mid<2>, k_ntt_dit<2>, k_ntt_brev<2>};
  for (auto k : kerns)
    if (cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
      return G3H_E_CUDA;
  // the multiexp's counting sort: a counter per bucket in each block
  const void* sort_kerns[] = {(const void*)k_msm_count, (const void*)k_msm_scatter};
  for (auto k : sort_kerns)
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMsmSortSmem) !=
        cudaSuccess)
      return G3H_E_CUDA;
  return G3H_OK;
}

int build_table(g3h_ctx* c, fr_const_t* tab, size_t count, int base, int scale, uint32_t brev) {
  if (count == 0) return G3H_OK;
  return run(c, "tables", [&] {
    k_pow_table<<<blocks_for(count, 256), 256, 0, c->stream>>>(tab, count, c->d_consts, base,
                                                                scale, brev);
  });
}

// The coset tables g^brev(p) (forward, at position p) and g^-j / n (inverse, at j),
// allocated and built by the first coset transform.
// They count as present only once both are allocated and their builds are enqueued; a
// failure frees what was allocated, so the next call starts over.
int ensure_coset_tables(g3h_ctx* c) {
  if (c->coset_ready) return G3H_OK;
  int rc = G3H_OK;
  if (!c->d_coset_fwd) rc = dalloc(&c->d_coset_fwd, c->n);
  if (rc == G3H_OK && !c->d_coset_inv) rc = dalloc(&c->d_coset_inv, c->n);
  // g^j stored at the bit-reversed position brev(j): the first kernel of a forward coset
  // transform loads position p from data[brev(p)] and reads its scale contiguously
  if (rc == G3H_OK) rc = build_table(c, c->d_coset_fwd, c->n, 2, -1, c->log_n);
  if (rc == G3H_OK) rc = build_table(c, c->d_coset_inv, c->n, 3, 4, 0);
  if (rc != G3H_OK) {
    cudaStreamSynchronize(c->stream);
    if (c->d_coset_fwd) cudaFree(c->d_coset_fwd);
    if (c->d_coset_inv) cudaFree(c->d_coset_inv);
    c->d_coset_fwd = c->d_coset_inv = nullptr;
    return rc;
  }
  c->coset_ready = true;
  return G3H_OK;
}

int ensure_stage(g3h_ctx* c, size_t elems) {
  if (c->stage_elems >= elems) return G3H_OK;
  if (c->d_stage) cudaFree(c->d_stage);
  c->d_stage = nullptr;
  c->stage_elems = 0;
  if (dalloc(&c->d_stage, elems) != G3H_OK) return G3H_E_NOMEM;
  c->stage_elems = elems;
  return G3H_OK;
}

int copy_on(cudaStream_t st, void* dst, const void* src, size_t bytes, cudaMemcpyKind kind) {
  if (bytes == 0) return G3H_OK;
  if (inject_fault(Fault::cuda)) return G3H_E_CUDA;
  return cudaMemcpyAsync(dst, src, bytes, kind, st) == cudaSuccess ? G3H_OK : G3H_E_CUDA;
}

int h2d(g3h_ctx* c, void* dst, const void* src, size_t bytes) {
  return copy_on(c->stream, dst, src, bytes, cudaMemcpyHostToDevice);
}

int d2h(g3h_ctx* c, void* dst, const void* src, size_t bytes) {
  return copy_on(c->stream, dst, src, bytes, cudaMemcpyDeviceToHost);
}

// Waits for the stream and reports (then clears) the device-side input check word.
int finish(g3h_ctx* c) {
  // the error word comes back in the same stream, so one synchronisation covers both
  if (cudaMemcpyAsync(c->h_err, c->d_err, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                      c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess)
    return G3H_E_CUDA;
  if (*c->h_err) {
    const uint32_t e = *c->h_err;
    *c->h_err = 0;
    if (cudaMemsetAsync(c->d_err, 0, sizeof(uint32_t), c->stream) != cudaSuccess)
      return G3H_E_CUDA;
    return (e & kMsmErrPoint) ? G3H_E_POINT : G3H_E_NONCANON;
  }
  return G3H_OK;
}

SliceArgs base_args(g3h_ctx* c, uint32_t flags) {
  SliceArgs a;
  std::memset(&a, 0, sizeof(a));
  a.err = c->d_err;
  a.log_n = c->log_n;
  (void)flags;
  return a;
}

int gather_on(g3h_ctx* c, cudaStream_t st, const fr_t* w, fr_t* a, fr_t* b, fr_t* cc,
              uint32_t flags);

Lane lane0(g3h_ctx* c) {
  Lane l = c->own;
  l.stream = c->stream;
  l.abc = c->d_abc;
  l.ab_in = c->d_ab_in;
  l.counters = c->d_counters;
  return l;
}

// Steps 2-5 on device vectors a, b, c -> h_mont, h_std (device), on a lane's stream and
// buffers. a, b, c may be the lane's scratch vectors. With a witness w (device) instead,
// steps 1-5: the gather writes a and b and the first inverse kernel forms c = a * b at
// its load (a, b, c are then ignored).
//
// The three vectors are independent until the join: vector v runs on vs[v], so one
// vector's gather latency and kernel tails overlap the others' transforms. With
// G3H_SERIALIZE everything runs on the lane's stream, one launch per phase covering the
// three vectors (grid rows 0, 1, 2), so each kernel runs alone. quotient_vectors issues
// the work of the forked streams; quotient_launches forks them and always joins them
// back, also when a launch fails, so that no work is left unjoined (and a stream capture
// in progress ends cleanly).
// A kernel launch that may begin while the previous kernel on the stream finishes
// (programmatic dependent launch; the kernel waits for it in wait_prior_grid before reading
// its output). Measured with the slice kernels launched the same way: 2^16 H 0.087 ->
// 0.085 ms, 2^22 coset NTT 0.8765 -> 0.8735 ms, 2^18 H within noise (0.2773 -> 0.2768).
template <class... K, class... A>
void launch_pdl(unsigned blocks, unsigned threads, cudaStream_t st, void (*kern)(K...),
                A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kern, args...);
}

fr_t* s_of(const Lane& ln, size_t n, int v) { return ln.abc + (size_t)v * n; }

int quotient_vectors(g3h_ctx* c, const Lane& ln, const cudaStream_t* vs, bool serial,
                     const fr_t* a, const fr_t* b, const fr_t* cc, const fr_t* w, fr_t* hm,
                     fr_t* hs, uint32_t flags) {
  const uint32_t k = c->log_n;
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  const size_t n = c->n;
  const uint32_t nv = serial ? 1u : 3u;    // launches per phase
  const unsigned rows = serial ? 3u : 1u;  // vectors per launch
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  int rc = G3H_OK;
  if (w) {
    // a and b by the gather, A on the stream of a, B on the stream of b; c = a * b is
    // formed by c's first inverse kernel at its load, once both are done. B's gather (the
    // longer rows) is issued first, so its blocks take the SMs first: 2^18 H 0.2771 ->
    // 0.2755 ms against A's first
    NvtxRange range("g3h gather");
    fr_t* ab = ln.ab_in;
    const uint32_t nn = (uint32_t)n;
    rc = run_on(c, vs[1], "gather_b", [&] {
      k_gather_rows<<<blocks_for(n, 256), 256, 0, vs[1]>>>(
          c->d_rpb, c->d_colb, c->d_valb, w, c->n_rows_b, nn, c->n_wires, ab + n, check,
          c->d_err, 0, 0);
    });
    if (rc == G3H_OK)
      rc = run_on(c, vs[0], "gather_a", [&] {
        k_gather_rows<<<blocks_for(n, 256), 256, 0, vs[0]>>>(
            c->d_rpa, c->d_cola, c->d_vala, w, c->n_rows_a, nn, c->n_wires, ab, check,
            c->d_err, 0, 0);
      });
    if (rc != G3H_OK) return rc;
    if (!ok(cudaEventRecord(ln.ev_ga, vs[0])) || !ok(cudaEventRecord(ln.ev_gb, vs[1])) ||
        !ok(cudaStreamWaitEvent(vs[2], ln.ev_ga, 0)) || !ok(cudaStreamWaitEvent(vs[2], ln.ev_gb, 0)))
      return G3H_E_CUDA;
    a = ab;
    b = ab + n;
    cc = nullptr;
  }
  fr_t* s[3] = {ln.abc, ln.abc + n, ln.abc + 2 * n};
  const Plan pl = plan_for(k);
  // Launches are issued phase by phase over the three vectors so that the vectors
  // advance together.
  {
    NvtxRange range("g3h inverse, top levels");
    for (int lvl = pl.levels - 1; lvl >= 1 && rc == G3H_OK; lvl--) {
      const bool first = lvl == pl.levels - 1;
      for (uint32_t v = 0; v < nv && rc == G3H_OK; v++) {
        SliceArgs x = base_args(c, flags);
        x.src[0] = first ? a : s[0];
        x.src[1] = first ? b : s[1];
        x.src[2] = first ? cc : s[2];
        for (int u = 0; u < 3; u++) x.dst[u] = s[u];
        x.tw = c->d_tw_inv;
        x.kk = pl.kk[lvl];
        x.c0 = pl.c0[lvl];
        x.mode = (first && check && !w) ? SL_CHECK : 0u;
        if (first && w) x.mode |= SL_C_FROM_AB;
        x.vbase = v;
        rc = launch_slice_on(c, vs[v], "ntt_dif", Slice::dif, x, rows);
      }
    }
  }
  {
    NvtxRange range("g3h inverse low levels, shift, forward low levels");
    for (uint32_t v = 0; v < nv && rc == G3H_OK; v++) {
      SliceArgs x = base_args(c, flags);
      for (int u = 0; u < 3; u++) x.dst[u] = s[u];
      x.tw = c->d_tw_inv;
      x.tw2 = c->d_tw_fwd;
      x.scale_tab = c->d_shift_br;
      x.kk = pl.kk[0];
      x.c0 = 0;
      x.vbase = v;
      rc = launch_slice_on(c, vs[v], "ntt_mid", Slice::mid, x, rows);
    }
  }
  {
    NvtxRange range("g3h forward, top levels");
    for (int lvl = 1; lvl < pl.levels && rc == G3H_OK; lvl++) {
      const bool top = lvl == pl.levels - 1;
      for (uint32_t v = 0; v < nv && rc == G3H_OK; v++) {
        SliceArgs x = base_args(c, flags);
        for (int u = 0; u < 3; u++) x.src[u] = x.dst[u] = s[u];
        x.tw = c->d_tw_fwd;
        x.kk = pl.kk[lvl];
        x.c0 = pl.c0[lvl];
        x.vbase = v;
        const bool fused = top && (flags & G3H_FUSED_JOIN);
        if (fused) {
          x.mode = SL_JOIN_LAST;
          x.h_mont = hm;
          x.h_std = hs;
          x.counters = ln.counters;
        }
        rc = launch_slice_on(c, vs[v], fused ? "ntt_dit_join" : "ntt_dit", Slice::dit, x, rows);
      }
    }
  }
  return rc;
}

int quotient_launches(g3h_ctx* c, const Lane& ln, const fr_t* a, const fr_t* b,
                      const fr_t* cc, const fr_t* w, fr_t* hm, fr_t* hs, uint32_t flags) {
  const uint32_t k = c->log_n;
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  const size_t n = c->n;
  const cudaStream_t st = ln.stream;
  if (k <= kSmallMaxLog) {
    if (w) {
      fr_t* s3 = ln.abc;
      const int rc = gather_on(c, st, w, s3, s3 + n, s3 + 2 * n, flags);
      if (rc != G3H_OK) return rc;
      a = s3;
      b = s3 + n;
      cc = s3 + 2 * n;
    }
    return run_on(c, st, "small_quotient", [&] {
      k_small_quotient<<<1, 32, 0, st>>>(a, b, cc, c->d_tw_inv, c->d_tw_fwd, c->d_shift_br, hm,
                                          hs, k, check, c->d_err);
    });
  }
  const bool serial = (flags & G3H_SERIALIZE) != 0u;
  const cudaStream_t vs[3] = {st, serial ? st : ln.aux[0], serial ? st : ln.aux[1]};
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!serial && (!ok(cudaEventRecord(ln.ev_fork, st)) ||
                  !ok(cudaStreamWaitEvent(vs[1], ln.ev_fork, 0)) ||
                  !ok(cudaStreamWaitEvent(vs[2], ln.ev_fork, 0))))
    return G3H_E_CUDA;
  int rc = quotient_vectors(c, ln, vs, serial, a, b, cc, w, hm, hs, flags);
  if (rc == G3H_OK && !(flags & G3H_FUSED_JOIN)) {
    // The join in two steps. The product p = a * b needs only vectors a and b, which are
    // done well before c (its chain starts once both gathers are done), so it is formed
    // on b's stream, over a, while c's last kernel still runs; the join then reduces on
    // c's stream, right after c's last kernel: h = p - c and its standard form.
    NvtxRange range("g3h join");
    fr_t* p = s_of(ln, n, 0);
    if (!serial && (!ok(cudaEventRecord(ln.ev_a, vs[0])) ||
                    !ok(cudaStreamWaitEvent(vs[1], ln.ev_a, 0))))
      rc = G3H_E_CUDA;
    if (rc == G3H_OK)
      rc = run_on(c, vs[1], "prejoin", [&] {
        launch_pdl(blocks_for(n, 256), 256, vs[1], k_join_product, p,
                   (const fr_t*)s_of(ln, n, 1), n);
      });
    if (rc == G3H_OK && !serial &&
        (!ok(cudaEventRecord(ln.ev_p, vs[1])) || !ok(cudaStreamWaitEvent(vs[2], ln.ev_p, 0))))
      rc = G3H_E_CUDA;
    if (rc == G3H_OK)
      rc = run_on(c, vs[2], "join", [&] {
        launch_pdl(blocks_for(n, 256), 256, vs[2], k_join_reduce, (const fr_t*)p,
                   (const fr_t*)s_of(ln, n, 2), hm, hs, n);
      });
  }
  // the lane's stream waits for streams b and c, also after a failed launch
  if (!serial)
    for (int i = 0; i < 2; i++)
      if (!ok(cudaEventRecord(ln.ev_end[i], vs[i + 1])) ||
          !ok(cudaStreamWaitEvent(st, ln.ev_end[i], 0)))
        rc = G3H_E_CUDA;
  return rc;
}

// quotient_launches through a launch graph: captured on the first call with a given lane,
// pointers and flags, replayed afterwards. Not when per-kernel timing is on (its events
// must be recorded per call), when the caller's stream is already being captured, or
// with G3H_NO_GRAPH.
constexpr size_t kMaxGraphs = 8;

int quotient(g3h_ctx* c, const Lane& ln, const fr_t* a, const fr_t* b, const fr_t* cc,
             const fr_t* w, fr_t* hm, fr_t* hs, uint32_t flags) {
  const cudaStream_t st = ln.stream;
  bool graph = !c->timing && !(flags & G3H_NO_GRAPH) && c->log_n > kSmallMaxLog;
  if (graph) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return G3H_E_CUDA;
    graph = cs == cudaStreamCaptureStatusNone;
  }
  if (!graph) return quotient_launches(c, ln, a, b, cc, w, hm, hs, flags);
  const void* key[6] = {a, b, cc, w, hm, hs};
  for (auto& g : c->graphs) {
    if (g.stream == st && g.flags == flags && std::memcmp(g.ptr, key, sizeof(key)) == 0)
      return cudaGraphLaunch(g.exec, st) == cudaSuccess ? G3H_OK : G3H_E_CUDA;
  }
  Lane cl = ln;  // the same buffers and streams, vector a captured on the private stream
  cl.stream = ln.cap;
  if (cudaStreamBeginCapture(cl.stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    return G3H_E_CUDA;
  int rc = quotient_launches(c, cl, a, b, cc, w, hm, hs, flags);
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cl.stream, &g);
  if (rc == G3H_OK && ec != cudaSuccess) rc = G3H_E_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (rc == G3H_OK && cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) rc = G3H_E_CUDA;
  if (g) cudaGraphDestroy(g);
  if (rc != G3H_OK) {
    cudaGetLastError();
    return rc;
  }
  if (c->graphs.size() == kMaxGraphs) {
    cudaGraphExecDestroy(c->graphs.front().exec);
    c->graphs.erase(c->graphs.begin());
  }
  g3h_ctx::Graph e;
  e.stream = st;
  std::memcpy(e.ptr, key, sizeof(key));
  e.flags = flags;
  e.exec = exec;
  c->graphs.push_back(e);
  return cudaGraphLaunch(exec, st) == cudaSuccess ? G3H_OK : G3H_E_CUDA;
}

int gather_on(g3h_ctx* c, cudaStream_t st, const fr_t* w, fr_t* a, fr_t* b, fr_t* cc,
              uint32_t flags) {
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  const uint32_t n = (uint32_t)c->n;
  return run_on(c, st, "gather", [&] {
    k_gather<<<blocks_for(n, 256), 256, 0, st>>>(
        c->d_rpa, c->d_cola, c->d_vala, c->d_rpb, c->d_colb, c->d_valb, w, c->n_rows_a,
        c->n_rows_b, n, a, b, cc, check, c->d_err);
  });
}

int gather(g3h_ctx* c, const fr_t* w, fr_t* a, fr_t* b, fr_t* cc, uint32_t flags) {
  return gather_on(c, c->stream, w, a, b, cc, flags);
}

int ntt(g3h_ctx* c, fr_t* data, int inverse, int coset, uint32_t flags) {
  const uint32_t k = c->log_n;
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  if (coset) {
    const int rc = ensure_coset_tables(c);
    if (rc != G3H_OK) return rc;
  }
  const fr_const_t* tw = inverse ? c->d_tw_inv : c->d_tw_fwd;
  const fr_const_t* scale_load = (!inverse && coset) ? c->d_coset_fwd : nullptr;
  const fr_const_t* scale_store = (inverse && coset) ? c->d_coset_inv : nullptr;
  const bool store_const = inverse && !coset;
  if (k <= kSmallMaxLog) {
    return run(c, "small_ntt", [&] {
      k_small_ntt<<<1, 32, 0, c->stream>>>(data, tw, scale_load, scale_store, c->h_ninv,
                                            store_const ? 1u : 0u, k, check, c->d_err);
    });
  }
  const Plan pl = plan_for(k);
  fr_t* s = c->d_abc;
  SliceArgs x = base_args(c, flags);
  x.src[0] = data;
  x.dst[0] = s;
  x.tw = tw;
  x.scale_tab = scale_load;
  x.kk = pl.kk[0];
  x.mode = (check ? SL_CHECK : 0u) | (scale_load ? SL_SCALE_TABLE : 0u);
  int rc = launch_slice(c, "ntt_brev", Slice::brev, x, 1);
  for (int lvl = 1; lvl < pl.levels && rc == G3H_OK; lvl++) {
    SliceArgs y = base_args(c, flags);
    const bool top = lvl == pl.levels - 1;
    y.src[0] = s;
    y.dst[0] = top ? data : s;
    y.tw = tw;
    y.kk = pl.kk[lvl];
    y.c0 = pl.c0[lvl];
    if (top) {
      if (scale_store) {
        y.scale_tab = scale_store;
        y.mode = SL_SCALE_TABLE;
      } else if (store_const) {
        y.kscale = c->h_ninv;
        y.mode = SL_SCALE_CONST;
      }
    }
    rc = launch_slice(c, "ntt_dit", Slice::dit, y, 1);
  }
  return rc;
}

bool validate_csr(const g3h_csr* m, size_t n, uint32_t n_wires, int* rc) {
  if (m->n_rows > n) {
    *rc = G3H_E_INVAL;
    return false;
  }
  if (!m->row_ptr) {
    *rc = G3H_E_INVAL;
    return false;
  }
  if (m->row_ptr[0] != 0) {
    *rc = G3H_E_RANGE;
    return false;
  }
  for (uint32_t i = 0; i < m->n_rows; i++) {
    if (m->row_ptr[i + 1] < m->row_ptr[i]) {
      *rc = G3H_E_RANGE;
      return false;
    }
  }
  const size_t nnz = m->row_ptr[m->n_rows];
  if (nnz && (!m->col || !m->val)) {
    *rc = G3H_E_INVAL;
    return false;
  }
  for (size_t k = 0; k < nnz; k++) {
    if (m->col[k] >= n_wires) {
      *rc = G3H_E_RANGE;
      return false;
    }
    if (!host_canonical(m->val + 8 * k)) {
      *rc = G3H_E_NONCANON;
      return false;
    }
  }
  return true;
}

int upload_csr(g3h_ctx* c, const g3h_csr* m, uint32_t** rp, uint32_t** col, fr_t** val) {
  const size_t nnz = m->row_ptr[m->n_rows];
  int rc = dalloc(rp, (size_t)m->n_rows + 1);
  if (rc == G3H_OK) rc = dalloc(col, nnz);
  if (rc == G3H_OK) rc = dalloc(val, nnz);
  if (rc != G3H_OK) return rc;
  rc = h2d(c, *rp, m->row_ptr, ((size_t)m->n_rows + 1) * sizeof(uint32_t));
  if (rc == G3H_OK) rc = h2d(c, *col, m->col, nnz * sizeof(uint32_t));
  if (rc == G3H_OK) rc = h2d(c, *val, m->val, nnz * sizeof(fr_t));
  return rc;
}

}  // namespace

extern "C" {

int g3h_prepare(uint32_t log_n, uint32_t n_wires, const g3h_csr* A, const g3h_csr* B,
                int device, void* stream, g3h_ctx** out) {
  if (!out) return G3H_E_INVAL;
  *out = nullptr;
  if (log_n > G3H_MAX_LOG_N) return G3H_E_RANGE;
  if ((A == nullptr) != (B == nullptr)) return G3H_E_INVAL;
  const size_t n = (size_t)1 << log_n;
  int rc = G3H_OK;
  if (A && (!validate_csr(A, n, n_wires, &rc) || !validate_csr(B, n, n_wires, &rc))) return rc;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev)
    return G3H_E_CUDA;
  DeviceGuard guard(device);
  g3h_ctx* c = new (std::nothrow) g3h_ctx();
  if (!c) return G3H_E_NOMEM;
  c->device = device;
  if (cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, device) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&c->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                             device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock,
                             device) != cudaSuccess) {
    delete c;
    return G3H_E_CUDA;
  }
  c->log_n = log_n;
  c->n = n;
  c->n_wires = n_wires;
  if (stream) {
    c->stream = (cudaStream_t)stream;
  } else {
    if (cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking) != cudaSuccess) {
      delete c;
      return G3H_E_CUDA;
    }
    c->own_stream = true;
  }
  rc = set_smem_limits();
  if (rc == G3H_OK) rc = make_lane_streams(c->own);
  if (rc == G3H_OK)
    rc = !inject_fault(Fault::alloc) &&
                 cudaMallocHost((void**)&c->h_err, sizeof(uint32_t)) == cudaSuccess
             ? G3H_OK
             : G3H_E_NOMEM;
  if (rc == G3H_OK) *c->h_err = 0;
  if (rc == G3H_OK) rc = dalloc(&c->d_err, 1);
  if (rc == G3H_OK)
    rc = cudaMemsetAsync(c->d_err, 0, sizeof(uint32_t), c->stream) == cudaSuccess ? G3H_OK
                                                                                  : G3H_E_CUDA;
  if (rc == G3H_OK) rc = dalloc(&c->d_consts, 6);
  if (rc == G3H_OK) rc = dalloc(&c->d_tw_fwd, n / 2);
  if (rc == G3H_OK) rc = dalloc(&c->d_tw_inv, n / 2);
  if (rc == G3H_OK) rc = dalloc(&c->d_shift_br, n);
  if (rc == G3H_OK) rc = dalloc(&c->d_abc, 3 * n);
  if (rc == G3H_OK && A) rc = dalloc(&c->d_ab_in, 2 * n);
  const size_t n_slices = n >> plan_for(log_n).kk[plan_for(log_n).levels - 1];
  if (rc == G3H_OK) rc = dalloc(&c->d_counters, n_slices);
  if (rc == G3H_OK)
    rc = cudaMemsetAsync(c->d_counters, 0, std::max<size_t>(n_slices, 1) * sizeof(uint32_t),
                         c->stream) == cudaSuccess
             ? G3H_OK
             : G3H_E_CUDA;
  if (rc == G3H_OK)
    rc = run(c, "tables", [&] { k_domain<<<1, 1, 0, c->stream>>>(c->d_consts, log_n); });
  if (rc == G3H_OK) rc = build_table(c, c->d_tw_fwd, n / 2, 0, -1, 0);
  if (rc == G3H_OK) rc = build_table(c, c->d_tw_inv, n / 2, 1, -1, 0);
  if (rc == G3H_OK) rc = build_table(c, c->d_shift_br, n, 2, 4, log_n);
  if (rc == G3H_OK) rc = dalloc(&c->d_ninv, 1);
  if (rc == G3H_OK) rc = build_table(c, c->d_ninv, 1, 5, 4, 0);  // 1^0 * n^-1
  if (rc == G3H_OK && A) {
    c->has_csr = true;
    c->n_rows_a = A->n_rows;
    c->n_rows_b = B->n_rows;
    rc = upload_csr(c, A, &c->d_rpa, &c->d_cola, &c->d_vala);
    if (rc == G3H_OK) rc = upload_csr(c, B, &c->d_rpb, &c->d_colb, &c->d_valb);
  }
  if (rc == G3H_OK)
    rc = cudaMemcpyAsync(&c->h_ninv, c->d_ninv, sizeof(c->h_ninv), cudaMemcpyDeviceToHost,
                         c->stream) == cudaSuccess
             ? G3H_OK
             : G3H_E_CUDA;
  if (rc == G3H_OK) rc = cudaStreamSynchronize(c->stream) == cudaSuccess ? G3H_OK : G3H_E_CUDA;
  if (rc != G3H_OK) {
    cudaGetLastError();
    release(c);
    delete c;
    return rc;
  }
  *out = c;
  return G3H_OK;
}

int g3h_compute_h(g3h_ctx* c, const uint32_t* witness, uint32_t* h_mont, uint32_t* h_std,
                  uint32_t flags) {
  if (!c || !c->has_csr || !h_mont || !h_std || (!witness && c->n_wires)) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  NvtxRange range("g3h_compute_h");
  const size_t n = c->n;
  fr_t* s[3] = {c->d_abc, c->d_abc + n, c->d_abc + 2 * n};
  if ((flags & G3H_DEVICE_PTRS) && misaligned({witness, h_mont, h_std})) return G3H_E_INVAL;
  if (flags & G3H_DEVICE_PTRS)
    return quotient(c, lane0(c), s[0], s[1], s[2], (const fr_t*)witness, (fr_t*)h_mont,
                    (fr_t*)h_std, flags);
  int rc = ensure_stage(c, (size_t)c->n_wires + 2 * n);
  if (rc != G3H_OK) return rc;
  fr_t* w = c->d_stage;
  fr_t* hm = c->d_stage + c->n_wires;
  fr_t* hs = hm + n;
  rc = h2d(c, w, witness, (size_t)c->n_wires * sizeof(fr_t));
  if (rc == G3H_OK) rc = quotient(c, lane0(c), s[0], s[1], s[2], w, hm, hs, flags);
  if (rc == G3H_OK) rc = d2h(c, h_mont, hm, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = d2h(c, h_std, hs, n * sizeof(fr_t));
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

int g3h_compute_h_abc(g3h_ctx* c, const uint32_t* a, const uint32_t* b, const uint32_t* cc,
                      uint32_t* h_mont, uint32_t* h_std, uint32_t flags) {
  if (!c || !a || !b || !cc || !h_mont || !h_std) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  NvtxRange range("g3h_compute_h_abc");
  const size_t n = c->n;
  if ((flags & G3H_DEVICE_PTRS) && misaligned({a, b, cc, h_mont, h_std})) return G3H_E_INVAL;
  if (flags & G3H_DEVICE_PTRS)
    return quotient(c, lane0(c), (const fr_t*)a, (const fr_t*)b, (const fr_t*)cc, nullptr,
                    (fr_t*)h_mont, (fr_t*)h_std, flags);
  int rc = ensure_stage(c, 5 * n);
  if (rc != G3H_OK) return rc;
  fr_t* in = c->d_stage;
  fr_t* hm = c->d_stage + 3 * n;
  fr_t* hs = hm + n;
  rc = h2d(c, in, a, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = h2d(c, in + n, b, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = h2d(c, in + 2 * n, cc, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = quotient(c, lane0(c), in, in + n, in + 2 * n, nullptr, hm, hs, flags);
  if (rc == G3H_OK) rc = d2h(c, h_mont, hm, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = d2h(c, h_std, hs, n * sizeof(fr_t));
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

}  // extern "C"

namespace {

// Domains whose batched calls take the z lanes, and the chunk size: enough witnesses per
// launch for about 2^20 elements per vector phase, at most 64.
constexpr uint32_t kZMinLog = 6, kZMaxLog = 16;

uint32_t z_chunk_for(uint32_t log_n) {
  return std::min<uint32_t>(64u, std::max<uint32_t>(1u, (1u << 20) >> log_n));
}

int ensure_zlanes(g3h_ctx* c, bool staged) {
  const uint32_t z = z_chunk_for(c->log_n);
  if (c->z_chunk == z && (c->z_staged || !staged)) return G3H_OK;
  const size_t n = c->n;
  for (ZLane& l : c->zl) {
    if (l.stream) cudaStreamSynchronize(l.stream);
    free_zlane(l);
  }
  c->z_chunk = 0;
  c->z_staged = false;
  for (ZLane& l : c->zl) {
    int rc = cudaStreamCreateWithFlags(&l.stream, cudaStreamNonBlocking) == cudaSuccess &&
                     cudaEventCreateWithFlags(&l.done, cudaEventDisableTiming) == cudaSuccess
                 ? G3H_OK
                 : G3H_E_CUDA;
    if (rc == G3H_OK) rc = dalloc(&l.ab_in, (size_t)z * 2 * n);
    if (rc == G3H_OK) rc = dalloc(&l.abc, (size_t)z * 3 * n);
    if (rc == G3H_OK && staged) rc = dalloc(&l.stage, (size_t)z * (c->n_wires + 2 * n));
    if (rc != G3H_OK) {
      for (ZLane& m : c->zl) free_zlane(m);
      return rc;
    }
  }
  c->z_chunk = z;
  c->z_staged = staged;
  return G3H_OK;
}

// Steps 1-5 for nz witnesses at w + i * w_stride (device) -> h_mont, h_std at hm, hs +
// i * h_stride (device), on a z lane: one launch per phase for all of them.
int quotient_z(g3h_ctx* c, const ZLane& l, uint32_t nz, const fr_t* w, size_t w_stride,
               fr_t* hm, fr_t* hs, size_t h_stride, uint32_t flags) {
  const uint32_t k = c->log_n;
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  const size_t n = c->n;
  const cudaStream_t st = l.stream;
  const uint32_t nn = (uint32_t)n;
  const dim3 ggrid(blocks_for(n, 256), nz);
  int rc = run_on(c, st, "gather_a", [&] {
    k_gather_rows<<<ggrid, 256, 0, st>>>(c->d_rpa, c->d_cola, c->d_vala, w, c->n_rows_a, nn,
                                         c->n_wires, l.ab_in, check, c->d_err, w_stride, 2 * n);
  });
  if (rc == G3H_OK)
    rc = run_on(c, st, "gather_b", [&] {
      k_gather_rows<<<ggrid, 256, 0, st>>>(c->d_rpb, c->d_colb, c->d_valb, w, c->n_rows_b, nn,
                                           c->n_wires, l.ab_in + n, check, c->d_err, w_stride,
                                           2 * n);
    });
  const Plan pl = plan_for(k);
  fr_t* s[3] = {l.abc, l.abc + n, l.abc + 2 * n};
  for (int lvl = pl.levels - 1; lvl >= 1 && rc == G3H_OK; lvl--) {
    const bool first = lvl == pl.levels - 1;
    SliceArgs x = base_args(c, flags);
    x.src[0] = first ? l.ab_in : s[0];
    x.src[1] = first ? l.ab_in + n : s[1];
    x.src[2] = first ? nullptr : s[2];
    for (int u = 0; u < 3; u++) x.dst[u] = s[u];
    x.zs_src = first ? 2 * n : 3 * n;
    x.zs_dst = 3 * n;
    x.tw = c->d_tw_inv;
    x.kk = pl.kk[lvl];
    x.c0 = pl.c0[lvl];
    x.mode = first ? SL_C_FROM_AB : 0u;
    rc = launch_slice_on(c, st, "ntt_dif", Slice::dif, x, 3, nz);
  }
  if (rc == G3H_OK) {
    SliceArgs x = base_args(c, flags);
    for (int u = 0; u < 3; u++) x.dst[u] = s[u];
    x.zs_dst = 3 * n;
    x.tw = c->d_tw_inv;
    x.tw2 = c->d_tw_fwd;
    x.scale_tab = c->d_shift_br;
    x.kk = pl.kk[0];
    rc = launch_slice_on(c, st, "ntt_mid", Slice::mid, x, 3, nz);
  }
  for (int lvl = 1; lvl < pl.levels && rc == G3H_OK; lvl++) {
    SliceArgs x = base_args(c, flags);
    for (int u = 0; u < 3; u++) x.src[u] = x.dst[u] = s[u];
    x.zs_src = x.zs_dst = 3 * n;
    x.tw = c->d_tw_fwd;
    x.kk = pl.kk[lvl];
    x.c0 = pl.c0[lvl];
    rc = launch_slice_on(c, st, "ntt_dit", Slice::dit, x, 3, nz);
  }
  if (rc == G3H_OK)
    rc = run_on(c, st, "join", [&] {
      k_join<<<dim3(blocks_for(n, 256), nz), 256, 0, st>>>(s[0], s[1], s[2], hm, hs, n, 0u,
                                                           c->d_err, 3 * n, h_stride);
    });
  return rc;
}

// A batched call on the z lanes: chunks of up to z_chunk witnesses, alternating lanes.
int batch_z(g3h_ctx* c, uint32_t count, const uint32_t* witnesses, uint32_t* h_mont,
            uint32_t* h_std, uint32_t flags) {
  const bool dev = (flags & G3H_DEVICE_PTRS) != 0u;
  int rc = ensure_zlanes(c, !dev);
  if (rc != G3H_OK) return rc;
  const size_t n = c->n, nw = c->n_wires;
  const uint32_t z = c->z_chunk;
  // the lanes start after everything already queued on the context's stream
  if (!c->batch_start &&
      cudaEventCreateWithFlags(&c->batch_start, cudaEventDisableTiming) != cudaSuccess)
    return G3H_E_CUDA;
  if (cudaEventRecord(c->batch_start, c->stream) != cudaSuccess) return G3H_E_CUDA;
  for (ZLane& l : c->zl)
    if (cudaStreamWaitEvent(l.stream, c->batch_start, 0) != cudaSuccess) return G3H_E_CUDA;
  uint32_t chunk = 0;
  for (uint32_t i = 0; i < count && rc == G3H_OK; i += z, chunk++) {
    const ZLane& l = c->zl[chunk & 1u];
    const uint32_t nz = std::min(z, count - i);
    const uint32_t* wi = witnesses + (size_t)i * 8 * nw;
    uint32_t* hmi = h_mont + (size_t)i * 8 * n;
    uint32_t* hsi = h_std + (size_t)i * 8 * n;
    if (dev) {
      rc = quotient_z(c, l, nz, (const fr_t*)wi, nw, (fr_t*)hmi, (fr_t*)hsi, n, flags);
      continue;
    }
    fr_t* w = l.stage;
    fr_t* hm = l.stage + (size_t)z * nw;
    fr_t* hs = hm + (size_t)z * n;
    rc = copy_on(l.stream, w, wi, (size_t)nz * nw * sizeof(fr_t), cudaMemcpyHostToDevice);
    if (rc == G3H_OK) rc = quotient_z(c, l, nz, w, nw, hm, hs, n, flags);
    if (rc == G3H_OK)
      rc = copy_on(l.stream, hmi, hm, (size_t)nz * n * sizeof(fr_t), cudaMemcpyDeviceToHost);
    if (rc == G3H_OK)
      rc = copy_on(l.stream, hsi, hs, (size_t)nz * n * sizeof(fr_t), cudaMemcpyDeviceToHost);
  }
  // the context's stream waits for both lanes: the batch ends in its order
  for (ZLane& l : c->zl)
    if (cudaEventRecord(l.done, l.stream) != cudaSuccess ||
        cudaStreamWaitEvent(c->stream, l.done, 0) != cudaSuccess)
      rc = G3H_E_CUDA;
  if (dev) return rc;
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

// Lanes of a batched call: the context's own plus up to kBatchLanes - 1 more, each with
// its stream and buffers, allocated on first use and kept.
constexpr uint32_t kBatchLanes = 3;

int ensure_lanes(g3h_ctx* c, uint32_t lanes, bool staged) {
  const size_t n = c->n;
  const Plan pl = plan_for(c->log_n);
  const size_t n_slices = std::max<size_t>(n >> pl.kk[pl.levels - 1], 1);
  while (c->extra_lanes.size() + 1 < lanes) {
    // a lane joins the context only once all its parts exist
    Lane l;
    int rc = cudaStreamCreateWithFlags(&l.stream, cudaStreamNonBlocking) == cudaSuccess
                 ? G3H_OK
                 : G3H_E_CUDA;
    l.own_stream = l.stream != nullptr;
    if (rc == G3H_OK) rc = dalloc(&l.abc, 3 * n);
    if (rc == G3H_OK) rc = dalloc(&l.ab_in, 2 * n);
    if (rc == G3H_OK) rc = dalloc(&l.counters, n_slices);
    if (rc == G3H_OK &&
        (cudaMemsetAsync(l.counters, 0, n_slices * sizeof(uint32_t), l.stream) != cudaSuccess ||
         cudaEventCreateWithFlags(&l.done, cudaEventDisableTiming) != cudaSuccess))
      rc = G3H_E_CUDA;
    if (rc == G3H_OK) rc = make_lane_streams(l);
    if (rc != G3H_OK) {
      if (l.stream) cudaStreamSynchronize(l.stream);
      free_lane(l);
      return rc;
    }
    c->extra_lanes.push_back(l);
  }
  if (!c->batch_start &&
      cudaEventCreateWithFlags(&c->batch_start, cudaEventDisableTiming) != cudaSuccess)
    return G3H_E_CUDA;
  if (staged) {
    const size_t elems = (size_t)c->n_wires + 2 * n;
    int rc = ensure_stage(c, elems);
    if (rc != G3H_OK) return rc;
    for (uint32_t i = 0; i + 1 < lanes; i++) {
      Lane& l = c->extra_lanes[i];
      if (l.stage_elems < elems) {
        if (l.stage) cudaFree(l.stage);
        l.stage = nullptr;
        l.stage_elems = 0;
        if (dalloc(&l.stage, elems) != G3H_OK) return G3H_E_NOMEM;
        l.stage_elems = elems;
      }
    }
  }
  return G3H_OK;
}

}  // namespace

extern "C" {

int g3h_compute_h_batch(g3h_ctx* c, uint32_t count, const uint32_t* witnesses,
                        uint32_t* h_mont, uint32_t* h_std, uint32_t flags) {
  if (!c || !c->has_csr) return G3H_E_INVAL;
  if (count == 0) return G3H_OK;
  if (!h_mont || !h_std || (!witnesses && c->n_wires)) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  NvtxRange range("g3h_compute_h_batch");
  const bool dev = (flags & G3H_DEVICE_PTRS) != 0u;
  if (dev && misaligned({witnesses, h_mont, h_std})) return G3H_E_INVAL;
  if (c->log_n >= kZMinLog && c->log_n <= kZMaxLog && count > 1 &&
      !(flags & G3H_FUSED_JOIN))
    return batch_z(c, count, witnesses, h_mont, h_std, flags);
  const uint32_t lanes = std::min(count, kBatchLanes);
  int rc = ensure_lanes(c, lanes, !dev);
  if (rc != G3H_OK) return rc;
  // the extra lanes start after everything already queued on the context's stream
  if (cudaEventRecord(c->batch_start, c->stream) != cudaSuccess) return G3H_E_CUDA;
  for (uint32_t i = 0; i + 1 < lanes; i++)
    if (cudaStreamWaitEvent(c->extra_lanes[i].stream, c->batch_start, 0) != cudaSuccess)
      return G3H_E_CUDA;
  const size_t n = c->n, nw = c->n_wires;
  for (uint32_t i = 0; i < count && rc == G3H_OK; i++) {
    const uint32_t li = i % lanes;
    Lane ln = li == 0 ? lane0(c) : c->extra_lanes[li - 1];
    if (li == 0) ln.stage = c->d_stage;
    const uint32_t* wi = witnesses + (size_t)i * 8 * nw;
    uint32_t* hmi = h_mont + (size_t)i * 8 * n;
    uint32_t* hsi = h_std + (size_t)i * 8 * n;
    if (dev) {
      // every witness has its own buffers here: launch directly rather than capture
      rc = quotient(c, ln, nullptr, nullptr, nullptr, (const fr_t*)wi, (fr_t*)hmi, (fr_t*)hsi,
                    flags | G3H_NO_GRAPH);
      continue;
    }
    fr_t* w = ln.stage;
    fr_t* hm = ln.stage + nw;
    fr_t* hs = hm + n;
    rc = copy_on(ln.stream, w, wi, nw * sizeof(fr_t), cudaMemcpyHostToDevice);
    if (rc == G3H_OK) rc = quotient(c, ln, nullptr, nullptr, nullptr, w, hm, hs, flags);
    if (rc == G3H_OK) rc = copy_on(ln.stream, hmi, hm, n * sizeof(fr_t), cudaMemcpyDeviceToHost);
    if (rc == G3H_OK) rc = copy_on(ln.stream, hsi, hs, n * sizeof(fr_t), cudaMemcpyDeviceToHost);
  }
  // the context's stream waits for the extra lanes: the batch ends in its order
  for (uint32_t i = 0; i + 1 < lanes; i++) {
    Lane& l = c->extra_lanes[i];
    if (cudaEventRecord(l.done, l.stream) != cudaSuccess ||
        cudaStreamWaitEvent(c->stream, l.done, 0) != cudaSuccess)
      return G3H_E_CUDA;
  }
  if (dev) return rc;
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

int g3h_gather(g3h_ctx* c, const uint32_t* witness, uint32_t* a, uint32_t* b, uint32_t* cc,
               uint32_t flags) {
  if (!c || !c->has_csr || !a || !b || !cc || (!witness && c->n_wires)) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  NvtxRange range("g3h_gather");
  const size_t n = c->n;
  if ((flags & G3H_DEVICE_PTRS) && misaligned({witness, a, b, cc})) return G3H_E_INVAL;
  if (flags & G3H_DEVICE_PTRS)
    return gather(c, (const fr_t*)witness, (fr_t*)a, (fr_t*)b, (fr_t*)cc, flags);
  int rc = ensure_stage(c, (size_t)c->n_wires + 3 * n);
  if (rc != G3H_OK) return rc;
  fr_t* w = c->d_stage;
  fr_t* o = c->d_stage + c->n_wires;
  rc = h2d(c, w, witness, (size_t)c->n_wires * sizeof(fr_t));
  if (rc == G3H_OK) rc = gather(c, w, o, o + n, o + 2 * n, flags);
  if (rc == G3H_OK) rc = d2h(c, a, o, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = d2h(c, b, o + n, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = d2h(c, cc, o + 2 * n, n * sizeof(fr_t));
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

int g3h_ntt(g3h_ctx* c, uint32_t* data, int inverse, int coset, uint32_t flags) {
  if (!c || !data) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  NvtxRange range("g3h_ntt");
  const size_t n = c->n;
  if ((flags & G3H_DEVICE_PTRS) && misaligned({data})) return G3H_E_INVAL;
  if (flags & G3H_DEVICE_PTRS) return ntt(c, (fr_t*)data, inverse, coset, flags);
  int rc = ensure_stage(c, n);
  if (rc != G3H_OK) return rc;
  rc = h2d(c, c->d_stage, data, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = ntt(c, c->d_stage, inverse, coset, flags);
  if (rc == G3H_OK) rc = d2h(c, data, c->d_stage, n * sizeof(fr_t));
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

int g3h_join(g3h_ctx* c, const uint32_t* ea, const uint32_t* eb, const uint32_t* ec,
             uint32_t* h_mont, uint32_t* h_std, uint32_t flags) {
  if (!c || !ea || !eb || !ec || !h_mont || !h_std) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  const size_t n = c->n;
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  auto launch = [&](const fr_t* x, const fr_t* y, const fr_t* z, fr_t* hm, fr_t* hs) {
    return run(c, "join", [&] {
      k_join<<<blocks_for(n, 256), 256, 0, c->stream>>>(x, y, z, hm, hs, n, check, c->d_err, 0,
                                                        0);
    });
  };
  if ((flags & G3H_DEVICE_PTRS) && misaligned({ea, eb, ec, h_mont, h_std})) return G3H_E_INVAL;
  if (flags & G3H_DEVICE_PTRS)
    return launch((const fr_t*)ea, (const fr_t*)eb, (const fr_t*)ec, (fr_t*)h_mont,
                  (fr_t*)h_std);
  int rc = ensure_stage(c, 5 * n);
  if (rc != G3H_OK) return rc;
  fr_t* in = c->d_stage;
  rc = h2d(c, in, ea, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = h2d(c, in + n, eb, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = h2d(c, in + 2 * n, ec, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = launch(in, in + n, in + 2 * n, in + 3 * n, in + 4 * n);
  if (rc == G3H_OK) rc = d2h(c, h_mont, in + 3 * n, n * sizeof(fr_t));
  if (rc == G3H_OK) rc = d2h(c, h_std, in + 4 * n, n * sizeof(fr_t));
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

int g3h_mul(g3h_ctx* c, const uint32_t* a, const uint32_t* b, uint32_t* out, size_t count,
            uint32_t flags) {
  if (!c || ((!a || !b || !out) && count)) return G3H_E_INVAL;
  if (count == 0) return G3H_OK;
  DeviceGuard guard(c->device);
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  auto launch = [&](const fr_t* x, const fr_t* y, fr_t* o) {
    return run(c, "mul", [&] {
      k_mul<<<blocks_for(count, 256), 256, 0, c->stream>>>(x, y, o, count, check, c->d_err);
    });
  };
  if ((flags & G3H_DEVICE_PTRS) && misaligned({a, b, out})) return G3H_E_INVAL;
  if (flags & G3H_DEVICE_PTRS) return launch((const fr_t*)a, (const fr_t*)b, (fr_t*)out);
  int rc = ensure_stage(c, 3 * count);
  if (rc != G3H_OK) return rc;
  fr_t* in = c->d_stage;
  rc = h2d(c, in, a, count * sizeof(fr_t));
  if (rc == G3H_OK) rc = h2d(c, in + count, b, count * sizeof(fr_t));
  if (rc == G3H_OK) rc = launch(in, in + count, in + 2 * count);
  if (rc == G3H_OK) rc = d2h(c, out, in + 2 * count, count * sizeof(fr_t));
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

int g3h_mont_to_std(g3h_ctx* c, const uint32_t* in, uint32_t* out, size_t count,
                    uint32_t flags) {
  if (!c || ((!in || !out) && count)) return G3H_E_INVAL;
  if (count == 0) return G3H_OK;
  DeviceGuard guard(c->device);
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  auto launch = [&](const fr_t* x, fr_t* o) {
    const size_t blocks = std::min<size_t>(blocks_for(count, 256), (size_t)c->sm_count * 8);
    return run(c, "mont_to_std", [&] {
      k_mont_to_std<<<(unsigned)blocks, 256, 0, c->stream>>>(x, o, count, check, c->d_err);
    });
  };
  if ((flags & G3H_DEVICE_PTRS) && misaligned({in, out})) return G3H_E_INVAL;
  if (flags & G3H_DEVICE_PTRS) return launch((const fr_t*)in, (fr_t*)out);
  int rc = ensure_stage(c, count);
  if (rc != G3H_OK) return rc;
  fr_t* buf = c->d_stage;
  rc = h2d(c, buf, in, count * sizeof(fr_t));
  if (rc == G3H_OK) rc = launch(buf, buf);
  if (rc == G3H_OK) rc = d2h(c, out, buf, count * sizeof(fr_t));
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

// ---------------------------------------------------------------------------------------
// Multi-scalar multiplication over G1.

}  // extern "C"

namespace {

template <class G>
int msm_launches(g3h_ctx* c, MsmState& m, const fr_t* s, uint32_t count, typename G::F* out,
                 uint32_t check) {
  using Pt = typename G::Pt;
  using Aff = typename G::Aff;
  constexpr uint32_t T = G::kTree;
  constexpr uint32_t chunks = msm_chunks<G>();
  cudaStream_t st = c->stream;
  // the long-run list's count starts at zero
  if (cudaMemsetAsync(m.counts + kMsmBuckets, 0, sizeof(uint32_t), st) != cudaSuccess)
    return G3H_E_CUDA;
  // sort blocks: one per SM, fewer for few scalars; block b owns scalars [b chunk, ...)
  const uint32_t sort_blocks = std::max<uint32_t>(
      1u, std::min<uint32_t>(m.sort_blocks, (count + kMsmSortThreads - 1) / kMsmSortThreads));
  const uint32_t sort_chunk = (count + sort_blocks - 1) / sort_blocks;
  const Aff* table = (const Aff*)m.table;
  Pt* buckets = (Pt*)m.buckets;
  Pt* chunk_sums = (Pt*)m.parts;
  Pt* parts = chunk_sums + kMsmSumParts * chunks;
  Pt* ones = parts + kMsmSumParts + 1;
  const unsigned ones_grid = (unsigned)c->sm_count * 2;
  Lane& ln = c->own;
  cudaStream_t os = ln.aux[0];
  int rc = run(c, "msm_count", [&] {
    k_msm_count<<<sort_blocks, kMsmSortThreads, kMsmSortSmem, st>>>(s, count, sort_chunk,
                                                                    m.block_counts, check,
                                                                    c->d_err);
  });
  if (rc == G3H_OK)
    rc = run(c, "msm_count_cols", [&] {
      k_msm_count_cols<<<kMsmBuckets / 32, 256, 0, st>>>(m.block_counts, sort_blocks, m.counts);
    });
  if (rc == G3H_OK)
    rc = run(c, "msm_scan", [&] {
      k_msm_scan<<<1, 1024, 0, st>>>(m.counts, m.offsets);
    });
  if (rc == G3H_OK)
    rc = run(c, "msm_scatter", [&] {
      k_msm_scatter<<<sort_blocks, kMsmSortThreads, kMsmSortSmem, st>>>(
          s, count, sort_chunk, m.offsets, m.block_counts, m.entries);
    });
  // the ones' sum runs on a second stream beside the bucket path from here on, joined
  // before the end; forked after the sort, whose blocks (one per SM, 128 KiB of shared
  // memory each) then run without the ones' blocks beside them (2^18 witness multiexp:
  // 0.63 -> 0.52 ms)
  if (rc == G3H_OK)
    rc = cudaEventRecord(ln.ev_fork, st) == cudaSuccess &&
                 cudaStreamWaitEvent(os, ln.ev_fork, 0) == cudaSuccess
             ? G3H_OK
             : G3H_E_CUDA;
  if (rc == G3H_OK)
    rc = run_on(c, os, "msm_ones", [&] {
      k_msm_ones<G><<<ones_grid, T, 0, os>>>(s, count, table, ones);
    });
  if (rc == G3H_OK)
    rc = run_on(c, os, "msm_ones_sum", [&] {
      k_msm_ones_sum<G><<<1, T, 0, os>>>(ones, ones_grid, parts);
    });
  if (rc == G3H_OK && cudaEventRecord(ln.ev_end[0], os) != cudaSuccess) rc = G3H_E_CUDA;
  // threads for slices of equal length, about one per resident thread of the accumulation
  // kernel for the most entries there can be; the kernels size the slices to the entries
  // present (at least kMsmMinSlice each), so n_slices <= count <= the spill slots
  const uint64_t max_entries = (uint64_t)count * kMsmWindows;
  const uint32_t slice = (uint32_t)std::max<uint64_t>(
      kMsmMinSlice, (max_entries + m.slots - 1) / std::max<uint32_t>(m.slots, 1));
  const uint32_t n_slices = (uint32_t)((max_entries + slice - 1) / slice);
  Pt* head = (Pt*)m.spill;
  Pt* tail = head + m.n + 1;
  if (rc == G3H_OK)
    rc = run(c, "msm_accumulate", [&] {
      k_msm_accumulate<G><<<blocks_for(n_slices, T), T, 0, st>>>(
          m.entries, m.offsets, table, buckets, head, tail, n_slices);
    });
  // the list of buckets with long runs (count first) lives after the scan's counters
  uint32_t* long_list = m.counts + kMsmBuckets;
  if (rc == G3H_OK)
    rc = run(c, "msm_merge", [&] {
      k_msm_merge<G><<<kMsmBuckets / 128, 128, 0, st>>>(m.offsets, buckets, head, tail, n_slices,
                                                         long_list);
    });
  if (rc == G3H_OK)
    rc = run(c, "msm_merge_long", [&] {
      k_msm_merge_long<G><<<(unsigned)c->sm_count, T, 0, st>>>(m.offsets, buckets, head, tail,
                                                               n_slices, long_list);
    });
  Pt* U = (Pt*)m.groups;
  Pt* V = U + kMsmPairs;
  if (rc == G3H_OK)
    rc = run(c, "msm_pairs", [&] {
      k_msm_pairs<G><<<kMsmPairs / 128, 128, 0, st>>>(buckets, U, V);
    });
  if (rc == G3H_OK)
    rc = run(c, "msm_part_chunks", [&] {
      k_msm_part_chunks<G><<<dim3(chunks, kMsmSumParts), T, 0, st>>>(U, V, chunk_sums);
    });
  if (rc == G3H_OK)
    rc = run(c, "msm_parts", [&] {
      k_msm_parts<G><<<kMsmSumParts, 32, 0, st>>>(chunk_sums, parts);
    });
  if (rc == G3H_OK && cudaStreamWaitEvent(st, ln.ev_end[0], 0) != cudaSuccess) rc = G3H_E_CUDA;
  if (rc == G3H_OK)
    rc = run(c, "msm_final", [&] { k_msm_final<G><<<1, 32, 0, st>>>(parts, out); });
  return rc;
}

template <class G>
int msm_prepare(g3h_ctx* c, MsmState& m, const uint32_t* bases, uint32_t n_bases,
                uint32_t flags) {
  using Pt = typename G::Pt;
  using Aff = typename G::Aff;
  if (!c || (!bases && n_bases)) return G3H_E_INVAL;
  if ((flags & G3H_DEVICE_PTRS) && misaligned({bases})) return G3H_E_INVAL;
  if (n_bases > (1u << G3H_MSM_MAX_LOG)) return G3H_E_RANGE;
  DeviceGuard guard(c->device);
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return G3H_E_CUDA;
  msm_free(m);
  if (n_bases == 0) return G3H_OK;
  const size_t n = n_bases;
  auto alloc = [](void** p, size_t bytes) { return raw_alloc(p, bytes); };
  int rc = alloc(&m.table, n * kMsmWindows * sizeof(Aff));
  if (rc == G3H_OK) rc = dalloc(&m.entries, n * kMsmWindows);
  // per-bucket counters, then the long-run list: its count and up to kMsmBuckets indices
  if (rc == G3H_OK) rc = dalloc(&m.counts, 2 * kMsmBuckets + 1);
  if (rc == G3H_OK) rc = dalloc(&m.offsets, kMsmBuckets + 1);
  m.sort_blocks = (uint32_t)c->sm_count;
  if (rc == G3H_OK) rc = dalloc(&m.block_counts, (size_t)m.sort_blocks * kMsmBuckets);
  if (rc == G3H_OK) rc = alloc(&m.buckets, kMsmBuckets * sizeof(Pt));
  if (rc == G3H_OK) rc = alloc(&m.spill, 2 * (n + 1) * sizeof(Pt));
  if (rc == G3H_OK) rc = alloc(&m.groups, 2 * kMsmPairs * sizeof(Pt));
  if (rc == G3H_OK)
    rc = alloc(&m.parts, (kMsmSumParts * msm_chunks<G>() + kMsmSumParts + 1 +
                          (size_t)c->sm_count * 2) * sizeof(Pt));
  if (rc == G3H_OK) rc = alloc(&m.result, 3 * sizeof(typename G::F));
  int per_sm = 0;
  if (rc == G3H_OK &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_msm_accumulate<G>, G::kTree, 0) !=
          cudaSuccess)
    rc = G3H_E_CUDA;
  m.slots = (uint32_t)std::max(per_sm, 1) * G::kTree * (uint32_t)c->sm_count;
  const Aff* src = (const Aff*)bases;
  void* tmp = nullptr;
  if (rc == G3H_OK && !(flags & G3H_DEVICE_PTRS)) {
    rc = alloc(&tmp, n * sizeof(Aff));
    if (rc == G3H_OK) rc = h2d(c, tmp, bases, n * sizeof(Aff));
    src = (const Aff*)tmp;
  }
  if (rc == G3H_OK)
    rc = run(c, "msm_precompute", [&] {
      k_msm_precompute<G><<<blocks_for(n, 128), 128, 0, c->stream>>>(src, n_bases, (Aff*)m.table,
                                                                     c->d_err);
    });
  const int rc2 = finish(c);
  if (tmp) cudaFree(tmp);
  if (rc == G3H_OK) rc = rc2;
  if (rc != G3H_OK) {
    msm_free(m);
    return rc;
  }
  m.n = n_bases;
  return G3H_OK;
}

template <class G>
int msm_run(g3h_ctx* c, MsmState& m, const uint32_t* scalars, uint32_t count, uint32_t* result,
            uint32_t flags) {
  using F = typename G::F;
  if (!c || !result || (!scalars && count)) return G3H_E_INVAL;
  if (count > m.n) return G3H_E_RANGE;
  DeviceGuard guard(c->device);
  NvtxRange range(G::kName);
  const bool dev = (flags & G3H_DEVICE_PTRS) != 0;
  if (dev && misaligned({scalars, result})) return G3H_E_INVAL;
  const uint32_t check = (flags & G3H_NOCHECK) ? 0u : 1u;
  if (count == 0) {  // the empty sum: infinity
    if (dev)
      return cudaMemsetAsync(result, 0, 3 * sizeof(F), c->stream) == cudaSuccess ? G3H_OK
                                                                                : G3H_E_CUDA;
    std::memset(result, 0, 3 * sizeof(F));
    return G3H_OK;
  }
  F* out = dev ? (F*)result : (F*)m.result;
  const fr_t* s = (const fr_t*)scalars;
  int rc = G3H_OK;
  if (!dev) {
    rc = ensure_stage(c, count);
    if (rc == G3H_OK) rc = h2d(c, c->d_stage, scalars, (size_t)count * sizeof(fr_t));
    s = c->d_stage;
  }
  if (rc == G3H_OK) rc = msm_launches<G>(c, m, s, count, out, check);
  if (dev) return rc;
  if (rc == G3H_OK) rc = d2h(c, result, out, 3 * sizeof(F));
  const int rc2 = finish(c);
  return rc != G3H_OK ? rc : rc2;
}

}  // namespace

extern "C" {

int g3h_msm_prepare(g3h_ctx* c, const uint32_t* bases, uint32_t n_bases, uint32_t flags) {
  if (!c) return G3H_E_INVAL;
  return msm_prepare<G1>(c, c->msm1, bases, n_bases, flags);
}

int g3h_msm(g3h_ctx* c, const uint32_t* scalars, uint32_t count, uint32_t* result,
            uint32_t flags) {
  if (!c) return G3H_E_INVAL;
  return msm_run<G1>(c, c->msm1, scalars, count, result, flags);
}

int g3h_msm_g2_prepare(g3h_ctx* c, const uint32_t* bases, uint32_t n_bases, uint32_t flags) {
  if (!c) return G3H_E_INVAL;
  return msm_prepare<G2>(c, c->msm2, bases, n_bases, flags);
}

int g3h_msm_g2(g3h_ctx* c, const uint32_t* scalars, uint32_t count, uint32_t* result,
               uint32_t flags) {
  if (!c) return G3H_E_INVAL;
  return msm_run<G2>(c, c->msm2, scalars, count, result, flags);
}

int g3h_sync(g3h_ctx* c) {
  if (!c) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  return finish(c);
}

void g3h_destroy(g3h_ctx* c) {
  if (!c) return;
  DeviceGuard guard(c->device);
  cudaStreamSynchronize(c->stream);
  release(c);
  delete c;
}

const char* g3h_strerror(int code) {
  switch (code) {
    case G3H_OK: return "ok";
    case G3H_E_INVAL: return "invalid argument";
    case G3H_E_NONCANON: return "input field element not canonical (>= r)";
    case G3H_E_RANGE: return "value out of range (log_n, CSR row pointers or column index)";
    case G3H_E_NOMEM: return "out of memory";
    case G3H_E_CUDA: return "CUDA runtime error";
    case G3H_E_POINT: return "a multiexp base point is not on its curve";
    default: return "unknown error";
  }
}

int g3h_info(const g3h_ctx* c, uint32_t* log_n, uint32_t* n_wires) {
  if (!c) return G3H_E_INVAL;
  if (log_n) *log_n = c->log_n;
  if (n_wires) *n_wires = c->n_wires;
  return G3H_OK;
}

int g3h_timing_enable(g3h_ctx* c, int enable) {
  if (!c) return G3H_E_INVAL;
  if (enable) {
    c->launches.clear();
    c->events_used = 0;
  }
  c->timing = enable != 0;
  return G3H_OK;
}

int g3h_timing_read(g3h_ctx* c, g3h_kernel_time* out, int max, int* count) {
  if (!c || (!out && max > 0)) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return G3H_E_CUDA;
  std::vector<g3h_kernel_time> agg;
  for (const TimedLaunch& l : c->launches) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, l.e0, l.e1) != cudaSuccess) return G3H_E_CUDA;
    size_t i = 0;
    while (i < agg.size() && std::strcmp(agg[i].name, l.name) != 0) i++;
    if (i == agg.size()) agg.push_back({l.name, 0u, 0.0});
    agg[i].launches++;
    agg[i].ms += ms;
  }
  for (int i = 0; i < max && i < (int)agg.size(); i++) out[i] = agg[i];
  if (count) *count = (int)agg.size();
  return G3H_OK;
}

}  // extern "C"

namespace g3h {

// Throughput probes of the integer multiply pipe, for the roofline's denominator: eight
// independent chains per thread, sixteen steps per chain and loop iteration, of
//   KIND 0: 32-bit multiply-adds, low word (mad.lo.u32, y <- y * c + a);
//   KIND 1: 32-bit multiply-adds, high word (mad.hi.u32, y <- hi(y * c) + a);
//   KIND 2: full 32 x 32 -> 64-bit multiply-adds (mad.wide.u32, x <- lo(x) * c + x).
// Every product takes the chain's value so far, so none can be computed once and reused.
// Nothing is read; sink[0] is written only if the chains' final values XOR to `seed`,
// which keeps them live. Launch: any grid of 256 threads.
template <int KIND>
__global__ void __launch_bounds__(256) k_imad_probe(uint64_t* sink, uint32_t iters, uint32_t seed) {
  uint32_t y[8], a[8];
  uint64_t x[8];
#pragma unroll
  for (int k = 0; k < 8; k++) {
    a[k] = seed * (threadIdx.x + 1u) + (uint32_t)k * 0x9e3779b9u;
    y[k] = a[k];
    x[k] = a[k];
  }
  const uint32_t c = seed ^ (blockIdx.x * 0x85ebca6bu);
  for (uint32_t it = 0; it < iters; it++) {
#pragma unroll
    for (int r = 0; r < 16; r++) {
#pragma unroll
      for (int k = 0; k < 8; k++) {
        if (KIND == 0)
          asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(y[k]) : "r"(c ^ a[k]), "r"(a[k]));
        else if (KIND == 1)
          asm volatile("mad.hi.u32 %0, %0, %1, %2;" : "+r"(y[k]) : "r"(c ^ a[k]), "r"(a[k]));
        else
          asm volatile("{\n\t.reg .u32 lo;\n\tcvt.u32.u64 lo, %0;\n\tmad.wide.u32 %0, lo, %1, %0;\n\t}"
                       : "+l"(x[k]) : "r"(c ^ a[k]));
      }
    }
  }
  uint64_t s = 0;
#pragma unroll
  for (int k = 0; k < 8; k++) s ^= (uint64_t)y[k] ^ x[k];
  if (s == (uint64_t)seed) sink[0] = s;
}

}  // namespace g3h

namespace {

int measure_mul(g3h_ctx* c, int kind, double* per_s) {
  if (!c || !per_s || kind < 0 || kind > 2) return G3H_E_INVAL;
  DeviceGuard guard(c->device);
  uint64_t* sink = nullptr;
  if (cudaMalloc((void**)&sink, sizeof(uint64_t)) != cudaSuccess) return G3H_E_NOMEM;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int rc = cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess
               ? G3H_OK
               : G3H_E_CUDA;
  // four blocks of eight warps per SM; a few ms a run
  const unsigned grid = (unsigned)c->sm_count * 4;
  const uint32_t iters = kind == 0 ? 4096u : 2048u;
  auto launch = [&](uint32_t it, uint32_t seed) {
    if (kind == 0) k_imad_probe<0><<<grid, 256, 0, c->stream>>>(sink, it, seed);
    else if (kind == 1) k_imad_probe<1><<<grid, 256, 0, c->stream>>>(sink, it, seed);
    else k_imad_probe<2><<<grid, 256, 0, c->stream>>>(sink, it, seed);
  };
  double best = 0.0;
  for (int run = 0; run < 4 && rc == G3H_OK; run++) {
    const uint32_t it = run == 0 ? 64u : iters;  // the first run warms up
    launch(it, 0x2545f491u + (uint32_t)run);
    if (cudaGetLastError() != cudaSuccess) rc = G3H_E_CUDA;
    if (run == 0 || rc != G3H_OK) continue;
    cudaEventRecord(e0, c->stream);
    launch(it, 0x9e3779b1u + (uint32_t)run);
    cudaEventRecord(e1, c->stream);
    float ms = 0.f;
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess || ms <= 0.f) {
      rc = G3H_E_CUDA;
      continue;
    }
    const double ops = (double)grid * 256.0 * it * 16.0 * 8.0;
    best = std::max(best, ops / (ms * 1e-3));
  }
  if (rc == G3H_OK && cudaStreamSynchronize(c->stream) != cudaSuccess) rc = G3H_E_CUDA;
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(sink);
  if (rc == G3H_OK) *per_s = best;
  return rc;
}

}  // namespace

extern "C" {

int g3h_measure_imad(g3h_ctx* c, double* results_per_s) {
  return measure_mul(c, G3H_MUL_LO, results_per_s);
}

int g3h_measure_int_mul(g3h_ctx* c, int kind, double* per_s) {
  return measure_mul(c, kind, per_s);
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// g3h_compute_h_abc_static: steps 2-5 without any allocation.
//
// For callers that cannot allocate device memory themselves or through this library: a
// framework whose caching allocator must own every device byte, or a latency-critical path
// that cannot take cudaMalloc's device-wide synchronisation.
// The working vectors and the domain tables live in one file-scope device array of fixed
// size, reserved on every GPU that loads this library until the process exits:
// (in 32-byte elements; a table entry (w, w') takes two)
//   [0, 3N)          the three working vectors a, b, c
//   [3N, 4N)         forward twiddles omega^j, j < n/2
//   [4N, 5N)         inverse twiddles omega^-j, j < n/2
//   [5N, 7N)         shift table g^brev(p) / n
//   [7N, 7N + 6)     domain constants
//   [7N + 6]         word 0: log_n + 1 of the domain whose tables [3N, 7N + 6) hold, 0 for
//                    none (the array starts zeroed when the library is loaded)
// with N = 2^16, the largest domain this entry point accepts: 7N + 8 elements of 32 bytes,
// 14 MiB. Whether the tables match a call's log_n is decided on the GPU, in stream order,
// by that call's own table kernels (k_static_domain, k_static_tables, k_static_tag): the
// host keeps no record of it, so the outcome does not depend on which calls the host made
// before. Every other element of the array that a call reads was written earlier in the
// same call, so nothing else has to start at zero.
namespace {
constexpr uint32_t kNoAllocMaxLog = 16;
constexpr size_t kNoAllocN = (size_t)1 << kNoAllocMaxLog;
constexpr size_t kNoAllocElems = 7 * kNoAllocN + 8;
}  // namespace

static __device__ __align__(256) fr_t g3h_noalloc_scratch[kNoAllocElems];

namespace g3h {

// The domain constants of 2^k into consts, unless *tag says the tables already hold 2^k.
// Launch: 1 block of 1 thread.
__global__ void k_static_domain(fr_t* consts, const uint32_t* tag, uint32_t k) {
  if (*tag == k + 1u) return;
  domain_constants(consts, k);
}

// The three tables of 2^k (forward and inverse twiddles, n/2 entries each, and the shift
// table, n entries), one entry per thread, unless *tag says they already hold 2^k.
// Launch: ceil(2n / 256) x 256.
__global__ void k_static_tables(fr_const_t* tw_fwd, fr_const_t* tw_inv, fr_const_t* shift,
                                const fr_t* consts, const uint32_t* tag, uint32_t k) {
  if (*tag == k + 1u) return;
  const size_t n = (size_t)1 << k, half = n >> 1;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < half)
    tw_fwd[i] = pow_table_entry(consts, 0, -1, (uint32_t)i);
  else if (i < 2 * half)
    tw_inv[i - half] = pow_table_entry(consts, 1, -1, (uint32_t)(i - half));
  else if (i < 2 * half + n)
    shift[i - 2 * half] = pow_table_entry(consts, 2, 4, bitrev((uint32_t)(i - 2 * half), k));
}

// Records that the tables hold 2^k. Launch: 1 block of 1 thread, after k_static_tables.
__global__ void k_static_tag(uint32_t* tag, uint32_t k) { *tag = k + 1u; }

}  // namespace g3h

namespace {

constexpr int kNoAllocMaxDevices = 64;
fr_t* g_noalloc_base[kNoAllocMaxDevices];  // device address of the array, per device
std::mutex g_noalloc_mu;

int noalloc_launch_ok() { return cudaGetLastError() == cudaSuccess ? G3H_OK : G3H_E_CUDA; }

}  // namespace

extern "C" int g3h_compute_h_abc_static(uint32_t log_n, const uint32_t* a, const uint32_t* b,
                                        const uint32_t* c, uint32_t* h_mont, uint32_t* h_std,
                                        void* stream) {
  if (!a || !b || !c || !h_mont || !h_std || misaligned({a, b, c, h_mont, h_std}))
    return G3H_E_INVAL;
  if (log_n > kNoAllocMaxLog) return G3H_E_RANGE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return G3H_E_CUDA;
  fr_t* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_base[dev]) {
      // One-time set-up on this device (the device is current): the host-side name of the
      // array is not a device address, so ask the runtime for the address.
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g3h_noalloc_scratch) != cudaSuccess || !p) return G3H_E_CUDA;
      g_noalloc_base[dev] = (fr_t*)p;
    }
    base = g_noalloc_base[dev];
  }
  const cudaStream_t s = (cudaStream_t)stream;
  const size_t n = (size_t)1 << log_n;
  fr_t* work = base;
  fr_const_t* tw_fwd = reinterpret_cast<fr_const_t*>(base + 3 * kNoAllocN);
  fr_const_t* tw_inv = tw_fwd + kNoAllocN / 2;
  fr_const_t* shift = tw_inv + kNoAllocN / 2;
  fr_t* consts = reinterpret_cast<fr_t*>(shift + kNoAllocN);
  uint32_t* tag = reinterpret_cast<uint32_t*>(consts + 6);
  k_static_domain<<<1, 1, 0, s>>>(consts, tag, log_n);
  k_static_tables<<<blocks_for(2 * n, 256), 256, 0, s>>>(tw_fwd, tw_inv, shift, consts, tag,
                                                          log_n);
  k_static_tag<<<1, 1, 0, s>>>(tag, log_n);
  if (noalloc_launch_ok() != G3H_OK) return G3H_E_CUDA;
  const fr_t* in[3] = {(const fr_t*)a, (const fr_t*)b, (const fr_t*)c};
  fr_t* hm = (fr_t*)h_mont;
  fr_t* hs = (fr_t*)h_std;
  if (log_n <= kSmallMaxLog) {
    k_small_quotient<<<1, 32, 0, s>>>(in[0], in[1], in[2], tw_inv, tw_fwd, shift, hm, hs, log_n,
                                       0u, nullptr);
    return noalloc_launch_ok();
  }
  fr_t* v[3] = {work, work + n, work + 2 * n};
  const Plan pl = plan_for(log_n);  // two levels: log_n <= 16
  auto args = [&]() {
    SliceArgs x;
    std::memset(&x, 0, sizeof(x));
    x.log_n = log_n;
    return x;
  };
  auto launch = [&](Slice which, const SliceArgs& x, unsigned nvec) {
    uint32_t threads = 0;
    void (*kern)(SliceArgs) = slice_kernel(which, x.kk, &threads);
    const dim3 grid((unsigned)(n >> x.kk), nvec);
    kern<<<grid, threads, (size_t)32 << x.kk, s>>>(x);
  };
  SliceArgs x = args();
  for (int i = 0; i < 3; i++) {
    x.src[i] = in[i];
    x.dst[i] = v[i];
  }
  x.tw = tw_inv;
  x.kk = pl.kk[1];
  x.c0 = pl.c0[1];
  launch(Slice::dif, x, 3);
  SliceArgs m = args();
  for (int i = 0; i < 3; i++) m.dst[i] = v[i];
  m.tw = tw_inv;
  m.tw2 = tw_fwd;
  m.scale_tab = shift;
  m.kk = pl.kk[0];
  launch(Slice::mid, m, 3);
  SliceArgs t = args();
  for (int i = 0; i < 3; i++) t.src[i] = t.dst[i] = v[i];
  t.tw = tw_fwd;
  t.kk = pl.kk[1];
  t.c0 = pl.c0[1];
  t.mode = SL_JOIN;
  t.h_mont = hm;
  t.h_std = hs;
  launch(Slice::dit, t, 1);
  return noalloc_launch_ok();
}
