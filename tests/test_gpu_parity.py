"""GPU parity: every entry point of the C ABI against the CPU oracle, bit for bit.

Field arithmetic is exact, so the bar is equality of every limb of every element. Sizes
run from 2^0 through the four proving-key-shaped domains (2^12, 2^14, 2^17, 2^18) to the
2^22 stress vectors, covering every slice geometry the launch plan uses: the small
one-block path (2^0..2^5), two levels with equal and unequal halves (2^6..2^22), and
three levels (2^23). Ragged cases: constraint rows fewer than the domain, empty
matrices, a single-row domain.
"""
import numpy as np
import pytest

import oracle
from bn254_scalar_field_gb300 import build, g3h, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()
    yield


def _torch():
    import torch

    return torch


def _dev(x):
    torch = _torch()
    return torch.from_numpy(x.view(np.int32)).cuda()


def _host(t):
    return t.cpu().numpy().view(np.uint32)


def _zeros(n):
    return np.zeros((n, 8), np.uint32)


def _edge_fr():
    from oracle import fr_int as F

    r = F.R_MOD
    vals = [0, 1, 2, r - 1, r - 2, (1 << 256) % r, (1 << 253), (r - 1) // 2, 0xFFFFFFFF,
            (1 << 32), (1 << 224) - 1, r - (1 << 128)]
    return F.ints_to_array(vals)


# -------------------------------------------------------------------------- field ----

def test_mul_edge_and_random_values():
    a = np.concatenate([_edge_fr(), synth.uniform_fr(synth.SplitMix64(1), 5000)])
    b = np.concatenate([_edge_fr()[::-1], synth.uniform_fr(synth.SplitMix64(2), 5000)])
    # every edge value against every edge value
    e = _edge_fr()
    ea = np.repeat(e, e.shape[0], axis=0)
    eb = np.tile(e, (e.shape[0], 1))
    a = np.concatenate([a, ea])
    b = np.concatenate([b, eb])
    with g3h.Context(4) as ctx:
        out = _zeros(a.shape[0])
        ctx.mul(a, b, out)
    assert np.array_equal(out, oracle.fr_mul_vec(a, b))


@pytest.mark.parametrize("count", [0, 1, 7, 4099, (1 << 22) + 5])
def test_mont_to_std(count):
    """Montgomery to standard form, host and device buffers, out of place and in place;
    counts ragged against the grid and one larger than L2."""
    x = np.concatenate([_edge_fr(), synth.uniform_fr(synth.SplitMix64(5 + count), count)])[:count]
    want = oracle.from_mont(x) if count else x.copy()
    with g3h.Context(3) as ctx:
        out = _zeros(count)
        ctx.mont_to_std(x, out)
        assert np.array_equal(out, want)
        d = _dev(x)
        ctx.mont_to_std(d, d)
        ctx.sync()
        assert np.array_equal(_host(d).reshape(-1, 8), want)


def test_mont_to_std_rejects_noncanonical():
    from oracle import fr_int as F

    x = synth.uniform_fr(synth.SplitMix64(9), 1000)
    x[517] = F.ints_to_array([F.R_MOD])[0]
    with g3h.Context(3) as ctx:
        with pytest.raises(g3h.G3HError) as e:
            ctx.mont_to_std(x, _zeros(1000))
        assert e.value.code == g3h.G3H_E_NONCANON
        out = _zeros(1000)
        x[517] = 0
        ctx.mont_to_std(x, out)
        assert np.array_equal(out, oracle.from_mont(x))


# ---------------------------------------------------------------------- transforms ----

NTT_SIZES = list(range(0, 13)) + [13, 14, 16, 17, 18]


@pytest.mark.parametrize("log_n", NTT_SIZES)
def test_ntt_all_modes(log_n):
    n = 1 << log_n
    x = synth.uniform_fr(synth.SplitMix64(100 + log_n), n)
    with g3h.Context(log_n) as ctx:
        for inverse in (False, True):
            for coset in (False, True):
                got = x.copy()
                ctx.ntt(got, inverse=inverse, coset=coset)
                want = oracle.ntt(x, log_n, inverse=inverse, coset=coset)
                assert np.array_equal(got, want), (inverse, coset)


@pytest.mark.parametrize("log_n", [19, 20, 21, 23])
def test_ntt_large_and_three_levels(log_n):
    """2^19 and 2^20 run radix-4 pass pairs on 2^10 slices, 2^21 mixes 2^10 and 2^11
    slices (the 256-thread radix-4 build on the latter), 2^23 takes three levels."""
    n = 1 << log_n
    x = synth.uniform_fr(synth.SplitMix64(200 + log_n), n)
    with g3h.Context(log_n) as ctx:
        got = x.copy()
        ctx.ntt(got, coset=True)
        assert np.array_equal(got, oracle.ntt(x, log_n, coset=True))
        ctx.ntt(got, inverse=True, coset=True)
        assert np.array_equal(got, x)


def test_ntt_largest_domain_sampled():
    """The largest domain, 2^27 (4 GiB per vector): the forward coset transform's outputs
    at sampled points against the oracle's Horner evaluation at g omega^i (the whole
    oracle transform would take minutes), then the inverse brings back the input exactly."""
    from oracle import fr_int as F

    log_n = g3h.G3H_MAX_LOG_N
    n = 1 << log_n
    x = synth.uniform_fr(synth.SplitMix64(271), n)
    omega, gen = (F.limbs_to_int(v) for v in oracle.domain(log_n))
    with g3h.Context(log_n) as ctx:
        got = x.copy()
        ctx.ntt(got, coset=True)
        for i in (0, 1, n // 2 + 12345, n - 1):
            z = F.ints_to_array([F.to_mont(gen * pow(omega, i, F.R_MOD) % F.R_MOD)])
            assert np.array_equal(got[i], oracle.poly_eval(x, z)), i
        ctx.ntt(got, inverse=True, coset=True)
        assert np.array_equal(got, x)


# -------------------------------------------------------------------------- gather ----

@pytest.mark.parametrize("log_n", [0, 1, 3, 7, 10, 12, 14])
def test_gather(log_n):
    A, B, w = synth.problem(log_n, seed=300 + log_n)
    n = 1 << log_n
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        a, b, c = _zeros(n), _zeros(n), _zeros(n)
        ctx.gather(w, a, b, c)
    ra, rb, rc = oracle.gather(log_n, A, B, w)
    assert np.array_equal(a, ra) and np.array_equal(b, rb) and np.array_equal(c, rc)


def test_join_unfused_kernel():
    n = 1 << 11
    rng = synth.SplitMix64(77)
    ea, eb, ec = (synth.uniform_fr(rng, n) for _ in range(3))
    with g3h.Context(11) as ctx:
        hm, hs = _zeros(n), _zeros(n)
        ctx.join(ea, eb, ec, hm, hs)
    prod = oracle.fr_mul_vec(ea, eb)
    want = np.stack([oracle.fr_sub(prod[i:i + 1], ec[i:i + 1])[0] for i in range(n)])
    assert np.array_equal(hm, want)
    assert np.array_equal(hs, oracle.from_mont(want))


# --------------------------------------------------------------------- whole path ----

@pytest.mark.parametrize("log_n", list(range(0, 12)))
def test_compute_h_small_domains(log_n):
    A, B, w = synth.problem(log_n, seed=400 + log_n)
    n = 1 << log_n
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        hm, hs = _zeros(n), _zeros(n)
        ctx.compute_h(w, hm, hs)
    want_m, want_s = oracle.compute_h(log_n, A, B, w)
    assert np.array_equal(hm, want_m)
    assert np.array_equal(hs, want_s)


@pytest.mark.parametrize("log_n", [12, 14, 17, 18])
def test_compute_h_proving_key_configs(log_n):
    """The four proving-key-shaped workloads, every output element compared."""
    A, B, w = synth.problem(log_n)
    n = 1 << log_n
    want_m, want_s = oracle.compute_h(log_n, A, B, w)
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        hm, hs = _zeros(n), _zeros(n)
        ctx.compute_h(w, hm, hs)
        assert np.array_equal(hm, want_m)
        assert np.array_equal(hs, want_s)
        # the join fused into the last forward kernel (POINTWISE_CU: the fused path the
        # standalone join kernel checks) gives the same bits
        hm2, hs2 = _zeros(n), _zeros(n)
        ctx.compute_h(w, hm2, hs2, flags=g3h.G3H_FUSED_JOIN)
        assert np.array_equal(hm2, hm) and np.array_equal(hs2, hs)
        # all on one stream, fused on one stream, and without the launch graph
        for fl in (g3h.G3H_SERIALIZE, g3h.G3H_SERIALIZE | g3h.G3H_FUSED_JOIN,
                   g3h.G3H_NO_GRAPH, g3h.G3H_NO_GRAPH | g3h.G3H_SERIALIZE):
            hm2, hs2 = _zeros(n), _zeros(n)
            ctx.compute_h(w, hm2, hs2, flags=fl)
            assert np.array_equal(hm2, hm) and np.array_equal(hs2, hs), fl
        # device pointers, asynchronous on the context's stream, twice in a row
        torch = _torch()
        wd = _dev(w)
        for _ in range(2):
            hmd = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
            hsd = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
            ctx.compute_h(wd, hmd, hsd)
            ctx.sync()
            assert np.array_equal(_host(hmd), want_m)
            assert np.array_equal(_host(hsd), want_s)


@pytest.mark.parametrize("max_len", [8, 9, 200])
def test_compute_h_row_lengths(max_len):
    """Rows of at most 8 terms are summed a lane each and longer ones by the whole warp:
    matrices whose rows stop at exactly 8 terms (every row a lane's), at 9, and reach 200,
    through the single and the batched path, against the oracle."""
    log_n = 10
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=800 + max_len, max_a=max_len, max_b=max_len)
    lens = np.diff(np.asarray(B[0], np.int64))
    assert lens.max() == max_len or max_len == 200
    want_m, want_s = oracle.compute_h(log_n, A, B, w)
    ws = np.stack([w, synth.witness(synth.SplitMix64(900 + max_len), w.shape[0], 0.5)])
    want2 = oracle.compute_h(log_n, A, B, ws[1])
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        for fl in (0, g3h.G3H_SERIALIZE):
            hm, hs = _zeros(n), _zeros(n)
            ctx.compute_h(w, hm, hs, flags=fl)
            assert np.array_equal(hm, want_m) and np.array_equal(hs, want_s), fl
        hm = np.zeros((2, n, 8), np.uint32)
        hs = np.zeros((2, n, 8), np.uint32)
        ctx.compute_h_batch(ws, hm, hs)
        assert np.array_equal(hm[0], want_m) and np.array_equal(hs[0], want_s)
        assert np.array_equal(hm[1], want2[0]) and np.array_equal(hs[1], want2[1])


@pytest.mark.parametrize("log_n", [4, 12, 14])
def test_compute_h_batch(log_n):
    """Batched H (several witnesses, one prepared context): every witness's output equals
    the oracle's, with more witnesses than lanes, in host and device memory."""
    A, B, w0 = synth.problem(log_n, seed=600 + log_n)
    n = 1 << log_n
    nw = w0.shape[0]
    count = 5
    ws = np.stack([w0] + [synth.witness(synth.SplitMix64(700 + i), nw, 0.9)
                          for i in range(count - 1)])
    want = [oracle.compute_h(log_n, A, B, ws[i]) for i in range(count)]
    with g3h.Context(log_n, nw, A, B) as ctx:
        hm = np.zeros((count, n, 8), np.uint32)
        hs = np.zeros((count, n, 8), np.uint32)
        ctx.compute_h_batch(ws, hm, hs)
        for i in range(count):
            assert np.array_equal(hm[i], want[i][0]) and np.array_equal(hs[i], want[i][1]), i
        torch = _torch()
        wd = torch.from_numpy(ws.view(np.int32)).cuda()
        hmd = torch.zeros((count, n, 8), dtype=torch.int32, device="cuda")
        hsd = torch.zeros((count, n, 8), dtype=torch.int32, device="cuda")
        ctx.compute_h_batch(wd, hmd, hsd)
        ctx.sync()
        for i in range(count):
            assert np.array_equal(_host(hmd[i]), want[i][0]), i
            assert np.array_equal(_host(hsd[i]), want[i][1]), i
        # one witness, and an empty batch
        h1m = np.zeros((1, n, 8), np.uint32)
        h1s = np.zeros((1, n, 8), np.uint32)
        ctx.compute_h_batch(ws[2:3], h1m, h1s)
        assert np.array_equal(h1m[0], want[2][0]) and np.array_equal(h1s[0], want[2][1])
        assert g3h.lib().g3h_compute_h_batch(ctx.handle, 0, None, None, None, 0) == g3h.G3H_OK


@pytest.mark.parametrize("log_n,count", [(6, 150), (14, 70), (16, 21)])
def test_compute_h_batch_chunks(log_n, count):
    """Batches on small and middle domains run one launch per phase for a chunk of
    witnesses (64 at 2^6 and 2^14, 16 at 2^16), chunks alternating between two lanes:
    several chunks, a ragged last one, every witness different, host and device memory,
    and the same context's single-witness call after it."""
    from concurrent.futures import ThreadPoolExecutor

    A, B, w0 = synth.problem(log_n, seed=900 + log_n)
    n = 1 << log_n
    nw = w0.shape[0]
    ws = np.stack([w0] + [synth.witness(synth.SplitMix64(910 + i), nw, 0.9)
                          for i in range(count - 1)])
    with ThreadPoolExecutor(8) as ex:
        want = list(ex.map(lambda i: oracle.compute_h(log_n, A, B, ws[i]), range(count)))
    with g3h.Context(log_n, nw, A, B) as ctx:
        hm = np.zeros((count, n, 8), np.uint32)
        hs = np.zeros((count, n, 8), np.uint32)
        ctx.compute_h_batch(ws, hm, hs)
        for i in range(count):
            assert np.array_equal(hm[i], want[i][0]) and np.array_equal(hs[i], want[i][1]), i
        torch = _torch()
        wd = torch.from_numpy(ws.view(np.int32)).cuda()
        hmd = torch.zeros((count, n, 8), dtype=torch.int32, device="cuda")
        hsd = torch.zeros((count, n, 8), dtype=torch.int32, device="cuda")
        ctx.compute_h_batch(wd, hmd, hsd)
        ctx.sync()
        got_m, got_s = _host(hmd), _host(hsd)
        for i in range(count):
            assert np.array_equal(got_m[i], want[i][0]), i
            assert np.array_equal(got_s[i], want[i][1]), i
        h1m, h1s = _zeros(n), _zeros(n)
        ctx.compute_h(ws[count - 1], h1m, h1s)
        assert np.array_equal(h1m, want[-1][0]) and np.array_equal(h1s, want[-1][1])


def test_compute_h_batch_reports_a_noncanonical_witness():
    """A batch on the z lanes with one witness holding a value >= r: the call reports
    G3H_E_NONCANON (host buffers) or the next sync does (device buffers), and the context
    computes bit-exact results afterwards."""
    log_n = 10
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=950)
    ws = np.stack([w] * 5)
    ws[3, :] = synth.MODULUS_LIMBS  # every wire of witness 3 (the gathers read some)
    want_m, want_s = oracle.compute_h(log_n, A, B, w)
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        hm = np.zeros((5, n, 8), np.uint32)
        hs = np.zeros((5, n, 8), np.uint32)
        with pytest.raises(g3h.G3HError) as ei:
            ctx.compute_h_batch(ws, hm, hs)
        assert ei.value.code == g3h.G3H_E_NONCANON
        torch = _torch()
        ctx.compute_h_batch(torch.from_numpy(ws.view(np.int32)).cuda(),
                            torch.zeros((5, n, 8), dtype=torch.int32, device="cuda"),
                            torch.zeros((5, n, 8), dtype=torch.int32, device="cuda"))
        with pytest.raises(g3h.G3HError) as ei:
            ctx.sync()
        assert ei.value.code == g3h.G3H_E_NONCANON
        good = np.stack([w] * 5)
        ctx.compute_h_batch(good, hm, hs)
        for i in range(5):
            assert np.array_equal(hm[i], want_m) and np.array_equal(hs[i], want_s), i


def test_compute_h_abc_stress_2_22():
    """The 2^22 NTT stress workload: a, b uniform, c = a*b, every element compared."""
    log_n = synth.STRESS_LOG_N
    n = 1 << log_n
    a, b = synth.stress_ab(log_n)
    c = oracle.fr_mul_vec(a, b)
    want_m, want_s = oracle.compute_h_abc(log_n, a, b, c)
    with g3h.Context(log_n) as ctx:
        c_gpu = _zeros(n)
        ctx.mul(a, b, c_gpu)
        assert np.array_equal(c_gpu, c)
        hm, hs = _zeros(n), _zeros(n)
        ctx.compute_h_abc(a, b, c, hm, hs)
    assert np.array_equal(hm, want_m)
    assert np.array_equal(hs, want_s)


@pytest.mark.parametrize("log_n", [19, 20])
def test_compute_h_abc_radix4_slices(log_n):
    """The quotient path on 2^10-element slices (radix-4 pass pairs in all three kernels)."""
    n = 1 << log_n
    rng = synth.SplitMix64(600 + log_n)
    a, b, c = (synth.uniform_fr(rng, n) for _ in range(3))
    want_m, want_s = oracle.compute_h_abc(log_n, a, b, c)
    with g3h.Context(log_n) as ctx:
        hm, hs = _zeros(n), _zeros(n)
        ctx.compute_h_abc(a, b, c, hm, hs)
    assert np.array_equal(hm, want_m) and np.array_equal(hs, want_s)


def test_compute_h_abc_three_levels():
    log_n = 23
    n = 1 << log_n
    rng = synth.SplitMix64(523)
    a, b, c = (synth.uniform_fr(rng, n) for _ in range(3))
    want_m, want_s = oracle.compute_h_abc(log_n, a, b, c)
    with g3h.Context(log_n) as ctx:
        hm, hs = _zeros(n), _zeros(n)
        ctx.compute_h_abc(a, b, c, hm, hs)
    assert np.array_equal(hm, want_m) and np.array_equal(hs, want_s)


# --------------------------------------------------------------------- edge cases ----

def test_ragged_rows_and_empty_matrices():
    log_n = 9
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=9)
    # fewer CSR rows than the domain: truncate both matrices to 300 and 123 rows
    def cut(m, rows):
        rp = m[0][:rows + 1].copy()
        nnz = int(rp[-1])
        return rp, m[1][:nnz].copy(), m[2][:nnz].copy()

    A2, B2 = cut(A, 300), cut(B, 123)
    with g3h.Context(log_n, w.shape[0], A2, B2) as ctx:
        hm, hs = _zeros(n), _zeros(n)
        ctx.compute_h(w, hm, hs)
    # the oracle takes one row count: pad the shorter matrices with empty rows
    def pad(m, rows):
        rp = np.concatenate([m[0], np.full(rows + 1 - m[0].shape[0], m[0][-1], np.uint32)])
        return rp, m[1], m[2]

    want_m, want_s = oracle.compute_h(log_n, pad(A2, n), pad(B2, n), w)
    assert np.array_equal(hm, want_m) and np.array_equal(hs, want_s)
    # empty matrices: a = b = c = 0, so h = 0
    E = (np.zeros(n + 1, np.uint32), np.zeros(0, np.uint32), np.zeros((0, 8), np.uint32))
    with g3h.Context(log_n, w.shape[0], E, E) as ctx:
        hm, hs = _zeros(n) + 7, _zeros(n) + 7
        ctx.compute_h(w, hm, hs)
    assert not hm.any() and not hs.any()


def test_noncanonical_inputs_reported_and_context_survives():
    log_n = 8
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=5)
    bad = w.copy()
    bad[0] = synth.MODULUS_LIMBS  # w[0] is referenced by the gather (the constant wire)
    bad[1:] = synth.MODULUS_LIMBS
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        hm, hs = _zeros(n), _zeros(n)
        with pytest.raises(g3h.G3HError) as ei:
            ctx.compute_h(bad, hm, hs)
        assert ei.value.code == g3h.G3H_E_NONCANON
        # device pointers: reported by the next sync
        torch = _torch()
        hmd = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
        hsd = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
        ctx.compute_h(_dev(bad), hmd, hsd)
        with pytest.raises(g3h.G3HError) as ei:
            ctx.sync()
        assert ei.value.code == g3h.G3H_E_NONCANON
        # and the context still computes correctly afterwards
        ctx.compute_h(w, hm, hs)
        want_m, want_s = oracle.compute_h(log_n, A, B, w)
        assert np.array_equal(hm, want_m) and np.array_equal(hs, want_s)
        x = _zeros(n)
        x[3] = synth.MODULUS_LIMBS
        with pytest.raises(g3h.G3HError):
            ctx.ntt(x)  # in place: x now holds the (unspecified) output
        x = _zeros(n)
        x[3] = synth.MODULUS_LIMBS
        with pytest.raises(g3h.G3HError):
            ctx.compute_h_abc(x, x, x, hm, hs)
        with pytest.raises(g3h.G3HError):
            ctx.join(x, x, x, hm, hs)
        with pytest.raises(g3h.G3HError):
            ctx.mul(x, x, hm)
        # gather: a non-canonical witness value referenced by the matrices
        a, b, c = _zeros(n), _zeros(n), _zeros(n)
        with pytest.raises(g3h.G3HError):
            ctx.gather(bad, a, b, c)
        # NOCHECK skips the checks: no error raised
        ctx.mul(x, x, hm, flags=g3h.G3H_NOCHECK)


def test_misaligned_device_pointers_refused():
    """A device pointer off a 16-byte boundary is refused at the C boundary before anything
    is launched (G3H_E_INVAL; the kernels move 16-byte vectors), and by the binding before
    the call; a tensor of another element width is refused by the binding."""
    import ctypes

    torch = _torch()
    L = g3h.lib()
    log_n = 6
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=9)
    buf = torch.zeros(8 * n + 8, dtype=torch.int32, device="cuda")
    good = ctypes.c_void_p(buf.data_ptr())
    off = ctypes.c_void_p(buf.data_ptr() + 4)
    D, INVAL = g3h.G3H_DEVICE_PTRS, g3h.G3H_E_INVAL
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        h = ctx.handle
        assert L.g3h_compute_h(h, off, good, good, D) == INVAL
        assert L.g3h_compute_h(h, good, good, off, D) == INVAL
        assert L.g3h_compute_h_abc(h, good, good, good, good, off, D) == INVAL
        assert L.g3h_compute_h_batch(h, 2, off, good, good, D) == INVAL
        assert L.g3h_gather(h, good, good, off, good, D) == INVAL
        assert L.g3h_ntt(h, off, 0, 1, D) == INVAL
        assert L.g3h_join(h, good, off, good, good, good, D) == INVAL
        assert L.g3h_mul(h, good, good, off, n, D) == INVAL
        assert L.g3h_mont_to_std(h, off, good, n, D) == INVAL
        assert L.g3h_msm_prepare(h, off, 4, D) == INVAL
        assert L.g3h_msm(h, good, 0, off, D) == INVAL
        assert L.g3h_msm_g2_prepare(h, off, 4, D) == INVAL
        assert L.g3h_msm_g2(h, off, 0, good, D) == INVAL
        ctx.sync()
        assert not buf.any()  # nothing ran
        # the binding refuses both before the call
        with pytest.raises(ValueError):
            ctx.mont_to_std(buf[1:1 + 8 * n], buf[8:8 + 8 * n])
        with pytest.raises(ValueError):
            ctx.mont_to_std(buf[:8 * n].view(torch.float32), buf[8:8 + 8 * n])
        # and the context still computes
        x = _edge_fr()
        xd = _dev(x)
        ctx.mont_to_std(xd, xd)
        from oracle import fr_int as F

        R = 1 << 256
        want = [v * pow(R, -1, F.R_MOD) % F.R_MOD for v in F.array_to_ints(x)]
        assert F.array_to_ints(_host(xd)) == want
    assert L.g3h_compute_h_abc_static(4, good, good, good, good, off, None) == INVAL


def test_measure_imad_probe():
    """The multiply-pipe probe returns a rate close to the derived peak (152 SMs x 64 32-bit
    IMAD results per clock at up to 2.07 GHz), its unit being the roofline's."""
    with g3h.Context(4) as ctx:
        rate = ctx.measure_imad()
    derived = 152 * 64 * 2.07e9
    assert 0.5 * derived < rate < 1.1 * derived


def test_domain_only_context_rejects_compute_h():
    with g3h.Context(6) as ctx:
        with pytest.raises(g3h.G3HError) as ei:
            ctx.compute_h(np.zeros((4, 8), np.uint32), _zeros(64), _zeros(64))
        assert ei.value.code == g3h.G3H_E_INVAL


def test_timing_records_kernels():
    log_n = 12
    A, B, w = synth.problem(log_n)
    n = 1 << log_n
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        ctx.timing_enable(True)
        hm, hs = _zeros(n), _zeros(n)
        ctx.compute_h(w, hm, hs)
        t = ctx.timing_read()
        ctx.timing_enable(False)
    # one stream per vector: the gathers of A and of B, three launches per transform phase,
    # the join's product and its reduction
    assert {k: v[0] for k, v in t.items()} == {"gather_a": 1, "gather_b": 1, "ntt_dif": 3,
                                               "ntt_mid": 3, "ntt_dit": 3, "prejoin": 1,
                                               "join": 1}
    assert all(v[1] > 0 for v in t.values())
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        ctx.timing_enable(True)
        hm2, hs2 = _zeros(n), _zeros(n)
        ctx.compute_h(w, hm2, hs2, flags=g3h.G3H_SERIALIZE)
        t = ctx.timing_read()
    assert {k: v[0] for k, v in t.items()} == {"gather_a": 1, "gather_b": 1, "ntt_dif": 1,
                                               "ntt_mid": 1, "ntt_dit": 1, "prejoin": 1,
                                               "join": 1}
    assert np.array_equal(hm2, hm) and np.array_equal(hs2, hs)
