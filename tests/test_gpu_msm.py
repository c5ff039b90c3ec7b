"""GPU parity of the H multiexp over G1 (g3h_msm_prepare / g3h_msm) against the oracle.

The sum is one group element; the library writes it in Jacobian coordinates, whose
representation is not unique, so each result is mapped to its affine point by the
oracle's own arithmetic and compared limb for limb with the oracle's sum of s_i P_i.

Cases: ragged sizes (1 .. 4099 bases, fewer scalars than bases, none), host and device
buffers, scalars at the digit boundaries (2^15, 2^15 + 1, 2^16 - 1 in a window: the
signed-digit carry), 0, 1, r - 1, one scalar for every base (all entries in a few
buckets: the slices' load balance), witness scalars (mostly 0 and 1), equal bases with equal scalars (the doubling case of
the mixed addition), P and -P (cancellation), bases at infinity, equal and opposite
sums meeting in the bucket sum's last additions, the chain from g3h_compute_h's h_std,
the full 2^18 workload, and the input checks.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
from oracle import fr_int as F
from oracle import g1_int as G
from bn254_scalar_field_gb300 import build, g3h, synth, synth_g1

pytestmark = pytest.mark.gpu

R = F.R_MOD


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()
    yield


def _dev(x):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x).view(np.int32)).cuda()


def _affine(jac):
    return oracle.g1_jacobian_to_affine(np.asarray(jac, np.uint32).reshape(24))


def _oracle_msm(points, scalars, workers=None):
    """The oracle's sum, split over host threads (the C calls release the GIL); the chunk
    sums are added with the oracle's own addition."""
    n = points.shape[0]
    workers = workers or max(1, min(32, os.cpu_count() or 1))
    if n < 4096 or workers == 1:
        return oracle.g1_msm(points, scalars)
    oracle.g1_on_curve(points[:1])  # one-time constant set-up before the threads start
    bounds = np.linspace(0, n, workers + 1).astype(int)
    with ThreadPoolExecutor(workers) as ex:
        parts = list(ex.map(lambda k: oracle.g1_msm(points[bounds[k]:bounds[k + 1]],
                                                    scalars[bounds[k]:bounds[k + 1]]),
                            range(workers)))
    acc = parts[0].reshape(1, 16)
    for p in parts[1:]:
        acc = oracle.g1_add(acc, p.reshape(1, 16))
    return acc.reshape(16)


def _run(points, scalars, count=None, device=False):
    count = scalars.shape[0] if count is None else count
    with g3h.Context(0) as ctx:
        if device:
            ctx.msm_prepare(_dev(points))
            res = _dev(np.zeros(24, np.uint32))
            ctx.msm(_dev(scalars[:count]), res)
            ctx.sync()
            return _affine(res.cpu().numpy().view(np.uint32))
        ctx.msm_prepare(points)
        res = np.zeros(24, np.uint32)
        ctx.msm(np.ascontiguousarray(scalars[:count]), res)
        return _affine(res)


@pytest.mark.parametrize("n", [1, 2, 3, 17, 1000, 4099])
def test_msm_ragged_sizes(n):
    pts = synth_g1.points(n, seed=100 + n)
    s = synth_g1.scalars(n, seed=200 + n)
    assert np.array_equal(_run(pts, s), oracle.g1_msm(pts, s))


def test_msm_device_buffers_and_fewer_scalars():
    n = 3000
    pts = synth_g1.points(n, seed=7)
    s = synth_g1.scalars(n, seed=8)
    assert np.array_equal(_run(pts, s, device=True), oracle.g1_msm(pts, s))
    assert np.array_equal(_run(pts, s, count=1234), oracle.g1_msm(pts[:1234], s[:1234]))


def test_msm_empty_is_infinity():
    pts = synth_g1.points(4, seed=9)
    with g3h.Context(0) as ctx:
        ctx.msm_prepare(pts)
        res = np.full(24, 7, np.uint32)
        ctx.msm(np.zeros((0, 8), np.uint32), res)
        assert not res.any()
        res = np.full(24, 7, np.uint32)
        ctx.msm(np.zeros((4, 8), np.uint32), res)  # all scalars zero
        assert not res[16:].any()  # Z = 0


def test_msm_digit_boundaries_and_special_scalars():
    vals = [0, 1, 2, R - 1, R - 2, 1 << 15, (1 << 15) + 1, (1 << 16) - 1, 1 << 16,
            (1 << 31) + (1 << 15), int("8000" * 15 + "8001", 16) % R, int("ffff" * 15, 16),
            (1 << 253) + (1 << 15), sum(0x8000 << (16 * w) for w in range(15)) % R]
    n = 200
    pts = synth_g1.points(n, seed=11)
    s = synth_g1.scalars(n, seed=12)
    s[:len(vals)] = F.ints_to_array(vals)
    assert np.array_equal(_run(pts, s), oracle.g1_msm(pts, s))


def test_msm_one_scalar_for_all_bases():
    """Every base with the same scalar: the entries fill only 16 buckets, so most slices
    lie inside one bucket's run and the merge adds many parts."""
    n = 5000
    pts = synth_g1.points(n, seed=13)
    s = np.repeat(synth_g1.scalars(1, seed=14), n, axis=0)
    assert np.array_equal(_run(pts, s), _oracle_msm(pts, s))


def test_msm_repeated_scalar_long_runs():
    """Most scalars equal to 2 (not 1): all their digits land in one bucket whose run covers
    hundreds of slices, which the merge hands to a block per bucket."""
    n = 1 << 15
    pts = synth_g1.points(n, seed=31)
    s = synth_g1.scalars(n, seed=32)
    two = F.ints_to_array([2])[0]
    s[np.arange(n) % 5 != 0] = two
    assert np.array_equal(_run(pts, s, device=True), _oracle_msm(pts, s))


def test_msm_exceptional_additions():
    """Equal bases with equal scalars meet in one bucket (the mixed addition's doubling
    case); P and -P with equal scalars cancel; bases at infinity add nothing."""
    base = synth_g1.points(6, seed=15)  # base[1] = -base[0]
    pts = np.concatenate([np.repeat(base[:1], 40, axis=0), base[:2], np.zeros((3, 16), np.uint32),
                          base[2:]])
    s = synth_g1.scalars(pts.shape[0], seed=16)
    s[:40] = s[0]
    s[40:42] = s[45]
    assert np.array_equal(_run(pts, s), oracle.g1_msm(pts, s))
    # everything cancels: P, -P with equal scalars only
    pts2 = np.repeat(base[:2], 8, axis=0)
    s2 = np.repeat(synth_g1.scalars(1, seed=17), 16, axis=0)
    got = _run(pts2, s2)
    assert not got.any() and not oracle.g1_msm(pts2, s2).any()


def test_msm_tail_equal_and_opposite_sums():
    """The bucket sum's last additions on equal or opposite points (the exceptional cases
    of the whole-warp addition): P with scalar 2 makes the V part 2P, and two bases with
    scalar 1 make the ones' sum 2P or -2P, so the final sum adds 2P to 2P (a doubling) or
    to -2P (infinity)."""
    base = synth_g1.points(2, seed=15)  # base[1] = -base[0]
    two, one = F.ints_to_array([2]), F.ints_to_array([1])
    for second, cancels in ((base[:1], False), (base[1:2], True)):
        pts = np.concatenate([base[:1], second, second])
        s = np.concatenate([two, one, one])
        want = oracle.g1_msm(pts, s)
        assert np.array_equal(_run(pts, s), want)
        assert (not want.any()) == cancels


def test_msm_on_h_std():
    """Stage 9's input: the standard-form h of g3h_compute_h, on the device."""
    import torch

    log_n = 10
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=18)
    pts = synth_g1.points(n, seed=19)
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        hm = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
        hs = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
        ctx.compute_h(_dev(w), hm, hs)
        ctx.msm_prepare(pts)
        res = _dev(np.zeros(24, np.uint32))
        ctx.msm(hs, res)
        ctx.sync()
        got = _affine(res.cpu().numpy().view(np.uint32))
    _, want_hs = oracle.compute_h(log_n, A, B, w)
    assert np.array_equal(got, oracle.g1_msm(pts, want_hs))


@pytest.mark.parametrize("log_n", [12, 14])
def test_witness_msm_over_g1(log_n):
    """A witness multiexp (MSM_CU stages 5, 6, 8 over G1): the witness of the proving-key
    workload (90 / 95 % of wires 0 or 1) brought to standard form on the device
    (g3h_mont_to_std), then summed against bases; zeros add no entry, ones one entry each
    in the first bucket, which the slices spread over many threads."""
    import torch

    _, _, w = synth.problem(log_n)
    n = w.shape[0]
    pts = synth_g1.points(n, seed=900 + log_n)
    with g3h.Context(0) as ctx:
        wd = _dev(w)
        ws = torch.empty_like(wd)
        ctx.mont_to_std(wd, ws)
        ctx.msm_prepare(_dev(pts))
        res = _dev(np.zeros(24, np.uint32))
        ctx.msm(ws, res)
        ctx.sync()
        got = _affine(res.cpu().numpy().view(np.uint32))
    assert np.array_equal(got, _oracle_msm(pts, oracle.from_mont(w)))


def test_msm_full_2p18():
    """The full workload: 2^18 bases, uniform scalars in [0, r)."""
    n = 1 << 18
    pts = synth_g1.points(n, seed=synth_g1.default_seed(18))
    s = synth_g1.scalars(n, seed=synth_g1.default_seed(18) + 1)
    got = _run(pts, s, device=True)
    assert np.array_equal(got, _oracle_msm(pts, s))


def test_msm_input_checks():
    pts = synth_g1.points(8, seed=20)
    s = synth_g1.scalars(8, seed=21)
    with g3h.Context(0) as ctx:
        bad = pts.copy()
        bad[3, 8] ^= 1
        with pytest.raises(g3h.G3HError) as e:
            ctx.msm_prepare(bad)
        assert e.value.code == g3h.G3H_E_POINT
        bad = pts.copy()
        bad[5, :8] = F.int_to_limbs(G.Q_MOD)
        with pytest.raises(g3h.G3HError) as e:
            ctx.msm_prepare(bad)
        assert e.value.code == g3h.G3H_E_NONCANON
        ctx.msm_prepare(pts)
        res = np.zeros(24, np.uint32)
        with pytest.raises(g3h.G3HError) as e:
            ctx.msm(np.zeros((9, 8), np.uint32), res)
        assert e.value.code == g3h.G3H_E_RANGE
        s_bad = s.copy()
        s_bad[2] = F.int_to_limbs(R)
        with pytest.raises(g3h.G3HError) as e:
            ctx.msm(s_bad, res)
        assert e.value.code == g3h.G3H_E_NONCANON
        ctx.msm(s, res)  # the context is still usable
        assert np.array_equal(_affine(res), oracle.g1_msm(pts, s))


# ---------------------------------------------------------------------------- G2 ----

def _affine2(jac):
    return oracle.g2_jacobian_to_affine(np.asarray(jac, np.uint32).reshape(48))


def _oracle_msm2(points, scalars, workers=None):
    n = points.shape[0]
    workers = workers or max(1, min(32, os.cpu_count() or 1))
    if n < 1024 or workers == 1:
        return oracle.g2_msm(points, scalars)
    oracle.g2_on_curve(points[:1])
    bounds = np.linspace(0, n, workers + 1).astype(int)
    with ThreadPoolExecutor(workers) as ex:
        parts = list(ex.map(lambda k: oracle.g2_msm(points[bounds[k]:bounds[k + 1]],
                                                    scalars[bounds[k]:bounds[k + 1]]),
                            range(workers)))
    acc = parts[0].reshape(1, 32)
    for p in parts[1:]:
        acc = oracle.g2_add(acc, p.reshape(1, 32))
    return acc.reshape(32)


def _run2(points, scalars, device=False):
    with g3h.Context(0) as ctx:
        if device:
            ctx.msm_g2_prepare(_dev(points))
            res = _dev(np.zeros(48, np.uint32))
            ctx.msm_g2(_dev(scalars), res)
            ctx.sync()
            return _affine2(res.cpu().numpy().view(np.uint32))
        ctx.msm_g2_prepare(points)
        res = np.zeros(48, np.uint32)
        ctx.msm_g2(np.ascontiguousarray(scalars), res)
        return _affine2(res)


@pytest.mark.parametrize("n", [1, 2, 7, 300])
def test_msm_g2_ragged_sizes(n):
    """The multiexp over the twist (MSM_CU stage 7), host buffers."""
    from bn254_scalar_field_gb300 import synth_g2

    pts = synth_g2.points(n, seed=1000 + n)
    s = synth_g1.scalars(n, seed=1100 + n)
    if n == 300:
        s[:4] = F.ints_to_array([0, 1, R - 1, (1 << 15) + 1])
    assert np.array_equal(_run2(pts, s), oracle.g2_msm(pts, s))


def test_msm_g2_witness_and_full_size():
    """A witness as scalars (mostly 0 and 1) on 4096 twist points, device buffers, and
    uniform scalars on 2^16 points."""
    from bn254_scalar_field_gb300 import synth_g2

    _, _, w = synth.problem(12)
    pts = synth_g2.points(w.shape[0], seed=1200)
    ws = oracle.from_mont(w)
    assert np.array_equal(_run2(pts, ws, device=True), _oracle_msm2(pts, ws))
    n = 1 << 16
    pts = synth_g2.points(n, seed=synth_g2.default_seed(16))
    s = synth_g1.scalars(n, seed=synth_g2.default_seed(16) + 1)
    assert np.array_equal(_run2(pts, s, device=True), _oracle_msm2(pts, s))


def test_msm_g2_cancellation_and_checks():
    from bn254_scalar_field_gb300 import synth_g2
    from oracle import g2_int as G2

    base = synth_g2.points(6, seed=1300)  # base[1] = -base[0]
    pts = np.concatenate([np.repeat(base[:1], 20, axis=0), base[:2], np.zeros((2, 32), np.uint32)])
    s = synth_g1.scalars(pts.shape[0], seed=1301)
    s[:20] = s[0]
    s[20:22] = s[5]
    assert np.array_equal(_run2(pts, s), oracle.g2_msm(pts, s))
    with g3h.Context(0) as ctx:
        bad = base.copy()
        bad[2, 16] ^= 1
        with pytest.raises(g3h.G3HError) as e:
            ctx.msm_g2_prepare(bad)
        assert e.value.code == g3h.G3H_E_POINT
        bad = base.copy()
        bad[3, 8:16] = F.int_to_limbs(G2.Q_MOD)
        with pytest.raises(g3h.G3HError) as e:
            ctx.msm_g2_prepare(bad)
        assert e.value.code == g3h.G3H_E_NONCANON
