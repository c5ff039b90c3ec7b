"""Failure paths, made on the host (no GPU fault, trap or hang is ever caused).

The library's fault hook (G3H_FAULT, read by the library at each allocation, launch and
copy) makes the N-th device allocation fail as if out of memory ("alloc:N") or the N-th
kernel launch or copy report a CUDA error without being issued ("cuda:N"). Every entry
point must then return its error code (G3H_E_NOMEM, G3H_E_CUDA) without crashing, free
what it allocated, and leave the context (or a fresh one) computing bit-exact results.
"""
import os

import numpy as np
import pytest

import oracle
from bn254_scalar_field_gb300 import build, g3h, synth, synth_g1

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    oracle.build()
    yield
    os.environ.pop("G3H_FAULT", None)


class _Fault:
    def __init__(self, spec):
        self.spec = spec

    def __enter__(self):
        os.environ["G3H_FAULT"] = self.spec

    def __exit__(self, *exc):
        os.environ.pop("G3H_FAULT", None)


def _code(fn):
    try:
        fn()
    except g3h.G3HError as e:
        return e.code
    return g3h.G3H_OK


def _h(ctx, w, n):
    hm = np.zeros((n, 8), np.uint32)
    hs = np.zeros((n, 8), np.uint32)
    ctx.compute_h(w, hm, hs)
    return hm, hs


def test_prepare_fails_cleanly_at_every_allocation():
    import torch

    log_n = 20  # tables and scratch of tens of MiB each: a leak shows in the free memory
    n = 1 << log_n
    A, B, w = synth.problem(10, seed=77)  # small matrices in the large domain
    # one successful prepare first: the library's device code and its static array are
    # loaded on first use, which the baseline must already include
    g3h.Context(log_n, w.shape[0], A, B, device=0).close()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    failures = 0
    for i in range(1, 60):
        with _Fault("alloc:%d" % i):
            rc = _code(lambda: g3h.Context(log_n, w.shape[0], A, B, device=0).close())
        if rc == g3h.G3H_OK:
            break
        assert rc == g3h.G3H_E_NOMEM, (i, rc)
        failures += 1
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] >= free0 - (4 << 20), i
    assert failures >= 10  # every device and pinned allocation of g3h_prepare was failed once
    # the process still prepares and computes
    A, B, w = synth.problem(10, seed=78)
    with g3h.Context(10, w.shape[0], A, B) as ctx:
        hm, hs = _h(ctx, w, 1 << 10)
    want_m, want_s = oracle.compute_h(10, A, B, w)
    assert np.array_equal(hm, want_m) and np.array_equal(hs, want_s)
    del n


@pytest.mark.parametrize("log_n,points", [(4, 5), (10, 14)])
def test_injected_launch_and_copy_errors_leave_the_context_usable(log_n, points):
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=79)
    want_m, want_s = oracle.compute_h(log_n, A, B, w)
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        # the launches and copies of a host-pointer call each fail in turn (2^4: witness
        # copy, gather, one-block quotient, two result copies; 2^10: the copy, then the
        # launches captured into the launch graph: two gathers, three per transform phase,
        # the join's product and its reduction)
        for i in range(1, points + 1):
            with _Fault("cuda:%d" % i):
                rc = _code(lambda: _h(ctx, w, n))
            assert rc == g3h.G3H_E_CUDA, (i, rc)
        for flags in (0, g3h.G3H_NO_GRAPH, g3h.G3H_SERIALIZE):
            hm = np.zeros((n, 8), np.uint32)
            hs = np.zeros((n, 8), np.uint32)
            ctx.compute_h(w, hm, hs, flags=flags)
            assert np.array_equal(hm, want_m) and np.array_equal(hs, want_s), flags


def test_injected_errors_in_batch_lanes_and_coset_tables():
    log_n = 10
    n = 1 << log_n
    A, B, w = synth.problem(log_n, seed=80)
    want_m, want_s = oracle.compute_h(log_n, A, B, w)
    ws = np.stack([w, w, w])
    x = synth.uniform_fr(synth.SplitMix64(81), n)
    with g3h.Context(log_n, w.shape[0], A, B) as ctx:
        # the batch's extra lanes are allocated by its first call: fail each allocation
        for i in range(1, 5):
            with _Fault("alloc:%d" % i):
                rc = _code(lambda: ctx.compute_h_batch(ws, np.zeros((3, n, 8), np.uint32),
                                                       np.zeros((3, n, 8), np.uint32)))
            assert rc == g3h.G3H_E_NOMEM, (i, rc)
        hm = np.zeros((3, n, 8), np.uint32)
        hs = np.zeros((3, n, 8), np.uint32)
        ctx.compute_h_batch(ws, hm, hs)
        for i in range(3):
            assert np.array_equal(hm[i], want_m) and np.array_equal(hs[i], want_s), i
        # the coset tables are allocated and built by the first coset transform
        for spec in ("alloc:1", "alloc:2", "cuda:1", "cuda:2"):
            with _Fault(spec):
                got = x.copy()
                rc = _code(lambda: ctx.ntt(got, coset=True))
            assert rc in (g3h.G3H_E_NOMEM, g3h.G3H_E_CUDA), (spec, rc)
        got = x.copy()
        ctx.ntt(got, coset=True)
        assert np.array_equal(got, oracle.ntt(x, log_n, coset=True))


def test_injected_errors_in_the_multiexp():
    pts = synth_g1.points(64, seed=82)
    sc = synth_g1.scalars(64, seed=83)
    want = oracle.g1_msm(pts, sc)
    with g3h.Context(0) as ctx:
        for i in range(1, 12):
            with _Fault("alloc:%d" % i):
                rc = _code(lambda: ctx.msm_prepare(pts))
            if rc == g3h.G3H_OK:
                break
            assert rc == g3h.G3H_E_NOMEM, (i, rc)
        ctx.msm_prepare(pts)
        for i in (1, 3, 6):
            with _Fault("cuda:%d" % i):
                rc = _code(lambda: ctx.msm(sc, np.zeros(24, np.uint32)))
            assert rc == g3h.G3H_E_CUDA, (i, rc)
        res = np.zeros(24, np.uint32)
        ctx.msm(sc, res)
    assert np.array_equal(oracle.g1_jacobian_to_affine(res), want)


def test_malformed_fault_specs_inject_nothing():
    log_n = 6
    A, B, w = synth.problem(log_n, seed=84)
    want_m, _ = oracle.compute_h(log_n, A, B, w)
    for spec in ("", "alloc:", "alloc:0", "alloc:x", "disk:1", "cuda:-1"):
        with _Fault(spec):
            with g3h.Context(log_n, w.shape[0], A, B) as ctx:
                hm, _ = _h(ctx, w, 1 << log_n)
        assert np.array_equal(hm, want_m), spec
