"""The allocation-free entry point g3h_compute_h_abc_static, through the C ABI.

Some callers cannot allocate device memory: a framework whose caching allocator must own
every device byte, or a latency-critical path that cannot take cudaMalloc's device-wide
synchronisation. This entry point serves them from a fixed array inside the library. It
must give the bits of g3h_compute_h_abc and of the CPU oracle, call after call (the array
keeps the previous call's contents), across changes of domain in either direction (the
tables in the array are rebuilt only when a call's domain differs from the one they
hold), and refuse domains beyond its fixed size and pointers it cannot use.

This file is named to be collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

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


def _dev(x):
    import torch

    return torch.from_numpy(x.view(np.int32)).cuda()


def _call_static(log_n, a, b, c, hm, hs):
    import torch

    L = g3h.lib()
    stream = torch.cuda.current_stream().cuda_stream
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return L.g3h_compute_h_abc_static(log_n, ptr(a), ptr(b), ptr(c), ptr(hm), ptr(hs),
                                      ctypes.c_void_p(stream) if stream else None)


def _with_context(log_n, a, b, c):
    n = 1 << log_n
    hm = np.zeros((n, 8), np.uint32)
    hs = np.zeros((n, 8), np.uint32)
    with g3h.Context(log_n) as ctx:
        ctx.compute_h_abc(a, b, c, hm, hs)
    return hm, hs


def _run_sequence(sizes, seed):
    import torch

    for call, log_n in enumerate(sizes):
        n = 1 << log_n
        rng = synth.SplitMix64(seed + 31 * call + log_n)
        a, b, c = (synth.uniform_fr(rng, n) for _ in range(3))
        want_m, want_s = oracle.compute_h_abc(log_n, a, b, c)
        ctx_m, ctx_s = _with_context(log_n, a, b, c)
        assert np.array_equal(ctx_m, want_m) and np.array_equal(ctx_s, want_s), log_n
        hm = torch.full((n, 8), -1, dtype=torch.int32, device="cuda")
        hs = torch.full((n, 8), -1, dtype=torch.int32, device="cuda")
        assert _call_static(log_n, _dev(a), _dev(b), _dev(c), hm, hs) == g3h.G3H_OK
        torch.cuda.synchronize()
        got_m = hm.cpu().numpy().view(np.uint32)
        got_s = hs.cpu().numpy().view(np.uint32)
        assert np.array_equal(got_m, want_m), (call, log_n)
        assert np.array_equal(got_s, want_s), (call, log_n)


@pytest.mark.parametrize("log_n", [3, 6, 11, 12, 13, 16])
def test_static_entry_twice_against_oracle_and_context(log_n):
    # two calls in a row on one domain: slices of equal halves (6, 12, 16: the largest,
    # two 2^8 slices) and unequal ones (11, 13), and the one-block path (3)
    _run_sequence([log_n, log_n], 0x5A7)


def test_static_entry_across_domain_changes():
    # up, down, back up: the tables follow every change of domain
    _run_sequence([12, 14, 12, 16, 5, 16, 0], 0x5B1)


def test_static_entry_limits():
    import torch

    big = torch.zeros((8, 8), dtype=torch.int32, device="cuda")
    # beyond the fixed array: refused, nothing launched
    assert _call_static(17, big, big, big, big, big) == g3h.G3H_E_RANGE
    L = g3h.lib()
    assert L.g3h_compute_h_abc_static(4, None, None, None, None, None, None) == g3h.G3H_E_INVAL
    # a pointer off a 16-byte boundary is refused and nothing is written
    n = 16
    buf = torch.zeros((n + 1, 8), dtype=torch.int32, device="cuda")
    out = torch.full((n, 8), 7, dtype=torch.int32, device="cuda")
    off = ctypes.c_void_p(buf.data_ptr() + 4)
    ok = ctypes.c_void_p(buf.data_ptr())
    rc = L.g3h_compute_h_abc_static(4, off, ok, ok, ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(out.data_ptr()), None)
    assert rc == g3h.G3H_E_INVAL
    torch.cuda.synchronize()
    assert int((out != 7).sum()) == 0
