"""The allocation-free entry point g3h_compute_h_abc_static, through the C ABI.

Callers that cannot allocate device memory (a framework allocator that must own every
byte, code running under stream capture, latency-critical paths) use this entry point; it
keeps its working vectors and tables in a fixed array inside the library. It must give
the same bits as g3h_compute_h_abc, call after call (the array keeps the previous call's
contents), across a change of domain, and refuse domains beyond its fixed size.

This file is named to be collected last, so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

from bn254_scalar_field_gb300 import build, g3h, synth

pytestmark = pytest.mark.gpu


def _dev(x):
    import torch

    return torch.from_numpy(x.view(np.int32)).cuda()


def _call_static(log_n, a, b, c, hm, hs):
    import torch

    L = g3h.lib()
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.g3h_compute_h_abc_static(
        log_n, ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()),
        ctypes.c_void_p(c.data_ptr()), ctypes.c_void_p(hm.data_ptr()),
        ctypes.c_void_p(hs.data_ptr()), ctypes.c_void_p(stream) if stream else None)
    return rc


def _reference(log_n, a, b, c):
    n = 1 << log_n
    hm = np.zeros((n, 8), np.uint32)
    hs = np.zeros((n, 8), np.uint32)
    with g3h.Context(log_n) as ctx:
        ctx.compute_h_abc(a, b, c, hm, hs)
    return hm, hs


@pytest.mark.parametrize("sizes", [(12, 12), (16, 14)])
def test_static_entry_matches_compute_h_abc(sizes):
    import torch

    assert torch.cuda.is_available()
    build.build()
    for call, log_n in enumerate(sizes):
        n = 1 << log_n
        rng = synth.SplitMix64(0x5A7 + 31 * call + log_n)
        a, b, c = (synth.uniform_fr(rng, n) for _ in range(3))
        want_m, want_s = _reference(log_n, a, b, c)
        hm = torch.full((n, 8), -1, dtype=torch.int32, device="cuda")
        hs = torch.full((n, 8), -1, dtype=torch.int32, device="cuda")
        assert _call_static(log_n, _dev(a), _dev(b), _dev(c), hm, hs) == g3h.G3H_OK
        torch.cuda.synchronize()
        assert np.array_equal(hm.cpu().numpy().view(np.uint32), want_m), (call, log_n)
        assert np.array_equal(hs.cpu().numpy().view(np.uint32), want_s), (call, log_n)


def test_static_entry_small_domain_and_limits():
    import torch

    build.build()
    log_n = 3
    n = 1 << log_n
    rng = synth.SplitMix64(0x5A8)
    a, b, c = (synth.uniform_fr(rng, n) for _ in range(3))
    want_m, want_s = _reference(log_n, a, b, c)
    hm = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
    hs = torch.zeros((n, 8), dtype=torch.int32, device="cuda")
    assert _call_static(log_n, _dev(a), _dev(b), _dev(c), hm, hs) == g3h.G3H_OK
    torch.cuda.synchronize()
    assert np.array_equal(hm.cpu().numpy().view(np.uint32), want_m)
    assert np.array_equal(hs.cpu().numpy().view(np.uint32), want_s)
    # beyond the fixed array: refused, nothing launched
    big = torch.zeros((8, 8), dtype=torch.int32, device="cuda")
    assert _call_static(17, big, big, big, big, big) == g3h.G3H_E_RANGE
    L = g3h.lib()
    assert L.g3h_compute_h_abc_static(4, None, None, None, None, None, None) == g3h.G3H_E_INVAL
