"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (for example a serving runtime that reserves all GPU
memory at start-up and forbids cudaMalloc afterwards, or a plugin hook that
must not allocate).  It keeps its scratch in a fixed device array inside the
library.  These tests call it through the C ABI and compare it, bit for bit,
with moe_dispatch run on a caller workspace, on two calls in a row (the
second smaller than the first, so stale scratch from the first call would
show).  The file is named to be collected last."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _entry(L):
    fn = L.moe_dispatch_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int] + [ctypes.c_void_p] * 5
    fn.restype = ctypes.c_int
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_dispatch_noalloc_matches_workspace_dispatch_two_calls():
    import mixture_experts_routed_top_gb300 as moe
    L = moe.lib()
    fn = _entry(L)
    stream = torch.cuda.current_stream()
    for T, E, k, seed in [(4096, 60, 4, 0), (333, 8, 2, 1)]:
        g = torch.Generator().manual_seed(seed)
        idx, _ = moe.route(torch.randn(T, E, generator=g).cuda(), k)
        outs = [torch.full((E,), -7, dtype=torch.int32, device="cuda"),
                torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
                torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
                torch.full((T * k,), -7, dtype=torch.int32, device="cuda")]
        st = fn(_p(idx), T, E, k, *[_p(o) for o in outs], ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, L.moe_last_error()
        torch.cuda.synchronize()
        ref = moe.dispatch(idx, E)
        for got, want in zip(outs, ref):
            assert torch.equal(got, want)


def test_dispatch_noalloc_rejects_out_of_range_sizes_before_any_launch():
    """E and k outside moe_dispatch's limits are rejected up front (every
    size inside them fits the fixed scratch, so the scratch-size guard is
    never what rejects a call)."""
    import mixture_experts_routed_top_gb300 as moe
    L = moe.lib()
    fn = _entry(L)
    nul = ctypes.c_void_p(0)
    n0 = moe.launch_count()
    st = fn(nul, 10_000_000, 4096, 8, nul, nul, nul, nul, nul)
    assert st == 2
    assert b"E must be" in L.moe_last_error()
    st = fn(nul, 100, 8, 9, nul, nul, nul, nul, nul)
    assert st == 2
    assert b"k must be" in L.moe_last_error()
    assert moe.launch_count() == n0
