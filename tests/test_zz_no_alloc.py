"""moe_route_noalloc: routing for callers that cannot allocate device memory at
call time (e.g. a serving loop whose own allocator already holds all free
device memory, or one whose rules forbid allocator calls after start-up).

Its logits scratch is a fixed array inside the library instead of a
stream-ordered allocation.  This test calls it through the C ABI twice in a
row, on different inputs, and checks each result against moe_route's: the
expert indices must be identical and the weights within the tolerance the
routing tests use.  The file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def capi():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    from fp4_expert_grouped_gb300 import capi as c
    return c


def _inputs(seed, T, d, E, with_bias):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.normal(0, 1, (T, d)).astype(np.float32)).to(torch.bfloat16).cuda()
    gw = torch.from_numpy((rng.normal(0, 1, (d, E)) / np.sqrt(d)).astype(np.float32)).cuda()
    b = torch.from_numpy(rng.normal(0, 1, E).astype(np.float32)).cuda() if with_bias else None
    return x, gw, b


def test_route_noalloc_matches_route_on_two_calls(capi):
    cases = [(1, 257, 4096, 256, 8, False), (2, 96, 1024, 64, 6, True)]
    for seed, T, d, E, k, bias in cases:
        x, gw, b = _inputs(seed, T, d, E, bias)
        ref_i = torch.empty((T, k), dtype=torch.int32, device="cuda")
        ref_w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        capi.moe_route(x, gw, b, ref_i, ref_w)
        got_i = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        got_w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
        capi.moe_route_noalloc(x, gw, b, got_i, got_w)
        assert capi.moe_get_device_status() == 0
        # both run the same kernels on the same logits: identical bits
        assert torch.equal(got_i, ref_i)
        assert torch.equal(got_w.view(torch.int32), ref_w.view(torch.int32))


def test_route_noalloc_second_call_takes_no_device_memory(capi):
    """After a first call (which, under lazy loading, is when the driver
    reserves the fixed array), a call leaves the device's free memory as it
    was: no allocation, in the library or the driver."""
    T, d, E, k = 257, 4096, 256, 8
    x, gw, b = _inputs(3, T, d, E, True)
    ti = torch.empty((T, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    capi.moe_route_noalloc(x, gw, b, ti, tw)
    torch.cuda.synchronize()
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    capi.moe_route_noalloc(x, gw, b, ti, tw)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert capi.moe_get_device_status() == 0
    assert free_after == free_before


def test_route_noalloc_rejects_shapes_beyond_its_scratch(capi):
    T, d, E, k = 4097, 128, 256, 8          # T * E = 1048832 > 1048576
    x = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    gw = torch.zeros((d, E), dtype=torch.float32, device="cuda")
    ti = torch.empty((T, k), dtype=torch.int32, device="cuda")
    tw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(capi.MoeError) as ei:
        capi.moe_route_noalloc(x, gw, None, ti, tw)
    assert ei.value.code == 4                # MOE_ERR_WORKSPACE
