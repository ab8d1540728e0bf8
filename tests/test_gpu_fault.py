"""Failure detection without a GPU fault: GEMM2's bounded wait for GEMM1's
per-tile completion count is made to run out (a count that is never
published, before any copy is issued).  The call must come back, the status
word must say MOE_ERR_TIMEOUT, and the next call must run normally."""
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"
MOE_FLAG_TEST_STALL_GEMM2 = 0x1
MOE_ERR_TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("T,d,inter,E,k", [(32, 256, 128, 8, 2), (256, 512, 256, 8, 2)])
def test_stalled_wait_reports_timeout_and_context_survives(T, d, inter, E, k):
    from fp4_expert_grouped_gb300 import capi, layer
    g = torch.Generator(device=DEV).manual_seed(T)
    w13 = torch.randn((E, 2 * inter, d), generator=g, device=DEV) / d ** 0.5
    w2 = torch.randn((E, d, inter), generator=g, device=DEV) / inter ** 0.5
    pk = layer.pack_experts(w13, w2)
    gw = torch.randn((d, E), generator=g, device=DEV) / d ** 0.5
    x = torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16)
    assert capi.moe_get_device_status() == 0
    want = layer.forward(x, gw, pk, k)
    assert capi.moe_get_device_status() == 0

    out = torch.empty_like(x)
    capi.moe_forward_ex(x, gw, pk.w13_fp4, pk.w13_scale, pk.w2_fp4, pk.w2_scale, out, k,
                        flags=MOE_FLAG_TEST_STALL_GEMM2)
    assert capi.moe_get_device_status() == MOE_ERR_TIMEOUT
    assert capi.moe_get_device_status() == 0                 # read and cleared

    again = layer.forward(x, gw, pk, k)
    assert capi.moe_get_device_status() == 0
    assert torch.equal(again, want)
