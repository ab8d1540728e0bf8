"""The CUDA-graph serving step (layer.GraphedForward) against eager calls:
the same kernels, so the same bits, and every replay reads the host buffer's
current tokens."""
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("T,d,inter,E,k,bias", [(64, 512, 256, 16, 4, False), (40, 768, 384, 32, 6, True)])
def test_graphed_step_matches_eager(T, d, inter, E, k, bias):
    from fp4_expert_grouped_gb300 import capi, layer
    g = torch.Generator(device=DEV).manual_seed(T + E)
    w13 = torch.randn((E, 2 * inter, d), generator=g, device=DEV) / d ** 0.5
    w2 = torch.randn((E, d, inter), generator=g, device=DEV) / inter ** 0.5
    pk = layer.pack_experts(w13, w2)
    gw = torch.randn((d, E), generator=g, device=DEV) / d ** 0.5
    gb = torch.randn((E,), generator=g, device=DEV) if bias else None
    xs = [torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16) for _ in range(3)]

    x_host = torch.empty((T, d), dtype=torch.bfloat16).pin_memory()
    x_host.copy_(xs[0].cpu())
    step = layer.GraphedForward(x_host, gw, pk, k, gate_bias=gb)
    for x in xs:
        x_host.copy_(x.cpu())
        step.replay()
        torch.cuda.synchronize()
        want = layer.forward(x, gw, pk, k, gate_bias=gb)
        torch.cuda.synchronize()
        assert torch.equal(step.out_host, want.cpu())
    assert capi.moe_get_device_status() == 0


def test_graphed_step_needs_pinned_buffers():
    from fp4_expert_grouped_gb300 import layer
    pk = layer.empty_packed(8, 256, 128, DEV)
    gw = torch.zeros((256, 8), device=DEV)
    with pytest.raises(ValueError):
        layer.GraphedForward(torch.zeros((4, 256), dtype=torch.bfloat16), gw, pk, 2)


@pytest.mark.parametrize("T,d,inter,E,k,depth", [(64, 512, 256, 16, 4, 2), (1100, 512, 256, 64, 4, 2),
                                                 (40, 768, 384, 32, 6, 1)])
def test_pipelined_steps_match_eager(T, d, inter, E, k, depth):
    """Five steps through layer.PipelinedForward (copies on two copy streams
    overlapping the neighbouring steps' kernels, device slots reused) give the
    eager forward's bits for each step's own tokens."""
    from fp4_expert_grouped_gb300 import capi, layer
    g = torch.Generator(device=DEV).manual_seed(T + d)
    w13 = torch.randn((E, 2 * inter, d), generator=g, device=DEV) / d ** 0.5
    w2 = torch.randn((E, d, inter), generator=g, device=DEV) / inter ** 0.5
    pk = layer.pack_experts(w13, w2)
    gw = torch.randn((d, E), generator=g, device=DEV) / d ** 0.5
    xs = [torch.randn((T, d), generator=g, device=DEV).to(torch.bfloat16) for _ in range(5)]
    x_hosts = [x.cpu().pin_memory() for x in xs]
    out_hosts = [torch.empty((T, d), dtype=torch.bfloat16).pin_memory() for _ in xs]
    pipe = layer.PipelinedForward(T, d, gw, pk, k, depth=depth)
    done = [pipe.step(xh, oh) for xh, oh in zip(x_hosts, out_hosts)]
    pipe.join()
    for ev in done:
        ev.synchronize()
    torch.cuda.synchronize()
    for x, oh in zip(xs, out_hosts):
        want = layer.forward(x, gw, pk, k)
        torch.cuda.synchronize()
        assert torch.equal(oh, want.cpu())
    assert capi.moe_get_device_status() == 0
