"""The tensor-core gate with certified routing, through the C ABI.

From MOE_GATE_TC_MIN_TOKENS tokens on (E a multiple of 64) the library
approximates the logits on the tensor cores, bounds each approximation's
distance to the fixed-order fp32 logit, and computes the fixed-order logit of
the candidate experts only.  Its routing must be bit-identical to the
oracle's (the fixed-order definition), on inputs chosen to stress the
certification: exact ties from duplicated gate columns, all logits equal
(every expert a candidate), rows of zeros, rows scaled far up or down (norms
that overflow, products near the underflow range), and a bias.  Every
approximation must lie within the stated bound; the largest ratio of error to
the bound's main term is printed (it is the measured margin of the
tensor-core accuracy assumption).
"""
import numpy as np
import pytest
import torch

import oracle
from fp4_expert_grouped_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def capi():
    from fp4_expert_grouped_gb300 import capi as c
    return c


def make_gate_case(T, d, E, case, seed):
    rng = np.random.default_rng(seed)
    xf = rng.normal(0, 1, (T, d)).astype(np.float32)
    gw = (rng.normal(0, 1, (d, E)) / np.sqrt(d)).astype(np.float32)
    bias = None
    if case == "ties":
        gw[:, E - 1] = gw[:, 0]
        gw[:, 5] = gw[:, 4]
        gw[:, 17] = gw[:, 16]
    elif case == "all-equal":
        gw[:, :] = gw[:, :1]
    elif case == "zero-rows":
        xf[::7] = 0.0
    elif case == "scaled-rows":
        xf[1::5] *= np.float32(1e18)        # sum of squares overflows fp32: no usable bound
        xf[2::5] *= np.float32(1e-19)       # products near the bottom of the normal range
        xf[3::5] *= np.float32(1e-3)
    elif case == "bias":
        bias = rng.normal(0, 1, E).astype(np.float32)
    elif case == "zipf":
        bias = inputs.zipf_bias(E).numpy()
    x = torch.from_numpy(xf).to(torch.bfloat16)
    return x, gw, bias


CASES = [
    (1024, 256, 64, 8, "plain"),
    (1024, 128, 64, 1, "plain"),
    (1500, 1024, 128, 6, "ties"),
    (1100, 640, 192, 4, "bias"),
    (3000, 7168, 256, 8, "bias"),
    (2048, 512, 256, 8, "zero-rows"),
    (1300, 384, 64, 8, "scaled-rows"),
    (1024, 512, 256, 8, "all-equal"),
    (4096, 4096, 256, 8, "zipf"),
]


@pytest.mark.parametrize("T,d,E,k,case", CASES)
def test_route_tc_gate_bitexact(T, d, E, k, case):
    assert T >= capi().MOE_GATE_TC_MIN_TOKENS and E % 64 == 0
    x, gw, bias = make_gate_case(T, d, E, case, seed=T + E + d)
    ti = torch.empty((T, k), dtype=torch.int32, device=DEV)
    tw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    capi().moe_route(x.to(DEV), torch.from_numpy(gw).to(DEV),
                     None if bias is None else torch.from_numpy(bias).to(DEV), ti, tw)
    assert capi().moe_get_device_status() == 0
    ridx, rw = oracle.route(inputs.bf16_bits(x), gw, k, bias)
    assert np.array_equal(ti.cpu().numpy(), ridx)
    assert np.allclose(tw.cpu().numpy(), rw, rtol=2e-7, atol=0)


def test_route_tc_gate_matches_the_cuda_core_gate_across_the_threshold():
    """The same tokens routed in a batch below the threshold (CUDA-core
    fixed-order logits) and in one above it (tensor-core gate): identical
    indices and weights, bit for bit."""
    T, d, E, k = 1200, 1024, 256, 8
    x, gw, bias = make_gate_case(T, d, E, "bias", seed=5)
    xd, gd, bd = x.to(DEV), torch.from_numpy(gw).to(DEV), torch.from_numpy(bias).to(DEV)
    big_i = torch.empty((T, k), dtype=torch.int32, device=DEV)
    big_w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    capi().moe_route(xd, gd, bd, big_i, big_w)
    n = 1000
    assert n < capi().MOE_GATE_TC_MIN_TOKENS
    small_i = torch.empty((n, k), dtype=torch.int32, device=DEV)
    small_w = torch.empty((n, k), dtype=torch.float32, device=DEV)
    capi().moe_route(xd[T - n:].contiguous(), gd, bd, small_i, small_w)
    assert torch.equal(small_i, big_i[T - n:])
    assert torch.equal(small_w.view(torch.int32), big_w[T - n:].view(torch.int32))


@pytest.mark.parametrize("T,d,inter,E,k,case", [
    (1100, 256, 128, 64, 6, "bias"),
    (1024, 512, 256, 128, 8, "ties"),
    (2000, 768, 128, 192, 4, "zero-rows"),
])
def test_forward_tc_gate_workspace_and_layer(T, d, inter, E, k, case):
    """The layer through the tensor-core gate: the logits region within the
    stated bound of the oracle's fixed-order logits, the selected experts'
    logits bit for bit, routing bit-exact, the layer within tolerance."""
    from test_gpu_parity import check_gate_workspace, check_layer_tolerance, small_case
    from fp4_expert_grouped_gb300 import layer
    w, _, _, _, w13, w2 = small_case(T, d, inter, E, k, seed=T + d)
    x, gw, bias = make_gate_case(T, d, E, case, seed=T)
    pk = layer.pack_experts(w13.to(DEV), w2.to(DEV))
    ws = layer.workspace(T, d, inter, E, k, DEV)
    xd, gd = x.to(DEV), torch.from_numpy(gw).to(DEV)
    bd = None if bias is None else torch.from_numpy(bias).to(DEV)
    out, ti, tw, pp = layer.forward(xd, gd, pk, k, gate_bias=bd, ws=ws, routing=True)
    assert capi().moe_get_device_status() == 0
    xb = inputs.bf16_bits(x)
    z = oracle.gate_logits(xb, gw, bias)
    oi, ow = oracle.topk(z, k)
    assert np.array_equal(ti.cpu().numpy(), oi)
    assert np.allclose(tw.cpu().numpy(), ow, rtol=2e-7, atol=0)
    ratio = check_gate_workspace(ws, w, xd, gd, z, oi, case)
    print("largest |a - z| / (c(d) ||x|| ||w||): %.3g" % ratio)
    f13, s13 = oracle.pack_fp4(w13.numpy())
    f2, s2 = oracle.pack_fp4(w2.numpy())
    ref, _, _ = oracle.moe_forward(xb, gw, f13, s13, f2, s2, k, bias)
    check_layer_tolerance(inputs.bf16_bits(out), ref)


@pytest.mark.parametrize("T,d,inter,E,k,case", [
    (1100, 256, 128, 64, 6, "bias"),
    (2000, 768, 128, 192, 4, "zero-rows"),
])
def test_forward_with_prepared_gate_is_the_same(T, d, inter, E, k, case):
    """moe_forward_opts.gate_prep (gate_w's split and norms prepared once by
    moe_prepare_gate): the same output and routing bits as computing them in
    the call, and the prepared parts equal the ones a call leaves in its
    workspace."""
    from test_gpu_parity import small_case
    from fp4_expert_grouped_gb300 import layer
    c = capi()
    _, _, _, _, w13, w2 = small_case(T, d, inter, E, k, seed=T + d)
    x, gw, bias = make_gate_case(T, d, E, case, seed=T)
    pk = layer.pack_experts(w13.to(DEV), w2.to(DEV))
    xd, gd = x.to(DEV), torch.from_numpy(gw).to(DEV)
    bd = None if bias is None else torch.from_numpy(bias).to(DEV)
    ws = layer.workspace(T, d, inter, E, k, DEV)
    out, ti, tw, pp = layer.forward(xd, gd, pk, k, gate_bias=bd, ws=ws, routing=True)
    prep = layer.prepare_gate(gd)
    ws2 = layer.workspace(T, d, inter, E, k, DEV)
    out2, ti2, tw2, pp2 = layer.forward(xd, gd, pk, k, gate_bias=bd, ws=ws2, routing=True, gate_prep=prep)
    assert c.moe_get_device_status() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(ti, ti2) and torch.equal(tw.view(torch.int32), tw2.view(torch.int32)) and torch.equal(pp, pp2)
    # the prepared parts are the bits a call computes into its workspace
    _, off, _ = c.moe_workspace_layout(T, d, inter, E, k)
    for name, nbytes in (("GATE_WT", E * d * 4), ("GATE_WHI", E * d * 2), ("GATE_WLO", E * d * 2), ("GATE_WNORM", E * 4)):
        o = off[getattr(c, "MOE_WS_" + name)]
        start = {"GATE_WT": 0, "GATE_WHI": 1, "GATE_WLO": 2, "GATE_WNORM": 3}[name]
        sizes = [E * d * 4, E * d * 2, E * d * 2, E * 4]
        po = sum((s + 255) // 256 * 256 for s in sizes[:start])
        assert torch.equal(ws[o:o + nbytes], prep[po:po + nbytes]), name
