"""The QAT backward pass's two dgrad GEMMs (moe_backward_h, moe_backward_x)
against the oracle.

dh = W2^T dy on the FP8 weights (moe_fp4_to_fp8t), the SwiGLU backward with
the forward's g and u, [dg; du] quantised to E4M3 per 128 channels -- per
token-expert pair, in the forward's expert order ("DeepSeek-V4揭秘…" section 4;
oracle/qat.py: pair_dgu).  The routing weights are set to 0.75 and 0.25 so
that dy = w * dout is exact in fp32 as in the oracle's float64 (dout is
bf16), which makes the FP8 operand dy the same codes on both sides.  The
unquantised dg, du must match at the layer tolerance (max|err| <= 1e-2
max|ref|, per-pair relative L2 <= 5e-3); the E4M3 codes of [dg; du] are
compared by fraction (a code flips where the GPU's fp32 sums and the oracle's
float64 fall on two sides of a rounding boundary).  dx = sum over a token's
slots of W13^T [dg; du] (oracle/qat.py: qat_backward) must match at the layer
tolerance; the routing and plan the oracle side uses are its own, checked equal
to the GPU's first.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import qat
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


def layer():
    from fp4_expert_grouped_gb300 import layer as l
    return l


def run_backward(T, d, inter, E, k, seed, bias=False):
    w = inputs.Workload("bwd", T, d, inter, E, k, seed)
    x, gw, _ = inputs.make_x_gate(w, "cpu")
    w13, w2 = inputs.make_all_experts(w, "cpu")
    b = torch.from_numpy(np.random.default_rng(seed).normal(0, 1, E).astype(np.float32)) if bias else None
    pk = layer().pack_experts(w13.to(DEV), w2.to(DEV))
    ws = layer().workspace(T, d, inter, E, k, DEV)
    gu = torch.empty((T * k, 2 * inter), dtype=torch.float32, device=DEV)
    _, ti, tw, pp = layer().forward(x.to(DEV), gw.to(DEV), pk, k, gate_bias=None if b is None else b.to(DEV),
                                    ws=ws, routing=True, gu_out=gu)
    c = capi()
    assert c.moe_get_device_status() == 0
    # routing weights with two significant bits: dy = w * dout exact in fp32
    wts = torch.tensor([0.75, 0.25, 0.5, 0.125, 0.375, 0.625, 0.875, 0.0625][:k], dtype=torch.float32)
    _, off, _ = c.moe_workspace_layout(T, d, inter, E, k)
    ws[off[c.MOE_WS_TOPK_W]:off[c.MOE_WS_TOPK_W] + 4 * T * k].view(torch.float32).copy_(wts.repeat(T).to(DEV))
    w8, s8 = torch.empty((E, inter, d), dtype=torch.uint8, device=DEV), \
        torch.empty((E, inter // 128, d // 128), dtype=torch.uint8, device=DEV)
    c.moe_fp4_to_fp8t(pk.w2_fp4, pk.w2_scale, w8, s8)
    dout = torch.from_numpy(np.random.default_rng(seed + 1).normal(0, 1, (T, d)).astype(np.float32)).to(torch.bfloat16)
    dgu = torch.empty((T * k, 2 * inter), dtype=torch.uint8, device=DEV)
    dgs = torch.empty((T * k, 2 * inter // 128), dtype=torch.uint8, device=DEV)
    dgf = torch.empty((T * k, 2 * inter), dtype=torch.float32, device=DEV)
    bws = torch.empty(c.moe_backward_h_workspace_size(T, d, inter, E, k), dtype=torch.uint8, device=DEV)
    c.moe_backward_h(dout.to(DEV), w8, s8, gu, ws, dgu, dgs, k, dgu_f32=dgf, workspace=bws)
    assert c.moe_get_device_status() == 0
    again = torch.empty_like(dgu)
    again_s = torch.empty_like(dgs)
    c.moe_backward_h(dout.to(DEV), w8, s8, gu, ws, again, again_s, k)
    assert torch.equal(again, dgu) and torch.equal(again_s, dgs)          # deterministic
    # dx through W13^T
    w8x = torch.empty((E, d, 2 * inter), dtype=torch.uint8, device=DEV)
    s8x = torch.empty((E, d // 128, 2 * inter // 128), dtype=torch.uint8, device=DEV)
    c.moe_fp4_to_fp8t(pk.w13_fp4, pk.w13_scale, w8x, s8x)
    dx = torch.empty((T, d), dtype=torch.bfloat16, device=DEV)
    c.moe_backward_x(dgu, dgs, w8x, s8x, ws, dx, k)
    dx2 = torch.empty_like(dx)
    c.moe_backward_x(dgu, dgs, w8x, s8x, ws, dx2, k)
    assert torch.equal(dx, dx2)                                          # deterministic
    dw = torch.empty((T, k), dtype=torch.float32, device=DEV)
    c.moe_backward_dw(dout.to(DEV), ws, dw, inter, E)
    # the master weights' gradients
    dW13 = torch.full((E, 2 * inter, d), float("nan"), dtype=torch.float32, device=DEV)
    dW2 = torch.full((E, d, inter), float("nan"), dtype=torch.float32, device=DEV)
    c.moe_backward_w(ws, bws, dgu, dgs, dW13, dW2, k)
    dW2b = torch.empty_like(dW2)
    dW13b = torch.empty_like(dW13)
    c.moe_backward_w(ws, bws, dgu, dgs, dW13b, dW2b, k)
    assert torch.equal(dW2, dW2b) and torch.equal(dW13, dW13b)          # deterministic
    assert c.moe_get_device_status() == 0
    return dict(x=x, gw=gw, b=b, w13=w13, w2=w2, ti=ti.cpu().numpy(), pp=pp.cpu().numpy(), wts=wts.numpy(),
                dout=dout, dgu=dgu.cpu().numpy(), dgs=dgs.cpu().numpy(), dgf=dgf.cpu().numpy().astype(np.float64),
                dx=inputs.bf16_bits(dx.cpu()), dw=dw.cpu().numpy().astype(np.float64),
                dW13=dW13.cpu().numpy().astype(np.float64), dW2=dW2.cpu().numpy().astype(np.float64))


def oracle_routing(r, E, k):
    """The oracle's own routing and dispatch plan of the case, checked equal to the GPU's."""
    xb = inputs.bf16_bits(r["x"])
    bias = None if r["b"] is None else r["b"].numpy()
    ti, _ = oracle.route(xb, r["gw"].numpy(), k, bias)
    _, _, pp = oracle.dispatch_plan(ti, E)
    assert np.array_equal(ti, r["ti"]) and np.array_equal(pp, r["pp"])
    return ti, pp


def check_against_oracle(r, T, d, inter, E, k, pairs=None):
    xb = inputs.bf16_bits(r["x"])
    xq, xs = oracle.quant_act(xb)
    f13, s13 = oracle.pack_fp4(r["w13"].numpy())
    f2, s2 = oracle.pack_fp4(r["w2"].numpy())
    W2 = qat.fp8_weights(f2, s2)
    do = (inputs.bf16_bits(r["dout"]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    E4M3 = np.array([oracle.e4m3_decode(c) for c in range(256)])
    ti, pp = oracle_routing(r, E, k)
    pairs = range(T * k) if pairs is None else pairs
    same_codes = same_scales = n_codes = n_scales = 0
    for p in pairs:
        t, j = divmod(p, k)
        e = int(ti[t, j])
        pos = int(pp[p])
        g, u = qat.forward_gu(xq[t], xs[t], e, f13, s13)
        dy = float(r["wts"][j]) * do[t]
        dyq, dg, du, dgu = qat.pair_dgu(g, u, dy, W2[e], quantize_grads=True)
        ref = np.concatenate([dg, du])
        got = r["dgf"][pos]
        err = np.abs(got - ref)
        assert err.max() <= 1e-2 * np.abs(ref).max() + 1e-30, (p, err.max(), np.abs(ref).max())
        assert np.linalg.norm(got - ref) <= 5e-3 * np.linalg.norm(ref) + 1e-30, (p, np.linalg.norm(got - ref))
        # the E4M3 output: dequantised codes against the oracle's quantised [dg; du]
        codes, scales = r["dgu"][pos], r["dgs"][pos].astype(np.int64) - 127
        deq = E4M3[codes] * np.ldexp(1.0, np.repeat(scales, 128))
        same_codes += int(np.count_nonzero(deq == dgu))
        n_codes += 2 * inter
        oscale = np.array([oracle.e4m3_scale_exp(float(np.abs(ref[g0:g0 + 128]).max()))
                           for g0 in range(0, 2 * inter, 128)])
        same_scales += int(np.count_nonzero(scales == oscale))
        n_scales += 2 * inter // 128
    # a code flips only where the two sides' dg, du straddle a rounding boundary:
    # about 1e-6 relative apart, against E4M3's 2^-4 to 2^-3 steps
    assert same_codes >= n_codes - max(2, n_codes // 500), (same_codes, n_codes)
    assert same_scales >= n_scales - max(1, n_scales // 200), (same_scales, n_scales)


def check_dx_against_oracle(r, T, d, inter, E, k):
    """dx of every token, dw of every pair and the master weights' gradients dW2,
    dW13 of every expert against the oracle's backward step (its own routing,
    the test's routing weights, quantised gradients) at the layer tolerance."""
    xb = inputs.bf16_bits(r["x"])
    f13, s13 = oracle.pack_fp4(r["w13"].numpy())
    f2, s2 = oracle.pack_fp4(r["w2"].numpy())
    ti, _ = oracle_routing(r, E, k)
    tw = np.tile(r["wts"], (T, 1)).astype(np.float32)
    ref, ref_dw, ref_dW13, ref_dW2 = qat.qat_backward(xb, ti, tw, f13, s13, f2, s2, inputs.bf16_bits(r["dout"]),
                                                      quantize_grads=True)
    # the master weights' gradients: exact zeros for experts without pairs; the
    # layer tolerance over each whole tensor; and per expert with at least 8
    # pairs.  (An expert with one or two pairs shows a single [dg; du] code that
    # the GPU's fp32 and the oracle's float64 round to neighbouring E4M3 values,
    # one step, as a whole row of its gradient: the per-pair comparison above
    # bounds how many such codes there are.)
    n_e = np.bincount(ti.reshape(-1), minlength=E)
    for name, got_w, ref_w in (("dW2", r["dW2"], ref_dW2), ("dW13", r["dW13"], ref_dW13)):
        assert np.all(np.isfinite(got_w)), name
        for e in range(E):
            if n_e[e] == 0:
                assert not np.any(got_w[e]) and not np.any(ref_w[e]), (name, e)
        assert np.abs(got_w - ref_w).max() <= 1e-2 * np.abs(ref_w).max(), (name, np.abs(got_w - ref_w).max())
        assert np.linalg.norm(got_w - ref_w) <= 5e-3 * np.linalg.norm(ref_w), name
        for e in np.nonzero(n_e >= 8)[0]:
            g_e, r_e = got_w[e], ref_w[e]
            assert np.abs(g_e - r_e).max() <= 1e-2 * np.abs(r_e).max(), (name, e, np.abs(g_e - r_e).max())
            assert np.linalg.norm(g_e - r_e) <= 5e-3 * np.linalg.norm(r_e), (name, e)
    # dw = dout . y per pair (y: each side's own bf16 expert output)
    dwe = np.abs(r["dw"] - ref_dw)
    assert dwe.max() <= 1e-2 * np.abs(ref_dw).max(), (dwe.max(), np.abs(ref_dw).max())
    assert np.linalg.norm(r["dw"] - ref_dw) <= 5e-3 * np.linalg.norm(ref_dw)
    got = (r["dx"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = np.abs(got - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max(), (err.max(), np.abs(ref).max())
    rel = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
    assert rel.max() <= 5e-3, (rel.max(), int(rel.argmax()))


@pytest.mark.parametrize("T,d,inter,E,k,bias", [
    (30, 256, 256, 8, 2, False),           # 16-row tiles (P <= 8 E)
    (60, 512, 256, 8, 2, True),            # 32-row tiles
    (150, 256, 256, 8, 2, False),          # 64-row tiles
    (700, 256, 512, 8, 2, True),           # 128-row tiles, two 256-channel blocks of dh
    (64, 256, 256, 4, 4, False),           # k == E
    (10, 256, 512, 32, 2, False),          # most experts without pairs: zero weight gradients
])
def test_backward_matches_oracle(T, d, inter, E, k, bias):
    r = run_backward(T, d, inter, E, k, seed=T + d, bias=bias)
    check_against_oracle(r, T, d, inter, E, k)
    check_dx_against_oracle(r, T, d, inter, E, k)
