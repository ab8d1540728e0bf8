"""Pins of the CPU oracle against facts fixed outside it.

Each test checks the oracle (oracle/moe_oracle.c) against something other than
itself: the format tables of the cited MX/FP8 formats, an independent library
conversion (PyTorch's float8/bfloat16 casts), brute-force search, closed-form
error bounds, invariants, or a float64 numpy brute force of the whole layer on
tiny shapes.  A plausible mistake in the oracle (a dropped term, a swapped
gate/up half, a wrong nibble order or index, a wrong rounding tie) fails one of
them.  None of these tests needs a GPU.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from fp4_expert_grouped_gb300 import inputs

E2M1 = np.array([float(v) for _, v in read_golden("e2m1_values.txt")])
E2M1_SIGNBIT = np.array([math.copysign(1.0, float(v)) < 0 for _, v in read_golden("e2m1_values.txt")])


# --------------------------------------------------------------------------
# helpers: an independent numpy/torch statement of the formats
# --------------------------------------------------------------------------

def t_e4m3_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def t_e4m3_encode(vals):
    """PyTorch's round-to-nearest-even float32 -> E4M3 cast (inputs within +-448)."""
    v = torch.from_numpy(np.asarray(vals, np.float32))
    return v.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def brute_e2m1_encode(v):
    """Nearest E2M1 magnitude, ties to the even code, saturating to 6; sign kept."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    mags = E2M1[:8]
    dist = np.abs(a[..., None] - mags)
    best = np.argmin(dist, axis=-1)
    # ties: argmin returns the lower code; switch to the upper code if that one is even
    dmin = np.take_along_axis(dist, best[..., None], -1)[..., 0]
    up = np.minimum(best + 1, 7)
    dup = np.take_along_axis(dist, up[..., None], -1)[..., 0]
    tie = (dup == dmin) & (up != best)
    best = np.where(tie & (up % 2 == 0), up, best)
    best = np.where(a >= 6.0, 7, best)
    return (best | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def brute_scale_exp_e4m3(amax):
    """Smallest integer e in [-127, 127] with amax <= 448 * 2^e (0 for amax == 0)."""
    if amax == 0:
        return 0
    for e in range(-127, 128):
        if amax <= 448.0 * 2.0 ** e:
            return e
    return 127


def brute_mx_exp(amax):
    """Largest integer X with 2^(X+2) <= amax, clamped to [-127, 127]; -127 for 0."""
    if amax == 0:
        return -127
    X = -200
    while 2.0 ** (X + 3) <= amax:
        X += 1
    return max(-127, min(127, X))


def np_pack_fp4(w):
    E, N, K = w.shape
    blk = w.astype(np.float64).reshape(E, N, K // 32, 32)
    amax = np.abs(blk).max(-1)
    X = np.vectorize(brute_mx_exp)(amax)
    codes = brute_e2m1_encode(np.ldexp(blk, -X[..., None])).reshape(E, N, K)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, (X + 127).astype(np.uint8)


def np_dequant_fp4(w_fp4, w_scale):
    lo = w_fp4 & 0xF
    hi = w_fp4 >> 4
    codes = np.stack([lo, hi], -1).reshape(*w_fp4.shape[:-1], w_fp4.shape[-1] * 2)
    X = np.repeat(w_scale.astype(np.int64) - 127, 32, axis=-1)
    return np.ldexp(E2M1[codes], X)


def np_fp8_quant(v):
    """Per-128 power-of-two scaled E4M3 quantisation of float32 rows; returns dequantised float64."""
    v = np.asarray(v, np.float32)
    n = v.shape[-1]
    g = v.reshape(*v.shape[:-1], n // 128, 128)
    amax = np.abs(g.astype(np.float64)).max(-1)
    e = np.vectorize(brute_scale_exp_e4m3)(amax)
    scaled = np.ldexp(g.astype(np.float64), -e[..., None]).astype(np.float32)
    q = t_e4m3_decode(t_e4m3_encode(scaled))
    return np.ldexp(q, e[..., None]).reshape(v.shape), e


def bf16_round(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def bf16_bits_of(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def from_bits(b):
    return np.asarray(b, np.uint16).astype(np.uint32).__lshift__(16).view(np.float32)


def check_tolerance(out_bits, ref_bits):
    """Output tolerance of the layer: max|err| <= 1e-2 max|ref| and per-token
    relative L2 <= 5e-3 (a zero reference row needs a zero output row)."""
    out = from_bits(out_bits).astype(np.float64)
    ref = from_bits(ref_bits).astype(np.float64)
    err = np.abs(out - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max() + 0.0, (err.max(), np.abs(ref).max())
    rn = np.linalg.norm(ref, axis=-1)
    en = np.linalg.norm(out - ref, axis=-1)
    zero = rn == 0
    assert np.all(en[zero] == 0)
    assert np.all(en[~zero] <= 5e-3 * rn[~zero]), (en / np.maximum(rn, 1e-30)).max()


# --------------------------------------------------------------------------
# codecs
# --------------------------------------------------------------------------

def test_e2m1_decode_table():
    for c in range(16):
        v = oracle.e2m1_decode(c)
        assert v == E2M1[c]
        assert math.copysign(1.0, v) < 0 if E2M1_SIGNBIT[c] else True


def test_e2m1_encode_matches_bruteforce():
    # every midpoint, every code value, values just around them, saturation and zeros
    mags = E2M1[:8]
    mids = (mags[:-1] + mags[1:]) / 2
    pts = np.concatenate([mags, mids, np.nextafter(mids, 0), np.nextafter(mids, 10),
                          [6.5, 7.9, 8.0, 100.0, 1e-30, 0.0]])
    rng = np.random.default_rng(0)
    pts = np.concatenate([pts, rng.uniform(0, 7, 20000)])
    vals = np.concatenate([pts, -pts])
    got = np.array([oracle.e2m1_encode(v) for v in vals], np.uint8)
    assert np.array_equal(got, brute_e2m1_encode(vals))
    # the tie cases spelled out (round half to even code)
    for v, c in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]:
        assert oracle.e2m1_encode(v) == c


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = t_e4m3_decode(codes)
    got = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(1) == 2.0 ** -9


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.normal(0, 50, 30000), rng.uniform(-448, 448, 30000),
        np.ldexp(rng.uniform(-1, 1, 20000), rng.integers(-14, 9, 20000)),
    ]).astype(np.float32)
    vals = vals[np.abs(vals) <= 448]
    # all exact codes and all midpoints between neighbours
    pos = t_e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, pos.astype(np.float32), mids, -mids, np.float32([-0.0, 0.0])])
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], np.uint8)
    assert np.array_equal(got, t_e4m3_encode(vals))
    # saturation of finite values beyond the largest code
    for v in (448.0, 460.0, 464.0, 500.0, 1e6):
        assert oracle.e4m3_encode(v) == 0x7E and oracle.e4m3_encode(-v) == 0xFE


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e30, 1000),
                           np.ldexp(rng.uniform(1, 2, 2000), rng.integers(-140, -120, 2000))]).astype(np.float32)
    # exact ties: low 16 bits == 0x8000
    ties = (rng.integers(0, 2 ** 31, 2000, dtype=np.int64).astype(np.uint32) & 0xFFFF0000) | 0x8000
    vals = np.concatenate([vals, ties.view(np.float32)])
    vals = vals[np.isfinite(vals)]
    got = np.array([oracle.f32_to_bf16(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, bf16_bits_of(vals))
    for b in (0x3F80, 0xBF80, 0x7F7F, 0x0001, 0x8000):
        assert bf16_bits_of([oracle.bf16_to_f32(b)])[0] == b


def test_e4m3_scale_exp_bruteforce():
    rng = np.random.default_rng(3)
    cases = [0.0, 448.0, 1.0, 1.75, 2.0 ** -130, 3e38]
    for e in range(-20, 20):
        b = 448.0 * 2.0 ** e
        cases += [b, float(np.nextafter(np.float32(b), np.float32(1e30))), float(np.nextafter(np.float32(b), np.float32(0)))]
    cases += list(np.abs(rng.normal(0, 3, 500)).astype(np.float32))
    for a in cases:
        assert oracle.e4m3_scale_exp(float(a)) == brute_scale_exp_e4m3(float(a)), a


def test_mx_scale_exp_bruteforce():
    rng = np.random.default_rng(4)
    cases = [0.0, 1.0, 4.0, 3.999, 2.0 ** -126, 2.0 ** -140, 1e30]
    for m in range(-30, 30):
        cases += [2.0 ** m, 2.0 ** m * 1.999999, float(np.nextafter(np.float32(2.0 ** m), np.float32(0)))]
    cases += list(np.abs(rng.normal(0, 0.05, 500)).astype(np.float32))
    for a in cases:
        assert oracle.mx_scale_exp(float(a)) == brute_mx_exp(float(a)), a


def test_fp4_to_fp8_lossless_range():
    """FP4 -> FP8 dequantisation is exact ("DeepSeek-V4揭秘…" section 4): every E2M1
    code times 2^D is an E4M3 value exactly iff D in [-8, 6], so a 128x128 FP8
    block can absorb 1x32 FP4 sub-block scales whose max/min ratio is <= 2^14."""
    codes = range(16)
    ok = []
    for D in range(-12, 10):
        exact = True
        for c in codes:
            v = E2M1[c] * 2.0 ** D
            q = oracle.e4m3_decode(oracle.e4m3_encode(v))
            if q != v:
                exact = False
        ok.append((D, exact))
    good = [D for D, ex in ok if ex]
    assert good == list(range(-8, 7))
    assert 2.0 ** (good[-1] - good[0]) == 2.0 ** 14


def test_gate_score_special_values():
    assert oracle.gate_score(0.0) == np.float32(math.sqrt(math.log(2.0)))
    for z in (-30.0, -3.0, -0.5, 0.7, 5.0, 40.0):
        ref = np.float32(math.sqrt(np.logaddexp(0.0, z)))
        assert abs(oracle.gate_score(z) - ref) <= 2 * np.spacing(ref)


# --------------------------------------------------------------------------
# quantisers on arrays
# --------------------------------------------------------------------------

def test_quant_act_matches_independent_quantiser():
    w = inputs.WORKLOADS["tiny"]
    x, _, _ = inputs.make_x_gate(w)
    xb = inputs.bf16_bits(x)
    # sprinkle exact zeros / a zero group / large values
    xb = xb.copy()
    xb[0, :128] = 0
    xb[1, 5] = bf16_bits_of([300.0])[0]
    xq, xs = oracle.quant_act(xb)
    xf = from_bits(xb)
    deq, e = np_fp8_quant(xf)
    assert np.array_equal(xs.astype(np.int64) - 127, e)
    got = np.ldexp(t_e4m3_decode(xq).reshape(xf.shape[0], -1, 128), e[..., None].astype(np.int64)).reshape(xf.shape)
    assert np.array_equal(got, deq)


def test_pack_fp4_matches_bruteforce():
    rng = np.random.default_rng(5)
    E, N, K = 3, 7, 256
    w = (rng.normal(0, 0.02, (E, N, K))).astype(np.float32)
    w[0, 0, :32] = 0.0                                     # all-zero block
    w[0, 1, :32] = np.float32(6.0 * 2.0 ** -7)             # at the top code
    w[0, 1, 0] = np.float32(7.9 * 2.0 ** -7)               # saturating element
    w[1, 2, 32:64] = np.float32(0.25 * 2.0 ** -5)          # exact ties
    w[1, 2, 32] = np.float32(4.0 * 2.0 ** -5)
    w[2, 3, 64:96] = -w[2, 3, 64:96]
    fp4, sc = oracle.pack_fp4(w)
    rf, rs = np_pack_fp4(w)
    assert np.array_equal(sc, rs)
    assert np.array_equal(fp4, rf)
    # nibble order: low nibble = even K index
    deq = np_dequant_fp4(fp4, sc)
    assert np.max(np.abs(deq - w)) <= np.max(np.abs(w)) / 4 + 1e-9


# --------------------------------------------------------------------------
# gate and routing
# --------------------------------------------------------------------------

def test_gate_logits_error_bound():
    rng = np.random.default_rng(6)
    for d, E in [(256, 8), (4096, 16), (7168, 4)]:
        x = bf16_bits_of(rng.normal(0, 1, (3, d)))
        gw = (rng.normal(0, 1, (d, E)) / math.sqrt(d)).astype(np.float32)
        z = oracle.gate_logits(x, gw)
        xf = from_bits(x).astype(np.float64)
        prod = xf[:, :, None] * gw.astype(np.float64)[None]           # exact products
        exact = np.array([[math.fsum(prod[t, :, e]) for e in range(E)] for t in range(3)])
        n = d // 32 + 5
        u = 2.0 ** -24
        gamma = n * u / (1 - n * u)
        bound = gamma * np.abs(prod).sum(1)
        assert np.all(np.abs(z - exact) <= bound)
        bias = rng.normal(0, 1, E).astype(np.float32)
        zb = oracle.gate_logits(x, gw, bias)
        assert np.array_equal(zb, (z + bias).astype(np.float32))


def test_gate_logits_exact_on_integer_products():
    # integer-valued products: every partial sum is exact, so the fixed order
    # must give the exact total whatever the order
    rng = np.random.default_rng(7)
    d, E = 512, 5
    x = bf16_bits_of(rng.integers(-8, 9, (2, d)).astype(np.float32))
    gw = rng.integers(-8, 9, (d, E)).astype(np.float32)
    z = oracle.gate_logits(x, gw)
    assert np.array_equal(z, (from_bits(x).astype(np.int64) @ gw.astype(np.int64)).astype(np.float32))


def _f32_round(q):
    """Nearest float32 to the exact rational q, ties to the even significand
    (IEEE round-to-nearest-even, found by exact comparison -- no double
    rounding through float64)."""
    from fractions import Fraction
    c = np.float32(float(q))
    best = None
    for cand in (np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))):
        dist = abs(Fraction(float(cand)) - q)
        even = (int(np.asarray(cand, np.float32).view(np.uint32)) & 1) == 0
        key = (dist, not even)
        if best is None or key < best[0]:
            best = (key, cand)
    return np.float32(best[1])


def _fmaf(a, b, c):
    """fmaf: a*b + c rounded once to float32 (exact rational arithmetic)."""
    from fractions import Fraction
    return _f32_round(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def _addf(a, b):
    from fractions import Fraction
    return _f32_round(Fraction(float(a)) + Fraction(float(b)))


def _logit_in_order(xr, wc, order):
    """One logit x . w in float32 under a named summation order.
    "strided32-tree": 32 chains over channels l, l+32, ... (fmaf), then the
    tree with offsets 16, 8, 4, 2, 1 -- the order the oracle states;
    the others are plausible misreadings of it."""
    d = len(xr)
    zero = np.float32(0.0)
    if order == "sequential":
        acc = zero
        for i in range(d):
            acc = _fmaf(xr[i], wc[i], acc)
        return acc
    if order in ("strided32-tree", "strided32-linear", "strided32-tree-up", "contiguous32-tree", "strided16-tree"):
        L = 16 if order == "strided16-tree" else 32
        part = []
        for l in range(L):
            acc = zero
            chans = range(l * (d // L), (l + 1) * (d // L)) if order == "contiguous32-tree" else range(l, d, L)
            for i in chans:
                acc = _fmaf(xr[i], wc[i], acc)
            part.append(acc)
        if order == "strided32-linear":
            acc = part[0]
            for l in range(1, L):
                acc = _addf(acc, part[l])
            return acc
        if order == "strided32-tree-up":                 # adjacent pairs first: (p0+p1), (p2+p3), ...
            step = 1
            while step < L:
                for l in range(0, L, 2 * step):
                    part[l] = _addf(part[l], part[l + step])
                step *= 2
            return part[0]
        off = L // 2
        while off >= 1:
            for l in range(off):
                part[l] = _addf(part[l], part[l + off])
            off //= 2
        return part[0]
    raise ValueError(order)


def test_gate_logits_fixed_order_exactly():
    """The oracle's logits equal the stated fixed order evaluated with exactly
    rounded float32 operations (every fused multiply-add and add rounded once,
    by rational arithmetic), bias added last; and each plausible misreading
    of the order (one sequential chain, contiguous chunks, 16 chains, a linear
    or bottom-up sum of the partials) disagrees with the oracle somewhere on
    the same inputs, so this test tells the orders apart."""
    rng = np.random.default_rng(61)
    T, d, E = 3, 256, 4
    x = bf16_bits_of(rng.normal(0, 1, (T, d)))
    gw = (rng.normal(0, 1, (d, E)) / math.sqrt(d)).astype(np.float32)
    bias = rng.normal(0, 1, E).astype(np.float32)
    xf = from_bits(x)
    want = np.empty((T, E), np.float32)
    for t in range(T):
        for e in range(E):
            want[t, e] = _addf(_logit_in_order(xf[t], gw[:, e], "strided32-tree"), bias[e])
    got = oracle.gate_logits(x, gw, bias)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    for order in ("sequential", "contiguous32-tree", "strided16-tree", "strided32-linear", "strided32-tree-up"):
        alt = np.array([[_addf(_logit_in_order(xf[t], gw[:, e], order), bias[e]) for e in range(E)]
                        for t in range(T)], np.float32)
        assert not np.array_equal(alt.view(np.uint32), got.view(np.uint32)), order


def test_gate_logits_hand_built_order_case():
    """A case worked out by hand.  d = 64, one expert, x = 1 on channels 0, 1
    and 33 (0 elsewhere); gate_w = 1 on channel 0 and b = 2^-24 on channels 1
    and 33.  In the fixed order, chain 1 holds channels 1 and 33:
    fmaf(1, b, fmaf(1, b, 0)) = 2b = 2^-23 exactly; chain 0 holds channel 0
    (= 1); the tree adds chain 1 into chain 0 at the last level (offset 1),
    after chain 1 has absorbed only zeros (chains 3, 5, 9, 17), giving
    1 + 2^-23, which is a float32 (one ulp above 1).  A single sequential
    chain gives 1: 1 + b is a tie between 1 and 1 + 2^-23 and rounds to the
    even significand, 1, and so does the second b.  Contiguous chunks of
    two channels put channel 1 beside channel 0 (1 + b -> 1) and channel 33
    alone in chunk 16, which meets chunk 0 first in the tree (1 + b -> 1):
    again 1."""
    d = 64
    x = np.zeros((1, d), np.float32)
    x[0, [0, 1, 33]] = 1.0
    gw = np.zeros((d, 1), np.float32)
    gw[0, 0] = 1.0
    gw[[1, 33], 0] = np.float32(2.0 ** -24)
    z = oracle.gate_logits(bf16_bits_of(x), gw)
    assert z[0, 0] == np.float32(1.0 + 2.0 ** -23)
    assert z[0, 0] != np.float32(1.0)


def test_topk_bruteforce_and_ties():
    rng = np.random.default_rng(8)
    T, E, k = 200, 32, 6
    z = rng.normal(0, 1, (T, E)).astype(np.float32)
    z[:20, :] = np.round(z[:20, :] * 2) / 2                 # many exact ties
    z[20] = 0.0                                             # all equal
    idx, w = oracle.topk(z, k)
    for t in range(T):
        order = np.lexsort((np.arange(E), -z[t].astype(np.float64)))[:k]
        assert list(idx[t]) == list(order)
    assert list(idx[20]) == list(range(k))
    # weights: proportional to sqrt(softplus(z)), sum 1 within k * 2^-24
    s = np.sqrt(np.logaddexp(0.0, np.take_along_axis(z, idx, 1).astype(np.float64)))
    ref = s / s.sum(1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-6, atol=1e-7)
    assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= k * 2.0 ** -24 + 1e-12)
    # k == E selects every expert in logit order
    idx2, _ = oracle.topk(z[:5], E)
    for t in range(5):
        assert sorted(idx2[t]) == list(range(E))


def test_route_duplicated_gate_columns_tie_to_lower_index():
    rng = np.random.default_rng(9)
    d, E = 256, 8
    x = bf16_bits_of(rng.normal(0, 1, (16, d)))
    gw = (rng.normal(0, 1, (d, E)) / 16).astype(np.float32)
    gw[:, 5] = gw[:, 2]
    z = oracle.gate_logits(x, gw)
    assert np.array_equal(z[:, 5], z[:, 2])
    idx, _ = oracle.topk(z, E)
    for t in range(16):
        pos = list(idx[t])
        assert pos.index(2) + 1 == pos.index(5)


# --------------------------------------------------------------------------
# dispatch plan
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (37, 8, 2), (300, 64, 8), (128, 256, 8)])
def test_dispatch_plan_is_stable_sort_and_bijection(T, E, k):
    rng = np.random.default_rng(T * 7 + E)
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    offs, sp, pp = oracle.dispatch_plan(idx, E)
    P = T * k
    assert np.array_equal(sp, np.argsort(idx.reshape(-1), kind="stable").astype(np.int32))
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(np.bincount(idx.reshape(-1), minlength=E))]))
    assert np.array_equal(np.sort(pp), np.arange(P))
    assert np.array_equal(pp[sp], np.arange(P))


# --------------------------------------------------------------------------
# whole layer
# --------------------------------------------------------------------------

def dense_bruteforce(xb, gw, bias, w13, w2, k):
    """float64 numpy restatement of the layer on dequantised tensors, with no
    permutation: out_t = sum over selected e of w_e * FFN_e(x_t)."""
    xf = from_bits(xb).astype(np.float64)
    z = xf @ gw.astype(np.float64) + (0 if bias is None else bias.astype(np.float64))
    T = xf.shape[0]
    inter = w13.shape[1] // 2
    sel = np.argsort(-z, axis=1, kind="stable")[:, :k]
    s = np.sqrt(np.logaddexp(0.0, np.take_along_axis(z, sel, 1)))
    wt = s / s.sum(1, keepdims=True)
    a, _ = np_fp8_quant(from_bits(xb))
    out = np.zeros_like(xf)
    for t in range(T):
        for j in range(k):
            e = sel[t, j]
            g = (w13[e, :inter] @ a[t]).astype(np.float32).astype(np.float64)
            u = (w13[e, inter:] @ a[t]).astype(np.float32).astype(np.float64)
            h = (g / (1 + np.exp(-g)) * u).astype(np.float32)
            hd, _ = np_fp8_quant(h[None])
            y = bf16_round((w2[e] @ hd[0]).astype(np.float32))
            out[t] += wt[t, j] * y
    return bf16_bits_of(out.astype(np.float32)), sel, z


def tiny_packed(w, rng_seed=None):
    x, gw, bias = inputs.make_x_gate(w)
    w13, w2 = inputs.make_all_experts(w)
    w13f, w13s = oracle.pack_fp4(w13.numpy())
    w2f, w2s = oracle.pack_fp4(w2.numpy())
    return (inputs.bf16_bits(x), gw.numpy(), None if bias is None else bias.numpy(),
            w13f, w13s, w2f, w2s)


def test_forward_matches_dense_bruteforce_tiny():
    w = inputs.WORKLOADS["tiny"]
    xb, gw, bias, w13f, w13s, w2f, w2s = tiny_packed(w)
    out, idx, wts = oracle.moe_forward(xb, gw, w13f, w13s, w2f, w2s, w.k, bias)
    ref, sel, z = dense_bruteforce(xb, gw, bias, np_dequant_fp4(w13f, w13s), np_dequant_fp4(w2f, w2s), w.k)
    # the float64 selection must agree (margins on this seed are far above fp32 rounding)
    zs = np.sort(z, 1)[:, ::-1]
    assert np.all(zs[:, w.k - 1] - zs[:, w.k] > 1e-4)
    assert np.array_equal(idx, sel)
    check_tolerance(out, ref)


def test_forward_dense_bruteforce_other_shapes():
    rng = np.random.default_rng(10)
    T, d, inter, E, k = 12, 384, 256, 6, 3
    xb = bf16_bits_of(rng.normal(0, 1, (T, d)))
    gw = (rng.normal(0, 1, (d, E)) / math.sqrt(d)).astype(np.float32)
    bias = rng.normal(0, 0.5, E).astype(np.float32)
    w13 = (rng.normal(0, 1, (E, 2 * inter, d)) / math.sqrt(d)).astype(np.float32)
    w2 = (rng.normal(0, 1, (E, d, inter)) / math.sqrt(inter)).astype(np.float32)
    w13f, w13s = oracle.pack_fp4(w13)
    w2f, w2s = oracle.pack_fp4(w2)
    out, idx, _ = oracle.moe_forward(xb, gw, w13f, w13s, w2f, w2s, k, bias)
    ref, sel, z = dense_bruteforce(xb, gw, bias, np_dequant_fp4(w13f, w13s), np_dequant_fp4(w2f, w2s), k)
    zs = np.sort(z, 1)[:, ::-1]
    assert np.all(zs[:, k - 1] - zs[:, k] > 1e-5)
    assert np.array_equal(idx, sel)
    check_tolerance(out, ref)


def test_identical_experts_reduce_to_one_expert():
    rng = np.random.default_rng(11)
    T, d, inter, E, k = 16, 256, 128, 8, 3
    xb = bf16_bits_of(rng.normal(0, 1, (T, d)))
    gw = (rng.normal(0, 1, (d, E)) / 16).astype(np.float32)
    w13 = np.repeat((rng.normal(0, 1, (1, 2 * inter, d)) / 16).astype(np.float32), E, 0)
    w2 = np.repeat((rng.normal(0, 1, (1, d, inter)) / math.sqrt(inter)).astype(np.float32), E, 0)
    w13f, w13s = oracle.pack_fp4(w13)
    w2f, w2s = oracle.pack_fp4(w2)
    out, _, wts = oracle.moe_forward(xb, gw, w13f, w13s, w2f, w2s, k)
    one, _, w1 = oracle.moe_forward(xb, gw[:, :1], w13f[:1], w13s[:1], w2f[:1], w2s[:1], 1)
    assert np.all(w1 == 1.0)
    a = from_bits(out).astype(np.float64)
    b = from_bits(one).astype(np.float64)
    ulp = np.abs(b) * 2.0 ** -7
    assert np.all(np.abs(a - b) <= ulp + 1e-30)


def test_one_hot_probe_gate_up_order_and_nibbles():
    """x = e_c; W13 nonzero only at gate row n, up row inter+n, column c; W2
    nonzero at row m, column n.  Then h_n = silu(g) u and y_m = h_n * W2[m, n];
    swapping gate and up, or the nibble order of column c, changes y_m."""
    d, inter, E, k = 256, 128, 2, 1
    c, n, m = 37, 5, 200           # odd column: high nibble of its byte
    x = np.zeros((1, d), np.float32)
    x[0, c] = 1.0
    xb = bf16_bits_of(x)
    gw = np.zeros((d, E), np.float32)
    gw[c, 1] = 1.0                 # route to expert 1
    w13 = np.zeros((E, 2 * inter, d), np.float32)
    w2 = np.zeros((E, d, inter), np.float32)
    w13[1, n, c] = -1.5            # gate
    w13[1, inter + n, c] = 4.0     # up
    w13[1, n, c - 1] = 0.5         # even neighbour sharing the byte (x is 0 there)
    w2[1, m, n] = 2.0
    w13f, w13s = oracle.pack_fp4(w13)
    w2f, w2s = oracle.pack_fp4(w2)
    out, idx, wts = oracle.moe_forward(xb, gw, w13f, w13s, w2f, w2s, k)
    assert idx[0, 0] == 1 and wts[0, 0] == 1.0
    g, u = -1.5, 4.0
    h = np.float32(g / (1 + math.exp(-g)) * u)
    hdq, _ = np_fp8_quant(np.array([[h] + [0.0] * (inter - 1)], np.float32))
    expect = bf16_round([hdq[0, 0] * 2.0])[0]
    got = from_bits(out)[0]
    assert got[m] == expect and np.count_nonzero(got) == 1


def test_expert_pair_intermediates():
    """One pair's intermediates: h against a float64 dense restatement (within
    fp32 rounding of g and u), and hq/hs against the brute-force scale rule and
    PyTorch's E4M3 cast applied to the same h."""
    rng = np.random.default_rng(12)
    d, inter, E = 256, 256, 2
    xb = bf16_bits_of(rng.normal(0, 1, (1, d)))
    xq, xs = oracle.quant_act(xb)
    w13 = (rng.normal(0, 1, (E, 2 * inter, d)) / 16).astype(np.float32)
    w2 = (rng.normal(0, 1, (E, d, inter)) / 16).astype(np.float32)
    w13f, w13s = oracle.pack_fp4(w13)
    w2f, w2s = oracle.pack_fp4(w2)
    h, hq, hs, y = oracle.expert_pair(xq[0], xs[0], 1, w13f, w13s, w2f, w2s)
    a = np.ldexp(t_e4m3_decode(xq[0]), np.repeat(xs[0].astype(np.int64) - 127, 128))
    W = np_dequant_fp4(w13f, w13s)[1]
    g = W[:inter] @ a
    u = W[inter:] @ a
    href = g / (1 + np.exp(-g)) * u
    assert np.allclose(h, href, rtol=1e-5, atol=1e-6 * np.abs(href).max())
    hd, e = np_fp8_quant(h[None])
    assert np.array_equal(hs.astype(np.int64) - 127, e[0])
    assert np.array_equal(t_e4m3_encode(np.ldexp(h.astype(np.float64), -np.repeat(e[0], 128)).astype(np.float32)), hq)
    yref = bf16_bits_of((np_dequant_fp4(w2f, w2s)[1] @ hd[0]).astype(np.float32))
    assert np.max(np.abs(from_bits(y) - from_bits(yref))) <= 2.0 ** -7 * np.abs(from_bits(yref)).max()


# --------------------------------------------------------------------------
# FP8 weights for the backward pass (FP4 QAT, "DeepSeek-V4揭秘…" section 4)
# --------------------------------------------------------------------------

def np_block_exponents(w_scale):
    """B = max(largest 1x32 exponent of each 128x128 block - 6, -127), as [E, K/128, N/128]."""
    E, N, KS = w_scale.shape
    X = w_scale.astype(np.int64).reshape(E, N // 128, 128, KS // 4, 4) - 127
    S = X.max(axis=(2, 4))                                   # [E, N/128, K/128]
    return np.maximum(S - 6, -127).transpose(0, 2, 1)


def test_fp8t_is_lossless_on_weights_within_the_scale_ratio():
    """The pages' claim: while each 128x128 block's sub-block scales stay within
    a 2^14 ratio, the FP8 weights are the FP4 weights exactly (here: transposed)."""
    rng = np.random.default_rng(11)
    E, N, K = 3, 256, 384
    w = (rng.normal(0, 1, (E, N, K)) / np.sqrt(K)).astype(np.float32)
    w[1, 128:, :128] = 0.0                                   # an all-zero block
    f, s = oracle.pack_fp4(w)
    w8t, s8t = oracle.fp4_to_fp8t(f, s)
    B = np_block_exponents(s)
    assert np.array_equal(s8t.astype(np.int64) - 127, B)
    X = s.astype(np.int64).reshape(E, N // 128, 128, K // 128, 4) - 127
    spread = X.max(axis=(2, 4)) - np.where(X.min(axis=(2, 4)) < -120, X.max(axis=(2, 4)), X.min(axis=(2, 4)))
    assert spread.max() <= 14
    got = t_e4m3_decode(w8t) * np.ldexp(1.0, np.repeat(np.repeat(B, 128, 1), 128, 2))
    assert np.array_equal(got, np_dequant_fp4(f, s).transpose(0, 2, 1))
    assert np.all(w8t[1, :128, 128:] == 0) and s8t[1, 0, 1] == 0   # zero block: B clamped to -127


def test_fp8t_rounds_sub_blocks_beyond_the_ratio():
    """A block whose sub-scales span more than 2^14: the large sub-block stays
    exact, the small one is rounded to nearest-even E4M3 at the block's scale."""
    rng = np.random.default_rng(12)
    w = np.zeros((1, 128, 128), np.float32)
    w[0, :, :32] = rng.uniform(-300, 300, (128, 32))          # exponents near 6
    w[0, :, 32:64] = rng.uniform(-1, 1, (128, 32)) * 2.0 ** -16   # about 2^22 smaller
    f, s = oracle.pack_fp4(w)
    w8t, s8t = oracle.fp4_to_fp8t(f, s)
    B = int(s8t[0, 0, 0]) - 127
    deq = np_dequant_fp4(f, s)[0]                             # [N, K]
    X = s[0].astype(np.int64) - 127
    assert X[:, 0].max() - X[:, 1].max() > 14
    want = t_e4m3_encode(np.ldexp(deq, -B).astype(np.float32)).T   # exact in fp32: codes times powers of two
    assert np.array_equal(w8t[0], want)
    big = t_e4m3_decode(w8t[0, :32, :]) * 2.0 ** B
    assert np.array_equal(big, deq[:, :32].T)
    assert not np.array_equal(t_e4m3_decode(w8t[0, 32:64, :]) * 2.0 ** B, deq[:, 32:64].T)


# --------------------------------------------------------------------------
# QAT backward step of the expert path (oracle/qat.py) against autograd
# --------------------------------------------------------------------------

class _QuantGrad(torch.autograd.Function):
    """Identity whose backward quantises the incoming gradient to E4M3 per 128
    channels (independent numpy/PyTorch statement of the activation rule)."""

    @staticmethod
    def forward(ctx, v):
        return v.clone()

    @staticmethod
    def backward(ctx, g):
        return torch.from_numpy(np_fp8_quant(g.detach().numpy())[0])


def _ste(v, value):
    """Forward value `value`, gradient of `v` (straight-through)."""
    return v + (torch.as_tensor(value, dtype=torch.float64) - v).detach()


def test_forward_gu_is_the_exact_sum_rounded_to_fp32():
    """oracle.qat.forward_gu (the g, u the backward's SwiGLU uses) equals, for
    every channel, the correctly rounded float32 of the exact dot product of the
    dequantised FP8 token and FP4 weight row (math.fsum of exact products; a
    float32 tie would show as one ulp), and the C oracle's h of the same pair
    is silu(g) * u of those values."""
    from oracle import qat
    rng = np.random.default_rng(31)
    E, inter, d = 3, 128, 256
    w13 = (rng.normal(0, 1, (E, 2 * inter, d)) / math.sqrt(d)).astype(np.float32)
    w2 = (rng.normal(0, 1, (E, d, inter)) / math.sqrt(inter)).astype(np.float32)
    f13, s13 = oracle.pack_fp4(w13)
    f2, s2 = oracle.pack_fp4(w2)
    W13 = np_dequant_fp4(f13, s13)
    xb = bf16_bits_of(rng.normal(0, 1, (2, d)))
    xq, xs = oracle.quant_act(xb)
    for t in range(2):
        xd = t_e4m3_decode(xq[t]) * np.ldexp(1.0, np.repeat(xs[t].astype(np.int64) - 127, 128))
        for e in range(E):
            g, u = qat.forward_gu(xq[t], xs[t], e, f13, s13)
            exact = np.array([math.fsum(xd * W13[e, n]) for n in range(2 * inter)])
            want = exact.astype(np.float32).astype(np.float64)
            got = np.concatenate([g, u])
            ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
            assert np.all(np.abs(got - want) <= ulp)
            h, _, _, _ = oracle.expert_pair(xq[t], xs[t], e, f13, s13, f2, s2)
            assert np.allclose(h, (g / (1.0 + np.exp(-g)) * u).astype(np.float32), rtol=1e-6, atol=0)


@pytest.mark.parametrize("quantize_grads", [False, True])
def test_qat_backward_matches_autograd(quantize_grads):
    """The oracle's backward step equals PyTorch float64 autograd of the same
    forward (straight-through quantisers, fixed routing; with quantize_grads,
    the gradients at y and at [g; u] quantised to E4M3 per 128 channels)."""
    from oracle import qat
    rng = np.random.default_rng(21)
    T, d, inter, E, k = 5, 256, 128, 4, 2
    w13 = (rng.normal(0, 1, (E, 2 * inter, d)) / np.sqrt(d)).astype(np.float32)
    w2 = (rng.normal(0, 1, (E, d, inter)) / np.sqrt(inter)).astype(np.float32)
    f13, s13 = oracle.pack_fp4(w13)
    f2, s2 = oracle.pack_fp4(w2)
    W13 = np_dequant_fp4(f13, s13)
    W2 = np_dequant_fp4(f2, s2)
    assert np.array_equal(qat.fp8_weights(f13, s13), W13)     # lossless: the backward's weights are the forward's
    assert np.array_equal(qat.fp8_weights(f2, s2), W2)
    xb = bf16_bits_of(rng.normal(0, 1, (T, d)))
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    tw = np.array([[0.75, 0.25]] * T, np.float32)              # dy = w * dout exact in fp32
    doutb = bf16_bits_of(rng.normal(0, 1, (T, d)))
    dx, dw, dW13, dW2 = qat.qat_backward(xb, idx, tw, f13, s13, f2, s2, doutb, quantize_grads=quantize_grads)

    xq, xs = oracle.quant_act(xb)
    xdq = np_fp8_quant(from_bits(xb))[0]
    Wt13 = torch.tensor(W13, requires_grad=True)
    Wt2 = torch.tensor(W2, requires_grad=True)
    xd = torch.tensor(xdq, requires_grad=True)
    wt = torch.tensor(tw.astype(np.float64), requires_grad=True)
    out = torch.zeros((T, d), dtype=torch.float64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            gu = Wt13[e] @ xd[t]
            if quantize_grads:
                gu = _QuantGrad.apply(gu)
            gu = _ste(gu, gu.detach().float().double())
            g, u = gu[:inter], gu[inter:]
            h = torch.nn.functional.silu(g) * u
            _, hq, hs, yb = oracle.expert_pair(xq[t], xs[t], e, f13, s13, f2, s2)
            hd = _ste(h, t_e4m3_decode(hq) * np.ldexp(1.0, np.repeat(hs.astype(np.int64) - 127, 128)))
            y = Wt2[e] @ hd
            if quantize_grads:
                y = _QuantGrad.apply(y)
            y = _ste(y, from_bits(yb).astype(np.float64))
            out[t] = out[t] + wt[t, j] * y
    (out * torch.from_numpy(from_bits(doutb).astype(np.float64))).sum().backward()

    def close(a, b):
        return np.linalg.norm(a - b) <= 1e-10 * max(np.linalg.norm(b), 1e-300)

    assert close(dx, xd.grad.numpy())
    assert close(dw, wt.grad.numpy())
    assert close(dW13, Wt13.grad.numpy())
    assert close(dW2, Wt2.grad.numpy())
    assert np.abs(dW13).max() > 0 and np.abs(dx).max() > 0
