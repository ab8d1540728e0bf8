"""Exhaustive parity of the GPU's FP4 and FP8 conversions with the oracle's
encoders, through the C ABI (the OCP MX / FP8 formats [P1] section 4 cites).

E2M1: every finite fp32 of magnitude <= 6, both signs (about 2.2e9 values),
goes through moe_pack_fp4.  Each 32-element block starts with a 6.0 marker,
which fixes the block's power-of-two scale at 2^0, so every other element's
code is the E2M1 encoding of that exact fp32 value: rounding ties, values
between codes, subnormals and signed zeros all included.

E4M3: every finite bf16 value goes through moe_quantize_act, once in
128-channel groups whose largest magnitude is 448 (scale 2^0: the codes are
the E4M3 encodings of the values themselves) and once in groups of
consecutive bit patterns (every scale the values produce).
"""
import numpy as np
import pytest
import torch

import oracle
from conftest import tile_codes, tile_fp8t, tile_scales

pytestmark = pytest.mark.gpu

DEV = "cuda"
SIX_BITS = 0x40C00000          # fp32 6.0, the largest E2M1 magnitude
BF16_448 = 0x43E0              # bf16 448.0, the largest E4M3 magnitude


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)


def capi():
    from fp4_expert_grouped_gb300 import capi as c
    return c


def test_e2m1_conversion_exhaustive():
    c = capi()
    N, K = 16384, 4096
    per = N * (K // 32) * 31                       # swept values per chunk
    top = SIX_BITS + 1                             # magnitudes 0 .. 6.0 as bit patterns
    fp4 = torch.empty((1, N, K // 2), dtype=torch.uint8, device=DEV)
    sc = torch.empty((1, N, K // 32), dtype=torch.uint8, device=DEV)
    blocks = np.empty((N, K // 32, 32), np.uint32)
    blocks[:, :, 0] = SIX_BITS
    swept = 0
    for sign in (0, 0x80000000):
        for start in range(0, top, per):
            n = min(per, top - start)
            body = np.zeros(per, np.uint32)
            body[:n] = np.arange(start, start + n, dtype=np.uint32) | np.uint32(sign)
            blocks[:, :, 1:] = body.reshape(N, K // 32, 31)
            w = blocks.view(np.float32).reshape(1, N, K)
            c.moe_pack_fp4(torch.from_numpy(w).to(DEV), fp4, sc)
            of, os_ = oracle.pack_fp4(w)
            got_codes = fp4.cpu().numpy().reshape(-1)
            want_codes = tile_codes(of).reshape(-1)
            if not np.array_equal(got_codes, want_codes):
                bad = np.flatnonzero(got_codes != want_codes)[:4]
                pytest.fail("E2M1 codes differ from the oracle in the chunk from %#x (sign %#x), tiled bytes %s"
                            % (start, sign, bad.tolist()))
            assert np.array_equal(sc.cpu().numpy().reshape(-1), tile_scales(os_).reshape(-1))
            assert np.all(os_ == 127)              # every block scaled by 2^0
            swept += n
    assert swept == 2 * top


def _finite_bf16_patterns():
    p = np.arange(1 << 16, dtype=np.uint32)
    return p[(p & 0x7F80) != 0x7F80].astype(np.uint16)     # drop Inf and NaN


def _quantize(bits_2d):
    c = capi()
    T, d = bits_2d.shape
    x = torch.from_numpy(bits_2d.view(np.int16).copy()).view(torch.bfloat16).to(DEV)
    xq = torch.empty((T, d), dtype=torch.uint8, device=DEV)
    xs = torch.empty((T, d // 128), dtype=torch.uint8, device=DEV)
    c.moe_quantize_act(x, xq, xs)
    oq, os_ = oracle.quant_act(bits_2d)
    assert np.array_equal(xs.cpu().numpy(), os_)
    assert np.array_equal(xq.cpu().numpy(), oq)
    return os_


def test_e4m3_conversion_exhaustive_over_bf16():
    p = _finite_bf16_patterns()
    # groups led by 448: every finite bf16 of magnitude <= 448, codes at scale 2^0
    small = p[(p & 0x7FFF) <= BF16_448]
    groups = -(-small.size // 127)
    body = np.zeros(groups * 127, np.uint16)
    body[:small.size] = small
    led = np.empty((groups, 128), np.uint16)
    led[:, 0] = BF16_448
    led[:, 1:] = body.reshape(groups, 127)
    rows = -(-groups // 8)
    x = np.zeros((rows * 8, 128), np.uint16)
    x[:groups] = led
    xs = _quantize(x.reshape(rows, 8 * 128))
    assert np.all(xs.reshape(-1)[:groups] == 127)
    # groups of consecutive patterns: every finite bf16, every scale it produces
    d = 1024
    full = np.zeros(-(-p.size // d) * d, np.uint16)
    full[:p.size] = p
    _quantize(full.reshape(-1, d))


@pytest.mark.parametrize("E,N,K", [(3, 512, 384), (1, 256, 128), (2, 384, 256)])   # N/128 odd: a lone last block
def test_fp4_to_fp8t_bitexact(E, N, K):
    """FP8 weights for the backward pass (transposed, one exponent per 128x128
    block) from the GPU pack: the oracle's codes and block exponents bit for bit,
    on trained-like weights, an all-zero block and a block whose sub-block
    scales span more than 2^14 (rounded, not lossless)."""
    rng = np.random.default_rng(E * N + K)
    w = (rng.normal(0, 1, (E, N, K)) / np.sqrt(K)).astype(np.float32)
    w[0, :128, :128] = 0.0
    if E > 1:
        w[E - 1, 128:256, 128:160] = rng.uniform(-300, 300, (128, 32))
        w[E - 1, 128:256, 160:192] = rng.uniform(-1, 1, (128, 32)) * 2.0 ** -16
    check_fp4_to_fp8t(w)


def test_fp4_to_fp8t_bitexact_scale_spread():
    """Every 1x32 sub-block at its own power of two, 2^-24 .. 2^8, so that inside
    each 128x128 block the shifts X - B run from 0 down far past E4M3's
    subnormals: exact codes, round-to-nearest-even below 2^-6, underflow to a
    signed zero; and one sub-block of every E2M1 value at both signs.  Bit-exact
    with the oracle."""
    rng = np.random.default_rng(2024)
    E, N, K = 2, 256, 512
    w = rng.normal(0, 1, (E, N, K)).astype(np.float32)
    shift = rng.integers(-24, 9, (E, N, K // 32))
    w *= np.repeat(np.exp2(shift.astype(np.float64)), 32, axis=2).astype(np.float32)
    vals = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float32)
    w[1, 5, 64:96] = np.concatenate([vals, -vals, vals * 4, -vals * 4])
    check_fp4_to_fp8t(w)


def check_fp4_to_fp8t(w):
    c = capi()
    E, N, K = w.shape
    wd = torch.from_numpy(w).to(DEV)
    fp4 = torch.empty((E, N, K // 2), dtype=torch.uint8, device=DEV)
    sc = torch.empty((E, N, K // 32), dtype=torch.uint8, device=DEV)
    c.moe_pack_fp4(wd, fp4, sc)
    w8t = torch.empty((E, K, N), dtype=torch.uint8, device=DEV)
    s8t = torch.empty((E, K // 128, N // 128), dtype=torch.uint8, device=DEV)
    c.moe_fp4_to_fp8t(fp4, sc, w8t, s8t)
    of, os_ = oracle.pack_fp4(w)
    rw, rs = oracle.fp4_to_fp8t(of, os_)
    assert np.array_equal(s8t.cpu().numpy(), rs)
    got = w8t.cpu().numpy().reshape(-1, 128, 128)
    want = tile_fp8t(rw)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)[:4]
        pytest.fail("codes differ at (block, row, column) %s" % bad.tolist())
    assert c.moe_get_device_status() == 0
