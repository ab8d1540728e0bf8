"""Host-side checks of the C ABI that need no GPU: the library builds and loads,
exports every function include/fp4moe.h declares, and rejects bad arguments
before it touches CUDA (nothing is launched in these tests)."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fp4moe.h")


@pytest.fixture(scope="module")
def capi():
    from fp4_expert_grouped_gb300 import build
    build.build()
    from fp4_expert_grouped_gb300 import capi as c
    return c


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declarations_exported(capi):
    names = declared_functions()
    assert names, "no declarations parsed"
    assert sorted(capi.EXPORTS) == names
    lib = capi.lib()
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    assert set(names) <= exported


def test_status_strings(capi):
    for code, name in capi.STATUS_NAMES.items():
        assert capi.moe_status_string(code) == name
    assert capi.moe_status_string(99) == "MOE_ERR_UNKNOWN"
    assert capi.moe_version() >= 100


FAKE = 0x100000          # an aligned address that is never dereferenced: every call below is rejected first


def fwd(lib, T=8, d=256, inter=128, E=8, k=2, x=FAKE, out=FAKE, w13=FAKE, w2=FAKE, opts=None):
    return lib.moe_forward_ex(x, FAKE, w13, FAKE, w2, FAKE, out, T, d, inter, E, k, None,
                              ctypes.byref(opts) if opts is not None else None)


def test_forward_argument_checks(capi):
    lib = capi.lib()
    INV, SHAPE, WS = 1, 2, 4
    assert fwd(lib, x=0) == INV
    assert fwd(lib, out=0) == INV
    assert fwd(lib, x=FAKE + 2) == INV                      # misaligned activations
    assert fwd(lib, w13=FAKE + 16) == INV                   # packed weights need 32-byte alignment
    assert fwd(lib, T=-1) == INV
    assert fwd(lib, d=320) == SHAPE                         # d % 128
    assert fwd(lib, inter=192) == SHAPE                     # inter % 128
    assert fwd(lib, k=9, E=16) == SHAPE
    assert fwd(lib, k=4, E=3) == SHAPE
    assert fwd(lib, E=300) == SHAPE
    assert fwd(lib, T=1 << 28, k=8) == SHAPE                # T*k >= 2^31
    o = capi.MoeForwardOpts()
    o.flags = 2                                             # no such flag
    assert fwd(lib, opts=o) == INV
    o = capi.MoeForwardOpts()
    o.workspace = FAKE
    o.workspace_bytes = 16
    assert fwd(lib, opts=o) == WS                           # caller workspace too small
    o = capi.MoeForwardOpts()
    o.workspace = FAKE + 16
    o.workspace_bytes = 1 << 40
    assert fwd(lib, opts=o) == WS                           # not 256-byte aligned
    assert fwd(lib, T=0) == 0                               # empty batch is a no-op


def test_other_entry_points_reject_bad_arguments(capi):
    lib = capi.lib()
    assert lib.moe_pack_fp4(None, FAKE, FAKE, 1, 128, 128, None) == 1
    assert lib.moe_pack_fp4(FAKE, FAKE, FAKE, 1, 128, 96, None) == 2     # K % 128
    assert lib.moe_pack_fp4(FAKE, FAKE, FAKE, 1, 64, 128, None) == 2     # N % 128
    assert lib.moe_pack_fp4(FAKE, FAKE, FAKE, 1, 320, 128, None) == 2
    assert lib.moe_pack_fp4(FAKE, FAKE, FAKE, 0, 256, 128, None) == 0
    assert lib.moe_quantize_act(FAKE, FAKE, FAKE, 4, 100, None) == 2
    assert lib.moe_quantize_act(FAKE, FAKE, FAKE, 0, 128, None) == 0
    assert lib.moe_route(FAKE, FAKE, None, FAKE, FAKE, 4, 128, 8, 9, None) == 2
    assert lib.moe_route(FAKE, None, None, FAKE, FAKE, 4, 128, 8, 2, None) == 1
    assert lib.moe_route(FAKE, FAKE, None, FAKE, FAKE, 0, 128, 8, 2, None) == 0
    assert lib.moe_dispatch_plan(FAKE, FAKE, FAKE, None, 4, 8, 2, None) == 1
    assert lib.moe_dispatch_plan(FAKE, FAKE, FAKE, FAKE, 4, 300, 2, None) == 2


def test_fp4_to_fp8t_argument_checks(capi):
    lib = capi._lib
    assert lib.moe_fp4_to_fp8t(None, FAKE, FAKE, FAKE, 1, 256, 128, None) == 1
    assert lib.moe_fp4_to_fp8t(FAKE, FAKE, FAKE + 8, FAKE, 1, 256, 128, None) == 1     # w8t not 16-byte aligned
    assert lib.moe_fp4_to_fp8t(FAKE, FAKE, FAKE, FAKE, -1, 256, 128, None) == 1
    assert lib.moe_fp4_to_fp8t(FAKE, FAKE, FAKE, FAKE, 1, 192, 128, None) == 2          # N % 128
    assert lib.moe_fp4_to_fp8t(FAKE, FAKE, FAKE, FAKE, 1, 256, 96, None) == 2           # K % 128
    assert lib.moe_fp4_to_fp8t(FAKE, FAKE, FAKE, FAKE, 0, 256, 128, None) == 0          # nothing to do


def test_workspace_layout(capi):
    # row tiles of 16 (the first two), 32, 64 and 128 pairs
    for (T, d, inter, E, k) in [(32, 256, 128, 8, 2), (128, 4096, 2048, 256, 8), (512, 4096, 2048, 256, 8),
                                (1536, 4096, 2048, 256, 8), (16384, 7168, 2048, 256, 8)]:
        total, off, st = capi.moe_workspace_layout(T, d, inter, E, k)
        assert total == capi.moe_workspace_size(T, d, inter, E, k) > 0
        P = T * k
        xs = ((d // 128) + 3) // 4 * 4
        R = 16 if P <= 8 * E else 32 if P <= 20 * E else 64 if P <= 48 * E else 128    # rows per GEMM row tile
        tiles = (P + R - 1) // R + min(P, E)
        gx, gh = (d // 128 + 3) // 4, (inter // 128 + 3) // 4
        chunks = (P + 2047) // 2048
        tc = T >= capi.MOE_GATE_TC_MIN_TOKENS and E % 64 == 0         # the tensor-core gate's scratch
        sizes = [T * d, T * xs, T * E * 4, P * 4, P * 4, (E + 1) * 4, P * 4, P * 4, (E + 1) * 4,
                 P * inter, tiles * gh * 512, P * d * 2, P * d, tiles * gx * 512,
                 chunks * E * 4 if chunks > 1 else 0, (tiles + 1) * 4, P * 4,
                 E * d * 4 * tc, E * d * 2 * tc, E * d * 2 * tc, E * 4 * tc, T * 4 * tc]
        assert len(sizes) == capi.MOE_WS_COUNT
        for i in range(capi.MOE_WS_COUNT):
            assert off[i] % 256 == 0
            end = off[i] + sizes[i]
            nxt = off[i + 1] if i + 1 < capi.MOE_WS_COUNT else total
            assert end <= nxt
        assert st[capi.MOE_WS_XS] == xs and st[capi.MOE_WS_HS_TILES] == gh * 512 and st[capi.MOE_WS_Y] == 2 * d
    assert capi.moe_workspace_size(8, 320, 128, 8, 2) == 0
    assert capi.moe_workspace_size(8, 384, 128, 8, 2) > 0                     # d % 128 is enough


def test_backward_h_argument_checks(capi):
    """moe_backward_h rejects bad shapes and pointers before touching CUDA."""
    lib = capi.lib()
    F = FAKE
    assert lib.moe_backward_h(F, F, F, F, F, None, 0, F, F, None, 8, 256, 384, 8, 2, None) == 2   # inter % 256
    assert lib.moe_backward_h(F, F, F, F, F, None, 0, F, F, None, 8, 384, 256, 8, 2, None) == 2   # d % 256
    assert lib.moe_backward_h(F, F, F, F, F, None, 0, None, F, None, 8, 256, 256, 8, 2, None) == 1  # no output
    assert lib.moe_backward_h(F, F, F, F + 16, F, None, 0, F, F, None, 8, 256, 256, 8, 2, None) == 1  # gu alignment
    assert lib.moe_backward_h(F, F, F, F, F, F, 16, F, F, None, 8, 256, 256, 8, 2, None) == 4      # workspace too small
    assert lib.moe_backward_h(F, F, F, F, F, None, 0, F, F, None, 0, 256, 256, 8, 2, None) == 0    # T == 0: no-op
    assert capi.moe_backward_h_workspace_size(8, 256, 384, 8, 2) == 0
    assert capi.moe_backward_h_workspace_size(8, 256, 256, 8, 2) > 0


def test_backward_x_argument_checks(capi):
    """moe_backward_x rejects bad shapes and pointers before touching CUDA."""
    lib = capi.lib()
    F = 0x100000
    assert lib.moe_backward_x(F, F, F, F, F, None, 0, F, 8, 256, 384, 8, 2, None) == 2      # inter % 256
    assert lib.moe_backward_x(F, F, F, F, F, None, 0, F, 8, 384, 256, 8, 2, None) == 2      # d % 256
    assert lib.moe_backward_x(F, F, F, F, F, None, 0, None, 8, 256, 256, 8, 2, None) == 1   # no output
    assert lib.moe_backward_x(F + 8, F, F, F, F, None, 0, F, 8, 256, 256, 8, 2, None) == 1  # dgu alignment
    assert lib.moe_backward_x(F, F, F, F, F, F, 16, F, 8, 256, 256, 8, 2, None) == 4        # workspace too small
    assert lib.moe_backward_x(F, F, F, F, F, None, 0, F, 0, 256, 256, 8, 2, None) == 0      # T == 0: no-op
    assert capi.moe_backward_x_workspace_size(8, 256, 384, 8, 2) == 0
    assert capi.moe_backward_x_workspace_size(8, 256, 256, 8, 2) > 0


def test_backward_dw_argument_checks(capi):
    """moe_backward_dw rejects bad shapes and pointers before touching CUDA."""
    lib = capi.lib()
    F = 0x100000
    assert lib.moe_backward_dw(F, F, None, 8, 256, 256, 8, 2, None) == 1       # no output
    assert lib.moe_backward_dw(F + 8, F, F, 8, 256, 256, 8, 2, None) == 1      # dout alignment
    assert lib.moe_backward_dw(F, F, F, 8, 320, 256, 8, 2, None) == 2          # d % 128
    assert lib.moe_backward_dw(F, F, F, 0, 256, 256, 8, 2, None) == 0          # T == 0: no-op


def test_backward_w_argument_checks(capi):
    """moe_backward_w rejects bad shapes and pointers before touching CUDA."""
    lib = capi.lib()
    F = 0x100000
    assert lib.moe_backward_w(F, F, F, F, F, F, None, 0, 8, 256, 384, 8, 2, None) == 2      # inter % 256
    assert lib.moe_backward_w(F, F, F, F, F, F, None, 0, 8, 384, 256, 8, 2, None) == 2      # d % 256
    assert lib.moe_backward_w(F, None, F, F, F, F, None, 0, 8, 256, 256, 8, 2, None) == 1   # no dy source
    assert lib.moe_backward_w(F, F, F, F, F + 16, F, None, 0, 8, 256, 256, 8, 2, None) == 1  # dW13 alignment
    assert lib.moe_backward_w(F, F, F, F, F, F, F, 16, 8, 256, 256, 8, 2, None) == 4        # workspace too small
    assert capi.moe_backward_w_workspace_size(8, 256, 384, 8, 2) == 0
    assert capi.moe_backward_w_workspace_size(8, 256, 256, 8, 2) > 0


def test_prepare_gate_argument_checks(capi):
    """moe_prepare_gate and moe_gate_prep_size reject bad shapes and pointers
    before touching CUDA; the size covers the four parts, 256-byte aligned."""
    lib = capi.lib()
    F = 0x100000
    assert capi.moe_gate_prep_size(320, 64) == 0                          # d % 128
    assert capi.moe_gate_prep_size(256, 300) == 0                         # E > 256
    d, E = 512, 64
    assert capi.moe_gate_prep_size(d, E) == E * d * 4 + 2 * E * d * 2 + 256
    assert lib.moe_prepare_gate(None, F, d, E, None) == 1
    assert lib.moe_prepare_gate(F, F + 16, d, E, None) == 1              # prep alignment
    assert lib.moe_prepare_gate(F, F, 320, E, None) == 2
