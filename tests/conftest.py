import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def read_golden(name):
    """Parse a whitespace table under tests/golden/, skipping '#' comment lines."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


# ---- the tiled MXFP4 byte order of moe_pack_fp4 (include/fp4moe.h) ---------
# A pure permutation of the plain layout the oracle writes ([E][N][K/2] codes,
# [E][N][K/32] scales), used to compare the two bit for bit.

def weight_block(e, n128, k128, N, K):
    """Block number of 128 x 128 block (n128, k128) of expert e in the tiled
    layout: row blocks pair as (j, j + H), H = ceil(NB/2), NB = N/128; a pair's
    two blocks are neighbours at each K block; with NB odd the last row block
    is alone, its K blocks consecutive after the pairs'."""
    NB, KB = N // 128, K // 128
    H = (NB + 1) // 2
    h = 1 if n128 >= H else 0
    j = n128 - h * H
    base = e * NB * KB
    return base + (j * KB + k128) * 2 + h if j < NB // 2 else base + 2 * (NB // 2) * KB + k128


def fp8t_block(e, rb, cb, R, C):
    """Block number of 128 x 128 block (rb, cb) of expert e's transposed FP8
    weights ([R][C] per expert): row blocks pair as (2j, 2j + 1), a pair's two
    blocks neighbours at every column block; an odd last row block alone, its
    column blocks after the pairs'."""
    RB, CB = R // 128, C // 128
    J = RB // 2
    base = e * RB * CB
    return base + ((rb // 2) * CB + cb) * 2 + rb % 2 if rb // 2 < J else base + 2 * J * CB + cb


def tile_fp8t(w8t):
    """plain transposed codes [E][R][C] -> tiled bytes [E * RB * CB blocks][128][128]."""
    import numpy as np
    E, R, C = w8t.shape
    out = np.empty((E * (R // 128) * (C // 128), 128, 128), np.uint8)
    for rb in range(R // 128):
        for cb in range(C // 128):
            idx = [fp8t_block(e, rb, cb, R, C) for e in range(E)]
            out[idx] = w8t[:, rb * 128:(rb + 1) * 128, cb * 128:(cb + 1) * 128]
    return out


def tile_codes(fp4):
    """plain codes [E][N][K/2] -> tiled bytes [E * NB * KB blocks][128 rows][64]."""
    import numpy as np
    E, N, K2 = fp4.shape
    K = 2 * K2
    NB, KB = N // 128, K // 128
    out = np.empty((E * NB * KB, 128, 64), np.uint8)
    for n128 in range(NB):
        for kb in range(KB):
            idx = [weight_block(e, n128, kb, N, K) for e in range(E)]
            out[idx] = fp4[:, n128 * 128:(n128 + 1) * 128, kb * 64:(kb + 1) * 64]
    return out


def tile_scales(sc):
    """plain scales [E][N][K/32] -> tiled bytes [E * NB * KB blocks][512] in the block
    order of tile_codes, the byte of row r and sub-block j at (r % 32) * 16 + (r / 32) * 4 + j."""
    import numpy as np
    E, N, K32 = sc.shape
    K = 32 * K32
    NB, KB = N // 128, K // 128
    out = np.empty((E * NB * KB, 512), np.uint8)
    r = np.arange(128)
    for n128 in range(NB):
        for kb in range(KB):
            idx = [weight_block(e, n128, kb, N, K) for e in range(E)]
            blk = sc[:, n128 * 128:(n128 + 1) * 128, kb * 4:(kb + 1) * 4]       # [E][128][4]
            img = np.empty((E, 512), np.uint8)
            for j in range(4):
                img[:, (r % 32) * 16 + (r // 32) * 4 + j] = blk[:, :, j]
            out[idx] = img
    return out


def sf_byte(r, j):
    return (r % 32) * 16 + (r // 32) * 4 + j
