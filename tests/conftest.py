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

def tile_codes(fp4):
    """plain codes [E][N][K/2] -> tiled bytes [E][N/256 pairs j][K/128][2 halves h][128 rows][64]:
    the 128-row block h * N/256 + j goes to block ((e * N/256 + j) * K/128 + k/128) * 2 + h."""
    import numpy as np
    E, N, K2 = fp4.shape
    a = fp4.reshape(E, 2, N // 256, 128, K2 // 64, 64)            # (e, h, j, r, kb, byte)
    return np.ascontiguousarray(a.transpose(0, 2, 4, 1, 3, 5))


def tile_scales(sc):
    """plain scales [E][N][K/32] -> tiled bytes [E][N/256][K/128][2][512] in the block
    order of tile_codes, the byte of row r and sub-block j at (r % 32) * 16 + (r / 32) * 4 + j."""
    import numpy as np
    E, N, K32 = sc.shape
    a = sc.reshape(E, 2, N // 256, 4, 32, K32 // 4, 4)       # (e, h, pair, r/32, r%32, kt, j)
    return np.ascontiguousarray(a.transpose(0, 2, 5, 1, 4, 3, 6)).reshape(E, N // 256, K32 // 4, 2, 512)


def sf_byte(r, j):
    return (r % 32) * 16 + (r // 32) * 4 + j
