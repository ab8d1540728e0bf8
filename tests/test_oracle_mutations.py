"""The oracle's pins catch plausible mistakes in it.

Each case plants one mistake in a copy of oracle/moe_oracle.c (a swapped
gate/up half, a wrong nibble order, a tie broken the wrong way, a scale rule
off by one, a dropped bias or routing weight, a wrong SiLU sign, an unstable
dispatch order, truncating instead of rounding, a different summation order of
the gate logits, ...), builds the copy with the oracle's own flags, routes the
oracle through it, and runs the pins named beside the mistake: every one of
them must fail.  The real oracle is restored after each case.  No GPU needed.
"""
import os
import tempfile

import pytest

import oracle
from oracle import build as obuild

import test_oracle_pins as pins

# (name, text in moe_oracle.c, its replacement, pins that must fail)
MUTATIONS = [
    ("gate and up halves swapped",
     "g += a[i] * dq_fp4(w13_fp4, w13_scale, row13 + n, d, i);\n"
     "            u += a[i] * dq_fp4(w13_fp4, w13_scale, row13 + inter + n, d, i);",
     "g += a[i] * dq_fp4(w13_fp4, w13_scale, row13 + inter + n, d, i);\n"
     "            u += a[i] * dq_fp4(w13_fp4, w13_scale, row13 + n, d, i);",
     [pins.test_one_hot_probe_gate_up_order_and_nibbles, pins.test_forward_matches_dense_bruteforce_tiny]),
    ("nibble order of the weight decode",
     "(i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xf)",
     "(i & 1) ? (uint8_t)(byte & 0xf) : (uint8_t)(byte >> 4)",
     [pins.test_one_hot_probe_gate_up_order_and_nibbles]),
    ("nibble order of the weight pack",
     "(uint8_t)(lo | (hi << 4))",
     "(uint8_t)(hi | (lo << 4))",
     [pins.test_pack_fp4_matches_bruteforce]),
    ("equal logits go to the higher expert",
     "if (best < 0 || zt[e] > zt[best])",
     "if (best < 0 || zt[e] >= zt[best])",
     [pins.test_topk_bruteforce_and_ties, pins.test_route_duplicated_gate_columns_tie_to_lower_index]),
    ("weights not renormalised",
     "(S == 0.0f) ? 1.0f / (float)k : s[j] / S;",
     "(S == 0.0f) ? 1.0f / (float)k : s[j];",
     [pins.test_topk_bruteforce_and_ties]),
    ("E4M3 scale boundary included",
     "((2.0 * f > 1.75) ? 1 : 0)",
     "((2.0 * f >= 1.75) ? 1 : 0)",
     [pins.test_e4m3_scale_exp_bruteforce]),
    ("MXFP4 exponent off by one",
     "int X = (ex - 1) - 2;",
     "int X = (ex - 1) - 1;",
     [pins.test_mx_scale_exp_bruteforce, pins.test_pack_fp4_matches_bruteforce]),
    ("gate bias dropped",
     "zz = zz + bias[e];",
     "zz = zz + 0.0f * bias[e];",
     [pins.test_gate_logits_error_bound, pins.test_gate_logits_fixed_order_exactly]),
    ("gate chains over contiguous channels",
     "for (int i = l; i < d; i += 32)",
     "for (int i = l * (d / 32); i < (l + 1) * (d / 32); i++)",
     [pins.test_gate_logits_fixed_order_exactly, pins.test_gate_logits_hand_built_order_case]),
    ("gate partials added in a chain",
     "for (int off = 16; off >= 1; off /= 2)\n                for (int l = 0; l < off; l++)\n"
     "                    part[l] = part[l] + part[l + off];",
     "for (int l = 1; l < 32; l++)\n                part[0] = part[0] + part[l];",
     [pins.test_gate_logits_fixed_order_exactly]),
    ("routing weight dropped in the combine",
     "acc = fmaf(w[j], orc_bf16_to_f32(y[(size_t)j * d + m]), acc);",
     "acc = fmaf(1.0f, orc_bf16_to_f32(y[(size_t)j * d + m]), acc);",
     [pins.test_forward_matches_dense_bruteforce_tiny]),
    ("SiLU with the wrong sign",
     "h[n] = (float)(gd / (1.0 + exp(-gd)) * (double)uf);",
     "h[n] = (float)(gd / (1.0 + exp(gd)) * (double)uf);",
     [pins.test_expert_pair_intermediates, pins.test_forward_matches_dense_bruteforce_tiny]),
    ("dispatch order descending within an expert",
     "for (long p = 0; p < P; p++) {\n        long pos = cnt[idx[p]]++;",
     "for (long p = P - 1; p >= 0; p--) {\n        long pos = cnt[idx[p]]++;",
     [lambda: pins.test_dispatch_plan_is_stable_sort_and_bijection(37, 8, 2)]),
    ("bf16 truncation instead of rounding",
     "u += 0x7fffu + lsb;",
     "u += 0u * lsb;",
     [pins.test_bf16_round_matches_torch_cast]),
    ("E4M3 truncation instead of rounding",
     "double mq = nearbyint(ldexp(a, 3 - E));",
     "double mq = floor(ldexp(a, 3 - E));",
     [pins.test_e4m3_encode_matches_torch_cast]),
    ("E2M1 ties away from zero",
     "double mq = nearbyint(ldexp(a, 1 - E));",
     "double mq = floor(ldexp(a, 1 - E) + 0.5);",
     [pins.test_e2m1_encode_matches_bruteforce]),
    ("backward FP8 block exponent one too low",
     "int B = S - 6;",
     "int B = S - 7;",
     [pins.test_fp8t_is_lossless_on_weights_within_the_scale_ratio]),
]


@pytest.fixture(scope="module")
def source():
    with open(obuild.SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_its_pins(name, old, new, catchers, source, tmp_path):
    assert source.count(old) == 1, "the text to mutate must occur exactly once: %r" % old
    path = obuild.build_source(source.replace(old, new), str(tmp_path / "liboracle_variant.so"))
    for pin in catchers:
        with oracle.use_library(path):
            try:
                pin()
            except Exception:       # the pin caught the mistake (AssertionError, or an error it raised)
                continue
        pytest.fail("%r was not caught by %s" % (name, getattr(pin, "__name__", pin)))


def test_unmutated_copy_passes_the_same_pins(source, tmp_path):
    """The procedure itself is sound: a copy built the same way without a
    mistake passes every pin used above."""
    path = obuild.build_source(source, str(tmp_path / "liboracle_copy.so"))
    with oracle.use_library(path):
        for _, _, _, catchers in MUTATIONS:
            for pin in catchers:
                pin()
