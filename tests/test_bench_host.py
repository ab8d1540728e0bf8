"""CPU tests of the benchmark's host logic: FLOP/byte accounting against the
cited identity, the max-over-ranks reduction on a 2-rank gloo group, and the
reference arm's JSON line (single process and under torchrun with 2 ranks)."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT, read_golden

sys.path.insert(0, ROOT)
import bench  # noqa: E402
from fp4_expert_grouped_gb300 import inputs  # noqa: E402


def test_flop_identity_matches_cited_ratio():
    g = dict(read_golden("flop_identity.txt"))
    assert g["flops_per_pair_formula"] == "6*h*d" and g["bytes_per_pair_formula"] == "3*h"
    w = inputs.Workload("x", T=3, d=7168, inter=3072, E=8, k=2, seed=0)
    t_roof, bound, flops, _ = bench.layer_roofline(w, touched=8, hbm_gbs=1.0, fp8_tflops=1.0)
    assert flops == 6 * w.d * w.inter * w.P
    # FLOPs per byte of (FP8 dispatch + BF16 combine) = 6hd / 3h = 2d; with the
    # inferred intermediate size d = 3072 this is the page's 6.1 TFLOP/s per GB/s
    ratio = (6 * w.d * w.inter) / (3 * w.d)
    assert abs(ratio / 1e3 - float(g["tflops_per_gbps_v4pro"])) < 0.05
    assert bench.gemm_flops(w, "gemm1") + bench.gemm_flops(w, "gemm2") == flops


def test_kernels_per_step_follow_the_library_thresholds():
    """gpu_launches claim: the gate and top-k (two kernels; on the tensor-core
    path from 1024 tokens with E a multiple of 64 two more for gate_w's split
    and norms unless they were prepared at load time, as the bench does), plan
    (one kernel up to 32768 pairs, a count and a scatter kernel above), the
    expert-ordered copy (from 16 pairs per expert on average), GEMM1, GEMM2,
    combine."""
    want = {"tiny": 6, "decode": 6, "mid": 7, "skew": 8, "prefill": 8}
    for name, n in want.items():
        assert bench.kernels_per_step(inputs.WORKLOADS[name]) == n, name
    assert bench.kernels_per_step(inputs.WORKLOADS["prefill"], gate_prepared=False) == 10
    edge = inputs.Workload("edge", T=4096, d=256, inter=128, E=256, k=8, seed=0)    # 32768 pairs: one plan kernel
    assert bench.kernels_per_step(edge) == 7
    edge = inputs.Workload("edge", T=4097, d=256, inter=128, E=256, k=8, seed=0)    # 32776 pairs: two
    assert bench.kernels_per_step(edge) == 8
    edge = inputs.Workload("edge", T=511, d=256, inter=128, E=256, k=8, seed=0)     # 4088 < 16 E: no copy
    assert bench.kernels_per_step(edge) == 6
    edge = inputs.Workload("edge", T=1023, d=256, inter=128, E=256, k=8, seed=0)    # below the tensor-core gate
    assert bench.kernels_per_step(edge) == 7
    edge = inputs.Workload("edge", T=2048, d=256, inter=128, E=40, k=8, seed=0)     # E not a multiple of 64
    assert bench.kernels_per_step(edge) == 7


def test_clock_window_keeps_the_gpu_busy_for_the_sampler():
    assert bench.clock_window_steps(0.555, 20) == 1782        # decode: 11 ms timed, ~1 s in all
    assert bench.clock_window_steps(6.2, 20) == 142           # prefill
    assert bench.clock_window_steps(60.0, 20) == 0            # already longer than the window
    assert bench.clock_window_steps(0.001, 1) == 20000        # capped
    assert bench.clock_window_steps(0.0, 5) == 0


def test_weight_bytes_per_expert():
    assert bench.weight_bytes_per_expert(4096, 2048) == 13_369_344
    assert bench.weight_bytes_per_expert(7168, 2048) == 23_396_352


def _rank_main(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    ws, r, _ = bench.dist_setup(want_nccl=False)
    bench.dist_barrier()
    v = bench.dist_max(10.0 + 5 * r, "cpu")
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, ws, v))


def test_dist_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29611
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
            "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"}


def test_reference_arm_json_line_cpu():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                        "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert REQUIRED <= set(d)
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_under_torchrun_two_ranks():
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", "29623", "bench.py", "--impl", "reference",
                        "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                                  # rank 0 alone prints
    assert json.loads(lines[0])["n_gpus"] == 2
