#!/usr/bin/env python
"""MoE-layer forward throughput on GB300 (tokens/s) with its roofline fraction.

One step = one moe_forward_ex call over one batch of a synthetic workload: gate
+ top-k + FP8 quantisation, dispatch plan, dispatch (rows of densely filled
tiles copied to expert order; the rows of sparse tiles are gathered inside
GEMM1), grouped GEMM1 (SwiGLU, FP8 re-quantisation), grouped GEMM2 and the
combine -- every stage of the layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
  python bench.py --impl reference ...     # the CPU oracle on the host cores

Timing: W untimed warm-up steps, then K steps, each timed with a pair of CUDA
events on the launching stream, with a 256 MiB write between steps to flush
L2; barrier + synchronize on both sides of the timed loop; the per-step time
is the max over ranks.  A second pass of K steps records an event between
every two stages (the library does it when given events) for the per-stage
times and the dominant kernel's roofline fraction; those events stop the
stages from overlapping their launches, so that pass is slightly slower and is
reported separately.  Under
torchrun (N > 1) every rank runs its own replica of the workload (token-sharded
data parallelism: there is no exchange between ranks), so scaling is weak.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "MoE-layer tokens/sec at 1 GB300; achieved TFLOP/s or HBM GB/s as % of roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0           # nominal dense FP8 / BF16 tensor-core ratio (4.5 / 2.25 PFLOP/s)
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="prefill",
                    help="tiny, decode, mid, skew or prefill (the largest configuration, the default)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8t", action="store_true",
                    help="instead of the layer: time moe_fp4_to_fp8t (FP8 weights for the backward pass) on "
                         "the workload's W13 and W2 shapes and print one JSON line per matrix")
    ap.add_argument("--dgrad", action="store_true",
                    help="instead of the layer: time moe_backward_h (the backward's dh = W2^T dy GEMM with the "
                         "SwiGLU backward, QAT) and moe_backward_x (dx = W13^T [dg; du] summed over a token's "
                         "slots) on the workload, against their FP8 tensor-core roofline; one JSON line each")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (a smaller case of the workload, e.g. for an ncu capture)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (a smaller case of the workload, e.g. for an ncu capture)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def dist_setup(want_nccl=True):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if (want_nccl and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def dist_max(v, device):
    """Max of a float over ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", FALLBACK_HBM_GBS), d.get("bf16_tflops", FALLBACK_BF16_TFLOPS), \
            d.get("bf16_tflops_sustained"), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, None, "fallback"


# How long the clock sampler watches the timed work: a short timed region
# (decode: ~11 ms) ends between two samples, so the same steps keep running,
# untimed, until the GPU has been under this load for about this long.
CLOCK_WINDOW_S = 1.0


def clock_window_steps(ms_per_step, timed_steps, window_s=CLOCK_WINDOW_S, cap=20000):
    """Untimed steps to run after `timed_steps` steps of `ms_per_step` so that
    the work lasts about `window_s` in all (at most `cap`)."""
    done = timed_steps * ms_per_step / 1e3
    if ms_per_step <= 0 or done >= window_s:
        return 0
    return min(cap, int(math.ceil((window_s - done) / (ms_per_step / 1e3))))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)              # the last sample under load, not a stretch of idle ones
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profile_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    if there is none or the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel, workload))
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    src = os.path.join(ROOT, "fp4_expert_grouped_gb300", "csrc", "gemm.cu" if "gemm" in kernel else "kernels.cu")
    if vals.get("source_sha") != file_sha(src):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# -------------------------------------------------------------- accounting

def weight_bytes_per_expert(d, inter):
    """FP4 codes (1/2 byte) + UE8M0 scales (1/32 byte) of W13 and W2."""
    return 3 * d * inter // 2 + 3 * d * inter // 32


def gemm_bytes(w, touched, which):
    """Algorithmic bytes of one grouped-GEMM launch: the touched experts' packed
    weights read once, the pair rows read once, the outputs written once."""
    d, I, P = w.d, w.inter, w.P
    if which == "gemm1":
        wb = touched * (2 * I * d // 2 + 2 * I * d // 32)
        return wb + P * d + P * (d // 128) + P * I + P * (I // 128)
    wb = touched * (d * I // 2 + d * I // 32)
    return wb + P * I + P * (I // 128) + P * d * 2


def gemm_flops(w, which):
    return 2 * w.P * w.d * (2 * w.inter if which == "gemm1" else w.inter)


GATE_TC_MIN_TOKENS = 1024      # the library's tensor-core gate threshold (include/fp4moe.h)


def kernels_per_step(w, gate_prepared=True):
    """Kernels the library launches for one forward of workload w: the gate
    and top-k (two kernels below 1024 tokens; from there, with E a multiple of
    64, the tensor-core logits and the certified top-k, plus gate_w's split
    and weight norms unless prepared at load time), the dispatch plan (a count
    and a scatter kernel beyond 32768 pairs, one kernel up to that), the
    expert-ordered copy (from 16 pairs per expert on average), GEMM1, GEMM2,
    combine."""
    gate = (2 if gate_prepared else 4) if w.T >= GATE_TC_MIN_TOKENS and w.E % 64 == 0 else 2
    plan = 2 if w.P > 32768 else 1
    dispatch = 1 if w.P >= 16 * w.E else 0
    return gate + plan + dispatch + 3


def layer_roofline(w, touched, hbm_gbs, fp8_tflops):
    """The layer's roofline time (us): the slower of 6*d*I FLOPs per pair at the
    FP8 peak and (touched weights + x + out + gate_w) bytes at HBM bandwidth."""
    flops = 6.0 * w.d * w.inter * w.P
    byts = touched * weight_bytes_per_expert(w.d, w.inter) + 2 * w.T * w.d * 2 + w.d * w.E * 4
    t_f = flops / (fp8_tflops * 1e12) * 1e6
    t_b = byts / (hbm_gbs * 1e9) * 1e6
    return max(t_f, t_b), ("tensor" if t_f > t_b else "hbm"), flops, byts


# ------------------------------------------------------------- CPU oracle

class OraclePacks:
    """The oracle's MXFP4 packs of a workload's experts, made on first use and
    kept for the rest of the run (plain [E][N][K/2] codes and [E][N][K/32]
    scales, packed by the oracle from the same seeded fp32 weights the GPU
    packs).  Packing an expert of the largest workload means generating and
    copying 176 MB of fp32 weights, so every sample packs only the experts no
    earlier sample needed; packing is never inside a timed region."""

    def __init__(self, w):
        self.w = w
        self.f13 = np.zeros((w.E, 2 * w.inter, w.d // 2), np.uint8)
        self.s13 = np.zeros((w.E, 2 * w.inter, w.d // 32), np.uint8)
        self.f2 = np.zeros((w.E, w.d, w.inter // 2), np.uint8)
        self.s2 = np.zeros((w.E, w.d, w.inter // 32), np.uint8)
        self.done = set()

    def need(self, experts):
        import oracle
        from fp4_expert_grouped_gb300 import inputs
        gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
        for e in sorted(set(int(v) for v in experts) - self.done):
            a, b = inputs.make_expert(self.w, e, gen_dev)
            r13 = oracle.pack_fp4(a.cpu().numpy()[None])
            r2 = oracle.pack_fp4(b.cpu().numpy()[None])
            self.f13[e], self.s13[e] = r13[0][0], r13[1][0]
            self.f2[e], self.s2[e] = r2[0][0], r2[1][0]
            self.done.add(e)


def oracle_sample(w, x, gw, bias, n_tok, seed=12345, packs=None):
    """Time the CPU oracle on a seeded sample of n_tok tokens of the workload.
    Returns (seconds, tokens, cores).  The experts those tokens route to are
    packed by the oracle first (outside the timed call; see OraclePacks)."""
    import oracle
    from fp4_expert_grouped_gb300 import inputs
    rng = np.random.default_rng(seed)
    tokens = np.sort(rng.choice(w.T, min(n_tok, w.T), replace=False)).astype(np.int32)
    xb = inputs.bf16_bits(x)
    gwn = gw.detach().cpu().numpy()
    bn = None if bias is None else bias.detach().cpu().numpy()
    ridx, _ = oracle.route(xb[tokens], gwn, w.k, bn)
    packs = OraclePacks(w) if packs is None else packs
    packs.need(ridx.reshape(-1))
    t0 = time.perf_counter()
    oracle.moe_forward(xb, gwn, packs.f13, packs.s13, packs.f2, packs.s2, w.k, bn, tokens=tokens)
    dt = time.perf_counter() - t0
    return dt, len(tokens), oracle.num_threads()


# ------------------------------------------------------------ reference arm

def run_reference(args, w, ws_, rank):
    if rank != 0:
        return
    from fp4_expert_grouped_gb300 import inputs
    import oracle
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    x, gw, b = inputs.make_x_gate(w, dev)
    cores = oracle.num_threads()
    n_tok = max(1, min(w.T, cores))
    packs = OraclePacks(w)
    for _ in range(args.warmup):
        oracle_sample(w, x, gw, b, 1, seed=999, packs=packs)
    times = []
    for s in range(args.steps):
        dt, n, _ = oracle_sample(w, x, gw, b, n_tok, seed=1000 + s, packs=packs)
        times.append(dt / n)
    per_tok = statistics.mean(times)
    value = 1.0 / per_tok
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_tok * n_tok * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 accumulate (oracle)", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d seeded tokens per step of the %s workload" % (n_tok, w.name)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w):
    return {"workload": w.name, "T": w.T, "d": w.d, "inter": w.inter, "E": w.E, "k": w.k,
            "zipf_bias": w.zipf_bias, "seed": w.seed,
            "weights": "experts packed to MXFP4 and gate_w prepared for the tensor-core gate at load time",
            "l2": "flushed (256 MiB write) before every timed step; weights %.2f GB >> 129 MB L2"
                  % (w.E * weight_bytes_per_expert(w.d, w.inter) / 1e9)}


# ------------------------------------------------------------------ our arm

def run_ours(args, w, world, rank, local):
    from fp4_expert_grouped_gb300 import capi, inputs, layer
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_gbs, bf16_tflops, bf16_sust, peak_src = measured_peaks()
    fp8_tflops = bf16_tflops * FP8_OVER_BF16

    x, gw, bias = inputs.make_x_gate(w, dev)
    pk = layer.pack_workload(w, dev)
    ws = layer.workspace(w.T, w.d, w.inter, w.E, w.k, dev)
    # gate_w's form for the tensor-core gate, prepared at load time like the
    # packed experts (a function of the weights only)
    gprep = layer.prepare_gate(gw)
    out = torch.empty_like(x)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    nst = len(capi.STAGES)

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)]
        for e in evs:
            e.record(stream)          # materialise the event handles
        return evs

    def step(evs):
        capi.moe_forward_ex(x, gw, pk.w13_fp4, pk.w13_scale, pk.w2_fp4, pk.w2_scale, out, w.k,
                            stream=stream, gate_bias=bias, workspace=ws, stage_events=evs, gate_prep=gprep)

    for _ in range(args.warmup):
        flush.zero_()
        step(None)
    torch.cuda.synchronize(dev)
    st = capi.moe_get_device_status()
    if st != 0:
        raise RuntimeError("device status after warm-up: " + capi.moe_status_string(st))

    # Timed region 1 (the headline number): one event pair per step around the
    # whole forward.  No events between the stages here: an event record
    # between two kernels stops the next one from launching early
    # (programmatic dependent launch), which costs ~25 us at decode.
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    dist_barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    for s in range(args.steps):
        flush.zero_()
        pairs[s][0].record(stream)
        step(None)
        pairs[s][1].record(stream)
    torch.cuda.synchronize(dev)
    dist_barrier()
    step_ms = [a.elapsed_time(b) for a, b in pairs]
    for _ in range(clock_window_steps(statistics.mean(step_ms), args.steps)):
        flush.zero_()
        step(None)
    torch.cuda.synchronize(dev)
    ck = clocks.stop()
    ms_local = statistics.mean(step_ms)
    ms = dist_max(ms_local, dev)
    value = world * w.T / (ms / 1e3)

    # Timed region 2 (the breakdown): the same steps with an event between
    # every two stages; gives each kernel's duration, the dominant kernel's
    # roofline numbers, and the step time with stage events.
    events = [new_events() for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    dist_barrier()
    torch.cuda.synchronize(dev)
    for s in range(args.steps):
        flush.zero_()
        step(events[s])
    torch.cuda.synchronize(dev)
    dist_barrier()
    st = capi.moe_get_device_status()
    if st != 0:
        raise RuntimeError("device status after timed steps: " + capi.moe_status_string(st))
    staged_ms = statistics.mean(events[s][0].elapsed_time(events[s][nst]) for s in range(args.steps))
    stage_ms = {name: statistics.mean(events[s][i].elapsed_time(events[s][i + 1]) for s in range(args.steps))
                for i, name in enumerate(capi.STAGES)}

    # ---- end to end through the public API with host buffers (pinned), every
    # step's copy in and copy out inside the timed region.  Headline: a serving
    # loop of K steps whose copies overlap the neighbouring steps' kernels
    # (layer.PipelinedForward: two copy streams, two device slots), timed from
    # before the first copy-in to after the last copy-out.  Beside it, steps
    # the host waits for one at a time (a decode loop): eager calls, and the
    # forward replayed as a CUDA graph (layer.GraphedForward).
    x_host = x.cpu().pin_memory()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def eager_e2e():
        x.copy_(x_host, non_blocking=True)
        step(None)
        out_host.copy_(out, non_blocking=True)

    graphed = layer.GraphedForward(x_host, gw, pk, w.k, gate_bias=bias, gate_prep=gprep)

    def time_e2e(run):
        for _ in range(2):
            run()
        torch.cuda.synchronize(dev)
        ms_ = []
        for s in range(args.steps):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            run()
            b.record(stream)
            b.synchronize()
            ms_.append(a.elapsed_time(b))
        return dist_max(statistics.mean(ms_), dev)

    e2e_eager_ms = time_e2e(eager_e2e)
    e2e_graph_ms = time_e2e(graphed.replay)
    if not torch.equal(graphed.out_host, out_host):
        raise RuntimeError("graphed and eager steps disagree")
    del graphed

    pipe = layer.PipelinedForward(w.T, w.d, gw, pk, w.k, gate_bias=bias, stream=stream, gate_prep=gprep)
    pipe_out = torch.empty_like(out_host).pin_memory()
    for _ in range(2):
        pipe.step(x_host, pipe_out)
    pipe.join()
    torch.cuda.synchronize(dev)
    dist_barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    pipe.h2d.wait_stream(stream)
    pipe.d2h.wait_stream(stream)
    for s in range(args.steps):
        pipe.step(x_host, pipe_out)
    pipe.join()
    b.record(stream)
    b.synchronize()
    e2e_pipe_ms = dist_max(a.elapsed_time(b) / args.steps, dev)
    if not torch.equal(pipe_out, out_host):
        raise RuntimeError("pipelined and eager steps disagree")
    del pipe
    e2e_v = world * w.T / (e2e_pipe_ms / 1e3)
    e2e_eager_v = world * w.T / (e2e_eager_ms / 1e3)
    e2e_graph_v = world * w.T / (e2e_graph_ms / 1e3)

    # ---- roofline of the dominant kernel and of the layer
    total, off, strides = capi.moe_workspace_layout(w.T, w.d, w.inter, w.E, w.k)
    offs = ws[off[capi.MOE_WS_EXPERT_OFFSETS]:off[capi.MOE_WS_EXPERT_OFFSETS] + 4 * (w.E + 1)].cpu().numpy()
    counts = np.diff(offs.view(np.int32))
    touched = int(np.count_nonzero(counts))
    dom = max(("gemm1", "gemm2"), key=lambda k: stage_ms[k])
    dom_ms = stage_ms[dom]
    fl = gemm_flops(w, dom)
    by = gemm_bytes(w, touched, dom)
    t_f = fl / (fp8_tflops * 1e12)
    t_b = by / (hbm_gbs * 1e9)
    if t_f > t_b:
        peak = fp8_tflops
        roof = {"bound": "tensor", "achieved": fl / (dom_ms / 1e3) / 1e12, "peak": peak, "unit": "TFLOP/s"}
        roof["peak_note"] = "FP8 = %.1f x %s bf16 burst" % (FP8_OVER_BF16, peak_src)
    else:
        peak = hbm_gbs
        roof = {"bound": "hbm", "achieved": by / (dom_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s"}
        roof["peak_note"] = "%s copy bandwidth" % peak_src
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dom
    roof["algorithmic_bytes_per_launch"] = by
    roof["algorithmic_flops_per_launch"] = fl
    roof["traffic"] = profile_traffic(dom, w.name)
    t_roof_us, lbound, lflops, lbytes = layer_roofline(w, touched, hbm_gbs, fp8_tflops)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp8_e4m3 x fp4_e2m1 (fp32 accumulate)",
        "data": "synthetic: seeded normal x / gate_w, N(0,1/fan_in) fp32 expert weights packed to MXFP4 on the GPU",
        "config": config_of(w),
        "roofline": roof,
        "layer": {"roofline_us": t_roof_us, "bound": lbound, "frac": t_roof_us / (ms * 1e3),
                  "weight_GBps": touched * weight_bytes_per_expert(w.d, w.inter) / (ms / 1e3) / 1e9,
                  "TFLOPs": lflops / (ms / 1e3) / 1e12, "touched_experts": touched,
                  "max_expert_load": int(counts.max()), "mean_expert_load": float(counts.mean())},
        "stages_us": {k: v * 1e3 for k, v in stage_ms.items()},
        "ms_per_step_with_stage_events": staged_ms,
        "e2e": {"value": e2e_v, "unit": UNIT, "h2d_bytes_per_step": int(x.numel() * x.element_size()),
                "d2h_bytes_per_step": int(out.numel() * out.element_size()),
                "path": "layer.PipelinedForward: K steps, each copying its tokens in from pinned host memory and "
                        "its output out, the copies on two copy streams overlapping the neighbouring steps' "
                        "kernels; timed from before the first copy-in to after the last copy-out",
                "l2": "not flushed between pipelined steps: the weights read every step (>= 3.4 GB) exceed L2"},
        "e2e_serial": {"value": e2e_eager_v, "unit": UNIT,
                       "path": "the host waits for every step: copy in, capi.moe_forward_ex, copy out (L2 flushed "
                               "before each step)"},
        "e2e_serial_graph": {"value": e2e_graph_v, "unit": UNIT,
                             "path": "as e2e_serial with the forward replayed as one CUDA graph "
                                     "(layer.GraphedForward)"},
        "gpu_launches": kernels_per_step(w) * args.steps,
        "clocks": ck,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, n, cores = oracle_sample(w, x, gw, bias, n_tok=max(1, min(w.T, 2 * os.cpu_count())))
        line["cpu_baseline"] = {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": "%d seeded tokens of the %s workload (oracle time %.1f s)"
                                          % (n, w.name, dt)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_fp8t(args, w):
    """Device time of the FP8 backward-weight conversion on the workload's
    packed W13 and W2 shapes (random packed bytes: the work does not depend on
    them), against the measured HBM bandwidth."""
    import torch
    from fp4_expert_grouped_gb300 import capi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_gbs, _, _, peak_src = measured_peaks()
    for name, N, K in (("W13", 2 * w.inter, w.d), ("W2", w.d, w.inter)):
        g = torch.Generator(device=dev).manual_seed(0)
        fp4 = torch.randint(0, 256, (w.E, N, K // 2), dtype=torch.uint8, device=dev, generator=g)
        sc = torch.randint(110, 135, (w.E, N, K // 32), dtype=torch.uint8, device=dev, generator=g)
        w8t = torch.empty((w.E, K, N), dtype=torch.uint8, device=dev)
        s8t = torch.empty((w.E, K // 128, N // 128), dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            capi.moe_fp4_to_fp8t(fp4, sc, w8t, s8t)
        torch.cuda.synchronize(dev)
        ms = []
        for _ in range(args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            capi.moe_fp4_to_fp8t(fp4, sc, w8t, s8t)
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        st = capi.moe_get_device_status()
        if st != 0:
            raise RuntimeError("device status: " + capi.moe_status_string(st))
        t = statistics.median(ms)
        byts = w.E * N * K // 2 + w.E * N * K // 32 + w.E * K * N + w.E * (K // 128) * (N // 128)
        gbs = byts / t / 1e6
        print(json.dumps({"metric": "moe_fp4_to_fp8t throughput", "matrix": name, "E": w.E, "N": N, "K": K,
                          "ms": t, "bytes": byts, "value": gbs, "unit": "GB/s",
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s",
                                       "peak_note": peak_src, "frac": gbs / hbm_gbs}}), flush=True)
        del fp4, sc, w8t, s8t
        torch.cuda.empty_cache()


def run_dgrad(args, w):
    """Device time of moe_backward_h on workload w: the forward runs once (keeping
    g and u), W2 is converted to its FP8 backward weights, then K timed calls
    (CUDA events, L2 flushed before each) of the three kernels: block-exponent
    scale image, dy dispatch + E4M3, and the grouped FP8 GEMM with the SwiGLU
    backward.  Roofline: 2 P d I FLOPs per call at the FP8 peak."""
    from fp4_expert_grouped_gb300 import capi, inputs, layer
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm_gbs, bf16_tflops, _, peak_src = measured_peaks()
    fp8_tflops = bf16_tflops * FP8_OVER_BF16
    x, gw, bias = inputs.make_x_gate(w, dev)
    pk = layer.pack_workload(w, dev)
    ws = layer.workspace(w.T, w.d, w.inter, w.E, w.k, dev)
    gu = torch.empty((w.P, 2 * w.inter), dtype=torch.float32, device=dev)
    layer.forward(x, gw, pk, w.k, gate_bias=bias, ws=ws, gu_out=gu)
    w8 = torch.empty((w.E, w.inter, w.d), dtype=torch.uint8, device=dev)
    s8 = torch.empty((w.E, w.inter // 128, w.d // 128), dtype=torch.uint8, device=dev)
    capi.moe_fp4_to_fp8t(pk.w2_fp4, pk.w2_scale, w8, s8)
    g = torch.Generator(device=dev).manual_seed(w.seed + 7)
    dout = torch.randn((w.T, w.d), device=dev, generator=g).to(torch.bfloat16)
    dgu = torch.empty((w.P, 2 * w.inter), dtype=torch.uint8, device=dev)
    dgs = torch.empty((w.P, 2 * w.inter // 128), dtype=torch.uint8, device=dev)
    bws = torch.empty(capi.moe_backward_h_workspace_size(w.T, w.d, w.inter, w.E, w.k), dtype=torch.uint8,
                      device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        capi.moe_backward_h(dout, w8, s8, gu, ws, dgu, dgs, w.k, workspace=bws)
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        capi.moe_backward_h(dout, w8, s8, gu, ws, dgu, dgs, w.k, workspace=bws)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    st = capi.moe_get_device_status()
    if st != 0:
        raise RuntimeError("device status: " + capi.moe_status_string(st))

    def report(metric, t, flops):
        tf = flops / (t / 1e3) / 1e12
        print(json.dumps({"metric": metric, "config": config_of(w), "ms": t, "flops": flops, "value": tf,
                          "unit": "TFLOP/s",
                          "roofline": {"bound": "tensor", "achieved": tf, "peak": fp8_tflops, "unit": "TFLOP/s",
                                       "peak_note": "FP8 = %.1f x %s bf16 burst" % (FP8_OVER_BF16, peak_src),
                                       "frac": tf / fp8_tflops}}), flush=True)

    report("moe_backward_h throughput (dh = W2^T dy + SwiGLU backward, FP8)", statistics.median(ms),
           2.0 * w.P * w.d * w.inter)

    # the second dgrad GEMM: dx = sum over slots of W13^T [dg; du]
    del w8, s8
    w8x = torch.empty((w.E, w.d, 2 * w.inter), dtype=torch.uint8, device=dev)
    s8x = torch.empty((w.E, w.d // 128, 2 * w.inter // 128), dtype=torch.uint8, device=dev)
    capi.moe_fp4_to_fp8t(pk.w13_fp4, pk.w13_scale, w8x, s8x)
    dx = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=dev)
    xws = torch.empty(capi.moe_backward_x_workspace_size(w.T, w.d, w.inter, w.E, w.k), dtype=torch.uint8,
                      device=dev)
    for _ in range(args.warmup):
        capi.moe_backward_x(dgu, dgs, w8x, s8x, ws, dx, w.k, workspace=xws)
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        capi.moe_backward_x(dgu, dgs, w8x, s8x, ws, dx, w.k, workspace=xws)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    st = capi.moe_get_device_status()
    if st != 0:
        raise RuntimeError("device status: " + capi.moe_status_string(st))
    report("moe_backward_x throughput (dx = W13^T [dg; du] summed over slots, FP8)", statistics.median(ms),
           4.0 * w.P * w.d * w.inter)

    # the master weights' gradients: dW2 = sum dy (x) h, dW13 = sum [dg; du] (x) x per expert (bf16 tensor
    # cores on the dequantised operands, fp32 out); bound by writing the fp32 gradients
    del w8x, s8x, xws
    dW13 = torch.empty((w.E, 2 * w.inter, w.d), dtype=torch.float32, device=dev)
    dW2 = torch.empty((w.E, w.d, w.inter), dtype=torch.float32, device=dev)
    wws = torch.empty(capi.moe_backward_w_workspace_size(w.T, w.d, w.inter, w.E, w.k), dtype=torch.uint8,
                      device=dev)
    for _ in range(args.warmup):
        capi.moe_backward_w(ws, bws, dgu, dgs, dW13, dW2, w.k, workspace=wws)
    torch.cuda.synchronize(dev)
    ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        capi.moe_backward_w(ws, bws, dgu, dgs, dW13, dW2, w.k, workspace=wws)
        b.record()
        b.synchronize()
        ms.append(a.elapsed_time(b))
    st = capi.moe_get_device_status()
    if st != 0:
        raise RuntimeError("device status: " + capi.moe_status_string(st))
    t = statistics.median(ms)
    flops = 6.0 * w.P * w.d * w.inter
    # algorithmic bytes: the fp32 gradients written, the E4M3 operands read once (dy, h, [dg; du] per pair,
    # x per token with its scales)
    by = 4.0 * w.E * 3 * w.d * w.inter + w.P * (w.d + w.inter + 2 * w.inter) + w.T * w.d
    print(json.dumps({"metric": "moe_backward_w throughput (dW2, dW13 over each expert's pairs)",
                      "config": config_of(w), "ms": t, "flops": flops, "bytes": by,
                      "value": by / (t / 1e3) / 1e9, "unit": "GB/s",
                      "roofline": {"bound": "hbm", "achieved": by / (t / 1e3) / 1e9, "peak": hbm_gbs, "unit": "GB/s",
                                   "peak_note": "%s copy bandwidth" % peak_src,
                                   "frac": by / (t / 1e3) / 1e9 / hbm_gbs},
                      "tflops_bf16": flops / (t / 1e3) / 1e12}), flush=True)


def main():
    args = parse()
    from fp4_expert_grouped_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    if args.tokens or args.experts:
        import dataclasses
        T = args.tokens or w.T
        E = args.experts or w.E
        w = dataclasses.replace(w, name="%s[T=%d,E=%d]" % (w.name, T, E), T=T, E=E)
    if args.fp8t:
        run_fp8t(args, w)
        return
    if args.dgrad:
        run_dgrad(args, w)
        return
    world, rank, local = dist_setup(want_nccl=(args.impl == "ours"))
    if args.impl == "reference":
        run_reference(args, w, world, rank)
    else:
        run_ours(args, w, world, rank, local)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
