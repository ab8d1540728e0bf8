"""Convenience layer over the C ABI: packed expert weights and a forward call.

Everything numeric runs in libfp4moe.so; this module only allocates device
tensors with PyTorch and passes pointers (see capi.py).
"""
from dataclasses import dataclass
from typing import Optional

import torch

from . import capi, inputs


@dataclass
class PackedExperts:
    w13_fp4: torch.Tensor     # uint8 [E, 2*inter, d/2]
    w13_scale: torch.Tensor   # uint8 [E, 2*inter, d/32]
    w2_fp4: torch.Tensor      # uint8 [E, d, inter/2]
    w2_scale: torch.Tensor    # uint8 [E, d, inter/32]

    @property
    def nbytes(self) -> int:
        return sum(t.numel() for t in (self.w13_fp4, self.w13_scale, self.w2_fp4, self.w2_scale))


def empty_packed(E: int, d: int, inter: int, device="cuda") -> PackedExperts:
    u8 = dict(dtype=torch.uint8, device=device)
    return PackedExperts(torch.empty((E, 2 * inter, d // 2), **u8), torch.empty((E, 2 * inter, d // 32), **u8),
                         torch.empty((E, d, inter // 2), **u8), torch.empty((E, d, inter // 32), **u8))


def pack_experts(w13: torch.Tensor, w2: torch.Tensor) -> PackedExperts:
    """Pack fp32 device weights W13 [E, 2I, d] and W2 [E, d, I] with moe_pack_fp4."""
    E, twoI, d = w13.shape
    pk = empty_packed(E, d, twoI // 2, w13.device)
    capi.moe_pack_fp4(w13.contiguous(), pk.w13_fp4, pk.w13_scale)
    capi.moe_pack_fp4(w2.contiguous(), pk.w2_fp4, pk.w2_scale)
    return pk


def pack_workload(w: inputs.Workload, device="cuda", gen_device=None) -> PackedExperts:
    """Generate every expert of a workload (one at a time, on `gen_device`) and
    pack it on `device`.  Peak extra memory: one expert's fp32 weights."""
    gen_device = device if gen_device is None else gen_device
    pk = empty_packed(w.E, w.d, w.inter, device)
    for e in range(w.E):
        w13, w2 = inputs.make_expert(w, e, gen_device)
        w13 = w13.to(device)
        w2 = w2.to(device)
        capi.moe_pack_fp4(w13, pk.w13_fp4[e], pk.w13_scale[e])
        capi.moe_pack_fp4(w2, pk.w2_fp4[e], pk.w2_scale[e])
    return pk


def workspace(T: int, d: int, inter: int, E: int, k: int, device="cuda") -> torch.Tensor:
    n = capi.moe_workspace_size(T, d, inter, E, k)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def prepare_gate(gate_w: torch.Tensor) -> torch.Tensor:
    """gate_w's form for the tensor-core gate (moe_prepare_gate), once per gate_w."""
    d, E = gate_w.shape
    prep = torch.empty(max(capi.moe_gate_prep_size(d, E), 256), dtype=torch.uint8, device=gate_w.device)
    capi.moe_prepare_gate(gate_w, prep)
    return prep


def forward(x: torch.Tensor, gate_w: torch.Tensor, pk: PackedExperts, k: int,
            gate_bias: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
            out: Optional[torch.Tensor] = None, stream=None, routing: bool = False,
            gu_out: Optional[torch.Tensor] = None, gate_prep: Optional[torch.Tensor] = None):
    """out bf16 [T, d] = MoE layer forward of bf16 x [T, d] (device tensors).
    With routing=True also returns (topk_idx, topk_w, pair_pos).  gu_out (fp32
    [T*k, 2*inter]) keeps GEMM1's g and u for the backward (moe_backward_h)."""
    T, d = x.shape
    if out is None:
        out = torch.empty_like(x)
    ti = tw = pp = None
    if routing:
        ti = torch.empty((T, k), dtype=torch.int32, device=x.device)
        tw = torch.empty((T, k), dtype=torch.float32, device=x.device)
        pp = torch.empty((T * k,), dtype=torch.int32, device=x.device)
    capi.moe_forward_ex(x, gate_w, pk.w13_fp4, pk.w13_scale, pk.w2_fp4, pk.w2_scale, out, k,
                        stream=stream, gate_bias=gate_bias, workspace=ws,
                        topk_idx_out=ti, topk_w_out=tw, pair_pos_out=pp, gu_out=gu_out, gate_prep=gate_prep)
    if routing:
        return out, ti, tw, pp
    return out


class GraphedForward:
    """A serving step whose forward is captured once as a CUDA graph and
    replayed per step: copy the step's tokens in from pinned host memory,
    replay the forward, copy the output back to pinned host memory.

    The captured work is exactly that of ``forward`` (the same kernels, with
    programmatic dependent launch between them kept as graph edges), on
    device buffers owned by this object.  Replaying costs the host one graph
    launch instead of the argument marshalling and the per-kernel launches of
    an eager call, which matters when every step waits for its result (a
    decode loop).  The two copies are issued around the replay rather than
    captured: with them inside the graph, a step of 16384 tokens of width
    7168 (235 MB each way) took 12.3 ms against 7.65 ms for the same eager
    copies.  Inputs are read from ``x_host`` at replay time: write the next
    step's tokens into it, then call ``replay``; ``out_host`` holds the
    result once the stream reaches the end of the replay.
    """

    def __init__(self, x_host: torch.Tensor, gate_w: torch.Tensor, pk: PackedExperts, k: int,
                 gate_bias: Optional[torch.Tensor] = None, out_host: Optional[torch.Tensor] = None,
                 gate_prep: Optional[torch.Tensor] = None):
        if not x_host.is_pinned():
            raise ValueError("x_host must be pinned host memory")
        dev = gate_w.device
        T, d = x_host.shape
        E = gate_w.shape[1]
        inter = pk.w13_fp4.shape[1] // 2
        self.x_host = x_host
        self.out_host = out_host if out_host is not None else torch.empty_like(x_host).pin_memory()
        if not self.out_host.is_pinned() or self.out_host.shape != x_host.shape:
            raise ValueError("out_host must be pinned host memory shaped like x_host")
        self.x = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev)
        self.out = torch.empty_like(self.x)
        self.ws = workspace(T, d, inter, E, k, dev)
        self._args = (gate_w, pk, k, gate_bias, gate_prep)
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self.x.copy_(self.x_host, non_blocking=True)
            self._forward()                   # eager once: kernel attributes set outside the capture
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="thread_local"):
            self._forward()

    def _forward(self):
        gate_w, pk, k, gate_bias, gate_prep = self._args
        capi.moe_forward_ex(self.x, gate_w, pk.w13_fp4, pk.w13_scale, pk.w2_fp4, pk.w2_scale, self.out, k,
                            gate_bias=gate_bias, workspace=self.ws, gate_prep=gate_prep)

    def replay(self):
        """Enqueue one step on the current stream."""
        self.x.copy_(self.x_host, non_blocking=True)
        self.graph.replay()
        self.out_host.copy_(self.out, non_blocking=True)


class PipelinedForward:
    """Consecutive serving steps with their host copies overlapped with the
    layer's kernels: step i's tokens are copied in on one copy stream while
    step i-1's forward runs, and its output is copied out on a second copy
    stream while step i+1's forward runs.  ``depth`` device slots of x and out
    alternate; one workspace serves every step, because the forwards run one
    after another on the compute stream.  Events order each slot's reuse: a
    slot's next copy-in waits for the forward that read it, and its next
    forward for the copy-out that read its output.

    ``step(x_host, out_host)`` enqueues one step and returns the event that
    completes once ``out_host`` holds the result; ``x_host`` may be rewritten
    once the step's copy-in is done (``in_event``).  Both must be pinned.
    """

    def __init__(self, T: int, d: int, gate_w: torch.Tensor, pk: PackedExperts, k: int,
                 gate_bias: Optional[torch.Tensor] = None, depth: int = 2, stream=None,
                 gate_prep: Optional[torch.Tensor] = None):
        if depth < 1:
            raise ValueError("depth must be at least 1")
        dev = gate_w.device
        E = gate_w.shape[1]
        inter = pk.w13_fp4.shape[1] // 2
        self.depth = depth
        self.x = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        self.out = [torch.empty((T, d), dtype=torch.bfloat16, device=dev) for _ in range(depth)]
        self.ws = workspace(T, d, inter, E, k, dev)
        self.compute = stream if stream is not None else torch.cuda.current_stream(dev)
        self.h2d = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        self.in_done = [torch.cuda.Event() for _ in range(depth)]
        self.fwd_done = [torch.cuda.Event() for _ in range(depth)]
        self.out_done = [torch.cuda.Event() for _ in range(depth)]
        self._used = [False] * depth
        self._args = (gate_w, pk, k, gate_bias, gate_prep)
        self.i = 0
        self.in_event = None

    def step(self, x_host: torch.Tensor, out_host: torch.Tensor) -> torch.cuda.Event:
        if not (x_host.is_pinned() and out_host.is_pinned()):
            raise ValueError("x_host and out_host must be pinned host memory")
        gate_w, pk, k, gate_bias, gate_prep = self._args
        s = self.i % self.depth
        if self._used[s]:
            self.h2d.wait_event(self.fwd_done[s])          # the forward that read x[s] is done
        with torch.cuda.stream(self.h2d):
            self.x[s].copy_(x_host, non_blocking=True)
            self.in_done[s].record(self.h2d)
        self.compute.wait_event(self.in_done[s])
        if self._used[s]:
            self.compute.wait_event(self.out_done[s])      # the copy-out that read out[s] is done
        capi.moe_forward_ex(self.x[s], gate_w, pk.w13_fp4, pk.w13_scale, pk.w2_fp4, pk.w2_scale, self.out[s], k,
                            stream=self.compute, gate_bias=gate_bias, workspace=self.ws, gate_prep=gate_prep)
        self.fwd_done[s].record(self.compute)
        self.d2h.wait_event(self.fwd_done[s])
        with torch.cuda.stream(self.d2h):
            out_host.copy_(self.out[s], non_blocking=True)
            self.out_done[s].record(self.d2h)
        self._used[s] = True
        self.in_event = self.in_done[s]
        self.i += 1
        return self.out_done[s]

    def join(self):
        """Make the compute stream wait for every copy enqueued so far."""
        self.compute.wait_stream(self.h2d)
        self.compute.wait_stream(self.d2h)
