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


def forward(x: torch.Tensor, gate_w: torch.Tensor, pk: PackedExperts, k: int,
            gate_bias: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
            out: Optional[torch.Tensor] = None, stream=None, routing: bool = False):
    """out bf16 [T, d] = MoE layer forward of bf16 x [T, d] (device tensors).
    With routing=True also returns (topk_idx, topk_w, pair_pos)."""
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
                        topk_idx_out=ti, topk_w_out=tw, pair_pos_out=pp)
    if routing:
        return out, ti, tw, pp
    return out
