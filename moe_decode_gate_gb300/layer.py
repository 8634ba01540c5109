"""A device-resident MoE decode layer: weights + workspace + the C-ABI call."""
from __future__ import annotations

import torch

from ._native import wd_moe_decode, wd_moe_workspace_init, wd_moe_workspace_size


def _to_device_u8(a, device):
    t = a if isinstance(a, torch.Tensor) else torch.from_numpy(a)
    if t.dtype != torch.uint8:
        t = t.view(torch.uint8)
    return t.to(device, non_blocking=False).contiguous()


class MoEDecodeLayer:
    """One MoE layer's MXFP8 expert weights held on the GPU.

    gate_up uint8 [E, 2I, H] (E4M3 codes; rows [0, I) gate, [I, 2I) up),
    gate_up_scale uint8 [E, 2I, H/32] (E8M0), down uint8 [E, H, I],
    down_scale uint8 [E, H, I/32].  The workspace is sized for ``max_batch``
    tokens and serves any smaller batch.
    """

    def __init__(self, gate_up, gate_up_scale, down, down_scale, K, max_batch=32, device="cuda"):
        self.device = torch.device(device)
        self.gate_up = _to_device_u8(gate_up, self.device)
        self.gate_up_scale = _to_device_u8(gate_up_scale, self.device)
        self.down = _to_device_u8(down, self.device)
        self.down_scale = _to_device_u8(down_scale, self.device)
        self.E, I2, self.H = self.gate_up.shape
        self.I = I2 // 2
        self.K = K
        self.max_batch = max_batch
        self.workspace = torch.empty(wd_moe_workspace_size(max_batch, K, self.I), dtype=torch.uint8,
                                     device=self.device)
        wd_moe_workspace_init(self.workspace)

    def weight_bytes(self) -> int:
        return sum(t.numel() for t in (self.gate_up, self.gate_up_scale, self.down, self.down_scale))

    def __call__(self, x, topk_ids, topk_w, out=None, stream=None):
        """x bf16 [B, H], topk_ids int32 [B, K], topk_w fp32 [B, K] -> out bf16 [B, H]."""
        if x.shape[0] > self.max_batch:
            raise ValueError(f"batch {x.shape[0]} exceeds max_batch {self.max_batch}")
        if out is None:
            out = torch.empty_like(x)
        wd_moe_decode(x, topk_ids, topk_w, self.gate_up, self.gate_up_scale, self.down,
                      self.down_scale, out, self.workspace, stream=stream)
        return out
