"""Device-side containers for one MoE layer: host arrays in storage form -> torch CUDA tensors.

Only data movement lives here (host -> device copies, workspace allocation); all
arithmetic of the block runs in the CUDA library.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional

import numpy as np
import torch

from . import MoEQ4, MoEShape, make_shape, moe_workspace_size


def to_device(a: Optional[np.ndarray], device, pin: bool = False) -> Optional[torch.Tensor]:
    """numpy array -> torch tensor; uint16 arrays are bf16 bit patterns and become torch.bfloat16."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    if device == "cpu":
        return t.pin_memory() if pin else t.clone()
    return t.to(device)


def bf16_tensor_bits(t: torch.Tensor) -> np.ndarray:
    """torch bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclasses.dataclass
class DeviceLayer:
    shape: MoEShape
    x: torch.Tensor
    w_router: torch.Tensor
    b_router: Optional[torch.Tensor]
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor
    q4: Optional[MoEQ4]
    scales: tuple

    @property
    def T(self):
        return self.shape.T

    def out_dtype(self):
        return torch.float32 if self.shape.act_dtype == 0 else torch.bfloat16

    def new_workspace(self) -> torch.Tensor:
        ws = torch.zeros(moe_workspace_size(self.shape), dtype=torch.uint8, device=self.x.device)
        assert ws.data_ptr() % 256 == 0
        return ws


def upload(inp, device="cuda") -> DeviceLayer:
    """Copy one layer's storage-form arrays (x, router, experts, q4 scales) to the device."""
    shape = make_shape(inp.T, inp.H, inp.E, inp.k, inp.I, inp.act, inp.w, inp.norm_topk, inp.q_block)
    d = lambda a: to_device(a, device)
    q4 = None
    scales = ()
    if inp.w == "q4":
        scales = (d(inp.gate_scales), d(inp.up_scales), d(inp.down_scales))
        q4 = MoEQ4(scales[0].data_ptr(), scales[1].data_ptr(), scales[2].data_ptr(),
                   (ctypes.c_float * 16)(*[float(v) for v in inp.codebook]))
    return DeviceLayer(shape, d(inp.x), d(inp.w_router), d(inp.b_router), d(inp.w_gate), d(inp.w_up),
                       d(inp.w_down), q4, scales)
