"""Convenience wrappers over the C ABI: resident layer weights and a layer
object that owns a plan. Argument marshalling only."""
from __future__ import annotations

from typing import Any, Optional

import numpy as np

from . import _abi

_DT = {"f32": _abi.MOE_DTYPE_F32, "bf16": _abi.MOE_DTYPE_BF16}


def _to_torch(a: np.ndarray, device, torch):
    """numpy storage array -> device tensor with the same bytes.
    uint32 -> int32, uint16 (bf16 bits) -> bfloat16, uint8 -> uint8 (6-bit
    down codes), float32 -> float32."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(device)
    if a.dtype == np.uint8:
        return torch.from_numpy(a).to(device)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    if a.dtype == np.float32:
        return torch.from_numpy(a).to(device)
    raise TypeError(a.dtype)


class DeviceLayer:
    """One MoE layer's weights resident on a CUDA device.

    router_w: [E, D] float32 or bf16; router_bias: [E] float32 or None;
    planes: the nine quantised arrays (see include/moe_decode.h)."""

    def __init__(self, router_w, router_bias, planes: dict, E: int, top_k: int, D: int, Dff: int):
        self.router_w = router_w
        self.router_bias = router_bias
        self.planes = planes
        self.E, self.top_k, self.D, self.Dff = E, top_k, D, Dff
        self.c_planes = _abi.make_planes(planes)

    @classmethod
    def from_host(cls, router_w_storage: np.ndarray, router_bias: Optional[np.ndarray], planes: Any,
                  top_k: int, device="cuda"):
        import torch
        arrs = {f: _to_torch(getattr(planes, f), device, torch) for f in _abi.PLANE_FIELDS}
        rw = _to_torch(router_w_storage, device, torch)
        rb = None if router_bias is None else _to_torch(router_bias.astype(np.float32), device, torch)
        E, Dff, D8 = arrs["gate_q"].shape
        return cls(rw, rb, arrs, E, top_k, D8 * 8, Dff)

    @property
    def plane_bytes_per_expert(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.planes.values()) // self.E


class MoeDecodeLayer:
    """Owns one plan (workspace sized for max_tokens) on the current device."""

    def __init__(self, E: int, top_k: int, D: int, Dff: int, max_tokens: int = 64,
                 act_dtype: str = "bf16", out_dtype: Optional[str] = None, flags: int = 0,
                 mma_min_tokens: int = 0, activation: int = _abi.MOE_ACT_SWIGLU,
                 act_limit: float = 0.0, down_bits: int = 0, experts=None):
        """experts: (begin, end) of the experts this plan owns (an expert-parallel
        shard), or None for all of them."""
        eb, ee = (0, 0) if experts is None else (int(experts[0]), int(experts[1]))
        self.cfg = _abi.make_config(E, top_k, D, Dff, max_tokens, x_dtype=_DT[act_dtype],
                                    router_dtype=_DT[act_dtype],
                                    out_dtype=_DT[out_dtype or act_dtype], flags=flags,
                                    mma_min_tokens=mma_min_tokens, activation=activation,
                                    act_limit=act_limit, down_bits=down_bits,
                                    expert_begin=eb, expert_end=ee)
        self.act_dtype = act_dtype
        self.out_dtype = out_dtype or act_dtype
        self.plan = _abi.moe_plan_create(self.cfg)

    def _out_torch_dtype(self):
        import torch
        return torch.float32 if self.out_dtype == "f32" else torch.bfloat16

    def forward(self, x, w: DeviceLayer, out=None, stream=None):
        import torch
        n = x.shape[0]
        if out is None:
            out = torch.empty((n, w.D), dtype=self._out_torch_dtype(), device=x.device)
        _abi.moe_decode_forward(self.plan, x, w.router_w, w.router_bias, w.c_planes, n,
                                self.cfg.top_k, out, stream)
        return out

    def forward_layers(self, steps, stream=None):
        """steps: sequence of (x, DeviceLayer, out), run in order as one chain
        (moe_decode_forward_layers); returns the outs."""
        _abi.moe_decode_forward_layers(
            self.plan, [(x, w.router_w, w.router_bias, w.c_planes, out) for x, w, out in steps],
            steps[0][0].shape[0], self.cfg.top_k, stream)
        return [out for _, _, out in steps]

    def forward_host(self, x_host, w: DeviceLayer, out_host, stream=None):
        n = x_host.shape[0]
        _abi.moe_decode_forward_host(self.plan, x_host, w.router_w, w.router_bias, w.c_planes, n,
                                     self.cfg.top_k, out_host, stream)
        return out_host

    def routing(self, n_tokens: int):
        return _abi.moe_get_routing(self.plan, n_tokens, self.cfg.E, self.cfg.top_k)

    def check(self):
        _abi.moe_plan_check(self.plan)

    def close(self):
        if getattr(self, "plan", None):
            _abi.moe_plan_free(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
