"""Device-resident copies of a layer's input bytes (torch CUDA tensors) and the
matching C-ABI descriptor/weight structs.  Plumbing only: uploads bytes and
takes pointers; no arithmetic of the layer happens here.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import _lib
from .synth import (BF16, FP8, HostLayer, LayerSpec, MXFP4, NVFP4, SIGMOID_BIAS, SOFTMAX,
                    SOFTMAX_BIAS)


def layer_desc(spec: LayerSpec) -> _lib.LayerDesc:
    d = _lib.LayerDesc()
    d.H, d.inter, d.E, d.top_k = spec.H, spec.inter, spec.E, spec.top_k
    d.scoring = {SOFTMAX: _lib.MOE_SCORE_SOFTMAX, SIGMOID_BIAS: _lib.MOE_SCORE_SIGMOID_BIAS,
                 SOFTMAX_BIAS: _lib.MOE_SCORE_SOFTMAX_BIAS}[spec.scoring]
    d.norm_topk_prob = int(spec.norm_topk_prob)
    d.routed_scaling_factor = float(spec.routed_scaling_factor)
    d.wfmt = {NVFP4: _lib.MOE_W_NVFP4, MXFP4: _lib.MOE_W_MXFP4, BF16: _lib.MOE_W_BF16,
              FP8: _lib.MOE_W_FP8}[spec.wfmt]
    d.shared_inter = spec.shared_inter
    d.router_fmt = _lib.MOE_R_NVFP4 if spec.router_fmt == NVFP4 else _lib.MOE_R_BF16
    d.zero_experts = spec.zero_experts
    d.hash_vocab = spec.hash_vocab
    return d


def to_device(a: Optional[np.ndarray], device="cuda") -> Optional[torch.Tensor]:
    """numpy array -> contiguous CUDA tensor with the same bytes (uint16 -> int16 view)."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    else:
        t = torch.from_numpy(a)
    return t.to(device, non_blocking=False)


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """BF16 bit pattern array -> torch.bfloat16 tensor on `device`."""
    return to_device(bits, device).view(torch.bfloat16)


@dataclasses.dataclass
class DeviceLayer:
    spec: LayerSpec
    tensors: dict
    desc: _lib.LayerDesc
    weights: _lib.Weights

    @staticmethod
    def upload(host: HostLayer, device="cuda") -> "DeviceLayer":
        ts = {k: to_device(v, device) for k, v in host.tensors().items()}
        return DeviceLayer.from_tensors(host.spec, ts)

    @staticmethod
    def from_tensors(spec: LayerSpec, ts: dict) -> "DeviceLayer":
        w = _lib.Weights()
        for name, _ in _lib.Weights._fields_:
            t = ts.get(name)
            setattr(w, name, None if t is None else t.data_ptr())
        return DeviceLayer(spec, ts, layer_desc(spec), w)

    def clone(self) -> "DeviceLayer":
        """A second copy of every tensor at new device addresses."""
        ts = {k: (None if v is None else v.clone()) for k, v in self.tensors.items()}
        return DeviceLayer.from_tensors(self.spec, ts)

    def nbytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.tensors.values() if v is not None)


def workspace(spec: LayerSpec, max_tokens: int, host_staging: bool = False,
              device="cuda") -> torch.Tensor:
    """Zero-initialised workspace (uint8 tensor) for up to max_tokens rows."""
    d = layer_desc(spec)
    n = _lib.moe_workspace_size(d, max_tokens)
    if n == 0:
        raise ValueError("invalid layer descriptor")
    if host_staging:
        n += _lib.moe_host_staging_size(d, max_tokens)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    _lib.moe_workspace_init(ws)
    return ws
