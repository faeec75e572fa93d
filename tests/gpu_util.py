"""Shared plumbing of the GPU tests: build/upload layers, run the C-ABI path,
fetch results as numpy."""
import functools

import numpy as np
import torch

from moe_decode_layer_topk_gb300 import _lib, synth
from moe_decode_layer_topk_gb300.device import DeviceLayer, bf16_tensor, workspace


def spec_from(base: str = "tiny", **kw) -> synth.LayerSpec:
    d = dict(synth.CONFIGS[base].__dict__)
    d.update(name=kw.pop("name", "case"), pool=kw.pop("pool", 1 << 30))
    d.update(kw)
    return synth.LayerSpec(**d)


@functools.lru_cache(maxsize=4)
def full_layer(name: str):
    """Host + device copy of one of the five full-size layers (cached)."""
    spec = synth.CONFIGS[name]
    host = synth.make_layer(spec)
    return host, DeviceLayer.upload(host)


def run_forward(dev: DeviceLayer, x_bits: np.ndarray, ws=None, token_ids=None):
    spec = dev.spec
    N = x_bits.shape[0]
    x = bf16_tensor(x_bits)
    out = torch.empty_like(x)
    idx = torch.full((N, spec.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((N, spec.top_k), float("nan"), dtype=torch.float32, device="cuda")
    ws = workspace(spec, N) if ws is None else ws
    if token_ids is None:
        _lib.moe_forward(dev.desc, dev.weights, x, out, ws, idx, w)
    else:
        tid = torch.from_numpy(np.ascontiguousarray(token_ids, dtype=np.int32)).cuda()
        _lib.moe_forward_ids(dev.desc, dev.weights, x, tid, out, ws, idx, w)
    torch.cuda.synchronize()
    assert _lib.moe_get_error(ws) == _lib.MOE_OK
    return (out.view(torch.int16).cpu().numpy().view(np.uint16), idx.cpu().numpy(),
            w.cpu().numpy())


def record_headroom(name: str, N: int, err: float, tol: float, path: str = None):
    """Append one parity case's max|err| and tolerance as a JSON line to the
    file named by MOE_PARITY_HEADROOM (nothing when it is unset)."""
    import json
    import os
    path = path or os.environ.get("MOE_PARITY_HEADROOM")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"case": name, "N": int(N), "max_err": float(err), "tol": float(tol),
                            "ratio": float(err) / float(tol)}) + "\n")
