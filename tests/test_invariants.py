"""Invariants of the GPU path that hold whatever the weights are.

- A batch of N tokens routes every token exactly as N one-token calls do and
  gives the same outputs within the tolerance (the only coupling between the
  tokens of a call is the shared power-of-two exponent of h within an expert's
  token batch).
- Renumbering the experts (router rows, bias and every expert table permuted
  together) renumbers the routing and leaves the output bit for bit the same.
- moe_forward captured in a CUDA graph and replayed on new token rows gives
  the eager call's bits.
"""
import numpy as np
import pytest
import torch

from moe_decode_layer_topk_gb300 import _lib, synth
from moe_decode_layer_topk_gb300.device import DeviceLayer, bf16_tensor, workspace
from oracle import compare, margin, oracle

from .gpu_util import run_forward, spec_from


def _layer(seed, **kw):
    spec = spec_from("tiny", name="inv", **kw)
    host = synth.make_layer(spec, seed=seed)
    return host, DeviceLayer.upload(host)


@pytest.mark.gpu
@pytest.mark.parametrize("kw", [dict(H=512, inter=256, E=16, top_k=4),
                                dict(H=256, inter=128, E=8, top_k=2, shared_inter=64,
                                     shared_gated=True, wfmt=synth.MXFP4)])
def test_batch_equals_single_token_calls(kw):
    host, dev = _layer(31, **kw)
    x = margin.tokens_with_margin(host, 4, seed=32)
    out, idx, w = run_forward(dev, x)
    ref = oracle.moe_forward(host, x)
    for n in range(4):
        o1, i1, w1 = run_forward(dev, x[n:n + 1])
        np.testing.assert_array_equal(i1[0], idx[n])
        np.testing.assert_allclose(w1[0], w[n], rtol=1e-6, atol=1e-7)
        compare.check_output(o1, ref["out_f64"][n:n + 1], what=f"token {n} alone")
    compare.check_output(out, ref["out_f64"], what="batch")


@pytest.mark.gpu
def test_expert_renumbering():
    import dataclasses
    host, dev = _layer(33, H=256, inter=128, E=12, top_k=3, scoring=synth.SIGMOID_BIAS,
                       routed_scaling_factor=2.0)
    perm = np.random.default_rng(34).permutation(12)     # new expert i = old expert perm[i]
    inv = np.argsort(perm)
    tables = {k: getattr(host, k) for k in ("router", "bias", "gate_q", "up_q", "down_q",
                                            "gate_s", "up_s", "down_s", "gate_s2", "up_s2",
                                            "down_s2")}
    hostp = dataclasses.replace(host, **{k: (None if v is None else v[perm].copy())
                                         for k, v in tables.items()})
    devp = DeviceLayer.upload(hostp)
    x = margin.tokens_with_margin(host, 4, seed=35)
    out, idx, w = run_forward(dev, x)
    outp, idxp, wp = run_forward(devp, x)
    np.testing.assert_array_equal(inv[idx], idxp)
    np.testing.assert_array_equal(w, wp)
    np.testing.assert_array_equal(out, outp)


@pytest.mark.gpu
def test_graph_capture_replays_the_eager_call():
    host, dev = _layer(36, H=512, inter=256, E=16, top_k=4, shared_inter=64)
    spec = host.spec
    xa = bf16_tensor(synth.make_tokens(spec, 3, seed=37))
    xb = bf16_tensor(synth.make_tokens(spec, 3, seed=38))
    ws = workspace(spec, 3)
    eager = []
    for x in (xa, xb):
        o = torch.empty_like(x)
        _lib.moe_forward(dev.desc, dev.weights, x, o, ws)
        eager.append(o.clone())
    xin = xa.clone()
    out = torch.empty_like(xin)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        _lib.moe_forward(dev.desc, dev.weights, xin, out, ws, stream=stream)
    for x, ref in zip((xa, xb, xa), (eager[0], eager[1], eager[0])):
        xin.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert _lib.moe_get_error(ws) == _lib.MOE_OK
