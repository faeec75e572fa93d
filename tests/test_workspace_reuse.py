"""One workspace through a sequence of calls of different layers, token
counts and paths, each checked against the FP64 oracle.

The fused kernels keep no per-call clearing of their cross-CTA words: every
such word carries the call's tag, and a word left by an earlier call of any
shape never carries the current one.  The output accumulator is zeroed and
released by each call itself.  Fresh-workspace parity tests cannot show a
fault in either; this sequence reuses one workspace across:

- two stream-kernel layers, one with a gated shared expert and one MXFP4;
- token counts that grow and shrink;
- route-only calls on both fused kernels;
- decode-kernel calls in between (a BF16 layer, and N = 12);
- on the Qwen3-shaped layer, the stream kernel and the grouped chain
  alternating, forwards and route-only calls.

Indices must match bit for bit, BF16 outputs within 1e-2*max|ref| + 2^-8.
"""
import numpy as np
import pytest

from moe_decode_layer_topk_gb300 import synth

NV, MX, BF = synth.NVFP4, synth.MXFP4, synth.BF16

LAYERS = {
    "nvfp4": dict(H=256, inter=128, E=16, top_k=4),
    "nvfp4_gated_shared": dict(H=160, inter=96, E=13, top_k=3, shared_inter=64, shared_gated=True),
    "mxfp4": dict(H=192, inter=160, E=9, top_k=2, wfmt=MX),
    "bf16_decode_path": dict(H=256, inter=128, E=16, top_k=4, wfmt=BF),
}

# (layer, N, forward or route-only)
SEQUENCE = [("nvfp4", 3, "fwd"), ("nvfp4", 1, "fwd"), ("nvfp4_gated_shared", 5, "fwd"),
            ("mxfp4", 8, "fwd"), ("nvfp4", 3, "route"), ("bf16_decode_path", 2, "fwd"),
            ("nvfp4", 2, "fwd"), ("nvfp4_gated_shared", 1, "fwd"), ("mxfp4", 4, "fwd"),
            ("nvfp4", 8, "fwd"), ("nvfp4", 8, "fwd"),
            # the decode kernel: route-only then forward, and N = 12 FP4 calls
            ("bf16_decode_path", 3, "route"), ("bf16_decode_path", 2, "fwd"),
            ("nvfp4", 12, "fwd"), ("nvfp4", 12, "route"), ("nvfp4", 12, "fwd"),
            ("nvfp4", 4, "fwd")]


@pytest.mark.gpu
def test_one_workspace_through_mixed_calls():
    import torch

    from moe_decode_layer_topk_gb300 import _lib
    from moe_decode_layer_topk_gb300.device import DeviceLayer, bf16_tensor
    from oracle import compare, margin, oracle

    from .gpu_util import run_forward, spec_from

    hosts, devs = {}, {}
    for i, (name, kw) in enumerate(LAYERS.items()):
        spec = spec_from("tiny", name=name, **kw)
        hosts[name] = synth.make_layer(spec, seed=9100 + i)
        devs[name] = DeviceLayer.upload(hosts[name])
    n = max(_lib.moe_workspace_size(d.desc, 16) for d in devs.values())
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    _lib.moe_workspace_init(ws)
    paths = set()
    for step, (name, N, kind) in enumerate(SEQUENCE):
        host, dev = hosts[name], devs[name]
        x = margin.tokens_with_margin(host, N, seed=9200 + step)
        ref = oracle.moe_forward(host, x)
        keys = margin.selection_keys(host, x)
        paths.add(_lib.moe_uses_grouped_path(dev.desc, N))
        if kind == "route":
            idx = torch.full((N, dev.spec.top_k), -1, dtype=torch.int32, device="cuda")
            w = torch.full((N, dev.spec.top_k), float("nan"), dtype=torch.float32, device="cuda")
            _lib.moe_route(dev.desc, dev.weights, bf16_tensor(x), idx, w, ws)
            torch.cuda.synchronize()
            assert _lib.moe_get_error(ws) == _lib.MOE_OK
            compare.check_routing(idx.cpu().numpy(), w.cpu().numpy(), ref["idx"], ref["w"], keys)
            continue
        out, idx, w = run_forward(dev, x, ws=ws)
        compare.check_routing(idx, w, ref["idx"], ref["w"], keys)
        compare.check_output(out, ref["out_f64"])
    assert paths == {0}   # the fused kernels throughout (stream and decode)


# the Qwen3-shaped layer: the stream kernel (N <= 8) and the grouped chain
# (N >= 9) alternating on one workspace, forwards and route-only calls
SEQUENCE_QWEN3 = [(4, "fwd"), (16, "fwd"), (2, "route"), (3, "fwd"), (12, "route"), (1, "fwd"),
                  (9, "fwd"), (8, "fwd")]


@pytest.mark.gpu
def test_one_workspace_across_stream_and_grouped_paths():
    import torch

    from moe_decode_layer_topk_gb300 import _lib
    from moe_decode_layer_topk_gb300.device import bf16_tensor
    from oracle import compare, margin, oracle

    from .gpu_util import full_layer, run_forward

    host, dev = full_layer("qwen3_30b_a3b")
    ws = torch.empty(_lib.moe_workspace_size(dev.desc, 16), dtype=torch.uint8, device="cuda")
    _lib.moe_workspace_init(ws)
    paths = set()
    for step, (N, kind) in enumerate(SEQUENCE_QWEN3):
        x = margin.tokens_with_margin(host, N, seed=9300 + step)
        ref = oracle.moe_forward(host, x)
        keys = margin.selection_keys(host, x)
        paths.add(_lib.moe_uses_grouped_path(dev.desc, N))
        if kind == "route":
            idx = torch.full((N, dev.spec.top_k), -1, dtype=torch.int32, device="cuda")
            w = torch.full((N, dev.spec.top_k), float("nan"), dtype=torch.float32, device="cuda")
            _lib.moe_route(dev.desc, dev.weights, bf16_tensor(x), idx, w, ws)
            torch.cuda.synchronize()
            assert _lib.moe_get_error(ws) == _lib.MOE_OK
            compare.check_routing(idx.cpu().numpy(), w.cpu().numpy(), ref["idx"], ref["w"], keys)
            continue
        out, idx, w = run_forward(dev, x, ws=ws)
        compare.check_routing(idx, w, ref["idx"], ref["w"], keys)
        compare.check_output(out, ref["out_f64"])
    assert paths == {0, 1}   # both the fused kernel and the grouped chain ran
