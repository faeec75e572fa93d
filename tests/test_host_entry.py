"""moe_forward_host, the end-to-end call with host activations: x goes to the
device through the workspace's staging area, the forward runs, the result
comes back to host memory.  Checked against the FP64 oracle (indices are not
returned by this call; outputs within 1e-2*max|ref| + 2^-8), reusing one
staging workspace across token counts, on the stream kernel (the
Qwen3-shaped layer at N = 1..4) and on the decode kernel (a small BF16 layer)."""
import numpy as np
import pytest

from moe_decode_layer_topk_gb300 import synth


@pytest.mark.gpu
@pytest.mark.parametrize("layer", ["qwen3_30b_a3b", "small_bf16"])
def test_host_entry_matches_the_oracle(layer):
    import torch

    from moe_decode_layer_topk_gb300 import _lib
    from moe_decode_layer_topk_gb300.device import DeviceLayer, workspace
    from oracle import compare, margin, oracle

    from .gpu_util import full_layer, spec_from

    if layer == "qwen3_30b_a3b":
        host, dev = full_layer(layer)
    else:
        spec = spec_from("tiny", name=layer, H=256, inter=128, E=16, top_k=4, wfmt=synth.BF16)
        host = synth.make_layer(spec, seed=9400)
        dev = DeviceLayer.upload(host)
    ws = workspace(dev.spec, 4, host_staging=True)
    for step, N in enumerate((3, 1, 4, 2)):
        x = margin.tokens_with_margin(host, N, seed=9500 + step)
        x_host = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
        out_host = torch.empty_like(x_host).pin_memory()
        _lib.moe_forward_host(dev.desc, dev.weights, x_host, out_host, ws)
        assert _lib.moe_get_error(ws) == _lib.MOE_OK
        ref = oracle.moe_forward(host, x)
        compare.check_output(out_host.numpy().view(np.uint16), ref["out_f64"])
