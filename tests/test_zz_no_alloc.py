"""moe_forward_noalloc: the layer forward for callers that cannot allocate
device memory (no workspace argument; the library's built-in device scratch
is used instead).  Its results must match moe_forward with a caller
workspace.  This file is collected after the parity files so a
stop-at-first-failure run has already run them; it builds everything it needs
itself, so it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest

from moe_decode_layer_topk_gb300 import _lib, synth


@pytest.fixture(scope="module")
def lib():
    from moe_decode_layer_topk_gb300 import build
    build.build()
    return _lib.load()


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    """Host-side refusal, before any CUDA call: 64 tokens of a layer with
    H 7168, inter 16384, top-4 need more than the 8 MiB built-in scratch."""
    d = _lib.LayerDesc()
    d.H, d.inter, d.E, d.top_k = 7168, 16384, 256, 4
    d.scoring, d.norm_topk_prob, d.routed_scaling_factor = 0, 1, 1.0
    d.wfmt, d.shared_inter = 0, 0
    assert _lib.moe_workspace_size(d, 64) > 8 << 20
    w = _lib.Weights()
    for i, (name, _) in enumerate(_lib.Weights._fields_):
        setattr(w, name, (1 << 20) + 256 * i)
    w.bias = w.sh_gate = w.sh_up = w.sh_down = w.sh_gate_w = None
    st = lib.moe_forward_noalloc(ctypes.byref(d), ctypes.byref(w), 1 << 24, 64, 1 << 25,
                                 None, None, None)
    assert st == _lib.MOE_ERR_WORKSPACE_TOO_SMALL


def _spec(**kw):
    base = dict(synth.CONFIGS["tiny"].__dict__)
    base.update(pool=64, **kw)
    return synth.LayerSpec(**base)


def _compare_call(spec, host, dev, N, seed, what):
    """One moe_forward_noalloc call against moe_forward on a fresh caller
    workspace (same routing bit for bit, outputs within the tolerance) and
    against the FP64 oracle."""
    import torch
    from moe_decode_layer_topk_gb300.device import bf16_tensor, workspace
    from oracle import compare, margin, oracle

    xb = margin.tokens_with_margin(host, N, seed=seed)
    x = bf16_tensor(xb)
    ref_out = torch.empty_like(x)
    ref_idx = torch.empty((N, spec.top_k), dtype=torch.int32, device="cuda")
    ref_w = torch.empty((N, spec.top_k), dtype=torch.float32, device="cuda")
    ws = workspace(spec, N)
    _lib.moe_forward(dev.desc, dev.weights, x, ref_out, ws, ref_idx, ref_w)
    out = torch.full_like(x, float("nan"))
    idx = torch.full((N, spec.top_k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((N, spec.top_k), float("nan"), dtype=torch.float32, device="cuda")
    _lib.moe_forward_noalloc(dev.desc, dev.weights, x, out, idx, w)
    torch.cuda.synchronize()
    assert _lib.moe_get_error(ws) == _lib.MOE_OK
    assert _lib.moe_get_error(None) == _lib.MOE_OK      # the built-in scratch's error word
    assert torch.equal(idx, ref_idx), what
    torch.testing.assert_close(w, ref_w, rtol=1e-6, atol=1e-7)
    bits = out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = compare.bf16_bits_to_f64(ref_out.view(torch.int16).cpu().numpy().view(np.uint16))
    compare.check_output(bits, ref, what=f"{what} vs moe_forward")
    orc = oracle.moe_forward(host, xb)
    compare.check_routing(idx.cpu().numpy(), w.cpu().numpy(), orc["idx"], orc["w"],
                          margin.selection_keys(host, xb))
    compare.check_output(bits, orc["out_f64"], what=f"{what} vs oracle")


@pytest.mark.gpu
def test_noalloc_matches_moe_forward_on_two_calls_in_a_row(lib):
    from moe_decode_layer_topk_gb300.device import DeviceLayer

    spec = _spec(name="noalloc", H=512, inter=256, E=16, top_k=4, shared_inter=128,
                 shared_gated=True)
    host = synth.make_layer(spec, seed=4242)
    dev = DeviceLayer.upload(host)
    for call, N in enumerate((4, 3)):           # two calls in a row, different batches
        _compare_call(spec, host, dev, N, 5000 + call, f"noalloc call {call}")


@pytest.mark.gpu
def test_noalloc_switches_between_the_paths_in_one_array(lib):
    """The one built-in array serves the grouped path (N*k > 256), the
    fused kernel for up to 8 rows and the fused kernel for more rows, one call
    after another; stale state of one layout must not leak into the next."""
    from moe_decode_layer_topk_gb300.device import DeviceLayer

    spec = _spec(name="noalloc_paths", H=256, inter=128, E=16, top_k=8)
    host = synth.make_layer(spec, seed=4343)
    dev = DeviceLayer.upload(host)
    d = dev.desc
    assert _lib.moe_uses_grouped_path(d, 40) == 1 and _lib.moe_uses_grouped_path(d, 3) == 0
    assert _lib.moe_workspace_size(d, 40) < 8 << 20
    for call, N in enumerate((40, 3, 12, 2, 40)):
        _compare_call(spec, host, dev, N, 5100 + call, f"noalloc path call {call} (N={N})")
