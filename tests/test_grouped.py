"""Grouped (many-token) path vs the FP64 oracle, through the C ABI.

When N * top_k exceeds the decode kernel's slot table (or reaches 128 for a
layer whose FP4 experts hold >= 1 MiB each), moe_forward runs the
per-expert token-group GEMMs on the tcgen05 tensor cores.  The small cases
span ragged 128-row weight tiles (32-row tails), a ragged K chunk, experts
with more positions than one 64-position token tile, both formats, both
scoring modes and per-expert scale2; the full-size case is the MXFP4
gpt-oss-shaped layer at N = 512 (routing and all 512 output rows, against the
expert-major restatement of the oracle).  Indices must match bit for bit, BF16 outputs within
1e-2*max|ref| + 2^-8.
"""
import numpy as np
import pytest

from moe_decode_layer_topk_gb300 import synth
from moe_decode_layer_topk_gb300.device import DeviceLayer
from oracle import compare, margin, oracle

from oracle.by_expert import moe_forward_by_expert

from .gpu_util import full_layer, record_headroom, run_forward, spec_from

NV, MX = synth.NVFP4, synth.MXFP4
SB = synth.SIGMOID_BIAS

GROUPED = {
    # two 128-row tiles with a 32-row tail, ~40 positions per expert
    "nvfp4_ragged_rows": (dict(H=256, inter=160, E=8, top_k=2), 160),
    # K = 288 = 2 x 128 + 32 in gate/up: a ragged last K chunk
    "mxfp4_ragged_k": (dict(H=288, inter=128, E=8, top_k=2, wfmt=MX), 200),
    # ~100 positions per expert: two token tiles per expert
    "multi_tile_experts_sigmoid": (dict(H=256, inter=128, E=4, top_k=2, scoring=SB,
                                        routed_scaling_factor=2.5), 200),
    "softmax_no_norm_k3": (dict(H=320, inter=192, E=16, top_k=3, norm_topk_prob=False), 100),
    # every token on the one expert: five token tiles of one expert
    "single_expert_all_tokens": (dict(H=256, inter=128, E=1, top_k=1), 300),
    "mxfp4_many_chunks": (dict(H=1024, inter=384, E=8, top_k=2, wfmt=MX), 160),
    "nvfp4_many_experts": (dict(H=512, inter=256, E=64, top_k=4), 96),
    # NVFP4-quantised router on the grouped router kernel
    "nvfp4_router": (dict(H=256, inter=128, E=16, top_k=4, router_fmt=NV), 100),
    # softmax + correction bias routing on the grouped top-k
    "softmax_bias": (dict(H=256, inter=128, E=16, top_k=4, scoring=synth.SOFTMAX_BIAS,
                          routed_scaling_factor=1.5), 100),
}


def _check(host, dev, x, sample=None):
    out, idx, w = run_forward(dev, x)
    sp = host.spec
    logits = oracle.layer_router_logits(host, x)
    ref_idx, ref_w, _ = oracle.route(logits, sp.top_k, sp.scoring, sp.norm_topk_prob,
                                     sp.routed_scaling_factor, host.bias)
    keys = margin.selection_keys(host, x)
    compare.check_routing(idx, w, ref_idx, ref_w, keys)
    rows = np.arange(x.shape[0]) if sample is None else np.asarray(sample)
    ref = oracle.moe_forward(host, x[rows])
    return compare.check_output(out[rows], ref["out_f64"])


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(GROUPED))
def test_grouped_small(case):
    kw, N = GROUPED[case]
    spec = spec_from("tiny", name=case, **kw)
    assert N * spec.top_k > 256
    host = synth.make_layer(spec, seed=9100 + len(case))
    dev = DeviceLayer.upload(host)
    x = margin.tokens_with_margin(host, N, seed=9200 + len(case))
    _check(host, dev, x)


@pytest.mark.gpu
def test_grouped_scale2_is_applied():
    spec = spec_from("tiny", name="g_scale2", H=256, inter=128, E=8, top_k=2)
    host = synth.make_layer(spec, seed=9301)
    rng = np.random.default_rng(9302)
    for name in ("gate_s2", "up_s2", "down_s2"):
        getattr(host, name)[:] = rng.uniform(0.5, 2, 8).astype(np.float32)
    dev = DeviceLayer.upload(host)
    x = margin.tokens_with_margin(host, 150, seed=9303)
    _check(host, dev, x)


@pytest.mark.gpu
def test_grouped_full_size_gpt_oss_n512():
    """All 512 output rows against the expert-major restatement of the oracle
    (oracle/by_expert.py, pinned to the per-token oracle on the CPU)."""
    host, dev = full_layer("gpt_oss_120b")
    x = margin.tokens_with_margin(host, 512)
    out, idx, w = run_forward(dev, x)
    ref = moe_forward_by_expert(host, x)
    compare.check_routing(idx, w, ref["idx"], ref["w"], margin.selection_keys(host, x))
    err, tol = compare.check_output(out, ref["out_f64"])
    record_headroom("gpt_oss_120b", 512, err, tol)


@pytest.mark.gpu
def test_grouped_matches_decode_path_at_the_boundary():
    """N*k = 256 runs the decode kernel, 257+ the grouped GEMMs: the same
    tokens give the same routing and outputs within the tolerance on both."""
    spec = spec_from("tiny", name="boundary", H=512, inter=256, E=16, top_k=4)
    host = synth.make_layer(spec, seed=9500)
    dev = DeviceLayer.upload(host)
    x = margin.tokens_with_margin(host, 65, seed=9501)
    out_g, idx_g, _ = run_forward(dev, x)            # 65 * 4 = 260 slots: grouped
    out_d, idx_d, _ = run_forward(dev, x[:64])       # 64 * 4 = 256 slots: decode
    for n in range(64):
        assert set(idx_g[n]) == set(idx_d[n])
    ref = oracle.moe_forward(host, x)
    compare.check_output(out_g, ref["out_f64"])
    compare.check_output(out_d, ref["out_f64"][:64])
