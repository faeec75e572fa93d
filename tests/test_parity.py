"""GPU path vs the FP64 oracle, element by element, through the C ABI.

Small cases use shapes that span several 32-row groups, several K chunks and
a ragged token tail (N not a multiple of the 4-token batch), both scale
layouts, both formats and every routing / shared-expert variant; the
full-size cases are the five layer shapes at their token counts, in the same
launch configuration the benchmark times.  Indices must match bit for bit,
BF16 outputs within 1e-2*max|ref| + 2^-8.
"""
import numpy as np
import pytest

from moe_decode_layer_topk_gb300 import synth
from moe_decode_layer_topk_gb300.device import DeviceLayer
from oracle import compare, margin, oracle

from .gpu_util import full_layer, record_headroom, run_forward, spec_from

NV, MX, BF, F8 = synth.NVFP4, synth.MXFP4, synth.BF16, synth.FP8
SM, SB, SMB = synth.SOFTMAX, synth.SIGMOID_BIAS, synth.SOFTMAX_BIAS

SMALL = {
    "tiny": (dict(), 1),
    "block_scales_ragged": (dict(H=160, inter=96, E=13, top_k=3), 5),
    "block_scales_gated_shared": (dict(H=160, inter=96, E=13, top_k=3, shared_inter=64,
                                       shared_gated=True), 5),
    "per_row_scales_5_chunks": (dict(H=1280, inter=256, E=16, top_k=4), 3),
    "mxfp4_block_scales": (dict(H=192, inter=160, E=9, top_k=2, wfmt=MX), 6),
    "mxfp4_per_row_scales": (dict(H=1024, inter=512, E=8, top_k=2, wfmt=MX), 2),
    "mxfp4_shared": (dict(H=2880 // 5, inter=2880 // 9, E=12, top_k=4, wfmt=MX,
                          shared_inter=96, shared_gated=True), 4),
    "sigmoid_bias_ungated_shared": (dict(H=256, inter=128, E=32, top_k=4, scoring=SB,
                                         routed_scaling_factor=2.5, shared_inter=96), 4),
    "sigmoid_bias_no_norm": (dict(H=256, inter=128, E=32, top_k=3, scoring=SB,
                                  norm_topk_prob=False, routed_scaling_factor=1.7), 3),
    "softmax_no_norm": (dict(H=256, inter=128, E=16, top_k=3, norm_topk_prob=False), 3),
    "single_expert": (dict(E=1, top_k=1), 2),
    "k_equals_E": (dict(E=4, top_k=4), 3),
    "max_slots_k32": (dict(H=128, inter=64, E=64, top_k=32), 8),
    "max_experts_1024": (dict(H=64, inter=32, E=1024, top_k=4), 3),
    "n64_sweep_shape": (dict(H=128, inter=64, E=32, top_k=4), 64),
    "zero_routed_weight": (dict(H=256, inter=128, E=8, top_k=2, scoring=SB,
                                routed_scaling_factor=0.0, shared_inter=64, shared_gated=True), 3),
    # BF16 routed experts: 3D boxes, 2D boxes with a partial last box, several
    # gate/up and down chunks, shared expert, sigmoid routing
    "bf16_experts": (dict(H=256, inter=128, E=16, top_k=4, wfmt=BF), 5),
    "bf16_experts_2d_boxes": (dict(H=160, inter=96, E=13, top_k=3, wfmt=BF), 5),
    "bf16_experts_5_chunks_gated_shared": (dict(H=1280, inter=256, E=16, top_k=4, wfmt=BF,
                                                shared_inter=96, shared_gated=True), 3),
    "bf16_experts_down_3_chunks": (dict(H=256, inter=640, E=8, top_k=2, wfmt=BF), 2),
    "bf16_experts_sigmoid_shared": (dict(H=256, inter=128, E=32, top_k=4, scoring=SB,
                                         routed_scaling_factor=2.5, wfmt=BF, shared_inter=96), 4),
    # FP8 block-scaled routed experts: several 128-row and 128-column scale
    # blocks, ragged blocks, 2D boxes, several chunks, shared expert, sigmoid
    "fp8_experts": (dict(H=256, inter=256, E=16, top_k=4, wfmt=F8), 5),
    "fp8_experts_ragged_blocks": (dict(H=160, inter=160, E=13, top_k=3, wfmt=F8), 5),
    "fp8_experts_4_chunks_gated_shared": (dict(H=2048, inter=384, E=16, top_k=4, wfmt=F8,
                                               shared_inter=96, shared_gated=True), 3),
    "fp8_experts_down_3_chunks": (dict(H=256, inter=1152, E=8, top_k=2, wfmt=F8), 2),
    "fp8_experts_sigmoid": (dict(H=512, inter=256, E=32, top_k=4, scoring=SB,
                                 routed_scaling_factor=2.5, wfmt=F8), 4),
    # NVFP4-quantised router (softmax and sigmoid routing, with other expert formats)
    "nvfp4_router": (dict(H=256, inter=128, E=16, top_k=4, router_fmt=NV), 5),
    "nvfp4_router_sigmoid_shared": (dict(H=320, inter=96, E=32, top_k=3, scoring=SB,
                                         routed_scaling_factor=2.5, shared_inter=64,
                                         router_fmt=NV), 4),
    "nvfp4_router_fp8_experts": (dict(H=512, inter=256, E=24, top_k=4, wfmt=F8,
                                      router_fmt=NV), 3),
    # softmax + correction bias, with and without zero experts
    "softmax_bias": (dict(H=256, inter=128, E=16, top_k=4, scoring=SMB,
                          routed_scaling_factor=1.5), 3),
    "zero_experts": (dict(H=256, inter=128, E=16, top_k=4, scoring=SMB, zero_experts=8), 5),
    "zero_experts_gated_shared": (dict(H=320, inter=96, E=32, top_k=6, scoring=SMB,
                                       zero_experts=16, shared_inter=64, shared_gated=True,
                                       routed_scaling_factor=2.0), 4),
    "zero_experts_width_1024": (dict(H=64, inter=32, E=768, top_k=4, scoring=SMB,
                                     zero_experts=256), 3),
}


def _check(host, dev, x):
    ref = oracle.moe_forward(host, x)
    out, idx, w = run_forward(dev, x)
    keys = margin.selection_keys(host, x)
    compare.check_routing(idx, w, ref["idx"], ref["w"], keys)
    return compare.check_output(out, ref["out_f64"])


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(SMALL))
def test_small_case(case):
    kw, N = SMALL[case]
    spec = spec_from("tiny", name=case, **kw)
    host = synth.make_layer(spec, seed=7000 + len(case))
    dev = DeviceLayer.upload(host)
    x = margin.tokens_with_margin(host, N, seed=8000 + len(case))
    _check(host, dev, x)


@pytest.mark.gpu
def test_many_tokens_on_one_expert():
    """Identical rows route every token to the same experts: each expert gets
    N = 9 tokens, i.e. three 4-token weight passes (ragged last pass)."""
    spec = spec_from("tiny", name="same_rows", H=256, inter=128, E=8, top_k=2,
                     shared_inter=64, shared_gated=True)
    host = synth.make_layer(spec, seed=11)
    dev = DeviceLayer.upload(host)
    x1 = margin.tokens_with_margin(host, 1, seed=12)
    x = np.repeat(x1, 9, axis=0)
    _check(host, dev, x)


@pytest.mark.gpu
def test_zero_down_codes_gives_shared_alone():
    spec = spec_from("tiny", name="zero_down", H=256, inter=128, E=8, top_k=2, shared_inter=64)
    host = synth.make_layer(spec, seed=13)
    host.down_q[:] = 0
    dev = DeviceLayer.upload(host)
    x = margin.tokens_with_margin(host, 2, seed=14)
    _check(host, dev, x)


@pytest.mark.gpu
def test_zero_experts_take_every_slot():
    """Zero experts pulled in by their bias for every slot: no routed expert
    runs, the output is the shared expert alone (and the routing outputs hold
    the zero-expert indices >= E)."""
    spec = spec_from("tiny", name="all_zero", H=256, inter=128, E=8, top_k=3, scoring=SMB,
                     zero_experts=4, shared_inter=64, shared_gated=True)
    host = synth.make_layer(spec, seed=19)
    host.bias[8:] = 10.0
    dev = DeviceLayer.upload(host)
    x = margin.tokens_with_margin(host, 3, seed=20)
    _check(host, dev, x)
    _, idx, _ = run_forward(dev, x)
    assert np.all(idx >= 8)


HASHED = {
    "hash_softmax": (dict(H=256, inter=128, E=16, top_k=4, hash_vocab=50), 5),
    "hash_sigmoid_shared": (dict(H=320, inter=96, E=32, top_k=3, scoring=SB,
                                 routed_scaling_factor=2.5, shared_inter=64, hash_vocab=1000), 4),
    "hash_softmax_no_norm_fp8": (dict(H=512, inter=256, E=24, top_k=2, wfmt=F8,
                                      norm_topk_prob=False, hash_vocab=7), 6),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(HASHED))
def test_hash_routing(case):
    """Hash routing through moe_forward_ids: experts from the tid2eid row of
    each token id (repeated ids included), weights by the layer's scoring."""
    kw, N = HASHED[case]
    spec = spec_from("tiny", name=case, **kw)
    host = synth.make_layer(spec, seed=7300 + len(case))
    dev = DeviceLayer.upload(host)
    x = synth.make_tokens(spec, N, seed=7400 + len(case))
    ids = np.random.default_rng(7500 + len(case)).integers(0, spec.hash_vocab, N).astype(np.int32)
    ids[-1] = ids[0]
    ref = oracle.moe_forward(host, x, token_ids=ids)
    out, idx, w = run_forward(dev, x, token_ids=ids)
    np.testing.assert_array_equal(idx, ref["idx"])          # table order, bit for bit
    np.testing.assert_allclose(w, ref["w"], rtol=1e-4, atol=1e-6)
    compare.check_output(out, ref["out_f64"])


@pytest.mark.gpu
def test_scale2_is_applied():
    spec = spec_from("tiny", name="scale2", H=256, inter=128, E=8, top_k=2)
    host = synth.make_layer(spec, seed=15)
    rng = np.random.default_rng(16)
    host.gate_s2[:] = rng.uniform(0.5, 2, 8).astype(np.float32)
    host.up_s2[:] = rng.uniform(0.5, 2, 8).astype(np.float32)
    host.down_s2[:] = rng.uniform(0.5, 2, 8).astype(np.float32)
    dev = DeviceLayer.upload(host)
    x = margin.tokens_with_margin(host, 3, seed=17)
    _check(host, dev, x)


FULL = [(name, N) for name in ("tiny", "qwen3_30b_a3b", "mtp_verify", "deepseek_v3", "gpt_oss_120b",
                               "qwen3_30b_a3b_bf16", "qwen3_30b_a3b_fp8", "qwen3_30b_a3b_nvfp4_router",
                               "qwen3_30b_a3b_zero_experts")
        for N in synth.CONFIGS[name].tokens if N <= 64]
# single-token calls of the shared-expert layers: at N = 1 the stream kernel
# prefetches token 0's gate/up tiles into L2 for every layer size (57 KB
# bursts of 16 rows on the DeepSeek-V3 shape)
FULL += [("mtp_verify", 1), ("deepseek_v3", 1)]


@pytest.mark.gpu
@pytest.mark.parametrize("name,N", FULL)
def test_full_size(name, N):
    host, dev = full_layer(name)
    x = margin.tokens_with_margin(host, N)
    err, tol = _check(host, dev, x)
    record_headroom(name, N, err, tol)
