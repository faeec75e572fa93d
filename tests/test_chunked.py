"""Layers the grouped path does not take (a shared expert, BF16 / FP8 routed
experts, zero experts, hash routing) with N * top_k > 256: moe_forward runs
the fused kernels in row chunks of floor(256 / top_k) tokens.  Each case is
checked against the FP64 oracle (indices bit for bit, weights to 1e-4
relative, BF16 outputs within 1e-2 * max|ref| + 2^-8): small layers against
the per-token oracle, the full-size MTP-verify and DeepSeek-V3 shapes at
N = 64 against the expert-major restatement of the oracle (pinned to the
per-token one on the CPU)."""
import numpy as np
import pytest

from moe_decode_layer_topk_gb300 import _lib, synth
from moe_decode_layer_topk_gb300.device import DeviceLayer
from oracle import compare, margin, oracle
from oracle.by_expert import moe_forward_by_expert

from .gpu_util import full_layer, record_headroom, run_forward, spec_from

SB, SMB, F8, BF = synth.SIGMOID_BIAS, synth.SOFTMAX_BIAS, synth.FP8, synth.BF16

CHUNKED = {
    # N * k > 256 in each case: 2 .. 4 row chunks, a ragged last one
    "shared_gated_nvfp4": (dict(H=256, inter=128, E=16, top_k=8, shared_inter=64,
                                shared_gated=True), 70),
    "bf16_experts": (dict(H=256, inter=128, E=16, top_k=4, wfmt=BF), 100),
    "fp8_experts_sigmoid": (dict(H=256, inter=128, E=16, top_k=4, wfmt=F8, scoring=SB,
                                 routed_scaling_factor=2.5), 90),
    "zero_experts": (dict(H=256, inter=128, E=16, top_k=4, scoring=SMB, zero_experts=8), 130),
}


@pytest.mark.gpu
@pytest.mark.parametrize("case", sorted(CHUNKED))
def test_row_chunks_small(case):
    kw, N = CHUNKED[case]
    spec = spec_from("tiny", name=case, **kw)
    assert N * spec.top_k > 256
    host = synth.make_layer(spec, seed=8100 + len(case))
    dev = DeviceLayer.upload(host)
    assert _lib.moe_uses_grouped_path(dev.desc, N) == 0
    x = margin.tokens_with_margin(host, N, seed=8200 + len(case))
    out, idx, w = run_forward(dev, x)
    ref = oracle.moe_forward(host, x)
    compare.check_routing(idx, w, ref["idx"], ref["w"], margin.selection_keys(host, x))
    compare.check_output(out, ref["out_f64"])


@pytest.mark.gpu
def test_row_chunks_hash_routing():
    spec = spec_from("tiny", name="hash_chunks", H=256, inter=128, E=16, top_k=4, hash_vocab=40)
    host = synth.make_layer(spec, seed=8300)
    dev = DeviceLayer.upload(host)
    N = 150
    x = synth.make_tokens(spec, N, seed=8301)
    ids = np.random.default_rng(8302).integers(0, spec.hash_vocab, N).astype(np.int32)
    ref = oracle.moe_forward(host, x, token_ids=ids)
    out, idx, w = run_forward(dev, x, token_ids=ids)
    np.testing.assert_array_equal(idx, ref["idx"])
    np.testing.assert_allclose(w, ref["w"], rtol=1e-4, atol=1e-6)
    compare.check_output(out, ref["out_f64"])


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["mtp_verify", "deepseek_v3"])
def test_row_chunks_full_size_n64(name):
    host, dev = full_layer(name)
    N = 64
    assert _lib.moe_uses_grouped_path(dev.desc, N) == 0
    x = margin.tokens_with_margin(host, N)
    out, idx, w = run_forward(dev, x)
    ref = moe_forward_by_expert(host, x)
    compare.check_routing(idx, w, ref["idx"], ref["w"], margin.selection_keys(host, x))
    err, tol = compare.check_output(out, ref["out_f64"])
    record_headroom(name, N, err, tol)
