"""The expert-major restatement of the oracle (oracle/by_expert.py) against
the oracle's per-token forward on small layers: the same routing bit for
bit and the same FP64 outputs up to summation order (relative 1e-12).
CPU only."""
import numpy as np
import pytest

from moe_decode_layer_topk_gb300 import synth
from oracle import oracle
from oracle.by_expert import moe_forward_by_expert


def _spec(**kw):
    d = dict(synth.CONFIGS["tiny"].__dict__)
    d.update(name=kw.pop("name", "case"), pool=1 << 30)
    d.update(kw)
    return synth.LayerSpec(**d)


CASES = {
    "nvfp4_softmax": dict(H=256, inter=128, E=16, top_k=4),
    "mxfp4_softmax": dict(H=288, inter=160, E=12, top_k=3, wfmt=synth.MXFP4),
    "nvfp4_sigmoid_bias": dict(H=256, inter=96, E=16, top_k=4, scoring=synth.SIGMOID_BIAS,
                               routed_scaling_factor=2.5),
    "zero_experts": dict(H=256, inter=128, E=16, top_k=4, scoring=synth.SOFTMAX_BIAS,
                         zero_experts=8),
    "shared_ungated": dict(H=256, inter=96, E=16, top_k=4, scoring=synth.SIGMOID_BIAS,
                           routed_scaling_factor=2.5, shared_inter=64),
    "shared_gated": dict(H=256, inter=128, E=24, top_k=6, shared_inter=96, shared_gated=True),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_by_expert_matches_the_per_token_oracle(case):
    spec = _spec(name=case, **CASES[case])
    host = synth.make_layer(spec, seed=4242)
    if host.gate_s2 is not None:   # exercise per-expert scale2
        host.gate_s2[:] = np.linspace(0.5, 2.0, spec.E, dtype=np.float32)
        host.down_s2[:] = np.linspace(1.5, 0.75, spec.E, dtype=np.float32)
    x = synth.make_tokens(spec, 9, seed=4343)
    ref = oracle.moe_forward(host, x)
    got = moe_forward_by_expert(host, x)
    assert np.array_equal(got["idx"], ref["idx"])
    assert np.array_equal(got["w"], ref["w"])
    scale = np.abs(ref["out_f64"]).max()
    assert scale > 0
    assert np.abs(got["out_f64"] - ref["out_f64"]).max() <= 1e-12 * scale


def test_by_expert_refuses_other_expert_formats():
    spec = _spec(name="bf16", H=256, inter=128, E=8, top_k=2, wfmt=synth.BF16)
    host = synth.make_layer(spec, seed=1)
    with pytest.raises(ValueError):
        moe_forward_by_expert(host, synth.make_tokens(spec, 2, seed=2))
