"""The switch between the fused kernels and the grouped chain on a full-size
layer.  The Qwen3-30B-A3B-shaped NVFP4 layer (2.65 MB experts) runs the
stream kernel up to 8 token rows and the grouped chain from 9 on (the
measured crossing); with the tuning hook's pair threshold at 128 it runs the
decode kernel below 128 (token, slot) pairs.  Each case is checked against
the FP64 oracle (indices bit for bit, BF16 outputs within
1e-2*max|ref| + 2^-8), with the library's own report of the path taken.
Collected last, so a stop-at-first-failure run has already run every other
test."""
import pytest

from moe_decode_layer_topk_gb300 import _lib
from oracle import compare, margin, oracle

from .gpu_util import full_layer, run_forward


def _check(host, dev, N, seed):
    x = margin.tokens_with_margin(host, N, seed=seed)
    out, idx, w = run_forward(dev, x)
    ref = oracle.moe_forward(host, x)
    compare.check_routing(idx, w, ref["idx"], ref["w"], margin.selection_keys(host, x))
    compare.check_output(out, ref["out_f64"])


@pytest.mark.gpu
@pytest.mark.parametrize("N,grouped", [(8, 0), (9, 1), (16, 1), (32, 1)])
def test_qwen3_shape_across_the_switch(N, grouped):
    host, dev = full_layer("qwen3_30b_a3b")
    assert _lib.moe_uses_grouped_path(dev.desc, N) == grouped
    _check(host, dev, N, 4100 + N)


@pytest.mark.gpu
@pytest.mark.parametrize("N,grouped", [(15, 0), (16, 1)])
def test_qwen3_shape_decode_kernel_under_a_pair_threshold(N, grouped):
    host, dev = full_layer("qwen3_30b_a3b")
    try:
        _lib.moe_debug_set_grouped_min_slots(128)
        assert _lib.moe_uses_grouped_path(dev.desc, N) == grouped
        _check(host, dev, N, 4200 + N)
    finally:
        _lib.moe_debug_set_grouped_min_slots(0)
