"""Token rows with a routing margin (test infrastructure only).

Parity compares routed expert indices bit for bit, so every token used in a
parity case must have a clear gap between its k-th and (k+1)-th selection key:
at least ``MARGIN`` (1e-3).  The key is the router logit for softmax routing
(softmax is monotone in the logit, so the order is the logit order) and
sigmoid(logit) + bias for sigmoid routing.  A row that falls short is redrawn
from its next sub-seed (synth.x_row attempt + 1).  The keys come from the FP64
oracle; the GPU never influences the inputs.
"""
from __future__ import annotations

import numpy as np

from moe_decode_layer_topk_gb300 import synth
from . import oracle

MARGIN = 1e-3
# softmax + bias keys are probabilities of about 1/(E + Z): the gap is taken
# relative to the largest key (still far above the GPU's FP32 error)
MARGIN_REL_SOFTMAX_BIAS = 1e-3


def selection_keys(layer, x: np.ndarray) -> np.ndarray:
    sp = layer.spec
    logits = oracle.layer_router_logits(layer, x)
    if sp.scoring == synth.SOFTMAX:
        return logits
    _, _, sel = oracle.route(logits, sp.top_k, sp.scoring, sp.norm_topk_prob,
                             sp.routed_scaling_factor, layer.bias)
    return sel


def margin_for(layer, keys_row: np.ndarray) -> float:
    if layer.spec.scoring == synth.SOFTMAX_BIAS:
        return MARGIN_REL_SOFTMAX_BIAS * float(np.max(np.abs(keys_row)))
    return MARGIN


def topk_gap(keys_row: np.ndarray, k: int) -> float:
    s = np.sort(keys_row)[::-1]
    return float(s[k - 1] - s[k]) if k < s.size else float("inf")


def tokens_with_margin(layer, N: int, seed=None, max_attempts: int = 2000) -> np.ndarray:
    """x [N, H] BF16 bits, each row redrawn until its top-k gap >= MARGIN."""
    sp = layer.spec
    seed = (synth.base_seed(sp) + N) if seed is None else seed
    rows = []
    for n in range(N):
        for attempt in range(max_attempts):
            r = synth.x_row(sp, seed, n, attempt)[None, :]
            keys = selection_keys(layer, r)[0]
            if topk_gap(keys, sp.top_k) >= margin_for(layer, keys):
                rows.append(r[0])
                break
        else:
            raise RuntimeError(f"no row with a top-k margin after {max_attempts} draws")
    if not rows:
        return np.zeros((0, sp.H), dtype=np.uint16)
    return np.stack(rows)
