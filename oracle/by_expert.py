"""Expert-major restatement of the oracle's layer forward, for token counts
where the per-token loop of oracle.moe_forward is too slow (gpt-oss shape at
N = 512: minutes).

TEST INFRASTRUCTURE ONLY: used by the test suite, never by the library.

The definition is the one oracle.moe_forward computes (the forward chain's
steps: router logits, top-k routing, per selected expert
y = Dq(Wd) (SiLU(Dq(Wg) x) * (Dq(Wu) x)), routing-weighted sum), with the
tokens of one expert taken together: each expert's projections are
dequantised once by the oracle (oracle_dequant, FP64) and applied to its
tokens with FP64 matrix products (numpy), so every token's result is the
same sum of the same FP64 products as in the per-token loop, in another
order.  Routing comes from the oracle (router logits + route).  A shared
expert (BF16) is added the same way over all tokens, times its gate
sigmoid(w_s . x) when the layer has a gate vector.  Hash-routed layers are
not taken here.
"""
from __future__ import annotations

import concurrent.futures
import os

import numpy as np

from . import oracle


def _bf16_rows(x_bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact: the upper half of an f32)."""
    u = np.ascontiguousarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def moe_forward_by_expert(layer, x: np.ndarray) -> dict:
    """-> dict(out_f64 [N, H], idx [N, k], w [N, k]) for a synth.HostLayer
    with FP4 routed experts (zero experts allowed: they add nothing)."""
    sp = layer.spec
    if sp.hash_vocab or sp.wfmt not in ("nvfp4", "mxfp4"):
        raise ValueError("by-expert oracle: FP4 experts, no hash routing")
    x = np.ascontiguousarray(x, dtype=np.uint16)
    N, H = x.shape
    logits = oracle.layer_router_logits(layer, x)
    idx, w, _ = oracle.route(logits, sp.top_k, sp.scoring, sp.norm_topk_prob,
                             sp.routed_scaling_factor, layer.bias)
    xf = _bf16_rows(x)
    out = np.zeros((N, H), dtype=np.float64)
    s2 = lambda a, e: 1.0 if a is None else float(a[e])

    def one(e):
        rows, slots = np.nonzero(idx == e)
        wg = oracle.dequant(layer.gate_q[e], layer.gate_s[e], s2(layer.gate_s2, e), sp.wfmt)
        wu = oracle.dequant(layer.up_q[e], layer.up_s[e], s2(layer.up_s2, e), sp.wfmt)
        wd = oracle.dequant(layer.down_q[e], layer.down_s[e], s2(layer.down_s2, e), sp.wfmt)
        xe = xf[rows]
        g = xe @ wg.T
        u = xe @ wu.T
        a = g / (1.0 + np.exp(-g)) * u
        return rows, w[rows, slots][:, None] * (a @ wd.T)

    # experts in parallel (the C dequantiser and numpy release the GIL); the
    # sums into `out` are taken in expert order
    experts = [int(e) for e in np.unique(idx[idx < sp.E])]
    with concurrent.futures.ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        for rows, part in ex.map(one, experts):
            out[rows] += part
    if sp.shared_inter:
        g = xf @ _bf16_rows(layer.sh_gate).T
        u = xf @ _bf16_rows(layer.sh_up).T
        sh = (g / (1.0 + np.exp(-g)) * u) @ _bf16_rows(layer.sh_down).T
        gate = np.ones(N)
        if layer.sh_gate_w is not None:
            d = xf @ _bf16_rows(layer.sh_gate_w)
            gate = 1.0 / (1.0 + np.exp(-d))
        out += gate[:, None] * sh
    return {"out_f64": out, "idx": idx, "w": w}
