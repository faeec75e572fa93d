"""GPU-vs-oracle comparison rules (test infrastructure only).

Output: BF16 values within max |gpu - ref| <= 1e-2 * max|ref| + 2^-8 over the
whole [N, H] output of one call, ref being the oracle's FP64 value before
rounding (the tolerance the method's target states; FP32 accumulation order on
the GPU is not fixed).
Routing: the set of selected experts per token is compared bit for bit, the
weights are matched by expert index (FP32 vs FP64: relative 1e-4), and the
order is compared wherever adjacent selection keys differ by >= 1e-3.
"""
from __future__ import annotations

import numpy as np

ORDER_GAP = 1e-3


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def output_tolerance(ref: np.ndarray) -> float:
    return 1e-2 * float(np.abs(ref).max()) + 2.0 ** -8


def check_output(out_bits: np.ndarray, ref: np.ndarray, what: str = "out"):
    got = bf16_bits_to_f64(out_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    tol = output_tolerance(ref)
    worst = np.unravel_index(int(np.argmax(err)), err.shape)
    assert err.max() <= tol, (f"{what}: max|err| {err.max():.3e} > tol {tol:.3e} at {worst} "
                              f"(gpu {got[worst]:.6f}, ref {ref[worst]:.6f})")
    return float(err.max()), tol


def check_routing(idx: np.ndarray, w: np.ndarray, ref_idx: np.ndarray, ref_w: np.ndarray,
                  keys: np.ndarray = None):
    N, k = ref_idx.shape
    for n in range(N):
        assert set(idx[n].tolist()) == set(ref_idx[n].tolist()), \
            f"token {n}: experts {sorted(idx[n])} != oracle {sorted(ref_idx[n])}"
        order = {int(e): j for j, e in enumerate(idx[n])}
        for j, e in enumerate(ref_idx[n]):
            gw = float(w[n, order[int(e)]])
            assert abs(gw - ref_w[n, j]) <= 1e-4 * abs(ref_w[n, j]) + 1e-6, \
                f"token {n} expert {e}: weight {gw} vs oracle {ref_w[n, j]}"
        if keys is not None:
            kk = keys[n, ref_idx[n]]
            for j in range(k - 1):
                if kk[j] - kk[j + 1] >= ORDER_GAP:
                    assert idx[n, j] == ref_idx[n, j] or order[int(ref_idx[n, j])] < order[int(ref_idx[n, j + 1])], \
                        f"token {n}: order differs at position {j}"
