"""ctypes front end of the FP64 CPU oracle (oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
bench's CPU-baseline leg, never by the library's product path.

Every function here only marshals numpy arrays into the C oracle; the
arithmetic lives in oracle.cpp.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so (g++ -O2 -fopenmp)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router", "bias", "gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s",
        "gate_s2", "up_s2", "down_s2", "sh_gate", "sh_up", "sh_down", "sh_gate_w",
        "router_s", "router_s2", "tid2eid")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # A test may point the wrapper at a deliberately broken build of
            # oracle.cpp (mutation check of the pins); otherwise build/load ours.
            path = os.environ.get("MOE_ORACLE_LIB")
            if not path:
                path = build()
            L = ctypes.CDLL(path)
            d, u32, i32, vp = ctypes.c_double, ctypes.c_uint32, ctypes.c_int, ctypes.c_void_p
            for name in ("oracle_e2m1", "oracle_e4m3", "oracle_e8m0", "oracle_bf16"):
                getattr(L, name).restype = d
                getattr(L, name).argtypes = [u32]
            L.oracle_round_bf16.restype = u32
            L.oracle_round_bf16.argtypes = [d]
            L.oracle_fp4_weight.restype = d
            L.oracle_fp4_weight.argtypes = [vp, vp, d, i32, i32, ctypes.c_long, ctypes.c_long]
            L.oracle_dequant.restype = None
            L.oracle_dequant.argtypes = [vp, vp, d, i32, i32, i32, vp]
            L.oracle_router_logits.restype = None
            L.oracle_router_logits.argtypes = [vp, vp, i32, i32, i32, vp]
            L.oracle_router_logits_fmt.restype = None
            L.oracle_router_logits_fmt.argtypes = [vp, vp, vp, d, i32, i32, i32, i32, vp]
            L.oracle_route.restype = None
            L.oracle_route.argtypes = [vp, vp, i32, i32, i32, i32, i32, d, vp, vp, vp]
            L.oracle_weight.restype = d
            L.oracle_weight.argtypes = [vp, vp, d, i32, i32, ctypes.c_long, ctypes.c_long]
            L.oracle_expert.restype = None
            L.oracle_expert.argtypes = [vp, vp, d, vp, vp, d, vp, vp, d, i32, i32, i32, vp, vp]
            L.oracle_shared_expert.restype = None
            L.oracle_shared_expert.argtypes = [vp, vp, vp, i32, i32, vp, vp]
            L.oracle_moe_forward.restype = i32
            L.oracle_moe_forward.argtypes = [i32, i32, i32, i32, i32, i32, d, i32, i32,
                                             ctypes.POINTER(_Weights), vp, i32,
                                             vp, vp, vp, vp, vp, i32, i32, vp]
            L.oracle_num_threads.restype = i32
            L.oracle_num_threads.argtypes = []
            L.oracle_set_num_threads.restype = None
            L.oracle_set_num_threads.argtypes = [i32]
            _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


# ------------------------------------------------------------------ decoders

def e2m1(code: int) -> float:
    return lib().oracle_e2m1(code)


def e4m3(code: int) -> float:
    return lib().oracle_e4m3(code)


def e8m0(code: int) -> float:
    return lib().oracle_e8m0(code)


def bf16(bits: int) -> float:
    return lib().oracle_bf16(bits)


def round_bf16(v: float) -> int:
    return lib().oracle_round_bf16(float(v))


def scoring_code(scoring: str) -> int:
    return {"softmax": 0, "sigmoid_bias": 1, "softmax_bias": 2}[scoring]


def fmt_code(wfmt: str) -> int:
    return {"nvfp4": 0, "mxfp4": 1, "bf16": 2, "fp8": 3}[wfmt]


def dequant(q: np.ndarray, s: np.ndarray, scale2: float, wfmt: str) -> np.ndarray:
    """One FP4 projection [rows, K/2] + scales -> float64 [rows, K]."""
    rows, kh = q.shape
    K = 2 * kh
    out = np.empty((rows, K), dtype=np.float64)
    q = np.ascontiguousarray(q)
    s = np.ascontiguousarray(s)
    lib().oracle_dequant(_p(q), _p(s), float(scale2), rows, K, fmt_code(wfmt), _p(out))
    return out


# ------------------------------------------------------------------- steps

def router_logits(x: np.ndarray, router: np.ndarray, router_s: Optional[np.ndarray] = None,
                  router_s2: Optional[np.ndarray] = None) -> np.ndarray:
    """Logits of a BF16 router [E, H] (uint16 bits), or of an NVFP4 router
    (router = codes [E, H/2], router_s = E4M3 scales [E, H/16], router_s2 =
    one float or None)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    N, H = x.shape
    E = router.shape[0]
    out = np.empty((N, E), dtype=np.float64)
    if router_s is None:
        router = np.ascontiguousarray(router, dtype=np.uint16)
        lib().oracle_router_logits(_p(x), _p(router), N, E, H, _p(out))
    else:
        router = np.ascontiguousarray(router, dtype=np.uint8)
        rs = np.ascontiguousarray(router_s, dtype=np.uint8)
        s2 = 1.0 if router_s2 is None else float(np.asarray(router_s2).ravel()[0])
        lib().oracle_router_logits_fmt(_p(x), _p(router), _p(rs), s2, 1, N, E, H, _p(out))
    return out


def layer_router_logits(layer, x: np.ndarray) -> np.ndarray:
    return router_logits(x, layer.router, layer.router_s, layer.router_s2)


def route(logits: np.ndarray, k: int, scoring: str, norm: bool, rsf: float = 1.0,
          bias: Optional[np.ndarray] = None):
    """-> (idx [N,k] int32, w [N,k] float64, selection scores [N,E] float64)."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    N, E = logits.shape
    idx = np.empty((N, k), dtype=np.int32)
    w = np.empty((N, k), dtype=np.float64)
    sel = np.empty((N, E), dtype=np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    lib().oracle_route(_p(logits), _p(b), N, E, k, scoring_code(scoring),
                       int(bool(norm)), float(rsf), _p(idx), _p(w), _p(sel))
    return idx, w, sel


def weight(q: np.ndarray, s: Optional[np.ndarray], scale2: float, K: int, wfmt: str,
           r: int, k: int) -> float:
    """Element (r, k) of one routed projection, as the oracle decodes it."""
    q = np.ascontiguousarray(q)
    s = None if s is None else np.ascontiguousarray(s)
    return lib().oracle_weight(_p(q), _p(s), float(scale2), K, fmt_code(wfmt), r, k)


def expert(layer, e: int, x_row: np.ndarray) -> np.ndarray:
    """One routed expert of a synth.HostLayer on one BF16 token row -> float64 [H]."""
    sp = layer.spec
    y = np.empty(sp.H, dtype=np.float64)
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    s2 = lambda a: 1.0 if a is None else float(a[e])
    sc = lambda a: None if a is None else np.ascontiguousarray(a[e])
    lib().oracle_expert(
        _p(np.ascontiguousarray(layer.gate_q[e])), _p(sc(layer.gate_s)), s2(layer.gate_s2),
        _p(np.ascontiguousarray(layer.up_q[e])), _p(sc(layer.up_s)), s2(layer.up_s2),
        _p(np.ascontiguousarray(layer.down_q[e])), _p(sc(layer.down_s)), s2(layer.down_s2),
        sp.H, sp.inter, fmt_code(sp.wfmt), _p(x_row), _p(y))
    return y


def shared_expert(layer, x_row: np.ndarray) -> np.ndarray:
    sp = layer.spec
    sh = np.empty(sp.H, dtype=np.float64)
    x_row = np.ascontiguousarray(x_row, dtype=np.uint16)
    lib().oracle_shared_expert(_p(layer.sh_gate), _p(layer.sh_up), _p(layer.sh_down),
                               sp.H, sp.shared_inter, _p(x_row), _p(sh))
    return sh


def _weights_struct(layer) -> _Weights:
    W = _Weights()
    for name, _ in _Weights._fields_:
        setattr(W, name, _p(getattr(layer, name)))
    return W


def moe_forward(layer, x: np.ndarray, token_ids: Optional[np.ndarray] = None):
    """Full layer forward.  Returns dict with out_f64 [N,H], out_bf16 [N,H]
    (uint16 bits), idx [N,k] int32, w [N,k] float64, logits [N,E]."""
    sp = layer.spec
    x = np.ascontiguousarray(x, dtype=np.uint16)
    N = x.shape[0]
    out = np.empty((N, sp.H), dtype=np.float64)
    outb = np.empty((N, sp.H), dtype=np.uint16)
    idx = np.empty((N, sp.top_k), dtype=np.int32)
    w = np.empty((N, sp.top_k), dtype=np.float64)
    logits = np.empty((N, sp.E + sp.zero_experts), dtype=np.float64)
    W = _weights_struct(layer)
    tid = None if token_ids is None else np.ascontiguousarray(token_ids, dtype=np.int32)
    rc = lib().oracle_moe_forward(
        sp.H, sp.inter, sp.E, sp.top_k, scoring_code(sp.scoring),
        int(sp.norm_topk_prob), float(sp.routed_scaling_factor), fmt_code(sp.wfmt),
        sp.shared_inter, ctypes.byref(W), _p(x), N, _p(out), _p(outb), _p(idx), _p(w),
        _p(logits), 1 if sp.router_fmt == "nvfp4" else 0, sp.zero_experts, _p(tid))
    if rc != 0:
        raise ValueError(f"oracle_moe_forward rejected its arguments (code {rc})")
    return {"out_f64": out, "out_bf16": outb, "idx": idx, "w": w, "logits": logits}


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (timing only: every
    output element is summed by one thread in index order either way)."""
    lib().oracle_set_num_threads(int(n))
