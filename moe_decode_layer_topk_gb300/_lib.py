"""ctypes binding of include/moe.h (libmoe.so), one Python function per C entry
point, same names.  Argument marshalling only: every step of the layer runs in
the CUDA library.  torch tensors supply device pointers and the current CUDA
stream.  There is no fallback: if libmoe.so is missing the import of a
function raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
ABI_VERSION = 3

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE_TOO_SMALL = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_RANGE = 6
MOE_SCORE_SOFTMAX = 0
MOE_SCORE_SIGMOID_BIAS = 1
MOE_SCORE_SOFTMAX_BIAS = 2
MOE_W_NVFP4 = 0
MOE_W_MXFP4 = 1
MOE_W_BF16 = 2
MOE_W_FP8 = 3
MOE_R_BF16 = 0
MOE_R_NVFP4 = 1

EXPORTED = ("moe_workspace_size", "moe_workspace_init", "moe_forward", "moe_route",
            "moe_host_staging_size", "moe_forward_host", "moe_get_error", "moe_status_string",
            "moe_abi_version", "moe_debug_set_wait_budget_ns", "moe_forward_noalloc",
            "moe_debug_set_grouped_min_slots",
            "moe_forward_ids", "moe_uses_grouped_path")


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {moe_status_string(status)} (status {status})")


class LayerDesc(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("inter", ctypes.c_int32), ("E", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("scoring", ctypes.c_int32),
                ("norm_topk_prob", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("wfmt", ctypes.c_int32), ("shared_inter", ctypes.c_int32),
                ("router_fmt", ctypes.c_int32), ("zero_experts", ctypes.c_int32),
                ("hash_vocab", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router", "bias", "gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s",
        "gate_s2", "up_s2", "down_s2", "sh_gate", "sh_up", "sh_down", "sh_gate_w",
        "router_s", "router_s2", "tid2eid")]


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libmoe.so (built by __graft_entry__.build / moe_decode_layer_topk_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build() first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        pd, pw = ctypes.POINTER(LayerDesc), ctypes.POINTER(Weights)
        L.moe_workspace_size.restype = sz
        L.moe_workspace_size.argtypes = [pd, i32]
        L.moe_uses_grouped_path.restype = i32
        L.moe_uses_grouped_path.argtypes = [pd, i32]
        L.moe_host_staging_size.restype = sz
        L.moe_host_staging_size.argtypes = [pd, i32]
        L.moe_workspace_init.restype = i32
        L.moe_workspace_init.argtypes = [vp, sz, vp]
        L.moe_forward.restype = i32
        L.moe_forward.argtypes = [pd, pw, vp, i32, vp, vp, vp, vp, sz, vp]
        L.moe_route.restype = i32
        L.moe_route.argtypes = [pd, pw, vp, i32, vp, vp, vp, sz, vp]
        L.moe_forward_host.restype = i32
        L.moe_forward_host.argtypes = [pd, pw, vp, i32, vp, vp, sz, vp]
        L.moe_get_error.restype = i32
        L.moe_get_error.argtypes = [vp, vp]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_abi_version.restype = i32
        L.moe_abi_version.argtypes = []
        L.moe_forward_noalloc.restype = i32
        L.moe_forward_noalloc.argtypes = [pd, pw, vp, i32, vp, vp, vp, vp]
        L.moe_forward_ids.restype = i32
        L.moe_forward_ids.argtypes = [pd, pw, vp, vp, i32, vp, vp, vp, vp, sz, vp]
        L.moe_debug_set_wait_budget_ns.restype = None
        L.moe_debug_set_wait_budget_ns.argtypes = [ctypes.c_ulonglong]
        L.moe_debug_set_grouped_min_slots.restype = None
        L.moe_debug_set_grouped_min_slots.argtypes = [i32]
        if L.moe_abi_version() != ABI_VERSION:
            raise RuntimeError("libmoe.so ABI version mismatch; rebuild it")
        _lib = L
        return L


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(status: int, what: str):
    if status != MOE_OK:
        raise MoeError(status, what)


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_abi_version() -> int:
    return load().moe_abi_version()


def moe_workspace_size(desc: LayerDesc, max_tokens: int) -> int:
    return load().moe_workspace_size(ctypes.byref(desc), int(max_tokens))


def moe_uses_grouped_path(desc: LayerDesc, N: int) -> int:
    return load().moe_uses_grouped_path(ctypes.byref(desc), int(N))


def moe_host_staging_size(desc: LayerDesc, max_tokens: int) -> int:
    return load().moe_host_staging_size(ctypes.byref(desc), int(max_tokens))


def moe_workspace_init(ws, stream=None):
    _check(load().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_workspace_init")


def moe_forward(desc: LayerDesc, weights: Weights, x, out, ws, topk_idx=None, topk_w=None,
                stream=None, check: bool = True) -> int:
    """out[N,H] = MoE layer(x[N,H]); x, out bf16 device tensors, ws a byte tensor."""
    st = load().moe_forward(ctypes.byref(desc), ctypes.byref(weights), _ptr(x), int(x.shape[0]),
                            _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                            ws.numel() * ws.element_size(), _stream(stream))
    if check:
        _check(st, "moe_forward")
    return st


def moe_forward_ids(desc: LayerDesc, weights: Weights, x, token_ids, out, ws, topk_idx=None,
                    topk_w=None, stream=None, check: bool = True) -> int:
    """moe_forward of a hash-routed layer; token_ids an int32 device tensor [N]."""
    st = load().moe_forward_ids(ctypes.byref(desc), ctypes.byref(weights), _ptr(x),
                                _ptr(token_ids), int(x.shape[0]), _ptr(out), _ptr(topk_idx),
                                _ptr(topk_w), _ptr(ws), ws.numel() * ws.element_size(),
                                _stream(stream))
    if check:
        _check(st, "moe_forward_ids")
    return st


def moe_route(desc: LayerDesc, weights: Weights, x, topk_idx, topk_w, ws, stream=None,
              check: bool = True) -> int:
    st = load().moe_route(ctypes.byref(desc), ctypes.byref(weights), _ptr(x), int(x.shape[0]),
                          _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                          ws.numel() * ws.element_size(), _stream(stream))
    if check:
        _check(st, "moe_route")
    return st


def moe_forward_host(desc: LayerDesc, weights: Weights, x_host, out_host, ws, stream=None,
                     check: bool = True) -> int:
    """Host (CPU, ideally pinned) bf16 x/out tensors; synchronises the stream."""
    st = load().moe_forward_host(ctypes.byref(desc), ctypes.byref(weights), _ptr(x_host),
                                 int(x_host.shape[0]), _ptr(out_host), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream))
    if check:
        _check(st, "moe_forward_host")
    return st


def moe_forward_noalloc(desc: LayerDesc, weights: Weights, x, out, topk_idx=None, topk_w=None,
                        stream=None, check: bool = True) -> int:
    """moe_forward in the library's built-in device scratch (no workspace
    argument, no allocation); for callers that cannot allocate device memory."""
    st = load().moe_forward_noalloc(ctypes.byref(desc), ctypes.byref(weights), _ptr(x),
                                    int(x.shape[0]), _ptr(out), _ptr(topk_idx), _ptr(topk_w),
                                    _stream(stream))
    if check:
        _check(st, "moe_forward_noalloc")
    return st


def moe_get_error(ws, stream=None) -> int:
    return load().moe_get_error(_ptr(ws), _stream(stream))


def moe_debug_set_wait_budget_ns(ns: int):
    load().moe_debug_set_wait_budget_ns(int(ns))


def moe_debug_set_grouped_min_slots(slots: int):
    """Pairs N x top_k from which large FP4 layers take the grouped path
    (0 restores the built-in threshold); size workspaces afterwards."""
    load().moe_debug_set_grouped_min_slots(int(slots))
