"""C-ABI checks: the library loads, exports every entry point include/moe.h
declares, and refuses bad arguments before touching the GPU (CPU tests); on a
GPU the error paths return their status and leave the context usable."""
import ctypes
import os
import re

import numpy as np
import pytest

from moe_decode_layer_topk_gb300 import _lib, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from moe_decode_layer_topk_gb300 import build
    build.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)


def test_header_declares_the_binding_names():
    assert sorted(_declared()) == sorted(_lib.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert lib.moe_abi_version() == _lib.ABI_VERSION


def test_status_strings(lib):
    for st in range(7):
        assert _lib.moe_status_string(st)
    assert "unknown" in _lib.moe_status_string(99)


def _desc(**kw):
    d = _lib.LayerDesc()
    d.H, d.inter, d.E, d.top_k = kw.get("H", 256), kw.get("inter", 128), kw.get("E", 8), kw.get("top_k", 2)
    d.scoring = kw.get("scoring", 0)
    d.norm_topk_prob = 1
    d.routed_scaling_factor = 1.0
    d.wfmt = kw.get("wfmt", 0)
    d.shared_inter = kw.get("shared_inter", 0)
    return d


def test_workspace_size_grows_with_tokens(lib):
    d = _desc()
    a, b = _lib.moe_workspace_size(d, 1), _lib.moe_workspace_size(d, 4)
    assert 0 < a < b
    assert _lib.moe_workspace_size(d, 0) == 0
    assert _lib.moe_host_staging_size(d, 4) >= 2 * 4 * 256 * 2


@pytest.mark.parametrize("bad", [dict(H=100), dict(inter=48), dict(E=0), dict(top_k=9),
                                 dict(E=2000), dict(top_k=40, E=64), dict(scoring=3), dict(wfmt=7), dict(wfmt=4),
                                 dict(shared_inter=40)])
def test_bad_descriptor_is_refused(lib, bad):
    assert _lib.moe_workspace_size(_desc(**bad), 1) == 0


def test_bad_router_format_is_refused(lib):
    d = _desc()
    d.router_fmt = 2
    assert _lib.moe_workspace_size(d, 1) == 0


@pytest.mark.parametrize("E,Z", [(8, -1), (1000, 25)])
def test_bad_zero_expert_count_is_refused(lib, E, Z):
    d = _desc(E=E)
    d.zero_experts = Z
    assert _lib.moe_workspace_size(d, 1) == 0


def _fake_weights(shared=False):
    w = _lib.Weights()
    base = 1 << 20
    for i, (name, _) in enumerate(_lib.Weights._fields_):
        setattr(w, name, base + 256 * i)
    w.bias = None
    if not shared:
        w.sh_gate = w.sh_up = w.sh_down = w.sh_gate_w = None
    return w


def _forward(lib, d, w, N=1, x=1 << 24, out=1 << 25, ws=1 << 26, ws_bytes=1 << 30):
    return lib.moe_forward(ctypes.byref(d), ctypes.byref(w), x, N, out, None, None, ws, ws_bytes, None)


def test_dispatch_rule(lib):
    """Fused kernels up to 256 (token, slot) pairs, grouped path beyond for
    the layers it takes (FP4 experts, no shared expert, zero experts or hash
    routing; the others stay fused, in row chunks); those whose experts hold
    >= 1 MiB of weights switch for N > 8 (the measured crossing); the tuning
    hook replaces that by a pair threshold.  Host-only."""
    from moe_decode_layer_topk_gb300.device import layer_desc

    def g(spec, N):
        return _lib.moe_uses_grouped_path(layer_desc(spec), N)

    oss, q3 = synth.CONFIGS["gpt_oss_120b"], synth.CONFIGS["qwen3_30b_a3b"]
    assert [g(oss, n) for n in (1, 4, 8, 9, 16, 64, 65, 512)] == [0, 0, 0, 1, 1, 1, 1, 1]
    assert [g(q3, n) for n in (1, 4, 8, 9, 16, 33)] == [0, 0, 0, 1, 1, 1]
    assert g(synth.CONFIGS["qwen3_30b_a3b_nvfp4_router"], 16) == 1
    try:
        _lib.moe_debug_set_grouped_min_slots(128)
        assert [g(oss, n) for n in (31, 32)] == [0, 1]
        assert [g(q3, n) for n in (15, 16)] == [0, 1]
    finally:
        _lib.moe_debug_set_grouped_min_slots(0)
    assert [g(oss, n) for n in (8, 9)] == [0, 1]
    for name in ("deepseek_v3", "mtp_verify", "qwen3_30b_a3b_bf16", "qwen3_30b_a3b_fp8",
                 "qwen3_30b_a3b_zero_experts"):       # no grouped path: fused, in row chunks
        sp = synth.CONFIGS[name]
        assert (g(sp, 256 // sp.top_k), g(sp, 256 // sp.top_k + 1), g(sp, 512)) == (0, 0, 0), name
    tiny = synth.CONFIGS["tiny"]                      # 55 KB experts
    assert (g(tiny, 128), g(tiny, 129)) == (0, 1)
    assert g(tiny, 0) == -1
    ws = [_lib.moe_workspace_size(layer_desc(oss), n) for n in range(1, 80)]
    assert all(a <= b for a, b in zip(ws, ws[1:]))


def test_argument_refusals_happen_before_any_cuda_call(lib):
    """Every case below is refused by the host checks (no GPU needed)."""
    d, w = _desc(), _fake_weights()
    assert _forward(lib, d, w, N=0) == _lib.MOE_ERR_INVALID_ARG
    # N*k > 256 takes the grouped path: its own workspace check; a layer it
    # does not take (here a shared expert) runs the fused kernels in row chunks
    assert _forward(lib, d, w, N=300, ws_bytes=1 << 20) == _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    assert _lib.moe_workspace_size(d, 300) > _lib.moe_workspace_size(d, 128)
    dsh = _desc(shared_inter=64)
    assert _lib.moe_uses_grouped_path(dsh, 300) == 0
    assert _lib.moe_workspace_size(dsh, 300) == _lib.moe_workspace_size(dsh, 128)
    assert _forward(lib, dsh, _fake_weights(shared=True), N=300, ws_bytes=1 << 10) == \
        _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    assert _forward(lib, d, w, x=(1 << 24) + 8) == _lib.MOE_ERR_INVALID_ARG
    assert _forward(lib, d, w, out=None) == _lib.MOE_ERR_INVALID_ARG
    assert _forward(lib, d, w, ws_bytes=16) == _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    w2 = _fake_weights()
    w2.gate_q = None
    assert _forward(lib, d, w2) == _lib.MOE_ERR_INVALID_ARG
    w3 = _fake_weights()
    w3.down_s = (1 << 20) + 3
    assert _forward(lib, d, w3) == _lib.MOE_ERR_INVALID_ARG
    w4 = _fake_weights()                                                  # FP4 experts need scales
    w4.up_s = None
    assert _forward(lib, d, w4) == _lib.MOE_ERR_INVALID_ARG
    # BF16 routed experts: no grouped path yet (N*k > 256: row chunks)
    db = _desc(wfmt=_lib.MOE_W_BF16)
    wb = _fake_weights()
    wb.gate_s = wb.up_s = wb.down_s = wb.gate_s2 = wb.up_s2 = wb.down_s2 = None
    assert _lib.moe_uses_grouped_path(db, 300) == 0
    wb.gate_q = None
    assert _forward(lib, db, wb) == _lib.MOE_ERR_INVALID_ARG
    # FP8 routed experts: block scales required, no grouped path yet
    d8 = _desc(wfmt=_lib.MOE_W_FP8)
    w8 = _fake_weights()
    assert _lib.moe_uses_grouped_path(d8, 300) == 0
    w8.down_s = None
    assert _forward(lib, d8, w8) == _lib.MOE_ERR_INVALID_ARG
    # NVFP4 router: its scales are required
    dr = _desc()
    dr.router_fmt = _lib.MOE_R_NVFP4
    wr = _fake_weights()
    wr.router_s = None
    assert _forward(lib, dr, wr) == _lib.MOE_ERR_INVALID_ARG
    # softmax + bias needs its bias; zero experts: no grouped path yet
    dz = _desc(scoring=_lib.MOE_SCORE_SOFTMAX_BIAS)
    dz.zero_experts = 64
    assert _forward(lib, dz, _fake_weights()) == _lib.MOE_ERR_INVALID_ARG
    wz = _fake_weights()
    wz.bias = 1 << 21
    assert _lib.moe_uses_grouped_path(dz, 300) == 0
    assert _lib.moe_workspace_size(dz, 4) > _lib.moe_workspace_size(_desc(), 4)
    # hash routing: token ids required (and only for hash routing), the table
    # required, no grouped path, no zero experts with it
    dh = _desc()
    dh.hash_vocab = 100
    assert _forward(lib, dh, _fake_weights()) == _lib.MOE_ERR_INVALID_ARG
    ids = 1 << 22
    assert _lib.moe_uses_grouped_path(dh, 300) == 0
    wt = _fake_weights()
    wt.tid2eid = None
    assert lib.moe_forward_ids(ctypes.byref(dh), ctypes.byref(wt), 1 << 24, ids, 1, 1 << 25,
                               None, None, 1 << 26, 1 << 30, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_ids(ctypes.byref(d), ctypes.byref(w), 1 << 24, ids, 1, 1 << 25,
                               None, None, 1 << 26, 1 << 30, None) == _lib.MOE_ERR_INVALID_ARG
    dh.zero_experts = 4
    assert _lib.moe_workspace_size(dh, 1) == 0
    ds = _desc(scoring=1)                                                 # sigmoid needs a bias
    assert _forward(lib, ds, _fake_weights()) == _lib.MOE_ERR_INVALID_ARG
    dsh = _desc(shared_inter=64)                                          # shared size, no weights
    assert _forward(lib, dsh, _fake_weights()) == _lib.MOE_ERR_INVALID_ARG
    assert _forward(lib, d, _fake_weights(shared=True)) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_route(ctypes.byref(d), ctypes.byref(w), 1 << 24, 1, None, None, 1 << 26,
                         1 << 30, None) == _lib.MOE_ERR_INVALID_ARG
    assert lib.moe_forward(None, ctypes.byref(w), 1 << 24, 1, 1 << 25, None, None, 1 << 26,
                           1 << 30, None) == _lib.MOE_ERR_INVALID_ARG


# ----------------------------------------------------------------- GPU paths

@pytest.mark.gpu
def test_gpu_error_statuses_leave_context_usable(lib):
    import torch
    from moe_decode_layer_topk_gb300.device import DeviceLayer, bf16_tensor, workspace
    spec = synth.CONFIGS["tiny"]
    dev = DeviceLayer.upload(synth.make_layer(spec))
    x = bf16_tensor(synth.make_tokens(spec, 2))
    out = torch.empty_like(x)
    ws = workspace(spec, 2)
    small = ws[: _lib.moe_workspace_size(dev.desc, 1)]
    assert _lib.moe_forward(dev.desc, dev.weights, x, out, small, check=False) == \
        _lib.MOE_ERR_WORKSPACE_TOO_SMALL
    _lib.moe_forward(dev.desc, dev.weights, x, out, ws)
    torch.cuda.synchronize()
    assert _lib.moe_get_error(ws) == _lib.MOE_OK
    assert torch.isfinite(out.float()).all()


@pytest.mark.gpu
def test_gpu_wait_timeout_is_reported_not_hung(lib):
    """A zero wait budget makes the first grid barrier expire; the call returns,
    moe_get_error reports MOE_ERR_TIMEOUT, and after re-initialising the
    workspace the next call is correct."""
    import torch
    from moe_decode_layer_topk_gb300.device import DeviceLayer, bf16_tensor, workspace
    spec = synth.CONFIGS["tiny"]
    dev = DeviceLayer.upload(synth.make_layer(spec))
    x = bf16_tensor(synth.make_tokens(spec, 1))
    out = torch.empty_like(x)
    ws = workspace(spec, 1)
    _lib.moe_forward(dev.desc, dev.weights, x, out, ws)
    torch.cuda.synchronize()
    ref = out.clone()
    try:
        _lib.moe_debug_set_wait_budget_ns(0)
        for _ in range(3):
            _lib.moe_forward(dev.desc, dev.weights, x, out, ws)
        torch.cuda.synchronize()
    finally:
        _lib.moe_debug_set_wait_budget_ns(1_000_000_000)
    assert _lib.moe_get_error(ws) == _lib.MOE_ERR_TIMEOUT
    _lib.moe_workspace_init(ws)
    _lib.moe_forward(dev.desc, dev.weights, x, out, ws)
    torch.cuda.synchronize()
    assert _lib.moe_get_error(ws) == _lib.MOE_OK
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16)) or \
        torch.allclose(out.float(), ref.float(), rtol=1e-2, atol=2 ** -8)


def test_every_entry_point_fails_loudly_without_the_library(monkeypatch):
    """No CPU fallback: with libmoe.so absent, each binding raises before it
    computes anything."""
    import inspect
    monkeypatch.setattr(_lib, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libmoe.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    called = 0
    for name in _lib.EXPORTED:
        fn = getattr(_lib, name, None)
        if fn is None:
            continue
        sig = inspect.signature(fn)
        args = [None for p in sig.parameters.values()
                if p.default is inspect.Parameter.empty and p.kind == p.POSITIONAL_OR_KEYWORD]
        with pytest.raises(RuntimeError, match="not built"):
            fn(*args)
        called += 1
    assert called >= 8
