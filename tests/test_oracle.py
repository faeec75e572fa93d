"""Pins of the FP64 oracle against facts that do not come from the oracle.

Each test checks one oracle function against a closed form, a format
specification table (tests/golden, each file cites its source), a library
routine (torch's float8 dtypes, numpy/scipy), or brute force on tiny inputs.
The pages themselves print no numeric example, so no test compares against a
value the pages give.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from moe_decode_layer_topk_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 0), float(v)))
    return rows


def _same(a, b):
    return (math.isnan(a) and math.isnan(b)) or (a == b and math.copysign(1, a) == math.copysign(1, b))


# ------------------------------------------------------------------ decoders

def test_e2m1_all_16_codes_match_ocp_table(oracle_mod):
    table = _golden("e2m1_codes.txt")
    assert len(table) == 16
    for code, val in table:
        assert _same(oracle_mod.e2m1(code), val), code


def test_e4m3_all_256_codes_match_torch_float8(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for c in range(256):
        assert _same(oracle_mod.e4m3(c), float(ref[c])), hex(c)


def test_e4m3_special_points_match_ocp_table(oracle_mod):
    for code, val in _golden("e4m3_special.txt"):
        assert _same(oracle_mod.e4m3(code), val), hex(code)


def test_e4m3_closed_form(oracle_mod):
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert math.isnan(oracle_mod.e4m3(c))
            continue
        mag = 2.0 ** -6 * m / 8 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8)
        assert oracle_mod.e4m3(c) == (-mag if s else mag)


def test_e8m0_all_codes(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    for c in range(256):
        v = oracle_mod.e8m0(c)
        if c == 255:
            assert math.isnan(v)
        else:
            assert v == math.ldexp(1.0, c - 127) == float(ref[c])
    for code, val in _golden("e8m0_special.txt"):
        assert _same(oracle_mod.e8m0(code), val)


def test_bf16_decode_matches_bit_widening(oracle_mod):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4000, dtype=np.uint32)
    ref = (bits << 16).astype(np.uint32).view(np.float32)
    for b, r in zip(bits, ref):
        assert _same(oracle_mod.bf16(int(b)), float(r))


def _bf16_val(b):
    return float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])


def _nearest_bf16_bruteforce(v):
    """Search the bf16 patterns around float32(v) for the nearest to v (ties to
    an even last bit)."""
    base = int(np.array([v], dtype=np.float32).view(np.uint32)[0]) >> 16
    best = None
    for b in range(max(0, (base & 0x7FFF) - 2), min(0x7F80, (base & 0x7FFF) + 3)):
        b |= base & 0x8000
        d = abs(_bf16_val(b) - v)
        if best is None or d < best[0] or (d == best[0] and (b & 1) == 0):
            best = (d, b)
    return best[1]


def test_round_bf16_nearest_even_bruteforce(oracle_mod):
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000))
    # exact midpoints between neighbouring bf16 values (ties)
    for b in rng.integers(0x0080, 0x7F00, size=400):
        lo, hi = _bf16_val(int(b)), _bf16_val(int(b) + 1)
        vals += [(lo + hi) / 2, -(lo + hi) / 2]
    # just above / below a midpoint (double precision only)
    vals += [1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 2.0 ** -8 - 2.0 ** -40]
    for v in vals:
        assert oracle_mod.round_bf16(float(v)) == _nearest_bf16_bruteforce(float(v)), v


# ------------------------------------------------------------ quantise/decode

def _decode_fp4_independent(q, s, wfmt):
    """Test-side decode: golden E2M1 table, torch float8 decode of the scales."""
    table = np.array([v for _, v in _golden("e2m1_codes.txt")])
    lo, hi = q & 0xF, q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1)
    gs = 16 if wfmt == synth.NVFP4 else 32
    dt = torch.float8_e4m3fn if wfmt == synth.NVFP4 else torch.float8_e8m0fnu
    sv = torch.from_numpy(np.ascontiguousarray(s)).view(dt).to(torch.float64).numpy()
    return table[codes] * np.repeat(sv, gs, axis=1)


@pytest.mark.parametrize("wfmt", [synth.NVFP4, synth.MXFP4])
def test_dequant_matches_independent_decode(oracle_mod, wfmt):
    rng = np.random.default_rng(2)
    w = rng.standard_normal((24, 96)).astype(np.float32) * 0.02
    q, s = synth.quantize_nvfp4(w) if wfmt == synth.NVFP4 else synth.quantize_mxfp4(w)
    dq = oracle_mod.dequant(q, s, 1.0, wfmt)
    np.testing.assert_array_equal(dq, _decode_fp4_independent(q, s, wfmt))


@pytest.mark.parametrize("wfmt", [synth.NVFP4, synth.MXFP4])
def test_dequant_recovers_source_within_quantisation_bound(oracle_mod, wfmt):
    """quantise(w) then decode is within one block-scale step of w, element by
    element: a wrong nibble order, scale axis or transposition breaks this."""
    rng = np.random.default_rng(3)
    rows, K = 40, 256
    w = (rng.standard_normal((rows, K)) * 0.02).astype(np.float32)
    if wfmt == synth.NVFP4:
        q, s = synth.quantize_nvfp4(w)
        sv = torch.from_numpy(s).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        gs = 16
    else:
        q, s = synth.quantize_mxfp4(w)
        sv = np.ldexp(1.0, s.astype(np.int64) - 127)
        gs = 32
    dq = oracle_mod.dequant(q, s, 1.0, wfmt)
    # |w|/s <= 6: nearest grid point, largest half-gap of the E2M1 grid is 1.
    # |w|/s > 6: saturated to 6 (the scale itself was rounded down, by up to a
    # quarter for E4M3 subnormal scales, or amax < 8X for E8M0).
    sv = np.repeat(sv, gs, axis=1)
    bound = np.maximum(sv, np.abs(w) - 6.0 * sv)
    assert np.all(np.abs(dq - w) <= bound + 1e-12)
    # and it is a real approximation, not a coincidence of the bound
    assert np.abs(dq - w).mean() < 0.25 * np.abs(w).mean()


def test_quantiser_round_trip_on_grid_values(oracle_mod):
    """Blocks made of exact E2M1 grid values times a representable scale come
    back bit-exactly (codes and scales)."""
    rng = np.random.default_rng(4)
    table = np.array([v for _, v in _golden("e2m1_codes.txt")])
    for wfmt in (synth.NVFP4, synth.MXFP4):
        gs = 16 if wfmt == synth.NVFP4 else 32
        codes = rng.integers(0, 16, size=(8, 64)).astype(np.uint8)
        codes[:, ::gs] = 7                         # every block reaches amax = 6
        codes[codes == 8] = 0                      # no negative zero
        if wfmt == synth.NVFP4:
            sc = rng.choice([0x30, 0x38, 0x21, 0x05, 0x44], size=(8, 64 // gs)).astype(np.uint8)
            sval = torch.from_numpy(sc).view(torch.float8_e4m3fn).to(torch.float64).numpy()
            w = table[codes] * np.repeat(sval, gs, axis=1)
            q, s = synth.quantize_nvfp4(w.astype(np.float32))
        else:
            sc = rng.integers(100, 140, size=(8, 64 // gs)).astype(np.uint8)
            w = table[codes] * np.repeat(np.ldexp(1.0, sc.astype(np.int64) - 127), gs, axis=1)
            q, s = synth.quantize_mxfp4(w.astype(np.float32))
        np.testing.assert_array_equal(s, sc)
        np.testing.assert_array_equal(q, synth.pack_nibbles(codes))
        np.testing.assert_array_equal(oracle_mod.dequant(q, s, 1.0, wfmt), w)


def test_scale_buffer_sizes_follow_group_size():
    """Scale bytes per projection are rows*K/16 (NVFP4) and rows*K/32 (E8M0),
    the sizes the pages give for the two scale buffers."""
    for name in ("tiny", "gpt_oss_120b"):
        sp = synth.CONFIGS[name]
        sp_small = synth.LayerSpec(**{**sp.__dict__, "H": 64, "inter": 64, "E": 2, "pool": 2,
                                     "shared_inter": 0})
        L = synth.make_layer(sp_small)
        assert L.gate_s.size == 2 * 64 * 64 // sp.gs
        assert L.down_q.size == 2 * 64 * 64 // 2


# ------------------------------------------------------------------- router

def _bf16_arr(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def test_router_logits_match_numpy_matmul(oracle_mod):
    rng = np.random.default_rng(5)
    x = synth.f32_to_bf16_bits(rng.standard_normal((3, 200)).astype(np.float32))
    wr = synth.f32_to_bf16_bits((rng.standard_normal((17, 200)) / 14).astype(np.float32))
    ref = _bf16_arr(x) @ _bf16_arr(wr).T
    np.testing.assert_allclose(oracle_mod.router_logits(x, wr), ref, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ routing

def _brute_topk(score, k):
    """Expert i is selected iff fewer than k experts beat it (higher score, or
    equal score and lower index); order by (score desc, index asc)."""
    E = len(score)
    sel = [i for i in range(E)
           if sum(1 for j in range(E) if score[j] > score[i] or (score[j] == score[i] and j < i)) < k]
    return sorted(sel, key=lambda i: (-score[i], i))


def test_topk_bruteforce_tiny_E_softmax(oracle_mod):
    rng = np.random.default_rng(6)
    for E in range(1, 9):
        for k in range(1, E + 1):
            for trial in range(6):
                logits = rng.standard_normal((1, E))
                if trial == 0:
                    logits[0, :] = np.round(logits[0, :] * 2) / 2     # exact ties
                for norm in (False, True):
                    idx, w, _ = oracle_mod.route(logits, k, "softmax", norm)
                    p = scipy.special.softmax(logits[0])
                    want = _brute_topk(p, k)
                    assert list(idx[0]) == want
                    ref = p[want] / (p[want].sum() if norm else 1.0)
                    np.testing.assert_allclose(w[0], ref, rtol=1e-14, atol=1e-16)


def test_topk_bruteforce_tiny_E_sigmoid_bias(oracle_mod):
    rng = np.random.default_rng(7)
    for E in range(1, 9):
        for k in range(1, E + 1):
            logits = rng.standard_normal((2, E))
            bias = (rng.standard_normal(E) * 0.5).astype(np.float32)
            for norm in (False, True):
                idx, w, sel = oracle_mod.route(logits, k, "sigmoid_bias", norm, 2.5, bias)
                for n in range(2):
                    s = scipy.special.expit(logits[n])
                    want = _brute_topk(s + bias.astype(np.float64), k)
                    assert list(idx[n]) == want
                    ref = s[want] / (s[want].sum() if norm else 1.0) * 2.5
                    np.testing.assert_allclose(w[n], ref, rtol=1e-14)


def test_topk_bruteforce_tiny_E_softmax_bias(oracle_mod):
    """Softmax scores plus a correction bias select (the zero-expert routers'
    softmax+bias arm); the weights are the selected softmax scores,
    renormalised if asked, times the routed scaling factor."""
    rng = np.random.default_rng(17)
    for E in range(1, 9):
        for k in range(1, E + 1):
            logits = rng.standard_normal((2, E))
            bias = (rng.standard_normal(E) * 0.2).astype(np.float32)
            for norm in (False, True):
                idx, w, sel = oracle_mod.route(logits, k, "softmax_bias", norm, 1.7, bias)
                for n in range(2):
                    p = scipy.special.softmax(logits[n])
                    want = _brute_topk(p + bias.astype(np.float64), k)
                    assert list(idx[n]) == want
                    ref = p[want] / (p[want].sum() if norm else 1.0) * 1.7
                    np.testing.assert_allclose(w[n], ref, rtol=1e-14)


def test_routing_weights_sum(oracle_mod):
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((16, 128)) * 2
    _, w, _ = oracle_mod.route(logits, 8, "softmax", True)
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-15 * 8)
    bias = (rng.standard_normal(128) * 0.1).astype(np.float32)
    _, w, _ = oracle_mod.route(logits, 8, "sigmoid_bias", True, 2.5, bias)
    assert np.all(np.abs(w.sum(1) - 2.5) <= 2.5e-15 * 8)
    _, w, _ = oracle_mod.route(logits, 8, "sigmoid_bias", False, 1.0, bias)
    assert np.all(w > 0) and np.all(w < 1)


def test_softmax_renorm_equals_softmax_over_selected(oracle_mod):
    """'softmax over the selected top-k' (the gpt-oss reading) is softmax over
    all experts followed by renormalisation."""
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((5, 128)) * 3
    idx, w, _ = oracle_mod.route(logits, 4, "softmax", True)
    for n in range(5):
        ref = scipy.special.softmax(logits[n, idx[n]])
        np.testing.assert_allclose(w[n], ref, rtol=1e-13)


def test_bias_selects_but_does_not_weight(oracle_mod):
    logits = np.array([[2.0, 1.0, 0.0, -1.0]])
    bias = np.array([0.0, 0.0, 0.0, 5.0], dtype=np.float32)   # pulls expert 3 in
    idx, w, _ = oracle_mod.route(logits, 2, "sigmoid_bias", False, 1.0, bias)
    assert list(idx[0]) == [3, 0]
    np.testing.assert_allclose(w[0], scipy.special.expit([-1.0, 2.0]), rtol=1e-15)


# ---------------------------------------------------------------- full layer

def _small_spec(**kw):
    base = dict(name="t", H=64, inter=32, E=4, top_k=2, scoring=synth.SOFTMAX,
                norm_topk_prob=True, routed_scaling_factor=1.0, wfmt=synth.NVFP4,
                shared_inter=0, shared_gated=False, x_rms_norm=False, tokens=(1,), pool=64)
    base.update(kw)
    return synth.LayerSpec(**base)


def _dense_swiglu(layer, e, x64):
    """Independent dense SwiGLU with numpy matmuls on test-side dequantised
    matrices (golden E2M1 table + torch float8 scales)."""
    sp = layer.spec
    s2 = (lambda a: 1.0 if a is None else float(a[e]))
    Wg = _decode_fp4_independent(layer.gate_q[e], layer.gate_s[e], sp.wfmt) * s2(layer.gate_s2)
    Wu = _decode_fp4_independent(layer.up_q[e], layer.up_s[e], sp.wfmt) * s2(layer.up_s2)
    Wd = _decode_fp4_independent(layer.down_q[e], layer.down_s[e], sp.wfmt) * s2(layer.down_s2)
    g, u = Wg @ x64, Wu @ x64
    return Wd @ (g * scipy.special.expit(g) * u)


def _dense_shared(layer, x64):
    Wg, Wu, Wd = _bf16_arr(layer.sh_gate), _bf16_arr(layer.sh_up), _bf16_arr(layer.sh_down)
    g, u = Wg @ x64, Wu @ x64
    return Wd @ (g * scipy.special.expit(g) * u)


@pytest.mark.parametrize("wfmt", [synth.NVFP4, synth.MXFP4])
def test_single_expert_equals_dense_swiglu(oracle_mod, wfmt):
    sp = _small_spec(E=1, top_k=1, H=96, inter=64, wfmt=wfmt)
    L = synth.make_layer(sp, seed=11)
    x = synth.make_tokens(sp, 3, seed=12)
    r = oracle_mod.moe_forward(L, x)
    for n in range(3):
        ref = _dense_swiglu(L, 0, _bf16_arr(x[n]))
        np.testing.assert_allclose(r["out_f64"][n], ref, rtol=1e-12, atol=1e-15)
    assert np.all(r["w"] == 1.0)
    rb = np.array([oracle_mod.round_bf16(v) for v in r["out_f64"].ravel()]).reshape(r["out_bf16"].shape)
    np.testing.assert_array_equal(r["out_bf16"], rb)


def _bf16_layer_from_fp4(layer):
    """The same layer with BF16 routed experts holding the FP4 experts' values
    (test-side decode; every E2M1 x E4M3 product has at most 6 significant bits,
    so it is a BF16 number exactly)."""
    import dataclasses
    sp = layer.spec
    assert sp.wfmt == synth.NVFP4 and all(np.all(a == 1.0) for a in (layer.gate_s2, layer.up_s2, layer.down_s2))

    def conv(q, s):
        out = []
        for e in range(q.shape[0]):
            v = _decode_fp4_independent(q[e], s[e], sp.wfmt)
            bits = synth.f32_to_bf16_bits(v.astype(np.float32))
            assert np.array_equal(_bf16_arr(bits), v)          # exact
            out.append(bits)
        return np.stack(out)

    spb = dataclasses.replace(sp, wfmt=synth.BF16)
    return dataclasses.replace(layer, spec=spb, gate_q=conv(layer.gate_q, layer.gate_s),
                               up_q=conv(layer.up_q, layer.up_s),
                               down_q=conv(layer.down_q, layer.down_s),
                               gate_s=None, up_s=None, down_s=None,
                               gate_s2=None, up_s2=None, down_s2=None)


def test_bf16_experts_equal_fp4_experts_with_the_same_values(oracle_mod):
    """BF16 routed experts (the pages' BF16 expert branch: the same chain with
    plain BF16 weights) holding exactly the values of NVFP4 experts give the
    NVFP4 layer's result to the last bit."""
    sp = _small_spec(E=6, top_k=3, H=96, inter=64)
    L = synth.make_layer(sp, seed=21)
    Lb = _bf16_layer_from_fp4(L)
    x = synth.make_tokens(sp, 4, seed=22)
    r, rb = oracle_mod.moe_forward(L, x), oracle_mod.moe_forward(Lb, x)
    assert set(r["idx"].ravel()) - {0}, "routing must reach experts past the first"
    np.testing.assert_array_equal(rb["idx"], r["idx"])
    np.testing.assert_array_equal(rb["out_f64"], r["out_f64"])
    np.testing.assert_array_equal(rb["out_bf16"], r["out_bf16"])


def test_bf16_single_expert_equals_dense_swiglu(oracle_mod):
    sp = _small_spec(E=1, top_k=1, H=96, inter=64, wfmt=synth.BF16)
    L = synth.make_layer(sp, seed=23)
    assert L.gate_s is None and L.gate_q.dtype == np.uint16 and L.gate_q.shape == (1, 64, 96)
    x = synth.make_tokens(sp, 2, seed=24)
    r = oracle_mod.moe_forward(L, x)
    Wg, Wu, Wd = (_bf16_arr(a[0]) for a in (L.gate_q, L.up_q, L.down_q))
    for n in range(2):
        x64 = _bf16_arr(x[n])
        g, u = Wg @ x64, Wu @ x64
        ref = Wd @ (g * scipy.special.expit(g) * u)
        np.testing.assert_allclose(r["out_f64"][n], ref, rtol=1e-12, atol=1e-15)
    for (rr, kk) in ((0, 0), (5, 17), (63, 95)):
        assert oracle_mod.weight(L.gate_q[0], None, 1.0, 96, synth.BF16, rr, kk) == Wg[rr, kk]


def test_bf16_expert_pool_copies_flip_whole_rows(oracle_mod):
    """With fewer drawn experts than slots, a BF16 slot is a pool expert with
    some rows negated (sign bit of every word of the row)."""
    sp = _small_spec(E=6, top_k=2, wfmt=synth.BF16, pool=2)
    L = synth.make_layer(sp, seed=25)
    b = _bf16_arr(L.gate_q)                       # [E, rows, K]
    assert not np.array_equal(np.abs(b[0]), np.abs(b[1]))
    for e in range(2, 6):
        src = [p for p in range(2) if np.array_equal(np.abs(b[e]), np.abs(b[p]))]
        assert len(src) == 1
        same = np.all(b[e] == b[src[0]], axis=1)
        neg = np.all(b[e] == -b[src[0]], axis=1)
        assert np.all(same | neg)


def _decode_fp8_independent(q, s):
    """Test-side FP8 decode: torch float8_e4m3fn bytes times the repeated
    128 x 128 block scales."""
    v = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    B = synth.FP8_BLOCK
    sc = np.repeat(np.repeat(s.astype(np.float64), B, axis=0), B, axis=1)[:q.shape[0], :q.shape[1]]
    return v * sc


def test_fp8_quantiser_and_decode(oracle_mod):
    """Block scale = amax/448, the block's largest element lands on +-448, and
    every element is within half an E4M3 step of the source."""
    rng = np.random.default_rng(31)
    w = (rng.standard_normal((300, 200)) * 0.02).astype(np.float32)
    w[130:140, 5:9] *= 50                                 # one loud corner
    q, s = synth.quantize_fp8_block(w)
    assert q.shape == (300, 200) and s.shape == (3, 2)
    for i in range(3):
        for j in range(2):
            blk = w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert s[i, j] == np.float32(np.abs(blk).max() / 448.0)
    dq = _decode_fp8_independent(q, s)
    for (r, k) in ((0, 0), (129, 7), (299, 199), (131, 6), (5, 150)):
        assert oracle_mod.weight(q, s, 1.0, 200, synth.FP8, r, k) == dq[r, k]
    sc = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:300, :200]
    a = np.abs(w.astype(np.float64)) / sc                 # magnitude in E4M3 units
    step = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3))
    assert np.all(np.abs(dq - w) <= 0.5 * step * sc * (1 + 1e-9))
    assert np.abs(_decode_fp8_independent(q, s)).max() == pytest.approx(np.abs(w).max(), rel=1e-7)


def test_fp8_experts_equal_bf16_experts_with_the_same_values(oracle_mod):
    """FP8 routed experts whose block scales are powers of two hold BF16
    numbers exactly (4 significant bits); the layer then equals the BF16-expert
    layer with those values to the last bit.  Rows > 128 give several row
    blocks per projection."""
    import dataclasses
    sp = _small_spec(E=5, top_k=2, H=256, inter=160, wfmt=synth.FP8)
    L = synth.make_layer(sp, seed=33)
    rng = np.random.default_rng(34)
    for a in (L.gate_s, L.up_s, L.down_s):
        a[:] = np.ldexp(1.0, rng.integers(-13, -6, size=a.shape)).astype(np.float32)

    def conv(q, s):
        out = []
        for e in range(q.shape[0]):
            v = _decode_fp8_independent(q[e], s[e])
            bits = synth.f32_to_bf16_bits(v.astype(np.float32))
            assert np.array_equal(_bf16_arr(bits), v)
            out.append(bits)
        return np.stack(out)

    Lb = dataclasses.replace(L, spec=dataclasses.replace(sp, wfmt=synth.BF16),
                             gate_q=conv(L.gate_q, L.gate_s), up_q=conv(L.up_q, L.up_s),
                             down_q=conv(L.down_q, L.down_s), gate_s=None, up_s=None, down_s=None)
    x = synth.make_tokens(sp, 3, seed=35)
    r, rb = oracle_mod.moe_forward(L, x), oracle_mod.moe_forward(Lb, x)
    assert set(r["idx"].ravel()) - {0}
    np.testing.assert_array_equal(r["out_f64"], rb["out_f64"])


def test_fp8_single_expert_equals_dense_swiglu(oracle_mod):
    sp = _small_spec(E=1, top_k=1, H=320, inter=192, wfmt=synth.FP8)
    L = synth.make_layer(sp, seed=36)
    x = synth.make_tokens(sp, 2, seed=37)
    r = oracle_mod.moe_forward(L, x)
    Wg = _decode_fp8_independent(L.gate_q[0], L.gate_s[0])
    Wu = _decode_fp8_independent(L.up_q[0], L.up_s[0])
    Wd = _decode_fp8_independent(L.down_q[0], L.down_s[0])
    for n in range(2):
        x64 = _bf16_arr(x[n])
        g, u = Wg @ x64, Wu @ x64
        np.testing.assert_allclose(r["out_f64"][n], Wd @ (g * scipy.special.expit(g) * u),
                                   rtol=1e-12, atol=1e-15)


def test_nvfp4_router_equals_bf16_router_with_the_same_values(oracle_mod):
    """An NVFP4 router (the pages' gate_nvfp4 into the w4a16 GEMV) whose values
    are BF16 numbers (E2M1 x E4M3 x 2) gives the BF16-router layer's routing
    and output to the last bit; its logits match a numpy matmul on the
    test-side decode."""
    import dataclasses
    sp = _small_spec(E=12, top_k=3, H=128, inter=64, router_fmt=synth.NVFP4)
    L = synth.make_layer(sp, seed=41)
    assert L.router.dtype == np.uint8 and L.router.shape == (12, 64) and L.router_s.shape == (12, 8)
    L.router_s2[:] = 2.0
    wr = _decode_fp4_independent(L.router, L.router_s, synth.NVFP4) * 2.0
    bits = synth.f32_to_bf16_bits(wr.astype(np.float32))
    assert np.array_equal(_bf16_arr(bits), wr)
    Lb = dataclasses.replace(L, spec=dataclasses.replace(sp, router_fmt=synth.BF16), router=bits,
                             router_s=None, router_s2=None)
    x = synth.make_tokens(sp, 5, seed=42)
    np.testing.assert_allclose(oracle_mod.layer_router_logits(L, x), _bf16_arr(x) @ wr.T,
                               rtol=1e-13, atol=1e-13)
    r, rb = oracle_mod.moe_forward(L, x), oracle_mod.moe_forward(Lb, x)
    np.testing.assert_array_equal(r["logits"], rb["logits"])
    np.testing.assert_array_equal(r["idx"], rb["idx"])
    np.testing.assert_array_equal(r["out_f64"], rb["out_f64"])


def test_zero_experts_add_nothing(oracle_mod):
    """Zero experts (router width E + Z): slots that select an index >= E run
    no expert.  (a) Zero experts pulled out by their bias: the layer equals
    the same E experts without zero experts (renormalised weights do not see
    the extra softmax terms).  (b) Zero experts pulled in for every slot: only
    the shared expert is left.  (c) A mix: the output is the weighted sum over
    the real-expert slots alone, computed expert by expert."""
    import dataclasses
    sp = _small_spec(E=6, top_k=3, H=96, inter=64, scoring=synth.SOFTMAX_BIAS,
                     zero_experts=4, shared_inter=32, shared_gated=True)
    L = synth.make_layer(sp, seed=51)
    assert L.router.shape == (10, 96) and L.bias.shape == (10,)
    x = synth.make_tokens(sp, 4, seed=52)
    # (a)
    # (the real experts' bias is zero here: the extra softmax terms scale every
    # real score by one factor, which keeps their order only without a bias)
    La = dataclasses.replace(L, bias=L.bias.copy())
    La.bias[:6] = 0.0
    La.bias[6:] = -10.0
    spE = dataclasses.replace(sp, zero_experts=0)
    LE = dataclasses.replace(L, spec=spE, router=L.router[:6].copy(), bias=La.bias[:6].copy())
    ra, rE = oracle_mod.moe_forward(La, x), oracle_mod.moe_forward(LE, x)
    assert ra["logits"].shape == (4, 10) and np.all(ra["idx"] < 6)
    np.testing.assert_array_equal(ra["idx"], rE["idx"])
    np.testing.assert_allclose(ra["out_f64"], rE["out_f64"], rtol=1e-12, atol=1e-15)
    # (b)
    Lb = dataclasses.replace(L, bias=L.bias.copy())
    Lb.bias[6:] = 10.0
    rb = oracle_mod.moe_forward(Lb, x)
    assert np.all(rb["idx"] >= 6)
    for n in range(4):
        d = float(_bf16_arr(L.sh_gate_w) @ _bf16_arr(x[n]))
        ref = scipy.special.expit(d) * _dense_shared(L, _bf16_arr(x[n]))
        np.testing.assert_allclose(rb["out_f64"][n], ref, rtol=1e-12, atol=1e-15)
    # (c)
    Lc = dataclasses.replace(L, bias=L.bias.copy())
    Lc.bias[6:8] = 10.0                      # two of the k = 3 slots are zero experts
    Lc.bias[8:] = -10.0
    rc = oracle_mod.moe_forward(Lc, x)
    for n in range(4):
        assert sum(int(e) >= 6 for e in rc["idx"][n]) == 2
        x64 = _bf16_arr(x[n])
        ref = sum(rc["w"][n, j] * _dense_swiglu(L, int(e), x64)
                  for j, e in enumerate(rc["idx"][n]) if e < 6)
        d = float(_bf16_arr(L.sh_gate_w) @ x64)
        ref = ref + scipy.special.expit(d) * _dense_shared(L, x64)
        np.testing.assert_allclose(rc["out_f64"][n], ref, rtol=1e-11, atol=1e-14)


@pytest.mark.parametrize("scoring", [synth.SOFTMAX, synth.SIGMOID_BIAS, synth.SOFTMAX_BIAS])
def test_hash_routing_with_the_topk_table_equals_topk_routing(oracle_mod, scoring):
    """Hash routing (experts from the tid2eid row of the token's id, weights by
    the layer's scoring): a table whose rows are the tokens' own top-k
    selections reproduces the top-k layer exactly, token ids permuted."""
    import dataclasses
    sp = _small_spec(E=12, top_k=3, H=96, inter=64, scoring=scoring, routed_scaling_factor=1.5)
    L = synth.make_layer(sp, seed=61)
    x = synth.make_tokens(sp, 5, seed=62)
    r = oracle_mod.moe_forward(L, x)
    perm = np.array([3, 0, 4, 1, 2], dtype=np.int32)            # token n has id perm[n]
    table = np.zeros((7, 3), dtype=np.int32)
    table[perm] = r["idx"]
    Lh = dataclasses.replace(L, spec=dataclasses.replace(sp, hash_vocab=7), tid2eid=table)
    rh = oracle_mod.moe_forward(Lh, x, token_ids=perm)
    np.testing.assert_array_equal(rh["idx"], r["idx"])
    np.testing.assert_allclose(rh["w"], r["w"], rtol=1e-15)
    np.testing.assert_array_equal(rh["out_f64"], r["out_f64"])


def test_hash_routing_weights(oracle_mod):
    """Weights of arbitrary table rows: the scoring's scores of those experts
    (softmax over all experts, or sigmoid), renormalised, times the scaling
    factor (not for plain softmax); the order is the table's."""
    import dataclasses
    for scoring, norm in ((synth.SOFTMAX, True), (synth.SOFTMAX, False),
                          (synth.SIGMOID_BIAS, True), (synth.SOFTMAX_BIAS, False)):
        sp = _small_spec(E=10, top_k=4, H=64, inter=32, scoring=scoring, norm_topk_prob=norm,
                         routed_scaling_factor=2.5, hash_vocab=6)
        L = synth.make_layer(sp, seed=63)
        assert L.tid2eid.shape == (6, 4)
        assert all(len(set(r)) == 4 and max(r) < 10 for r in L.tid2eid.tolist())
        x = synth.make_tokens(sp, 3, seed=64)
        ids = np.array([5, 0, 5], dtype=np.int32)
        rh = oracle_mod.moe_forward(L, x, token_ids=ids)
        for n in range(3):
            row = L.tid2eid[ids[n]]
            assert list(rh["idx"][n]) == list(row)
            l = rh["logits"][n]
            s = scipy.special.expit(l) if scoring == synth.SIGMOID_BIAS else scipy.special.softmax(l)
            ref = s[row] / (s[row].sum() if norm else 1.0)
            if scoring != synth.SOFTMAX:
                ref = ref * 2.5
            np.testing.assert_allclose(rh["w"][n], ref, rtol=1e-13)


def test_scale2_scales_each_projection(oracle_mod):
    sp = _small_spec(E=1, top_k=1)
    L = synth.make_layer(sp, seed=13)
    x = synth.make_tokens(sp, 1, seed=14)
    base = oracle_mod.moe_forward(L, x)["out_f64"]
    L.gate_s2[:] = 2.0
    L.up_s2[:] = 0.5
    L.down_s2[:] = 3.0
    # g -> 2g changes SiLU non-linearly; compare with the dense form instead
    ref = _dense_swiglu(L, 0, _bf16_arr(x[0]))
    out = oracle_mod.moe_forward(L, x)["out_f64"][0]
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)
    assert not np.allclose(out, base[0])


@pytest.mark.parametrize("gated", [False, True])
def test_zero_routed_weight_gives_shared_expert_alone(oracle_mod, gated):
    sp = _small_spec(scoring=synth.SIGMOID_BIAS, routed_scaling_factor=0.0,
                     shared_inter=48, shared_gated=gated)
    L = synth.make_layer(sp, seed=15)
    x = synth.make_tokens(sp, 2, seed=16)
    r = oracle_mod.moe_forward(L, x)
    for n in range(2):
        x64 = _bf16_arr(x[n])
        gate = scipy.special.expit(_bf16_arr(L.sh_gate_w) @ x64) if gated else 1.0
        np.testing.assert_allclose(r["out_f64"][n], gate * _dense_shared(L, x64), rtol=1e-12, atol=1e-15)


def test_zero_down_codes_gives_shared_expert_alone(oracle_mod):
    sp = _small_spec(shared_inter=32, shared_gated=False)
    L = synth.make_layer(sp, seed=17)
    L.down_q[:] = 0
    x = synth.make_tokens(sp, 2, seed=18)
    r = oracle_mod.moe_forward(L, x)
    for n in range(2):
        np.testing.assert_allclose(r["out_f64"][n], _dense_shared(L, _bf16_arr(x[n])), rtol=1e-12, atol=1e-15)


def test_weighted_sum_of_experts(oracle_mod):
    """Routed output = sum_j w_j * SwiGLU_{idx_j}(x) with w from the routing."""
    sp = _small_spec(E=6, top_k=3)
    L = synth.make_layer(sp, seed=19)
    x = synth.make_tokens(sp, 2, seed=20)
    r = oracle_mod.moe_forward(L, x)
    for n in range(2):
        x64 = _bf16_arr(x[n])
        ref = sum(r["w"][n, j] * _dense_swiglu(L, r["idx"][n, j], x64) for j in range(3))
        np.testing.assert_allclose(r["out_f64"][n], ref, rtol=1e-12, atol=1e-15)
        p = scipy.special.softmax(_bf16_arr(L.router) @ x64)
        assert list(r["idx"][n]) == _brute_topk(p, 3)


def test_per_token_independence(oracle_mod):
    sp = _small_spec(E=8, top_k=2, shared_inter=32, shared_gated=True)
    L = synth.make_layer(sp, seed=21)
    x = synth.make_tokens(sp, 4, seed=22)
    full = oracle_mod.moe_forward(L, x)
    for n in range(4):
        one = oracle_mod.moe_forward(L, x[n:n + 1])
        np.testing.assert_array_equal(one["out_f64"][0], full["out_f64"][n])
        np.testing.assert_array_equal(one["idx"][0], full["idx"][n])


def test_thread_count_does_not_change_results(oracle_mod):
    """Every output element is summed by one thread in index order, so one
    thread and all threads give the same bits (the benchmark times both)."""
    sp = _small_spec(E=8, top_k=2, shared_inter=32, shared_gated=True)
    L = synth.make_layer(sp, seed=23)
    x = synth.make_tokens(sp, 5, seed=24)
    full = oracle_mod.num_threads()
    ref = oracle_mod.moe_forward(L, x)
    oracle_mod.set_num_threads(1)
    try:
        one = oracle_mod.moe_forward(L, x)
    finally:
        oracle_mod.set_num_threads(full)
    assert oracle_mod.num_threads() == full
    for key in ("out_f64", "idx", "w", "logits"):
        np.testing.assert_array_equal(one[key], ref[key])


def test_expert_permutation_invariance(oracle_mod):
    sp = _small_spec(E=8, top_k=3, scoring=synth.SIGMOID_BIAS, routed_scaling_factor=1.7)
    L = synth.make_layer(sp, seed=23)
    x = synth.make_tokens(sp, 3, seed=24)
    base = oracle_mod.moe_forward(L, x)
    perm = np.random.default_rng(25).permutation(8)          # new slot i holds old expert perm[i]
    import dataclasses
    P = dataclasses.replace(L)
    for name in ("router", "bias", "gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s",
                 "gate_s2", "up_s2", "down_s2"):
        setattr(P, name, np.ascontiguousarray(getattr(L, name)[perm]))
    out = oracle_mod.moe_forward(P, x)
    inv = np.argsort(perm)
    np.testing.assert_array_equal(perm[out["idx"]], base["idx"])
    np.testing.assert_array_equal(inv[base["idx"]], out["idx"])
    np.testing.assert_array_equal(out["out_f64"], base["out_f64"])


def test_margin_rows_have_margin(oracle_mod):
    from oracle import margin
    sp = synth.CONFIGS["tiny"]
    L = synth.make_layer(sp)
    x = margin.tokens_with_margin(L, 3)
    keys = margin.selection_keys(L, x)
    for n in range(3):
        assert margin.topk_gap(keys[n], sp.top_k) >= margin.MARGIN


def test_softmax_weights_ignore_routed_scaling_factor(oracle_mod):
    """Reading: the softmax top-k op is not given the routed scaling factor."""
    rng = np.random.default_rng(26)
    logits = rng.standard_normal((3, 16))
    _, w1, _ = oracle_mod.route(logits, 4, "softmax", True, 1.0)
    _, w2, _ = oracle_mod.route(logits, 4, "softmax", True, 2.5)
    np.testing.assert_array_equal(w1, w2)
