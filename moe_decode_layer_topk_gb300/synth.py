"""Seeded synthetic inputs for the MoE decode layer (shared by the CUDA path's
tests/bench and by the FP64 oracle).

This module only *builds input bytes*: it draws Gaussian tensors with numpy's
PCG64 generator and encodes them into the storage formats the layer reads
(BF16, E2M1 codes with E4M3 or E8M0 block scales).  It contains none of the
layer's arithmetic (no router, routing, decode, GEMV or blend); both the GPU
path and the oracle consume the bytes produced here.

Workload shapes follow the five layer shapes the method is run on (tiny,
Qwen3-30B-A3B, MTP verify with a gated shared expert, DeepSeek-V3 with an
always-on shared expert, gpt-oss-120b MXFP4).  The expert formats are the two
the pages name: NVFP4 (E2M1 + per-16 E4M3 scale + per-tensor FP32 "scale2")
and MXFP4 (E2M1 + per-32 E8M0 scale), see forward_k3.rs (the E8M0 guard above
the GS16 batch3 kernel) and forward_batched.rs (the `_e8m0` kernel choice).

Expert pool: drawing every expert of a 256-expert DeepSeek-V3 layer means
11.3e9 normals; instead ``pool`` experts per projection are drawn and
quantised exactly per recipe, and expert slot ``e`` holds a copy of pool entry
``src[e]`` whose rows are sign-flipped by a seeded per-(slot,row) mask.  Each
slot is distinct, the value distribution is unchanged (the Gaussian and both
encodings are symmetric), and each slot occupies its own HBM bytes.  With
``pool >= E`` every expert is an independent draw.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

NVFP4 = "nvfp4"
MXFP4 = "mxfp4"
BF16 = "bf16"
FP8 = "fp8"
FP8_BLOCK = 128   # FP8 experts: one FP32 scale per 128 x 128 block
SOFTMAX = "softmax"
SIGMOID_BIAS = "sigmoid_bias"
SOFTMAX_BIAS = "softmax_bias"   # softmax scores + correction bias for selection


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    name: str
    H: int
    inter: int
    E: int
    top_k: int
    scoring: str            # SOFTMAX | SIGMOID_BIAS | SOFTMAX_BIAS
    norm_topk_prob: bool
    routed_scaling_factor: float
    wfmt: str               # NVFP4 | MXFP4 | BF16 | FP8
    shared_inter: int       # 0 = no shared expert
    shared_gated: bool      # sigmoid(w_s . x) gate on the shared expert
    x_rms_norm: bool        # x rows RMS-normalised before the BF16 cast
    tokens: tuple           # token counts the layer is run at
    pool: int               # distinct experts drawn per projection
    router_fmt: str = BF16  # BF16 router, or NVFP4 (E2M1 + per-16 E4M3 + scale2)
    zero_experts: int = 0   # Z extra router outputs whose expert adds nothing
    hash_vocab: int = 0     # V > 0: hash routing, experts from a [V, top_k] token-id table

    @property
    def gs(self) -> int:
        """Block-scale group size along K (0 for BF16 experts, which have no
        scales; FP8 blocks are 128 x 128)."""
        return {NVFP4: 16, MXFP4: 32, BF16: 0, FP8: FP8_BLOCK}[self.wfmt]

    def expert_bytes(self) -> int:
        """Bytes of one routed expert (gate+up+down packed codes + block scales,
        BF16 words, or E4M3 bytes + FP32 block scales)."""
        if self.wfmt == BF16:
            return 3 * self.inter * self.H * 2
        if self.wfmt == FP8:
            nb = -(-self.inter // FP8_BLOCK) * -(-self.H // FP8_BLOCK)
            return 3 * self.inter * self.H + 3 * nb * 4
        return 3 * self.inter * self.H // 2 + 3 * self.inter * self.H // self.gs

    def router_bytes(self) -> int:
        R = self.E + self.zero_experts
        if self.router_fmt == NVFP4:
            return R * self.H // 2 + R * self.H // 16
        return R * self.H * 2

    def shared_bytes(self) -> int:
        return 3 * self.shared_inter * self.H * 2


# The five layer shapes (sizes, routing and input distributions per workload).
CONFIGS = {
    "tiny": LayerSpec("tiny", 256, 128, 8, 2, SOFTMAX, True, 1.0, NVFP4,
                      0, False, False, (1,), 8),
    "qwen3_30b_a3b": LayerSpec("qwen3_30b_a3b", 2048, 768, 128, 8, SOFTMAX, True, 1.0,
                               NVFP4, 0, False, True, (1, 2, 3, 4), 16),
    "mtp_verify": LayerSpec("mtp_verify", 2048, 512, 512, 10, SOFTMAX, True, 1.0, NVFP4,
                            512, True, True, (3,), 16),
    "deepseek_v3": LayerSpec("deepseek_v3", 7168, 2048, 256, 8, SIGMOID_BIAS, True, 2.5,
                             NVFP4, 2048, False, True, (4,), 4),
    # "softmax over the selected top-k" == softmax over E then renormalise.
    "gpt_oss_120b": LayerSpec("gpt_oss_120b", 2880, 2880, 128, 4, SOFTMAX, True, 1.0,
                              MXFP4, 0, False, False, (1, 2, 3, 4, 8, 16, 32, 64, 512), 8),
    # BF16 routed experts (the pages' third expert format) on the Qwen3 shape.
    "qwen3_30b_a3b_bf16": LayerSpec("qwen3_30b_a3b_bf16", 2048, 768, 128, 8, SOFTMAX, True,
                                    1.0, BF16, 0, False, True, (1, 2, 3, 4), 16),
    # FP8 block-scaled routed experts on the Qwen3 shape.
    "qwen3_30b_a3b_fp8": LayerSpec("qwen3_30b_a3b_fp8", 2048, 768, 128, 8, SOFTMAX, True,
                                   1.0, FP8, 0, False, True, (1, 2, 3, 4), 16),
    # Zero-expert routing (router of width E + Z, softmax + correction bias)
    # on the Qwen3 shape: 128 experts and 64 zero experts.
    "qwen3_30b_a3b_zero_experts": LayerSpec("qwen3_30b_a3b_zero_experts", 2048, 768, 128, 8,
                                            SOFTMAX_BIAS, True, 1.0, NVFP4, 0, False, True,
                                            (1, 2, 3, 4), 16, BF16, 64),
    # NVFP4-quantised router on the Qwen3 shape.
    "qwen3_30b_a3b_nvfp4_router": LayerSpec("qwen3_30b_a3b_nvfp4_router", 2048, 768, 128, 8,
                                            SOFTMAX, True, 1.0, NVFP4, 0, False, True,
                                            (1, 2, 3, 4), 16, NVFP4),
}
CONFIG_INDEX = {"tiny": 0, "qwen3_30b_a3b": 1, "mtp_verify": 2, "deepseek_v3": 3,
                "gpt_oss_120b": 4, "qwen3_30b_a3b_bf16": 5, "qwen3_30b_a3b_fp8": 6,
                "qwen3_30b_a3b_nvfp4_router": 7, "qwen3_30b_a3b_zero_experts": 8}


def base_seed(spec: LayerSpec) -> int:
    return 1000 + CONFIG_INDEX.get(spec.name, 99)


# ----------------------------------------------------------------------------
# Encoders (value -> storage bytes).  Inputs only; decode lives on each side.
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest BF16 (ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def encode_e2m1(v: np.ndarray) -> np.ndarray:
    """Round to the nearest E2M1 magnitude (ties to even code), saturate at 6.

    Grid 0,0.5,1,1.5,2,3,4,6 (codes 0..7); bit 3 is the sign.  A magnitude that
    rounds to 0 gets code 0 (no negative zero)."""
    a = np.abs(v)
    code = ((a > 0.25).astype(np.uint8) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
            + (a > 2.5) + (a >= 3.5) + (a > 5.0)).astype(np.uint8)
    neg = (v < 0) & (code != 0)
    return code | (neg.astype(np.uint8) << np.uint8(3))


def encode_e4m3(v: np.ndarray) -> np.ndarray:
    """Non-negative float -> E4M3 (OCP 'fn', bias 7), nearest-even, saturating at 448."""
    v = np.minimum(np.asarray(v, dtype=np.float64), 448.0)
    out = np.zeros(v.shape, dtype=np.uint8)
    sub = v < 2.0 ** -6
    # subnormal grid m * 2^-9 (m = 8 lands exactly on the smallest normal, code 8)
    out[sub] = np.rint(v[sub] * 2.0 ** 9).astype(np.uint8)
    nv = v[~sub]
    mant, ex = np.frexp(nv)                 # nv = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1                              # nv = (2*mant) * 2^e, 2*mant in [1, 2)
    m = np.rint((2.0 * mant - 1.0) * 8.0)   # ties to even
    carry = m >= 8
    e = np.where(carry, e + 1, e)
    m = np.where(carry, 0, m)
    code = ((e + 7) << 3).astype(np.int64) + m.astype(np.int64)
    out[~sub] = np.minimum(code, 0x7E).astype(np.uint8)
    return out


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[..., K] uint8 codes -> [..., K/2] bytes; element 2j low nibble, 2j+1 high."""
    c = codes.reshape(codes.shape[:-1] + (codes.shape[-1] // 2, 2))
    return (c[..., 0] | (c[..., 1] << np.uint8(4))).astype(np.uint8)


def quantize_nvfp4(w: np.ndarray, scale2: float = 1.0):
    """[rows, K] float32 -> (packed [rows, K/2], E4M3 scales [rows, K/16]).

    Per 16 consecutive elements along K: s = E4M3(amax/6/scale2); codes are
    E2M1(w / (s*scale2)); an all-zero scale zeroes the block."""
    rows, K = w.shape
    blk = w.reshape(rows, K // 16, 16).astype(np.float32)
    amax = np.abs(blk).max(axis=-1)
    s_code = encode_e4m3(amax / 6.0 / scale2)
    s_val = _e4m3_grid()[s_code] * scale2
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(s_val[..., None] > 0, blk / s_val[..., None], 0.0)
    codes = encode_e2m1(ratio).reshape(rows, K)
    return pack_nibbles(codes), s_code


def quantize_mxfp4(w: np.ndarray):
    """[rows, K] float32 -> (packed [rows, K/2], E8M0 scales [rows, K/32]).

    Per 32 elements: X = 2^(floor(log2 amax) - 2) (emax of E2M1 is 2), codes are
    E2M1(w / X) saturated to +-6; amax == 0 gives X = 2^-127 and zero codes."""
    rows, K = w.shape
    blk = w.reshape(rows, K // 32, 32).astype(np.float64)
    amax = np.abs(blk).max(axis=-1)
    with np.errstate(divide="ignore"):
        ex = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, -127)
    ex = np.clip(ex, -127, 127)
    s_code = (ex + 127).astype(np.uint8)
    x = np.ldexp(1.0, ex.astype(np.int64))
    codes = encode_e2m1(blk / x[..., None]).reshape(rows, K)
    return pack_nibbles(codes), s_code


def quantize_fp8_block(w: np.ndarray):
    """[rows, K] float32 -> (E4M3 bytes [rows, K], FP32 scales [ceil(rows/128),
    ceil(K/128)]).

    Per 128 x 128 block: s = amax / 448 (FP32), codes E4M3(w / s) with the
    sign in bit 7, nearest even, saturating at 448; an all-zero block gets
    s = 1 and zero codes."""
    rows, K = w.shape
    B = FP8_BLOCK
    nr, nk = -(-rows // B), -(-K // B)
    s = np.ones((nr, nk), dtype=np.float32)
    q = np.zeros((rows, K), dtype=np.uint8)
    for i in range(nr):
        for j in range(nk):
            blk = w[i * B:(i + 1) * B, j * B:(j + 1) * B].astype(np.float32)
            amax = float(np.abs(blk).max()) if blk.size else 0.0
            if amax > 0:
                s[i, j] = np.float32(amax / 448.0)
            r = blk.astype(np.float64) / np.float64(s[i, j])
            code = encode_e4m3(np.abs(r))
            neg = (r < 0) & (code != 0)
            q[i * B:(i + 1) * B, j * B:(j + 1) * B] = code | (neg.astype(np.uint8) << np.uint8(7))
    return q, s


_E4M3_GRID = None


def _e4m3_grid() -> np.ndarray:
    """Value of every E4M3 code, used only to divide by the chosen scale when
    encoding (the quantiser needs the scale it picked)."""
    global _E4M3_GRID
    if _E4M3_GRID is None:
        g = np.zeros(256)
        for c in range(256):
            e, m = (c >> 3) & 15, c & 7
            mag = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
            g[c] = -mag if c & 0x80 else mag
        g[0x7F] = g[0xFF] = np.nan
        _E4M3_GRID = g
    return _E4M3_GRID


# ----------------------------------------------------------------------------
# Layer and token generation
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class HostLayer:
    """Host-resident input bytes of one MoE layer (numpy arrays)."""
    spec: LayerSpec
    router: np.ndarray            # uint16 [E, H] BF16 bits
    bias: Optional[np.ndarray]    # float32 [E] or None
    gate_q: np.ndarray            # uint8 [E, inter, H/2] (BF16: uint16 [E, inter, H]; FP8: uint8 [E, inter, H])
    up_q: np.ndarray
    down_q: np.ndarray            # uint8 [E, H, inter/2] (BF16: uint16 [E, H, inter]; FP8: uint8 [E, H, inter])
    gate_s: Optional[np.ndarray]  # uint8 [E, inter, H/gs] (None for BF16; FP8: float32 [E, inter/128, H/128])
    up_s: Optional[np.ndarray]
    down_s: Optional[np.ndarray]  # uint8 [E, H, inter/gs] (FP8: float32 [E, H/128, inter/128])
    gate_s2: Optional[np.ndarray]  # float32 [E] (NVFP4) or None (MXFP4)
    up_s2: Optional[np.ndarray]
    down_s2: Optional[np.ndarray]
    sh_gate: Optional[np.ndarray]  # uint16 [inter_s, H]
    sh_up: Optional[np.ndarray]
    sh_down: Optional[np.ndarray]  # uint16 [H, inter_s]
    sh_gate_w: Optional[np.ndarray]  # uint16 [H] or None
    router_s: Optional[np.ndarray] = None   # NVFP4 router: uint8 E4M3 [E, H/16] (router: uint8 [E, H/2])
    router_s2: Optional[np.ndarray] = None  # NVFP4 router: float32 [1]
    tid2eid: Optional[np.ndarray] = None    # hash routing: int32 [V, top_k]

    def tensors(self):
        return {k: getattr(self, k) for k in (
            "router", "bias", "gate_q", "up_q", "down_q", "gate_s", "up_s", "down_s",
            "gate_s2", "up_s2", "down_s2", "sh_gate", "sh_up", "sh_down", "sh_gate_w",
            "router_s", "router_s2", "tid2eid")}


def _quantize(spec: LayerSpec, w: np.ndarray):
    if spec.wfmt == BF16:
        return f32_to_bf16_bits(w), None
    if spec.wfmt == FP8:
        return quantize_fp8_block(w)
    return quantize_nvfp4(w) if spec.wfmt == NVFP4 else quantize_mxfp4(w)


def _expert_projection(spec, rng, rows, K, pool, E):
    """Draw `pool` experts [rows, K] ~ N(0, 0.02), quantise (or round to BF16),
    and fill E slots."""
    qs, ss = [], []
    for _ in range(pool):
        w = rng.standard_normal((rows, K), dtype=np.float32) * np.float32(0.02)
        q, s = _quantize(spec, w)
        qs.append(q)
        ss.append(s)
    qp = np.stack(qs)
    sp = None if ss[0] is None else np.stack(ss)
    if pool >= E:
        return qp[:E].copy(), None if sp is None else sp[:E].copy()
    src = rng.integers(0, pool, size=E)
    src[:pool] = np.arange(pool)            # every pool entry is used
    flip = rng.random((E, rows)) < 0.5
    flip[:pool] = False
    q = qp[src]
    if spec.wfmt == BF16:                    # sign bit of every BF16 word of the row
        q ^= (flip.astype(np.uint16) * np.uint16(0x8000))[..., None]
    elif spec.wfmt == FP8:                   # sign bit of every E4M3 byte of the row
        q ^= (flip.astype(np.uint8) * np.uint8(0x80))[..., None]
    else:                                    # sign bits of both E2M1 codes of each byte
        q ^= (flip.astype(np.uint8) * np.uint8(0x88))[..., None]
    return q, None if sp is None else sp[src].copy()


def make_layer(spec: LayerSpec, seed: Optional[int] = None, pool: Optional[int] = None) -> HostLayer:
    seed = base_seed(spec) if seed is None else seed
    pool = min(spec.E, spec.pool if pool is None else pool)
    rng = np.random.default_rng(seed)
    H, I, E = spec.H, spec.inter, spec.E
    R = E + spec.zero_experts    # router width
    router_w = rng.standard_normal((R, H), dtype=np.float32) * np.float32(1.0 / np.sqrt(H))
    router_s = router_s2 = None
    if spec.router_fmt == NVFP4:
        router, router_s = quantize_nvfp4(router_w)
        router_s2 = np.ones(1, dtype=np.float32)
    else:
        router = f32_to_bf16_bits(router_w)
    bias = None
    if spec.scoring == SIGMOID_BIAS:
        bias = (rng.standard_normal(R, dtype=np.float32) * np.float32(0.1)).astype(np.float32)
    elif spec.scoring == SOFTMAX_BIAS:
        # on the scale of the softmax scores (about 1/R each)
        bias = (rng.standard_normal(R, dtype=np.float32) * np.float32(0.5 / R)).astype(np.float32)
    gate_q, gate_s = _expert_projection(spec, rng, I, H, pool, E)
    up_q, up_s = _expert_projection(spec, rng, I, H, pool, E)
    down_q, down_s = _expert_projection(spec, rng, H, I, pool, E)
    s2 = np.ones(E, dtype=np.float32) if spec.wfmt == NVFP4 else None   # MXFP4, BF16: none
    sh_gate = sh_up = sh_down = sh_gate_w = None
    if spec.shared_inter:
        Is = spec.shared_inter
        sh_gate = f32_to_bf16_bits(rng.standard_normal((Is, H), dtype=np.float32) * np.float32(0.02))
        sh_up = f32_to_bf16_bits(rng.standard_normal((Is, H), dtype=np.float32) * np.float32(0.02))
        sh_down = f32_to_bf16_bits(rng.standard_normal((H, Is), dtype=np.float32) * np.float32(0.02))
        if spec.shared_gated:
            sh_gate_w = f32_to_bf16_bits(rng.standard_normal(H, dtype=np.float32)
                                         * np.float32(1.0 / np.sqrt(H)))
    tid2eid = None
    if spec.hash_vocab > 0:   # k distinct experts per token id, uniformly drawn
        tid2eid = np.stack([rng.permutation(E)[:spec.top_k]
                            for _ in range(spec.hash_vocab)]).astype(np.int32)
    return HostLayer(spec, router, bias, gate_q, up_q, down_q, gate_s, up_s, down_s,
                     s2, None if s2 is None else s2.copy(), None if s2 is None else s2.copy(),
                     sh_gate, sh_up, sh_down, sh_gate_w, router_s, router_s2, tid2eid)


def x_row(spec: LayerSpec, seed: int, row: int, attempt: int = 0) -> np.ndarray:
    """One token's activation row as BF16 bits (uint16 [H]).

    Drawn N(0,1) from the sub-seed (seed, row, attempt); RMS-normalised
    (x / sqrt(mean(x^2) + 1e-6), no weight) for the shapes whose input is the
    normed MoE input."""
    rng = np.random.default_rng([seed, row, attempt])
    x = rng.standard_normal(spec.H).astype(np.float64)
    if spec.x_rms_norm:
        x = x / np.sqrt(np.mean(x * x) + 1e-6)
    return f32_to_bf16_bits(x.astype(np.float32))


def make_tokens(spec: LayerSpec, N: int, seed: Optional[int] = None, attempts=None) -> np.ndarray:
    """x [N, H] BF16 bits; ``attempts[n]`` selects the redraw of row n."""
    seed = (base_seed(spec) + N) if seed is None else seed
    attempts = attempts if attempts is not None else [0] * N
    if N == 0:
        return np.zeros((0, spec.H), dtype=np.uint16)
    return np.stack([x_row(spec, seed, n, attempts[n]) for n in range(N)])

