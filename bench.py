"""Benchmark of the MoE decode-layer forward on one GB300 (or N replicas).

Workload: the Qwen3-30B-A3B-shaped layer (H 2048, inter 768, 128 NVFP4
experts, top-8 softmax with renormalisation) at N = 1, 2, 3, 4 tokens.  One
step = four moe_forward calls, N = 1, 2, 3, 4, on one layer copy; step s runs
on copy s mod R (L2 defeat: one round of copies touches many times the
129 MB L2).  The metric is the achieved HBM rate over algorithmic bytes:
    bytes(call) = U * expert_bytes + router_bytes + shared_bytes + x/out bytes
with U the number of distinct routed experts the call's tokens touched (read
back from the routing outputs before timing).  value = sum of bytes / time.

Timed region: exactly --steps steps after exactly --warmup untimed ones, each
step a replay of its copy's captured CUDA graph, bracketed by a barrier and
torch.cuda.synchronize(), CUDA events on the launch stream; the maximum over
ranks is taken.  "per_n" gives each token count's latency (median of five
repeats of a round-robin loop) and "per_n_l2_flush" the same from single
calls after an L2-sized buffer write.  "configs" holds every layer shape of
the workload list at its token counts (the small layer, Qwen3 N=1-4,
MTP-verify N=3, DeepSeek-V3 N=4, gpt-oss N=1-64 and N=512 on the grouped
tcgen05 path); "bf16_experts", "fp8_experts", "nvfp4_router" and
"zero_experts" the Qwen3 shape with BF16 or FP8 routed experts, an NVFP4
router, or 64 zero experts; all timed on the same GPU after the main
measurement.  --impl reference times the FP64 CPU oracle on a bounded sample
of the same workload instead; "cpu_baseline" also holds the oracle's
single-thread per-call times.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAK_FALLBACK_GBS = 6800.0
PER_N_REPEATS = 5   # per-N latency: median over this many repeats of the timed loop
NOMINAL_HBM_GBS = 8000.0
METRIC = "MoE layer us and expert-weight HBM GB/s (fraction of 8 TB/s) at N=1-4 tokens"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback"


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device="cuda") -> float:
    """The largest x over all ranks of the initialised process group (the
    timed region's length is the slowest replica's); x itself when world == 1."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(bytes_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every replica moves bytes_per_rank in the timed
    region, whose length is the maximum over ranks (ms)."""
    return bytes_per_rank * world / (ms / 1e3) / 1e9


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if not self.path or not os.path.exists(self.path):
            return out
        sms, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if sms:
            out.update(sm_mhz=float(np.median(sms)), sm_max_mhz=float(max(mx)),
                       reasons=sorted(reasons), samples=len(sms))
        return out


def algorithmic_bytes(spec, idx: np.ndarray, N: int) -> dict:
    """Bytes one call must move: touched routed experts, router, shared expert,
    x in and out."""
    U = len(np.unique(idx[idx < spec.E]))   # zero experts (index >= E) read no weights
    routed = U * spec.expert_bytes()
    other = spec.router_bytes() + spec.shared_bytes() + 2 * N * spec.H * 2
    return {"U": U, "routed": routed, "total": routed + other}


def stream_traffic(calls):
    """DRAM bytes per stream-kernel launch from the committed ncu record
    (profiles/traffic.json), or None when the kernel source changed since the
    counters were taken.  Calls whose token count has no capture are scaled
    from the captured ones by algorithmic bytes (mean traffic/algorithmic
    ratio of the captured launches)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))
        src = os.path.join(ROOT, rec["kernel_source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except (OSError, ValueError, KeyError):
        return None, "no record"
    if rec.get("kernel_source_sha256") != h:
        return None, f"{rec['kernel_source']} changed since the ncu capture"
    meas, alg = rec["dram_bytes_per_launch"], rec["algorithmic_bytes_per_launch"]
    ratio = float(np.mean([meas[k] / alg[k] for k in meas]))
    tot = sum(ratio * c[5]["total"] for c in calls)
    note = f"ncu dram read+write (profiles/traffic.json) = {ratio:.4f} x algorithmic bytes"
    return tot / len(calls), note


def kernels_per_call(spec, N: int) -> int:
    """Kernels one moe_forward enqueues, as the library reports its path: one
    fused kernel (the stream or the decode kernel), or the grouped chain
    (router, top-k, plan, gather, gate/up GEMM, pack, down GEMM, combine)."""
    from moe_decode_layer_topk_gb300 import _lib
    from moe_decode_layer_topk_gb300.device import layer_desc
    g = _lib.moe_uses_grouped_path(layer_desc(spec), N)
    if g < 0:
        raise ValueError(f"invalid layer or token count: {spec.name}, N={N}")
    return 8 if g else 1


def measure_grouped(stream, name: str = "gpt_oss_120b", N: int = 512, reps: int = 10) -> dict:
    """The grouped many-token path (tcgen05 GEMMs) on its headline workload:
    one layer (1.69 GB of MXFP4 experts, far above L2, so every call streams
    the weights from HBM), N tokens, CUDA-graph replays timed with events."""
    import torch
    from moe_decode_layer_topk_gb300 import _lib, synth
    from moe_decode_layer_topk_gb300.device import DeviceLayer, bf16_tensor, workspace
    spec = synth.CONFIGS[name]
    dev = DeviceLayer.upload(synth.make_layer(spec))
    x = bf16_tensor(synth.make_tokens(spec, N, seed=90512))
    out = torch.empty_like(x)
    ws = workspace(spec, N)
    idx = torch.empty((N, spec.top_k), dtype=torch.int32, device="cuda")
    _lib.moe_forward(dev.desc, dev.weights, x, out, ws, idx)
    torch.cuda.synchronize()
    b = algorithmic_bytes(spec, idx.cpu().numpy(), N)
    with torch.cuda.stream(stream):
        for _ in range(3):
            _lib.moe_forward(dev.desc, dev.weights, x, out, ws, stream=stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        _lib.moe_forward(dev.desc, dev.weights, x, out, ws, stream=stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    assert _lib.moe_get_error(ws) == _lib.MOE_OK
    us = e0.elapsed_time(e1) * 1e3 / reps
    flops = 2.0 * N * spec.top_k * 3 * spec.H * spec.inter
    peak, _ = _peaks()
    del dev, ws
    torch.cuda.empty_cache()
    return {"workload": f"{name} layer at N={N} (grouped tcgen05 path)", "us_per_layer": round(us, 2),
            "tokens_per_s": round(N / us * 1e6, 1), "U": b["U"], "bytes": int(b["total"]),
            "GBps": round(b["total"] / us / 1e3, 1),
            "hbm_frac_of_measured": round(b["total"] / us / 1e3 / peak, 4),
            "tensor_tflops": round(flops / us / 1e6, 2), "launches_per_call": kernels_per_call(spec, N),
            "reps": reps}


def layer_bytes(spec) -> int:
    """Device bytes of one copy of the layer's weights."""
    return spec.E * spec.expert_bytes() + spec.router_bytes() + spec.shared_bytes()


def measure_config(stream, name: str, tokens, l2_bytes: int, max_copies: int = 16,
                   reps: int = 200) -> dict:
    """Latency of one layer shape at each token count: enough device copies of
    the layer (each with its own token rows) that a round of calls touches
    about three times the L2, replayed round-robin from one CUDA graph, so
    consecutive calls read different weight bytes; the median of five timed
    loops.  A layer too small for that (the tiny shape) stays L2-resident, and
    the record says so."""
    import torch
    from moe_decode_layer_topk_gb300 import _lib, synth
    from moe_decode_layer_topk_gb300.device import DeviceLayer, bf16_tensor, workspace
    spec = synth.CONFIGS[name]
    peak, _ = _peaks()
    lb = layer_bytes(spec)
    base = DeviceLayer.upload(synth.make_layer(spec))
    res = {}
    devs = [base]
    for N in tokens:
        touched = min(spec.E, N * spec.top_k) * spec.expert_bytes() + spec.router_bytes() + \
            spec.shared_bytes()
        copies = max(2, min(max_copies, -(-3 * l2_bytes // touched), (48 << 30) // lb))
        while len(devs) < copies:
            devs.append(base.clone())
        calls = []
        for i, dev in enumerate(devs[:copies]):
            x = bf16_tensor(synth.make_tokens(spec, N, seed=77000 + 97 * N + i))
            out, ws = torch.empty_like(x), workspace(spec, N)
            idx = torch.empty((N, spec.top_k), dtype=torch.int32, device="cuda")
            _lib.moe_forward(dev.desc, dev.weights, x, out, ws, idx)
            calls.append((dev, x, out, ws, algorithmic_bytes(spec, idx.cpu().numpy(), N)))
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for dev, x, out, ws, _ in calls:
                _lib.moe_forward(dev.desc, dev.weights, x, out, ws, stream=stream)
        rounds = max(1, reps // len(calls))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        rep_us = []
        for _ in range(PER_N_REPEATS):
            with torch.cuda.stream(stream):
                g.replay()
                e0.record(stream)
                for _ in range(rounds):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            rep_us.append(e0.elapsed_time(e1) * 1e3 / (rounds * len(calls)))
        for c in calls:
            assert _lib.moe_get_error(c[3]) == _lib.MOE_OK
        us = float(np.median(rep_us))
        b = float(np.mean([c[4]["total"] for c in calls]))
        round_bytes = sum(c[4]["total"] for c in calls)
        res[str(N)] = {"us_per_layer": round(us, 3), "tokens_per_s": round(N / us * 1e6, 1),
                       "GBps": round(b / us / 1e3, 1),
                       "hbm_frac_of_measured": round(b / us / 1e3 / peak, 4),
                       "U_mean": float(np.mean([c[4]["U"] for c in calls])), "bytes_mean": int(b),
                       "copies": copies, "l2_resident": bool(round_bytes < l2_bytes),
                       "launches_per_call": kernels_per_call(spec, N),
                       "us_repeats": [round(u, 3) for u in rep_us]}
        del calls, g
    del devs, base
    torch.cuda.empty_cache()
    return {"workload": f"{name} layer: H {spec.H}, inter {spec.inter}, E {spec.E}, top-{spec.top_k}, "
                        f"{spec.wfmt} experts" + (f", shared inter {spec.shared_inter}"
                                                  if spec.shared_inter else ""),
            "per_n": res}


def measure_all_configs(stream, l2_bytes: int) -> dict:
    """Every layer shape of the workload list at its token counts: the small
    layer (N=1), the Qwen3 shape (N=1-4), the MTP-verify layer (N=3), the
    DeepSeek-V3 shape (N=4) and the gpt-oss shape (N=1-64 on the fused
    kernels, N=512 on the grouped path)."""
    from moe_decode_layer_topk_gb300 import synth
    out = {}
    for name in ("tiny", "qwen3_30b_a3b", "mtp_verify", "deepseek_v3", "gpt_oss_120b"):
        spec = synth.CONFIGS[name]
        toks = [n for n in spec.tokens if n <= 64]
        out[name] = measure_config(stream, name, toks, l2_bytes)
        big = [n for n in spec.tokens if n > 64]
        for n in big:
            out[name]["per_n"][str(n)] = measure_grouped(stream, name, n)
    return out


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from moe_decode_layer_topk_gb300 import _lib, synth
    from moe_decode_layer_topk_gb300.device import DeviceLayer, bf16_tensor, workspace

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    spec = synth.CONFIGS[args.config]
    tokens = [n for n in spec.tokens if n <= 64] if args.tokens is None else args.tokens
    base = DeviceLayer.upload(synth.make_layer(spec))
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    R = args.copies
    copies = [base] + [base.clone() for _ in range(R - 1)]
    stream = torch.cuda.Stream()
    maxN = max(tokens)
    calls = []   # [layer copy, N, x, out, ws, bytes]
    for r in range(R):
        for N in tokens:
            x = bf16_tensor(synth.make_tokens(spec, N, seed=90000 + 1000 * rank + 17 * r + N))
            calls.append([copies[r], N, x, torch.empty_like(x), workspace(spec, maxN)])
    # routing of every call (untimed) to count its algorithmic bytes
    per_cycle_bytes = 0
    for c in calls:
        dev, N, x, out, ws = c
        idx = torch.empty((N, spec.top_k), dtype=torch.int32, device="cuda")
        w = torch.empty((N, spec.top_k), dtype=torch.float32, device="cuda")
        _lib.moe_forward(dev.desc, dev.weights, x, out, ws, idx, w)
        torch.cuda.synchronize()
        c.append(algorithmic_bytes(spec, idx.cpu().numpy(), N))
        per_cycle_bytes += c[-1]["total"]
    for c in calls:
        assert _lib.moe_get_error(c[4]) == _lib.MOE_OK
    launches_per_cycle = len(calls)
    kernels_per_cycle = sum(kernels_per_call(spec, c[1]) for c in calls)
    ntok = len(tokens)

    # one step = the N sweep on one layer copy; step s uses copy s mod R, so
    # consecutive steps read different weight bytes
    def enqueue_step(r):
        for dev, N, x, out, ws, _ in calls[r * ntok:(r + 1) * ntok]:
            _lib.moe_forward(dev.desc, dev.weights, x, out, ws, stream=stream)

    graphs = None
    if not args.no_graph:
        with torch.cuda.stream(stream):
            for r in range(R):
                enqueue_step(r)
        stream.synchronize()
        graphs = []
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                enqueue_step(r)
            graphs.append(g)

    def run_step(s_):
        if graphs is not None:
            graphs[s_ % R].replay()
        else:
            enqueue_step(s_ % R)

    with torch.cuda.stream(stream):
        for s_ in range(args.warmup):
            run_step(s_)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for s_ in range(args.warmup, args.warmup + args.steps):
                run_step(s_)
            ev1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    for c in calls:
        assert _lib.moe_get_error(c[4]) == _lib.MOE_OK, "device-side wait expired during timing"
    steps = args.steps
    step_bytes = [sum(c[5]["total"] for c in calls[r * ntok:(r + 1) * ntok]) for r in range(R)]
    timed_bytes = sum(step_bytes[s_ % R] for s_ in range(args.warmup, args.warmup + steps))
    value = job_gbps(timed_bytes, world, ms)
    launches = steps * ntok
    avg_launch_us = ms * 1e3 / launches
    achieved = timed_bytes / launches / (avg_launch_us * 1e-6) / 1e9
    kernels_timed = sum(kernels_per_call(spec, N) for N in tokens) * steps

    # per-token-count latency (separate loop after the timed region)
    per_n = {}
    for N in tokens:
        sub = [c for c in calls if c[1] == N]
        reps = max(32, min(args.steps, 400))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g = None
        if not args.no_graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for dev, n_, x, out, ws, _ in sub:
                    _lib.moe_forward(dev.desc, dev.weights, x, out, ws, stream=stream)
        rounds = max(1, reps // len(sub))
        rep_us = []
        for _ in range(PER_N_REPEATS):
            with torch.cuda.stream(stream):
                if g is not None:
                    g.replay()
                e0.record(stream)
                for _ in range(rounds):
                    if g is not None:
                        g.replay()
                    else:
                        for dev, n_, x, out, ws, _ in sub:
                            _lib.moe_forward(dev.desc, dev.weights, x, out, ws, stream=stream)
                e1.record(stream)
            torch.cuda.synchronize()
            rep_us.append(e0.elapsed_time(e1) * 1e3 / (rounds * len(sub)))
        us = float(np.median(rep_us))
        b = float(np.mean([c[5]["total"] for c in sub]))
        br = float(np.mean([c[5]["routed"] for c in sub]))
        per_n[str(N)] = {"us_per_layer": round(us, 3),
                         "us_repeats": [round(u, 3) for u in rep_us],
                         "calls_per_repeat": rounds * len(sub),
                         "tokens_per_s": round(N / us * 1e6, 1),
                         "GBps": round(b / us / 1e3, 1),
                         "frac_of_8TBs": round(b / us / 1e3 / NOMINAL_HBM_GBS, 4),
                         "U_mean": float(np.mean([c[5]["U"] for c in sub])),
                         "bytes_mean": int(b), "routed_bytes_mean": int(br)}

    # cross-check of the L2 defeat: one call at a time on layer copy 0 after
    # writing a buffer twice the L2 size (so nothing of the call is cached)
    per_n_flush = None
    if rank == 0 and not args.no_l2_flush:
        per_n_flush = l2_flush_latency(stream, calls, tokens, l2)

    # end to end through the host-buffer entry point (pinned host x / out)
    e2e = None
    if rank == 0 and not args.no_e2e:
        wsh = workspace(spec, maxN, host_staging=True)
        hx = [calls[i][2].cpu().pin_memory() for i in range(len(tokens))]
        ho = [torch.empty_like(h).pin_memory() for h in hx]
        for i in range(len(tokens)):
            _lib.moe_forward_host(base.desc, base.weights, hx[i], ho[i], wsh, stream=stream)
        e2e_steps = max(3, min(args.steps, 100))
        t0 = time.perf_counter()
        for s_ in range(e2e_steps):
            cp = copies[s_ % R]
            for i in range(len(tokens)):
                _lib.moe_forward_host(cp.desc, cp.weights, hx[i], ho[i], wsh, stream=stream)
        dt = time.perf_counter() - t0
        b_step = sum(c[5]["total"] for c in calls[: len(tokens)])
        io = int(sum(N * spec.H * 2 for N in tokens))
        e2e = {"value": round(b_step * e2e_steps / dt / 1e9, 2), "unit": "GB/s",
               "us_per_step": round(dt / e2e_steps * 1e6, 2),
               "h2d_bytes_per_step": io, "d2h_bytes_per_step": io}

    peak, peak_kind = _peaks()
    traffic, traffic_note = (args.traffic, "--traffic") if args.traffic else stream_traffic(calls)
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1/e4m3 weights, f16x2 block sums, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) NVFP4 experts, N(0,1/H) bf16 router, RMS-normed bf16 x)",
        "config": {"workload": f"{spec.name} layer, one step = moe_forward at N={','.join(map(str, tokens))}",
                   "H": spec.H, "inter": spec.inter, "E": spec.E, "top_k": spec.top_k,
                   "wfmt": spec.wfmt, "shared_inter": spec.shared_inter,
                   "layer_copies": R, "l2_bytes": l2,
                   "l2_defeat": f"inputs larger than L2: {R} layer copies cycled, step s on "
                                f"copy s mod {R}; {per_cycle_bytes / l2:.1f}x L2 touched per cycle",
                   "cuda_graph": graphs is not None,
                   "parallelism": f"{world} replicas" if world > 1 else "single GPU"},
        "frac_of_8TBs": round(value / world / NOMINAL_HBM_GBS, 4),
        "us_per_layer_mean": round(avg_launch_us, 3),
        "per_n": per_n,
        "per_n_l2_flush": per_n_flush,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": None if traffic is None else int(traffic),
                     "traffic_source": traffic_note,
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                     "kernel": "moe::moe_stream_kernel"},
        "gpu_launches": kernels_timed,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_configs:
        result["configs"] = measure_all_configs(stream, l2)
    if rank == 0 and not args.no_bf16:
        result["bf16_experts"] = measure_config(stream, "qwen3_30b_a3b_bf16", (1, 2, 3, 4), l2)
    if rank == 0 and not args.no_fp8:
        result["fp8_experts"] = measure_config(stream, "qwen3_30b_a3b_fp8", (1, 2, 3, 4), l2)
    if rank == 0 and not args.no_nvfp4_router:
        result["nvfp4_router"] = measure_config(stream, "qwen3_30b_a3b_nvfp4_router",
                                                (1, 2, 3, 4), l2)
    if rank == 0 and not args.no_zero_experts:
        result["zero_experts"] = measure_config(stream, "qwen3_30b_a3b_zero_experts",
                                                (1, 2, 3, 4), l2)
    if rank == 0:
        result["clocks"] = clk.summary()
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(spec, tokens, args.cpu_seconds)
        print(json.dumps(result))
    if world > 1:
        dist.destroy_process_group()


def l2_flush_latency(stream, calls, tokens, l2_bytes: int, reps: int = 30) -> dict:
    """Per token count: median CUDA-event time of single moe_forward calls on
    layer copy 0, each one after a write of 2 x L2 bytes on the same stream
    (L2 holds none of the call's bytes), as a check on the round-robin
    figures, which defeat L2 by cycling layer copies instead."""
    import torch
    from moe_decode_layer_topk_gb300 import _lib
    flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device="cuda")
    res = {}
    for N in tokens:
        dev, _, x, out, ws, b = next(c for c in calls if c[1] == N)
        evs = []
        with torch.cuda.stream(stream):
            for i in range(reps + 3):
                flush.fill_(i & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                _lib.moe_forward(dev.desc, dev.weights, x, out, ws, stream=stream)
                e1.record(stream)
                if i >= 3:
                    evs.append((e0, e1))
        torch.cuda.synchronize()
        assert _lib.moe_get_error(ws) == _lib.MOE_OK
        us = float(np.median([a.elapsed_time(z) * 1e3 for a, z in evs]))
        res[str(N)] = {"us_per_layer": round(us, 3), "GBps": round(b["total"] / us / 1e3, 1),
                       "U": b["U"], "calls": reps}
    del flush
    torch.cuda.empty_cache()
    return {"method": f"write of {2 * l2_bytes} bytes before each call, layer copy 0, "
                      f"median of {reps} calls", "per_n": res}


def oracle_single_thread(budget_s: float = 8.0) -> dict:
    """The oracle on one host thread, one call each on the small, Qwen3 and
    MTP-verify layers (per-call milliseconds), then the thread count restored."""
    from moe_decode_layer_topk_gb300 import synth
    from oracle import oracle
    full = oracle.num_threads()
    oracle.set_num_threads(1)
    res, t_all = {}, 0.0
    try:
        for name, N, calls in (("tiny", 1, 20), ("qwen3_30b_a3b", 1, 1), ("mtp_verify", 3, 1)):
            if t_all > budget_s:
                break
            spec = synth.CONFIGS[name]
            host = synth.make_layer(spec)
            x = synth.make_tokens(spec, N, seed=71000 + N)
            t0 = time.perf_counter()
            for _ in range(calls):
                oracle.moe_forward(host, x)
            dt = time.perf_counter() - t0
            t_all += dt
            res[f"{name}_n{N}"] = {"ms_per_call": round(dt / calls * 1e3, 2), "calls": calls}
    finally:
        oracle.set_num_threads(full)
    return {"cores": 1, "per_config": res}


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline(spec, tokens, budget_s: float):
    """The FP64 oracle (as it stands) on a bounded sample of the workload, on
    all host threads, plus the single-thread per-call times of the small,
    Qwen3 and MTP-verify layers."""
    from moe_decode_layer_topk_gb300 import synth
    from oracle import oracle
    host = synth.make_layer(spec)
    nbytes, t_total, steps = 0, 0.0, 0
    while t_total < budget_s:
        for N in tokens:
            x = synth.make_tokens(spec, N, seed=70000 + 31 * steps + N)
            t0 = time.perf_counter()
            r = oracle.moe_forward(host, x)
            t_total += time.perf_counter() - t0
            nbytes += algorithmic_bytes(spec, r["idx"], N)["total"]
        steps += 1
    return {"value": round(nbytes / t_total / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{steps} steps of moe_forward at N={','.join(map(str, tokens))} on "
                      f"{spec.name} ({t_total:.1f} s of CPU time)",
            "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
            "single_thread": oracle_single_thread()}


def run_reference(args):
    """Reference arm: the FP64 oracle on the host cores (rank 0 only).  Each
    step is a bounded sample of our arm's step: one moe_forward call of the N
    sweep, round-robin over the token counts (the whole sweep takes over a
    second on the host); when K such steps would exceed --ref-seconds (timed
    on the warm-up steps), every step is the N = 1 call instead.  Exactly W
    warm-up and K timed steps."""
    rank, world, _ = _dist()
    if rank != 0:
        return
    from moe_decode_layer_topk_gb300 import synth
    from oracle import oracle
    spec = synth.CONFIGS[args.config]
    tokens = [n for n in spec.tokens if n <= 64] if args.tokens is None else args.tokens
    host = synth.make_layer(spec)
    xs = {N: synth.make_tokens(spec, N, seed=70000 + N) for N in tokens}
    t0 = time.perf_counter()
    for s_ in range(args.warmup):
        oracle.moe_forward(host, xs[tokens[s_ % len(tokens)]])
    per_call = (time.perf_counter() - t0) / max(1, args.warmup)
    if args.warmup == 0:
        t0 = time.perf_counter()
        oracle.moe_forward(host, xs[tokens[0]])
        per_call = time.perf_counter() - t0
    order = tokens if per_call * args.steps <= args.ref_seconds else [min(tokens)]
    nbytes, t0 = 0, time.perf_counter()
    for s_ in range(args.steps):
        N = order[s_ % len(order)]
        r = oracle.moe_forward(host, xs[N])
        nbytes += algorithmic_bytes(spec, r["idx"], N)["total"]
    dt = time.perf_counter() - t0
    v = nbytes / dt / 1e9
    sample = (f"{args.steps} steps, each one moe_forward call on {spec.name}, N round-robin over "
              f"{','.join(map(str, order))} ({dt:.1f} s)")
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (same seeded layer as our arm)",
        "config": {"workload": f"{spec.name} layer, one step = moe_forward at N={','.join(map(str, tokens))}"},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3_30b_a3b")
    ap.add_argument("--tokens", type=int, nargs="*", default=None)
    ap.add_argument("--copies", type=int, default=16)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=180.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram read+write bytes per launch from an ncu capture of this kernel")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-l2-flush", action="store_true",
                    help="skip the per-N L2-flush cross-check")
    ap.add_argument("--no-bf16", action="store_true",
                    help="skip the BF16 routed-expert decode measurement")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the FP8 routed-expert decode measurement")
    ap.add_argument("--no-nvfp4-router", action="store_true",
                    help="skip the NVFP4-router decode measurement")
    ap.add_argument("--no-zero-experts", action="store_true",
                    help="skip the zero-expert routing decode measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-layer-shape records (all five shapes, gpt-oss N=512 "
                         "on the grouped path)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        import __graft_entry__
        __graft_entry__.build()
        run_gpu(args)


if __name__ == "__main__":
    main()
