"""The oracle's pins must catch plausible mistakes in the oracle.

Each mutant below plants one mistake in a copy of oracle/oracle.cpp (a
swapped nibble order, a wrong scale group, a dropped term, a wrong sign, a
transposed operand, a wrong tie order, ...), builds it, and runs the pin suite
(tests/test_oracle.py) against it in a child process.  Every mutant must make
at least one pin fail; the unmodified oracle passes them (test_oracle.py).
"""
import concurrent.futures
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTANTS = {
    "nibble_order": ("(k % 2 == 0) ? (byte & 0xF) : (byte >> 4)",
                     "(k % 2 == 0) ? (byte >> 4) : (byte & 0xF)"),
    "scale_group_16_for_mx": ("s[r * (K / gs) + k / gs]", "s[r * (K / gs) + k / 16 % (K / gs)]"),
    "scale_axis": ("s[r * (K / gs) + k / gs]", "s[(k / gs) * (K / gs) % 1 + r % (K / gs) + 0 * k]"),
    "dropped_up_term": ("a[i] = silu(g) * u;\n    }\n#pragma omp parallel for schedule(static)\n    for (int r = 0; r < H; ++r) {\n        double acc = 0.0;\n        for (int i = 0; i < inter; ++i)",
                        "a[i] = silu(g);\n    }\n#pragma omp parallel for schedule(static)\n    for (int r = 0; r < H; ++r) {\n        double acc = 0.0;\n        for (int i = 0; i < inter; ++i)"),
    "silu_sign": ("return g / (1.0 + std::exp(-g));", "return g / (1.0 + std::exp(g));"),
    "bias_in_weights": ("base[e] = 1.0 / (1.0 + std::exp(-l[e]));",
                        "base[e] = 1.0 / (1.0 + std::exp(-l[e])) + (bias ? (double)bias[e] : 0.0);"),
    "ties_to_higher_index": ("return a < b;", "return a > b;"),
    "ascending_sort": ("return score[a] > score[b];", "return score[a] < score[b];"),
    "no_renorm": ("if (norm)\n", "if (0)\n"),
    "rsf_on_softmax": ("if (scoring != 0)\n        for (int j = 0; j < k; ++j) w[j] *= rsf;",
                       "for (int j = 0; j < k; ++j) w[j] *= rsf;"),
    "softmax_denominator": ("den += std::exp(l[e] - mx);", "den += std::exp(l[e]);"),
    "down_transposed": ("oracle_weight(dq, dsc, d2, inter, fmt, r, i)",
                        "oracle_weight(dq, dsc, d2, inter, fmt, i % H, r % inter)"),
    "bf16_byte_order": ("(uint32_t)q[i] | ((uint32_t)q[i + 1] << 8)",
                        "(uint32_t)q[i + 1] | ((uint32_t)q[i] << 8)"),
    "bf16_adjacent_swap": ("const long i = 2 * (r * (long)K + k);",
                           "const long i = 2 * ((r * (long)K + k) ^ 1);"),
    "bf16_expert_stride": ("const long gq_e = bf ? 2L * inter * H", "const long gq_e = bf ? 1L * inter * H"),
    "router_nvfp4_as_mxfp4": ("return oracle_fp4_weight(wr, rs, rs2, H, 0, e, h);",
                              "return oracle_fp4_weight(wr, rs, rs2, H, 1, e, h);"),
    "router_scale2_ignored": ("W->router_s2 ? (double)W->router_s2[0] : 1.0", "1.0"),
    "softmax_bias_ignored": ("score[e] = base[e] + ((scoring == 2 && bias) ? (double)bias[e] : 0.0);",
                             "score[e] = base[e];"),
    "softmax_bias_no_rsf": ("if (scoring != 0)\n        for (int j = 0; j < k; ++j) w[j] *= rsf;",
                            "if (scoring == 1)\n        for (int j = 0; j < k; ++j) w[j] *= rsf;"),
    "zero_expert_runs_expert_0": ("if (e >= E) continue;", "if (e >= E) { }"),
    "hash_row_by_position": ("W->tid2eid + (long)token_ids[n] * k", "W->tid2eid + (long)n * k"),
    "hash_sigmoid_as_softmax": ("w[j] = (scoring == 1) ? 1.0 / (1.0 + std::exp(-l[e])) : std::exp(l[e] - mx) / den;",
                                "w[j] = std::exp(l[e] - mx) / den;"),
    "fp8_row_block_ignored": ("s + 4 * ((r / 128) * kb + k / 128)", "s + 4 * (k / 128)"),
    "fp8_scale_ignored": ("return oracle_e4m3(q[r * (long)K + k]) * (double)sc;",
                          "return oracle_e4m3(q[r * (long)K + k]) * (sc > 0 ? 1.0 : 0.0);"),
    "fp8_scale_stride": ("const long gs_e = bf ? 0 : f8 ? 4 * bi * bh", "const long gs_e = bf ? 0 : f8 ? 4 * bi"),
    "router_transposed": ("oracle_bf16(wr[(long)e * H + h])", "oracle_bf16(wr[(long)h * E + e])"),
    "shared_gate_no_sigmoid": ("gsig = 1.0 / (1.0 + std::exp(-d));", "gsig = d;"),
    "shared_down_dropped": ("acc[h] += gsig * sh[h];", "acc[h] += gsig;"),
    "e4m3_subnormal_exp": ("std::ldexp(m / 8.0, -6)", "std::ldexp(m / 8.0, -7)"),
    "e2m1_bias": ("std::ldexp(1.0 + 0.5 * m, e - 1)", "std::ldexp(1.0 + 0.5 * m, e - 2)"),
    "e8m0_bias": ("(int)(byte & 0xFF) - 127", "(int)(byte & 0xFF) - 128"),
    "bf16_ties_away": ("(frac == 0.5 && std::fmod(r, 2.0) != 0.0)", "(frac == 0.5)"),
    "routed_weight_dropped": ("acc[h] += wj * y[h];", "acc[h] += y[h];"),
    "scale2_ignored": ("return oracle_e2m1(code) * bs * scale2;", "return oracle_e2m1(code) * bs;"),
}


def _run_mutant(name, tmp):
    src = open(SRC).read()
    if name == "control":
        mut = src
    else:
        old, new = MUTANTS[name]
        assert src.count(old) >= 1, f"mutant {name}: pattern not found"
        mut = src.replace(old, new, 1)
    cpp = os.path.join(tmp, f"{name}.cpp")
    so = os.path.join(tmp, f"{name}.so")
    open(cpp, "w").write(mut)
    subprocess.run(["g++", "-std=c++17", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", so, cpp],
                   check=True, capture_output=True)
    env = dict(os.environ, MOE_ORACLE_LIB=so, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    # pytest exit code 1 = some test failed (an assertion in a pin), as
    # opposed to 0 (all passed) or 2-4 (collection/usage/internal errors).
    return name, r.returncode, ("FAILED" in r.stdout) or ("failed" in r.stdout)


def test_every_planted_mistake_is_caught():
    names = ["control"] + sorted(MUTANTS)
    with tempfile.TemporaryDirectory() as tmp:
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            results = {n: (rc, failed) for n, rc, failed in ex.map(lambda n: _run_mutant(n, tmp), names)}
    assert results.pop("control")[0] == 0, "the unmodified oracle must pass its pins"
    survivors = [n for n, (rc, failed) in results.items() if not (rc == 1 and failed)]
    assert not survivors, f"mutants not caught by a failing pin: {survivors}"
