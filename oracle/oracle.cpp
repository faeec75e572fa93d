// FP64 CPU oracle for the mixture-of-experts decode-layer forward.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
// calls this file; the test suite, the smoke check and the bench's CPU
// baseline do.  It shares no code, header, table or constant with the CUDA
// library: every decode below is written from the format definitions.
//
// What it computes (plain definition, no blocking, no fusion), following the
// layer the pages describe:
//   * forward_k3.rs, doc comment of MoeLayer::forward_k3 — the chain
//     router logits -> top-k -> expert gate+up -> SiLU+down -> weighted sum
//     + shared-expert blend;
//   * forward_k3.rs, the batched top-k step (moe_topk_sigmoid_batched /
//     moe_topk_softmax_batched arguments) — softmax with optional
//     renormalisation, or sigmoid + correction bias with norm_topk_prob and
//     routed_scaling_factor;
//   * forward_k3.rs, the E8M0 guard (GS16 vs GS32 scale groups) — NVFP4
//     (E2M1 + per-16 E4M3) and MXFP4 (E2M1 + per-32 E8M0) expert formats;
//   * forward_batched.rs, the BF16 expert branch (bf16_gate/up/down weight
//     pointers, run through the plain forward's kernels) — BF16 routed experts,
//     the same chain with plain BF16 weights (no block scales);
//   * forward_k3.rs / forward_batched.rs, the FP8 expert branch (fp8 gate/up/
//     down weight_ptrs + scale_ptrs into moe_expert_gate_up_shared_fp8 and
//     moe_expert_silu_down_shared_fp8) — FP8 routed experts: E4M3 weights
//     with block scales.  The pages do not give the scale granularity; the
//     reading taken is one FP32 scale per 128 x 128 block of each projection;
//   * forward_k3.rs / forward_batched.rs / forward_ep.rs, step 1 (gate_nvfp4
//     into w4a16_gemv_batch3 / w4a16_gemm / w4a16_decode_gemv) — the router
//     weight may be NVFP4 (E2M1 + per-16 E4M3 scale + FP32 scale2) against the
//     BF16 activations;
//   * forward_k3.rs / forward_batched.rs, the zero-expert guards (a router of
//     width num_experts + zero_expert_num, run only with softmax + bias
//     scoring) — routing over E + Z router outputs
//     with softmax scores plus a correction bias for selection; a selected
//     zero expert runs no expert.  The pages do not say what a zero expert
//     adds; the reading taken is nothing (its output is zero);
//   * forward_batched.rs, hash routing (moe_hash_route with the gate logits,
//     tid2eid, the token's id, num_experts, top_k, norm_topk_prob and
//     routed_scaling_factor) — the k experts of a token are row token_id of
//     the tid2eid table; the weights come from the gate logits with the
//     layer's scoring (the pages do not spell the rule out; the reading taken
//     is the top-k rule applied to the table's experts);
//   * forward_atomic_c4.rs, doc comment — routed outputs accumulated as
//     routing-weighted sums, then cast to BF16 and blended with the shared
//     expert;
//   * forward_k3.rs, the EP all-reduce block (the sigmoid-gated shared-expert
//     add) — a null shared_expert_gate adds the shared expert as is,
//     otherwise it is blended with sigmoid(w_s . x).
// Readings where the pages are silent (nibble order, tie order, bias only in
// selection, scaling only on the sigmoid path) are stated at each function.
//
// All arithmetic is double precision; OpenMP only splits independent output
// rows (each output element is still summed by one thread in index order).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>
#include <numeric>

#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// ---------------------------------------------------------------- decoders

// OCP Microscaling Formats (MX) v1.0, FP4 E2M1: sign(1) exponent(2, bias 1)
// mantissa(1); exponent 0 is subnormal (0.5 * m); no inf or NaN.
double oracle_e2m1(uint32_t nibble) {
    const int s = (nibble >> 3) & 1, e = (nibble >> 1) & 3, m = nibble & 1;
    const double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

// OCP 8-bit Floating Point spec, E4M3 ("fn": bias 7, no inf, S.1111.111 = NaN,
// max 448); exponent 0 is subnormal m/8 * 2^-6.
double oracle_e4m3(uint32_t byte) {
    const int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    if (e == 15 && m == 7) return std::nan("");
    const double mag = (e == 0) ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

// OCP MX v1.0 E8M0 shared scale: 2^(e-127); 0xFF is NaN.
double oracle_e8m0(uint32_t byte) {
    if ((byte & 0xFF) == 0xFF) return std::nan("");
    return std::ldexp(1.0, (int)(byte & 0xFF) - 127);
}

// BF16 = the upper 16 bits of an IEEE binary32.
double oracle_bf16(uint32_t bits16) {
    const uint32_t u = (bits16 & 0xFFFFu) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// Round a double to the nearest BF16 (8 significant bits, exponent range of
// binary32), ties to even, overflow to infinity; returns the 16-bit pattern.
uint32_t oracle_round_bf16(double v) {
    if (std::isnan(v)) return 0x7FC0;
    const uint32_t sign = std::signbit(v) ? 0x8000u : 0u;
    double a = std::fabs(v);
    if (a == 0.0) return sign;
    // quantum of the bf16 grid at |v|: 2^(e-7) for normals (e = floor(log2 a)),
    // 2^-133 below the smallest normal 2^-126.
    int e = std::ilogb(a);
    const double quantum = (e < -126) ? std::ldexp(1.0, -133) : std::ldexp(1.0, e - 7);
    const double q = a / quantum;                 // exact (power-of-two division)
    double r = std::floor(q);
    const double frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && std::fmod(r, 2.0) != 0.0)) r += 1.0;
    const double rounded = r * quantum;
    if (rounded >= std::ldexp(1.0, 128)) return sign | 0x7F80u;   // inf
    const float f = (float)rounded;               // exact: rounded is on the bf16 grid
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return sign | ((u >> 16) & 0x7FFFu);
}

// ------------------------------------------------------------ dequantisation

// Value of element (r, k) of one FP4 projection matrix [rows, K]:
//   E2M1(code) * blockscale(scale[r, k/gs]) * scale2
// with code = low nibble of byte q[r, k/2] for even k, high nibble for odd k
// (element 2j in the low nibble: not stated on the pages; plainest reading),
// and the scale group running along K, the input dimension (the pages size
// the scale buffer as rows*K/16 for NVFP4 and rows*K/32 for E8M0).
// fmt 0 = NVFP4 (gs 16, E4M3 scales), fmt 1 = MXFP4 (gs 32, E8M0 scales).
double oracle_fp4_weight(const uint8_t* q, const uint8_t* s, double scale2,
                         int K, int fmt, long r, long k) {
    const int gs = (fmt == 0) ? 16 : 32;
    const uint8_t byte = q[r * (K / 2) + k / 2];
    const uint32_t code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    const uint8_t sb = s[r * (K / gs) + k / gs];
    const double bs = (fmt == 0) ? oracle_e4m3(sb) : oracle_e8m0(sb);
    return oracle_e2m1(code) * bs * scale2;
}

// Value of element (r, k) of a routed projection [rows, K] in weight format
// `fmt`: 0/1 as oracle_fp4_weight; 2 = BF16 experts, the BF16 number stored in
// the 16-bit little-endian word r*K + k of q (no block scales: s and scale2
// are not read).
// fmt 3 = FP8 experts: E4M3(q[r*K + k]) times the FP32 block scale
// S[r/128][k/128] of the [ceil(rows/128), ceil(K/128)] scale table at s
// (floats, native byte order); scale2 is not read.
double oracle_weight(const uint8_t* q, const uint8_t* s, double scale2, int K, int fmt,
                     long r, long k) {
    if (fmt == 2) {
        const long i = 2 * (r * (long)K + k);
        return oracle_bf16((uint32_t)q[i] | ((uint32_t)q[i + 1] << 8));
    }
    if (fmt == 3) {
        const long kb = (K + 127) / 128;
        float sc;
        std::memcpy(&sc, s + 4 * ((r / 128) * kb + k / 128), 4);
        return oracle_e4m3(q[r * (long)K + k]) * (double)sc;
    }
    return oracle_fp4_weight(q, s, scale2, K, fmt, r, k);
}

void oracle_dequant(const uint8_t* q, const uint8_t* s, double scale2, int rows, int K,
                    int fmt, double* out) {
    for (long r = 0; r < rows; ++r)
        for (long k = 0; k < K; ++k)
            out[r * K + k] = oracle_weight(q, s, scale2, K, fmt, r, k);
}

// ------------------------------------------------------------------- router

// logits[n, e] = sum_h x[n, h] * Wr[e, h]   (BF16 inputs, FP64 products/sums)
void oracle_router_logits(const uint16_t* x, const uint16_t* wr, int N, int E, int H,
                          double* logits) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; ++n)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += oracle_bf16(x[(long)n * H + h]) * oracle_bf16(wr[(long)e * H + h]);
            logits[(long)n * E + e] = acc;
        }
}

// Router weight (e, h): fmt 0 = BF16 router [E, H] (16-bit little-endian
// words at wr); fmt 1 = NVFP4 router, E2M1 codes [E, H/2] at wr, E4M3 scales
// [E, H/16] at rs, times the router's scale2 (rs2).
double oracle_router_weight(const uint8_t* wr, const uint8_t* rs, double rs2, int H, int fmt,
                            long e, long h) {
    if (fmt == 1) return oracle_fp4_weight(wr, rs, rs2, H, 0, e, h);
    const long i = 2 * (e * (long)H + h);
    return oracle_bf16((uint32_t)wr[i] | ((uint32_t)wr[i + 1] << 8));
}

// logits[n, e] = sum_h x[n, h] * Wr[e, h] for either router format.
void oracle_router_logits_fmt(const uint16_t* x, const uint8_t* wr, const uint8_t* rs, double rs2,
                              int fmt, int N, int E, int H, double* logits) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int n = 0; n < N; ++n)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += oracle_bf16(x[(long)n * H + h]) * oracle_router_weight(wr, rs, rs2, H, fmt, e, h);
            logits[(long)n * E + e] = acc;
        }
}

// ------------------------------------------------------------------ routing

// Routing of one token, from its logits row.
//   scoring 0 (softmax): p = softmax(l); selection score = p;
//       w = p of the selected experts, divided by their sum if norm != 0.
//       The routed scaling factor is not applied (the softmax top-k op is not
//       given it on the pages).
//   scoring 1 (sigmoid + correction bias): s = 1/(1+exp(-l)); selection score
//       = s + bias; w = s of the selected experts (bias only selects), divided
//       by their sum if norm != 0, then multiplied by rsf.
//   scoring 2 (softmax + correction bias, the zero-expert routers): p =
//       softmax(l); selection score = p + bias; w = p of the selected, divided
//       by their sum if norm != 0, then multiplied by rsf.
// Top-k: sort by selection score descending, ties to the lower expert index;
// the first k in that order are the selected experts, in that order.
// sel_score (optional, [E]) receives the selection score of every expert.
void oracle_route_one(const double* l, const float* bias, int E, int k, int scoring,
                      int norm, double rsf, int32_t* idx, double* w, double* sel_score) {
    std::vector<double> score(E), base(E);
    if (scoring == 0 || scoring == 2) {
        double mx = l[0];
        for (int e = 1; e < E; ++e) mx = std::max(mx, l[e]);
        double den = 0.0;
        for (int e = 0; e < E; ++e) den += std::exp(l[e] - mx);
        for (int e = 0; e < E; ++e) {
            base[e] = std::exp(l[e] - mx) / den;
            score[e] = base[e] + ((scoring == 2 && bias) ? (double)bias[e] : 0.0);
        }
    } else {
        for (int e = 0; e < E; ++e) {
            base[e] = 1.0 / (1.0 + std::exp(-l[e]));
            score[e] = base[e] + (bias ? (double)bias[e] : 0.0);
        }
    }
    std::vector<int> order(E);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
        if (score[a] != score[b]) return score[a] > score[b];
        return a < b;
    });
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
        idx[j] = order[j];
        w[j] = base[order[j]];
        sum += w[j];
    }
    if (norm)
        for (int j = 0; j < k; ++j) w[j] /= sum;
    if (scoring != 0)
        for (int j = 0; j < k; ++j) w[j] *= rsf;
    if (sel_score)
        for (int e = 0; e < E; ++e) sel_score[e] = score[e];
}

// Hash routing of one token: the selected experts are the table row `row`
// (k expert ids, in that order); their weights follow the scoring as in
// oracle_route_one (softmax over all E for scorings 0 and 2, sigmoid for 1;
// divided by their sum if norm != 0; times rsf unless scoring 0).  The bias
// does not enter (it only ever selects).
void oracle_route_hash_one(const double* l, const int32_t* row, int E, int k, int scoring,
                           int norm, double rsf, int32_t* idx, double* w) {
    double mx = l[0], den = 0.0;
    for (int e = 1; e < E; ++e) mx = std::max(mx, l[e]);
    for (int e = 0; e < E; ++e) den += std::exp(l[e] - mx);
    double sum = 0.0;
    for (int j = 0; j < k; ++j) {
        const int e = row[j];
        idx[j] = e;
        w[j] = (scoring == 1) ? 1.0 / (1.0 + std::exp(-l[e])) : std::exp(l[e] - mx) / den;
        sum += w[j];
    }
    if (norm)
        for (int j = 0; j < k; ++j) w[j] /= sum;
    if (scoring != 0)
        for (int j = 0; j < k; ++j) w[j] *= rsf;
}

void oracle_route(const double* logits, const float* bias, int N, int E, int k, int scoring,
                  int norm, double rsf, int32_t* idx, double* w, double* sel_score) {
    for (int n = 0; n < N; ++n)
        oracle_route_one(logits + (long)n * E, bias, E, k, scoring, norm, rsf,
                         idx + (long)n * k, w + (long)n * k,
                         sel_score ? sel_score + (long)n * E : nullptr);
}

// ------------------------------------------------------------------ experts

static double silu(double g) { return g / (1.0 + std::exp(-g)); }

// One routed expert on one token (weight format fmt, see oracle_weight):
//   g = Dq(Wg) x,  u = Dq(Wu) x,  a = SiLU(g) * u,  y = Dq(Wd) a.
// Wg, Wu are [inter, H]; Wd is [H, inter]; x is BF16 [H]; y is [H].
void oracle_expert(const uint8_t* gq, const uint8_t* gsc, double g2,
                       const uint8_t* uq, const uint8_t* usc, double u2,
                       const uint8_t* dq, const uint8_t* dsc, double d2,
                       int H, int inter, int fmt, const uint16_t* x, double* y) {
    std::vector<double> xv(H), a(inter);
    for (int h = 0; h < H; ++h) xv[h] = oracle_bf16(x[h]);
#pragma omp parallel for schedule(static)
    for (int i = 0; i < inter; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            g += oracle_weight(gq, gsc, g2, H, fmt, i, h) * xv[h];
            u += oracle_weight(uq, usc, u2, H, fmt, i, h) * xv[h];
        }
        a[i] = silu(g) * u;
    }
#pragma omp parallel for schedule(static)
    for (int r = 0; r < H; ++r) {
        double acc = 0.0;
        for (int i = 0; i < inter; ++i)
            acc += oracle_weight(dq, dsc, d2, inter, fmt, r, i) * a[i];
        y[r] = acc;
    }
}

// Shared expert, BF16 weights: sh = Wd (SiLU(Wg x) * (Wu x)); Wg, Wu [Is, H],
// Wd [H, Is].
void oracle_shared_expert(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd,
                          int H, int Is, const uint16_t* x, double* sh) {
    std::vector<double> xv(H), a(Is);
    for (int h = 0; h < H; ++h) xv[h] = oracle_bf16(x[h]);
#pragma omp parallel for schedule(static)
    for (int i = 0; i < Is; ++i) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            g += oracle_bf16(wg[(long)i * H + h]) * xv[h];
            u += oracle_bf16(wu[(long)i * H + h]) * xv[h];
        }
        a[i] = silu(g) * u;
    }
#pragma omp parallel for schedule(static)
    for (int r = 0; r < H; ++r) {
        double acc = 0.0;
        for (int i = 0; i < Is; ++i) acc += oracle_bf16(wd[(long)r * Is + i]) * a[i];
        sh[r] = acc;
    }
}

// ------------------------------------------------------------- full forward

// Weights of one layer, host memory, canonical layout:
//   router [E, H] bf16; bias [E] f32 or null;
//   gate_q/up_q [E, inter, H/2] u8, gate_s/up_s [E, inter, H/gs] u8,
//   down_q [E, H, inter/2] u8, down_s [E, H, inter/gs] u8,
//   *_s2 [E] f32 or null (null = 1.0; MXFP4 has none);
//   BF16 experts (fmt 2): gate_q/up_q [E, inter, H] and down_q [E, H, inter]
//   hold BF16 words, the scale pointers are not read;
//   FP8 experts (fmt 3): gate_q/up_q [E, inter, H], down_q [E, H, inter] E4M3
//   bytes; gate_s/up_s [E, ceil(inter/128), ceil(H/128)] and down_s
//   [E, ceil(H/128), ceil(inter/128)] f32 block scales; *_s2 not read;
//   sh_gate/sh_up [Is, H] bf16, sh_down [H, Is] bf16 (null when Is == 0);
//   sh_gate_w [H] bf16 or null (null = ungated shared expert).
struct oracle_weights {
    const uint16_t* router;
    const float* bias;
    const uint8_t *gate_q, *up_q, *down_q;
    const uint8_t *gate_s, *up_s, *down_s;
    const float *gate_s2, *up_s2, *down_s2;
    const uint16_t *sh_gate, *sh_up, *sh_down;
    const uint16_t* sh_gate_w;
    const uint8_t* router_s;     // NVFP4 router: E4M3 scales [E, H/16]
    const float* router_s2;      // NVFP4 router: scale2 (one float) or null = 1.0
    const int32_t* tid2eid;      // hash routing: [V, k] expert ids per token id, or null
};

// out_f64 [N, H] = sum_j w[n,j] * expert_{idx[n,j]}(x_n) + g_s(x_n) * shared(x_n)
// with g_s = sigmoid(w_s . x_n) when sh_gate_w is given, 1 otherwise, and no
// shared term when Is == 0.  The routed scaling factor is not applied to the
// shared expert.  out_bf16 is out_f64 rounded to BF16 (nearest even).
// idx/w receive the routing ([N, k]); logits (optional) the router output.
// router_fmt: 0 = BF16 router, 1 = NVFP4 router (router holds the codes).
// Z zero experts: the router (and bias) has E + Z rows, routing runs over all
// E + Z, and a slot that selects index >= E adds nothing; logits_out is
// [N, E + Z].
int oracle_moe_forward(int H, int inter, int E, int k, int scoring, int norm, double rsf,
                       int fmt, int Is, const oracle_weights* W, const uint16_t* x, int N,
                       double* out_f64, uint16_t* out_bf16, int32_t* idx, double* w,
                       double* logits_out, int router_fmt, int Z, const int32_t* token_ids) {
    if (H <= 0 || inter <= 0 || E <= 0 || Z < 0 || k <= 0 || k > E + Z || N < 0) return 1;
    if (scoring < 0 || scoring > 2) return 1;
    const int R = E + Z;   // router width
    if (fmt < 0 || fmt > 3 || router_fmt < 0 || router_fmt > 1) return 1;
    const int gs = (fmt == 0) ? 16 : 32;
    std::vector<double> logits((size_t)N * R);
    if (router_fmt == 0)
        oracle_router_logits(x, W->router, N, R, H, logits.data());
    else
        oracle_router_logits_fmt(x, reinterpret_cast<const uint8_t*>(W->router), W->router_s,
                                 W->router_s2 ? (double)W->router_s2[0] : 1.0, 1, N, R, H,
                                 logits.data());
    if (logits_out) std::copy(logits.begin(), logits.end(), logits_out);
    if (W->tid2eid) {   // hash routing: token n takes table row token_ids[n]
        if (!token_ids || Z != 0) return 1;
        for (int n = 0; n < N; ++n)
            oracle_route_hash_one(logits.data() + (long)n * R, W->tid2eid + (long)token_ids[n] * k,
                                  R, k, scoring, norm, rsf, idx + (long)n * k, w + (long)n * k);
    } else {
        oracle_route(logits.data(), W->bias, N, R, k, scoring, norm, rsf, idx, w, nullptr);
    }

    // bytes per expert of each table (BF16: two bytes per element, no scales;
    // FP8: one byte per element, 4-byte scales per 128 x 128 block)
    const bool bf = (fmt == 2), f8 = (fmt == 3);
    const long bi = (inter + 127) / 128, bh = (H + 127) / 128;
    const long gq_e = bf ? 2L * inter * H : f8 ? (long)inter * H : (long)inter * (H / 2);
    const long gs_e = bf ? 0 : f8 ? 4 * bi * bh : (long)inter * (H / gs);
    const long dq_e = bf ? 2L * H * inter : f8 ? (long)H * inter : (long)H * (inter / 2);
    const long ds_e = bf ? 0 : f8 ? 4 * bh * bi : (long)H * (inter / gs);
    std::vector<double> y(H), sh(H);
    for (int n = 0; n < N; ++n) {
        const uint16_t* xn = x + (long)n * H;
        std::vector<double> acc(H, 0.0);
        for (int j = 0; j < k; ++j) {
            const int e = idx[(long)n * k + j];
            if (e >= E) continue;              // zero expert: adds nothing
            const bool fp4 = !bf && !f8;   // only the FP4 formats have scale2
            const double g2 = (fp4 && W->gate_s2) ? W->gate_s2[e] : 1.0;
            const double u2 = (fp4 && W->up_s2) ? W->up_s2[e] : 1.0;
            const double d2 = (fp4 && W->down_s2) ? W->down_s2[e] : 1.0;
            oracle_expert(W->gate_q + e * gq_e, bf ? nullptr : W->gate_s + e * gs_e, g2,
                          W->up_q + e * gq_e, bf ? nullptr : W->up_s + e * gs_e, u2,
                          W->down_q + e * dq_e, bf ? nullptr : W->down_s + e * ds_e, d2,
                          H, inter, fmt, xn, y.data());
            const double wj = w[(long)n * k + j];
            for (int h = 0; h < H; ++h) acc[h] += wj * y[h];
        }
        if (Is > 0) {
            oracle_shared_expert(W->sh_gate, W->sh_up, W->sh_down, H, Is, xn, sh.data());
            double gsig = 1.0;
            if (W->sh_gate_w) {
                double d = 0.0;
                for (int h = 0; h < H; ++h) d += oracle_bf16(W->sh_gate_w[h]) * oracle_bf16(xn[h]);
                gsig = 1.0 / (1.0 + std::exp(-d));
            }
            for (int h = 0; h < H; ++h) acc[h] += gsig * sh[h];
        }
        for (int h = 0; h < H; ++h) {
            if (out_f64) out_f64[(long)n * H + h] = acc[h];
            if (out_bf16) out_bf16[(long)n * H + h] = (uint16_t)oracle_round_bf16(acc[h]);
        }
    }
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

// Threads of the oracle's later parallel loops (n >= 1).  Each output element
// is still summed by one thread in index order, so the results do not depend
// on it; only the timing does.
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

}  // extern "C"
