// Fused MoE decode-layer forward for small N on sm_103a (one launch per call).
//
// Computes, for N token rows (see forward_k3.rs MoeLayer::forward_k3 for the
// step chain and forward_atomic_c4.rs for the FP32 routing-weighted
// accumulation followed by the BF16 cast and shared-expert blend):
//   router logits -> top-k routing -> per-expert gate+up (FP4 or BF16) ->
//   SiLU(g)*u -> down -> routing-weighted FP32 sum + shared expert -> BF16.
//
// Execution model: a persistent grid, one CTA per SM, every CTA resident at
// once (cooperative launch).  Each CTA has 8 compute ("consumer") warps and
// one producer warp that streams weight rows into a ring of shared-memory
// stages with 1D bulk copies (TMA), completion tracked by mbarriers.
//
// Phases of one call (per CTA):
//   P0  router GEMV for rows e = cta, cta+G, ... (direct 128-bit loads);
//       per-token prep for n = cta, cta+G, ...: f16 copy of x scaled by a
//       power of two, shared-expert gate sigmoid(w_s . x);
//       zero the FP32 accumulator and the row-block counters.
//   --  grid barrier B1 (arrive); shared-expert gate/up row groups need only x,
//       so they are streamed and computed before waiting on B1.
//   P1  every CTA computes the same top-k for all N tokens from the logits,
//       then the same table of unique experts (ascending id), per-expert token
//       lists and the list of (expert, token batch) units.  Each routed
//       expert's weights are then read once for all its tokens
//       (forward_batched.rs: "streams its weights once for all rows").
//   P2  routed gate/up row groups -> h = SiLU(g)*u (FP32, workspace).
//   --  grid barrier B2 (the producer keeps prefetching down weights).
//   P3  down row groups (routed and shared) -> routing-weighted FP32 red.add
//       into acc[N,H]; the CTA completing an aligned 32-row block of acc casts
//       it to BF16 into out (no third grid barrier).
//
// Work split: a row group (RG) is 32 consecutive weight rows of one
// (expert, token batch) unit; each kind's RG list is split evenly over the
// CTAs.  Inside a CTA, lane j of every consumer warp owns row j of the RG and
// the 8 warps split the K range; partial sums meet in shared memory at the
// end of the RG.  Weight rows land in stages with an odd multiple of 16 bytes
// as row stride, so the lane-per-row 128-bit shared loads are conflict free;
// activations are read as broadcasts.
//
// FP4 arithmetic: E2M1 codes become f16x2 with cvt.rn.f16x2.e2m1x2; each
// 16-element (NVFP4) or 32-element (MXFP4) block is summed with f16x2 FMAs
// against x (or h) held as f16 scaled by a per-row power of two that keeps
// every partial below 2^14; each block partial is then multiplied by its
// E4M3/E8M0 scale and accumulated in FP32.  The shared expert (BF16) uses
// fma.rn.f32.bf16 (BF16 products, FP32 accumulation).
//
// Every wait (grid barrier, stage, routing-ready) is bounded by a time budget;
// on expiry the kernel records an error bit in the workspace and drains.

#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {

struct Tables {
  int16_t sel_e[kMaxSlots];    // routing per slot s = n*k + j
  float sel_w[kMaxSlots];
  uint32_t cnt[kMaxE];         // per expert: count, then unique index
  int16_t uexp[kMaxSlots];     // unique experts, ascending id
  uint16_t ucnt[kMaxSlots];    // tokens routed to unique expert u
  uint16_t hoff[kMaxSlots];    // first slot of u in the (expert, token) order
  uint8_t utok[kMaxSlots];     // token of (expert, position) slot
  float uw[kMaxSlots];         // routing weight of that slot
  uint16_t unit_u[kMaxSlots];  // units = (unique expert, token batch)
  uint8_t unit_tb[kMaxSlots];
  int U, n_units;
  int abort;                   // set when a bounded wait expired
  int fin;                     // this CTA completes the current row block
  int hb_kind, hb_unit;        // unit whose activations sit in hbuf
  int hexp[kTB];               // power-of-two exponents of hbuf rows
  float rscratch[kConsumerWarps * 8];
  uint32_t uscratch[kConsumerWarps * 2];
};

// ----------------------------------------------------------------- helpers

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ void consumer_sync() { named_bar_sync(1, kConsumerThreads); }

// Sum over the 256 consumer threads of M values each; result valid in all threads.
template <int M>
__device__ __forceinline__ void block_sum(float (&v)[M], Tables& tb, int ctid) {
  const int lane = ctid & 31, warp = ctid >> 5;
#pragma unroll
  for (int m = 0; m < M; ++m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[m] += __shfl_xor_sync(0xffffffffu, v[m], o);
  }
  if (lane == 0) {
#pragma unroll
    for (int m = 0; m < M; ++m) tb.rscratch[warp * 8 + m] = v[m];
  }
  consumer_sync();
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) s += tb.rscratch[w * 8 + m];
    v[m] = s;
  }
  consumer_sync();
}

template <int M>
__device__ __forceinline__ void block_max(float (&v)[M], Tables& tb, int ctid) {
  const int lane = ctid & 31, warp = ctid >> 5;
#pragma unroll
  for (int m = 0; m < M; ++m) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[m] = fmaxf(v[m], __shfl_xor_sync(0xffffffffu, v[m], o));
  }
  if (lane == 0) {
#pragma unroll
    for (int m = 0; m < M; ++m) tb.rscratch[warp * 8 + m] = v[m];
  }
  consumer_sync();
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) s = fmaxf(s, tb.rscratch[w * 8 + m]);
    v[m] = s;
  }
  consumer_sync();
}

// Exclusive scan over the 256 consumer threads (one value each); returns the
// prefix, total in *total.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, Tables& tb, int ctid,
                                                    uint32_t* total) {
  const int lane = ctid & 31, warp = ctid >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) tb.uscratch[warp] = inc;
  consumer_sync();
  uint32_t base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) {
    const uint32_t s = tb.uscratch[w];
    if (w < warp) base += s;
    tot += s;
  }
  consumer_sync();
  *total = tot;
  return base + inc - v;
}

// Power-of-two exponent e such that max|v| * 2^-e lies in [64, 128).
__device__ __forceinline__ int scale_exponent(float amax) {
  if (!(amax > 0.f) || !isfinite(amax)) return 0;
  return ilogbf(amax) - 6;
}

// ------------------------------------------------------------ grid barrier
// Self-resetting barrier in the workspace: ctrl[0] counts arrivals, ctrl[1]
// is the generation.  The last arriver resets the count and bumps the
// generation; waiters spin (bounded) until the generation changes.
__device__ uint32_t grid_arrive(uint32_t* ctrl, uint32_t G) {
  const uint32_t gen = ld_acquire_u32(ctrl + 1);
  __threadfence();
  const uint32_t old = atomicAdd(ctrl + 0, 1u);
  if (old == G - 1) {
    atomicExch(ctrl + 0, 0u);
    __threadfence();
    atomicAdd(ctrl + 1, 1u);
  }
  return gen;
}

__device__ bool grid_wait(uint32_t* ctrl, uint32_t gen, uint64_t budget_ns) {
  if (ld_acquire_u32(ctrl + 1) != gen) return true;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_u32(ctrl + 1) == gen) {
    if (global_timer_ns() - t0 > budget_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- router
// logits[n, e] = sum_h x[n, h] * Wr[e, h], FP32 accumulation of BF16 products.
__device__ void router_phase(const Params& p, int cta, int G, Tables& tb, int ctid) {
  const int H = p.H;
  for (int e = cta; e < p.E; e += G) {
    const uint16_t* wr = p.router + (size_t)e * H;
    for (int n0 = 0; n0 < p.N; n0 += 8) {
      const int nn = min(8, p.N - n0);
      float acc[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t] = 0.f;
      for (int kk = ctid * 8; kk < H; kk += kConsumerThreads * 8) {
        const uint4 w = ld_nc_u4(wr + kk);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (t < nn) {
            const uint4 xv = ld_nc_u4(p.x + (size_t)(n0 + t) * H + kk);
            const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              acc[t] = fmaf(bf16_lo(wv[i]), bf16_lo(xa[i]), acc[t]);
              acc[t] = fmaf(bf16_hi(wv[i]), bf16_hi(xa[i]), acc[t]);
            }
          }
        }
      }
      block_sum<8>(acc, tb, ctid);
      if (ctid < nn) {
        float v = acc[0];
#pragma unroll
        for (int t = 1; t < 8; ++t)
          if (ctid == t) v = acc[t];
        p.logits[(size_t)(n0 + ctid) * p.E + e] = v;
      }
    }
  }
}

// Per-token prep: x16 = f16(x * 2^-xexp) and the shared-expert gate.
__device__ void token_prep(const Params& p, int cta, int G, Tables& tb, int ctid) {
  const int H = p.H;
  for (int n = cta; n < p.N; n += G) {
    const uint16_t* xr = p.x + (size_t)n * H;
    float m[1] = {0.f};
    float d[1] = {0.f};
    for (int kk = ctid * 8; kk < H; kk += kConsumerThreads * 8) {
      const uint4 xv = ld_nc_u4(xr + kk);
      const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        m[0] = fmaxf(m[0], fmaxf(fabsf(bf16_lo(xa[i])), fabsf(bf16_hi(xa[i]))));
      if (p.shw) {
        const uint4 wv = ld_nc_u4(p.shw + kk);
        const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          d[0] = fmaf(bf16_lo(wa[i]), bf16_lo(xa[i]), d[0]);
          d[0] = fmaf(bf16_hi(wa[i]), bf16_hi(xa[i]), d[0]);
        }
      }
    }
    block_max<1>(m, tb, ctid);
    block_sum<1>(d, tb, ctid);
    const int ex = scale_exponent(m[0]);
    const float sc = ldexpf(1.0f, -ex);
    for (int kk = ctid * 8; kk < H; kk += kConsumerThreads * 8) {
      const uint4 xv = ld_nc_u4(xr + kk);
      const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __half2 hv = __floats2half2_rn(bf16_lo(xa[i]) * sc, bf16_hi(xa[i]) * sc);
        o[i] = *reinterpret_cast<uint32_t*>(&hv);
      }
      *reinterpret_cast<uint4*>(p.x16 + (size_t)n * H + kk) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (ctid == 0) {
      p.xexp[n] = ex;
      p.gsig[n] = p.shw ? 1.0f / (1.0f + expf(-d[0])) : 1.0f;
    }
  }
}

// ------------------------------------------------------------------- top-k
// Selection key, order preserving as unsigned: larger key = larger score.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp routes token n: softmax (selection by logit, weights softmax over
// all E, optionally renormalised over the selected) or sigmoid + bias
// (selection by sigmoid(l) + bias, weights sigmoid(l), optional
// renormalisation, times the routed scaling factor).  Ties go to the lower
// expert index.  Results to tb.sel_e / tb.sel_w in selection order.
template <int PER>
__device__ void topk_token(const Params& p, int n, Tables& tb, int lane) {
  const int E = p.E, k = p.k;
  uint32_t key[PER];
  float lg[PER];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0u;
    lg[i] = -INFINITY;
    if (e < E) {
      const float l = ld_cg_f32(p.logits + (size_t)n * E + e);
      lg[i] = l;
      mx = fmaxf(mx, l);
      float s = l;
      if (p.scoring == 1) s = 1.0f / (1.0f + expf(-l)) + p.bias[e];
      key[i] = order_key(s);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float den = 0.f;
  if (p.scoring == 0) {
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (lane + 32 * i < E) den += expf(lg[i] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  }
  // lane-local best (lowest index among equal keys)
  uint32_t bk = 0u, be = 0xFFFFFFFFu;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (key[i] > bk) { bk = key[i]; be = lane + 32 * i; }
  float wsum = 0.f;
  float wsel = 0.f;  // weight of selection j, held by lane j
  int esel = 0;
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    uint32_t we = __reduce_min_sync(0xffffffffu, (bk == m) ? be : 0xFFFFFFFFu);
    if (we >= (uint32_t)E) we = 0;   // only if fewer than k keys are valid (k <= E is checked)
    float lw = 0.f;
    if (lane == (int)(we & 31u)) {
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (lane + 32 * i == (int)we) { lw = lg[i]; key[i] = 0u; }
      bk = 0u;
      be = 0xFFFFFFFFu;
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (key[i] > bk) { bk = key[i]; be = lane + 32 * i; }
    }
    lw = __shfl_sync(0xffffffffu, lw, we & 31u);
    const float w = (p.scoring == 0) ? expf(lw - mx) / den : 1.0f / (1.0f + expf(-lw));
    wsum += w;
    if (lane == j) { wsel = w; esel = (int)we; }
  }
  if (lane < k) {
    float w = wsel;
    if (p.norm) w = w / wsum;
    if (p.scoring == 1) w *= p.rsf;
    tb.sel_e[n * k + lane] = (int16_t)esel;
    tb.sel_w[n * k + lane] = w;
  }
}

// Routing for all tokens + unique-expert tables (identical in every CTA).
__device__ void routing_phase(const Params& p, int cta, Tables& tb, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int E = p.E, k = p.k, S = p.N * p.k;
  for (int n = warp; n < p.N; n += kConsumerWarps) {
    if (E <= 32) topk_token<1>(p, n, tb, lane);
    else if (E <= 64) topk_token<2>(p, n, tb, lane);
    else if (E <= 128) topk_token<4>(p, n, tb, lane);
    else if (E <= 256) topk_token<8>(p, n, tb, lane);
    else if (E <= 512) topk_token<16>(p, n, tb, lane);
    else topk_token<32>(p, n, tb, lane);
  }
  for (int e = ctid; e < E; e += kConsumerThreads) tb.cnt[e] = 0u;
  consumer_sync();
  for (int s = ctid; s < S; s += kConsumerThreads) atomicAdd(&tb.cnt[tb.sel_e[s]], 1u);
  consumer_sync();
  // scan over experts: (present, count) packed as (1 << 16) | count
  const int per = (E + kConsumerThreads - 1) / kConsumerThreads;   // <= 4
  const int e0 = ctid * per;
  uint32_t loc = 0;
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E && tb.cnt[e]) loc += (1u << 16) | tb.cnt[e];
  }
  uint32_t tot;
  uint32_t pre = block_excl_scan(loc, tb, ctid, &tot);
  for (int i = 0; i < per; ++i) {
    const int e = e0 + i;
    if (e < E && tb.cnt[e]) {
      const uint32_t u = pre >> 16, off = pre & 0xFFFFu, c = tb.cnt[e];
      tb.uexp[u] = (int16_t)e;
      tb.ucnt[u] = (uint16_t)c;
      tb.hoff[u] = (uint16_t)off;
      tb.cnt[e] = u;
      pre += (1u << 16) | c;
    }
  }
  const int U = (int)(tot >> 16);
  consumer_sync();
  // place each slot at hoff[u] + (number of earlier slots routed to the same expert)
  for (int s = ctid; s < S; s += kConsumerThreads) {
    const int e = tb.sel_e[s];
    int pos = 0;
    for (int s2 = 0; s2 < s; ++s2) pos += (tb.sel_e[s2] == e);
    const int u = (int)tb.cnt[e];
    tb.utok[tb.hoff[u] + pos] = (uint8_t)(s / k);
    tb.uw[tb.hoff[u] + pos] = tb.sel_w[s];
  }
  // units (u, token batch), u-major
  uint32_t nb = 0;
  if (ctid < U) nb = (tb.ucnt[ctid] + kTB - 1) / kTB;
  uint32_t ntot;
  const uint32_t ub = block_excl_scan(nb, tb, ctid, &ntot);
  if (ctid < U)
    for (uint32_t b = 0; b < nb; ++b) {
      tb.unit_u[ub + b] = (uint16_t)ctid;
      tb.unit_tb[ub + b] = (uint8_t)b;
    }
  if (ctid == 0) {
    tb.U = U;
    tb.n_units = (int)ntot;
  }
  if (cta == 0) {
    for (int s = ctid; s < S; s += kConsumerThreads) {
      if (p.topk_idx) p.topk_idx[s] = tb.sel_e[s];
      if (p.topk_w) p.topk_w[s] = tb.sel_w[s];
    }
  }
  consumer_sync();
}

// ------------------------------------------------------- row-group plumbing

struct RG {
  int unit, rg;   // unit index within the kind, row group within the unit
  int e, u, tb;   // expert id (routed), unique index, token batch
  int nt;         // tokens in this batch (1..kTB)
};

__device__ __forceinline__ int kind_units(const Params& p, const Tables& tb, int kind) {
  if (kind == KIND_AS || kind == KIND_BS) return p.Is > 0 ? (p.N + kTB - 1) / kTB : 0;
  return tb.n_units;
}

__device__ __forceinline__ void kind_range(const Params& p, const Tables& tb, int kind, int cta,
                                           int G, int& lo, int& hi) {
  const int rpu = p.geo[kind].rows_total / kRows;
  const long long T = (long long)kind_units(p, tb, kind) * rpu;
  lo = (int)(T * cta / G);
  hi = (int)(T * (cta + 1) / G);
}

__device__ __forceinline__ RG decode_rg(const Params& p, const Tables& tb, int kind, int g) {
  RG r;
  const int rpu = p.geo[kind].rows_total / kRows;
  r.unit = g / rpu;
  r.rg = g % rpu;
  if (kind == KIND_AS || kind == KIND_BS) {
    r.u = 0;
    r.e = -1;
    r.tb = r.unit;
    r.nt = min(kTB, p.N - r.tb * kTB);
  } else {
    r.u = tb.unit_u[r.unit];
    r.tb = tb.unit_tb[r.unit];
    r.e = tb.uexp[r.u];
    r.nt = min(kTB, (int)tb.ucnt[r.u] - r.tb * kTB);
  }
  return r;
}

// Token (row of x / out) of batch slot t of an RG.
__device__ __forceinline__ int rg_token(const Tables& tb, int kind, const RG& r, int t) {
  if (kind == KIND_AS || kind == KIND_BS) return r.tb * kTB + t;
  return tb.utok[tb.hoff[r.u] + r.tb * kTB + t];
}

// Global address of weight row `row` (chunk 0) of projection pj.
__device__ __forceinline__ const uint8_t* weight_row(const Params& p, int kind, int pj, int e,
                                                     int row) {
  switch (kind) {
    case KIND_AR: {
      const uint8_t* base = pj == 0 ? p.gq : p.uq;
      return base + ((size_t)e * p.inter + row) * (size_t)(p.H / 2);
    }
    case KIND_BR:
      return p.dq + ((size_t)e * p.H + row) * (size_t)(p.inter / 2);
    case KIND_AS: {
      const uint16_t* base = pj == 0 ? p.shg : p.shu;
      return reinterpret_cast<const uint8_t*>(base + (size_t)row * p.H);
    }
    default:
      return reinterpret_cast<const uint8_t*>(p.shd + (size_t)row * p.Is);
  }
}

__device__ __forceinline__ const uint8_t* scale_row(const Params& p, int kind, int pj, int e,
                                                    int row) {
  const int sr = p.geo[kind].sr;
  if (kind == KIND_AR) {
    const uint8_t* base = pj == 0 ? p.gsc : p.usc;
    return base + ((size_t)e * p.inter + row) * (size_t)sr;
  }
  return p.dsc + ((size_t)e * p.H + row) * (size_t)sr;
}

// ------------------------------------------------------------------ producer

__device__ __forceinline__ uint32_t stage_tx_bytes(const Geo& g, int kind, int nt) {
  uint32_t b = (uint32_t)(g.nproj * kRows * g.row_bytes);
  if (g.scale_mode == SCALES_PER_ROW) b += (uint32_t)(g.nproj * kRows * g.scale_bytes);
  if (g.scale_mode == SCALES_BLOCK) b += (uint32_t)(g.nproj * kRows * g.sr);
  if (kind == KIND_AS || kind == KIND_AR) b += (uint32_t)(nt * g.Kc * 2);
  return b;
}

__device__ void produce_stage(const Params& p, const Tables& tb, int kind, const RG& r, int c,
                              uint8_t* st, uint64_t* full, int lane) {
  const Geo& g = p.geo[kind];
  if (lane == 0) mbar_arrive_expect_tx(full, stage_tx_bytes(g, kind, r.nt));
  __syncwarp();
  const int row = r.rg * kRows + lane;
  for (int pj = 0; pj < g.nproj; ++pj) {
    const uint8_t* src = weight_row(p, kind, pj, r.e, row) + (size_t)c * g.row_bytes;
    bulk_g2s(st + (pj * kRows + lane) * g.row_stride, src, (uint32_t)g.row_bytes, full);
    if (g.scale_mode == SCALES_PER_ROW) {
      const uint8_t* ss = scale_row(p, kind, pj, r.e, row) + (size_t)c * g.scale_bytes;
      bulk_g2s(st + g.scale_off + (pj * kRows + lane) * g.scale_stride, ss,
               (uint32_t)g.scale_bytes, full);
    }
  }
  if (g.scale_mode == SCALES_BLOCK && lane < g.nproj) {
    const uint8_t* ss = scale_row(p, kind, lane, r.e, r.rg * kRows);
    bulk_g2s(st + g.scale_off + lane * kRows * g.sr, ss, (uint32_t)(kRows * g.sr), full);
  }
  if ((kind == KIND_AS || kind == KIND_AR) && lane < r.nt) {
    const int n = rg_token(tb, kind, r, lane);
    const uint16_t* xs = (kind == KIND_AR) ? p.x16 : p.x;
    bulk_g2s(st + g.opnd_off + lane * g.Kc * 2, xs + (size_t)n * p.H + (size_t)c * g.Kc,
             (uint32_t)(g.Kc * 2), full);
  }
}

struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  int nstages, stage_bytes;
};

// Streams every stage of one kind's row groups; returns false on abort.
__device__ bool produce_kind(const Params& p, Tables& tb, const Ring& ring, int kind, int cta,
                             int G, int& ctr, int lane) {
  if (kind_units(p, tb, kind) == 0) return true;
  int lo, hi;
  kind_range(p, tb, kind, cta, G, lo, hi);
  const Geo& geo = p.geo[kind];
  for (int gi = lo; gi < hi; ++gi) {
    const RG r = decode_rg(p, tb, kind, gi);
    for (int c = 0; c < geo.nchunks; ++c) {
      const int slot = ctr % ring.nstages;
      const uint32_t round = (uint32_t)(ctr / ring.nstages);
      if (*(volatile int*)&tb.abort) return false;
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(ring.empty + slot, (round & 1u) ^ 1u, p.timeout_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          atomicOr(p.ctrl + 2, kErrTimeoutProducer);
          *(volatile int*)&tb.abort = 1;
        }
        return false;
      }
      produce_stage(p, tb, kind, r, c, ring.base + (size_t)slot * ring.stage_bytes,
                    ring.full + slot, lane);
      ++ctr;
    }
  }
  return true;
}

// ------------------------------------------------------------------ consumer

// One stage of FP4 weights: lane = weight row, steps [s0, s1) of this warp.
template <int FMT, int NPROJ>
__device__ __forceinline__ void compute_fp4(const Geo& g, uint32_t st, int c, uint32_t obase,
                                            int otstride, int nt, int s0, int s1, int lane,
                                            float (&acc)[2][kTB]) {
  for (int s = s0; s < s1; ++s) {
    uint32_t wd[NPROJ][16];
    uint32_t scl[NPROJ];
#pragma unroll
    for (int pj = 0; pj < NPROJ; ++pj) {
      const uint4 w = lds128(st + (pj * kRows + lane) * g.row_stride + s * 16);
      uint32_t o[4];
      e2m1x8_to_f16x2x4(w.x, o);
      wd[pj][0] = o[0]; wd[pj][1] = o[1]; wd[pj][2] = o[2]; wd[pj][3] = o[3];
      e2m1x8_to_f16x2x4(w.y, o);
      wd[pj][4] = o[0]; wd[pj][5] = o[1]; wd[pj][6] = o[2]; wd[pj][7] = o[3];
      e2m1x8_to_f16x2x4(w.z, o);
      wd[pj][8] = o[0]; wd[pj][9] = o[1]; wd[pj][10] = o[2]; wd[pj][11] = o[3];
      e2m1x8_to_f16x2x4(w.w, o);
      wd[pj][12] = o[0]; wd[pj][13] = o[1]; wd[pj][14] = o[2]; wd[pj][15] = o[3];
      if (FMT == FMT_NVFP4) {
        uint32_t sa;
        if (g.scale_mode == SCALES_PER_ROW)
          sa = st + g.scale_off + (pj * kRows + lane) * g.scale_stride + s * 2;
        else
          sa = st + g.scale_off + (pj * kRows + lane) * g.sr + (c * g.Kc + s * 32) / 16;
        scl[pj] = e4m3x2_to_f16x2(lds_u16(sa));
      } else {
        uint32_t sa;
        if (g.scale_mode == SCALES_PER_ROW)
          sa = st + g.scale_off + (pj * kRows + lane) * g.scale_stride + s;
        else
          sa = st + g.scale_off + (pj * kRows + lane) * g.sr + (c * g.Kc + s * 32) / 32;
        scl[pj] = __float_as_uint(e8m0_to_f32(lds_u8(sa)));
      }
    }
#pragma unroll
    for (int t = 0; t < kTB; ++t) {
      if (t < nt) {
        const uint32_t oa = obase + t * otstride + s * 64;
        uint32_t xo[16];
        const uint4 x0 = lds128(oa), x1 = lds128(oa + 16), x2 = lds128(oa + 32),
                    x3 = lds128(oa + 48);
        xo[0] = x0.x; xo[1] = x0.y; xo[2] = x0.z; xo[3] = x0.w;
        xo[4] = x1.x; xo[5] = x1.y; xo[6] = x1.z; xo[7] = x1.w;
        xo[8] = x2.x; xo[9] = x2.y; xo[10] = x2.z; xo[11] = x2.w;
        xo[12] = x3.x; xo[13] = x3.y; xo[14] = x3.z; xo[15] = x3.w;
#pragma unroll
        for (int pj = 0; pj < NPROJ; ++pj) {
          if (FMT == FMT_NVFP4) {
            uint32_t p0 = hmul2(wd[pj][0], xo[0]);
            uint32_t p1 = hmul2(wd[pj][8], xo[8]);
#pragma unroll
            for (int i = 1; i < 8; ++i) {
              p0 = hfma2(wd[pj][i], xo[i], p0);
              p1 = hfma2(wd[pj][8 + i], xo[8 + i], p1);
            }
            float a = acc[pj][t];
            a = fma_f16pair_scalar(p0, (uint16_t)(scl[pj] & 0xFFFFu), a);
            a = fma_f16pair_scalar(p1, (uint16_t)(scl[pj] >> 16), a);
            acc[pj][t] = a;
          } else {
            uint32_t p0 = hmul2(wd[pj][0], xo[0]);
            uint32_t p1 = hmul2(wd[pj][1], xo[1]);
#pragma unroll
            for (int i = 2; i < 16; i += 2) {
              p0 = hfma2(wd[pj][i], xo[i], p0);
              p1 = hfma2(wd[pj][i + 1], xo[i + 1], p1);
            }
            const float2 f0 = f16x2_to_f32x2(p0), f1 = f16x2_to_f32x2(p1);
            acc[pj][t] = fmaf((f0.x + f0.y) + (f1.x + f1.y), __uint_as_float(scl[pj]), acc[pj][t]);
          }
        }
      }
    }
  }
}

// One stage of BF16 weights (shared expert).
template <int NPROJ>
__device__ __forceinline__ void compute_bf16(const Geo& g, uint32_t st, uint32_t obase,
                                             int otstride, int nt, int s0, int s1, int lane,
                                             float (&acc)[2][kTB]) {
  for (int s = s0; s < s1; ++s) {
    uint32_t wv[NPROJ][16];
#pragma unroll
    for (int pj = 0; pj < NPROJ; ++pj) {
      const uint32_t wa = st + (pj * kRows + lane) * g.row_stride + s * 64;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = lds128(wa + q * 16);
        wv[pj][4 * q + 0] = w.x; wv[pj][4 * q + 1] = w.y;
        wv[pj][4 * q + 2] = w.z; wv[pj][4 * q + 3] = w.w;
      }
    }
#pragma unroll
    for (int t = 0; t < kTB; ++t) {
      if (t < nt) {
        const uint32_t oa = obase + t * otstride + s * 64;
        uint32_t xo[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 x = lds128(oa + q * 16);
          xo[4 * q + 0] = x.x; xo[4 * q + 1] = x.y; xo[4 * q + 2] = x.z; xo[4 * q + 3] = x.w;
        }
#pragma unroll
        for (int pj = 0; pj < NPROJ; ++pj) {
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            a0 = fma2_bf16_to_f32(wv[pj][i], xo[i], a0);
            a1 = fma2_bf16_to_f32(wv[pj][i + 1], xo[i + 1], a1);
          }
          acc[pj][t] += a0 + a1;
        }
      }
    }
  }
}

// Stage activations of a down-projection unit into hbuf: routed h as f16
// scaled per token by a power of two, shared h as BF16.
__device__ void stage_hbuf(const Params& p, Tables& tb, int kind, const RG& r, uint8_t* hbuf,
                           int ctid) {
  const int K = p.geo[kind].K;
  if (kind == KIND_BR) {
    float m[kTB];
#pragma unroll
    for (int t = 0; t < kTB; ++t) m[t] = 0.f;
#pragma unroll
    for (int t = 0; t < kTB; ++t) {
      if (t < r.nt) {
        const float* src = p.h + (size_t)(tb.hoff[r.u] + r.tb * kTB + t) * p.inter;
        for (int kk = ctid * 4; kk < K; kk += kConsumerThreads * 4) {
          const float4 v = ld_cg_f32x4(src + kk);
          m[t] = fmaxf(m[t], fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
      }
    }
    block_max<kTB>(m, tb, ctid);
#pragma unroll
    for (int t = 0; t < kTB; ++t) {
      if (t < r.nt) {
        const int ex = scale_exponent(m[t]);
        if (ctid == 0) tb.hexp[t] = ex;
        const float sc = ldexpf(1.0f, -ex);
        const float* src = p.h + (size_t)(tb.hoff[r.u] + r.tb * kTB + t) * p.inter;
        __half* dst = reinterpret_cast<__half*>(hbuf) + (size_t)t * K;
        for (int kk = ctid * 4; kk < K; kk += kConsumerThreads * 4) {
          const float4 v = ld_cg_f32x4(src + kk);
          __half2 a = __floats2half2_rn(v.x * sc, v.y * sc);
          __half2 b = __floats2half2_rn(v.z * sc, v.w * sc);
          *reinterpret_cast<__half2*>(dst + kk) = a;
          *reinterpret_cast<__half2*>(dst + kk + 2) = b;
        }
      }
    }
  } else {
    for (int t = 0; t < r.nt; ++t) {
      const int n = r.tb * kTB + t;
      const float* src = p.hs + (size_t)n * p.Is;
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(hbuf) + (size_t)t * K;
      for (int kk = ctid * 4; kk < K; kk += kConsumerThreads * 4) {
        const float4 v = ld_cg_f32x4(src + kk);
        *reinterpret_cast<__nv_bfloat162*>(dst + kk) = __floats2bfloat162_rn(v.x, v.y);
        *reinterpret_cast<__nv_bfloat162*>(dst + kk + 2) = __floats2bfloat162_rn(v.z, v.w);
      }
    }
  }
  consumer_sync();
}

// Reduce the 8 warps' partial sums of the current RG and apply its epilogue.
__device__ void rg_epilogue(const Params& p, Tables& tb, int kind, const RG& r, float* red,
                            const float (&acc)[2][kTB], int ctid, uint32_t b_units) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const Geo& g = p.geo[kind];
#pragma unroll
  for (int pj = 0; pj < 2; ++pj)
#pragma unroll
    for (int t = 0; t < kTB; ++t)
      if (pj < g.nproj) red[((warp * 2 + pj) * kTB + t) * 32 + lane] = acc[pj][t];
  consumer_sync();
  const bool aborted = *(volatile int*)&tb.abort;
  if (ctid < r.nt * 32 && !aborted) {
    const int t = ctid >> 5, j = ctid & 31;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      s0 += red[((w * 2 + 0) * kTB + t) * 32 + j];
      if (g.nproj == 2) s1 += red[((w * 2 + 1) * kTB + t) * 32 + j];
    }
    const int row = r.rg * kRows + j;
    const int n = rg_token(tb, kind, r, t);
    if (kind == KIND_AR) {
      const float xs = ldexpf(1.0f, ld_cg_s32(p.xexp + n));
      const float gg = s0 * xs * (p.g2 ? p.g2[r.e] : 1.0f);
      const float uu = s1 * xs * (p.u2 ? p.u2[r.e] : 1.0f);
      p.h[(size_t)(tb.hoff[r.u] + r.tb * kTB + t) * p.inter + row] = silu(gg) * uu;
    } else if (kind == KIND_AS) {
      p.hs[(size_t)n * p.Is + row] = silu(s0) * s1;
    } else if (kind == KIND_BR) {
      const float y = s0 * ldexpf(1.0f, tb.hexp[t]) * (p.d2 ? p.d2[r.e] : 1.0f);
      red_add_f32(p.acc + (size_t)n * p.H + row, y * tb.uw[tb.hoff[r.u] + r.tb * kTB + t]);
    } else {
      red_add_f32(p.acc + (size_t)n * p.H + row, s0 * ld_cg_f32(p.gsig + n));
    }
  }
  if (kind == KIND_BR || kind == KIND_BS) {
    __threadfence();
    consumer_sync();
    if (ctid == 0) {
      int fin = 0;
      if (!aborted) {
        const uint32_t old = atomicAdd(p.rbcnt + r.rg, 1u);
        fin = (old + 1u == b_units);
        if (fin) __threadfence();
      }
      tb.fin = fin;
    }
    consumer_sync();
    if (tb.fin) {
      for (int i = ctid; i < p.N * kRows; i += kConsumerThreads) {
        const int n = i / kRows, row = r.rg * kRows + (i % kRows);
        const float v = ld_cg_f32(p.acc + (size_t)n * p.H + row);
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        p.out[(size_t)n * p.H + row] = *reinterpret_cast<const uint16_t*>(&b);
      }
    }
  }
  consumer_sync();
}

struct ConsumerCtx {
  uint8_t* ring_base;
  uint64_t* full;
  uint64_t* empty;
  int nstages, stage_bytes;
  float* red;
  uint8_t* hbuf;
};

// Consumes every stage of one kind's row groups.
__device__ void consume_kind(const Params& p, Tables& tb, const ConsumerCtx& cx, int kind,
                             int cta, int G, int& ctr, int ctid, uint32_t b_units) {
  if (kind_units(p, tb, kind) == 0) return;
  const int warp = ctid >> 5, lane = ctid & 31;
  int lo, hi;
  kind_range(p, tb, kind, cta, G, lo, hi);
  const Geo& g = p.geo[kind];
  const int spc = g.Kc / 32;
  const int s0 = warp * spc / kConsumerWarps, s1 = (warp + 1) * spc / kConsumerWarps;
  for (int gi = lo; gi < hi; ++gi) {
    const RG r = decode_rg(p, tb, kind, gi);
    if ((kind == KIND_BR || kind == KIND_BS) &&
        (tb.hb_kind != kind || tb.hb_unit != r.unit)) {
      consumer_sync();
      if (!*(volatile int*)&tb.abort) stage_hbuf(p, tb, kind, r, cx.hbuf, ctid);
      if (ctid == 0) {
        tb.hb_kind = kind;
        tb.hb_unit = r.unit;
      }
      consumer_sync();
    }
    float acc[2][kTB];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int t = 0; t < kTB; ++t) acc[a][t] = 0.f;
    for (int c = 0; c < g.nchunks; ++c) {
      const int slot = ctr % cx.nstages;
      const uint32_t round = (uint32_t)(ctr / cx.nstages);
      ++ctr;
      bool ok = !*(volatile int*)&tb.abort;
      if (ok) ok = mbar_wait_bounded(cx.full + slot, round & 1u, p.timeout_ns);
      if (!ok) {
        if (lane == 0 && !*(volatile int*)&tb.abort) {
          atomicOr(p.ctrl + 2, kErrTimeoutStage);
          *(volatile int*)&tb.abort = 1;
        }
      } else {
        const uint32_t st = smem_u32(cx.ring_base + (size_t)slot * cx.stage_bytes);
        uint32_t obase;
        int ots;
        if (kind == KIND_AS || kind == KIND_AR) {
          obase = st + g.opnd_off;
          ots = g.Kc * 2;
        } else {
          obase = smem_u32(cx.hbuf) + c * g.Kc * 2;
          ots = g.K * 2;
        }
        if (g.fmt == FMT_BF16) {
          if (g.nproj == 2) compute_bf16<2>(g, st, obase, ots, r.nt, s0, s1, lane, acc);
          else compute_bf16<1>(g, st, obase, ots, r.nt, s0, s1, lane, acc);
        } else if (g.fmt == FMT_NVFP4) {
          if (g.nproj == 2) compute_fp4<FMT_NVFP4, 2>(g, st, c, obase, ots, r.nt, s0, s1, lane, acc);
          else compute_fp4<FMT_NVFP4, 1>(g, st, c, obase, ots, r.nt, s0, s1, lane, acc);
        } else {
          if (g.nproj == 2) compute_fp4<FMT_MXFP4, 2>(g, st, c, obase, ots, r.nt, s0, s1, lane, acc);
          else compute_fp4<FMT_MXFP4, 1>(g, st, c, obase, ots, r.nt, s0, s1, lane, acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cx.empty + slot);
    }
    rg_epilogue(p, tb, kind, r, cx.red, acc, ctid, b_units);
  }
}

// ------------------------------------------------------------------- kernel

__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Tables& tb = *reinterpret_cast<Tables*>(smem + p.smem_tab_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.smem_bar_off);
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxStages;
  uint64_t* rr = bars + 2 * kMaxStages;  // routing tables ready (consumers -> producer)
  const int tid = threadIdx.x;
  const int cta = blockIdx.x, G = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < p.nstages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kConsumerWarps);
    }
    mbar_init(rr, 1);
    fence_mbar_init();
    tb.abort = 0;
    tb.hb_kind = -1;
    tb.hb_unit = -1;
    tb.n_units = 0;
    tb.U = 0;
  }
  __syncthreads();

  const uint32_t b_units_shared = (p.Is > 0) ? (uint32_t)((p.N + kTB - 1) / kTB) : 0u;

  if (tid >= kConsumerThreads) {
    // ------------------------------------------------------------ producer
    const int lane = tid - kConsumerThreads;
    if (p.route_only) return;
    Ring ring{smem + p.smem_ring_off, full, empty, p.nstages, p.stage_bytes};
    int ctr = 0;
    bool ok = produce_kind(p, tb, ring, KIND_AS, cta, G, ctr, lane);
    if (ok) {
      bool got = true;
      if (lane == 0) got = mbar_wait_bounded(rr, 0, p.timeout_ns);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) {
          atomicOr(p.ctrl + 2, kErrTimeoutProducer);
          *(volatile int*)&tb.abort = 1;
        }
        ok = false;
      }
    }
    if (ok) {
      fence_proxy_async_global();   // x16 was written by other CTAs before B1
      ok = produce_kind(p, tb, ring, KIND_AR, cta, G, ctr, lane) &&
           produce_kind(p, tb, ring, KIND_BR, cta, G, ctr, lane) &&
           produce_kind(p, tb, ring, KIND_BS, cta, G, ctr, lane);
    }
    if (!ok && lane == 0) {
      // drain: wait (bounded) for copies still in flight into our stages
      const int first = ctr > p.nstages ? ctr - p.nstages : 0;
      for (int i = first; i < ctr; ++i)
        mbar_wait_bounded(full + (i % p.nstages), (uint32_t)(i / p.nstages) & 1u, p.timeout_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = tid;
  float* red = reinterpret_cast<float*>(smem + p.smem_red_off);
  ConsumerCtx cx{smem + p.smem_ring_off, full, empty, p.nstages, p.stage_bytes, red,
                 smem + p.smem_hbuf_off};

  // P0: router, token prep, zero the accumulator
  router_phase(p, cta, G, tb, ctid);
  if (!p.route_only) {
    token_prep(p, cta, G, tb, ctid);
    const size_t nacc = (size_t)p.N * p.H;
    for (size_t i = (size_t)cta * kConsumerThreads + ctid; i < nacc; i += (size_t)G * kConsumerThreads)
      p.acc[i] = 0.f;
    for (int i = cta * kConsumerThreads + ctid; i < p.H / kRows; i += G * kConsumerThreads)
      p.rbcnt[i] = 0u;
  }
  __threadfence();
  consumer_sync();
  uint32_t gen = 0;
  if (ctid == 0) gen = grid_arrive(p.ctrl, (uint32_t)G);

  int ctr = 0;
  if (!p.route_only) consume_kind(p, tb, cx, KIND_AS, cta, G, ctr, ctid, 0);

  if (ctid == 0) {
    if (!grid_wait(p.ctrl, gen, p.timeout_ns)) {
      atomicOr(p.ctrl + 2, kErrTimeoutBarrier);
      *(volatile int*)&tb.abort = 1;
    }
  }
  consumer_sync();
  if (*(volatile int*)&tb.abort) {
    if (ctid == 0) mbar_arrive(rr);
    return;   // producer sees abort / rr and drains
  }

  // P1: routing
  routing_phase(p, cta, tb, ctid);
  if (p.route_only) return;
  if (ctid == 0) mbar_arrive(rr);

  const uint32_t b_units = (uint32_t)tb.n_units + b_units_shared;

  // P2: routed gate/up
  consume_kind(p, tb, cx, KIND_AR, cta, G, ctr, ctid, b_units);
  __threadfence();
  consumer_sync();
  if (ctid == 0) {
    const uint32_t gen2 = grid_arrive(p.ctrl, (uint32_t)G);
    if (!*(volatile int*)&tb.abort && !grid_wait(p.ctrl, gen2, p.timeout_ns)) {
      atomicOr(p.ctrl + 2, kErrTimeoutBarrier);
      *(volatile int*)&tb.abort = 1;
    }
  }
  consumer_sync();

  // P3: down projections (routed, then shared) + finalize
  consume_kind(p, tb, cx, KIND_BR, cta, G, ctr, ctid, b_units);
  consume_kind(p, tb, cx, KIND_BS, cta, G, ctr, ctid, b_units);
}

// ------------------------------------------------------------------- host

static int pad_odd16(int b) { return ((b / 16) % 2 == 1) ? b : b + 16; }

static int largest_divisor(int K, int mult, int cap) {
  int best = 0;
  for (int c = mult; c <= cap && c <= K; c += mult)
    if (K % c == 0) best = c;
  return best;
}

static bool plan_kind(Geo& g, int fmt, int nproj, int K, int rows, bool with_operand) {
  g.fmt = fmt;
  g.nproj = nproj;
  g.K = K;
  g.rows_total = rows;
  g.opnd_off = -1;
  if (K % 32 != 0 || rows % kRows != 0 || K <= 0 || rows <= 0) return false;
  int off = 0;
  if (fmt == FMT_BF16) {
    g.Kc = largest_divisor(K, 32, 256);
    g.row_bytes = g.Kc * 2;
    g.row_stride = pad_odd16(g.row_bytes);
    g.scale_mode = SCALES_NONE;
    g.sr = g.scale_bytes = g.scale_stride = 0;
    off = nproj * kRows * g.row_stride;
    g.scale_off = off;
  } else {
    const int gs = (fmt == FMT_NVFP4) ? 16 : 32;
    g.sr = K / gs;
    int kc = 0;
    if (g.sr % 16 == 0) kc = largest_divisor(K, 16 * gs, 1024);
    if (kc) {
      g.scale_mode = SCALES_PER_ROW;
      g.Kc = kc;
      g.scale_bytes = kc / gs;
      g.scale_stride = pad_odd16(g.scale_bytes);
    } else {
      g.scale_mode = SCALES_BLOCK;
      g.Kc = largest_divisor(K, 32, 1024);
      g.scale_bytes = g.sr;
      g.scale_stride = g.sr;
    }
    g.row_bytes = g.Kc / 2;
    g.row_stride = pad_odd16(g.row_bytes);
    off = nproj * kRows * g.row_stride;
    g.scale_off = off;
    if (g.scale_mode == SCALES_PER_ROW) off += nproj * kRows * g.scale_stride;
    else off += (nproj * kRows * g.sr + 15) / 16 * 16;
  }
  if (g.Kc <= 0) return false;
  g.nchunks = K / g.Kc;
  if (with_operand) {
    g.opnd_off = off;
    off += kTB * g.Kc * 2;
  }
  g.stage_bytes = (off + 127) / 128 * 128;
  return true;
}

bool plan_decode(Params& p, int smem_budget) {
  const int wf = (p.fmt == 0) ? FMT_NVFP4 : FMT_MXFP4;
  if (!plan_kind(p.geo[KIND_AR], wf, 2, p.H, p.inter, true)) return false;
  if (!plan_kind(p.geo[KIND_BR], wf, 1, p.inter, p.H, false)) return false;
  int stage = std::max(p.geo[KIND_AR].stage_bytes, p.geo[KIND_BR].stage_bytes);
  int hb = kTB * p.inter * 2;
  if (p.Is > 0) {
    if (!plan_kind(p.geo[KIND_AS], FMT_BF16, 2, p.H, p.Is, true)) return false;
    if (!plan_kind(p.geo[KIND_BS], FMT_BF16, 1, p.Is, p.H, false)) return false;
    stage = std::max(stage, std::max(p.geo[KIND_AS].stage_bytes, p.geo[KIND_BS].stage_bytes));
    hb = std::max(hb, kTB * p.Is * 2);
  } else {
    p.geo[KIND_AS] = p.geo[KIND_AR];
    p.geo[KIND_BS] = p.geo[KIND_BR];
    p.geo[KIND_AS].rows_total = kRows;
    p.geo[KIND_BS].rows_total = kRows;
  }
  const int red = kConsumerWarps * 2 * kTB * 32 * 4;
  const int tab = ((int)sizeof(Tables) + 127) / 128 * 128;
  const int bars = (2 * kMaxStages + 1) * 8;
  const int fixed = red + ((hb + 127) / 128 * 128) + tab + ((bars + 127) / 128 * 128);
  int ns = (smem_budget - fixed) / stage;
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return false;
  p.nstages = ns;
  p.stage_bytes = stage;
  p.hbuf_bytes = hb;
  p.smem_ring_off = 0;
  p.smem_red_off = ns * stage;
  p.smem_hbuf_off = p.smem_red_off + red;
  p.smem_tab_off = p.smem_hbuf_off + (hb + 127) / 128 * 128;
  p.smem_bar_off = p.smem_tab_off + tab;
  p.smem_total = p.smem_bar_off + (bars + 127) / 128 * 128;
  return p.smem_total <= smem_budget;
}

int decode_smem_budget(int device) {
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
    return 0;
  return v - 1024;   // headroom for static / reserved shared memory
}

int decode_grid(int device, int smem_bytes) {
  int sms = 0, nb = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  if (cudaFuncSetAttribute(moe_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_bytes) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, moe_decode_kernel, kThreads,
                                                    smem_bytes) != cudaSuccess)
    return 0;
  if (nb < 1) return 0;
  return sms;   // one CTA per SM
}

// The kernel's dynamic shared-memory limit was raised to the device budget
// once, in decode_grid.
cudaError_t launch_decode(const Params& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem_total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_decode_kernel, p);
}

}  // namespace moe
