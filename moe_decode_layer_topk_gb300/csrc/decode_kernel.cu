// Fused MoE decode-layer forward for small N on sm_103a (one launch per call).
//
// Computes, for N token rows, the chain of forward_k3.rs (doc comment of
// MoeLayer::forward_k3: gate GEMV -> batched top-k -> expert gate+up ->
// SiLU+down -> weighted sum + shared blend) with the routed experts
// accumulated as routing-weighted FP32 sums and cast to BF16 once at the end
// (forward_atomic_c4.rs, doc comment of forward_atomic_c4_decode).
//
// Execution model: a persistent grid, one CTA per SM, every CTA resident at
// once (cooperative launch).  Each CTA has 8 compute ("consumer") warps and
// one producer thread that streams weights into a ring of shared-memory
// stages with TMA (2D tensor-map boxes of 32 rows x 128 bytes, 128-byte
// swizzle), completion tracked by mbarriers.
//
// Phases of one call (per CTA):
//   P0  router GEMV for rows e = cta, cta+G, ... (128-bit loads); token prep
//       (f16 copy of x scaled by a power of two, shared-expert gate) on the
//       last CTAs; zero the FP32 accumulator and the row-block counters.
//   --  grid barrier B1 (arrive).  Shared-expert gate/up row groups need only
//       x, so they are streamed and computed before waiting on B1.
//   P1  every CTA computes the same top-k for all N tokens and the same table
//       of unique experts (ascending id), per-expert token lists and
//       (expert, token batch) units: each routed expert's weights are then read
//       once for all its tokens (forward_batched.rs: "streams its weights once
//       for all rows").
//   P2  routed gate/up row groups -> h = SiLU(g)*u (FP32, workspace).
//   --  grid barrier B2 (the producer keeps prefetching down weights).
//   P3  down row groups (routed, then shared) -> routing-weighted FP32 red.add
//       into acc[N,H]; at the end each CTA bumps the completion counters of the
//       32-row output blocks it touched, and the CTA that completes a block
//       casts it to BF16 into out (no third grid barrier).
//
// Work split: a row group (RG) is 32 consecutive weight rows of one
// (expert, token batch) unit; each kind's RG list is split evenly over the
// CTAs.  Inside a CTA, lane j of every consumer warp owns row j of the RG and
// the 8 warps split the K range; partial sums meet in shared memory at the
// end of the RG.  The 128-byte swizzle of the boxes makes the lane-per-row
// 128-bit shared loads conflict free; activations are read as broadcasts.
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
#include "routing.cuh"

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
  uint16_t brg[kMaxRgList];    // output row blocks this CTA added to (pending)
  uint8_t bfin[kMaxRgList];    // ... and whether this CTA completed them
  int nbrg;
  int U, n_units;
  int abort;                   // set when a bounded wait expired
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
__device__ __forceinline__ bool aborted(const Tables& tb) {
  return *(volatile const int*)&tb.abort != 0;
}
__device__ __forceinline__ void set_abort(const Params& p, Tables& tb, uint32_t bit) {
  atomicOr(&p.ctrl->error, bit);
  *(volatile int*)&tb.abort = 1;
}

// Sum / max over the 256 consumer threads of M values each (all threads get it).
template <int M, bool MAX>
__device__ __forceinline__ void block_reduce(float (&v)[M], Tables& tb, int ctid) {
  const int lane = ctid & 31, warp = ctid >> 5;
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float t = __shfl_xor_sync(0xffffffffu, v[m], o);
      v[m] = MAX ? fmaxf(v[m], t) : v[m] + t;
    }
  if (lane == 0)
#pragma unroll
    for (int m = 0; m < M; ++m) tb.rscratch[warp * 8 + m] = v[m];
  consumer_sync();
#pragma unroll
  for (int m = 0; m < M; ++m) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w)
      s = MAX ? fmaxf(s, tb.rscratch[w * 8 + m]) : s + tb.rscratch[w * 8 + m];
    v[m] = s;
  }
  consumer_sync();
}

// Exclusive scan over the 256 consumer threads (one value each).
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
// The workspace keeps one monotonic 64-bit arrival counter.  Every CTA
// arrives exactly twice per call, so at kernel start the counter lies in
// [base, base + G) with base a multiple of 2G (no CTA can pass B1 before all
// have arrived).  Arrivals are fire-and-forget release reductions; a waiter
// polls with acquire loads until the counter reaches base + G*(b+1).
__device__ __forceinline__ void grid_arrive(Ctrl* c) { red_release_add_u64(&c->arrivals, 1ull); }

__device__ bool grid_wait(Ctrl* c, unsigned long long target, uint64_t budget_ns) {
  if (ld_acquire_u64(&c->arrivals) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_u64(&c->arrivals) < target) {
    if (global_timer_ns() - t0 > budget_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- router
// logits[n, e] = sum_h x[n, h] * Wr[e, h], FP32 accumulation of BF16 products.
__device__ __noinline__ void router_phase(const Params& p, int cta, int G, Tables& tb, int ctid) {
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
      block_reduce<8, false>(acc, tb, ctid);
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

// Per-token prep on the last CTAs (those past the router rows when E < G):
// x16 = f16(x * 2^-xexp) and the shared-expert gate sigmoid(w_s . x).
__device__ __noinline__ void token_prep(const Params& p, int cta, int G, Tables& tb, int ctid) {
  const int H = p.H;
  for (int n = G - 1 - cta; n < p.N; n += G) {
    const uint16_t* xr = p.x + (size_t)n * H;
    float md[2] = {0.f, 0.f};
    float d[1] = {0.f};
    for (int kk = ctid * 8; kk < H; kk += kConsumerThreads * 8) {
      const uint4 xv = ld_nc_u4(xr + kk);
      const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        md[0] = fmaxf(md[0], fmaxf(fabsf(bf16_lo(xa[i])), fabsf(bf16_hi(xa[i]))));
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
    float m1[1] = {md[0]};
    block_reduce<1, true>(m1, tb, ctid);
    block_reduce<1, false>(d, tb, ctid);
    const int ex = scale_exponent(m1[0]);
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
// One warp routes token n (logits from L2: other CTAs wrote them) into the
// per-slot selection tables.
template <int PER>
__device__ __forceinline__ void topk_token(int E, int k, int scoring, int norm, float rsf,
                                           const float* bias, const float* lrow, int n,
                                           Tables& tb, int lane) {
  float lg[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    lg[i] = (e < E) ? ld_cg_f32(lrow + e) : -INFINITY;
  }
  int se = 0;
  float sw = 0.f;
  topk_warp<PER>(E, k, scoring, norm, rsf, bias, lg, lane, &se, &sw);
  if (lane < k) {
    tb.sel_e[n * k + lane] = (int16_t)se;
    tb.sel_w[n * k + lane] = sw;
  }
}

// Small case (S = N*k <= 32, every expert has <= kTB tokens): the same tables
// as build_tables, from one slot per lane in registers.
__device__ __forceinline__ bool build_tables_small(int k, int S, Tables& tb, int lane) {
  const bool v = lane < S;
  const int e = v ? tb.sel_e[lane] : -1 - lane;
  const float wv = v ? tb.sel_w[lane] : 0.f;
  const uint32_t lt = (1u << lane) - 1u;
  const uint32_t peers = __match_any_sync(0xffffffffu, e);
  const int cnt = __popc(peers), pos = __popc(peers & lt);
  if (!__all_sync(0xffffffffu, !v || cnt <= kTB)) return false;
  const bool isfirst = v && pos == 0;
  const uint32_t fmask = __ballot_sync(0xffffffffu, isfirst);
  const int leader = __ffs(peers) - 1;
  const int u = __shfl_sync(0xffffffffu, __popc(fmask & lt), leader);   // unique index
  int inc = isfirst ? cnt : 0;                       // slot offsets over first lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  const int hoff = __shfl_sync(0xffffffffu, inc - (isfirst ? cnt : 0), leader);
  if (v) {
    tb.utok[hoff + pos] = (uint8_t)(lane / k);
    tb.uw[hoff + pos] = wv;
  }
  if (isfirst) {
    tb.uexp[u] = (int16_t)e;
    tb.ucnt[u] = (uint16_t)cnt;
    tb.hoff[u] = (uint16_t)hoff;
    tb.unit_u[u] = (uint16_t)u;
    tb.unit_tb[u] = 0;
  }
  if (lane == 0) {
    tb.U = __popc(fmask);
    tb.n_units = __popc(fmask);
  }
  return true;
}

// Unique experts and per-expert token lists from the S = N*k selections, by
// one warp.  Unique experts are ordered by their first selection slot
// (token-major), tokens of an expert by token index; every CTA builds the
// same tables from the same routing.
__device__ __forceinline__ void build_tables(int E, int k, int S, Tables& tb, int lane) {
  uint32_t* first = tb.cnt;              // first slot of each expert, then its unique index
  for (int e = lane; e < E; e += 32) first[e] = 0xFFFFFFFFu;
  __syncwarp();
  for (int s = lane; s < S; s += 32) atomicMin(&first[tb.sel_e[s]], (uint32_t)s);
  __syncwarp();
  const uint32_t lt = (1u << lane) - 1u;
  int U = 0;
  for (int b = 0; b < S; b += 32) {          // unique experts in first-slot order
    const int s = b + lane;
    const int e = (s < S) ? tb.sel_e[s] : 0;
    const bool isfirst = (s < S) && first[e] == (uint32_t)s;
    const uint32_t mask = __ballot_sync(0xffffffffu, isfirst);
    if (isfirst) {
      const int u = U + __popc(mask & lt);
      tb.uexp[u] = (int16_t)e;
      tb.ucnt[u] = 0;
      first[e] = 0x80000000u | (uint32_t)u;   // from now on: the expert's unique index
    }
    U += __popc(mask);
    __syncwarp();
  }
  // token positions within each expert, in slot order (peers = same expert)
  for (int b = 0; b < S; b += 32) {
    const int s = b + lane;
    const bool v = s < S;
    const int e = v ? tb.sel_e[s] : -1 - lane;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int u = 0, pos = 0;
    if (v) {
      u = (int)(first[e] & 0x7FFFFFFFu);
      pos = tb.ucnt[u] + __popc(peers & lt);
    }
    __syncwarp();
    if (v) {
      tb.unit_tb[s] = (uint8_t)pos;        // position of slot s within its expert
      if ((peers & lt) == 0) tb.ucnt[u] = (uint16_t)(pos + __popc(peers));
    }
    __syncwarp();
  }
  // slot offsets hoff[u] = sum of ucnt over earlier unique experts
  int run = 0;
  for (int b = 0; b < U; b += 32) {
    const int u = b + lane;
    const int c = (u < U) ? tb.ucnt[u] : 0;
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (u < U) tb.hoff[u] = (uint16_t)(run + inc - c);
    run += __shfl_sync(0xffffffffu, inc, 31);
  }
  __syncwarp();
  for (int s = lane; s < S; s += 32) {
    const int u = (int)(first[tb.sel_e[s]] & 0x7FFFFFFFu);
    const int slot = tb.hoff[u] + tb.unit_tb[s];
    tb.utok[slot] = (uint8_t)(s / k);
    tb.uw[slot] = tb.sel_w[s];
  }
  __syncwarp();
  // units (u, token batch), u-major
  int nu = 0;
  for (int b = 0; b < U; b += 32) {
    const int u = b + lane;
    const int nb = (u < U) ? (tb.ucnt[u] + kTB - 1) / kTB : 0;
    int inc = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    if (u < U)
      for (int q = 0; q < nb; ++q) {
        tb.unit_u[nu + inc - nb + q] = (uint16_t)u;
        tb.unit_tb[nu + inc - nb + q] = (uint8_t)q;
      }
    nu += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) {
    tb.U = U;
    tb.n_units = nu;
  }
}

// Routing for all tokens + unique-expert tables (identical in every CTA).
__device__ __noinline__ void routing_phase(const Params& p, int write_out, Tables& tb, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int E = p.E, k = p.k, S = p.N * p.k, scoring = p.scoring, norm = p.norm;
  const float rsf = p.rsf;
  const float* bias = p.bias;
  for (int n = warp; n < p.N; n += kConsumerWarps) {
    const float* lrow = p.logits + (size_t)n * E;
    if (E <= 128) topk_token<4>(E, k, scoring, norm, rsf, bias, lrow, n, tb, lane);
    else if (E <= 256) topk_token<8>(E, k, scoring, norm, rsf, bias, lrow, n, tb, lane);
    else if (E <= 512) topk_token<16>(E, k, scoring, norm, rsf, bias, lrow, n, tb, lane);
    else topk_token<32>(E, k, scoring, norm, rsf, bias, lrow, n, tb, lane);
  }
  consumer_sync();
  if (warp == 0) {
    const bool done = (S <= 32) && build_tables_small(k, S, tb, lane);
    if (!done) build_tables(E, k, S, tb, lane);
  }
  if (write_out && warp == 1) {
    for (int s = lane; s < S; s += 32) {
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
  int row0;       // first row in the 2D tensor-map view [E*rows, ...]
};

template <int KIND>
__device__ __forceinline__ int kind_units(const Params& p, const Tables& tb) {
  if (KIND == KIND_AS || KIND == KIND_BS) return p.Is > 0 ? (p.N + kTB - 1) / kTB : 0;
  return tb.n_units;
}

template <int KIND>
__device__ __forceinline__ void kind_range(const Params& p, const Tables& tb, int cta, int G,
                                           int& lo, int& hi) {
  const uint32_t rpu = (uint32_t)(p.geo[KIND].rows_total / kRows);
  const uint32_t T = (uint32_t)kind_units<KIND>(p, tb) * rpu;   // < 2^22: products fit 32 bits
  lo = (int)(T * (uint32_t)cta / (uint32_t)G);
  hi = (int)(T * (uint32_t)(cta + 1) / (uint32_t)G);
}

template <int KIND>
__device__ __forceinline__ RG decode_rg(const Params& p, const Tables& tb, int g) {
  RG r;
  const int rows = p.geo[KIND].rows_total;
  const int rpu = rows / kRows;
  r.unit = g / rpu;
  r.rg = g % rpu;
  if (KIND == KIND_AS || KIND == KIND_BS) {
    r.u = 0;
    r.e = 0;
    r.tb = r.unit;
    r.nt = min(kTB, p.N - r.tb * kTB);
    r.row0 = r.rg * kRows;
  } else {
    r.u = tb.unit_u[r.unit];
    r.tb = tb.unit_tb[r.unit];
    r.e = tb.uexp[r.u];
    r.nt = min(kTB, (int)tb.ucnt[r.u] - r.tb * kTB);
    r.row0 = r.e * rows + r.rg * kRows;
  }
  return r;
}

// Token (row of x / out) of batch slot t of an RG.
template <int KIND>
__device__ __forceinline__ int rg_token(const Tables& tb, const RG& r, int t) {
  if (KIND == KIND_AS || KIND == KIND_BS) return r.tb * kTB + t;
  return tb.utok[tb.hoff[r.u] + r.tb * kTB + t];
}

// Bytes of row data (whole row of one projection) in chunk c.
__device__ __forceinline__ int chunk_row_bytes(const Geo& g, int c) {
  return min(kChunkBytes, g.kb - c * kChunkBytes);
}
__device__ __forceinline__ bool swizzled(const Geo& g) { return g.kb >= kBoxBytes; }

// ------------------------------------------------------------------ producer

template <int KIND>
__device__ __forceinline__ void produce_stage(const Params& p, const Tables& tb, const RG& r,
                                              int c, uint8_t* st, uint64_t* full) {
  const Geo& g = p.geo[KIND];
  const int rb = chunk_row_bytes(g, c);
  const bool sw = swizzled(g);
  const int nbox = sw ? (rb + kBoxBytes - 1) / kBoxBytes : 1;
  const int box_bytes = sw ? kBoxTileBytes : kRows * g.kb;
  const bool has_opnd = (KIND == KIND_AS || KIND == KIND_AR);
  const int elems = rb * 8 / (g.fmt == FMT_BF16 ? 16 : 4);   // K elements in this chunk
  uint32_t bytes = (uint32_t)(g.nproj * nbox * box_bytes);
  if (g.scale_mode == SCALES_TMAP) bytes += (uint32_t)(g.nproj * kRows * g.scb);
  if (g.scale_mode == SCALES_BLOCK) bytes += (uint32_t)(g.nproj * kRows * g.sr);
  if (has_opnd) bytes += (uint32_t)(r.nt * elems * 2);
  mbar_arrive_expect_tx(full, bytes);
  const int wmap0 = (KIND == KIND_AR) ? TM_GQ : (KIND == KIND_BR) ? TM_DQ
                  : (KIND == KIND_AS) ? TM_SG : TM_SD;
  for (int pj = 0; pj < g.nproj; ++pj) {
    const CUtensorMap* tm = &p.tm[wmap0 + pj];
    for (int b = 0; b < nbox; ++b)
      tma_load_2d(st + (sw ? (pj * kBoxesPerChunk + b) * kBoxTileBytes : pj * kRows * g.kb), tm,
                  c * kChunkBytes + b * kBoxBytes, r.row0, full);
  }
  if (g.scale_mode == SCALES_TMAP) {
    const int smap0 = (KIND == KIND_AR) ? TM_GS : TM_DS;
    for (int pj = 0; pj < g.nproj; ++pj)
      tma_load_2d(st + g.scale_off + pj * kRows * g.scb, &p.tm[smap0 + pj], c * g.scb, r.row0,
                  full);
  } else if (g.scale_mode == SCALES_BLOCK) {
    for (int pj = 0; pj < g.nproj; ++pj) {
      const uint8_t* base = (KIND == KIND_AR) ? (pj == 0 ? p.gsc : p.usc) : p.dsc;
      bulk_g2s(st + g.scale_off + pj * kRows * g.sr, base + (size_t)r.row0 * g.sr,
               (uint32_t)(kRows * g.sr), full);
    }
  }
  if (has_opnd) {
    const uint16_t* xs = (KIND == KIND_AR) ? p.x16 : p.x;
    for (int t = 0; t < r.nt; ++t) {
      const int n = rg_token<KIND>(tb, r, t);
      bulk_g2s(st + g.opnd_off + t * g.Kc * 2, xs + (size_t)n * p.H + (size_t)c * g.Kc,
               (uint32_t)(elems * 2), full);
    }
  }
}

struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  int nstages, stage_bytes;
};

// Streams every stage of one kind's row groups; returns false on abort.
template <int KIND>
__device__ __noinline__ bool produce_kind(const Params& p, Tables& tb, const Ring ring, int cta,
                                          int G, int* ctr_io) {
  int ctr = *ctr_io;
  if (kind_units<KIND>(p, tb) == 0) return true;
  int lo, hi;
  kind_range<KIND>(p, tb, cta, G, lo, hi);
  const int nch = p.geo[KIND].nchunks;
  for (int gi = lo; gi < hi; ++gi) {
    const RG r = decode_rg<KIND>(p, tb, gi);
    for (int c = 0; c < nch; ++c) {
      const int slot = ctr % ring.nstages;
      const uint32_t round = (uint32_t)(ctr / ring.nstages);
      if (aborted(tb)) return false;
      if (!mbar_wait_bounded(ring.empty + slot, (round & 1u) ^ 1u, p.timeout_ns)) {
        set_abort(p, tb, kErrTimeoutProducer);
        return false;
      }
      produce_stage<KIND>(p, tb, r, c, ring.base + (size_t)slot * ring.stage_bytes,
                          ring.full + slot);
      ++ctr;
      *ctr_io = ctr;
    }
  }
  return true;
}

// ------------------------------------------------------------------ consumer

struct ConsumerCtx {
  uint8_t* ring_base;
  uint64_t* full;
  uint64_t* empty;
  int nstages, stage_bytes;
  float* red;
  uint8_t* hbuf;
};

template <typename T>
__device__ __forceinline__ T lds(const uint8_t* p) {
  return *reinterpret_cast<const T*>(p);
}

// Stage geometry of one kind, held in registers by the consumer.
struct SG {
  int kb, Kc, K, nchunks, scale_mode, scale_off, scb, sr, opnd_off, scale_swz;
};
__device__ __forceinline__ SG load_sg(const Geo& g) {
  SG r;
  r.kb = g.kb; r.Kc = g.Kc; r.K = g.K; r.nchunks = g.nchunks; r.scale_mode = g.scale_mode;
  r.scale_off = g.scale_off; r.scb = g.scb; r.sr = g.sr; r.opnd_off = g.opnd_off;
  r.scale_swz = (g.scale_mode == SCALES_TMAP && g.scb == 64) ? 1 : 0;
  return r;
}

// Address of the 16-byte piece `piece` of weight row `lane` in a stage, for
// projection pj: 128-byte-swizzled boxes (rows of >= 128 bytes) or plain rows.
__device__ __forceinline__ const uint8_t* wptr(const uint8_t* st, int kb, int pj, int lane,
                                               int piece) {
  if (kb >= kBoxBytes)
    return st + (pj * kBoxesPerChunk + (piece >> 3)) * kBoxTileBytes + lane * kBoxBytes +
           (((piece & 7) ^ (lane & 7)) << 4);
  return st + pj * kRows * kb + lane * kb + piece * 16;
}

// Scale byte `b` of row `lane` in a tensor-map scale box (64-byte swizzle when
// the box rows are 64 bytes).
__device__ __forceinline__ const uint8_t* sptr(const uint8_t* st, const SG& g, int pj, int lane,
                                               int b) {
  const uint8_t* base = st + g.scale_off + pj * kRows * g.scb;
  if (g.scale_swz) return base + lane * 64 + ((((b >> 4) ^ ((lane >> 1) & 3)) << 4) | (b & 15));
  return base + lane * g.scb + b;
}

// Block scales of the (at most 4) steps [s0, s1) of this warp, per projection:
// NVFP4: f16x2 of the two 16-element block scales of a step; MXFP4: the
// 32-element block scale as f32 bits.
template <int FMT, int NPROJ>
__device__ __forceinline__ void load_scales(const uint8_t* st, const SG& g, int c, int s0, int s1,
                                            int lane, uint32_t (&sc)[NPROJ][4]) {
  const int nsw = s1 - s0;
#pragma unroll
  for (int pj = 0; pj < NPROJ; ++pj) {
    if (FMT == FMT_NVFP4) {
      if (g.scale_mode == SCALES_TMAP && nsw == 4 && (s0 & 3) == 0) {
        const uint2 v = lds<uint2>(sptr(st, g, pj, lane, 2 * s0));
        sc[pj][0] = e4m3x2_to_f16x2(v.x & 0xFFFFu);
        sc[pj][1] = e4m3x2_to_f16x2(v.x >> 16);
        sc[pj][2] = e4m3x2_to_f16x2(v.y & 0xFFFFu);
        sc[pj][3] = e4m3x2_to_f16x2(v.y >> 16);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i < nsw) {
            const int s = s0 + i;
            const uint8_t* a = (g.scale_mode == SCALES_TMAP)
                                   ? sptr(st, g, pj, lane, 2 * s)
                                   : st + g.scale_off + (pj * kRows + lane) * g.sr + (c * g.Kc + s * 32) / 16;
            sc[pj][i] = e4m3x2_to_f16x2(lds<uint16_t>(a));
          }
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i < nsw) {
          const int s = s0 + i;
          const uint8_t* a = (g.scale_mode == SCALES_TMAP)
                                 ? sptr(st, g, pj, lane, s)
                                 : st + g.scale_off + (pj * kRows + lane) * g.sr + (c * g.Kc + s * 32) / 32;
          sc[pj][i] = __float_as_uint(e8m0_to_f32(lds<uint8_t>(a)));
        }
      }
    }
  }
}

// One stage of FP4 weights for NT tokens: lane = weight row, steps [s0, s1)
// of this warp (a step is 32 elements = 16 bytes of a row, at most 4 steps).
template <int FMT, int NPROJ, int NT>
__device__ __forceinline__ void compute_fp4(const uint8_t* st, const SG& g, int c,
                                            const uint8_t* obase, int otstride, int s0, int s1,
                                            int lane, float (&acc)[NPROJ][NT]) {
  uint32_t sc[NPROJ][4];
  load_scales<FMT, NPROJ>(st, g, c, s0, s1, lane, sc);
  const int nsw = s1 - s0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i < nsw) {
      const int s = s0 + i;
      uint32_t wd[NPROJ][16];
#pragma unroll
      for (int pj = 0; pj < NPROJ; ++pj) {
        const uint4 w = lds<uint4>(wptr(st, g.kb, pj, lane, s));
        uint32_t o[4];
        e2m1x8_to_f16x2x4(w.x, o);
        wd[pj][0] = o[0]; wd[pj][1] = o[1]; wd[pj][2] = o[2]; wd[pj][3] = o[3];
        e2m1x8_to_f16x2x4(w.y, o);
        wd[pj][4] = o[0]; wd[pj][5] = o[1]; wd[pj][6] = o[2]; wd[pj][7] = o[3];
        e2m1x8_to_f16x2x4(w.z, o);
        wd[pj][8] = o[0]; wd[pj][9] = o[1]; wd[pj][10] = o[2]; wd[pj][11] = o[3];
        e2m1x8_to_f16x2x4(w.w, o);
        wd[pj][12] = o[0]; wd[pj][13] = o[1]; wd[pj][14] = o[2]; wd[pj][15] = o[3];
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const uint8_t* oa = obase + t * otstride + s * 64;
        uint32_t xo[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 x = lds<uint4>(oa + q * 16);
          xo[4 * q + 0] = x.x; xo[4 * q + 1] = x.y; xo[4 * q + 2] = x.z; xo[4 * q + 3] = x.w;
        }
#pragma unroll
        for (int pj = 0; pj < NPROJ; ++pj) {
          if (FMT == FMT_NVFP4) {
            uint32_t p0 = hmul2(wd[pj][0], xo[0]);
            uint32_t p1 = hmul2(wd[pj][8], xo[8]);
#pragma unroll
            for (int e = 1; e < 8; ++e) {
              p0 = hfma2(wd[pj][e], xo[e], p0);
              p1 = hfma2(wd[pj][8 + e], xo[8 + e], p1);
            }
            float a = acc[pj][t];
            a = fma_f16pair_scalar(p0, (uint16_t)(sc[pj][i] & 0xFFFFu), a);
            a = fma_f16pair_scalar(p1, (uint16_t)(sc[pj][i] >> 16), a);
            acc[pj][t] = a;
          } else {
            uint32_t p0 = hmul2(wd[pj][0], xo[0]);
            uint32_t p1 = hmul2(wd[pj][1], xo[1]);
#pragma unroll
            for (int e = 2; e < 16; e += 2) {
              p0 = hfma2(wd[pj][e], xo[e], p0);
              p1 = hfma2(wd[pj][e + 1], xo[e + 1], p1);
            }
            const float2 f0 = f16x2_to_f32x2(p0), f1 = f16x2_to_f32x2(p1);
            acc[pj][t] = fmaf((f0.x + f0.y) + (f1.x + f1.y), __uint_as_float(sc[pj][i]), acc[pj][t]);
          }
        }
      }
    }
  }
}

// One stage of BF16 weights (shared expert) for NT tokens; a step is 32
// elements = 64 bytes of a row.
template <int NPROJ, int NT>
__device__ __forceinline__ void compute_bf16(const uint8_t* st, const SG& g,
                                             const uint8_t* obase, int otstride, int s0, int s1,
                                             int lane, float (&acc)[NPROJ][NT]) {
#pragma unroll 1
  for (int s = s0; s < s1; ++s) {
    uint32_t wv[NPROJ][16];
#pragma unroll
    for (int pj = 0; pj < NPROJ; ++pj)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 w = lds<uint4>(wptr(st, g.kb, pj, lane, s * 4 + q));
        wv[pj][4 * q + 0] = w.x; wv[pj][4 * q + 1] = w.y;
        wv[pj][4 * q + 2] = w.z; wv[pj][4 * q + 3] = w.w;
      }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint8_t* oa = obase + t * otstride + s * 64;
      uint32_t xo[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 x = lds<uint4>(oa + q * 16);
        xo[4 * q + 0] = x.x; xo[4 * q + 1] = x.y; xo[4 * q + 2] = x.z; xo[4 * q + 3] = x.w;
      }
#pragma unroll
      for (int pj = 0; pj < NPROJ; ++pj) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          a0 = fma2_bf16_to_f32(wv[pj][e], xo[e], a0);
          a1 = fma2_bf16_to_f32(wv[pj][e + 1], xo[e + 1], a1);
        }
        acc[pj][t] += a0 + a1;
      }
    }
  }
}

// Activations of a down-projection unit into hbuf: routed h as f16 scaled
// per token by a power of two, shared h as BF16.
template <int KIND>
__device__ __noinline__ void stage_hbuf(const Params& p, Tables& tb, const RG& r, uint8_t* hbuf,
                                        int ctid) {
  const int K = p.geo[KIND].K;
  if (KIND == KIND_BR) {
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
    block_reduce<kTB, true>(m, tb, ctid);
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
          *reinterpret_cast<__half2*>(dst + kk) = __floats2half2_rn(v.x * sc, v.y * sc);
          *reinterpret_cast<__half2*>(dst + kk + 2) = __floats2half2_rn(v.z * sc, v.w * sc);
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

// Row-block completion for the down phase: every CTA, after its last down row
// group, publishes its red.adds (fence), bumps the counter of each 32-row
// output block it added to, and casts the blocks it completed to BF16.
__device__ __noinline__ void flush_row_blocks(const Params& p, Tables& tb, int ctid,
                                              uint32_t b_units) {
  __threadfence();
  consumer_sync();
  const int nb = tb.nbrg;
  const bool ab = aborted(tb);
  for (int i = ctid; i < nb; i += kConsumerThreads) {
    int fin = 0;
    if (!ab) {
      const uint32_t old = atomicAdd(p.rbcnt + tb.brg[i], 1u);
      fin = (old + 1u == b_units);
      if (fin) __threadfence();
    }
    tb.bfin[i] = (uint8_t)fin;
  }
  consumer_sync();
  for (int i = 0; i < nb; ++i) {
    if (!tb.bfin[i]) continue;
    const int rb = tb.brg[i];
    for (int j = ctid; j < p.N * kRows; j += kConsumerThreads) {
      const int n = j / kRows, row = rb * kRows + (j % kRows);
      const float v = ld_cg_f32(p.acc + (size_t)n * p.H + row);
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      p.out[(size_t)n * p.H + row] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
  consumer_sync();
  if (ctid == 0) tb.nbrg = 0;
  consumer_sync();
}

// Reduce the 8 warps' partial sums of an RG (already in `red`) and apply the
// epilogue of its kind.
// Per-thread epilogue factors of an RG (thread ctid < nt*32 serves token
// ctid/32), loaded when the RG starts so their latency hides behind the
// stage compute: gate/up scales for AR, output weight for BR/BS.
template <int KIND>
__device__ __forceinline__ float2 epi_factors(const Params& p, const Tables& tb, const RG& r,
                                              int ctid) {
  float2 f = make_float2(1.f, 1.f);
  if (ctid >= r.nt * 32) return f;
  const int t = ctid >> 5;
  const int n = rg_token<KIND>(tb, r, t);
  if (KIND == KIND_AR) {
    const float xs = ldexpf(1.0f, ld_cg_s32(p.xexp + n));
    f.x = xs * (p.g2 ? __ldg(p.g2 + r.e) : 1.0f);
    f.y = xs * (p.u2 ? __ldg(p.u2 + r.e) : 1.0f);
  } else if (KIND == KIND_BR) {
    f.x = ldexpf(1.0f, tb.hexp[t]) * (p.d2 ? __ldg(p.d2 + r.e) : 1.0f) *
          tb.uw[tb.hoff[r.u] + r.tb * kTB + t];
  } else if (KIND == KIND_BS) {
    f.x = ld_cg_f32(p.gsig + n);
  }
  return f;
}

template <int KIND>
__device__ __noinline__ void rg_epilogue(const Params& p, Tables& tb, const RG& r,
                                         const float* red, int ctid, uint32_t b_units, float2 ef) {
  const Geo& g = p.geo[KIND];
  if (ctid < r.nt * 32 && !aborted(tb)) {
    const int t = ctid >> 5, j = ctid & 31;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      s0 += red[((w * 2 + 0) * kTB + t) * 32 + j];
      if (g.nproj == 2) s1 += red[((w * 2 + 1) * kTB + t) * 32 + j];
    }
    const int row = r.rg * kRows + j;
    const int n = rg_token<KIND>(tb, r, t);
    if (KIND == KIND_AR) {
      p.h[(size_t)(tb.hoff[r.u] + r.tb * kTB + t) * p.inter + row] = silu(s0 * ef.x) * (s1 * ef.y);
    } else if (KIND == KIND_AS) {
      p.hs[(size_t)n * p.Is + row] = silu(s0) * s1;
    } else {
      red_add_f32(p.acc + (size_t)n * p.H + row, s0 * ef.x);
    }
  }
  consumer_sync();
  if (KIND == KIND_BR || KIND == KIND_BS) {
    if (ctid == 0) {
      tb.brg[tb.nbrg] = (uint16_t)r.rg;
      tb.nbrg = tb.nbrg + 1;
    }
    consumer_sync();
    if (tb.nbrg == kMaxRgList) flush_row_blocks(p, tb, ctid, b_units);
  }
}

// Streams the chunks of one RG for NT tokens and leaves the 8 warps' partial
// sums in `red` (layout [warp][proj][token][lane]).
template <int FMT, int NPROJ, int KIND, int NT>
__device__ __forceinline__ void consume_rg(const Params& p, Tables& tb, const ConsumerCtx& cx,
                                           const SG& g, int& ctr, int warp, int lane) {
  constexpr int kStepBytes = (FMT == FMT_BF16) ? 64 : 16;
  float acc[NPROJ][NT];
#pragma unroll
  for (int a = 0; a < NPROJ; ++a)
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[a][t] = 0.f;
  for (int c = 0; c < g.nchunks; ++c) {
    const int slot = ctr % cx.nstages;
    const uint32_t round = (uint32_t)(ctr / cx.nstages);
    ++ctr;
    bool ok = !aborted(tb);
    if (ok) ok = mbar_wait_bounded(cx.full + slot, round & 1u, p.timeout_ns);
    if (!ok) {
      if (lane == 0 && !aborted(tb)) set_abort(p, tb, kErrTimeoutStage);
    } else {
      const uint8_t* st = cx.ring_base + (size_t)slot * cx.stage_bytes;
      const int ns = min(kChunkBytes, g.kb - c * kChunkBytes) / kStepBytes;
      const int s0 = warp * ns / kConsumerWarps, s1 = (warp + 1) * ns / kConsumerWarps;
      const uint8_t* ob;
      int ots;
      if (KIND == KIND_AS || KIND == KIND_AR) {
        ob = st + g.opnd_off;
        ots = g.Kc * 2;
      } else {
        ob = cx.hbuf + c * g.Kc * 2;
        ots = g.K * 2;
      }
      if (FMT == FMT_BF16) compute_bf16<NPROJ, NT>(st, g, ob, ots, s0, s1, lane, acc);
      else compute_fp4<FMT, NPROJ, NT>(st, g, c, ob, ots, s0, s1, lane, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.empty + slot);
  }
#pragma unroll
  for (int pj = 0; pj < NPROJ; ++pj)
#pragma unroll
    for (int t = 0; t < NT; ++t) cx.red[((warp * 2 + pj) * kTB + t) * 32 + lane] = acc[pj][t];
}

// Consumes every stage of one kind's row groups.
template <int FMT, int NPROJ, int KIND>
__device__ __noinline__ void consume_kind(const Params& p, Tables& tb, const ConsumerCtx cx,
                                          int cta, int G, int* ctr_io, int ctid, uint32_t b_units) {
  if (kind_units<KIND>(p, tb) == 0) return;
  const int warp = ctid >> 5, lane = ctid & 31;
  int lo, hi;
  kind_range<KIND>(p, tb, cta, G, lo, hi);
  const SG g = load_sg(p.geo[KIND]);
  int ctr = *ctr_io;
  for (int gi = lo; gi < hi; ++gi) {
    const RG r = decode_rg<KIND>(p, tb, gi);
    if ((KIND == KIND_BR || KIND == KIND_BS) && (tb.hb_kind != KIND || tb.hb_unit != r.unit)) {
      if (!aborted(tb)) stage_hbuf<KIND>(p, tb, r, cx.hbuf, ctid);
      if (ctid == 0) {
        tb.hb_kind = KIND;
        tb.hb_unit = r.unit;
      }
      consumer_sync();
    }
    const float2 ef = epi_factors<KIND>(p, tb, r, ctid);
    switch (r.nt) {
      case 1: consume_rg<FMT, NPROJ, KIND, 1>(p, tb, cx, g, ctr, warp, lane); break;
      case 2: consume_rg<FMT, NPROJ, KIND, 2>(p, tb, cx, g, ctr, warp, lane); break;
      case 3: consume_rg<FMT, NPROJ, KIND, 3>(p, tb, cx, g, ctr, warp, lane); break;
      default: consume_rg<FMT, NPROJ, KIND, 4>(p, tb, cx, g, ctr, warp, lane); break;
    }
    consumer_sync();
    rg_epilogue<KIND>(p, tb, r, cx.red, ctid, b_units, ef);
  }
  *ctr_io = ctr;
}

// ------------------------------------------------------------------- kernel

template <int WF>
__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte-swizzled TMA boxes need a 1024-byte aligned destination
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
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
    tb.nbrg = 0;
  }
  __syncthreads();

  if (tid >= kConsumerThreads) {
    // -------------------------------------------------- producer (one thread)
    if (tid != kConsumerThreads || p.route_only) return;
    for (int i = 0; i < TM_COUNT; ++i)
      if (p.tm_valid & (1u << i)) prefetch_tensormap(&p.tm[i]);
    Ring ring{smem + p.smem_ring_off, full, empty, p.nstages, p.stage_bytes};
    int ctr = 0;
    bool ok = produce_kind<KIND_AS>(p, tb, ring, cta, G, &ctr);
    if (ok && !mbar_wait_bounded(rr, 0, p.timeout_ns)) {
      set_abort(p, tb, kErrTimeoutProducer);
      ok = false;
    }
    if (ok && aborted(tb)) ok = false;
    if (ok) {
      fence_proxy_async_global();   // x16 was written by other CTAs before B1
      ok = produce_kind<KIND_AR>(p, tb, ring, cta, G, &ctr) &&
           produce_kind<KIND_BR>(p, tb, ring, cta, G, &ctr) &&
           produce_kind<KIND_BS>(p, tb, ring, cta, G, &ctr);
    }
    if (!ok) {
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
  unsigned long long base = 0;
  if (ctid == 0) {
    const unsigned long long c0 = ld_relaxed_u64(&p.ctrl->arrivals);
    base = c0 - c0 % (2ull * (unsigned long long)G);
  }

  // P0: router, token prep, zero the accumulator
  router_phase(p, cta, G, tb, ctid);
  if (!p.route_only) {
    token_prep(p, cta, G, tb, ctid);
    const size_t nacc = (size_t)p.N * p.H;
    for (size_t i = (size_t)cta * kConsumerThreads + ctid; i < nacc;
         i += (size_t)G * kConsumerThreads)
      p.acc[i] = 0.f;
    for (int i = cta * kConsumerThreads + ctid; i < p.H / kRows; i += G * kConsumerThreads)
      p.rbcnt[i] = 0u;
  }
  consumer_sync();
  if (ctid == 0) {
    __threadfence();
    grid_arrive(p.ctrl);    // B1
  }

  int ctr = 0;
  if (!p.route_only) consume_kind<FMT_BF16, 2, KIND_AS>(p, tb, cx, cta, G, &ctr, ctid, 0);

  if (ctid == 0 && !grid_wait(p.ctrl, base + (unsigned long long)G, p.timeout_ns))
    set_abort(p, tb, kErrTimeoutBarrier);
  consumer_sync();
  if (aborted(tb)) {
    if (ctid == 0) {
      grid_arrive(p.ctrl);  // keep two arrivals per call
      mbar_arrive(rr);
    }
    return;   // the producer sees the abort and drains
  }

  // P1: routing
  routing_phase(p, cta == 0, tb, ctid);
  if (p.route_only) {
    if (ctid == 0) grid_arrive(p.ctrl);   // B2 arrival, nothing waits on it
    return;
  }
  if (ctid == 0) mbar_arrive(rr);

  const uint32_t b_units = (uint32_t)tb.n_units + ((p.Is > 0) ? (uint32_t)((p.N + kTB - 1) / kTB) : 0u);

  // P2: routed gate/up
  consume_kind<WF, 2, KIND_AR>(p, tb, cx, cta, G, &ctr, ctid, b_units);
  __threadfence();
  consumer_sync();
  if (ctid == 0) {
    grid_arrive(p.ctrl);    // B2
    if (!aborted(tb) && !grid_wait(p.ctrl, base + 2ull * (unsigned long long)G, p.timeout_ns))
      set_abort(p, tb, kErrTimeoutBarrier);
  }
  consumer_sync();

  // P3: down projections (routed, then shared) + row-block completion
  consume_kind<WF, 1, KIND_BR>(p, tb, cx, cta, G, &ctr, ctid, b_units);
  consume_kind<FMT_BF16, 1, KIND_BS>(p, tb, cx, cta, G, &ctr, ctid, b_units);
  flush_row_blocks(p, tb, ctid, b_units);
}

// ------------------------------------------------------------------- host

static bool plan_kind(Geo& g, int fmt, int nproj, int K, int rows, bool with_operand) {
  g.fmt = fmt;
  g.nproj = nproj;
  g.K = K;
  g.rows_total = rows;
  g.opnd_off = -1;
  if (K % 32 != 0 || rows % kRows != 0 || K <= 0 || rows <= 0) return false;
  g.kb = (fmt == FMT_BF16) ? K * 2 : K / 2;
  g.Kc = (fmt == FMT_BF16) ? kChunkBytes / 2 : kChunkBytes * 2;
  g.nchunks = (g.kb + kChunkBytes - 1) / kChunkBytes;
  int off = (g.kb >= kBoxBytes) ? nproj * kBoxesPerChunk * kBoxTileBytes : nproj * kRows * g.kb;
  off = (off + 1023) / 1024 * 1024;
  g.scale_off = off;
  g.sr = g.scb = 0;
  g.scale_mode = SCALES_NONE;
  if (fmt != FMT_BF16) {
    const int gs = (fmt == FMT_NVFP4) ? 16 : 32;
    g.sr = K / gs;
    if (g.sr % 16 == 0) {
      g.scale_mode = SCALES_TMAP;
      g.scb = std::min(g.Kc / gs, g.sr);
      off += nproj * kRows * g.scb;
    } else {
      g.scale_mode = SCALES_BLOCK;
      off += nproj * kRows * g.sr;
    }
    off = (off + 127) / 128 * 128;
  }
  if (with_operand) {
    g.opnd_off = off;
    off += kTB * g.Kc * 2;
  }
  g.stage_bytes = (off + 1023) / 1024 * 1024;
  return true;
}

// Tables plus the reduction scratch; the ring needs 1024-byte alignment.
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
  return v - 2048;   // 1024 B alignment headroom of the ring + reserved
}

int decode_grid(int device, int smem_bytes) {
  smem_bytes += 1024;   // alignment headroom of the ring (see the kernel prologue)
  int sms = 0, nb0 = 0, nb1 = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  if (cudaFuncSetAttribute(moe_decode_kernel<FMT_NVFP4>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess ||
      cudaFuncSetAttribute(moe_decode_kernel<FMT_MXFP4>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb0, moe_decode_kernel<FMT_NVFP4>, kThreads,
                                                    smem_bytes) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb1, moe_decode_kernel<FMT_MXFP4>, kThreads,
                                                    smem_bytes) != cudaSuccess)
    return 0;
  if (nb0 < 1 || nb1 < 1) return 0;
  return sms;   // one CTA per SM
}

cudaError_t launch_decode(const Params& p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem_total + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.fmt == 0) return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_NVFP4>, p);
  return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_MXFP4>, p);
}

}  // namespace moe
