// Fused MoE decode-layer forward for small N on sm_103a (one launch per call).
//
// Computes, for N token rows, the chain of forward_k3.rs (doc comment of
// MoeLayer::forward_k3: gate GEMV -> batched top-k -> expert gate+up ->
// SiLU+down -> weighted sum + shared blend) with the routed experts summed as
// routing-weighted FP32 partials and cast to BF16 once at the end
// (forward_atomic_c4.rs, doc comment of forward_atomic_c4_decode).
//
// Execution model: a persistent grid, one CTA per SM, every CTA resident at
// once (cooperative launch).  Each CTA has 8 compute ("consumer") warps, one
// epilogue warp, and 4 producer threads (lane 0 of 4 warps, stage k issued by
// producer k mod 4: a TMA instruction from DRAM holds its thread for a few
// hundred cycles) that stream weights into a ring of shared-memory stages
// with TMA (3D tensor-map copies of whole 512-byte chunks, or 2D boxes of 16
// or 32 rows x 128 bytes; 128-byte swizzle), completion tracked by mbarriers.
//
// Instruction fetch is a first-order cost here (the code a launch runs does
// not stay in the SM's instruction cache), so the kernel is built twice per
// weight format (the routing variants apart) and count-dependent steps
// dispatch to one template instance per token count.
//
// Phases of one call (per CTA):
//   P0  router GEMV for rows e = cta, cta+G, ... (128-bit loads; BF16 or NVFP4
//       router, E + Z rows with zero experts); token prep
//       (f16 copy of x scaled by a power of two, shared-expert gate) on the
//       last CTAs; zero the per-unit readiness counters.
//   --  grid barrier B1 (arrive).  Shared-expert gate/up row groups need only
//       x, so they are streamed and computed before waiting on B1.
//   P1  every CTA computes the same top-k (or hash routing) for all N tokens
//       and the same table
//       of unique experts, per-expert token lists and (expert, token batch)
//       units (zero-expert slots run nothing): each routed expert's weights
//       are then read once for all its tokens (forward_batched.rs: one pass
//       over an expert's weights serves every row routed to it).
//   P2  routed gate/up row groups of 16 rows (gate rows and up rows stacked
//       as one 32-row tile, lane j < 16 gate, lane j >= 16 up); the epilogue
//       warp forms h = SiLU(g)*u, stored as f16 with one power-of-two
//       exponent per 16 rows, and publishes the CTA's row groups to the
//       units' readiness counters.
//   P3  down: each CTA owns whole 16-row blocks of the output.  Every unit
//       (and shared-expert token batch) is one job for S = 8 / jobs-per-block
//       warps (half-warps split K); the producer prefetches the down weights during P2 and adds
//       a job's activations to its stage once the unit's counter says its h
//       is complete.  Jobs add their routing-weighted rows into shared
//       memory; the block is cast to BF16 and written once: no second grid
//       barrier, no global atomics, no accumulator in global memory.
//
// Inside a row group, lane j owns weight row j and the 8 warps split the K
// range; partial sums meet in shared memory at the end of the group.  The
// 128-byte swizzle makes the lane-per-row 128-bit shared loads conflict free;
// activations are read as broadcasts.
//
// FP4 arithmetic: E2M1 codes become f16x2 with cvt.rn.f16x2.e2m1x2; each
// 16-element block is summed with f16x2 FMAs against x or h held as f16
// scaled by a power of two that keeps every partial below 2^14; each block
// partial is then multiplied by its E4M3/E8M0 scale (times the h exponent in
// the down projection) and accumulated in FP32.  The shared expert (BF16)
// uses fma.rn.f32.bf16 (BF16 products, FP32 accumulation).  FP8 experts:
// E4M3 -> f16 (exact), products with f16 x or h formed and summed in FP32,
// each 32-element step times its 128 x 128 block scale.  BF16 experts: BF16
// products with the BF16 x (gate/up) or the f16 h (down) in FP32.
//
// Every wait (grid barrier, stage, readiness) is bounded by a time budget; on
// expiry the kernel records an error bit in the workspace and drains.

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
  uint32_t cnt[kMaxE];         // per expert: first slot, then unique index
  int16_t uexp[kMaxSlots];     // unique experts
  uint16_t ucnt[kMaxSlots];    // tokens routed to unique expert u
  uint16_t hoff[kMaxSlots];    // first slot of u in the (expert, token) order
  uint8_t utok[kMaxSlots];     // token of (expert, position) slot
  float uw[kMaxSlots];         // routing weight of that slot
  uint16_t unit_u[kMaxSlots];  // units = (unique expert, token batch)
  uint8_t unit_tb[kMaxSlots];
  int16_t xe[kMaxSlots];       // power-of-two exponent of each token's f16 x
  float s2[2][kMaxSlots];      // gate / up scale2 of unique expert u
  int U, n_units;
  int abort;                   // set when a bounded wait expired
  float rscratch[kConsumerWarps * 8];
  uint32_t uscratch[kConsumerWarps * 2];
};

// ----------------------------------------------------------------- helpers

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
// SiLU with the fast exponential and divide (h is rounded to f16 afterwards).
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }
// 2^e for e in [-252, 254] (two normal factors; 0 or inf outside the float range).
__device__ __forceinline__ float exp2i(int e) {
  const int e1 = e >> 1;
  return __int_as_float((e1 + 127) << 23) * __int_as_float((e - e1 + 127) << 23);
}
// floor(log2(m)) of a positive finite float, subnormals included.
__device__ __forceinline__ int ilog2_pos(float m) {
  const uint32_t b = __float_as_uint(m);
  const int ex = (int)((b >> 23) & 0xFFu);
  return ex ? ex - 127 : -118 - __clz(b & 0x7FFFFFu);
}
__device__ __forceinline__ void consumer_sync() { named_bar_sync(1, kConsumerThreads); }
__device__ __forceinline__ bool aborted(const Tables& tb) {
  return *(volatile const int*)&tb.abort != 0;
}
__device__ __noinline__ void set_abort(const Params& p, Tables& tb, uint32_t bit) {
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
  return ilog2_pos(amax) - 6;
}

// ------------------------------------------------------------ grid barrier
// The workspace keeps one monotonic 64-bit arrival counter.  Every CTA
// arrives exactly once per call, so at kernel start the counter is a multiple
// of G (no CTA can pass B1 before all have arrived).  Arrivals are
// fire-and-forget release reductions; a waiter polls with acquire loads until
// the counter reaches base + G.
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
// Logits of expert e for tokens n0 .. n0 + nn - 1 (nn <= NT): one thread per
// 8 elements of H, then a block reduction.  Only the NT-token variant that
// runs is fetched, so small token counts execute little code.
template <bool EXT, int NT>
__device__ __forceinline__ void router_group(const Params& p, Tables& tb, int ctid, int R, int e,
                                             int n0, int nn, float rs2) {
  const int H = p.H;
  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
  for (int kk = ctid * 8; kk < H; kk += kConsumerThreads * 8) {
    float wf[8];
    router_w8(p.router, EXT ? p.router_fmt : 0, p.router_s, rs2, H, e, kk, wf);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (t < nn) {
        const uint4 xv = ld_nc_u4(p.x + (size_t)(n0 + t) * H + kk);
        const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[t] = fmaf(wf[2 * i], bf16_lo(xa[i]), acc[t]);
          acc[t] = fmaf(wf[2 * i + 1], bf16_hi(xa[i]), acc[t]);
        }
      }
    }
  }
  block_reduce<NT, false>(acc, tb, ctid);
  if (ctid < nn) {
    float v = acc[0];
#pragma unroll
    for (int t = 1; t < NT; ++t)
      if (ctid == t) v = acc[t];
    p.logits[(size_t)(n0 + ctid) * R + e] = v;
  }
}

// EXT = false: a BF16 router of width E only (the common layers).
template <bool EXT>
__device__ __noinline__ void router_phase(const Params& p, int cta, int G, Tables& tb, int ctid) {
  const float rs2 = (EXT && p.router_fmt == 1 && p.router_s2) ? __ldg(p.router_s2) : 1.0f;
  const int R = EXT ? p.E + p.Z : p.E;   // router width (zero experts included)
  for (int e = cta; e < R; e += G) {
    for (int n0 = 0; n0 < p.N; n0 += 8) {
      const int nn = min(8, p.N - n0);
      if (nn == 1) router_group<EXT, 1>(p, tb, ctid, R, e, n0, nn, rs2);
      else if (nn == 2) router_group<EXT, 2>(p, tb, ctid, R, e, n0, nn, rs2);
      else if (nn <= 4) router_group<EXT, 4>(p, tb, ctid, R, e, n0, nn, rs2);
      else router_group<EXT, 8>(p, tb, ctid, R, e, n0, nn, rs2);
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
    const float sc = exp2i(-ex);
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
template <int PER, bool EXT>
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
  topk_warp<PER, EXT>(E, k, scoring, norm, rsf, bias, lg, lane, &se, &sw);
  if (lane < k) {
    tb.sel_e[n * k + lane] = (int16_t)se;
    tb.sel_w[n * k + lane] = sw;
  }
}

// Hash routing of token n (experts from its tid2eid row), out of line so the
// top-k path's code stays compact.
template <int PER>
__device__ __noinline__ void hash_token(int E, int k, int scoring, int norm, float rsf,
                                        const float* lrow, int n, const int32_t* hash_row,
                                        Tables& tb, int lane) {
  float lg[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    lg[i] = (e < E) ? ld_cg_f32(lrow + e) : -INFINITY;
  }
  int se = 0;
  float sw = 0.f;
  hash_warp<PER>(E, k, scoring, norm, rsf, hash_row, lg, lane, &se, &sw);
  if (lane < k) {
    tb.sel_e[n * k + lane] = (int16_t)se;
    tb.sel_w[n * k + lane] = sw;
  }
}

// Small case (S = N*k <= 32, every expert has <= kTB tokens): the same tables
// as build_tables, from one slot per lane in registers.
__device__ __forceinline__ bool build_tables_small(int E, int k, int S, Tables& tb, int lane) {
  // slots that selected a zero expert (index >= E) run no expert
  const bool v = lane < S && tb.sel_e[lane] < E;
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
  for (int s = lane; s < S; s += 32)
    if (tb.sel_e[s] < E) atomicMin(&first[tb.sel_e[s]], (uint32_t)s);   // zero experts: none
  __syncwarp();
  const uint32_t lt = (1u << lane) - 1u;
  int U = 0;
  for (int b = 0; b < S; b += 32) {          // unique experts in first-slot order
    const int s = b + lane;
    const int e = (s < S) ? tb.sel_e[s] : 0;
    const bool isfirst = (s < S) && e < E && first[e] == (uint32_t)s;
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
    const bool v = s < S && tb.sel_e[s] < E;
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
    if (tb.sel_e[s] >= E) continue;
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
// EXT = false: top-k routing with the softmax / sigmoid + bias scorings over E
// router outputs only (no zero experts, no hash routing).
template <bool EXT>
__device__ __noinline__ void routing_phase(const Params& p, int write_out, Tables& tb, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31;
  const int E = p.E, k = p.k, S = p.N * p.k, scoring = p.scoring, norm = p.norm;
  const int R = EXT ? E + p.Z : E;   // top-k runs over the whole router width
  const float rsf = p.rsf;
  const float* bias = p.bias;
  for (int n = warp; n < p.N; n += kConsumerWarps) {
    const float* lrow = p.logits + (size_t)n * R;
    if (EXT && p.hash_V > 0) {
      // hash routing: the token id's row of tid2eid (ids clamped into the table)
      const int32_t* hrow =
          p.tid2eid + (size_t)min(max(__ldg(p.token_ids + n), 0), p.hash_V - 1) * k;
      if (R <= 128) hash_token<4>(R, k, scoring, norm, rsf, lrow, n, hrow, tb, lane);
      else if (R <= 256) hash_token<8>(R, k, scoring, norm, rsf, lrow, n, hrow, tb, lane);
      else if (R <= 512) hash_token<16>(R, k, scoring, norm, rsf, lrow, n, hrow, tb, lane);
      else hash_token<32>(R, k, scoring, norm, rsf, lrow, n, hrow, tb, lane);
      continue;
    }
    if (R <= 128) topk_token<4, EXT>(R, k, scoring, norm, rsf, bias, lrow, n, tb, lane);
    else if (R <= 256) topk_token<8, EXT>(R, k, scoring, norm, rsf, bias, lrow, n, tb, lane);
    else if (R <= 512) topk_token<16, EXT>(R, k, scoring, norm, rsf, bias, lrow, n, tb, lane);
    else topk_token<32, EXT>(R, k, scoring, norm, rsf, bias, lrow, n, tb, lane);
  }
  if (!p.route_only && warp == kConsumerWarps - 1)
    for (int n = lane; n < p.N; n += 32) tb.xe[n] = (int16_t)ld_cg_s32(p.xexp + n);
  consumer_sync();
  if (warp == 0) {
    const bool done = (S <= 32) && build_tables_small(E, k, S, tb, lane);
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

// Per-unique-expert gate/up scale2 factors into shared memory (the epilogue
// warp, off the compute warps' path; read only by its own epilogues).
__device__ __forceinline__ void load_scale2(const Params& p, Tables& tb, int lane) {
  for (int u = lane; u < tb.U; u += 32) {
    const int e = tb.uexp[u];
    tb.s2[0][u] = p.g2 ? __ldg(p.g2 + e) : 1.0f;
    tb.s2[1][u] = p.u2 ? __ldg(p.u2 + e) : 1.0f;
  }
  __syncwarp();
}

// ------------------------------------------------------- row-group plumbing
// Gate/up row groups (AS: 32 shared-expert rows; AR: 16 routed rows of gate
// and of up).

struct RG {
  int unit, rg;   // unit index within the kind, row group within the unit
  int e, u, tb;   // expert id (routed), unique index, token batch
  int nt;         // tokens in this batch (1..kTB)
  int row0;       // first row in the 2D tensor-map view [E*rows, ...]
};

template <int KIND>
__device__ __forceinline__ int kind_units(const Params& p, const Tables& tb) {
  if (KIND == KIND_AS) return p.Is > 0 ? (p.N + kTB - 1) / kTB : 0;
  return tb.n_units;
}

template <int KIND>
__device__ __forceinline__ void kind_range(const Params& p, const Tables& tb, int cta, int G,
                                           int& lo, int& hi) {
  const uint32_t rpu = (uint32_t)(p.geo[KIND].rows_total / p.geo[KIND].rg_rows);
  const uint32_t T = (uint32_t)kind_units<KIND>(p, tb) * rpu;   // < 2^22: products fit 32 bits
  lo = (int)(T * (uint32_t)cta / (uint32_t)G);
  hi = (int)(T * (uint32_t)(cta + 1) / (uint32_t)G);
}

template <int KIND>
__device__ __forceinline__ RG decode_rg(const Params& p, const Tables& tb, int g) {
  RG r;
  const int rows = p.geo[KIND].rows_total;
  const int rr = p.geo[KIND].rg_rows;
  const int rpu = rows / rr;
  r.unit = g / rpu;
  r.rg = g % rpu;
  if (KIND == KIND_AS) {
    r.u = 0;
    r.e = 0;
    r.tb = r.unit;
    r.nt = min(kTB, p.N - r.tb * kTB);
    r.row0 = r.rg * rr;
  } else {
    r.u = tb.unit_u[r.unit];
    r.tb = tb.unit_tb[r.unit];
    r.e = tb.uexp[r.u];
    r.nt = min(kTB, (int)tb.ucnt[r.u] - r.tb * kTB);
    r.row0 = r.e * rows + r.rg * rr;
  }
  return r;
}

// Token (row of x / out) of batch slot t of a gate/up row group.
template <int KIND>
__device__ __forceinline__ int rg_token(const Tables& tb, const RG& r, int t) {
  if (KIND == KIND_AS) return r.tb * kTB + t;
  return tb.utok[tb.hoff[r.u] + r.tb * kTB + t];
}

// Bytes of row data (whole row of one projection) in chunk c.
__device__ __forceinline__ int chunk_row_bytes(const Geo& g, int c) {
  return min(kChunkBytes, g.kb - c * kChunkBytes);
}
__device__ __forceinline__ bool swizzled(const Geo& g) { return g.kb >= kBoxBytes; }

// Down jobs of a CTA: for each owned 16-row output block i (rows
// (cta + i*G)*16 ..), the routed units 0..nr-1, then the shared-expert token
// batches; each job is nchunks stages.
struct DnIt {
  int i, jb, c;
};
__device__ __forceinline__ void dn_next(DnIt& it, int J, int nr, int nch_r, int nch_s) {
  ++it.c;
  if (it.c == (it.jb < nr ? nch_r : nch_s)) {
    it.c = 0;
    if (++it.jb == J) {
      it.jb = 0;
      ++it.i;
    }
  }
}
__device__ __forceinline__ int dn_blocks(const Params& p, int cta, int G) {
  return cta < p.nrb ? (p.nrb - cta + G - 1) / G : 0;
}

// ------------------------------------------------------------------ producer

// Weight boxes (and block scales) of chunk c of one stage; `opnd_bytes` of
// activations will complete the stage's transaction count (issued now or
// later by produce_operand).
template <int KIND>
__device__ __forceinline__ void produce_weights(const Params& p, int row0, int c, uint8_t* st,
                                                uint64_t* full, uint32_t opnd_bytes) {
  const Geo& g = p.geo[KIND];
  const int rb = chunk_row_bytes(g, c);
  const bool sw = swizzled(g);
  const int nbox = sw ? (rb + kBoxBytes - 1) / kBoxBytes : 1;
  const int box_bytes = sw ? g.brows * kBoxBytes : g.brows * g.kb;
  // projection stride inside the stage: one tile of 4 columns x brows rows
  const int pstride = sw ? kBoxesPerChunk * g.brows * kBoxBytes : g.brows * g.kb;
  uint32_t bytes = (uint32_t)(g.nproj * (g.use3d ? kBoxesPerChunk : nbox) * box_bytes) + opnd_bytes;
  if (g.scale_mode == SCALES_TMAP) bytes += (uint32_t)(g.nproj * g.brows * g.scb);
  if (g.scale_mode == SCALES_BLOCK) bytes += (uint32_t)(g.nproj * g.brows * g.sr);
  mbar_arrive_expect_tx(full, bytes);
  const int wmap0 = (KIND == KIND_AR) ? TM_GQ : (KIND == KIND_BR) ? TM_DQ
                  : (KIND == KIND_AS) ? TM_SG : TM_SD;
  const int wmap3 = (KIND == KIND_AR) ? TM3_GQ : (KIND == KIND_BR) ? TM3_DQ
                  : (KIND == KIND_AS) ? TM3_SG : TM3_SD;
  for (int pj = 0; pj < g.nproj; ++pj) {
    if (g.use3d) {
      // columns 4c .. 4c+3 (beyond the row: zero fill, counted in the box bytes)
      tma_load_3d(st + pj * pstride, &p.tm[wmap3 + pj], 0, row0, c * kBoxesPerChunk, full);
    } else {
      const CUtensorMap* tm = &p.tm[wmap0 + pj];
      for (int b = 0; b < nbox; ++b)
        tma_load_2d(st + pj * pstride + b * g.tile_bytes, tm, c * kChunkBytes + b * kBoxBytes,
                    row0, full);
    }
  }
  if (g.scale_mode == SCALES_TMAP) {
    const int smap0 = (KIND == KIND_AR) ? TM_GS : TM_DS;
    for (int pj = 0; pj < g.nproj; ++pj)
      tma_load_2d(st + g.scale_off + pj * g.brows * g.scb, &p.tm[smap0 + pj], c * g.scb, row0,
                  full);
  } else if (g.scale_mode == SCALES_BLOCK) {
    for (int pj = 0; pj < g.nproj; ++pj) {
      const uint8_t* base = (KIND == KIND_AR) ? (pj == 0 ? p.gsc : p.usc) : p.dsc;
      bulk_g2s(st + g.scale_off + pj * g.brows * g.sr, base + (size_t)row0 * g.sr,
               (uint32_t)(g.brows * g.sr), full);
    }
  }
}

// K elements of chunk c.
__device__ __forceinline__ int chunk_elems(const Geo& g, int c) {
  const int rb = chunk_row_bytes(g, c);
  return g.fmt == FMT_BF16 ? rb / 2 : g.fmt == FMT_FP8 ? rb : rb * 2;
}

template <int KIND>
__device__ __forceinline__ uint32_t gateup_opnd_bytes(const Geo& g, int c, int nt) {
  return (uint32_t)(nt * chunk_elems(g, c) * 2);
}

// One stage of a gate/up row group: weights, scales and the x chunk.
template <int KIND>
__device__ __forceinline__ void produce_stage(const Params& p, const Tables& tb, const RG& r,
                                              int c, uint8_t* st, uint64_t* full) {
  const Geo& g = p.geo[KIND];
  const int elems = chunk_elems(g, c);
  produce_weights<KIND>(p, r.row0, c, st, full, gateup_opnd_bytes<KIND>(g, c, r.nt));
  // FP4 experts take the scaled f16 copy of x; BF16 weights (shared expert,
  // BF16 routed experts) take the BF16 x itself
  const uint16_t* xs = (KIND == KIND_AR && g.fmt != FMT_BF16) ? p.x16 : p.x;
  for (int t = 0; t < r.nt; ++t) {
    const int n = rg_token<KIND>(tb, r, t);
    bulk_g2s(st + g.opnd_off + t * g.Kc * 2, xs + (size_t)n * p.H + (size_t)c * g.Kc,
             (uint32_t)(elems * 2), full);
  }
}

struct Ring {
  uint8_t* base;
  uint64_t* full;
  uint64_t* empty;
  int nstages, stage_bytes;
};

// Streams the stages k = pid (mod kProducers) of one gate/up kind's row
// groups; returns false on abort.  `*ctr_io` counts all stages.
template <int KIND>
__device__ __noinline__ bool produce_kind(const Params& p, Tables& tb, const Ring ring, int cta,
                                          int G, int* ctr_io, int pid) {
  int ctr = *ctr_io;
  if (kind_units<KIND>(p, tb) == 0) return true;
  int lo, hi;
  kind_range<KIND>(p, tb, cta, G, lo, hi);
  const int nch = p.geo[KIND].nchunks;
  for (int gi = lo; gi < hi; ++gi) {
    const RG r = decode_rg<KIND>(p, tb, gi);
    for (int c = 0; c < nch; ++c) {
      if (ctr % kProducers != pid) {
        *ctr_io = ++ctr;
        continue;
      }
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

// Job parameters of a down stage.
struct DnJob {
  bool routed;
  int row0;    // tensor-map row of the block
  int nt;      // tokens
  int src0;    // first activation row: h16 slot (routed) or token (shared)
  int unit;    // routed unit (readiness counter, hexp row)
};
__device__ __forceinline__ DnJob dn_job(const Params& p, const Tables& tb, int cta, int G,
                                        const DnIt& it, int nr) {
  DnJob j;
  const int rb = cta + it.i * G;
  j.routed = it.jb < nr;
  if (j.routed) {
    const int u = tb.unit_u[it.jb], tbi = tb.unit_tb[it.jb];
    j.unit = it.jb;
    j.nt = min(kTB, (int)tb.ucnt[u] - tbi * kTB);
    j.src0 = tb.hoff[u] + tbi * kTB;
    j.row0 = tb.uexp[u] * p.H + rb * kDnRows;
  } else {
    const int b = it.jb - nr;
    j.unit = -1;
    j.nt = min(kTB, p.N - b * kTB);
    j.src0 = b * kTB;
    j.row0 = rb * kDnRows;
  }
  return j;
}
__device__ __forceinline__ uint32_t dn_opnd_bytes(const Params& p, const DnJob& j, int c) {
  const Geo& g = p.geo[j.routed ? KIND_BR : KIND_BS];
  const int elems = chunk_elems(g, c);
  uint32_t b = (uint32_t)(j.nt * elems * 2);
  if (j.routed) b += (uint32_t)(((elems / 16) + 15) & ~15);
  return b;
}
__device__ __forceinline__ void dn_operand(const Params& p, const DnJob& j, int c, uint8_t* st,
                                           uint64_t* full) {
  const Geo& g = p.geo[j.routed ? KIND_BR : KIND_BS];
  const int elems = chunk_elems(g, c);
  if (j.routed) {
    for (int t = 0; t < j.nt; ++t)
      bulk_g2s(st + g.opnd_off + t * g.Kc * 2,
               p.h16 + (size_t)(j.src0 + t) * p.inter + (size_t)c * g.Kc, (uint32_t)(elems * 2),
               full);
    bulk_g2s(st + g.hx_off, p.hexp + (size_t)j.unit * p.hstride + c * (g.Kc / 16),
             (uint32_t)(((elems / 16) + 15) & ~15), full);
  } else {
    for (int t = 0; t < j.nt; ++t)
      bulk_g2s(st + g.opnd_off + t * g.Kc * 2,
               p.hs + (size_t)(j.src0 + t) * p.Is + (size_t)c * g.Kc, (uint32_t)(elems * 2), full);
  }
}

// Down stages: weights are issued as soon as ring slots free up (prefetch
// during the gate/up phase); a stage's activations follow once its unit's
// gate/up row groups are all done everywhere (readiness counters, acquire).
__device__ __noinline__ bool produce_down(const Params& p, Tables& tb, const Ring ring, int cta,
                                          int G, int* ctr_io, int pid) {
  const int nrbl = dn_blocks(p, cta, G);
  const int nr = tb.n_units, nsh = p.Is > 0 ? (p.N + kTB - 1) / kTB : 0, J = nr + nsh;
  if (nrbl == 0 || J == 0) return true;
  const int nch_r = p.geo[KIND_BR].nchunks, nch_s = nsh ? p.geo[KIND_BS].nchunks : 1;
  const int total = nrbl * (nr * nch_r + nsh * nch_s);
  const uint32_t need_r = (uint32_t)(p.inter / kDnRows);
  const uint32_t need_s = nsh ? (uint32_t)(nsh * (p.Is / kRows)) : 0u;
  const int ctr0 = *ctr_io;
  DnIt W{0, 0, 0}, O{0, 0, 0};
  int kw = 0, ko = 0;
  uint64_t idle0 = 0;
  bool ok = true;
  // units already seen complete (units beyond 64 are re-checked each time)
  unsigned long long seen = 0ull;
  bool as_seen = false;
  auto unit_ready = [&](const DnJob& j) -> bool {
    if (!j.routed) {
      if (!as_seen) as_seen = ld_acquire_u32(p.ready + kReadyAS) >= need_s;
      return as_seen;
    }
    if (j.unit < 64 && (seen >> j.unit & 1ull)) return true;
    const bool r = ld_acquire_u32(p.ready + j.unit) >= need_r;
    if (r && j.unit < 64) seen |= 1ull << j.unit;
    return r;
  };
  // skip the stages of the other producers (both cursors)
  auto skip_w = [&]() {
    while (kw < total && (ctr0 + kw) % kProducers != pid) {
      dn_next(W, J, nr, nch_r, nch_s);
      ++kw;
    }
  };
  auto skip_o = [&]() {
    while (ko < kw && (ctr0 + ko) % kProducers != pid) {
      dn_next(O, J, nr, nch_r, nch_s);
      ++ko;
    }
  };
  skip_w();
  while (ko < total) {
    if (aborted(tb)) { ok = false; break; }
    skip_o();
    if (ko >= total) break;
    bool did = false;
    if (ko < kw) {
      const DnJob j = dn_job(p, tb, cta, G, O, nr);
      if (unit_ready(j)) {
        fence_proxy_async_global();   // h16 / hs were written by other CTAs
        const int k = ctr0 + ko;
        dn_operand(p, j, O.c, ring.base + (size_t)(k % ring.nstages) * ring.stage_bytes,
                   ring.full + k % ring.nstages);
        dn_next(O, J, nr, nch_r, nch_s);
        ++ko;
        skip_o();
        did = true;
      }
    }
    if (!did && kw < total) {
      const int k = ctr0 + kw;
      const int slot = k % ring.nstages;
      if (mbar_test_wait(ring.empty + slot, ((uint32_t)(k / ring.nstages) & 1u) ^ 1u)) {
        const DnJob j = dn_job(p, tb, cta, G, W, nr);
        uint8_t* st = ring.base + (size_t)slot * ring.stage_bytes;
        if (j.routed) produce_weights<KIND_BR>(p, j.row0, W.c, st, ring.full + slot, dn_opnd_bytes(p, j, W.c));
        else produce_weights<KIND_BS>(p, j.row0, W.c, st, ring.full + slot, dn_opnd_bytes(p, j, W.c));
        dn_next(W, J, nr, nch_r, nch_s);
        ++kw;
        skip_w();
        did = true;
      }
    }
    if (did) {
      idle0 = 0;
    } else {
      const uint64_t now = global_timer_ns();
      if (idle0 == 0) idle0 = now;
      else if (now - idle0 > p.timeout_ns) {
        set_abort(p, tb, kErrTimeoutProducer);
        ok = false;
        break;
      }
      __nanosleep(64);
    }
  }
  if (!ok) {
    // complete the transaction counts of our stages whose weights are in flight
    while (ko < kw) {
      if ((ctr0 + ko) % kProducers == pid) {
        const DnJob j = dn_job(p, tb, cta, G, O, nr);
        const int k = ctr0 + ko;
        dn_operand(p, j, O.c, ring.base + (size_t)(k % ring.nstages) * ring.stage_bytes,
                   ring.full + k % ring.nstages);
      }
      dn_next(O, J, nr, nch_r, nch_s);
      ++ko;
    }
  }
  *ctr_io = ctr0 + kw;
  return ok;
}

// ------------------------------------------------------------------ consumer

struct ConsumerCtx {
  uint8_t* ring_base;
  uint64_t* full;
  uint64_t* empty;
  int nstages, stage_bytes;
  float* red;        // two partial-sum buffers of kRedFloats
  float* sacc;
  uint64_t* rfull;   // [2] compute warps -> epilogue warp (buffer filled)
  uint64_t* rempty;  // [2] epilogue warp -> compute warps (buffer free)
};

// Loads from the stage ring and tables in shared memory.  The pointers reach
// the consumer through structures, so the address space is stated explicitly
// (a generic load would take the slower generic-address path).
template <typename T>
__device__ __forceinline__ T lds(const uint8_t* p) {
  const uint32_t a = smem_u32(p);
  if constexpr (sizeof(T) == 16) {
    const uint4 v = lds128(a);
    return *reinterpret_cast<const T*>(&v);
  } else if constexpr (sizeof(T) == 8) {
    const uint2 v = lds64(a);
    return *reinterpret_cast<const T*>(&v);
  } else if constexpr (sizeof(T) == 4) {
    const uint32_t v = lds32(a);
    return *reinterpret_cast<const T*>(&v);
  } else if constexpr (sizeof(T) == 2) {
    return (T)lds_u16(a);
  } else {
    return (T)lds_u8(a);
  }
}

// Stage geometry of one kind, held in registers by the consumer.
struct SG {
  int kb, Kc, K, nchunks, scale_mode, scale_off, scb, sr, opnd_off, hx_off, scale_swz;
};
__device__ __forceinline__ SG load_sg(const Geo& g) {
  SG r;
  r.kb = g.kb; r.Kc = g.Kc; r.K = g.K; r.nchunks = g.nchunks; r.scale_mode = g.scale_mode;
  r.scale_off = g.scale_off; r.scb = g.scb; r.sr = g.sr; r.opnd_off = g.opnd_off;
  r.hx_off = g.hx_off;
  r.scale_swz = (g.scale_mode == SCALES_TMAP && g.scb == 64) ? 1 : 0;
  return r;
}

// Routed gate/up stage: lane j < 16 reads gate row j, lane j >= 16 up row
// j-16; tiles [proj][128-byte column][16 rows][128 bytes] (128-byte swizzle),
// or plain rows (gate rows then up rows) when the row is under 128 bytes.
__device__ __forceinline__ const uint8_t* wptr_ar(const uint8_t* st, int kb, int lane,
                                                  int piece) {
  if (kb >= kBoxBytes)
    return st + (lane >> 4) * (kBoxesPerChunk * kDnRows * kBoxBytes) +
           (piece >> 3) * (kDnRows * kBoxBytes) + (lane & 15) * kBoxBytes +
           (((piece & 7) ^ (lane & 7)) << 4);
  return st + lane * kb + piece * 16;
}

// Address of the 16-byte piece `piece` of tile row `lane` (32-row tiles of
// 128-byte-swizzled boxes, rows >= 128 bytes) or of plain rows.
__device__ __forceinline__ const uint8_t* wptr(const uint8_t* st, int kb, int pj, int lane,
                                               int piece) {
  if (kb >= kBoxBytes)
    return st + (pj * kBoxesPerChunk + (piece >> 3)) * kBoxTileBytes + lane * kBoxBytes +
           (((piece & 7) ^ (lane & 7)) << 4);
  return st + pj * kRows * kb + lane * kb + piece * 16;
}
// Same for the 16-row tiles of the down blocks.
__device__ __forceinline__ const uint8_t* wptr16(const uint8_t* st, int kb, int row, int piece) {
  if (kb >= kBoxBytes)
    return st + (piece >> 3) * (kDnRows * kBoxBytes) + row * kBoxBytes +
           (((piece & 7) ^ (row & 7)) << 4);
  return st + row * kb + piece * 16;
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
        const uint4 w = lds<uint4>(wptr_ar(st, g.kb, lane, s));
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

// One stage of BF16 routed gate/up weights (16 gate rows over 16 up rows of
// the stacked tile, lane = row) for NT tokens against the BF16 x chunk; a
// step is 32 elements = 64 bytes of a row, products and sums in f32.
template <int NT>
__device__ __forceinline__ void compute_bf16_ar(const uint8_t* st, const SG& g,
                                                const uint8_t* obase, int otstride, int s0,
                                                int s1, int lane, float (&acc)[1][NT]) {
#pragma unroll 1
  for (int s = s0; s < s1; ++s) {
    uint32_t wv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = lds<uint4>(wptr_ar(st, g.kb, lane, s * 4 + q));
      wv[4 * q + 0] = w.x; wv[4 * q + 1] = w.y; wv[4 * q + 2] = w.z; wv[4 * q + 3] = w.w;
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
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        a0 = fma2_bf16_to_f32(wv[e], xo[e], a0);
        a1 = fma2_bf16_to_f32(wv[e + 1], xo[e + 1], a1);
      }
      acc[0][t] += a0 + a1;
    }
  }
}

// One stage of FP8 routed gate/up weights (16 gate rows over 16 up rows,
// lane = row) for NT tokens against the scaled f16 x chunk; a step is 32
// elements = 32 bytes of a row.  E4M3 -> f16 is exact, products and sums in
// f32; each step is scaled by its 128 x 128 block scale (srow: this lane's
// row of block scales, indexed by K / 128).
template <int NT>
__device__ __forceinline__ void compute_fp8_ar(const uint8_t* st, const SG& g, int c,
                                               const uint8_t* obase, int otstride, int s0,
                                               int s1, int lane, const float* srow,
                                               float (&acc)[1][NT]) {
#pragma unroll 1
  for (int s = s0; s < s1; ++s) {
    const float sc = __ldg(srow + ((c * g.Kc + s * 32) >> 7));
    const uint4 w0 = lds<uint4>(wptr_ar(st, g.kb, lane, 2 * s));
    const uint4 w1 = lds<uint4>(wptr_ar(st, g.kb, lane, 2 * s + 1));
    const uint32_t wb[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    uint32_t wv[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      wv[2 * i] = e4m3x2_to_f16x2(wb[i] & 0xFFFFu);
      wv[2 * i + 1] = e4m3x2_to_f16x2(wb[i] >> 16);
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
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        a0 = fma2_f16_to_f32(wv[e], xo[e], a0);
        a1 = fma2_f16_to_f32(wv[e + 1], xo[e + 1], a1);
      }
      acc[0][t] = fmaf(a0 + a1, sc, acc[0][t]);
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

// ------------------------------------------------------------- down compute
// 2^e for e in [-126, 127].
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

// One 16-byte piece s of a routed down job for NT tokens: per-token sum of
// its two 16-element blocks, each scaled by block scale x 2^(h exponent).
template <int FMT, int NT>
__device__ __forceinline__ void dn_piece(const uint8_t* st, const SG& g, int c, int s, int row,
                                         const uint8_t* ob, const int8_t* hx, float (&part)[kTB]) {
  const uint4 w = lds<uint4>(wptr16(st, g.kb, row, s));
  uint32_t wd[16];
  uint32_t o[4];
  e2m1x8_to_f16x2x4(w.x, o);
  wd[0] = o[0]; wd[1] = o[1]; wd[2] = o[2]; wd[3] = o[3];
  e2m1x8_to_f16x2x4(w.y, o);
  wd[4] = o[0]; wd[5] = o[1]; wd[6] = o[2]; wd[7] = o[3];
  e2m1x8_to_f16x2x4(w.z, o);
  wd[8] = o[0]; wd[9] = o[1]; wd[10] = o[2]; wd[11] = o[3];
  e2m1x8_to_f16x2x4(w.w, o);
  wd[12] = o[0]; wd[13] = o[1]; wd[14] = o[2]; wd[15] = o[3];
  float f0, f1;
  if (FMT == FMT_NVFP4) {
    const uint8_t* sa = (g.scale_mode == SCALES_TMAP)
                            ? sptr(st, g, 0, row, 2 * s)
                            : st + g.scale_off + row * g.sr + (c * g.Kc + s * 32) / 16;
    const float2 sc = f16x2_to_f32x2(e4m3x2_to_f16x2(lds<uint16_t>(sa)));
    f0 = sc.x * pow2i((int8_t)lds<uint8_t>(reinterpret_cast<const uint8_t*>(hx + 2 * s)));
    f1 = sc.y * pow2i((int8_t)lds<uint8_t>(reinterpret_cast<const uint8_t*>(hx + 2 * s + 1)));
  } else {
    const uint8_t* sa = (g.scale_mode == SCALES_TMAP)
                            ? sptr(st, g, 0, row, s)
                            : st + g.scale_off + row * g.sr + (c * g.Kc + s * 32) / 32;
    const float sc = e8m0_to_f32(lds<uint8_t>(sa));
    f0 = sc * pow2i((int8_t)lds<uint8_t>(reinterpret_cast<const uint8_t*>(hx + 2 * s)));
    f1 = sc * pow2i((int8_t)lds<uint8_t>(reinterpret_cast<const uint8_t*>(hx + 2 * s + 1)));
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const uint8_t* oa = ob + t * g.Kc * 2 + s * 64;
    uint32_t xo[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 x = lds<uint4>(oa + q * 16);
      xo[4 * q + 0] = x.x; xo[4 * q + 1] = x.y; xo[4 * q + 2] = x.z; xo[4 * q + 3] = x.w;
    }
    // four independent f16x2 chains of four
    uint32_t q0 = hmul2(wd[0], xo[0]), q1 = hmul2(wd[4], xo[4]);
    uint32_t q2 = hmul2(wd[8], xo[8]), q3 = hmul2(wd[12], xo[12]);
#pragma unroll
    for (int e = 1; e < 4; ++e) {
      q0 = hfma2(wd[e], xo[e], q0);
      q1 = hfma2(wd[4 + e], xo[4 + e], q1);
      q2 = hfma2(wd[8 + e], xo[8 + e], q2);
      q3 = hfma2(wd[12 + e], xo[12 + e], q3);
    }
    const float2 a = f16x2_to_f32x2(q0), a1 = f16x2_to_f32x2(q1);
    const float2 b = f16x2_to_f32x2(q2), b1 = f16x2_to_f32x2(q3);
    part[t] = fmaf((a.x + a.y) + (a1.x + a1.y), f0, part[t]);
    part[t] = fmaf((b.x + b.y) + (b1.x + b1.y), f1, part[t]);
  }
}

// One chunk of a routed down job: 16 weight rows (row = lane & 15) against
// the f16 h of NT tokens; the half-warp covers 16-byte pieces [p0, p1) of the
// chunk, two pieces in flight (independent partial sums).
template <int FMT, int NT>
__device__ __forceinline__ void compute_dn_fp4(const uint8_t* st, const SG& g, int c, int p0,
                                               int p1, int row, float (&acc)[kTB]) {
  const uint8_t* ob = st + g.opnd_off;
  const int8_t* hx = reinterpret_cast<const int8_t*>(st + g.hx_off);
  float pa[kTB], pb[kTB];
#pragma unroll
  for (int t = 0; t < kTB; ++t) pa[t] = pb[t] = 0.f;
  int s = p0;
  for (; s + 1 < p1; s += 2) {
    dn_piece<FMT, NT>(st, g, c, s, row, ob, hx, pa);
    dn_piece<FMT, NT>(st, g, c, s + 1, row, ob, hx, pb);
  }
  if (s < p1) dn_piece<FMT, NT>(st, g, c, s, row, ob, hx, pa);
#pragma unroll
  for (int t = 0; t < kTB; ++t) acc[t] += pa[t] + pb[t];
}

// One chunk of a routed down job with BF16 weights: 16 rows (row = lane & 15)
// against the f16 h of NT tokens; a step is 32 elements (64 bytes of a row),
// its two 16-element halves scaled by 2^(h exponent); the half-warp covers
// steps [p0, p1).  Products and sums in f32.
template <int NT>
__device__ __forceinline__ void compute_dn_bf16r(const uint8_t* st, const SG& g, int p0, int p1,
                                                 int row, float (&acc)[kTB]) {
  const uint8_t* ob = st + g.opnd_off;
  const uint8_t* hx = st + g.hx_off;
  for (int s = p0; s < p1; ++s) {
    uint32_t wv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = lds<uint4>(wptr16(st, g.kb, row, s * 4 + q));
      wv[4 * q + 0] = w.x; wv[4 * q + 1] = w.y; wv[4 * q + 2] = w.z; wv[4 * q + 3] = w.w;
    }
    const float f0 = pow2i((int8_t)lds<uint8_t>(hx + 2 * s));
    const float f1 = pow2i((int8_t)lds<uint8_t>(hx + 2 * s + 1));
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint8_t* oa = ob + t * g.Kc * 2 + s * 64;
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 x = lds<uint4>(oa + q * 16);
        const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 h = f16x2_to_f32x2(xv[i]);
          const uint32_t w = wv[4 * q + i];
          float& a = (q < 2) ? a0 : a1;
          a = fmaf(bf16_lo(w), h.x, a);
          a = fmaf(bf16_hi(w), h.y, a);
        }
      }
      acc[t] = fmaf(a0, f0, fmaf(a1, f1, acc[t]));
    }
  }
}

// One chunk of a routed down job with FP8 weights: 16 rows (row = lane & 15)
// against the f16 h of NT tokens; a step is 32 elements (32 bytes of a row),
// its two 16-element halves scaled by 2^(h exponent) and the step by its
// 128 x 128 block scale (srow: the 16 rows' row of block scales); the
// half-warp covers steps [p0, p1).  Products and sums in f32.
template <int NT>
__device__ __forceinline__ void compute_dn_fp8(const uint8_t* st, const SG& g, int c, int p0,
                                               int p1, int row, const float* srow,
                                               float (&acc)[kTB]) {
  const uint8_t* ob = st + g.opnd_off;
  const uint8_t* hx = st + g.hx_off;
  for (int s = p0; s < p1; ++s) {
    const float sc = __ldg(srow + ((c * g.Kc + s * 32) >> 7));
    const uint4 w0 = lds<uint4>(wptr16(st, g.kb, row, 2 * s));
    const uint4 w1 = lds<uint4>(wptr16(st, g.kb, row, 2 * s + 1));
    const uint32_t wb[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    uint32_t wv[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      wv[2 * i] = e4m3x2_to_f16x2(wb[i] & 0xFFFFu);
      wv[2 * i + 1] = e4m3x2_to_f16x2(wb[i] >> 16);
    }
    const float f0 = sc * pow2i((int8_t)lds<uint8_t>(hx + 2 * s));
    const float f1 = sc * pow2i((int8_t)lds<uint8_t>(hx + 2 * s + 1));
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint8_t* oa = ob + t * g.Kc * 2 + s * 64;
      uint32_t xo[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 x = lds<uint4>(oa + q * 16);
        xo[4 * q + 0] = x.x; xo[4 * q + 1] = x.y; xo[4 * q + 2] = x.z; xo[4 * q + 3] = x.w;
      }
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        a0 = fma2_f16_to_f32(wv[e], xo[e], a0);
        a1 = fma2_f16_to_f32(wv[8 + e], xo[8 + e], a1);
      }
      acc[t] = fmaf(a0, f0, fmaf(a1, f1, acc[t]));
    }
  }
}

// One chunk of a shared-expert down job: BF16 weights against BF16 h; a step
// is 32 elements (64 bytes) of the row, the half-warp covers steps [p0, p1).
template <int NT>
__device__ __forceinline__ void compute_dn_bf16(const uint8_t* st, const SG& g, int p0, int p1,
                                                int row, float (&acc)[kTB]) {
  const uint8_t* ob = st + g.opnd_off;
  for (int s = p0; s < p1; ++s) {
    uint32_t wv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = lds<uint4>(wptr16(st, g.kb, row, s * 4 + q));
      wv[4 * q + 0] = w.x; wv[4 * q + 1] = w.y; wv[4 * q + 2] = w.z; wv[4 * q + 3] = w.w;
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint8_t* oa = ob + t * g.Kc * 2 + s * 64;
      uint32_t xo[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 x = lds<uint4>(oa + q * 16);
        xo[4 * q + 0] = x.x; xo[4 * q + 1] = x.y; xo[4 * q + 2] = x.z; xo[4 * q + 3] = x.w;
      }
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        a0 = fma2_bf16_to_f32(wv[e], xo[e], a0);
        a1 = fma2_bf16_to_f32(wv[e + 1], xo[e + 1], a1);
      }
      acc[t] += a0 + a1;
    }
  }
}

// ---------------------------------------------------------- gate/up epilogue
// Epilogue of one gate/up row group, by the epilogue warp: reduce the compute
// warps' partial sums (`red`, layout [warp][proj][token][lane]) and store h.
// Shared expert: BF16 h of 32 rows.  Routed: lanes 0-15 of the tile are gate
// rows, 16-31 up rows; h = SiLU(g)*u for the 16 rows, stored as f16 times
// 2^-e with e chosen from the group's largest |h| (max in [64, 128)).
// Routed group epilogue for NT token slots (nt <= NT of them used).
template <int NT>
__device__ __forceinline__ void rg_epilogue_ar(const Params& p, const Tables& tb, const RG& r,
                                               const float* red, int lane) {
  const int j = lane;
  const float g2 = tb.s2[0][r.u], u2 = tb.s2[1][r.u];
  float h[NT];
  float m = 0.f;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    h[t] = 0.f;
    if (t < r.nt) {
      float g = 0.f, u = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        g += red[((w * 2) * kTB + t) * 32 + j];
        u += red[((w * 2) * kTB + t) * 32 + 16 + j];
      }
      // FP4 / FP8 experts ran on x * 2^-xe; BF16 routed experts on x itself
      const float xs = (p.fmt == FMT_BF16) ? 1.0f : exp2i(tb.xe[rg_token<KIND_AR>(tb, r, t)]);
      g *= xs * g2;
      u *= xs * u2;
      h[t] = silu(g) * u;
      m = fmaxf(m, fabsf(h[t]));
    }
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0x0000ffffu, m, o));
  const int e = min(max(scale_exponent(m), -126), 127);
  const float sc = pow2i(-e);
  const int slot0 = tb.hoff[r.u] + r.tb * kTB;
#pragma unroll
  for (int t = 0; t < NT; ++t)
    if (t < r.nt)
      p.h16[(size_t)(slot0 + t) * p.inter + r.rg * kDnRows + j] =
          __half_as_ushort(__float2half_rn(h[t] * sc));
  if (j == 0) p.hexp[(size_t)r.unit * p.hstride + r.rg] = (int8_t)e;
}

template <int KIND>
__device__ __forceinline__ void rg_epilogue(const Params& p, const Tables& tb, const RG& r,
                                            const float* red, int lane) {
  if (KIND == KIND_AS) {
    for (int t = 0; t < r.nt; ++t) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        s0 += red[((w * 2 + 0) * kTB + t) * 32 + lane];
        s1 += red[((w * 2 + 1) * kTB + t) * 32 + lane];
      }
      const int n = rg_token<KIND>(tb, r, t);
      const __nv_bfloat16 hb = __float2bfloat16_rn(silu(s0) * s1);
      p.hs[(size_t)n * p.Is + r.rg * kRows + lane] = *reinterpret_cast<const uint16_t*>(&hb);
    }
  } else if (lane < 16) {
    if (r.nt == 1) rg_epilogue_ar<1>(p, tb, r, red, lane);
    else if (r.nt == 2) rg_epilogue_ar<2>(p, tb, r, red, lane);
    else rg_epilogue_ar<kTB>(p, tb, r, red, lane);
  }
}

// The epilogue warp's loop over one gate/up kind's row groups (same order as
// the compute warps); routed groups are then published to the units'
// readiness counters (release: every lane's h stores, the warp barrier, lane
// 0's fence and counts).  Returns the number of row groups, or -1 on abort.
template <int KIND>
__device__ __noinline__ int epilogue_kind(const Params& p, Tables& tb, const ConsumerCtx cx,
                                          int cta, int G, int* rgk_io, int lane) {
  if (kind_units<KIND>(p, tb) == 0) return 0;
  int lo, hi;
  kind_range<KIND>(p, tb, cta, G, lo, hi);
  int kk = *rgk_io;
  for (int gi = lo; gi < hi; ++gi, ++kk) {
    const RG r = decode_rg<KIND>(p, tb, gi);
    const int buf = kk & 1;
    bool ok = !aborted(tb) && mbar_wait_bounded(cx.rfull + buf, (uint32_t)(kk >> 1) & 1u,
                                                 p.timeout_ns);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) {
      if (lane == 0 && !aborted(tb)) set_abort(p, tb, kErrTimeoutStage);
      return -1;
    }
    rg_epilogue<KIND>(p, tb, r, cx.red + buf * kRedFloats, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.rempty + buf);
  }
  *rgk_io = kk;
  if (KIND == KIND_AR && lane == 0 && lo < hi) {
    const int rpu = p.inter / kDnRows;
    __threadfence();
    for (int u = lo / rpu; u <= (hi - 1) / rpu; ++u)
      atomicAdd(p.ready + u, (uint32_t)(min(hi, (u + 1) * rpu) - max(lo, u * rpu)));
  }
  return hi - lo;
}

// Streams the chunks of one gate/up row group for NT tokens and leaves the 8
// warps' partial sums in `red` (layout [warp][proj][token][lane]).
template <int FMT, int NPROJ, int KIND, int NT>
__device__ __forceinline__ void consume_rg(const Params& p, Tables& tb, const ConsumerCtx& cx,
                                           const SG& g, int& ctr, int warp, int lane, float* red,
                                           const float* srow) {
  constexpr int kStepBytes = (FMT == FMT_BF16) ? 64 : (FMT == FMT_FP8) ? 32 : 16;
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
      const uint8_t* ob = st + g.opnd_off;
      const int ots = g.Kc * 2;
      if constexpr (FMT == FMT_BF16 && KIND == KIND_AR)
        compute_bf16_ar<NT>(st, g, ob, ots, s0, s1, lane, acc);
      else if constexpr (FMT == FMT_FP8)
        compute_fp8_ar<NT>(st, g, c, ob, ots, s0, s1, lane, srow, acc);
      else if constexpr (FMT == FMT_BF16)
        compute_bf16<NPROJ, NT>(st, g, ob, ots, s0, s1, lane, acc);
      else
        compute_fp4<FMT, NPROJ, NT>(st, g, c, ob, ots, s0, s1, lane, acc);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.empty + slot);
  }
#pragma unroll
  for (int pj = 0; pj < NPROJ; ++pj)
#pragma unroll
    for (int t = 0; t < NT; ++t)
      sts32(smem_u32(red + ((warp * 2 + pj) * kTB + t) * 32 + lane), __float_as_uint(acc[pj][t]));
}

// Compute warps: every stage of one gate/up kind's row groups; each group's
// partial sums go to one of two buffers that the epilogue warp finishes.
template <int FMT, int NPROJ, int KIND>
__device__ __noinline__ void consume_kind(const Params& p, Tables& tb, const ConsumerCtx cx,
                                          int cta, int G, int* ctr_io, int* rgk_io, int ctid) {
  if (kind_units<KIND>(p, tb) == 0) return;
  const int warp = ctid >> 5, lane = ctid & 31;
  int lo, hi;
  kind_range<KIND>(p, tb, cta, G, lo, hi);
  const SG g = load_sg(p.geo[KIND]);
  int ctr = *ctr_io, kk = *rgk_io;
  for (int gi = lo; gi < hi; ++gi, ++kk) {
    const RG r = decode_rg<KIND>(p, tb, gi);
    const int buf = kk & 1;
    // the buffer's previous group (kk - 2) must be finished by the epilogue warp
    if (!aborted(tb) &&
        !mbar_wait_bounded(cx.rempty + buf, ((uint32_t)(kk >> 1) & 1u) ^ 1u, p.timeout_ns) &&
        lane == 0)
      set_abort(p, tb, kErrTimeoutStage);
    float* red = cx.red + buf * kRedFloats;
    const float* srow = nullptr;   // FP8: this lane's row of 128 x 128 block scales
    if constexpr (FMT == FMT_FP8) {
      const int nkb = (p.H + kFp8Block - 1) / kFp8Block;
      const int nrb = (p.inter + kFp8Block - 1) / kFp8Block;
      const float* tab = reinterpret_cast<const float*>(lane < 16 ? p.gsc : p.usc);
      srow = tab + ((size_t)r.e * nrb + (r.rg * kDnRows) / kFp8Block) * nkb;
    }
    switch (r.nt) {
      case 1: consume_rg<FMT, NPROJ, KIND, 1>(p, tb, cx, g, ctr, warp, lane, red, srow); break;
      case 2: consume_rg<FMT, NPROJ, KIND, 2>(p, tb, cx, g, ctr, warp, lane, red, srow); break;
      case 3: consume_rg<FMT, NPROJ, KIND, 3>(p, tb, cx, g, ctr, warp, lane, red, srow); break;
      default: consume_rg<FMT, NPROJ, KIND, 4>(p, tb, cx, g, ctr, warp, lane, red, srow); break;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(cx.rfull + buf);
  }
  *ctr_io = ctr;
  *rgk_io = kk;
}

// Down jobs of this CTA's output blocks (same order as produce_down).  With
// J jobs per block and W consumer warps, a job belongs to S = W / J (a power
// of two, at least 1) consecutive warps, each taking one K slice per
// half-warp; every warp passes every stage (the ring's release count is W),
// only the owners compute.  Each owner adds its routing-weighted partial into
// the block accumulator in shared memory.
template <int FMT>
__device__ __noinline__ void consume_down(const Params& p, Tables& tb, const ConsumerCtx cx,
                                          int cta, int G, int* ctr_io, int ctid) {
  const int warp = ctid >> 5, lane = ctid & 31, row = lane & 15, half = lane >> 4;
  const int nrbl = dn_blocks(p, cta, G);
  const int nr = tb.n_units, nsh = p.Is > 0 ? (p.N + kTB - 1) / kTB : 0, J = nr + nsh;
  if (nrbl == 0 || J == 0) return;
  const SG gr = load_sg(p.geo[KIND_BR]);
  const SG gsh = load_sg(p.geo[nsh ? KIND_BS : KIND_BR]);
  int S = 1;
  while (S * 2 * J <= kConsumerWarps) S *= 2;
  int ctr = *ctr_io;
  int q = 0;
  for (int i = 0; i < nrbl; ++i) {
    for (int jb = 0; jb < J; ++jb, ++q) {
      const int w0 = (q * S) & (kConsumerWarps - 1);
      const bool own = warp >= w0 && warp < w0 + S;
      const int slice = (warp - w0) * 2 + half, nslice = 2 * S;
      const bool routed = jb < nr;
      const SG& g = routed ? gr : gsh;
      int nt, src0;
      float d2 = 1.0f;   // down scale2, loaded at job start (latency hidden by the compute)
      const float* srow = nullptr;   // FP8: the block's row of 128 x 128 block scales
      if (routed) {
        const int u = tb.unit_u[jb], tbi = tb.unit_tb[jb];
        nt = min(kTB, (int)tb.ucnt[u] - tbi * kTB);
        src0 = tb.hoff[u] + tbi * kTB;
        if (own && p.d2) d2 = __ldg(p.d2 + tb.uexp[u]);
        if constexpr (FMT == FMT_FP8) {
          const int nkb = (p.inter + kFp8Block - 1) / kFp8Block;
          const int nrb = (p.H + kFp8Block - 1) / kFp8Block;
          srow = reinterpret_cast<const float*>(p.dsc) +
                 ((size_t)tb.uexp[u] * nrb + ((cta + i * G) * kDnRows) / kFp8Block) * nkb;
        }
      } else {
        const int b = jb - nr;
        nt = min(kTB, p.N - b * kTB);
        src0 = b * kTB;
      }
      float acc[kTB];
#pragma unroll
      for (int t = 0; t < kTB; ++t) acc[t] = 0.f;
      for (int c = 0; c < g.nchunks; ++c) {
        const int slot = ctr % cx.nstages;
        const uint32_t round = (uint32_t)(ctr / cx.nstages);
        ++ctr;
        bool ok = !aborted(tb);
        if (ok) ok = mbar_wait_bounded(cx.full + slot, round & 1u, p.timeout_ns);
        if (!ok) {
          if (lane == 0 && !aborted(tb)) set_abort(p, tb, kErrTimeoutStage);
        } else if (own) {
          const uint8_t* st = cx.ring_base + (size_t)slot * cx.stage_bytes;
          const int rb = min(kChunkBytes, g.kb - c * kChunkBytes);
          if (routed) {
            if constexpr (FMT == FMT_BF16) {
              const int np = rb / 64;
              const int p0 = slice * np / nslice, p1 = (slice + 1) * np / nslice;
              switch (nt) {
                case 1: compute_dn_bf16r<1>(st, g, p0, p1, row, acc); break;
                case 2: compute_dn_bf16r<2>(st, g, p0, p1, row, acc); break;
                case 3: compute_dn_bf16r<3>(st, g, p0, p1, row, acc); break;
                default: compute_dn_bf16r<4>(st, g, p0, p1, row, acc); break;
              }
            } else if constexpr (FMT == FMT_FP8) {
              const int np = rb / 32;
              const int p0 = slice * np / nslice, p1 = (slice + 1) * np / nslice;
              switch (nt) {
                case 1: compute_dn_fp8<1>(st, g, c, p0, p1, row, srow, acc); break;
                case 2: compute_dn_fp8<2>(st, g, c, p0, p1, row, srow, acc); break;
                case 3: compute_dn_fp8<3>(st, g, c, p0, p1, row, srow, acc); break;
                default: compute_dn_fp8<4>(st, g, c, p0, p1, row, srow, acc); break;
              }
            } else {
              const int np = rb / 16;
              const int p0 = slice * np / nslice, p1 = (slice + 1) * np / nslice;
              switch (nt) {
                case 1: compute_dn_fp4<FMT, 1>(st, g, c, p0, p1, row, acc); break;
                case 2: compute_dn_fp4<FMT, 2>(st, g, c, p0, p1, row, acc); break;
                case 3: compute_dn_fp4<FMT, 3>(st, g, c, p0, p1, row, acc); break;
                default: compute_dn_fp4<FMT, 4>(st, g, c, p0, p1, row, acc); break;
              }
            }
          } else {
            const int np = rb / 64;
            const int p0 = slice * np / nslice, p1 = (slice + 1) * np / nslice;
            switch (nt) {
              case 1: compute_dn_bf16<1>(st, g, p0, p1, row, acc); break;
              case 2: compute_dn_bf16<2>(st, g, p0, p1, row, acc); break;
              case 3: compute_dn_bf16<3>(st, g, p0, p1, row, acc); break;
              default: compute_dn_bf16<4>(st, g, p0, p1, row, acc); break;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(cx.empty + slot);
      }
      if (own && !aborted(tb)) {
#pragma unroll
        for (int t = 0; t < kTB; ++t) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], 16);
        if (lane < 16) {
#pragma unroll
          for (int t = 0; t < kTB; ++t) {
            if (t < nt) {
              const int n = routed ? tb.utok[src0 + t] : src0 + t;
              const float wgt = routed ? tb.uw[src0 + t] * d2 : ld_cg_f32(p.gsig + n);
              red_add_shared_f32(smem_u32(cx.sacc + ((size_t)i * p.N + n) * kDnRows + row),
                                 acc[t] * wgt);
            }
          }
        }
      }
    }
  }
  *ctr_io = ctr;
}

// ------------------------------------------------------------------- kernel

// EXT: the routing variants (softmax + bias scoring, zero experts, hash
// routing, NVFP4 router) are compiled in; the common layers launch EXT = false.
template <int WF, bool EXT>
__global__ void __launch_bounds__(kThreads, 1) moe_decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte-swizzled TMA boxes need a 1024-byte aligned destination
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Tables& tb = *reinterpret_cast<Tables*>(smem + p.smem_tab_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.smem_bar_off);
  uint64_t* full = bars;
  uint64_t* empty = bars + kMaxStages;
  uint64_t* rr = bars + 2 * kMaxStages;  // routing tables ready (consumers -> producer)
  uint64_t* rfull = rr + 1;
  uint64_t* rempty = rr + 3;
  const int tid = threadIdx.x;
  const int cta = blockIdx.x, G = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < p.nstages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kConsumerWarps);
    }
    mbar_init(rr, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(rfull + i, kConsumerWarps);
      mbar_init(rempty + i, 1);
    }
    fence_mbar_init();
    tb.abort = 0;
    tb.n_units = 0;
    tb.U = 0;
  }
  __syncthreads();

  float* red = reinterpret_cast<float*>(smem + p.smem_red_off);
  float* sacc = reinterpret_cast<float*>(smem + p.smem_sacc_off);
  ConsumerCtx cx{smem + p.smem_ring_off, full, empty, p.nstages, p.stage_bytes, red, sacc,
                 rfull, rempty};

  if ((tid >> 5) == kEpiWarp) {
    // ------------------------------------------------------ epilogue warp
    if (p.route_only) return;
    const int lane = tid & 31;
    int kk = 0;
    const int as_done = epilogue_kind<KIND_AS>(p, tb, cx, cta, G, &kk, lane);
    bool ok = as_done >= 0 && mbar_wait_bounded(rr, 0, p.timeout_ns);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok || aborted(tb)) return;
    // shared-expert h rows of this CTA are complete; the readiness counters
    // were zeroed everywhere before B1, which the routing (rr) came after
    __syncwarp();
    if (lane == 0 && as_done > 0) {
      __threadfence();
      atomicAdd(p.ready + kReadyAS, (uint32_t)as_done);
    }
    load_scale2(p, tb, lane);
    epilogue_kind<KIND_AR>(p, tb, cx, cta, G, &kk, lane);
    return;
  }
  if (tid >= kConsumerThreads) {
    // ------------------------------- producers (lane 0 of each producer warp)
    if ((tid & 31) != 0 || p.route_only) return;
    const int pid = (tid - kConsumerThreads - 32) >> 5;
    for (int i = pid; i < TM_COUNT; i += kProducers)
      if (p.tm_valid & (1u << i)) prefetch_tensormap(&p.tm[i]);
    Ring ring{smem + p.smem_ring_off, full, empty, p.nstages, p.stage_bytes};
    int ctr = 0;
    bool ok = produce_kind<KIND_AS>(p, tb, ring, cta, G, &ctr, pid);
    if (ok && !mbar_wait_bounded(rr, 0, p.timeout_ns)) {
      set_abort(p, tb, kErrTimeoutProducer);
      ok = false;
    }
    if (ok && aborted(tb)) ok = false;
    if (ok) {
      fence_proxy_async_global();   // x16 was written by other CTAs before B1
      ok = produce_kind<KIND_AR>(p, tb, ring, cta, G, &ctr, pid) &&
           produce_down(p, tb, ring, cta, G, &ctr, pid);
    }
    if (!ok) {
      // drain: wait (bounded) for copies still in flight into our stages
      const int first = ctr > p.nstages ? ctr - p.nstages : 0;
      for (int i = first; i < ctr; ++i)
        if (i % kProducers == pid)
          mbar_wait_bounded(full + (i % p.nstages), (uint32_t)(i / p.nstages) & 1u, p.timeout_ns);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = tid;
  unsigned long long base = 0;
  if (ctid == 0) {
    const unsigned long long c0 = ld_relaxed_u64(&p.ctrl->arrivals);
    base = c0 - c0 % (unsigned long long)G;
  }

  // P0: router, token prep, zero the readiness counters and the block accumulator
  router_phase<EXT>(p, cta, G, tb, ctid);
  const int nrbl = p.route_only ? 0 : dn_blocks(p, cta, G);
  if (!p.route_only) {
    token_prep(p, cta, G, tb, ctid);
    for (int i = cta * kConsumerThreads + ctid; i <= kReadyAS; i += G * kConsumerThreads)
      p.ready[i] = 0u;
    for (int i = ctid; i < nrbl * p.N * kDnRows; i += kConsumerThreads) sacc[i] = 0.f;
  }
  consumer_sync();
  if (ctid == 0) {
    __threadfence();
    grid_arrive(p.ctrl);    // B1
  }

  int ctr = 0, kk = 0;
  if (!p.route_only) consume_kind<FMT_BF16, 2, KIND_AS>(p, tb, cx, cta, G, &ctr, &kk, ctid);

  if (ctid == 0 && !grid_wait(p.ctrl, base + (unsigned long long)G, p.timeout_ns))
    set_abort(p, tb, kErrTimeoutBarrier);
  consumer_sync();
  if (aborted(tb)) {
    if (ctid == 0) mbar_arrive(rr);
    return;   // the producer sees the abort and drains
  }

  // P1: routing
  routing_phase<EXT>(p, cta == 0, tb, ctid);
  if (p.route_only) return;
  if (ctid == 0) mbar_arrive(rr);

  // P2: routed gate/up; P3: down jobs of the owned output blocks
  consume_kind<WF, 1, KIND_AR>(p, tb, cx, cta, G, &ctr, &kk, ctid);
  consume_down<WF>(p, tb, cx, cta, G, &ctr, ctid);
  consumer_sync();
  if (aborted(tb)) return;
  for (int idx = ctid; idx < nrbl * p.N * kDnRows; idx += kConsumerThreads) {
    const int i = idx / (p.N * kDnRows), rem = idx - i * p.N * kDnRows;
    const int n = rem / kDnRows, j = rem - n * kDnRows;
    const __nv_bfloat16 b = __float2bfloat16_rn(sacc[idx]);
    p.out[(size_t)n * p.H + (size_t)(cta + i * G) * kDnRows + j] =
        *reinterpret_cast<const uint16_t*>(&b);
  }
}

// ------------------------------------------------------------------- host

// Stage geometry of one kind: weight tiles, block scales, activation chunk.
static bool plan_kind(Geo& g, int kind, int fmt, int K, int rows, int ntok) {
  const int nproj = (kind == KIND_AS || kind == KIND_AR) ? 2 : 1;
  g.fmt = fmt;
  g.nproj = nproj;
  g.brows = (kind == KIND_AS) ? kRows : kDnRows;
  g.rg_rows = g.brows;
  g.K = K;
  g.rows_total = rows;
  g.opnd_off = -1;
  if (K % 32 != 0 || rows % g.rg_rows != 0 || K <= 0 || rows <= 0) return false;
  g.kb = (fmt == FMT_BF16) ? K * 2 : (fmt == FMT_FP8) ? K : K / 2;
  g.Kc = (fmt == FMT_BF16) ? kChunkBytes / 2 : (fmt == FMT_FP8) ? kChunkBytes : kChunkBytes * 2;
  g.nchunks = (g.kb + kChunkBytes - 1) / kChunkBytes;
  const bool sw = g.kb >= kBoxBytes;
  // AS: one 32-row tile per projection; AR: gate and up 16-row boxes stacked
  // into one 32-row tile; BR/BS: one 16-row tile
  int wbytes;
  if (kind == KIND_AS) {
    g.tile_bytes = kBoxTileBytes;
    wbytes = sw ? nproj * kBoxesPerChunk * kBoxTileBytes : nproj * kRows * g.kb;
  } else if (kind == KIND_AR) {
    g.tile_bytes = kDnRows * kBoxBytes;
    wbytes = sw ? 2 * kBoxesPerChunk * kDnRows * kBoxBytes : kRows * g.kb;
  } else {
    g.tile_bytes = kDnRows * kBoxBytes;
    wbytes = sw ? kBoxesPerChunk * kDnRows * kBoxBytes : kDnRows * g.kb;
  }
  g.use3d = (g.kb % kBoxBytes == 0) ? 1 : 0;   // whole 128-byte columns only
  int off = (wbytes + 1023) / 1024 * 1024;
  g.scale_off = off;
  g.sr = g.scb = 0;
  g.scale_mode = SCALES_NONE;
  if (fmt == FMT_NVFP4 || fmt == FMT_MXFP4) {   // FP8 block scales are read from global
    const int gs = (fmt == FMT_NVFP4) ? 16 : 32;
    g.sr = K / gs;
    if (g.sr % 16 == 0) {
      g.scale_mode = SCALES_TMAP;
      g.scb = std::min(g.Kc / gs, g.sr);
      off += nproj * g.brows * g.scb;
    } else {
      g.scale_mode = SCALES_BLOCK;
      off += nproj * g.brows * g.sr;
    }
    off = (off + 127) / 128 * 128;
  }
  g.opnd_off = off;
  off += ntok * g.Kc * 2;                  // activation chunk of up to ntok tokens
  g.hx_off = off;
  if (kind == KIND_BR) off += g.Kc / 16;   // h exponents of the chunk
  g.stage_bytes = (off + 1023) / 1024 * 1024;
  return true;
}

bool plan_decode(Params& p, int smem_budget, int grid) {
  const int wf = (p.fmt == 0) ? FMT_NVFP4 : (p.fmt == 1) ? FMT_MXFP4
               : (p.fmt == 2) ? FMT_BF16 : FMT_FP8;
  const int ntok = std::min(p.N, kTB);   // tokens per activation chunk
  if (!plan_kind(p.geo[KIND_AR], KIND_AR, wf, p.H, p.inter, ntok)) return false;
  if (!plan_kind(p.geo[KIND_BR], KIND_BR, wf, p.inter, p.H, ntok)) return false;
  int stage = std::max(p.geo[KIND_AR].stage_bytes, p.geo[KIND_BR].stage_bytes);
  if (p.Is > 0) {
    if (!plan_kind(p.geo[KIND_AS], KIND_AS, FMT_BF16, p.H, p.Is, ntok)) return false;
    if (!plan_kind(p.geo[KIND_BS], KIND_BS, FMT_BF16, p.Is, p.H, ntok)) return false;
    stage = std::max(stage, std::max(p.geo[KIND_AS].stage_bytes, p.geo[KIND_BS].stage_bytes));
  } else {
    p.geo[KIND_AS] = p.geo[KIND_AR];
    p.geo[KIND_BS] = p.geo[KIND_BR];
  }
  p.hstride = ((p.inter / kDnRows) + 15) / 16 * 16;
  p.nrb = p.H / kDnRows;
  p.nrb_cta = (p.nrb + grid - 1) / grid;
  const int red = 2 * kRedFloats * 4;
  const int sacc = ((p.nrb_cta * p.N * kDnRows * 4) + 127) / 128 * 128;
  const int tab = ((int)sizeof(Tables) + 127) / 128 * 128;
  const int bars = (2 * kMaxStages + 5) * 8;
  const int fixed = red + sacc + tab + ((bars + 127) / 128 * 128);
  int ns = (smem_budget - fixed) / stage;
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) return false;
  p.nstages = ns;
  p.stage_bytes = stage;
  p.smem_ring_off = 0;
  p.smem_red_off = ns * stage;
  p.smem_sacc_off = p.smem_red_off + red;
  p.smem_tab_off = p.smem_sacc_off + sacc;
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
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  const void* kernels[8] = {(const void*)moe_decode_kernel<FMT_NVFP4, false>,
                            (const void*)moe_decode_kernel<FMT_MXFP4, false>,
                            (const void*)moe_decode_kernel<FMT_BF16, false>,
                            (const void*)moe_decode_kernel<FMT_FP8, false>,
                            (const void*)moe_decode_kernel<FMT_NVFP4, true>,
                            (const void*)moe_decode_kernel<FMT_MXFP4, true>,
                            (const void*)moe_decode_kernel<FMT_BF16, true>,
                            (const void*)moe_decode_kernel<FMT_FP8, true>};
  for (const void* k : kernels) {
    int nb = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, k, kThreads, smem_bytes) != cudaSuccess ||
        nb < 1)
      return 0;
  }
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
  // the routing variants run the EXT build of the kernel
  const bool ext = p.scoring == 2 || p.Z > 0 || p.hash_V > 0 || p.router_fmt != 0;
  if (ext) {
    if (p.fmt == 0) return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_NVFP4, true>, p);
    if (p.fmt == 1) return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_MXFP4, true>, p);
    if (p.fmt == 2) return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_BF16, true>, p);
    return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_FP8, true>, p);
  }
  if (p.fmt == 0) return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_NVFP4, false>, p);
  if (p.fmt == 1) return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_MXFP4, false>, p);
  if (p.fmt == 2) return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_BF16, false>, p);
  return cudaLaunchKernelEx(&cfg, moe_decode_kernel<FMT_FP8, false>, p);
}

}  // namespace moe
