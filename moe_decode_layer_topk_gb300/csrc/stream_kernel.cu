// Fused MoE decode-layer forward for up to 8 token rows with FP4 routed
// experts (NVFP4 or MXFP4) and an optional BF16 shared expert, on sm_103a:
// one cooperative launch per call.
//
// The chain is the one forward_k3.rs's MoeLayer::forward_k3 doc comment lists
// (router GEMV over the token batch, batched top-k, expert gate+up, SiLU and
// down, weighted sum + shared blend), with each touched expert's weights read
// once for all rows of the call (forward_batched.rs: one pass over an expert's
// weights serves every row routed to it) and the experts summed in FP32
// before one BF16 cast (forward_atomic_c4.rs, forward_atomic_c4_decode).
//
// Execution model: one CTA per SM, 16 warps, every CTA resident at once.
//
//   P0  the router weight rows of this CTA (e = cta, cta + G, ...) are
//       requested first; meanwhile every CTA builds its f16 copy of x (scaled
//       by a power of two per token) in shared memory, in the order the MMA B
//       fragments read it, and the shared-expert gate sigmoid(w_s . x).  The
//       logits (FP32) are stored as 64-bit words tagged with the call number.
//   PS  shared-expert gate/up (independent of the routing, so it runs while
//       the logits land): its 16-row tiles are split along K over the last
//       CTAs; parts meet in an FP32 buffer, the last part stores the tile's
//       h = gate * SiLU(g) * u as BF16 and tags the tile.
//   P1  every CTA polls the N x E tagged logits (no grid barrier: a word
//       carries its own validity), computes the same top-k and the same table
//       of unique experts.
//   P2  routed gate/up: the U x inter/16 tiles (16 rows of gate and of up of
//       one expert) go round-robin to the CTAs, so the experts complete one
//       after another; inside a CTA the warps split the (tile, 128-column K
//       segment, projection) items evenly.  A tile finished by one warp is
//       finalised from registers; one shared by several warps meets in a
//       shared-memory accumulator and the last warp finalises it:
//       h = w * scale2_down * SiLU(g) * u goes to f16 per (token, slot) and
//       the tile is tagged with the call number.
//   P3  down: the grid's (shared K segment, row tile) and (expert, K segment,
//       32-row tile) items are split over all warps in order; a routed item
//       waits only for the eight gate/up tiles its K segment reads.  Partial
//       sums go to an FP32 accumulator in global memory by vector reductions;
//       once every CTA has counted itself done at the end counter, each CTA
//       converts its H / G output rows to BF16.  The item pipeline runs from
//       P2 straight into P3, so the first down weights are in flight while
//       the last gate/up items compute.
//
// Weight streaming: an item's code rows (16 rows x 64 bytes of gate and of
// up, or 32 rows x 64 bytes of down) come by TMA, issued by lane 0, into the
// warp's two-stage ring, with their block scales as a 16-byte column of the
// scale rows by TMA too (by per-lane 4-byte copies when scale rows are not
// 16-byte multiples); one mbarrier per stage counts the bytes.  With one item
// in flight per warp the grid keeps about 6 MB of weight reads queued.
//
// Arithmetic: E2M1 -> f16 by cvt, times the E4M3 block scale (exact in f16:
// at most 6 significant bits, range 2^-10 .. 2688), or for MXFP4 times
// 2^(E8M0 - segment maximum) with 2^(maximum - 127) applied to the FP32 MMA
// result.  The dot products are mma.sync m16n8k16 (f16 or bf16 in, FP32
// accumulate): 16 weight rows x 16 K x 8 tokens, the token rows being the B
// columns, so the instruction count does not grow with N up to 8.  Inside a
// lane's piece, MMA K step s takes elements 4s .. 4s+3; B is read with the
// same permutation, so every product pairs the right x (or h) element.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kW = kSkWarps;
constexpr int kT = kSkThreads;
constexpr int kMaxRouterRows = 8;     // router rows per CTA (E <= 1024, G >= 128)

struct SkTab {
  int U;
  int abort;
  uint32_t tag;
  int pad0;
  int xe[kSkMaxTok];
  float xf[kSkMaxTok];
  float gsig[kSkMaxTok];
  int16_t sel_e[kMaxSlots];
  float sel_w[kMaxSlots];
  uint32_t first[kMaxE];
  float bias[kMaxE];
  float s2[kMaxE][3];   // per-expert second-level scales: gate, up, down (1 without)
  int16_t u_e[kMaxSlots];
  uint32_t u_mask[kMaxSlots];
  float u_w[kMaxSlots][kSkMaxTok];
  int16_t u_slot[kMaxSlots][kSkMaxTok];
  uint32_t split_cnt[kSkSplitSlots];
  uint64_t full[kSkWarps][kSkStages];   // per warp and ring stage: the stage's TMA bytes have landed
  float part[kSkMaxTok][8][2];   // per token and 128-expert part: max, sum exp(l - max)
  uint32_t xmax[kSkMaxTok];   // max |x| per token (float bits)
  float xdot[kSkMaxTok];       // w_s . x per token
  float gmax[kSkMaxTok], gden[kSkMaxTok];
};

// ------------------------------------------------------------------ helpers
// 16-byte weight piece (zero fill past n bytes) with a 256-byte L2 prefetch
// (the row's next pieces are other items of the same CTA or its neighbours).
__device__ __forceinline__ void cpa16w(uint32_t dst, const void* src, uint32_t n) {
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
// 4-byte block-scale word.
__device__ __forceinline__ void cpa4w(uint32_t dst, const void* src, uint32_t n) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
// Prior generic-proxy accesses to shared memory before later async-proxy
// (TMA) writes of this thread.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 16-byte activation piece (x or h), default L2 policy.
__device__ __forceinline__ void cpa16(uint32_t dst, const void* src, uint32_t n) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// D += A * B, m16n8k16, FP32 accumulators; f16 or bf16 operands.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t dup_lo(uint32_t v) { return __byte_perm(v, v, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t v) { return __byte_perm(v, v, 0x3232); }

// f16x2 {2^d, 2^d} for d <= 0 (0 below the f16 subnormal range).
__device__ __forceinline__ uint32_t pow2_f16x2(int d) {
  const uint32_t b = d >= -14 ? (uint32_t)(15 + d) << 10 : (d >= -24 ? 1u << (d + 24) : 0u);
  return b | (b << 16);
}

__device__ __forceinline__ void st_relaxed64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// floor(log2(m)) of a positive finite float.
__device__ __forceinline__ int ilog2f(float m) {
  const uint32_t b = __float_as_uint(m);
  const int ex = (int)((b >> 23) & 0xFFu);
  return ex ? ex - 127 : -118 - __clz(b & 0x7FFFFFu);
}
// 2^e as a float for e in [-252, 254].
__device__ __forceinline__ float pow2f(int e) {
  const int e1 = e >> 1;
  return __int_as_float((e1 + 127) << 23) * __int_as_float((e - e1 + 127) << 23);
}
// e^x as 2^(x log2 e) on the hardware base-2 exponential, and 1/x on the
// hardware reciprocal (both approximate, denormals flushed to zero: the
// non-flushing forms carry fix-up code, and most of this file runs once per
// launch, where every instruction is a cold fetch).
__device__ __forceinline__ float exp_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * 1.44269504088896341f));
  return y;
}
__device__ __forceinline__ float rcp_fast(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_fast(float v) { return rcp_fast(1.0f + exp_fast(-v)); }
__device__ __forceinline__ float silu(float v) { return v * sigmoid_fast(v); }
// a / d for 0 <= a < 2^21 and 0 < d < 2^21: a float quotient (error well
// under one unit) corrected by one step; a few instructions where the integer
// division takes dozens, which matters in code that runs once per launch.
__device__ __forceinline__ int divs(int a, int d) {
  int q = __float2int_rz((float)a * rcp_fast((float)d));
  const int r = a - q * d;
  q += r >= d ? 1 : (r < 0 ? -1 : 0);
  return q;
}

__device__ __noinline__ void set_error(const StreamParams& p, SkTab& tb, uint32_t bit) {
  atomicOr(&p.ctrl->error, bit);
  *(volatile int*)&tb.abort = 1;
}

// Lanes 0..n-1 each wait until *(words[lane]) == tag (bounded, with backoff);
// then every lane's later reads are ordered after the observed writes.
__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire_tag(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return (uint32_t)(v >> 32);
}
__device__ __forceinline__ void st_flag(unsigned long long* p, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"((unsigned long long)tag << 32)
               : "memory");
}
// Waits (bounded) until flags words[0 .. n) (n <= 32) carry this call's tag.
// Acquire loads: once a lane has seen its flag, the writes published before
// it are visible to the whole warp after the __syncwarp.  (A fence here would
// also wait for this warp's weight copies in flight.)
__device__ __noinline__ void wait_tags(const StreamParams& p, SkTab& tb,
                                       const unsigned long long* words, int n, uint32_t tag,
                                       int lane) {
  bool ok = lane >= n || ld_acquire_tag(words + lane) == tag;
  if (!__all_sync(0xffffffffu, ok)) {
    const uint64_t t0 = global_timer_ns();
    while (!__all_sync(0xffffffffu, ok)) {
      if (*(volatile int*)&tb.abort) break;
      if (global_timer_ns() - t0 > p.timeout_ns) {
        if (lane == 0) set_error(p, tb, kErrTimeoutStage);
        break;
      }
      __nanosleep(200);
      if (!ok) ok = ld_acquire_tag(words + lane) == tag;
    }
  }
  __syncwarp();
}
__device__ __forceinline__ void st_tagged(unsigned long long* p, uint32_t v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p),
               "l"(((unsigned long long)tag << 32) | v)
               : "memory");
}
// Adds a lane's C fragment (rows r, r + 8; columns 2t, 2t+1) to the FP32
// output accumulator [H][ld] (ld even) at o = row r, column 2t: two vector
// reductions, fire and forget.
__device__ __forceinline__ void red_out(float* o, int ld, const float (&c)[4]) {
  asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" ::"l"(o), "f"(c[0]), "f"(c[1])
               : "memory");
  asm volatile("red.relaxed.gpu.global.add.v2.f32 [%0], {%1, %2};" ::"l"(o + 8 * ld), "f"(c[2]),
               "f"(c[3])
               : "memory");
}
// This lane's 32 h values (16 tagged words from w) as f16 pairs in b, once
// every word carries this call's tag (bounded wait); zeros where !have.
__device__ __forceinline__ void load_h(const StreamParams& p, SkTab& tb, const unsigned long long* w,
                                    bool have, uint32_t tag, uint32_t (&b)[16]) {
  uint64_t t0 = 0;
#pragma unroll 1
  for (int it = 0;; ++it) {
    bool ok = true;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      unsigned long long a = 0ull, c = 0ull;
      if (have)
        asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
                     : "=l"(a), "=l"(c) : "l"(w + 2 * i) : "memory");
      b[2 * i] = (uint32_t)a;
      b[2 * i + 1] = (uint32_t)c;
      ok = ok && (!have || ((uint32_t)(a >> 32) == tag && (uint32_t)(c >> 32) == tag));
    }
    if (__all_sync(0xffffffffu, ok)) return;
    if (it == 0) t0 = global_timer_ns();
    if (*(volatile int*)&tb.abort) return;
    if (global_timer_ns() - t0 > p.timeout_ns) {
      set_error(p, tb, kErrTimeoutStage);
      return;
    }
    __nanosleep(100);
  }
}
// Adds one to a counter word (tag << 32 | count) of this call, restarting it
// at 1 when it holds another call's tag; returns the new count (0 if the CAS
// loop, which only fails when another part got in first, did not finish).
__device__ __forceinline__ uint32_t tagged_count(const StreamParams& p, SkTab& tb,
                                                 unsigned long long* w, uint32_t tag) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(w);
#pragma unroll 1
  for (int it = 0; it < (1 << 16); ++it) {
    const unsigned long long nv =
        (uint32_t)(old >> 32) == tag ? old + 1ull : (((unsigned long long)tag << 32) | 1ull);
    const unsigned long long seen = atomicCAS(w, old, nv);
    if (seen == old) return (uint32_t)nv;
    old = seen;
  }
  set_error(p, tb, kErrTimeoutStage);
  return 0u;
}

// ---------------------------------------------------- one K segment of MMAs
// rg / rg8: 32 E2M1 codes of rows g and g+8 (this lane's piece); b: the B
// fragments of the segment (b[m] = elements 2m, 2m+1 of the lane's piece of
// token column g).  seg_scales gives the f16x2 multipliers of the codes
// (sa* for row g, sb* for row g+8; *0 for piece elements 0-15, *1 for 16-31)
// and the FP32 factors of the segment's partial sums (fa row g, fb row g+8).
// NVFP4: s0 / s8 = the piece's two E4M3 block scales (low byte: elements
// 0-15), E2M1 x E4M3 exact in f16, factors 1.  MXFP4: s0 / s8 = the piece's
// E8M0 byte; the four lanes of a row hold the four 32-element blocks of the
// segment; each is scaled by 2^(its code - the largest of the four) in f16
// and the segment's partial by 2^(largest - 127).
template <int FMT>
__device__ __forceinline__ void seg_scales(uint32_t s0, uint32_t s8, uint32_t& sa0, uint32_t& sa1,
                                           uint32_t& sb0, uint32_t& sb1, float& fa, float& fb) {
  if (FMT == FMT_NVFP4) {
    const uint32_t fg = e4m3x2_to_f16x2(s0), fh = e4m3x2_to_f16x2(s8);
    sa0 = dup_lo(fg);
    sa1 = dup_hi(fg);
    sb0 = dup_lo(fh);
    sb1 = dup_hi(fh);
    fa = fb = 1.f;
  } else {
    int mg = (int)s0, mh = (int)s8;
    mg = max(mg, __shfl_xor_sync(0xffffffffu, mg, 1));
    mh = max(mh, __shfl_xor_sync(0xffffffffu, mh, 1));
    mg = max(mg, __shfl_xor_sync(0xffffffffu, mg, 2));
    mh = max(mh, __shfl_xor_sync(0xffffffffu, mh, 2));
    sa0 = sa1 = pow2_f16x2((int)s0 - mg);
    sb0 = sb1 = pow2_f16x2((int)s8 - mh);
    fa = e8m0_to_f32((uint32_t)mg);
    fb = e8m0_to_f32((uint32_t)mh);
  }
}
// The segment's 8 MMA K steps of one row pair: even steps into c0, odd ones
// into c1 (two accumulator chains; c0 and c1 may be the same array).
template <int FMT>
__device__ __forceinline__ void seg_mma(float (&c0)[4], float (&c1)[4], const uint4& rg,
                                        const uint4& rg8, uint32_t sa0, uint32_t sa1, uint32_t sb0,
                                        uint32_t sb1, const uint32_t (&b)[16]) {
  const uint32_t wg[4] = {rg.x, rg.y, rg.z, rg.w};
  const uint32_t wh[4] = {rg8.x, rg8.y, rg8.z, rg8.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t og[4], oh[4];
    e2m1x8_to_f16x2x4(wg[w], og);
    e2m1x8_to_f16x2x4(wh[w], oh);
    const uint32_t sa = w < 2 ? sa0 : sa1, sb = w < 2 ? sb0 : sb1;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int s = 2 * w + h;
      const uint32_t a[4] = {hmul2(og[2 * h], sa), hmul2(oh[2 * h], sb), hmul2(og[2 * h + 1], sa),
                             hmul2(oh[2 * h + 1], sb)};
      mma_f16(h == 0 ? c0 : c1, a, b[2 * s], b[2 * s + 1]);
    }
  }
}

// BF16 segment (32 K): rg / rg8 = 8 BF16 weights of rows g and g+8, bv = the
// 8 BF16 B elements of the lane's piece of column g.  Two MMA K steps.
__device__ __forceinline__ void seg_bf16(float (&c)[4], const uint4& rg, const uint4& rg8,
                                         const uint4& bv) {
  const uint32_t a0[4] = {rg.x, rg8.x, rg.y, rg8.y};
  const uint32_t a1[4] = {rg.z, rg8.z, rg.w, rg8.w};
  mma_bf16(c, a0, bv.x, bv.y);
  mma_bf16(c, a1, bv.z, bv.w);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ P0 / P1
// Piece idx of the f16 fragment copy of x -> token n and first element k0:
// piece ((seg*4 + i)*N + n)*4 + t holds x[n][128 seg + 32 t + 8 i .. +8].
__device__ __forceinline__ void x_coords(int idx, int N, int& n, int& k0) {
  int r = idx >> 2;
  const int rq = divs(r, N);
  n = r - rq * N;
  k0 = 128 * (rq >> 2) + 32 * (idx & 3) + 8 * (rq & 3);
}

// Copies issued at kernel start (the first DRAM round trip of the call):
// the raw BF16 x into its fragment slots and this CTA's router rows into the
// ring (free until the shared expert or the logits use it).
__device__ void issue_inputs(const StreamParams& p, uint8_t* smem, int c, int G, int nq, int tid) {
  const int H = p.H, N = p.N;
  const int pieces = ((H + 127) >> 7) * 16 * N;
  const uint32_t xs = smem_u32(smem + p.off_x16);
#pragma unroll 1
  for (int idx = tid; idx < pieces; idx += kT) {
    int n, k0;
    x_coords(idx, N, n, k0);
    const bool in = k0 < H;
    cpa16(xs + idx * 16, p.x + (in ? (size_t)n * H + k0 : 0), in ? 16u : 0u);
  }
  const uint32_t rw = smem_u32(smem + p.off_ring);
#pragma unroll 1
  for (int q = 0; q < nq; ++q) {
    const uint16_t* row = p.router + (size_t)(c + G * q) * H;
#pragma unroll 1
    for (int k8 = tid; k8 < (H >> 3); k8 += kT) cpa16(rw + (q * H + 8 * k8) * 2, row + 8 * k8, 16u);
  }
  cpa_commit();
}

// x in fragment order as f16 scaled by 2^-xe[n] (max |x_n| * 2^-xe[n] in
// [2^14, 2^15): every BF16 value down to 2^-10 of the maximum stays exact),
// converted in place; and the shared-expert gate sigmoid(w_s . x_n) (1
// without a gate vector).
__device__ void x_prep(const StreamParams& p, SkTab& tb, uint8_t* smem, int tid) {
  const int H = p.H, N = p.N;
  const int pieces = ((H + 127) >> 7) * 16 * N;
  uint4* xs = reinterpret_cast<uint4*>(smem + p.off_x16);
  const int lane = tid & 31;
  // whole warps per step (every lane runs every step), so the per-token
  // maxima reduce within the warp first: one shared atomic per warp and token
#pragma unroll 1
  for (int base = tid & ~31; base < pieces; base += kT) {
    const int idx = base + lane;
    int n = -1, k0 = 0;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (idx < pieces) {
      x_coords(idx, N, n, k0);
      v = xs[idx];
    }
    const uint32_t xa[4] = {v.x, v.y, v.z, v.w};
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf_lo(xa[j])), fabsf(bf_hi(xa[j]))));
#pragma unroll 1
    for (int t = 0; t < N; ++t) {   // non-negative floats order as integers
      const uint32_t mt = __reduce_max_sync(0xffffffffu, n == t ? __float_as_uint(m) : 0u);
      if (lane == 0 && mt) atomicMax(&tb.xmax[t], mt);
    }
    if (n >= 0 && p.shw && k0 < H) {
      const uint4 wv = ld_nc_u4(p.shw + k0);
      const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
      float d = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        d = fmaf(bf_lo(wa[j]), bf_lo(xa[j]), d);
        d = fmaf(bf_hi(wa[j]), bf_hi(xa[j]), d);
      }
      atomicAdd(&tb.xdot[n], d);
    }
  }
  __syncthreads();
  if (tid < N) {
    const float m = __uint_as_float(tb.xmax[tid]);
    const int e = (m > 0.f && isfinite(m)) ? ilog2f(m) - 14 : 0;
    tb.xe[tid] = e;
    tb.xf[tid] = pow2f(e);
    tb.gsig[tid] = p.shw ? sigmoid_fast(tb.xdot[tid]) : 1.0f;
  }
  __syncthreads();
#pragma unroll 1
  for (int idx = tid; idx < pieces; idx += kT) {
    int n, k0;
    x_coords(idx, N, n, k0);
    const uint4 v = xs[idx];
    const uint32_t xa[4] = {v.x, v.y, v.z, v.w};
    const float sc = pow2f(-tb.xe[n]);
    uint32_t h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2 hv = __floats2half2_rn(bf_lo(xa[j]) * sc, bf_hi(xa[j]) * sc);
      h[j] = *reinterpret_cast<uint32_t*>(&hv);
    }
    xs[idx] = make_uint4(h[0], h[1], h[2], h[3]);
  }
  __syncthreads();
}

// Router logits of this CTA's rows e = c + G q (q < nq) for the N tokens:
// FP32 dot products of the BF16 rows (staged in the ring) with the raw BF16 x
// (in its fragment slots, before x_prep scales it), one warp per (row, token,
// 256-element block) with a fixed-order sum of the blocks; published as
// tagged words (tag << 32 | f32 bits).
__device__ void router_phase(const StreamParams& p, SkTab& tb, uint8_t* smem, int c, int G, int nq,
                             int warp, int lane, int tid) {
  const int H = p.H, N = p.N, E = p.E;
  const int nb = (H + 255) >> 8;
  const uint32_t xs = smem_u32(smem + p.off_x16);
  const uint32_t rw = smem_u32(smem + p.off_ring);
  float* part = reinterpret_cast<float*>(smem + p.off_split);   // [nq * N][nb]
#pragma unroll 1
  for (int w = warp; w < nq * N * nb; w += kW) {
    const int qn = divs(w, nb), b = w - qn * nb;
    const int q = divs(qn, N), n = qn - q * N;
    const int k0 = 256 * b + 8 * lane;
    float a = 0.f;
    if (k0 < H) {
      const uint4 wv = lds128(rw + (q * H + k0) * 2);
      const uint4 xv = lds128(xs + ((((k0 >> 7) * 4 + ((k0 >> 3) & 3)) * N + n) * 4 +
                                    ((k0 >> 5) & 3)) * 16);
      const uint32_t wa[4] = {wv.x, wv.y, wv.z, wv.w};
      const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a = fmaf(bf_lo(wa[j]), bf_lo(xa[j]), a);
        a = fmaf(bf_hi(wa[j]), bf_hi(xa[j]), a);
      }
    }
    a = warp_sum(a);
    if (lane == 0) part[w] = a;
  }
  // published by the last nq * N threads, whose fence at kernel start
  // released this CTA's zeroed accumulator rows
  __syncthreads();
  {
    const int qn = kT - 1 - tid;
    if (qn < nq * N) {
      const int q = divs(qn, N), n = qn - q * N;
    float s = 0.f;
#pragma unroll 1
      for (int b = 0; b < nb; ++b) s += part[qn * nb + b];
      st_relaxed64(p.logits + (size_t)n * E + c + G * q,
                   ((unsigned long long)tb.tag << 32) | __float_as_uint(s));
    }
  }
  __syncthreads();   // x_prep converts the x slots in place afterwards
}

// Poll the call's tagged logits into shared memory (float [N][E]).  The
// reads are acquires: with the barrier after this, every thread's later
// reductions follow the publishing CTAs' release of their zeroed rows.
__device__ void gather_logits(const StreamParams& p, SkTab& tb, float* lg, int tid) {
  const int total = p.N * p.E;
  const uint32_t tag = tb.tag;
  #pragma unroll 1
  for (int w = tid; w < total; w += kT) {
    unsigned long long v = ld_acquire64(p.logits + w);
    if ((uint32_t)(v >> 32) != tag) {
      const uint64_t t0 = global_timer_ns();
      do {
        if (*(volatile int*)&tb.abort) break;
        if (global_timer_ns() - t0 > p.timeout_ns) {
          set_error(p, tb, kErrTimeoutBarrier);
          break;
        }
        __nanosleep(100);
        v = ld_acquire64(p.logits + w);
      } while ((uint32_t)(v >> 32) != tag);
    }
    lg[w] = __uint_as_float((uint32_t)v);
  }
}

// Selection key, order preserving as unsigned: larger key = larger score.
__device__ __forceinline__ uint32_t okey(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// k rounds of warp arg-max over 4 (key, index) pairs per lane (key 0 =
// empty, with index 0xFFFFFFFF); lane j < k returns selection j (key,
// index; index 0xFFFFFFFF if none).  Equal keys go to the lower index.  The
// lane that held a round's winner drops it and rescans its slots (all lanes
// scan before round 0).
__device__ __forceinline__ uint2 select_rounds(uint32_t (&key)[4], const uint32_t (&idx)[4], int k,
                                               int lane) {
  uint2 mine = make_uint2(0u, 0xFFFFFFFFu);
  uint32_t bk = 0u, bi = 0xFFFFFFFFu, we = 0xFFFFFFFFu;
#pragma unroll 1
  for (int j = 0;; ++j) {
    if (bi == we) {
      bk = 0u;
      bi = 0xFFFFFFFFu;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if (idx[s] == we) key[s] = 0u;
        if (key[s] > bk || (key[s] == bk && idx[s] < bi)) {
          bk = key[s];
          bi = idx[s];
        }
      }
    }
    if (j == k) break;
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    we = __reduce_min_sync(0xffffffffu, bk == m ? bi : 0xFFFFFFFFu);
    if (lane == j) mine = make_uint2(m, we);
  }
  return mine;
}

// Top-k routing of the N tokens from the logits in shared memory: softmax
// (selection by logit, weights softmax over all E, optionally renormalised
// over the selected), sigmoid + correction bias (selection by sigmoid(l) +
// bias, weights sigmoid(l), optional renormalisation, times the routed
// scaling factor), or softmax + correction bias (selection by softmax(l) +
// bias, weights softmax(l), likewise).  Ties go to the lower expert index
// (forward_k3.rs, the batched top-k step).
//
// Level 0: a warp owns 128 experts of one token (4 keys per lane) and selects
// their top k.  Level 1 (more than 128 experts): a warp selects the final k
// of one token from its W local lists (W*k <= 128 candidates).  Both levels
// read (key, expert) pairs from shared memory: `pairs` [N][E] for level 0,
// `cand` [N][W*k] for level 1.
// Selection key of logit v (expert e) given the token's softmax max / sum.
__device__ __forceinline__ uint32_t sel_key(const StreamParams& p, const SkTab& tb, float v, int e,
                                            float gm, float gd) {
  float sc = v;
  if (p.scoring == 1) sc = sigmoid_fast(v) + tb.bias[e];
  if (p.scoring == 2) sc = exp_fast(v - gm) * rcp_fast(gd) + tb.bias[e];
  return okey(sc);
}
// Routing weights of token n's selections (lane j < k holds selection j,
// expert e), stored with the experts.
__device__ __forceinline__ void sel_weights(const StreamParams& p, SkTab& tb, const float* lg, int n,
                                            int e, float gm, float gd, int lane) {
  const int k = p.k;
  float w = 0.f;
  if (lane < k) {
    const float v = lg[n * p.E + e];
    w = p.scoring != 1 ? exp_fast(v - gm) * rcp_fast(gd) : sigmoid_fast(v);
  }
  const float ws = warp_sum(w);
  if (lane < k) {
    if (p.norm) w *= rcp_fast(ws);
    if (p.scoring != 0) w *= p.rsf;
    tb.sel_e[n * k + lane] = (int16_t)e;
    tb.sel_w[n * k + lane] = w;
  }
}

__device__ void routing(const StreamParams& p, SkTab& tb, const float* lg, uint2* pairs,
                        uint2* cand, int warp, int lane) {
  const int E = p.E, N = p.N, k = p.k;
  const int W = (E + 127) >> 7;   // warps per token
  if (W == 1) {
    // at most 128 experts: one warp per token, keys in registers
    if (warp < N) {
      const int n = warp;
      const int scoring = p.scoring;
      float v[4], m = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? lg[n * E + e] : -INFINITY;
        m = fmaxf(m, v[i]);
      }
      // the softmax statistics over all E: needed by softmax + bias keys and
      // by softmax weights left unnormalised; softmax weights renormalised
      // over the selection only need a common reference (the top logit)
      const bool stats = scoring == 2 || (scoring == 0 && !p.norm);
      float d = 1.f;
      if (stats) {
        m = warp_max(m);
        d = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) d += exp_fast(v[i] - m);   // exp(-inf) = 0
        d = warp_sum(d);
      }
      uint32_t key[4], idx[4];
      if (scoring == 0) {   // selection by the logit itself
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = lane + 32 * i;
          idx[i] = e < E ? (uint32_t)e : 0xFFFFFFFFu;
          key[i] = e < E ? okey(v[i]) : 0u;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = lane + 32 * i;
          idx[i] = e < E ? (uint32_t)e : 0xFFFFFFFFu;
          key[i] = e < E ? sel_key(p, tb, v[i], e, m, d) : 0u;
        }
      }
      const uint2 sel = select_rounds(key, idx, k, lane);
      const int es = sel.y < (uint32_t)E ? (int)sel.y : 0;
      if (!stats) m = lg[n * E + __shfl_sync(0xffffffffu, es, 0)];
      sel_weights(p, tb, lg, n, es, m, d, lane);
    }
    return;
  }
  // softmax statistics of each token's 128-expert parts
#pragma unroll 1
  for (int task = warp; task < N * W; task += kW) {
    const int n = divs(task, W), w = task - n * W;
    float v[4], m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 128 * w + lane + 32 * i;
      v[i] = e < E ? lg[n * E + e] : -INFINITY;
      m = fmaxf(m, v[i]);
    }
    m = warp_max(m);
    float d = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) d += exp_fast(v[i] - m);   // exp(-inf) = 0
    d = warp_sum(d);
    if (lane == 0) {
      tb.part[n][w][0] = m;
      tb.part[n][w][1] = d;
    }
  }
  __syncthreads();
  if (warp < N && lane == 0) {
    float gm = -INFINITY, gd = 0.f;
#pragma unroll 1
    for (int q = 0; q < W; ++q) gm = fmaxf(gm, tb.part[warp][q][0]);
#pragma unroll 1
    for (int q = 0; q < W; ++q) gd += tb.part[warp][q][1] * exp_fast(tb.part[warp][q][0] - gm);
    tb.gmax[warp] = gm;
    tb.gden[warp] = gd;
  }
  __syncthreads();
  // selection keys of all N x E scores
#pragma unroll 1
  for (int w = threadIdx.x; w < N * E; w += kT) {
    const int n = divs(w, E), e = w - n * E;
    pairs[w] = make_uint2(sel_key(p, tb, lg[w], e, tb.gmax[n], tb.gden[n]), (uint32_t)e);
  }
  __syncthreads();
#pragma unroll 1
  for (int level = 0; level < (W > 1 ? 2 : 1); ++level) {
    const int ntask = level == 0 ? N * W : N;
    const int M = W * k;
#pragma unroll 1
    for (int task = warp; task < ntask; task += kW) {
      // this task's candidates
      const uint2* src;
      int cnt;
      if (level == 0) {
        const int n = divs(task, W), w = task - n * W;
        src = pairs + n * E + 128 * w;
        cnt = min(128, E - 128 * w);
      } else {
        src = cand + task * M;
        cnt = M;
      }
      uint32_t key[4], idx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ci = lane + 32 * i;
        const uint2 cv = ci < cnt ? src[ci] : make_uint2(0u, 0xFFFFFFFFu);
        key[i] = cv.x;
        idx[i] = cv.y;
      }
      const uint2 sel = select_rounds(key, idx, k, lane);
      if (lane < k) {
        if (level == 0 && W > 1)
          cand[task * k + lane] = sel;
        else
          tb.sel_e[task * k + lane] = (int16_t)(sel.y < (uint32_t)E ? sel.y : 0u);
      }
    }
    __syncthreads();
  }
  // weights of the selected experts
  if (warp < N)
    sel_weights(p, tb, lg, warp, lane < k ? tb.sel_e[warp * k + lane] : 0, tb.gmax[warp],
                tb.gden[warp], lane);
}

// Unique experts of the N*k selections (first-selection order), with the
// token mask, routing weight and h slot of every (expert, token) pair.
__device__ void build_tables(const StreamParams& p, SkTab& tb, int lane) {
  const int S = p.N * p.k, k = p.k;
  if (S <= 32) {
    // one selection per lane: the lanes that hold the same expert, the lowest
    // of them (its first selection) stands for the unit, and units are
    // numbered in first-selection order; no shared-memory atomics
    const bool v = lane < S;
    const int e = v ? (int)tb.sel_e[lane] : -1 - lane;   // idle lanes: keys of their own
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const uint32_t below = (1u << lane) - 1u;
    const bool lead = v && (same & below) == 0u;
    const uint32_t leads = __ballot_sync(0xffffffffu, lead);
    const int first = __ffs(same) - 1;
    const int u = __popc(leads & ((1u << first) - 1u));
    if (v) {
      const int n = divs(lane, k);
      tb.u_w[u][n] = tb.sel_w[lane];
      tb.u_slot[u][n] = (int16_t)lane;
      if (lead) {
        // token n holds this expert if one of its k slots n*k .. n*k+k-1 does
        // (n*k < 32 for every n < N since N*k <= 32)
        const uint32_t km = k >= 32 ? 0xFFFFFFFFu : (1u << k) - 1u;
        uint32_t tm = 0u;
#pragma unroll 1
        for (int t = 0; t < p.N; ++t)
          if ((same >> (t * k)) & km) tm |= 1u << t;
        tb.u_e[u] = (int16_t)e;
        tb.u_mask[u] = tm;
      }
    }
    if (lane == 0) tb.U = __popc(leads);
    return;
  }
  #pragma unroll 1
  for (int s = lane; s < S; s += 32) atomicMin(&tb.first[tb.sel_e[s]], (uint32_t)s);
  __syncwarp();
  const uint32_t lt = (1u << lane) - 1u;
  int U = 0;
  #pragma unroll 1
  for (int b = 0; b < S; b += 32) {
    const int s = b + lane;
    const int e = s < S ? tb.sel_e[s] : 0;
    const bool isfirst = s < S && tb.first[e] == (uint32_t)s;
    const uint32_t mask = __ballot_sync(0xffffffffu, isfirst);
    __syncwarp();
    if (isfirst) {
      const int u = U + __popc(mask & lt);
      tb.u_e[u] = (int16_t)e;
      tb.u_mask[u] = 0u;
      tb.first[e] = 0x80000000u | (uint32_t)u;
    }
    U += __popc(mask);
    __syncwarp();
  }
  #pragma unroll 1
  for (int s = lane; s < S; s += 32) {
    const int u = (int)(tb.first[tb.sel_e[s]] & 0x7FFFFFFFu);
    const int n = divs(s, k);
    atomicOr(&tb.u_mask[u], 1u << n);
    tb.u_w[u][n] = tb.sel_w[s];
    tb.u_slot[u][n] = (int16_t)s;
  }
  if (lane == 0) tb.U = U;
}

// ------------------------------------------------- PS shared-expert gate/up
// Ring layout of one warp: stage s holds 4 pieces; piece k of lane l sits at
// ring + (s*4 + k)*512 + l*16 (conflict-free 16-byte accesses), its side slot
// at aux + s*512 + l*16.
__device__ __forceinline__ uint32_t piece(uint32_t ring, int slot, int k) {
  return ring + (uint32_t)((slot * 4 + k) * 512);
}

// This CTA's unit (if any): 16-row tile j of the shared gate/up, K part q of
// sh_parts, split over the 16 warps as 32-column segment items (gate rows g,
// g+8 and up rows g, g+8 in one stage, with this lane's BF16 x piece).
template <int D>
__device__ void shared_gate_up(const StreamParams& p, SkTab& tb, uint8_t* smem, int c, int G,
                               int warp, int lane) {
  const int Ts = p.Is >> 4, parts = p.sh_parts;
  const int v = G - 1 - c;
  if (v < 0 || v >= Ts * parts) return;
  const int g = lane >> 2, t = lane & 3;
  const int j = divs(v, parts), q = v - j * parts;
  const int Sb = p.H >> 5;
  const int sa = divs(q * Sb, parts), sb = divs((q + 1) * Sb, parts);
  const int h0 = sa + warp * (sb - sa) / kW, h1 = sa + (warp + 1) * (sb - sa) / kW;
  const uint32_t ring = smem_u32(smem + p.off_ring) + (uint32_t)(warp * D * kSkStageCodes + lane * 16);
  const uint32_t aux = smem_u32(smem + p.off_aux) + (uint32_t)(warp * D * kSkStageAux + lane * 16);
  const int rb = 2 * p.H;   // bytes per row
  const uint8_t* g0 = reinterpret_cast<const uint8_t*>(p.shg) + (size_t)(16 * j + g) * rb + 16 * t;
  const uint8_t* u0 = reinterpret_cast<const uint8_t*>(p.shu) + (size_t)(16 * j + g) * rb + 16 * t;
  const bool vx = g < p.N;
  const uint8_t* x0 = reinterpret_cast<const uint8_t*>(p.x) + (vx ? (size_t)g * rb + 16 * t : 0);
  float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
  int islot = 0, cslot = 0;
  const int n = h1 - h0;
#pragma unroll 1
  for (int it = 0; it < n + D - 1; ++it) {
    if (it < n) {
      const int o = 64 * (h0 + it);
      cpa16w(piece(ring, islot, 0), g0 + o, 16u);
      cpa16w(piece(ring, islot, 1), g0 + o + 8 * rb, 16u);
      cpa16w(piece(ring, islot, 2), u0 + o, 16u);
      cpa16w(piece(ring, islot, 3), u0 + o + 8 * rb, 16u);
      cpa16(aux + islot * 512, x0 + (vx ? o : 0), vx ? 16u : 0u);
      islot = islot + 1 == D ? 0 : islot + 1;
    }
    cpa_commit();
    if (it < D - 1) continue;
    asm volatile("cp.async.wait_group %0;" ::"n"(D - 1) : "memory");
    const uint4 bv = lds128(aux + cslot * 512);
    seg_bf16(ag, lds128(piece(ring, cslot, 0)), lds128(piece(ring, cslot, 1)), bv);
    seg_bf16(au, lds128(piece(ring, cslot, 2)), lds128(piece(ring, cslot, 3)), bv);
    cslot = cslot + 1 == D ? 0 : cslot + 1;
  }
  cpa_wait_all();
  // the 16 warps' partial tiles meet in split slot 0
  float* acc = reinterpret_cast<float*>(smem + p.off_split) + lane * 8;
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    atomicAdd(acc + qq, ag[qq]);
    atomicAdd(acc + 4 + qq, au[qq]);
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      ag[qq] = acc[qq];
      au[qq] = acc[4 + qq];
    }
    bool fin = parts == 1;
    if (!fin) {
      // the K parts of this tile (one per CTA) leave their partial sums in
      // their own slots; the part that counts last adds them in part order
      float* mine = p.shpart + ((size_t)j * parts + q) * 256 + lane * 8;
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        __stcg(mine + qq, ag[qq]);
        __stcg(mine + 4 + qq, au[qq]);
      }
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        fence_gpu();   // no weight copies are in flight here
        last = tagged_count(p, tb, p.scnt + j, tb.tag) == (uint32_t)parts;
      }
      fin = __shfl_sync(0xffffffffu, last, 0) != 0;
      if (fin) {
        fence_gpu();
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) ag[qq] = au[qq] = 0.f;
#pragma unroll 1
        for (int pq = 0; pq < parts; ++pq) {
          const float* o = p.shpart + ((size_t)j * parts + pq) * 256 + lane * 8;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            ag[qq] += __ldcg(o + qq);
            au[qq] += __ldcg(o + 4 + qq);
          }
        }
      }
    }
    if (fin) {
      __nv_bfloat16* hs = reinterpret_cast<__nv_bfloat16*>(p.hs);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const int nn = 2 * t + (qq & 1), r = g + 8 * (qq >> 1);
        if (nn < p.N)
          hs[(size_t)nn * p.Is + 16 * j + r] =
              __float2bfloat16_rn(silu(ag[qq]) * au[qq] * tb.gsig[nn]);
      }
      __syncwarp();
      if (lane == 0) {
        fence_gpu();
        st_flag(p.sflag + j, tb.tag);
      }
    }
  }
  __syncthreads();
  // split slot 0 is reused by the routed tiles
  if (warp == 0) {
#pragma unroll
    for (int qq = 0; qq < 8; ++qq) acc[qq] = 0.f;
  }
}

// ------------------------------------------------ P2 + P3 item pipeline
// Items of one warp: its share of this CTA's routed gate/up items (tile,
// 128-column segment: gate rows g, g+8 and up rows g, g+8), then its share of
// the grid's down items (shared-expert (segment, row tile) items first, then
// routed (expert, segment, 32-row tile) items; rows g + 8 i of the tile).  The down
// list is split over all warps of the grid in order, so a warp's items mostly
// share one (expert, segment) and its B operand; their partial sums go to the
// FP32 output accumulator in global memory.  One loop; the first down items
// are copied while the last gate/up items compute.
struct Pipe {
  int c, G, g, t, lane;
  uint32_t ring, aux;
  int S, tpe, a0, a1;                    // gate/up: segments per row, tiles per expert, items
  int Sd, Sds, MT, nsh, b0, b1;          // down: segments, shared segments, row tiles, entries
  int sst, spar, sdp;                    // down segment step (1, or 2 when paired), parity, Sd / sst
};

// Down item cursor: shared-expert items (u < 0) over (segment, row tile),
// then routed items over (expert, segment, row tile).  Paired order (sst =
// 2): the list runs over segment pairs, and the two warps of a pair take
// segments 2p and 2p + 1 of the same entries (spar = the warp's parity), so
// the two 64-byte halves of each 128-byte row piece are read together.
struct DCur {
  int u, seg, m;
};
template <bool SH>
__device__ __forceinline__ void dcur_init(const Pipe& P, int b, DCur& d) {
  if (SH && b < P.nsh) {
    d.u = -1;
    const int sp = divs(b, P.MT);
    d.m = b - sp * P.MT;
    d.seg = sp * P.sst + P.spar;
  } else {
    const int unit = divs(b - P.nsh, P.MT);
    d.m = (b - P.nsh) - unit * P.MT;
    d.u = divs(unit, P.sdp);
    d.seg = (unit - d.u * P.sdp) * P.sst + P.spar;
  }
}
template <bool SH>
__device__ __forceinline__ void dcur_next(const Pipe& P, DCur& d) {
  if (++d.m == P.MT) {
    d.m = 0;
    d.seg += P.sst;
    if (SH && d.u < 0) {
      if (d.seg >= P.Sds) {
        d.seg = P.spar;
        d.u = 0;
      }
    } else if (d.seg >= P.Sd) {
      d.seg = P.spar;
      ++d.u;
    }
  }
}

template <int D>
__device__ __forceinline__ void cpa_wait_d() {
  asm volatile("cp.async.wait_group %0;" ::"n"(D - 1) : "memory");
}

// Copy state of the gate/up items: this lane's pointers into the current
// tile (gate and up rows g; row g+8 is 8 * rb further), advanced by one
// segment per item.
struct GuIssue {
  const uint8_t *sg, *su;   // this lane's scale words (row g)
  int row0;                 // first row of the tile in the [E * inter] code tensors
  int seg, tl;
};
template <int FMT>
__device__ __forceinline__ void gu_issue_tile(const StreamParams& p, const SkTab& tb, const Pipe& P,
                                              GuIssue& s) {
  constexpr int gsz = FMT == FMT_NVFP4 ? 16 : 32;
  const int i = P.c + P.G * s.tl;
  const int u = divs(i, P.tpe), j = i - u * P.tpe;
  s.row0 = tb.u_e[u] * p.inter + 16 * j;
  const size_t row = (size_t)s.row0 + P.g;
  const size_t so = row * (p.H / gsz) + (FMT == FMT_NVFP4 ? 2 * P.t : P.t);
  s.sg = p.gsc + (so & ~(size_t)3);
  s.su = p.usc + (so & ~(size_t)3);
}

// Copies of down item d (cursor), this lane's rows g and g+8.  Scale tensors
// hold rows * K / gs bytes with rows a multiple of 32, so a 4-byte word never
// reaches past the end.
template <int FMT, bool SH>
__device__ __forceinline__ void dn_issue(const StreamParams& p, SkTab& tb, const Pipe& P,
                                         const DCur& d, uint8_t* dst, uint64_t* bar, uint32_t da,
                                         uint8_t* daux, bool& sh_waited) {
  constexpr int gsz = FMT == FMT_NVFP4 ? 16 : 32;
  const int rr = 32 * d.m + P.g;   // rows rr + 8 i, i < 4 (H is a multiple of 32)
  const int o = 64 * d.seg + 16 * P.t;
  if (SH && d.u < 0) {
    // shared-expert down: BF16 rows [H, Is] and this lane's piece of h_s,
    // copied only once every shared tile of the call is published
    if (!sh_waited) {
      const int Ts = p.Is >> 4;
#pragma unroll 1
      for (int bb = 0; bb < Ts; bb += 32)
        wait_tags(p, tb, p.sflag + bb, min(32, Ts - bb), tb.tag, P.lane);
      sh_waited = true;
    }
    const int rb = 2 * p.Is;
    if (P.lane == 0) {
      mbar_arrive_expect_tx(bar, 2048u);
      tma_load_2d(dst, &p.tm_shd, 64 * d.seg, 32 * d.m, bar);
    }
    const bool vx = P.g < p.N;
    cpa16(da, reinterpret_cast<const uint8_t*>(p.hs) + (vx ? (size_t)P.g * rb + o : 0),
          vx ? 16u : 0u);
  } else {
    const int rb = p.inter / 2, scb = p.inter / gsz;
    const size_t row = (size_t)tb.u_e[d.u] * p.H + rr;
    const bool kin = o < rb;
    if (P.lane == 0) {
      const int y = tb.u_e[d.u] * p.H + 32 * d.m;
      mbar_arrive_expect_tx(bar, p.sc_tma ? 2560u : 2048u);
      tma_load_2d(dst, &p.tm_dq, 64 * d.seg, y, bar);
      if (p.sc_tma)   // the 16-byte scale column holding this segment's, 32 rows
        tma_load_2d(daux, &p.tm_ds, ((FMT == FMT_NVFP4 ? 8 : 4) * d.seg) & ~15, y, bar);
    }
    if (!p.sc_tma) {
      const size_t so = row * scb + (FMT == FMT_NVFP4 ? 8 : 4) * d.seg + (FMT == FMT_NVFP4 ? 2 * P.t : P.t);
      const uint8_t* s0 = p.dsc + (so & ~(size_t)3);
#pragma unroll
      for (int i = 0; i < 4; ++i) cpa4w(da + 4 * i, kin ? s0 + 8 * i * scb : p.dsc, kin ? 4u : 0u);
    }
  }
}

// Byte offset of lane t's scale word for K segment seg within a 16-byte row
// of a scale box (NVFP4: 8 bytes per segment, two per box row, the lane's
// two scales at byte 2t; MXFP4: 4 bytes per segment, four per row, its scale
// at byte t); the shift inside the word is the one of the per-lane copies.
template <int FMT>
__device__ __forceinline__ int scw_t(int seg, int t) {
  return FMT == FMT_NVFP4 ? ((seg & 1) * 8 + 2 * t) & ~3 : (seg & 3) * 4;
}

template <int FMT, int D, bool SH>
__device__ void pipeline(const StreamParams& p, SkTab& tb, uint8_t* smem, const Pipe& P) {
  constexpr int gsz = FMT == FMT_NVFP4 ? 16 : 32;
  constexpr int sstep = FMT == FMT_NVFP4 ? 8 : 4;   // scale bytes per 128-column segment
  const int ngu = P.a1 - P.a0, ndn = P.b1 - P.b0;
  const int total = ngu + ndn;
  const int g = P.g, t = P.t, lane = P.lane;
  const int rb = p.H / 2;
  const int s8 = 8 * (p.H / gsz);   // scale bytes of 8 rows
  const uint32_t xs = smem_u32(smem + p.off_x16) + (uint32_t)((g * 4 + t) * 16);
  const int xstride = p.N * 64;   // bytes between the x pieces i of one segment
  const bool xlane = g < p.N;
  float* split = reinterpret_cast<float*>(smem + p.off_split);
  const uint32_t tag = tb.tag;
  const bool olane = 2 * t < p.N;   // this lane's output columns 2t, 2t+1 hold tokens
  const int old = (p.N + 1) & ~1;   // row stride of the output accumulator
  const int soff_t = FMT == FMT_NVFP4 ? 2 * t : t;
  auto scw = [](int seg, int tt) { return scw_t<FMT>(seg, tt); };

  // ---- copy-side cursors; the code rows of a stage come by TMA (lane 0),
  // their scale words by per-lane cp.async
  const int warp = threadIdx.x >> 5;
  uint8_t* wring = smem + p.off_ring + warp * D * kSkStageCodes;
  uint8_t* daux = smem + p.off_aux + warp * D * kSkStageAux;   // this warp's side slots
  const uint32_t auxw = smem_u32(daux);
  uint64_t* full = tb.full[warp];
  int islot = 0;
  GuIssue gi;
  gi.tl = divs(P.a0, P.S);
  gi.seg = P.a0 - gi.tl * P.S;
  if (ngu) gu_issue_tile<FMT>(p, tb, P, gi);
  DCur di;
  dcur_init<SH>(P, P.b0, di);
  int dleft = ndn;   // down items not yet copied
  bool sh_waited = false;
  auto issue_next = [&](int k) {   // k-th item of this warp's sequence
    const uint32_t da = P.aux + (uint32_t)(islot * 512);
    uint8_t* dst = wring + islot * 2048;
    if (k < total) {
      // the stage was last read (generic proxy) by the item consumed just
      // before; order those reads before the TMA's writes
      __syncwarp();
      if (lane == 0) fence_proxy_async_smem();
    }
    if (k < ngu) {
      const int o = 64 * gi.seg;
      const bool kin = o + 16 * t < rb;
      if (lane == 0) {
        mbar_arrive_expect_tx(full + islot, p.sc_tma ? 2560u : 2048u);
        tma_load_2d(dst, &p.tm_gq, o, gi.row0, full + islot);
        tma_load_2d(dst + 1024, &p.tm_uq, o, gi.row0, full + islot);
        if (p.sc_tma) {   // the 16-byte scale column holding this segment's, 16 rows
          const int sx = (sstep * gi.seg) & ~15;
          tma_load_2d(daux + islot * 512, &p.tm_gs, sx, gi.row0, full + islot);
          tma_load_2d(daux + islot * 512 + 256, &p.tm_us, sx, gi.row0, full + islot);
        }
      }
      if (!p.sc_tma) {
        const int so = kin ? sstep * gi.seg : 0;
        const uint32_t n4 = kin ? 4u : 0u;
        cpa4w(da, gi.sg + so, n4);
        cpa4w(da + 4, gi.sg + so + s8, n4);
        cpa4w(da + 8, gi.su + so, n4);
        cpa4w(da + 12, gi.su + so + s8, n4);
      }
      if (++gi.seg == P.S) {
        gi.seg = 0;
        ++gi.tl;
        if (k + 1 < ngu) gu_issue_tile<FMT>(p, tb, P, gi);
      }
    } else if (dleft > 0) {
      dn_issue<FMT, SH>(p, tb, P, di, dst, full + islot, da, daux + islot * 512, sh_waited);
      dcur_next<SH>(P, di);
      --dleft;
    }
    islot = islot + 1 == D ? 0 : islot + 1;
  };
  int cslot = 0;
  // item h's stage: its TMA bytes (phase h / D of the stage's mbarrier) and
  // its scale copies (cp.async group)
  auto wait_stage = [&](int h) {
    if (!mbar_wait_bounded(full + cslot, (uint32_t)(h / D) & 1u, p.timeout_ns) && lane == 0)
      set_error(p, tb, kErrTimeoutStage);
    cpa_wait_d<D>();
  };
  // gate/up consume state
  int ctl = divs(P.a0, P.S), cseg = P.a0 - ctl * P.S;
  int cur_tile = -1, done = 0, u = 0, j = 0, csh = 0, useg = 0;
  float ag[4] = {0.f, 0.f, 0.f, 0.f}, au[4] = {0.f, 0.f, 0.f, 0.f};
  float s2g = 1.f, s2u = 1.f, s2d = 1.f;
  // down consume state
  DCur cd;
  dcur_init<SH>(P, P.b0, cd);
  int du = -2, dseg = -1, dsh = 0;
  uint32_t b[16];
  // one loop over this warp's items (gate/up, then down) with the copies of
  // item h + D - 1 issued at step h; steps before 0 only fill the ring
#pragma unroll 1
  for (int h = 1 - D; h <= total; ++h) {
    if (cur_tile >= 0 && (h >= ngu || ctl != cur_tile)) {
      // ---- tile done: the only place a gate/up tile ends
      const int first = cur_tile * P.S;
      bool epi = first >= P.a0 && first + P.S <= P.a1;
      if (!epi) {
        int slot = cur_tile;
        const int Tc = divs(tb.U * P.tpe - 1 - P.c, P.G) + 1;
        if (Tc > kSkSplitSlots) {
          // the warp boundary that cuts this tile (at most one does)
          const int tot = Tc * P.S;
          int wf = 0;
#pragma unroll 1
          for (int bb = 1; bb < kW; ++bb)
            if (bb * tot / kW <= first) wf = bb;
          slot = wf + 1;
        }
        float* acc = split + slot * 256 + lane * 8;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          atomicAdd(acc + qq, ag[qq]);
          atomicAdd(acc + 4 + qq, au[qq]);
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          __threadfence_block();
          last = atomicAdd(&tb.split_cnt[slot], (uint32_t)done) + done == (uint32_t)P.S;
        }
        epi = __shfl_sync(0xffffffffu, last, 0) != 0;
        if (epi) {
          __threadfence_block();
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            ag[qq] = *(volatile float*)(acc + qq);
            au[qq] = *(volatile float*)(acc + 4 + qq);
          }
        }
      }
      if (epi) {
        // h of rows r, r+1 (lanes g, g+1) of token n in one tagged word,
        // written by the even-g lane: no fence and no flag, the word
        // carries its own readiness
        const uint32_t mask = tb.u_mask[u];
        bool over = false;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int n = 2 * t + (qq & 1), r = g + 8 * (qq >> 1);
          const bool routed = n < p.N && ((mask >> n) & 1u);
          float hv = 0.f;
          if (routed) {
            const float xf = tb.xf[n];
            hv = silu(ag[qq] * s2g * xf) * (au[qq] * s2u * xf) * tb.u_w[u][n] * s2d;
          }
          if (fabsf(hv) > 65504.f) {   // saturate (NaN passes through) and report
            over = true;
            hv = copysignf(65504.f, hv);
          }
          const uint32_t lo = __half_as_ushort(__float2half_rn(hv));
          const uint32_t hi = __shfl_down_sync(0xffffffffu, lo, 4);
          if (!(g & 1) && routed)
            st_tagged(p.hw + (((size_t)tb.u_slot[u][n] * p.inter + 16 * j + r) >> 1),
                      lo | (hi << 16), tag);
        }
        if (__any_sync(0xffffffffu, over) && lane == 0) atomicOr(&p.ctrl->error, kErrRange);
      }
      cur_tile = -1;
    }
    if (h == total) break;
    issue_next(h + D - 1);
    cpa_commit();
    if (h < 0) continue;
    if (h < ngu) {
      if (ctl != cur_tile) {
        cur_tile = ctl;
        const int i = P.c + P.G * ctl;
        u = divs(i, P.tpe);
        j = i - u * P.tpe;
        const int e = tb.u_e[u];
        const size_t row = (size_t)e * p.inter + 16 * j + g;
        csh = 8 * (int)((row * (p.H / gsz) + soff_t) & 3u);
        s2g = tb.s2[e][0];
        s2u = tb.s2[e][1];
        s2d = tb.s2[e][2];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) ag[qq] = au[qq] = 0.f;
        done = 0;
      }
      // B = this lane's f16 x piece of the segment (column g)
      const uint32_t xa = xs + (uint32_t)(cseg * 4 * xstride);
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (xlane) v = lds128(xa + (uint32_t)(ii * xstride));
        b[4 * ii] = v.x;
        b[4 * ii + 1] = v.y;
        b[4 * ii + 2] = v.z;
        b[4 * ii + 3] = v.w;
      }
      useg = cseg;
      ++done;
      if (++cseg == P.S) {
        cseg = 0;
        ++ctl;
      }
    } else if (SH && cd.u < 0) {
      // shared-expert down item (BF16 rows, B copied with them)
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t sc = P.ring + (uint32_t)(cslot * 2048);
      wait_stage(h);
      const uint4 bv = lds128(P.aux + (uint32_t)(cslot * 512));
      seg_bf16(c0, lds128(sc), lds128(sc + 512), bv);
      seg_bf16(c1, lds128(sc + 1024), lds128(sc + 1536), bv);
      if (olane) {
        red_out(p.oacc + (32 * cd.m + g) * old + 2 * t, old, c0);
        red_out(p.oacc + (32 * cd.m + 16 + g) * old + 2 * t, old, c1);
      }
      dcur_next<SH>(P, cd);
      cslot = cslot + 1 == D ? 0 : cslot + 1;
      continue;
    } else if (cd.u != du || cd.seg != dseg) {
      // routed down item of a new (unit, segment): B = this lane's f16 h
      // piece of column g (waits for the eight gate/up tiles it reads)
      if (cd.u != du) {
        // byte position of the scales in their word: the same for rows
        // 32 m + g + 8 i of every row tile m (8 x the scale bytes per row is
        // a multiple of 4)
        const size_t row = (size_t)tb.u_e[cd.u] * p.H + g;
        dsh = 8 * (int)((row * (p.inter / gsz) + soff_t) & 3u);
      }
      du = cd.u;
      dseg = cd.seg;
      const int kk = 128 * cd.seg + 32 * t;
      const bool have = xlane && ((tb.u_mask[cd.u] >> g) & 1u) && kk < p.inter;
      load_h(p, tb, p.hw + (have ? ((size_t)tb.u_slot[cd.u][g] * p.inter + kk) >> 1 : 0), have,
             tag, b);
    }
    // the item's FP4 rows: gate and up (two row pairs) or down (one)
    wait_stage(h);
    {
      const uint32_t m16 = FMT == FMT_NVFP4 ? 0xFFFFu : 0xFFu;
      const uint32_t sc = P.ring + (uint32_t)(cslot * 2048), sa = P.aux + (uint32_t)(cslot * 512);
      uint32_t a0, a1, b0, b1;
      float fa, fb;
      if (h < ngu) {
        // gate and up: two independent MMA chains
        uint4 av;
        if (p.sc_tma) {
          // box rows of 16 bytes: gate rows at 0, up rows at 256
          const uint32_t wb = auxw + (uint32_t)(cslot * 512 + g * 16 + scw(useg, t));
          av = make_uint4(lds32(wb), lds32(wb + 128), lds32(wb + 256), lds32(wb + 384));
        } else {
          av = lds128(sa);
        }
        const uint4 g0 = lds128(sc), g8 = lds128(sc + 512);
        const uint4 u0 = lds128(sc + 1024), u8 = lds128(sc + 1536);
        if (FMT == FMT_NVFP4) {
          seg_scales<FMT>((av.x >> csh) & m16, (av.y >> csh) & m16, a0, a1, b0, b1, fa, fb);
          seg_mma<FMT>(ag, ag, g0, g8, a0, a1, b0, b1, b);
          seg_scales<FMT>((av.z >> csh) & m16, (av.w >> csh) & m16, a0, a1, b0, b1, fa, fb);
          seg_mma<FMT>(au, au, u0, u8, a0, a1, b0, b1, b);
        } else {
          float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
          float ga, gb;
          seg_scales<FMT>((av.x >> csh) & m16, (av.y >> csh) & m16, a0, a1, b0, b1, ga, gb);
          seg_mma<FMT>(cg, cg, g0, g8, a0, a1, b0, b1, b);
          seg_scales<FMT>((av.z >> csh) & m16, (av.w >> csh) & m16, a0, a1, b0, b1, fa, fb);
          seg_mma<FMT>(cu, cu, u0, u8, a0, a1, b0, b1, b);
          ag[0] = fmaf(cg[0], ga, ag[0]);
          ag[1] = fmaf(cg[1], ga, ag[1]);
          ag[2] = fmaf(cg[2], gb, ag[2]);
          ag[3] = fmaf(cg[3], gb, ag[3]);
          au[0] = fmaf(cu[0], fa, au[0]);
          au[1] = fmaf(cu[1], fa, au[1]);
          au[2] = fmaf(cu[2], fb, au[2]);
          au[3] = fmaf(cu[3], fb, au[3]);
        }
      } else {
        // down: two row pairs (rows 32m + g + 8i, i < 4), two MMA chains;
        // the partial sums (columns 2t, 2t+1) go to the output accumulator
        uint4 sw;
        if (p.sc_tma) {   // box rows of 16 bytes: rows g, g + 8, g + 16, g + 24
          const uint32_t wb = auxw + (uint32_t)(cslot * 512 + g * 16 + scw(cd.seg, t));
          sw = make_uint4(lds32(wb), lds32(wb + 128), lds32(wb + 256), lds32(wb + 384));
        } else {
          sw = lds128(sa);
        }
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        float fc, fd;
        seg_scales<FMT>((sw.x >> dsh) & m16, (sw.y >> dsh) & m16, a0, a1, b0, b1, fa, fb);
        seg_mma<FMT>(c0, c0, lds128(sc), lds128(sc + 512), a0, a1, b0, b1, b);
        seg_scales<FMT>((sw.z >> dsh) & m16, (sw.w >> dsh) & m16, a0, a1, b0, b1, fc, fd);
        seg_mma<FMT>(c1, c1, lds128(sc + 1024), lds128(sc + 1536), a0, a1, b0, b1, b);
        if (FMT != FMT_NVFP4) {
          c0[0] *= fa;
          c0[1] *= fa;
          c0[2] *= fb;
          c0[3] *= fb;
          c1[0] *= fc;
          c1[1] *= fc;
          c1[2] *= fd;
          c1[3] *= fd;
        }
        if (olane) {
          red_out(p.oacc + (32 * cd.m + g) * old + 2 * t, old, c0);
          red_out(p.oacc + (32 * cd.m + 16 + g) * old + 2 * t, old, c1);
        }
        dcur_next<SH>(P, cd);
      }
    }
    cslot = cslot + 1 == D ? 0 : cslot + 1;
  }
  cpa_wait_all();
}

// ------------------------------------------------------------------ kernel
template <int FMT, int D, bool SH>
__global__ void __launch_bounds__(kSkThreads, 1) moe_stream_kernel(const __grid_constant__ StreamParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  SkTab& tb = *reinterpret_cast<SkTab*>(smem + p.off_tab);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;

  // the call's inputs: the first DRAM round trip on the critical path
  const int nq = c < p.E ? divs(p.E - 1 - c, G) + 1 : 0;   // router rows of this CTA
  issue_inputs(p, smem, c, G, nq, tid);
  {
    // this CTA's rows of the FP32 output accumulator start at zero.  The
    // threads that later publish the logits (the last nq * N) release these
    // stores now, while the input copies are in flight: a fence here and
    // their logit stores after it make the release pattern that orders the
    // zeros before every other CTA's reductions, which follow its acquire
    // reads of the logits
    const int r0 = divs(c * p.H, G), r1 = divs((c + 1) * p.H, G), ld = (p.N + 1) & ~1;
#pragma unroll 1
    for (int i = r0 * ld + tid; i < r1 * ld; i += kT) p.oacc[i] = 0.f;
    __syncthreads();
    if (tid >= kT - nq * p.N) fence_gpu();
  }
  if (tid == 0) {
    // the call's tag: the counter moves by exactly 256 per call (G <= 256):
    // CTA 0 adds 257 - G and the others 1, so every CTA of call c reads a
    // value in [256 c, 256 c + 255]
    const unsigned long long v = atomicAdd(&p.ctrl->calls, c == 0 ? 257ull - G : 1ull);
    tb.tag = (uint32_t)(v >> 8) + 1u;
    tb.abort = 0;
  }
  #pragma unroll 1
  for (int e = tid; e < p.E; e += kT) {
    tb.first[e] = 0xFFFFFFFFu;
    if (p.scoring != 0) tb.bias[e] = __ldg(p.bias + e);
    // read once here, off the weight stream's path
    tb.s2[e][0] = p.g2 ? __ldg(p.g2 + e) : 1.f;
    tb.s2[e][1] = p.u2 ? __ldg(p.u2 + e) : 1.f;
    tb.s2[e][2] = p.d2 ? __ldg(p.d2 + e) : 1.f;
  }
  if (tid < kSkSplitSlots) tb.split_cnt[tid] = 0u;
  if (lane == 0) {
    // this warp's ring stages: one arrival (lane 0's expect_tx) per use
#pragma unroll 1
    for (int s = 0; s < D; ++s) mbar_init(&tb.full[warp][s], 1u);
    fence_mbar_init();
  }
  if (tid < kSkMaxTok) {
    tb.xmax[tid] = 0u;
    tb.xdot[tid] = 0.f;
  }
  // the copies have landed; the barrier also publishes the tag and the
  // zeroed tables
  cpa_wait_all();
  __syncthreads();
  router_phase(p, tb, smem, c, G, nq, warp, lane, tid);
  x_prep(p, tb, smem, tid);
  {
    // the router's partial sums are done with the split area
    float* sp = reinterpret_cast<float*>(smem + p.off_split);
    for (int i = tid; i < kSkSplitSlots * 256; i += kT) sp[i] = 0.f;
    __syncthreads();
  }

  // PS: shared-expert gate/up while the logits land
  if (SH) shared_gate_up<D>(p, tb, smem, c, G, warp, lane);

  // P1: routing (the ring holds the float logits and keys until the weights stream)
  float* lg = reinterpret_cast<float*>(smem + p.off_ring);
  uint2* pairs = reinterpret_cast<uint2*>(smem + p.off_ring + ((p.N * p.E * 4 + 15) & ~15));
  uint2* cand = pairs + p.N * p.E;
  gather_logits(p, tb, lg, tid);
  __syncthreads();
  routing(p, tb, lg, pairs, cand, warp, lane);
  __syncthreads();
  if (c == 0) {
    const int S = p.N * p.k;
    #pragma unroll 1
    for (int s = tid; s < S; s += kT) {
      if (p.topk_idx) p.topk_idx[s] = tb.sel_e[s];
      if (p.topk_w) p.topk_w[s] = tb.sel_w[s];
    }
  }
  if (p.route_only) {
    // the end counter moves with the call counter (+256 per call), so the
    // next full call's end target stays reachable
    if (tid == 0) atomicAdd(&p.ctrl->fin, c == 0 ? 257ull - G : 1ull);
    return;
  }
  if ((p.N == 1 || (p.N <= 3 && (size_t)p.k * p.inter * p.H <= (16u << 20))) && warp == 1) {
    // a head start for the weight stream: the first k units are token 0's
    // selections in order, so this CTA's gate/up tiles among them (i = c +
    // G tl < k tpe, unit i / tpe) are known now; their gate and up rows (16
    // contiguous rows each) go to L2 while warp 0 builds the tables.  At
    // N = 1 these are all of the CTA's tiles.  Above that, warps whose first
    // tiles come later wait behind the burst: measured faster for bursts up
    // to 16 MB at N <= 3, slower at N = 4 or with larger bursts
    const int tpe = p.inter >> 4;
    const uint32_t rb = (uint32_t)(p.H >> 1);
#pragma unroll 1
    for (int i = c + G * lane; i < p.k * tpe; i += 32 * G) {
      const int u = divs(i, tpe), j = i - u * tpe;
      const size_t row0 = (size_t)tb.sel_e[u] * p.inter + 16 * j;   // u < k: token 0's
      bulk_prefetch_l2(p.gq + row0 * rb, 16u * rb);
      bulk_prefetch_l2(p.uq + row0 * rb, 16u * rb);
    }
  }
  if (warp == 0) build_tables(p, tb, lane);
  __syncthreads();

  // P2 + P3
  Pipe P;
  P.c = c;
  P.G = G;
  P.g = lane >> 2;
  P.t = lane & 3;
  P.lane = lane;
  P.ring = smem_u32(smem + p.off_ring) + (uint32_t)(warp * D * kSkStageCodes + lane * 16);
  P.aux = smem_u32(smem + p.off_aux) + (uint32_t)(warp * D * kSkStageAux + lane * 16);
  P.S = (p.H + 127) >> 7;
  P.tpe = p.inter >> 4;
  {
    const int Tr = tb.U * P.tpe;
    const int Tc = c < Tr ? divs(Tr - 1 - c, G) + 1 : 0;
    const int tot = Tc * P.S;
    P.a0 = (int)((long long)warp * tot / kW);
    P.a1 = (int)((long long)(warp + 1) * tot / kW);
  }
  P.Sd = (p.inter + 127) >> 7;
  P.Sds = SH ? p.Is >> 5 : 0;
  P.MT = p.H >> 5;   // 32-row down tiles
  // paired down order where the host chose it (long lists, an even number
  // of segments per unit)
  const bool paired = p.dpair != 0;
  P.sst = paired ? 2 : 1;
  P.spar = paired ? (warp & 1) : 0;
  P.sdp = paired ? P.Sd >> 1 : P.Sd;
  P.nsh = (paired ? P.Sds >> 1 : P.Sds) * P.MT;
  {
    // the grid's down items split over all warps in order
    // floor(gw * tot / nw) in 32-bit pieces: gw * r < nw^2 <= 2^24; a pair
    // of warps shares one range when paired
    const uint32_t tot = (uint32_t)(P.nsh + tb.U * P.sdp * P.MT);
    const uint32_t gw = (uint32_t)(c * kW + warp) >> (paired ? 1 : 0);
    const uint32_t nw = (uint32_t)(G * kW) >> (paired ? 1 : 0);
    const uint32_t q = tot / nw, r = tot - q * nw;
    P.b0 = (int)(gw * q + gw * r / nw);
    P.b1 = (int)((gw + 1) * q + (gw + 1) * r / nw);
  }
  if (!tb.abort) pipeline<FMT, D, SH>(p, tb, smem, P);

  // every CTA's reductions into the output accumulator are done when the
  // end counter (+ 256 per call, like the call counter) reaches 256 x tag
  __syncthreads();
  if (tid == 0) {
    fence_gpu();   // no weight copies are in flight here
    atomicAdd(&p.ctrl->fin, c == 0 ? 257ull - G : 1ull);
    const unsigned long long target = (unsigned long long)tb.tag << 8;
    if (ld_acquire64(&p.ctrl->fin) < target) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire64(&p.ctrl->fin) < target) {
        if (global_timer_ns() - t0 > p.timeout_ns) {
          set_error(p, tb, kErrTimeoutBarrier);
          break;
        }
        __nanosleep(64);
      }
    }
  }
  __syncthreads();
  if (tb.abort) return;
  {
    // this CTA's output rows in BF16
    const int r0 = divs(c * p.H, G), r1 = divs((c + 1) * p.H, G);
    const int nr = r1 - r0;
#pragma unroll 1
    for (int idx = tid; idx < nr * p.N; idx += kT) {
      const int n = divs(idx, nr), r = r0 + idx - n * nr;
      p.out[(size_t)n * p.H + r] =
          __bfloat16_as_ushort(__float2bfloat16_rn(__ldcg(p.oacc + r * ((p.N + 1) & ~1) + n)));
    }
  }
}

}  // namespace

bool plan_stream(StreamParams& p, int smem_budget, int grid) {
  if (p.N < 1 || p.N > kSkMaxTok) return false;
  if (p.fmt != FMT_NVFP4 && p.fmt != FMT_MXFP4) return false;
  if (p.H % 32 || p.inter % 32 || p.Is % 32) return false;
  if (p.E > kMaxE || p.N * p.k > kMaxSlots) return false;
  if (grid < 128 || grid > kSkMaxGrid || (p.E + grid - 1) / grid > kMaxRouterRows) return false;
  if (p.Is > 0) {
    const int Ts = p.Is / 16, Sb = p.H / 32;
    if (Ts > grid) return false;   // one shared unit per CTA at most
    int parts = grid / Ts;
    if (parts > Sb) parts = Sb;
    p.sh_parts = parts;
  } else {
    p.sh_parts = 0;
  }
  const int S = (p.H + 127) / 128;
  auto al = [](int v) { return (v + 1023) & ~1023; };
  int off = 0;
  p.off_tab = off;
  off = al(off + (int)sizeof(SkTab));
  p.off_split = off;
  off = al(off + kSkSplitSlots * 256 * 4);
  p.off_x16 = off;
  off = al(off + S * 4 * p.N * 64);
  // the ring region: kSkStages code stages per warp once the weights
  // stream; before that it holds this CTA's router rows, then the float
  // logits, their (key, expert) pairs and the top-k candidates
  const int Wt = (p.E + 127) / 128;
  if (Wt * p.k > 128) return false;   // the second top-k level holds 4 candidates per lane
  const int nq = (p.E + grid - 1) / grid;
  int ring = kSkStages * kSkWarps * kSkStageCodes;
  ring = max(ring, ((p.N * p.E * 4 + 15) & ~15) + p.N * p.E * 8 + p.N * Wt * p.k * 8);
  ring = max(ring, nq * p.H * 2);
  // the router's partial sums sit in the split area
  if (nq * p.N * ((p.H + 255) / 256) > kSkSplitSlots * 256) return false;
  p.stages = kSkStages;
  p.off_ring = off;
  off = al(off + ring);
  p.off_aux = off;
  off += kSkStages * kSkWarps * kSkStageAux;
  p.smem_bytes = off;
  return off <= smem_budget;
}

// The kernel instances: block-scale format x shared expert.
template <int FMT, bool SH>
constexpr const void* sk_fn() {
  return (const void*)moe_stream_kernel<FMT, kSkStages, SH>;
}
const void* stream_fn(int fmt, bool sh) {
  return fmt == FMT_NVFP4 ? (sh ? sk_fn<FMT_NVFP4, true>() : sk_fn<FMT_NVFP4, false>())
                          : (sh ? sk_fn<FMT_MXFP4, true>() : sk_fn<FMT_MXFP4, false>());
}

cudaError_t stream_set_smem(int smem_bytes) {
  for (int fmt : {FMT_NVFP4, FMT_MXFP4})
    for (bool sh : {false, true}) {
      const cudaError_t e = cudaFuncSetAttribute(stream_fn(fmt, sh),
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

cudaError_t launch_stream(const StreamParams& p, int grid, cudaStream_t stream) {
  void* args[] = {const_cast<StreamParams*>(&p)};
  return cudaLaunchCooperativeKernel(stream_fn(p.fmt, p.Is > 0), dim3(grid),
                                     dim3(kSkThreads), args, (size_t)p.smem_bytes, stream);
}

}  // namespace moe
