// Grouped MoE layer forward for many tokens (prefill-sized N) on sm_103a.
//
// Same mathematics as the decode kernel (forward chain of forward_k3.rs:
// router GEMV -> top-k -> expert gate+up -> SiLU -> down -> weighted sum),
// organised as per-expert token groups so that each routed expert's weights
// are streamed once for all of its tokens (the grouped GEMM that
// forward_batched.rs switches to for larger row counts) and the contractions
// run on the tcgen05 tensor cores.  Stream-ordered launches:
//
//   router    logits[n,e] (FP32, CUDA cores)
//   top-k     warp top-k per token; per-token power-of-two exponent of x
//   plan      per-expert token counts, expert-sorted positions of the
//             (token, slot) pairs, token tiles of <= 64 positions (one CTA)
//   gather    xg[pos] = x[token(pos)] * 2^-xexp as f16, in expert order
//   gemm(2)   per (token tile, 128-row block): g = Dq(Wg) xg^T, u = Dq(Wu) xg^T,
//             h = SiLU(g) * u (FP32)
//   pack      h16[pos] = h[pos] * 2^-hexp as f16 (per-row power of two)
//   gemm(1)   y = w(pos) * Dq(Wd) h16^T (FP32, one row per position)
//   combine   out[n] = bf16(sum over the k slots of n of y)
//
// GEMM kernel (persistent, one CTA per SM, 25 warps):
//   warp 0      TMA producer: FP4 weight boxes (64 bytes x 128 rows, 64-byte
//               swizzle), activation boxes (64 f16 x 64 rows, 128-byte
//               swizzle), the unit's block scales (1D bulk copy)
//   warps 1,22-24  TMEM allocation (warp 1); lane 0 of each issues tcgen05.mma kind::f16
//               (A from tensor memory, B from shared memory, FP32 accumulators
//               in tensor memory, M = 128 weight rows, N = tokens rounded to 16,
//               one partial accumulator per issuer)
//   warps 2-17  dequantisation: thread = weight row; E2M1 -> f16 with
//               cvt.rn.f16x2.e2m1x2, times the block scale (E4M3 as f16:
//               exact; E8M0 as a power of two relative to the row's largest
//               scale), written to tensor memory with tcgen05.st
//   warps 18-21 epilogue: tcgen05.ld of the accumulators, scale factors,
//               SiLU(g)*u or the routing weight, FP32 stores
//
// The f16 A and B operands are exact images of the FP4 weights and of the
// BF16 activations (up to f16 subnormal flushing of values more than ~2^28
// below the row maximum), and f16 x f16 products are exact in FP32, so the
// only rounding besides FP32 accumulation is the f16 image of h.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_internal.h"
#include "ptx.cuh"
#include "routing.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kRtTok = 8;          // tokens per router CTA
constexpr int kGThreads = 800;     // GEMM kernel: 25 warps
constexpr int kTileRows = 128;     // weight rows per unit (MMA M)
constexpr int kKChunk = 128;       // K elements per stage
constexpr int kABox = 8192;        // 128 rows x 64 bytes of FP4
constexpr int kBBox = 8192;        // 64 positions x 128 bytes of f16
constexpr int kNA = 4;             // A slots in tensor memory
constexpr uint32_t kTmemCols = 512;

// power-of-two exponent e with max * 2^-e in [2^14, 2^15) (0 for max == 0)
__device__ __forceinline__ int f16_exponent(float mx) {
  if (!(mx > 0.f) || isinf(mx)) return 0;
  int ex;
  frexpf(mx, &ex);   // mx = f * 2^ex, f in [0.5, 1)
  return ex - 15;
}

__device__ __forceinline__ uint32_t f16x2_pack(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

}  // namespace

// ------------------------------------------------------------------ router
// Grid (token groups of 8) x (expert groups of 16): each CTA holds its 8 x
// rows in shared memory; each warp computes 2 experts for the 8 tokens, with
// the router row's loads issued 8 vectors at a time (latency, not bandwidth,
// bounds this kernel).
constexpr int kRtExp = 16;   // experts per router CTA

__global__ void __launch_bounds__(256) grouped_router_kernel(const GroupedParams p) {
  extern __shared__ __align__(1024) uint8_t rsmem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(rsmem);   // [8][H]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * kRtTok;
  const int nt = min(kRtTok, p.N - n0);
  const int H = p.H, E = p.E;
  for (int i = tid * 8; i < nt * H; i += 256 * 8)
    *reinterpret_cast<uint4*>(xs + i) = ld_nc_u4(p.x + (size_t)n0 * H + i);
  __syncthreads();
  const float rs2 = (p.router_fmt == 1 && p.router_s2) ? __ldg(p.router_s2) : 1.0f;
  for (int e = blockIdx.y * kRtExp + warp; e < min(E, (int)(blockIdx.y + 1) * kRtExp); e += 8) {
    float acc[kRtTok];
#pragma unroll
    for (int t = 0; t < kRtTok; ++t) acc[t] = 0.f;
    if (p.router_fmt == 1) {   // NVFP4 router: eight decoded weights per lane and step
      for (int h = lane * 8; h < H; h += 32 * 8) {
        float wf[8];
        router_w8(p.router, 1, p.router_s, rs2, H, e, h, wf);
#pragma unroll
        for (int t = 0; t < kRtTok; ++t) {
          if (t < nt) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * H + h);
            const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
            float a2 = acc[t];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              a2 = fmaf(wf[2 * q], __uint_as_float(xa[q] << 16), a2);
              a2 = fmaf(wf[2 * q + 1], __uint_as_float(xa[q] & 0xFFFF0000u), a2);
            }
            acc[t] = a2;
          }
        }
      }
    }
    const uint16_t* wr = p.router + (size_t)e * H;
    for (int hb = 0; p.router_fmt == 0 && hb < H; hb += 8 * 256) {
      uint4 wv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int h = hb + (i * 32 + lane) * 8;
        wv[i] = (h < H) ? ld_nc_u4(wr + h) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int h = hb + (i * 32 + lane) * 8;
        if (h >= H) continue;
        const uint32_t wa[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
        for (int t = 0; t < kRtTok; ++t) {
          if (t < nt) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xs + t * H + h);
            const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w};
            float a2 = acc[t];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              a2 = fmaf(__uint_as_float(wa[q] << 16), __uint_as_float(xa[q] << 16), a2);
              a2 = fmaf(__uint_as_float(wa[q] & 0xFFFF0000u),
                        __uint_as_float(xa[q] & 0xFFFF0000u), a2);
            }
            acc[t] = a2;
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kRtTok; ++t) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t < nt) p.logits[(size_t)(n0 + t) * E + e] = v;
    }
  }
}

// One warp per token: top-k over the FP32 logits, and the power-of-two
// exponent of the token's f16 image.
__global__ void __launch_bounds__(256) grouped_topk_kernel(const GroupedParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + warp;
  if (n >= p.N) return;
  const int E = p.E;
  float mx = 0.f;
  const uint16_t* xr = p.x + (size_t)n * p.H;
  for (int h = lane * 8; h < p.H; h += 256) {
    const uint4 v = ld_nc_u4(xr + h);
    const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(a[q] << 16)),
                           fabsf(__uint_as_float(a[q] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) p.xexp[n] = f16_exponent(mx);
  const float* lrow = p.logits + (size_t)n * E;
  int se = 0;
  float sw = 0.f;
#define MOE_TOPK_CASE(PER)                                                         \
  {                                                                                \
    float lg[PER];                                                                 \
    _Pragma("unroll") for (int i = 0; i < PER; ++i) {                              \
      const int e = lane + 32 * i;                                                 \
      lg[i] = (e < E) ? lrow[e] : -INFINITY;                                       \
    }                                                                              \
    topk_warp<PER>(E, p.k, p.scoring, p.norm, p.rsf, p.bias, lg, lane, &se, &sw); \
  }
  if (E <= 128) MOE_TOPK_CASE(4)
  else if (E <= 256) MOE_TOPK_CASE(8)
  else if (E <= 512) MOE_TOPK_CASE(16)
  else MOE_TOPK_CASE(32)
#undef MOE_TOPK_CASE
  if (lane < p.k) {
    p.sel_e[n * p.k + lane] = se;
    p.sel_w[n * p.k + lane] = sw;
    if (p.topk_idx) p.topk_idx[n * p.k + lane] = se;
    if (p.topk_w) p.topk_w[n * p.k + lane] = sw;
  }
}

// -------------------------------------------------------------------- plan
// Block-wide exclusive scan of one value per thread (1024 threads).
__device__ int scan1024(int v, int* sh, int* total) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = sh[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    sh[32 + lane] = wi - w;
    if (lane == 31) sh[64] = wi;
  }
  __syncthreads();
  const int r = sh[32 + warp] + inc - v;
  *total = sh[64];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) grouped_plan_kernel(const GroupedParams p) {
  __shared__ int cnt[kMaxE];
  __shared__ int cursor[kMaxE];
  __shared__ int sh[96];
  const int tid = threadIdx.x;
  const int S = p.N * p.k;
  for (int e = tid; e < p.E; e += 1024) cnt[e] = 0;
  __syncthreads();
  for (int s = tid; s < S; s += 1024) atomicAdd(&cnt[p.sel_e[s]], 1);
  __syncthreads();
  const int c = (tid < p.E) ? cnt[tid] : 0;
  const int nt = (c + kGTileTok - 1) / kGTileTok;
  int tot_pos = 0, tot_tiles = 0;
  const int off = scan1024(c, sh, &tot_pos);
  const int toff = scan1024(nt, sh, &tot_tiles);
  if (tid < p.E) {
    cursor[tid] = off;
    for (int q = 0; q < nt; ++q) {
      int* t = p.tiles + 3 * (toff + q);
      t[0] = tid;
      t[1] = off + q * kGTileTok;
      t[2] = min(kGTileTok, c - q * kGTileTok);
    }
  }
  if (tid == 0) p.ntiles[0] = tot_tiles;
  __syncthreads();
  for (int s = tid; s < S; s += 1024) {
    const int pos = atomicAdd(&cursor[p.sel_e[s]], 1);
    p.pos_of[s] = pos;
    p.tok_of[pos] = s / p.k;
    p.w_of[pos] = p.sel_w[s];
  }
}

// ------------------------------------------------------------------ gather
__global__ void __launch_bounds__(128) grouped_gather_kernel(const GroupedParams p) {
  const int pos = blockIdx.x;
  const int n = p.tok_of[pos];
  const int ex = p.xexp[n];
  if (threadIdx.x == 0) p.bexp[pos] = ex;
  const uint16_t* src = p.x + (size_t)n * p.H;
  uint16_t* dst = p.xg + (size_t)pos * p.H;
  for (int h = threadIdx.x * 8; h < p.H; h += 128 * 8) {
    const uint4 v = ld_nc_u4(src + h);
    const uint32_t a[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = f16x2_pack(ldexpf(__uint_as_float(a[q] << 16), -ex),
                        ldexpf(__uint_as_float(a[q] & 0xFFFF0000u), -ex));
    *reinterpret_cast<uint4*>(dst + h) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// -------------------------------------------------------------------- pack
__global__ void __launch_bounds__(256) grouped_pack_kernel(const GroupedParams p) {
  __shared__ float red[8];
  const int pos = blockIdx.x, tid = threadIdx.x;
  const float* src = p.hbuf + (size_t)pos * p.inter;
  float mx = 0.f;
  for (int i = tid * 4; i < p.inter; i += 256 * 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + i);
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) mx = fmaxf(mx, red[w]);
  const int ex = f16_exponent(mx);
  if (tid == 0) p.hexp[pos] = ex;
  uint16_t* dst = p.h16 + (size_t)pos * p.inter;
  for (int i = tid * 4; i < p.inter; i += 256 * 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + i);
    *reinterpret_cast<uint2*>(dst + i) =
        make_uint2(f16x2_pack(ldexpf(v.x, -ex), ldexpf(v.y, -ex)),
                   f16x2_pack(ldexpf(v.z, -ex), ldexpf(v.w, -ex)));
  }
}

// ----------------------------------------------------------------- combine
__global__ void __launch_bounds__(256) grouped_combine_kernel(const GroupedParams p) {
  const int n = blockIdx.x;
  int pos[kMaxTopK];
  for (int j = 0; j < p.k; ++j) pos[j] = p.pos_of[n * p.k + j];
  for (int r = threadIdx.x; r < p.H; r += 256) {
    float s = 0.f;
    for (int j = 0; j < p.k; ++j) s += p.hbuf[(size_t)pos[j] * p.H + r];
    const __nv_bfloat16 b = __float2bfloat16_rn(s);
    p.out[(size_t)n * p.H + r] = *reinterpret_cast<const uint16_t*>(&b);
  }
}

// -------------------------------------------------------------------- GEMM
namespace {

// Roles: warp 0 producer, warp 1 TMEM owner + MMA issuer 0, warps 2-17
// dequantisation (one 32-element piece of one projection per A slot each),
// warps 18-21 epilogue, warps 22-24 MMA issuers 1-3.  One thread issues a
// small-N tcgen05.mma only every ~45-60 cycles whatever N (<= 64), while the
// tensor core takes far more; so four issuers share the MMAs, each with its
// own accumulator, each owning whole stages (two projections: issuer =
// projection x stage parity; one projection: issuer = stage index mod 4), so
// that every barrier has a fixed set of arrivals.  The epilogue sums the
// issuers' partial accumulators.
constexpr int kDeqWarps = 16;
constexpr int kEpiWarps = 4;
constexpr int kIssuers = 4;
constexpr int kDeq0 = 2, kEpi0 = kDeq0 + kDeqWarps, kMma1 = kEpi0 + kEpiWarps;

struct GBars {
  uint64_t* full;     // [8]   stage ring: TMA -> dequant + MMA
  uint64_t* empty;    // [8]   16 dequant warps + MMA commit -> producer
  uint64_t* afull;    // [4]   dequant -> MMA (tensor-memory A slot written)
  uint64_t* aempty;   // [4]   MMA commits of the issuers that read the slot -> dequant
  uint64_t* dfull;    // [2]   all issuers' commits -> epilogue (accumulators ready)
  uint64_t* dempty;   // [2]   epilogue -> MMA
  uint64_t* scfull;   // [2]   unit scales landed
  uint64_t* scempty;  // [2]   dequant + epilogue done with the unit's scales
  uint64_t* fin;      // [4]   final MMA commit of each issuer
  uint32_t* tslot;
  int* abort;
};

struct GUnit {
  int e, p0, nt, rt;
};

__device__ __forceinline__ GUnit gunit(const GemmParams& p, int u, int RT) {
  const int t = u / RT;
  GUnit r;
  r.e = __ldg(p.tiles + 3 * t);
  r.p0 = __ldg(p.tiles + 3 * t + 1);
  r.nt = __ldg(p.tiles + 3 * t + 2);
  r.rt = u - t * RT;
  return r;
}

__device__ __forceinline__ bool gwait(const GemmParams& p, const GBars& b, uint64_t* bar,
                                      uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*reinterpret_cast<volatile int*>(b.abort)) return false;
  if (mbar_wait_bounded(bar, parity, p.timeout_ns)) return true;
  atomicExch(b.abort, 1);
  atomicOr(p.err, kErrTimeoutStage);
  return false;
}
// all lanes wait; the warp agrees on the outcome
__device__ __forceinline__ bool gwait_warp(const GemmParams& p, const GBars& b, uint64_t* bar,
                                           uint32_t parity) {
  const bool ok = gwait(p, b, bar, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint8_t* gstage(uint8_t* smem, const GemmParams& p, int s) {
  return smem + (size_t)s * p.stage_bytes;
}
__device__ __forceinline__ uint8_t* gscbuf(uint8_t* smem, const GemmParams& p, int ub) {
  return smem + p.off_sc + (size_t)ub * p.sc_bytes;
}
// Tensor-memory columns: accumulators [2 buffers][4 issuers][32 tokens], then
// 4 A slots of 64 columns: [2 proj][32 columns = 64 K] (two projections) or
// [64 columns = 128 K] (one projection).
__device__ __forceinline__ int dcol(int b, int i) { return b * 128 + i * 32; }
__device__ __forceinline__ int acol(int a, int pj) { return 256 + a * 64 + pj * 32; }
// K elements of one A slot: 16 MMA K-steps' worth of dequantisation work
// (16 warps x one 32-element piece) whatever the projection count.
template <int NPROJ>
__host__ __device__ constexpr int slot_k() { return 128 / NPROJ; }

// largest non-NaN E8M0 code of a row's scales (0 if none)
__device__ __forceinline__ int row_max_e8m0(const uint8_t* s, int n) {
  int mx = 0;
  for (int i = 0; i < n; ++i) {
    const int v = s[i];
    if (v != 0xFF) mx = max(mx, v);
  }
  return mx;
}

template <int NPROJ>
__device__ void g_producer(const GemmParams& p, uint8_t* smem, const GBars& b, int RT,
                           int nunits) {
  for (int i = 0; i < NPROJ; ++i) prefetch_tensormap(&p.tmA[i]);
  prefetch_tensormap(&p.tmB);
  const int nch = (p.K + kKChunk - 1) / kKChunk;
  int sctr = 0, it = 0, nsc = 0;   // stages and scale copies issued
  bool ok = true;
  for (int u = blockIdx.x; ok && u < nunits; u += gridDim.x, ++it) {
    const GUnit un = gunit(p, u, RT);
    const int rv = min(kTileRows, p.rows - un.rt * kTileRows);
    const int ub = it % p.nscbuf;
    const uint32_t ur = (uint32_t)(it / p.nscbuf);
    if (!gwait(p, b, b.scempty + ub, (ur & 1u) ^ 1u)) { ok = false; break; }
    mbar_arrive_expect_tx(b.scfull + ub, (uint32_t)(NPROJ * rv * p.sr));
    const size_t srow = ((size_t)un.e * p.rows + (size_t)un.rt * kTileRows) * p.sr;
    for (int pj = 0; pj < NPROJ; ++pj)
      bulk_g2s(gscbuf(smem, p, ub) + pj * kTileRows * p.sr, p.sc[pj] + srow,
               (uint32_t)(rv * p.sr), b.scfull + ub);
    ++nsc;
    const int arow = un.e * p.rows + un.rt * kTileRows;
    for (int c = 0; c < nch; ++c, ++sctr) {
      const int s = sctr % p.nstages;
      const uint32_t r = (uint32_t)(sctr / p.nstages);
      if (!gwait(p, b, b.empty + s, (r & 1u) ^ 1u)) { ok = false; break; }
      const int nb = min(2, (p.K - c * kKChunk + 63) / 64);
      mbar_arrive_expect_tx(b.full + s, (uint32_t)(NPROJ * kABox + nb * kBBox));
      uint8_t* st = gstage(smem, p, s);
      for (int pj = 0; pj < NPROJ; ++pj)
        tma_load_2d(st + pj * kABox, &p.tmA[pj], c * (kKChunk / 2), arow, b.full + s);
      for (int j = 0; j < nb; ++j)
        tma_load_2d(st + NPROJ * kABox + j * kBBox, &p.tmB, (c * kKChunk + j * 64) * 2, un.p0,
                    b.full + s);
    }
  }
  if (!ok) {   // drain copies still in flight into our buffers
    const int first = sctr > p.nstages ? sctr - p.nstages : 0;
    for (int i = first; i < sctr; ++i)
      mbar_wait_bounded(b.full + (i % p.nstages), (uint32_t)(i / p.nstages) & 1u, p.timeout_ns);
    const int f2 = nsc > p.nscbuf ? nsc - p.nscbuf : 0;
    for (int i = f2; i < nsc; ++i)
      mbar_wait_bounded(b.scfull + (i % p.nscbuf), (uint32_t)(i / p.nscbuf) & 1u, p.timeout_ns);
  }
}

// One dequantisation warp: rows q*32 .. q*32+31 of the tile (its tensor-memory
// lane quarter), one projection, one 32-element piece of every A slot.
template <int NPROJ, int FMT>
__device__ void g_dequant(const GemmParams& p, uint8_t* smem, const GBars& b, uint32_t tbase,
                          int RT, int nunits) {
  constexpr int SK = slot_k<NPROJ>();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int role = (warp - kDeq0) >> 2;   // 0..3
  const int q = warp & 3;                 // tensor-memory lane quarter
  const int m = q * 32 + lane;            // weight row within the tile
  const int pj = (NPROJ == 2) ? (role >> 1) : 0;
  const int pc = (NPROJ == 2) ? (role & 1) : role;   // piece within the slot
  const int nch = (p.K + kKChunk - 1) / kKChunk;
  int sctr = 0, actr = 0, it = 0;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++it) {
    const GUnit un = gunit(p, u, RT);
    const int rv = min(kTileRows, p.rows - un.rt * kTileRows);
    const bool live = m < rv;   // warp-uniform: rv is a multiple of 32
    const int ub = it % p.nscbuf;
    if (!gwait_warp(p, b, b.scfull + ub, (uint32_t)(it / p.nscbuf) & 1u)) return;
    const uint8_t* srow = gscbuf(smem, p, ub) + pj * kTileRows * p.sr + m * p.sr;
    int mref = 0;
    if (FMT == FMT_MXFP4 && live) mref = row_max_e8m0(srow, p.sr) - 13;
    for (int c = 0; c < nch; ++c, ++sctr) {
      const int s = sctr % p.nstages;
      if (!gwait_warp(p, b, b.full + s, (uint32_t)(sctr / p.nstages) & 1u)) return;
      const uint8_t* at = gstage(smem, p, s) + pj * kABox + m * 64;
      const int nslot = min(NPROJ, (p.K - c * kKChunk + SK - 1) / SK);
      for (int j = 0; j < nslot; ++j, ++actr) {
        const int a = actr % kNA;
        const int pi = j * (SK / 32) + pc;   // 16-byte piece of the 64-byte row
        const int k0 = c * kKChunk + pi * 32;
        const bool work = live && k0 < p.K;
        // load and convert before waiting for the slot
        uint32_t v[16];
        if (work) {
          const uint4 w = *reinterpret_cast<const uint4*>(at + ((pi ^ ((m >> 1) & 3)) << 4));
          uint32_t o[4];
          e2m1x8_to_f16x2x4(w.x, o);
          v[0] = o[0]; v[1] = o[1]; v[2] = o[2]; v[3] = o[3];
          e2m1x8_to_f16x2x4(w.y, o);
          v[4] = o[0]; v[5] = o[1]; v[6] = o[2]; v[7] = o[3];
          e2m1x8_to_f16x2x4(w.z, o);
          v[8] = o[0]; v[9] = o[1]; v[10] = o[2]; v[11] = o[3];
          e2m1x8_to_f16x2x4(w.w, o);
          v[12] = o[0]; v[13] = o[1]; v[14] = o[2]; v[15] = o[3];
          uint32_t s0, s1;
          if (FMT == FMT_NVFP4) {
            const uint32_t sv =
                e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(srow + k0 / 16));
            s0 = __byte_perm(sv, 0, 0x1010);
            s1 = __byte_perm(sv, 0, 0x3232);
          } else {
            // 2^j2 as f16, j2 = code - (row max code - 13) <= 13
            const int code = srow[k0 / 32];
            const int j2 = code - mref;
            uint32_t bits;
            if (code == 0xFF) bits = 0x7E00u;                      // NaN scale
            else if (j2 >= -14) bits = (uint32_t)(j2 + 15) << 10;  // normal
            else if (j2 >= -24) bits = 1u << (j2 + 24);            // subnormal
            else bits = 0u;                                        // below f16: flushed
            s0 = s1 = bits | (bits << 16);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = hmul2(v[i], s0);
#pragma unroll
          for (int i = 8; i < 16; ++i) v[i] = hmul2(v[i], s1);
        }
        if (!gwait_warp(p, b, b.aempty + a, ((uint32_t)(actr / kNA) & 1u) ^ 1u)) return;
        tc_fence_after();
        if (work) {
          tmem_st16(tmem_addr(tbase, q * 32, acol(a, pj) + pc * 16), v);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(b.afull + a);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(b.empty + s);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(b.scempty + ub);
  }
}

// Does issuer `i` own stage `sctr`?  Two projections: stage parity = i & 1
// (the projection is i >> 1); one projection: stage index mod 4 = i.
template <int NPROJ>
__device__ __forceinline__ bool owns_stage(int i, int sctr) {
  return NPROJ == 2 ? ((sctr & 1) == (i & 1)) : ((sctr & 3) == i);
}

// MMA issuer `me` (0..3): every A slot of the stages it owns, into its own
// partial accumulator.  Full slots are issued as straight-line code (a branch
// between MMAs slows the issue).
template <int NPROJ>
__device__ void g_mma(const GemmParams& p, uint8_t* smem, const GBars& b, uint32_t tbase, int RT,
                      int nunits, int me) {
  constexpr int SK = slot_k<NPROJ>();
  constexpr int KS = SK / 16;   // MMA K-steps per slot
  const int pj = (NPROJ == 2) ? (me >> 1) : 0;
  const int nch = (p.K + kKChunk - 1) / kKChunk;
  int sctr = 0, actr = 0, it = 0;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++it) {
    const GUnit un = gunit(p, u, RT);
    const int db = it & 1;
    if (!gwait(p, b, b.dempty + db, ((uint32_t)(it >> 1) & 1u) ^ 1u)) break;
    tc_fence_after();
    const uint32_t idesc = idesc_f16_f32(kTileRows, (un.nt + 15) & ~15);
    const uint32_t d = tmem_addr(tbase, 0, dcol(db, me));
    uint32_t accum = 0u;
    bool ok = true;
    for (int c = 0; c < nch && ok; ++c, ++sctr) {
      const int s = sctr % p.nstages;
      const int kleft = p.K - c * kKChunk;
      const int nslot = min(NPROJ, (kleft + SK - 1) / SK);
      if (!owns_stage<NPROJ>(me, sctr)) {
        actr += nslot;
        continue;
      }
      if (!gwait(p, b, b.full + s, (uint32_t)(sctr / p.nstages) & 1u)) { ok = false; break; }
      const uint64_t bdesc = sdesc_sw128(smem_u32(gstage(smem, p, s) + NPROJ * kABox));
      for (int j = 0; j < nslot; ++j, ++actr) {
        const int a = actr % kNA;
        if (!gwait(p, b, b.afull + a, (uint32_t)(actr / kNA) & 1u)) { ok = false; break; }
        tc_fence_after();
        const uint32_t at = tmem_addr(tbase, 0, acol(a, pj));
        // B: box kk/64 of the stage, 32 bytes per K-step inside the 128-byte swizzled row
        const uint64_t bd = bdesc + (uint64_t)((j * SK / 64) * (kBBox >> 4));
        if (kleft - j * SK >= SK) {
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            mma_f16_ts(d, at + ks * 8, bd + (uint64_t)((ks >> 2) * (kBBox >> 4) + (ks & 3) * 2),
                       idesc, accum);
            accum = 1u;
          }
        } else {
          for (int ks = 0; ks * 16 < kleft - j * SK; ++ks) {
            mma_f16_ts(d, at + ks * 8, bd + (uint64_t)((ks >> 2) * (kBBox >> 4) + (ks & 3) * 2),
                       idesc, accum);
            accum = 1u;
          }
        }
        mma_commit(b.aempty + a);
      }
      if (ok) mma_commit(b.empty + s);
    }
    if (!ok) break;
    mma_commit(b.dfull + db);
  }
  mma_commit(b.fin + me);   // completes once every MMA issued above has finished
  mbar_wait_bounded(b.fin + me, 0, p.timeout_ns);
}

template <int NPROJ, int FMT>
__device__ void g_epilogue(const GemmParams& p, uint8_t* smem, const GBars& b, uint32_t tbase,
                           int RT, int nunits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;
  const int m = q * 32 + lane;
  int it = 0;
  for (int u = blockIdx.x; u < nunits; u += gridDim.x, ++it) {
    const GUnit un = gunit(p, u, RT);
    const int rv = min(kTileRows, p.rows - un.rt * kTileRows);
    const bool live = m < rv;
    const int db = it & 1;
    const int ub = it % p.nscbuf;
    // per-token factors, token t held by lane t % 32 (t < 64): 2^bexp (and weight)
    float tf0 = 0.f, tf1 = 0.f;
    if (lane < un.nt) {
      tf0 = ldexpf(1.0f, __ldg(p.bexp + un.p0 + lane));
      if (NPROJ == 1) tf0 *= __ldg(p.wpos + un.p0 + lane);
    }
    if (lane + 32 < un.nt) {
      tf1 = ldexpf(1.0f, __ldg(p.bexp + un.p0 + 32 + lane));
      if (NPROJ == 1) tf1 *= __ldg(p.wpos + un.p0 + 32 + lane);
    }
    if (!gwait_warp(p, b, b.scfull + ub, (uint32_t)(it / p.nscbuf) & 1u)) return;
    // per-row factors: scale2 (NVFP4) or 2^(row reference exponent - 127) (MXFP4)
    float rf[2] = {1.f, 1.f};
#pragma unroll
    for (int pj = 0; pj < NPROJ; ++pj) {
      if (FMT == FMT_NVFP4) {
        rf[pj] = p.s2[pj] ? __ldg(p.s2[pj] + un.e) : 1.0f;
      } else if (live) {
        const uint8_t* srow = gscbuf(smem, p, ub) + pj * kTileRows * p.sr + m * p.sr;
        rf[pj] = ldexpf(1.0f, row_max_e8m0(srow, p.sr) - 13 - 127);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(b.scempty + ub);
    if (!gwait_warp(p, b, b.dfull + db, (uint32_t)(it >> 1) & 1u)) return;
    tc_fence_after();
    const int nmma = (un.nt + 15) & ~15;
    // issuers that owned a stage of this unit (its stages are it*nch .. +nch-1)
    const int nch = (p.K + kKChunk - 1) / kKChunk;
    uint32_t used = 0u;
    for (int c = 0; c < nch && c < 4; ++c)
#pragma unroll
      for (int is = 0; is < kIssuers; ++is)
        if (owns_stage<NPROJ>(is, it * nch + c)) used |= 1u << is;
    float* dst = p.out + (size_t)un.p0 * p.rows + un.rt * kTileRows + m;
    for (int cb = 0; cb < nmma; cb += 16) {
      // partial accumulators of the issuers that owned at least one stage
      float v0[16], v1[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v0[i] = v1[i] = 0.f;
#pragma unroll
      for (int is = 0; is < kIssuers; ++is) {
        if (!(used >> is & 1)) continue;
        uint32_t r[16];
        tmem_ld16(tmem_addr(tbase, q * 32, dcol(db, is) + cb), r);
        tmem_wait_ld();
        if (NPROJ == 2 && is >= 2) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v1[i] += __uint_as_float(r[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v0[i] += __uint_as_float(r[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = cb + i;
        const float tf = __shfl_sync(0xffffffffu, t < 32 ? tf0 : tf1, t & 31);
        if (live && t < un.nt) {
          if (NPROJ == 2) {
            const float g = v0[i] * rf[0] * tf;
            const float uu = v1[i] * rf[1] * tf;
            dst[(size_t)t * p.rows] = g / (1.0f + expf(-g)) * uu;
          } else {
            dst[(size_t)t * p.rows] = v0[i] * rf[0] * tf;
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(b.dempty + db);
  }
}

}  // namespace

template <int NPROJ, int FMT>
__global__ void __launch_bounds__(kGThreads, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  GBars b;
  b.full = bars;
  b.empty = bars + 8;
  b.afull = bars + 16;
  b.aempty = bars + 20;
  b.dfull = bars + 24;
  b.dempty = bars + 26;
  b.scfull = bars + 28;
  b.scempty = bars + 30;
  b.fin = bars + 32;
  b.tslot = reinterpret_cast<uint32_t*>(bars + 36);
  b.abort = reinterpret_cast<int*>(bars + 37);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < p.nstages; ++s) {
      mbar_init(b.full + s, 1);
      mbar_init(b.empty + s, kDeqWarps + (NPROJ == 2 ? 2 : 1));
    }
    for (int a = 0; a < kNA; ++a) {
      mbar_init(b.afull + a, kDeqWarps);
      mbar_init(b.aempty + a, NPROJ == 2 ? 2 : 1);   // issuers reading the slot
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b.dfull + i, kIssuers);
      mbar_init(b.dempty + i, kEpiWarps);
      mbar_init(b.scfull + i, 1);
      mbar_init(b.scempty + i, kDeqWarps + kEpiWarps);
    }
    for (int i = 0; i < kIssuers; ++i) mbar_init(b.fin + i, 1);
    *b.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(b.tslot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *b.tslot;
  const int RT = (p.rows + kTileRows - 1) / kTileRows;
  const int nunits = p.ntiles[0] * RT;

  if (warp == 0) {
    if ((tid & 31) == 0) g_producer<NPROJ>(p, smem, b, RT, nunits);
  } else if (warp == 1) {
    if ((tid & 31) == 0) g_mma<NPROJ>(p, smem, b, tbase, RT, nunits, 0);
  } else if (warp >= kMma1) {
    if ((tid & 31) == 0) g_mma<NPROJ>(p, smem, b, tbase, RT, nunits, warp - kMma1 + 1);
  } else if (warp < kEpi0) {
    g_dequant<NPROJ, FMT>(p, smem, b, tbase, RT, nunits);
  } else {
    g_epilogue<NPROJ, FMT>(p, smem, b, tbase, RT, nunits);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// -------------------------------------------------------------------- host
int grouped_plan_gemm(GemmParams& g, int nproj, int smem_budget) {
  g.stage_bytes = nproj * kABox + 2 * kBBox;
  const int scb = ((nproj * kTileRows * g.sr) + 1023) / 1024 * 1024;
  g.sc_bytes = scb;
  const int bar_bytes = 1024;
  for (int nsc = 2; nsc >= 1; --nsc) {
    const int room = smem_budget - nsc * scb - bar_bytes;
    int ns = room / g.stage_bytes;
    ns = std::min(ns, 8);
    if (ns >= 2) {
      g.nscbuf = nsc;
      g.nstages = ns;
      g.off_sc = ns * g.stage_bytes;
      g.off_bar = g.off_sc + nsc * scb;
      return g.off_bar + bar_bytes;
    }
  }
  return 0;
}

cudaError_t grouped_set_smem(int smem_bytes) {
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<2, FMT_NVFP4>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<2, FMT_MXFP4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<1, FMT_NVFP4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_kernel<1, FMT_MXFP4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes);
  return e;
}

cudaError_t launch_grouped(const GroupedParams& gp, GemmParams gu, GemmParams gd, int grid,
                           int smem_gu, int smem_gd, cudaStream_t st) {
  const int S = gp.N * gp.k;
  const int rsmem = kRtTok * gp.H * 2;
  const dim3 rgrid((gp.N + kRtTok - 1) / kRtTok, (gp.E + kRtExp - 1) / kRtExp);
  grouped_router_kernel<<<rgrid, 256, rsmem, st>>>(gp);
  grouped_topk_kernel<<<(gp.N + 7) / 8, 256, 0, st>>>(gp);
  if (gp.route_only) return cudaGetLastError();
  grouped_plan_kernel<<<1, 1024, 0, st>>>(gp);
  grouped_gather_kernel<<<S, 128, 0, st>>>(gp);
  // gate/up: smem + 1024 for the manual 1024-byte alignment
  if (gp.fmt == FMT_NVFP4)
    grouped_gemm_kernel<2, FMT_NVFP4><<<grid, kGThreads, smem_gu + 1024, st>>>(gu);
  else
    grouped_gemm_kernel<2, FMT_MXFP4><<<grid, kGThreads, smem_gu + 1024, st>>>(gu);
  grouped_pack_kernel<<<S, 256, 0, st>>>(gp);
  if (gp.fmt == FMT_NVFP4)
    grouped_gemm_kernel<1, FMT_NVFP4><<<grid, kGThreads, smem_gd + 1024, st>>>(gd);
  else
    grouped_gemm_kernel<1, FMT_MXFP4><<<grid, kGThreads, smem_gd + 1024, st>>>(gd);
  grouped_combine_kernel<<<gp.N, 256, 0, st>>>(gp);
  return cudaGetLastError();
}

}  // namespace moe
