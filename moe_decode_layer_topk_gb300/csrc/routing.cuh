// Warp-level top-k routing of one token, shared by the decode and grouped
// kernels.  Scoring follows the gating step of the forward chain: softmax
// (selection by logit, weights softmax over all E, optionally renormalised
// over the selected), sigmoid + correction bias (selection by
// sigmoid(l) + bias, weights sigmoid(l) without the bias, optional
// renormalisation, then times the routed scaling factor), or softmax +
// correction bias (the zero-expert routers: selection by softmax(l) + bias,
// weights softmax(l), optional renormalisation, times the routed scaling
// factor).  Ties go to the lower expert index.
#pragma once
#include <math.h>
#include <stdint.h>

#include "ptx.cuh"

namespace moe {

// Eight router weights of row e, elements h .. h+7 (h a multiple of 8), as
// FP32: a BF16 router [E, H], or an NVFP4 router (E2M1 codes [E, H/2], element
// 2j in the low nibble; one E4M3 scale per 16 elements [E, H/16]; times the
// router's scale2).  E2M1 x E4M3 is exact in FP32.
__device__ __forceinline__ void router_w8(const uint16_t* router, int fmt, const uint8_t* rs,
                                          float s2, int H, int e, int h, float (&w)[8]) {
  if (fmt == 0) {
    const uint4 v = ld_nc_u4(router + (size_t)e * H + h);
    const uint32_t a[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[2 * i] = __uint_as_float(a[i] << 16);
      w[2 * i + 1] = __uint_as_float(a[i] & 0xFFFF0000u);
    }
  } else {
    const uint8_t* q = reinterpret_cast<const uint8_t*>(router) + (size_t)e * (H / 2) + h / 2;
    const uint32_t codes = __ldg(reinterpret_cast<const uint32_t*>(q));
    const uint32_t sb = __ldg(rs + (size_t)e * (H / 16) + h / 16);
    const float sc = f16x2_to_f32x2(e4m3x2_to_f16x2(sb)).x * s2;
    uint32_t o[4];
    e2m1x8_to_f16x2x4(codes, o);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = f16x2_to_f32x2(o[i]);
      w[2 * i] = f.x * sc;
      w[2 * i + 1] = f.y * sc;
    }
  }
}

// Selection key, order preserving as unsigned: larger key = larger score.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// lg[i] = logit of expert lane + 32*i (-inf where that index is >= E).  The k
// selections are k rounds of a warp arg-max; lane j < k returns selection j
// (expert and weight) in *e_out / *w_out, in selection order.  EXT = false
// compiles only the softmax and sigmoid + bias scorings (a smaller routine for
// the common layers).
template <int PER, bool EXT = true>
__device__ __forceinline__ void topk_warp(int E, int k, int scoring, int norm, float rsf,
                                          const float* bias, const float (&lg)[PER], int lane,
                                          int* e_out, float* w_out) {
  uint32_t key[PER];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (lane + 32 * i < E) mx = fmaxf(mx, lg[i]);
  float den = 0.f;
  // softmax max and denominator over all E: before the selection when the
  // keys need them (scoring 2), after it when only the weights do (scoring 0)
  auto softmax_den = [&]() {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (lane + 32 * i < E) den += expf(lg[i] - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  };
  if (EXT && scoring == 2) softmax_den();
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0u;
    if (e < E) {
      const float l = lg[i];
      const float sc = (scoring == 0) ? l
                     : (!EXT || scoring == 1) ? 1.0f / (1.0f + expf(-l)) + bias[e]
                                              : expf(l - mx) / den + bias[e];
      key[i] = order_key(sc);
    }
  }
  uint32_t bk = 0u, be = 0xFFFFFFFFu;   // lane-local best, lowest index among equals
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (key[i] > bk) { bk = key[i]; be = lane + 32 * i; }
  uint32_t mine = 0u;                   // lane j: expert of selection j
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
    uint32_t we = __reduce_min_sync(0xffffffffu, (bk == m) ? be : 0xFFFFFFFFu);
    if (we >= (uint32_t)E) we = 0;      // only if fewer than k valid keys (k <= E is checked)
    if (lane == j) mine = we;
    if ((we & 31u) == (uint32_t)lane) {
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (lane + 32 * i == (int)we) key[i] = 0u;
      bk = 0u;
      be = 0xFFFFFFFFu;
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (key[i] > bk) { bk = key[i]; be = lane + 32 * i; }
    }
  }
  if (scoring == 0) softmax_den();
  // logit of this lane's selection, from the lane that holds it
  float l = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const float v = __shfl_sync(0xffffffffu, lg[i], mine & 31u);
    if ((int)(mine >> 5) == i) l = v;
  }
  float w = 0.f;
  if (lane < k) w = (scoring != 1) ? expf(l - mx) / den : 1.0f / (1.0f + expf(-l));
  float wsum = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  if (lane < k) {
    if (norm) w = w / wsum;
    if (scoring != 0) w *= rsf;
    *e_out = (int)mine;
    *w_out = w;
  }
}

// Hash routing of one token: the k experts are `row` (the token id's row of
// the tid2eid table, in table order; ids clamped into [0, E)); their weights
// follow the scoring as in topk_warp (softmax over all E for scorings 0 and 2,
// sigmoid for 1; renormalised if asked; times rsf unless plain softmax).
// Lane j < k returns slot j in *e_out / *w_out.
template <int PER>
__device__ __forceinline__ void hash_warp(int E, int k, int scoring, int norm, float rsf,
                                          const int32_t* row, const float (&lg)[PER], int lane,
                                          int* e_out, float* w_out) {
  float mx = -INFINITY, den = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (lane + 32 * i < E) mx = fmaxf(mx, lg[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (lane + 32 * i < E) den += expf(lg[i] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  int e = 0;
  if (lane < k) e = min(max(__ldg(row + lane), 0), E - 1);
  float l = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const float v = __shfl_sync(0xffffffffu, lg[i], e & 31);
    if ((e >> 5) == i) l = v;
  }
  float w = 0.f;
  if (lane < k) w = (scoring == 1) ? 1.0f / (1.0f + expf(-l)) : expf(l - mx) / den;
  float wsum = w;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  if (lane < k) {
    if (norm) w = w / wsum;
    if (scoring != 0) w *= rsf;
    *e_out = e;
    *w_out = w;
  }
}

}  // namespace moe
