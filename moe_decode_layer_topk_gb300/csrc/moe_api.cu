// C ABI of the MoE decode-layer forward (include/moe.h): argument checks,
// workspace carve-out, and the launch of the fused decode kernel.
//
// Checks follow the pages' rule of refusing an unsupported case by name
// rather than computing a wrong result (forward_k3.rs, the zero-expert guard) and the scratch-size check of
// forward_atomic_c4.rs: every refusal returns a status before anything is
// enqueued.

#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

constexpr int32_t kAbiVersion = 3;
constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The stream kernel's cross-CTA words (router logits, the routed
// intermediate h, shared-expert readiness flags and part counters) are 64-bit
// words tagged with the call number,
// in a region right after the control block that no other path writes and
// that the stream kernel writes only with such words, so no stale word can
// look current whatever shapes ran before.  Its layout depends on the layer
// alone (sized for kSkMaxTok rows), not on N.
struct TaggedLayout {
  size_t logits, hw, sflag, scnt, total;
};

TaggedLayout tagged_layout(const moe_layer_desc_t& d) {
  TaggedLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  const size_t Ts = (size_t)std::max(d.shared_inter, 0) / 16;
  L.logits = take((size_t)moe::kSkMaxTok * (d.E + d.zero_experts) * 8);
  L.hw = take((size_t)moe::kSkMaxTok * d.top_k * (d.inter / 2) * 8);
  L.sflag = take(Ts * 8);
  L.scnt = take(Ts * 8);
  L.total = off;
  return L;
}

size_t tagged_bytes(const moe_layer_desc_t& d) { return tagged_layout(d).total; }

// Workspace of the stream kernel (FP4 experts, N <= kSkMaxTok).
struct SWsLayout {
  size_t ctrl, tagged, hs, shpart, oacc, total;
};

SWsLayout sws_layout(const moe_layer_desc_t& d, int32_t N) {
  SWsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  const size_t Ts = (size_t)std::max(d.shared_inter, 0) / 16;
  L.ctrl = take(256);
  L.tagged = take(tagged_bytes(d));
  L.hs = take((size_t)N * std::max(d.shared_inter, 0) * 2);
  // K parts x tiles <= the grid (at most kSkMaxGrid CTAs)
  L.shpart = take(Ts ? (size_t)std::max<size_t>(Ts, moe::kSkMaxGrid) * 256 * 4 : 0);
  L.oacc = take((size_t)d.H * ((N + 1) & ~1) * 4);
  L.total = off;
  return L;
}

struct WsLayout {
  size_t ctrl, logits, x16, xexp, gsig, h16, hexp, hs, ready, total;
};

WsLayout ws_layout(const moe_layer_desc_t& d, int32_t N) {
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  L.ctrl = take(256);
  take(tagged_bytes(d));
  L.logits = take((size_t)N * (d.E + d.zero_experts) * 4);
  L.x16 = take((size_t)N * d.H * 2);
  L.xexp = take((size_t)N * 4);
  L.gsig = take((size_t)N * 4);
  const size_t S = (size_t)N * d.top_k;
  L.h16 = take(S * d.inter * 2);
  L.hexp = take(S * (size_t)(((d.inter / 16) + 15) / 16 * 16));   // units <= S
  L.hs = take((size_t)N * std::max(d.shared_inter, 0) * 2);
  L.ready = take((size_t)(moe::kMaxSlots + 1) * 4);
  L.total = off;
  return L;
}

// Workspace of the grouped (many-token) path.  The control block sits at the
// same offset as in the decode layout so moe_get_error reads both.
struct GWsLayout {
  size_t ctrl, logits, xexp, sel_e, sel_w, tiles, ntiles, pos_of, tok_of, w_of, bexp, hexp, xg,
      hbuf, h16, total;
};

GWsLayout gws_layout(const moe_layer_desc_t& d, int32_t N) {
  GWsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  const size_t S = (size_t)N * d.top_k;
  const size_t T = S / moe::kGTileTok + std::min((size_t)d.E, S) + 1;   // token tiles, bound
  L.ctrl = take(256);
  take(tagged_bytes(d));
  L.logits = take((size_t)N * d.E * 4);
  L.xexp = take((size_t)N * 4);
  L.sel_e = take(S * 4);
  L.sel_w = take(S * 4);
  L.tiles = take(T * 3 * 4);
  L.ntiles = take(4);
  L.pos_of = take(S * 4);
  L.tok_of = take(S * 4);
  L.w_of = take(S * 4);
  L.bexp = take(S * 4);
  L.hexp = take(S * 4);
  L.xg = take(S * d.H * 2);
  L.hbuf = take(S * std::max(d.inter, d.H) * 4);
  L.h16 = take(S * d.inter * 2);
  L.total = off;
  return L;
}

// Layers the grouped path runs: FP4 experts, no shared expert, no zero
// experts, no hash routing.
bool grouped_capable(const moe_layer_desc_t& d) {
  return (d.wfmt == MOE_W_NVFP4 || d.wfmt == MOE_W_MXFP4) && d.shared_inter == 0 &&
         d.zero_experts == 0 && d.hash_vocab == 0;
}

// The decode kernel takes up to kMaxSlots (token, slot) pairs.  Layers the
// grouped path runs, with experts of at least kGroupedMinExpertBytes, take it
// for every N beyond the stream kernel's kSkMaxTok rows: measured on GB300
// (decode kernel against grouped path, layer copies cycled past L2), the
// grouped GEMMs win from N = 9 on (gpt-oss shape 414 / 254 us at N = 9,
// 677 / 377 us at N = 16, 2045 / 750 us at N = 64; Qwen3 shape 125 / 119 us
// at N = 9, 188 / 146 us at N = 16).  moe_debug_set_grouped_min_slots
// replaces the rule by a (token, slot) pair threshold.  Monotone in N, so a
// workspace sized for max_tokens covers every smaller N.
constexpr double kGroupedMinExpertBytes = 1024.0 * 1024.0;
long long g_grouped_min_slots = 0;   // 0: the N > kSkMaxTok rule

bool grouped_path(const moe_layer_desc_t& d, int32_t N) {
  const long long slots = (long long)N * d.top_k;
  if (!grouped_capable(d)) return false;   // run() splits such calls into row chunks
  if (slots > moe::kMaxSlots) return true;
  if (g_grouped_min_slots > 0 ? slots < g_grouped_min_slots : N <= moe::kSkMaxTok) return false;
  const double per_byte = 0.5 + (d.wfmt == MOE_W_NVFP4 ? 1.0 / 16 : 1.0 / 32);   // codes + scales
  return 3.0 * d.inter * d.H * per_byte >= kGroupedMinExpertBytes;
}

// Workspace bytes for any N <= max_tokens (decode layout up to the slot
// limit, grouped layout where grouped_path takes max_tokens).
size_t ws_total(const moe_layer_desc_t& d, int32_t max_tokens) {
  const int32_t ndec = std::min(max_tokens, (int32_t)(moe::kMaxSlots / d.top_k));
  size_t t = ndec >= 1 ? ws_layout(d, ndec).total : 0;
  if (grouped_path(d, max_tokens)) t = std::max(t, gws_layout(d, max_tokens).total);
  t = std::max(t, sws_layout(d, std::min(max_tokens, (int32_t)moe::kSkMaxTok)).total);
  return t;
}

moe_status_t check_desc(const moe_layer_desc_t* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->H <= 0 || d->inter <= 0 || d->E <= 0 || d->top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (d->scoring != MOE_SCORE_SOFTMAX && d->scoring != MOE_SCORE_SIGMOID_BIAS &&
      d->scoring != MOE_SCORE_SOFTMAX_BIAS)
    return MOE_ERR_INVALID_ARG;
  if (d->zero_experts < 0) return MOE_ERR_INVALID_ARG;
  if (d->hash_vocab < 0) return MOE_ERR_INVALID_ARG;
  if (d->hash_vocab > 0 && d->zero_experts > 0) return MOE_ERR_UNSUPPORTED;
  if (d->wfmt != MOE_W_NVFP4 && d->wfmt != MOE_W_MXFP4 && d->wfmt != MOE_W_BF16 &&
      d->wfmt != MOE_W_FP8)
    return MOE_ERR_INVALID_ARG;
  if (d->shared_inter < 0) return MOE_ERR_INVALID_ARG;
  if (d->router_fmt != MOE_R_BF16 && d->router_fmt != MOE_R_NVFP4) return MOE_ERR_INVALID_ARG;
  if (d->H % 32 || d->inter % 32 || d->shared_inter % 32) return MOE_ERR_UNSUPPORTED;
  if (d->E + d->zero_experts > moe::kMaxE || d->top_k > d->E + d->zero_experts ||
      d->top_k > moe::kMaxTopK)
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t check_weights(const moe_layer_desc_t* d, const moe_weights_t* w) {
  if (!w) return MOE_ERR_INVALID_ARG;
  const void* req[] = {w->router, w->gate_q, w->up_q, w->down_q};
  for (const void* p : req)
    if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  if (d->wfmt != MOE_W_BF16) {   // BF16 experts have no block scales
    const void* sc[] = {w->gate_s, w->up_s, w->down_s};
    for (const void* p : sc)
      if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
  }
  if (d->scoring != MOE_SCORE_SOFTMAX && !w->bias) return MOE_ERR_INVALID_ARG;
  if (d->router_fmt == MOE_R_NVFP4 && (!w->router_s || !aligned16(w->router_s)))
    return MOE_ERR_INVALID_ARG;
  if (d->hash_vocab > 0 && !w->tid2eid) return MOE_ERR_INVALID_ARG;
  if (d->shared_inter > 0) {
    const void* sh[] = {w->sh_gate, w->sh_up, w->sh_down};
    for (const void* p : sh)
      if (!p || !aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (w->sh_gate_w && !aligned16(w->sh_gate_w)) return MOE_ERR_INVALID_ARG;
  } else if (w->sh_gate || w->sh_up || w->sh_down || w->sh_gate_w) {
    return MOE_ERR_INVALID_ARG;   // shared weights without a shared size
  }
  return MOE_OK;
}

struct DeviceInfo {
  int budget = 0;
  int grid = 0;
  bool ready = false;
};

std::mutex g_mu;
DeviceInfo g_dev[64];

moe_status_t device_info(int* budget, int* grid) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    di.budget = moe::decode_smem_budget(dev);
    if (di.budget <= 0) return MOE_ERR_CUDA;
    di.grid = moe::decode_grid(dev, di.budget);
    if (di.grid <= 0) return MOE_ERR_CUDA;
    if (moe::grouped_set_smem(di.budget + 1024) != cudaSuccess) return MOE_ERR_CUDA;
    if (moe::stream_set_smem(di.budget) != cudaSuccess) return MOE_ERR_CUDA;
    di.ready = true;
  }
  *budget = di.budget;
  *grid = di.grid;
  return MOE_OK;
}

unsigned long long g_timeout_ns = 1000000000ull;   // bounded waits: 1 s

// ------------------------------------------------------------ tensor maps
// 2D views of the weight tensors for the kernel's TMA loads: rows of `inner`
// bytes, `rows` rows, boxes of 32 rows x `box` bytes (128-byte swizzle when
// the box is a full 128-byte line).  Encodings are cached by their key.
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

struct TmKey {
  const void* ptr;
  uint64_t inner, rows;
  uint32_t box, box_rows;
  int swz;
  int promo;   // L2 promotion of the loads, bytes
  bool operator==(const TmKey& o) const {
    return ptr == o.ptr && inner == o.inner && rows == o.rows && box == o.box &&
           box_rows == o.box_rows && swz == o.swz && promo == o.promo;
  }
};
struct TmEntry {
  TmKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kTmCache = 64;
TmEntry g_tm_cache[kTmCache];
int g_tm_next = 0;

bool encode_2d(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box,
               int swz, uint32_t box_rows = moe::kRows,
               int promo = 256) {   // swz: 0 none, 64 or 128 (bytes); promo: 128 or 256 (bytes)
  const TmKey key{ptr, inner, rows, box, box_rows, swz, promo};
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& e : g_tm_cache)
    if (e.used && e.key == key) {
      *out = e.map;
      return true;
    }
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t boxd[2] = {box, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUtensorMap m;
  if (g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, boxd,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
               promo == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  TmEntry& e = g_tm_cache[g_tm_next];
  g_tm_next = (g_tm_next + 1) % kTmCache;
  e.key = key;
  e.map = m;
  e.used = true;
  *out = m;
  return true;
}

// 3D view of weight rows: [column of 128 bytes][row][byte], boxes of 4
// columns x brows rows x 128 bytes (128-byte swizzle); rows must be whole
// columns (kb % 128 == 0) so no box reaches past a row or the tensor.
bool encode_3d(CUtensorMap* out, const void* ptr, uint64_t kb, uint64_t rows, uint32_t brows) {
  constexpr uint32_t kKey3d = 0x3D3Du;   // cache key marker of the 3D views
  const TmKey key{ptr, kb, rows, kKey3d, brows, 128, 256};
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& e : g_tm_cache)
    if (e.used && e.key == key) {
      *out = e.map;
      return true;
    }
  if (!g_encode) return false;
  cuuint64_t dims[3] = {128, rows, kb / 128};
  cuuint64_t strides[2] = {kb, 128};
  cuuint32_t boxd[3] = {128, brows, (cuuint32_t)moe::kBoxesPerChunk};
  cuuint32_t es[3] = {1, 1, 1};
  CUtensorMap m;
  if (g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, boxd,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  TmEntry& e = g_tm_cache[g_tm_next];
  g_tm_next = (g_tm_next + 1) % kTmCache;
  e.key = key;
  e.map = m;
  e.used = true;
  *out = m;
  return true;
}

// Weight-row map of one projection (packed FP4 or BF16 bytes), boxes of
// g.brows rows; plus its 3D view when the stage loads whole chunks.
bool encode_rows(moe::Params& p, int slot, const void* ptr, const moe::Geo& g, uint64_t rows) {
  const bool sw = g.kb >= moe::kBoxBytes;
  if (!encode_2d(&p.tm[slot], ptr, (uint64_t)g.kb, rows, sw ? moe::kBoxBytes : (uint32_t)g.kb,
                 sw ? 128 : 0, (uint32_t)g.brows))
    return false;
  p.tm_valid |= 1u << slot;
  if (g.use3d) {
    const int s3 = slot == moe::TM_GQ ? moe::TM3_GQ : slot == moe::TM_UQ ? moe::TM3_UQ
                 : slot == moe::TM_DQ ? moe::TM3_DQ : slot == moe::TM_SG ? moe::TM3_SG
                 : slot == moe::TM_SU ? moe::TM3_SU : moe::TM3_SD;
    if (!encode_3d(&p.tm[s3], ptr, (uint64_t)g.kb, rows, (uint32_t)g.brows)) return false;
    p.tm_valid |= 1u << s3;
  }
  return true;
}

// Block-scale map of one projection (tensor-map scale mode only); 64-byte box
// rows are swizzled so the kernel's per-lane scale loads avoid bank conflicts.
bool encode_scales(moe::Params& p, int slot, const void* ptr, const moe::Geo& g, uint64_t rows) {
  if (g.scale_mode != moe::SCALES_TMAP) return true;
  if (!encode_2d(&p.tm[slot], ptr, (uint64_t)g.sr, rows, (uint32_t)g.scb, g.scb == 64 ? 64 : 0,
                 (uint32_t)g.brows))
    return false;
  p.tm_valid |= 1u << slot;
  return true;
}

// Grouped path: router/top-k, plan, gather, gate/up GEMM, pack, down GEMM,
// combine (grouped_kernel.cu).  Arguments are already checked.
template <class Head>
moe_status_t run_grouped(const moe_layer_desc_t* d, const moe_weights_t* w, const void* x,
                         int32_t N, void* out, int32_t* topk_idx, float* topk_w, void* ws,
                         size_t ws_bytes, void* stream, int route_only, Head head) {
  if (d->shared_inter > 0) return MOE_ERR_UNSUPPORTED;   // shared expert: decode sizes only
  if (d->wfmt == MOE_W_BF16 || d->wfmt == MOE_W_FP8)
    return MOE_ERR_UNSUPPORTED;   // BF16 / FP8 experts: decode sizes only
  if (d->zero_experts > 0) return MOE_ERR_UNSUPPORTED;   // zero experts: decode sizes only
  if (d->hash_vocab > 0) return MOE_ERR_UNSUPPORTED;     // hash routing: decode sizes only
  const GWsLayout L = gws_layout(*d, N);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int budget = 0, grid = 0;
  moe_status_t st = device_info(&budget, &grid);
  if (st != MOE_OK) return st;
  if ((size_t)8 * d->H * 2 > (size_t)budget) return MOE_ERR_UNSUPPORTED;

  uint8_t* b = static_cast<uint8_t*>(ws);
  moe::GroupedParams gp;
  memset(&gp, 0, sizeof(gp));
  gp.N = N;
  gp.H = d->H;
  gp.inter = d->inter;
  gp.E = d->E;
  gp.k = d->top_k;
  gp.scoring = d->scoring;
  gp.norm = d->norm_topk_prob ? 1 : 0;
  gp.rsf = d->routed_scaling_factor;
  gp.fmt = d->wfmt;
  gp.route_only = route_only;
  gp.x = static_cast<const uint16_t*>(x);
  gp.router = static_cast<const uint16_t*>(w->router);
  gp.router_fmt = d->router_fmt;
  gp.router_s = d->router_fmt == MOE_R_NVFP4 ? w->router_s : nullptr;
  gp.router_s2 = d->router_fmt == MOE_R_NVFP4 ? w->router_s2 : nullptr;
  gp.bias = d->scoring != MOE_SCORE_SOFTMAX ? w->bias : nullptr;
  gp.topk_idx = topk_idx;
  gp.topk_w = topk_w;
  gp.out = static_cast<uint16_t*>(out);
  gp.logits = reinterpret_cast<float*>(b + L.logits);
  gp.xexp = reinterpret_cast<int*>(b + L.xexp);
  gp.sel_e = reinterpret_cast<int*>(b + L.sel_e);
  gp.sel_w = reinterpret_cast<float*>(b + L.sel_w);
  gp.tiles = reinterpret_cast<int*>(b + L.tiles);
  gp.ntiles = reinterpret_cast<int*>(b + L.ntiles);
  gp.pos_of = reinterpret_cast<int*>(b + L.pos_of);
  gp.tok_of = reinterpret_cast<int*>(b + L.tok_of);
  gp.w_of = reinterpret_cast<float*>(b + L.w_of);
  gp.bexp = reinterpret_cast<int*>(b + L.bexp);
  gp.hexp = reinterpret_cast<int*>(b + L.hexp);
  gp.xg = reinterpret_cast<uint16_t*>(b + L.xg);
  gp.hbuf = reinterpret_cast<float*>(b + L.hbuf);
  gp.h16 = reinterpret_cast<uint16_t*>(b + L.h16);

  const int gs = d->wfmt == MOE_W_NVFP4 ? 16 : 32;
  const uint64_t S = (uint64_t)N * d->top_k;
  moe::GemmParams gu, gd;
  memset(&gu, 0, sizeof(gu));
  memset(&gd, 0, sizeof(gd));
  uint32_t* err = &reinterpret_cast<moe::Ctrl*>(b + L.ctrl)->error;
  int smem_gu = 0, smem_gd = 0;
  if (!route_only) {
    gu.sc[0] = w->gate_s;
    gu.sc[1] = w->up_s;
    gu.s2[0] = w->gate_s2;
    gu.s2[1] = w->up_s2;
    gu.tiles = gp.tiles;
    gu.ntiles = gp.ntiles;
    gu.bexp = gp.bexp;
    gu.wpos = nullptr;
    gu.out = gp.hbuf;
    gu.err = err;
    gu.rows = d->inter;
    gu.K = d->H;
    gu.sr = d->H / gs;
    gu.timeout_ns = g_timeout_ns;
    gd = gu;
    gd.sc[0] = w->down_s;
    gd.sc[1] = nullptr;
    gd.s2[0] = w->down_s2;
    gd.s2[1] = nullptr;
    gd.bexp = gp.hexp;
    gd.wpos = gp.w_of;
    gd.rows = d->H;
    gd.K = d->inter;
    gd.sr = d->inter / gs;
    smem_gu = moe::grouped_plan_gemm(gu, 2, budget);
    smem_gd = moe::grouped_plan_gemm(gd, 1, budget);
    if (!smem_gu || !smem_gd) return MOE_ERR_UNSUPPORTED;
    // at least half of the SM's shared memory, so one CTA (and one TMEM
    // allocation of all 512 columns) per SM
    smem_gu = std::max(smem_gu, budget / 2 + 1024);
    smem_gd = std::max(smem_gd, budget / 2 + 1024);
    const uint64_t ER = (uint64_t)d->E;
    bool ok = encode_2d(&gu.tmA[0], w->gate_q, (uint64_t)d->H / 2, ER * d->inter, 64, 64, 128) &&
              encode_2d(&gu.tmA[1], w->up_q, (uint64_t)d->H / 2, ER * d->inter, 64, 64, 128) &&
              encode_2d(&gu.tmB, gp.xg, (uint64_t)d->H * 2, S, 128, 128, 64) &&
              encode_2d(&gd.tmA[0], w->down_q, (uint64_t)d->inter / 2, ER * d->H, 64, 64, 128) &&
              encode_2d(&gd.tmB, gp.h16, (uint64_t)d->inter * 2, S, 128, 128, 64);
    if (!ok) return MOE_ERR_CUDA;
  }
  st = head();
  if (st != MOE_OK) return st;
  if (moe::launch_grouped(gp, gu, gd, grid, smem_gu, smem_gd,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// Layers the stream kernel takes: FP4 experts, BF16 router, no zero experts,
// no hash routing; up to kSkMaxTok rows.
bool stream_capable(const moe_layer_desc_t& d, int32_t N) {
  return (d.wfmt == MOE_W_NVFP4 || d.wfmt == MOE_W_MXFP4) && d.router_fmt == MOE_R_BF16 &&
         d.zero_experts == 0 && d.hash_vocab == 0 && N >= 1 && N <= moe::kSkMaxTok;
}

// Fills the stream kernel's parameters; false if the shape does not fit it.
bool stream_params(moe::StreamParams& p, const moe_layer_desc_t* d, const moe_weights_t* w,
                   const void* x, int32_t N, void* out, int32_t* topk_idx, float* topk_w,
                   void* ws, int route_only, int budget, int grid) {
  memset(&p, 0, sizeof(p));
  p.H = d->H;
  p.inter = d->inter;
  p.E = d->E;
  p.k = d->top_k;
  p.scoring = d->scoring;
  p.norm = d->norm_topk_prob ? 1 : 0;
  p.rsf = d->routed_scaling_factor;
  p.fmt = d->wfmt;
  p.N = N;
  p.Is = d->shared_inter;
  p.route_only = route_only;
  p.router = static_cast<const uint16_t*>(w->router);
  p.bias = d->scoring != MOE_SCORE_SOFTMAX ? w->bias : nullptr;
  p.gq = w->gate_q;
  p.uq = w->up_q;
  p.dq = w->down_q;
  p.gsc = w->gate_s;
  p.usc = w->up_s;
  p.dsc = w->down_s;
  p.g2 = w->gate_s2;
  p.u2 = w->up_s2;
  p.d2 = w->down_s2;
  if (d->shared_inter > 0) {
    p.shg = static_cast<const uint16_t*>(w->sh_gate);
    p.shu = static_cast<const uint16_t*>(w->sh_up);
    p.shd = static_cast<const uint16_t*>(w->sh_down);
    p.shw = static_cast<const uint16_t*>(w->sh_gate_w);
  }
  p.x = static_cast<const uint16_t*>(x);
  p.out = static_cast<uint16_t*>(out);
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  const SWsLayout L = sws_layout(*d, N);
  uint8_t* b = static_cast<uint8_t*>(ws);
  p.ctrl = reinterpret_cast<moe::Ctrl*>(b + L.ctrl);
  const TaggedLayout T = tagged_layout(*d);
  p.logits = reinterpret_cast<unsigned long long*>(b + L.tagged + T.logits);
  p.hw = reinterpret_cast<unsigned long long*>(b + L.tagged + T.hw);
  p.sflag = reinterpret_cast<unsigned long long*>(b + L.tagged + T.sflag);
  p.scnt = reinterpret_cast<unsigned long long*>(b + L.tagged + T.scnt);
  p.hs = reinterpret_cast<uint16_t*>(b + L.hs);
  p.shpart = reinterpret_cast<float*>(b + L.shpart);
  p.oacc = reinterpret_cast<float*>(b + L.oacc);
  p.timeout_ns = g_timeout_ns;
  if (!moe::plan_stream(p, budget, grid)) return false;
  // weight codes by TMA: gate / up rows [E*inter, H/2] (16-row boxes), down
  // rows [E*H, inter/2] (32-row boxes), the shared down rows [H, 2*Is] bytes
  const uint64_t E = (uint64_t)d->E;
  // Long down lists (at least 8 items per warp at the N * k upper bound on
  // the units) with an even number of 128-column segments per unit run in
  // the paired order: warp pairs read the down rows in 128-byte pieces, so
  // the L2 promotion is the piece, not beyond it.  Short lists keep the
  // plain order, whose partner segments already run at about the same time.
  const long long sd = (d->inter + 127) / 128, mt = d->H / 32;
  p.dpair = sd % 2 == 0 && (d->shared_inter / 32) % 2 == 0 &&
            (long long)N * d->top_k * sd * mt >= 8LL * grid * moe::kSkWarps;
  const int dpromo = p.dpair ? 128 : 256;
  if (!encode_2d(&p.tm_gq, w->gate_q, d->H / 2, E * d->inter, 64, 0, 16) ||
      !encode_2d(&p.tm_uq, w->up_q, d->H / 2, E * d->inter, 64, 0, 16) ||
      !encode_2d(&p.tm_dq, w->down_q, d->inter / 2, E * d->H, 64, 0, 32, dpromo))
    return false;
  if (d->shared_inter > 0 &&
      !encode_2d(&p.tm_shd, w->sh_down, 2 * (uint64_t)d->shared_inter, d->H, 64, 0, 32, dpromo))
    return false;
  // block scales by TMA where each scale row is a multiple of 16 bytes,
  // otherwise by per-lane 4-byte copies
  const int gs = d->wfmt == MOE_W_NVFP4 ? 16 : 32;
  const uint64_t shb = d->H / gs, sib = d->inter / gs;
  p.sc_tma = shb % 16 == 0 && sib % 16 == 0 &&
             encode_2d(&p.tm_gs, w->gate_s, shb, E * d->inter, 16, 0, 16) &&
             encode_2d(&p.tm_us, w->up_s, shb, E * d->inter, 16, 0, 16) &&
             encode_2d(&p.tm_ds, w->down_s, sib, E * d->H, 16, 0, 32);
  return true;
}

moe_status_t run(const moe_layer_desc_t* d, const moe_weights_t* w, const void* x, int32_t N,
                 void* out, int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                 void* stream, int route_only, const int32_t* token_ids = nullptr,
                 bool clear_head = false) {
  moe_status_t st = check_desc(d);
  if (st != MOE_OK) return st;
  st = check_weights(d, w);
  if (st != MOE_OK) return st;
  // hash routing needs the call's token ids, and only hash routing takes them
  if ((d->hash_vocab > 0) != (token_ids != nullptr)) return MOE_ERR_INVALID_ARG;
  if (N < 1) return MOE_ERR_INVALID_ARG;
  if (!x || !aligned16(x) || !ws || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (!route_only && (!out || !aligned16(out))) return MOE_ERR_INVALID_ARG;
  if (route_only && (!topk_idx || !topk_w)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_total(*d, N)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  // clear_head: the built-in scratch of moe_forward_noalloc restarts its
  // call counter and tagged logits each call, once every check has passed
  auto head = [&]() -> moe_status_t {
    if (!clear_head) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, 24, s) != cudaSuccess) return MOE_ERR_CUDA;   // call counters
    if (cudaMemsetAsync(static_cast<uint8_t*>(ws) + 256, 0, tagged_bytes(*d), s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  };
  if ((long long)N * d->top_k > moe::kMaxSlots && !grouped_capable(*d)) {
    // layers the grouped path does not take (a shared expert, BF16 / FP8
    // experts, zero experts, hash routing): the fused kernels in row chunks
    // of kMaxSlots / top_k tokens, one after another on the stream (each
    // chunk streams its experts again)
    const int32_t C = moe::kMaxSlots / d->top_k;
    for (int32_t n0 = 0; n0 < N; n0 += C) {
      const int32_t nc = std::min(C, N - n0);
      const size_t xo = (size_t)n0 * d->H, so = (size_t)n0 * d->top_k;
      st = run(d, w, static_cast<const uint16_t*>(x) + xo, nc,
               out ? static_cast<uint16_t*>(out) + xo : nullptr, topk_idx ? topk_idx + so : nullptr,
               topk_w ? topk_w + so : nullptr, ws, ws_bytes, stream, route_only,
               token_ids ? token_ids + n0 : nullptr, clear_head);
      if (st != MOE_OK) return st;
    }
    return MOE_OK;
  }
  if (grouped_path(*d, N))
    return run_grouped(d, w, x, N, out, topk_idx, topk_w, ws, ws_bytes, stream, route_only, head);
  if (stream_capable(*d, N)) {
    if (ws_bytes < sws_layout(*d, N).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
    int budget = 0, grid = 0;
    moe_status_t st2 = device_info(&budget, &grid);
    if (st2 != MOE_OK) return st2;
    moe::StreamParams sp;
    if (stream_params(sp, d, w, x, N, out, topk_idx, topk_w, ws, route_only, budget, grid)) {
      st2 = head();
      if (st2 != MOE_OK) return st2;
      if (moe::launch_stream(sp, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_CUDA;
      return MOE_OK;
    }
  }
  const WsLayout L = ws_layout(*d, N);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;

  int budget = 0, grid = 0;
  st = device_info(&budget, &grid);
  if (st != MOE_OK) return st;

  moe::Params p;
  memset(&p, 0, sizeof(p));
  p.H = d->H;
  p.inter = d->inter;
  p.E = d->E;
  p.k = d->top_k;
  p.scoring = d->scoring;
  p.norm = d->norm_topk_prob ? 1 : 0;
  p.rsf = d->routed_scaling_factor;
  p.fmt = d->wfmt;
  p.Is = d->shared_inter;
  p.N = N;
  p.route_only = route_only;
  p.router = static_cast<const uint16_t*>(w->router);
  p.router_fmt = d->router_fmt;
  p.router_s = d->router_fmt == MOE_R_NVFP4 ? w->router_s : nullptr;
  p.router_s2 = d->router_fmt == MOE_R_NVFP4 ? w->router_s2 : nullptr;
  p.bias = d->scoring != MOE_SCORE_SOFTMAX ? w->bias : nullptr;
  p.Z = d->zero_experts;
  p.hash_V = d->hash_vocab;
  p.tid2eid = d->hash_vocab > 0 ? w->tid2eid : nullptr;
  p.token_ids = token_ids;
  // BF16 experts read no scales; FP8 experts their f32 block scales; only
  // the FP4 formats have scale2
  const bool scales = d->wfmt != MOE_W_BF16;
  const bool fp4 = d->wfmt == MOE_W_NVFP4 || d->wfmt == MOE_W_MXFP4;
  p.gsc = scales ? w->gate_s : nullptr;
  p.usc = scales ? w->up_s : nullptr;
  p.dsc = scales ? w->down_s : nullptr;
  p.g2 = fp4 ? w->gate_s2 : nullptr;
  p.u2 = fp4 ? w->up_s2 : nullptr;
  p.d2 = fp4 ? w->down_s2 : nullptr;
  p.shw = d->shared_inter > 0 ? static_cast<const uint16_t*>(w->sh_gate_w) : nullptr;
  p.x = static_cast<const uint16_t*>(x);
  p.out = static_cast<uint16_t*>(out);
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  uint8_t* b = static_cast<uint8_t*>(ws);
  p.ctrl = reinterpret_cast<moe::Ctrl*>(b + L.ctrl);
  p.logits = reinterpret_cast<float*>(b + L.logits);
  p.x16 = reinterpret_cast<uint16_t*>(b + L.x16);
  p.xexp = reinterpret_cast<int*>(b + L.xexp);
  p.gsig = reinterpret_cast<float*>(b + L.gsig);
  p.h16 = reinterpret_cast<uint16_t*>(b + L.h16);
  p.hexp = reinterpret_cast<int8_t*>(b + L.hexp);
  p.hs = reinterpret_cast<uint16_t*>(b + L.hs);
  p.ready = reinterpret_cast<uint32_t*>(b + L.ready);
  p.timeout_ns = g_timeout_ns;
  if (!moe::plan_decode(p, budget, grid)) return MOE_ERR_UNSUPPORTED;
  if (!route_only) {
    const uint64_t ER = (uint64_t)d->E;
    const moe::Geo& ga = p.geo[moe::KIND_AR];
    const moe::Geo& gb = p.geo[moe::KIND_BR];
    bool ok = encode_rows(p, moe::TM_GQ, w->gate_q, ga, ER * d->inter) &&
              encode_rows(p, moe::TM_UQ, w->up_q, ga, ER * d->inter) &&
              encode_rows(p, moe::TM_DQ, w->down_q, gb, ER * d->H) &&
              encode_scales(p, moe::TM_GS, w->gate_s, ga, ER * d->inter) &&
              encode_scales(p, moe::TM_US, w->up_s, ga, ER * d->inter) &&
              encode_scales(p, moe::TM_DS, w->down_s, gb, ER * d->H);
    if (ok && d->shared_inter > 0)
      ok = encode_rows(p, moe::TM_SG, w->sh_gate, p.geo[moe::KIND_AS], (uint64_t)d->shared_inter) &&
           encode_rows(p, moe::TM_SU, w->sh_up, p.geo[moe::KIND_AS], (uint64_t)d->shared_inter) &&
           encode_rows(p, moe::TM_SD, w->sh_down, p.geo[moe::KIND_BS], (uint64_t)d->H);
    if (!ok) return MOE_ERR_CUDA;
  }
  st = head();
  if (st != MOE_OK) return st;
  if (moe::launch_decode(p, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

// ---------------------------------------------------------------------------
// Built-in scratch for moe_forward_noalloc.  Some callers cannot allocate
// device memory at all (an allocator-free runtime, a plug-in that only
// receives input/output buffers, code that must not touch the CUDA memory
// pool); this array stands in for the caller workspace.  It is zero at module
// load, lives on every GPU that loads the library until the process exits,
// and is shared by every call on that GPU.  In host code its name is only a
// host-side stand-in: the device address is obtained with
// cudaGetSymbolAddress, once per device, with that device current.
constexpr size_t kNoAllocScratchBytes = 8u << 20;   // 8 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
// The address is looked up once per (device, CUDA context): a reset device or
// another context current on the device gets its own lookup.
struct NoallocEntry {
  CUcontext ctx;
  void* ptr;
};
NoallocEntry g_noalloc[64] = {};
PFN_cuCtxGetCurrent_v4000 g_ctx_get = nullptr;

moe_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  // make the runtime's context current for this thread before reading it
  if (cudaFree(nullptr) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_ctx_get) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return MOE_ERR_CUDA;
    g_ctx_get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get(&ctx) != CUDA_SUCCESS || !ctx) return MOE_ERR_CUDA;
  NoallocEntry& en = g_noalloc[dev];
  if (!en.ptr || en.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    en.ptr = p;
    en.ctx = ctx;
  }
  *out = en.ptr;
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_size(const moe_layer_desc_t* desc, int32_t max_tokens) {
  if (check_desc(desc) != MOE_OK || max_tokens < 1) return 0;
  return ws_total(*desc, max_tokens);
}

int32_t moe_uses_grouped_path(const moe_layer_desc_t* desc, int32_t N) {
  if (check_desc(desc) != MOE_OK || N < 1) return -1;
  return grouped_path(*desc, N) ? 1 : 0;
}

size_t moe_host_staging_size(const moe_layer_desc_t* desc, int32_t max_tokens) {
  if (check_desc(desc) != MOE_OK || max_tokens < 1) return 0;
  return 2 * align_up((size_t)max_tokens * desc->H * 2, kAlign);
}

moe_status_t moe_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || ws_bytes == 0) return MOE_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_forward(const moe_layer_desc_t* desc, const moe_weights_t* weights, const void* x,
                         int32_t N, void* out, int32_t* topk_idx, float* topk_w, void* workspace,
                         size_t ws_bytes, void* stream) {
  return run(desc, weights, x, N, out, topk_idx, topk_w, workspace, ws_bytes, stream, 0);
}

moe_status_t moe_forward_ids(const moe_layer_desc_t* desc, const moe_weights_t* weights,
                             const void* x, const int32_t* token_ids, int32_t N, void* out,
                             int32_t* topk_idx, float* topk_w, void* workspace, size_t ws_bytes,
                             void* stream) {
  if (!token_ids) return MOE_ERR_INVALID_ARG;
  return run(desc, weights, x, N, out, topk_idx, topk_w, workspace, ws_bytes, stream, 0,
             token_ids);
}

moe_status_t moe_route(const moe_layer_desc_t* desc, const moe_weights_t* weights, const void* x,
                       int32_t N, int32_t* topk_idx, float* topk_w, void* workspace,
                       size_t ws_bytes, void* stream) {
  return run(desc, weights, x, N, nullptr, topk_idx, topk_w, workspace, ws_bytes, stream, 1);
}

moe_status_t moe_forward_host(const moe_layer_desc_t* desc, const moe_weights_t* weights,
                              const void* x_host, int32_t N, void* out_host, void* workspace,
                              size_t ws_bytes, void* stream) {
  moe_status_t st = check_desc(desc);
  if (st != MOE_OK) return st;
  if (!x_host || !out_host || N < 1 || !workspace) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_workspace_size(desc, N);
  const size_t stage = align_up((size_t)N * desc->H * 2, kAlign);
  if (ws_bytes < need + 2 * stage) return MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* b = static_cast<uint8_t*>(workspace);
  void* xd = b + need;
  void* od = b + need + stage;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)N * desc->H * 2;
  if (cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  st = run(desc, weights, xd, N, od, nullptr, nullptr, workspace, need, stream, 0);
  if (st != MOE_OK) return st;
  if (cudaMemcpyAsync(out_host, od, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_get_error(void* workspace, void* stream) {
  if (!workspace) {   // the built-in scratch of moe_forward_noalloc on this device
    const moe_status_t st = noalloc_scratch(&workspace);
    if (st != MOE_OK) return st;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  uint32_t* err = &static_cast<moe::Ctrl*>(workspace)->error;
  if (cudaMemcpyAsync(&word, err, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (word == 0) return MOE_OK;
  if (cudaMemsetAsync(err, 0, 4, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return (word & ~moe::kErrRange) ? MOE_ERR_TIMEOUT : MOE_ERR_RANGE;
}

const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, N < 1 or misaligned buffer)";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or format";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than moe_workspace_size()";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "a bounded device-side wait expired";
    case MOE_ERR_RANGE: return "an expert activation exceeded the f16 range and was saturated";
  }
  return "unknown status";
}

int32_t moe_abi_version(void) { return kAbiVersion; }

/* moe_forward without a caller workspace: the scratch is the library's
 * built-in 8 MiB device array (see the declaration in moe.h). */
moe_status_t moe_forward_noalloc(const moe_layer_desc_t* desc, const moe_weights_t* weights,
                                 const void* x, int32_t N, void* out, int32_t* topk_idx,
                                 float* topk_w, void* stream) {
  moe_status_t st = check_desc(desc);
  if (st != MOE_OK) return st;
  st = check_weights(desc, weights);
  if (st != MOE_OK) return st;
  if (N < 1) return MOE_ERR_INVALID_ARG;
  if (!x || !aligned16(x) || !out || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (ws_total(*desc, N) > kNoAllocScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  st = noalloc_scratch(&ws);
  if (st != MOE_OK) return st;
  // the call counter and the tagged logits restart every call (enqueued by
  // run() once every check has passed); the kernels zero their own
  // accumulators and counters, and the error word stays sticky
  return run(desc, weights, x, N, out, topk_idx, topk_w, ws, kNoAllocScratchBytes, stream, 0,
             nullptr, true);
}

/* Test hook: budget of every bounded device wait, in nanoseconds, for calls
 * enqueued afterwards (default 1e9).  A budget of 0 makes any wait that is not
 * already satisfied expire at once, which exercises the MOE_ERR_TIMEOUT path
 * without hanging the GPU. */
void moe_debug_set_wait_budget_ns(unsigned long long ns) { g_timeout_ns = ns; }

/* Tuning hook: (token, slot) pairs from which layers with large FP4 experts
 * take the grouped path; slots <= 0 restores the built-in rule. */
void moe_debug_set_grouped_min_slots(int32_t slots) { g_grouped_min_slots = slots > 0 ? slots : 0; }

}  // extern "C"
