/*
 * moe.h — C ABI of the GB300 (sm_103a) mixture-of-experts decode-layer forward.
 *
 * One call computes, for N token rows x[N,H] (BF16):
 *   1. router logits   l[n,e] = x[n,:] . Wr[e,:]                 (FP32 accumulate)
 *                      with a BF16 router, or an NVFP4 router
 *                      (Wr = E2M1(code) * E4M3 scale per 16 * scale2);
 *   2. top-k routing   softmax (optionally renormalised over the selected k)
 *                      or sigmoid + correction bias for selection, sigmoid
 *                      for the weights, optional renormalisation, times the
 *                      routed scaling factor; or softmax + correction bias
 *                      (the zero-expert routers) likewise; with Z zero
 *                      experts the router has E + Z outputs and a selected
 *                      zero expert runs no expert; or hash routing: the k
 *                      experts of a token are the tid2eid row of its token
 *                      id, weighted by the scoring of their logits;
 *   3. routed experts  SwiGLU with block-scaled FP4 weights:
 *                      h = SiLU(Dq(Wg) x) * (Dq(Wu) x),  y = Dq(Wd) h,
 *                      Dq(w) = E2M1(code) * blockscale * scale2;
 *                      or with plain BF16 weights (Dq(w) = w), or with
 *                      FP8 weights (Dq(w) = E4M3(code) * blockscale, one
 *                      FP32 scale per 128 x 128 block);
 *   4. output          out[n] = BF16( sum_j w[n,j] * y_{idx[n,j]}
 *                                     + g_s(x_n) * shared(x_n) ),
 *                      g_s = sigmoid(w_s . x_n) if a shared-expert gate vector
 *                      is given, 1 if not; no shared term without a shared
 *                      expert.
 *
 * The layer follows the MoE forward of the pages this library is built from:
 *   - forward_k3.rs (MoeLayer::forward_k3): the step chain "gate GEMV ->
 *     batched topK -> expert gate+up -> silu+down -> weighted sum + blend", the
 *     batched top-k calls (moe_topk_sigmoid_batched with bias, norm_topk_prob
 *     and routed_scaling_factor; moe_topk_softmax_batched with norm_topk_prob),
 *     the per-expert weight tables (packed_ptrs, scale_ptrs, scale2_vals), the
 *     GS16/E4M3 vs GS32/E8M0 scale formats (the E8M0 guard), and the shared
 *     expert blend (null shared_expert_gate -> residual add, else sigmoid gate);
 *   - forward_atomic_c4.rs (forward_atomic_c4_decode): routing-weighted FP32
 *     accumulation of the routed down projections, then a BF16 cast and the
 *     shared-expert blend; the scratch carve-out and its size check;
 *   - forward_batched.rs: one router GEMM for N rows, per-token routing, and
 *     every routed and shared expert's weights read in one pass for all rows;
 *     its BF16 expert branch (bf16 gate/up/down weight pointers, the same
 *     kernels as the FP4 forward) for the BF16 routed-expert format, and the
 *     FP8 expert branch (weight_ptrs + scale_ptrs of moe_expert_gate_up_
 *     shared_fp8 / moe_expert_silu_down_shared_fp8).  The pages do not give the
 *     FP8 scale granularity; this library takes one FP32 scale per 128 x 128
 *     block of each projection.
 *
 * Memory: every pointer passed to moe_forward / moe_route is a DEVICE pointer
 * (weights, x, out, topk outputs, workspace) unless the name says _host.  The
 * caller owns all buffers.  The library never allocates device memory and
 * never synchronises inside moe_forward/moe_route: work is enqueued on the
 * given stream (a cudaStream_t passed as void*; NULL = legacy default stream).
 *
 * Weight layout (canonical, row-major, K contiguous):
 *   router     [E + Z, H]      bf16 (Z = zero experts, usually 0)
 *   bias       [E + Z]         f32, the bias scorings only (NULL otherwise)
 *   gate_q     [E, inter, H/2] u8  two E2M1 codes per byte, element 2j in the
 *   up_q       [E, inter, H/2] u8  low nibble, 2j+1 in the high nibble
 *   down_q     [E, H, inter/2] u8
 *   gate_s     [E, inter, H/gs]   u8  block scales along K (the input dim),
 *   up_s       [E, inter, H/gs]   u8  gs = 16 (E4M3, NVFP4) or 32 (E8M0, MXFP4)
 *   down_s     [E, H, inter/gs]   u8
 *   gate_s2, up_s2, down_s2 [E] f32 per-expert global scale (NULL = 1.0)
 * BF16 routed experts (wfmt MOE_W_BF16): gate_q, up_q [E, inter, H] bf16 and
 *   down_q [E, H, inter] bf16; the scale pointers and *_s2 are not read (NULL
 *   allowed).
 * NVFP4 router (router_fmt MOE_R_NVFP4, the pages' gate_nvfp4 into the w4a16
 *   GEMV of forward_k3.rs step 1): router points to E2M1 codes [E, H/2] u8,
 *   router_s to E4M3 scales [E, H/16] u8, router_s2 to one f32 scale2 (NULL =
 *   1.0).
 * FP8 routed experts (wfmt MOE_W_FP8): gate_q, up_q [E, inter, H] and down_q
 *   [E, H, inter] E4M3 bytes (OCP "fn"); gate_s, up_s point to f32
 *   [E, ceil(inter/128), ceil(H/128)] and down_s to f32 [E, ceil(H/128),
 *   ceil(inter/128)] block scales; *_s2 are not read.
 *   sh_gate, sh_up [Is, H] bf16; sh_down [H, Is] bf16  (NULL when Is == 0)
 *   sh_gate_w  [H] bf16 or NULL (NULL = ungated, always-on shared expert)
 * All weight, x, out and workspace pointers must be 16-byte aligned.
 */
#ifndef MOE_DECODE_LAYER_TOPK_GB300_MOE_H
#define MOE_DECODE_LAYER_TOPK_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  A refusal names what is wrong instead of computing a wrong
 * answer (the rule of forward_k3.rs's zero-expert guard). */
typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null required pointer, N < 1, bad alignment */
  MOE_ERR_UNSUPPORTED = 2,          /* shape/format outside what the kernels take */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < moe_workspace_size(desc, N) */
  MOE_ERR_CUDA = 4,                 /* a CUDA runtime call failed */
  MOE_ERR_TIMEOUT = 5,              /* a bounded device-side wait gave up */
  MOE_ERR_RANGE = 6                 /* an activation held as f16 exceeded +-65504 and was
                                       saturated (the result is not reliable) */
} moe_status_t;

typedef enum {
  MOE_SCORE_SOFTMAX = 0,        /* softmax; routed_scaling_factor not applied */
  MOE_SCORE_SIGMOID_BIAS = 1,   /* sigmoid + correction bias */
  MOE_SCORE_SOFTMAX_BIAS = 2    /* softmax + correction bias (zero-expert routers) */
} moe_scoring_t;
/* Routed-expert weight formats: NVFP4 (E2M1 + per-16 E4M3 scale + FP32
 * scale2), MXFP4 (E2M1 + per-32 E8M0 scale), BF16 (plain weights), FP8 (E4M3
 * + FP32 scale per 128 x 128 block). */
typedef enum { MOE_W_NVFP4 = 0, MOE_W_MXFP4 = 1, MOE_W_BF16 = 2, MOE_W_FP8 = 3 } moe_wfmt_t;
/* Router weight formats. */
typedef enum { MOE_R_BF16 = 0, MOE_R_NVFP4 = 1 } moe_rfmt_t;

/* Layer configuration: the config fields the pages' MoE forward reads
 * (hidden_size, moe_intermediate_size, num_experts, num_experts_per_tok,
 * norm_topk_prob, routed_scaling_factor, the expert scale kind, and
 * shared_expert_intermediate_size). */
typedef struct {
  int32_t H;                     /* hidden size, multiple of 32 */
  int32_t inter;                 /* routed expert intermediate size, multiple of 32 */
  int32_t E;                     /* number of routed experts, 1..1024 */
  int32_t top_k;                 /* experts per token, 1..min(E, 32) */
  int32_t scoring;               /* moe_scoring_t */
  int32_t norm_topk_prob;        /* 0/1: renormalise the selected weights */
  float routed_scaling_factor;   /* the bias scorings only; ignored for plain softmax */
  int32_t wfmt;                  /* moe_wfmt_t */
  int32_t shared_inter;          /* shared expert intermediate size; 0 = none */
  int32_t router_fmt;            /* moe_rfmt_t (0 = BF16 router) */
  int32_t zero_experts;          /* Z >= 0: router width E + Z (the pages' num_experts +
                                    zero_expert_num); E + Z <= 1024 */
  int32_t hash_vocab;            /* V > 0: hash routing with a [V, top_k] tid2eid table
                                    (forward_batched.rs, moe_hash_route); calls go
                                    through moe_forward_ids; needs zero_experts == 0 */
} moe_layer_desc_t;

typedef struct {
  const void* router;            /* bf16 [E, H], or E2M1 codes [E, H/2] (NVFP4 router) */
  const float* bias;             /* f32 [E + Z] (required iff the scoring has a bias) */
  const uint8_t* gate_q;
  const uint8_t* up_q;
  const uint8_t* down_q;
  const uint8_t* gate_s;
  const uint8_t* up_s;
  const uint8_t* down_s;
  const float* gate_s2;          /* NULL = 1.0 */
  const float* up_s2;
  const float* down_s2;
  const void* sh_gate;           /* bf16, NULL iff shared_inter == 0 */
  const void* sh_up;
  const void* sh_down;
  const void* sh_gate_w;         /* bf16 [H] or NULL (ungated) */
  const uint8_t* router_s;       /* NVFP4 router: E4M3 scales [E, H/16]; else NULL */
  const float* router_s2;        /* NVFP4 router: one f32 scale2, NULL = 1.0 */
  const int32_t* tid2eid;        /* hash routing: int32 [V, top_k] expert ids per token id
                                    (in [0, E)), else NULL */
} moe_weights_t;

/* Bytes of device workspace moe_forward needs for any 1 <= N <= max_tokens.
 * Returns 0 if the descriptor is invalid.  The workspace holds the router
 * logits, the routing table, the gate/up activations, the FP32 output
 * accumulator and the grid-barrier words (the scratch the pages carve out of
 * ctx.buffers.scratch() in forward_atomic_c4.rs); when max_tokens runs the
 * grouped path (see moe_forward) it also covers that path's expert-sorted
 * activation copies (about S * (2H + 4 max(H, inter) + 2 inter) bytes,
 * S = max_tokens * top_k). */
MOE_API size_t moe_workspace_size(const moe_layer_desc_t* desc, int32_t max_tokens);

/* The path moe_forward (and moe_route, moe_forward_ids, moe_forward_host)
 * takes for N token rows of this layer: 1 = the grouped path (eight
 * kernels: router, top-k, plan, gather, gate/up GEMM, pack, down GEMM,
 * combine; moe_route stops after the top-k), 0 = the fused kernels (the
 * stream or the decode kernel, one launch per row chunk), -1 = invalid
 * descriptor or N < 1.  Host-only: makes no CUDA call.  The rule is the one
 * moe_forward's description states. */
MOE_API int32_t moe_uses_grouped_path(const moe_layer_desc_t* desc, int32_t N);

/* Zero a workspace before its first use (and after MOE_ERR_TIMEOUT).  Enqueues
 * a memset on `stream`.  Afterwards moe_forward keeps the workspace's barrier
 * and error words consistent by itself. */
MOE_API moe_status_t moe_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* The layer forward for N token rows.
 *   x         bf16 [N, H] device
 *   out       bf16 [N, H] device, fully overwritten
 *   topk_idx  int32 [N, top_k] device or NULL: selected experts, in order of
 *             decreasing selection score (ties to the lower expert index)
 *   topk_w    f32 [N, top_k] device or NULL: their routing weights
 *   workspace device, >= moe_workspace_size(desc, N) bytes, zeroed once by
 *             moe_workspace_init; one workspace per concurrently running call
 * Paths: up to 8 token rows of a layer with NVFP4 / MXFP4 experts, a BF16
 * router, no zero experts and no hash routing run one cooperative stream
 * kernel (router, top-k, gate/up, SiLU, down and the shared-expert blend in
 * one launch); other layers with N*top_k <= 256 run one fused decode kernel;
 * N*top_k > 256 runs the grouped path (per-expert token groups on the tcgen05
 * tensor cores, the grouped GEMM forward_batched.rs switches to for larger
 * row counts).  Layers the grouped path runs (NVFP4 / MXFP4 experts, no
 * shared expert, no zero experts, no hash routing) whose experts hold >= 1 MiB
 * of weights (3 * inter * H * (1/2 + 1/gs) bytes) take it for every N > 8,
 * where it is the faster path.  The grouped path takes neither a shared
 * expert, BF16 / FP8 routed experts, zero experts nor hash routing yet: such
 * layers with N*top_k > 256 run the fused kernels in row chunks of
 * floor(256 / top_k) tokens, one after another on the stream (each chunk
 * reads its touched experts' weights again).  With zero experts, topk_idx
 * holds indices up to E + Z - 1 (>= E: a zero expert).  Asynchronous on `stream`; no host synchronisation,
 * no allocation, so it may be captured in a CUDA graph.  Argument errors are
 * returned before anything is enqueued; device-side timeouts are reported by
 * moe_get_error. */
MOE_API moe_status_t moe_forward(const moe_layer_desc_t* desc, const moe_weights_t* weights,
                         const void* x, int32_t N, void* out,
                         int32_t* topk_idx, float* topk_w,
                         void* workspace, size_t ws_bytes, void* stream);

/* moe_forward for a hash-routed layer (desc->hash_vocab > 0): token_ids is
 * int32 [N] device, the token ids of the rows of x (each clamped into
 * [0, hash_vocab)); token n's experts are tid2eid row token_ids[n] in table
 * order (ids outside [0, E) are clamped), weighted as top-k routing weights
 * are for the layer's scoring.  A hash-routed layer refuses moe_forward,
 * moe_route and the other entry points (MOE_ERR_INVALID_ARG: no token ids).
 * N*top_k > 256 runs in row chunks as moe_forward describes.  Otherwise as
 * moe_forward. */
MOE_API moe_status_t moe_forward_ids(const moe_layer_desc_t* desc, const moe_weights_t* weights,
                                     const void* x, const int32_t* token_ids, int32_t N,
                                     void* out, int32_t* topk_idx, float* topk_w,
                                     void* workspace, size_t ws_bytes, void* stream);

/* Router logits and top-k routing only (steps 1-2): writes topk_idx/topk_w
 * (both required).  Same constraints and ownership as moe_forward. */
MOE_API moe_status_t moe_route(const moe_layer_desc_t* desc, const moe_weights_t* weights,
                       const void* x, int32_t N, int32_t* topk_idx, float* topk_w,
                       void* workspace, size_t ws_bytes, void* stream);

/* End-to-end convenience call with HOST activations: copies x_host (bf16
 * [N,H], pinned memory recommended) to the device through the workspace,
 * runs moe_forward, copies the result to out_host and synchronises `stream`
 * before returning.  Weights and workspace stay device pointers.  Needs
 * moe_workspace_size(desc, N) + moe_host_staging_size(desc, N) bytes. */
MOE_API size_t moe_host_staging_size(const moe_layer_desc_t* desc, int32_t max_tokens);
MOE_API moe_status_t moe_forward_host(const moe_layer_desc_t* desc, const moe_weights_t* weights,
                              const void* x_host, int32_t N, void* out_host,
                              void* workspace, size_t ws_bytes, void* stream);

/* Sticky device-side error of a workspace: MOE_OK, MOE_ERR_TIMEOUT (a bounded
 * wait expired; re-initialise the workspace), or MOE_ERR_RANGE (the fused
 * decode kernel holds the routed experts' SiLU(g)*u, times the routing weight
 * and the down scale2, as f16; a value beyond +-65504 was saturated).
 * Enqueues a 4-byte read on `stream`, synchronises the stream, clears the
 * word, and returns the status of the calls that ran since the last check.
 * workspace == NULL reads the built-in scratch of moe_forward_noalloc on the
 * current device. */
MOE_API moe_status_t moe_get_error(void* workspace, void* stream);

/* Static description of a status code. */
MOE_API const char* moe_status_string(moe_status_t status);

/* Library version, for the binding to check it loaded the library it expects. */
MOE_API int32_t moe_abi_version(void);

/* moe_forward for callers that cannot allocate device memory.  Some callers
 * have no way to obtain a workspace: an allocator-free embedded runtime, a
 * plug-in that is handed only its input and output buffers, or code that must
 * not call cudaMalloc or touch a framework's memory pool.  This entry point
 * computes exactly what moe_forward computes (same arguments minus the
 * workspace, same constraints, same outputs) but runs in a fixed 8 MiB scratch
 * array that the library keeps in device memory (a file-scope __device__
 * array: every GPU that loads the library holds it until the process exits).
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 *   - A shape whose moe_workspace_size(desc, N) exceeds 8 MiB is refused with
 *     MOE_ERR_WORKSPACE_TOO_SMALL; use moe_forward with a caller workspace.
 *   - The first call on a device (and the first after the current CUDA
 *     context changed, e.g. after cudaDeviceReset) looks up the array's device
 *     address with cudaGetSymbolAddress, with that device current; make that
 *     first call before any stream capture.
 *   - Every call on a device shares the one array and it keeps the last call's
 *     contents; each call, once its arguments have passed every check,
 *     restarts the array's call counter and tagged router logits (async
 *     memsets on `stream`), and the kernels clear their own accumulators, so
 *     nothing carries over between calls that run one after another.  Calls
 *     that overlap on the GPU (different streams, no ordering between them)
 *     race on the array: order them on one stream.
 *   - Device-side errors stay in the array's sticky error word until read:
 *     moe_get_error(NULL, stream) reports and clears them for the current
 *     device.
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate. */
MOE_API moe_status_t moe_forward_noalloc(const moe_layer_desc_t* desc,
                                         const moe_weights_t* weights, const void* x,
                                         int32_t N, void* out, int32_t* topk_idx,
                                         float* topk_w, void* stream);

/* Test hook: time budget, in nanoseconds, of every bounded device-side wait
 * (grid barrier, stage arrival) for calls enqueued afterwards; default 1e9.
 * A budget of 0 makes a wait that is not already satisfied expire at once, so
 * a test can drive the MOE_ERR_TIMEOUT path without stalling the GPU.  After
 * such a call, re-initialise the workspace with moe_workspace_init. */
MOE_API void moe_debug_set_wait_budget_ns(unsigned long long ns);

/* Tuning hook: the number of (token, slot) pairs, N x top_k, from which a
 * layer with FP4 experts of at least 1 MiB (and no shared expert, zero experts
 * or hash routing) takes the grouped path instead of the fused kernels; 0 or a
 * negative value restores the built-in rule (grouped for N > 8, measured to
 * win there on GB300).  Affects calls and moe_workspace_size /
 * moe_uses_grouped_path from then on; size workspaces after setting it.  Used
 * to measure where the paths cross. */
MOE_API void moe_debug_set_grouped_min_slots(int32_t slots);

#ifdef __cplusplus
}
#endif

#endif /* MOE_DECODE_LAYER_TOPK_GB300_MOE_H */
