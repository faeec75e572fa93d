// Internal interface between the C ABI layer (moe_api.cu) and the fused
// decode kernel (decode_kernel.cu).  Host and device code.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kConsumerWarps = 8;                 // compute warps per CTA
constexpr int kConsumerThreads = kConsumerWarps * 32;
// A TMA copy instruction from DRAM keeps its issuing thread busy for a few
// hundred cycles whatever its size, so one thread cannot feed an SM at HBM
// speed: several producer warps (lane 0 each) issue alternate stages.
constexpr int kProducers = 4;
// + one epilogue warp that finishes each gate/up row group (reduction over the
// compute warps, SiLU(g)*u, h stores) while the compute warps go on
constexpr int kEpiWarp = kConsumerWarps;
constexpr int kThreads = kConsumerThreads + 32 + 32 * kProducers;
constexpr int kTB = 4;                            // token rows per weight pass
constexpr int kRedFloats = kConsumerWarps * 2 * kTB * 32;   // one partial-sum buffer
constexpr int kRows = 32;                         // weight rows per row group
constexpr int kMaxSlots = 256;                    // N * top_k per call
constexpr int kMaxE = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxStages = 8;
constexpr int kBoxBytes = 128;                    // inner extent of a weight box
constexpr int kBoxesPerChunk = 4;                 // chunk = 512 bytes of each row
constexpr int kChunkBytes = kBoxBytes * kBoxesPerChunk;
constexpr int kBoxTileBytes = kRows * kBoxBytes;  // 4 KB: one 32-row tile in smem
constexpr int kDnRows = 16;                       // output rows per down block
constexpr int kReadyAS = kMaxSlots;               // ready[] index of the shared expert

// AS shared gate/up (32-row groups), AR routed gate/up (16 gate + 16 up rows
// stacked as one 32-row tile), BR routed down / BS shared down (16-row blocks).
enum Kind { KIND_AS = 0, KIND_AR = 1, KIND_BR = 2, KIND_BS = 3 };
enum Fmt { FMT_NVFP4 = 0, FMT_MXFP4 = 1, FMT_BF16 = 2, FMT_FP8 = 3 };
constexpr int kFp8Block = 128;   // FP8 experts: one FP32 scale per 128 x 128 block
enum ScaleMode { SCALES_NONE = 0, SCALES_TMAP = 1, SCALES_BLOCK = 2 };
// tensor map slots
// 2D maps of weight rows (boxes of 128 bytes x brows), of scales, and 3D
// maps of the weight rows viewed as [128-byte column][row][byte] (boxes of 4
// columns: a whole 512-byte chunk of brows rows in one copy) where the row
// length is a multiple of 128 bytes.
enum TMap { TM_GQ = 0, TM_UQ, TM_DQ, TM_GS, TM_US, TM_DS, TM_SG, TM_SU, TM_SD,
            TM3_GQ, TM3_UQ, TM3_DQ, TM3_SG, TM3_SU, TM3_SD, TM_COUNT };

// Device-side error word bits (workspace control block).
constexpr uint32_t kErrTimeoutBarrier = 1u;
constexpr uint32_t kErrTimeoutStage = 2u;
constexpr uint32_t kErrTimeoutProducer = 4u;

// Workspace control block (first 256 bytes of the workspace).
struct Ctrl {
  unsigned long long arrivals;   // grid-barrier arrivals, monotonic (1 per CTA per call)
  unsigned long long calls;      // stream-kernel call counter: + 256 per call (tag = calls / 256)
  unsigned long long fin;        // stream-kernel end counter: + 256 per call
  uint32_t error;                // sticky error bits
  uint32_t pad[57];
};
static_assert(sizeof(Ctrl) == 256, "control block is the first 256 bytes of a workspace");

// Stage geometry of one kind of row group (see decode_kernel.cu).
struct Geo {
  int fmt;          // Fmt
  int nproj;        // weight matrices streamed together (2 = gate+up, 1 = down)
  int brows;        // rows per TMA box (32 shared gate/up, 16 routed gate/up and down)
  int rg_rows;      // output rows per row group / down block
  int K;            // reduction length (input dim of the projection)
  int kb;           // bytes of one full weight row
  int Kc;           // K elements per full chunk (512 bytes of row)
  int nchunks;      // ceil(kb / 512)
  int scale_mode;   // ScaleMode
  int sr;           // scale bytes per full weight row (K / gs); 0 for bf16
  int scb;          // scale bytes per row per chunk (TMAP mode)
  int scale_off;    // offset of the scale region in the stage
  int opnd_off;     // offset of the activation chunk region
  int hx_off;       // offset of the chunk's h exponents (routed down stages)
  int stage_bytes;  // bytes used in a stage
  int rows_total;   // weight rows of one projection (inter, H or Is)
  int tile_bytes;   // bytes between 128-byte box columns of one projection
  int use3d;        // weight chunks by one 3D copy per projection
};

struct Params {
  CUtensorMap tm[TM_COUNT];   // weight (swizzle 128B) and scale maps
  uint32_t tm_valid;          // bit i set when tm[i] is encoded
  // layer
  int H, inter, E, k, scoring, norm;
  int Z;     // zero experts: router width E + Z, selected zero experts run nothing
  int hash_V;                 // > 0: hash routing with a [hash_V, k] tid2eid table
  const int32_t* tid2eid;     // hash routing: expert ids per token id
  const int32_t* token_ids;   // hash routing: [N] token ids of this call
  float rsf;
  int fmt;   // FMT_NVFP4 / FMT_MXFP4 / FMT_BF16 / FMT_FP8 for the routed experts
  int Is;    // shared expert intermediate size (0 = none)
  int N;
  int route_only;
  // weights (device)
  const uint16_t* router;            // bf16 [E, H], or E2M1 codes [E, H/2] (router_fmt 1)
  int router_fmt;                    // 0 = BF16 router, 1 = NVFP4 router
  const uint8_t* router_s;           // NVFP4 router: E4M3 scales [E, H/16]
  const float* router_s2;            // NVFP4 router: scale2 (one float) or null
  const float* bias;
  const uint8_t *gsc, *usc, *dsc;   // FP4 scales (1D block copies); FP8: f32 block scales
  const float *g2, *u2, *d2;
  const uint16_t* shw;
  // activations / outputs (device)
  const uint16_t* x;
  uint16_t* out;
  int32_t* topk_idx;
  float* topk_w;
  // workspace (device)
  Ctrl* ctrl;
  float* logits;     // [N, E]
  uint16_t* x16;     // [N, H] f16, x * 2^-xexp[n]
  int* xexp;         // [N]
  float* gsig;       // [N] shared-expert gate
  uint16_t* h16;     // [N*k, inter] f16 SiLU(g)*u by (expert, token) slot, x 2^-hexp
  int8_t* hexp;      // [units][hstride] power-of-two exponent per 16 rows of h16
  uint16_t* hs;      // [N, Is] bf16 shared expert SiLU(g)*u
  uint32_t* ready;   // [kMaxSlots + 1] finished gate/up row groups per unit (+ shared)
  int hstride;       // bytes per unit row of hexp (inter/16 rounded up to 16)
  // geometry
  Geo geo[4];
  int nstages, stage_bytes;
  int smem_ring_off, smem_red_off, smem_sacc_off, smem_tab_off, smem_bar_off, smem_total;
  int nrb, nrb_cta;  // down blocks (H/16) and at most this many per CTA
  unsigned long long timeout_ns;
};

// ------------------------------------------------------------ stream kernel
// Fused forward for up to kSkMaxTok token rows with FP4 routed experts
// (stream_kernel.cu): every lane streams its own 16-byte pieces of the
// touched experts' rows with cp.async into a per-warp shared-memory ring,
// dequantises them in registers and runs the dot products as m16n8k16
// tensor-core MMAs with the token rows as the 8 MMA columns.
constexpr int kSkWarps = 16;
constexpr int kSkThreads = kSkWarps * 32;
constexpr int kSkMaxTok = 8;       // MMA N: every token of a call is one column
// Weight ring depth per warp: the item being computed plus one in flight.
// One 2.5 KB item per warp in flight (about 6 MB over the grid) keeps HBM
// busy, and a shallower queue lets the first items and the gate/up -> down
// hand-off through sooner (2 stages measured faster than 3 or 4 at every N).
constexpr int kSkStages = 2;
constexpr int kSkSplitSlots = 16;  // gate/up tiles shared by several warps of one CTA
constexpr int kSkStageCodes = 4 * 32 * 16;   // bytes per warp and stage: 4 pieces of 16 B per lane
constexpr int kSkStageAux = 32 * 16;     // 16 B per lane: block-scale words or a B piece
constexpr int kSkMaxGrid = 256;   // CTAs; bounds the shared-expert K-part slots
constexpr uint32_t kErrRange = 8u;       // an activation left the f16 range

struct StreamParams {
  // tensor maps of the weight codes (2D uint8 [rows, row bytes]): gate / up
  // box 64 B x 16 rows, down box 64 B x 32 rows; the shared expert's down rows
  // (BF16 [H, Is] as bytes) box 64 B x 32 rows
  CUtensorMap tm_gq, tm_uq, tm_dq, tm_shd;
  // and of the block scales (2D uint8 [rows, K / gs]) when their rows are
  // 16-byte multiples (sc_tma): gate / up box 16 B x 16 rows (two NVFP4 or
  // four MXFP4 K segments), down box 16 B x 32 rows
  CUtensorMap tm_gs, tm_us, tm_ds;
  int sc_tma;
  int dpair;   // down items in the paired order (warp pairs take segments 2p, 2p + 1)
  // layer
  int H, inter, E, k, scoring, norm, fmt, N, Is, route_only;
  float rsf;
  // weights (device)
  const uint16_t* router;            // bf16 [E, H]
  const float* bias;                 // [E] or null
  const uint8_t *gq, *uq, *dq;       // E2M1 codes [E, rows, K/2]
  const uint8_t *gsc, *usc, *dsc;    // block scales [E, rows, K/gs]
  const float *g2, *u2, *d2;         // per-expert scale2 or null
  const uint16_t *shg, *shu, *shd;   // shared expert, bf16 (null if Is == 0)
  const uint16_t* shw;               // shared-expert gate vector [H] or null
  // activations / outputs (device)
  const uint16_t* x;
  uint16_t* out;
  int32_t* topk_idx;
  float* topk_w;
  // workspace (device)
  Ctrl* ctrl;
  // Words whose upper half is a call tag, in a region that only this kernel
  // writes and only with 64-bit words of that form, so a word left by an
  // earlier call (of any shape) never carries the current tag.
  unsigned long long* logits;   // [N, E]: (call tag << 32) | f32 bits
  unsigned long long* hw;       // [N*k, inter/2]: (call tag << 32) | two f16 of
                                //   w * scale2 * SiLU(g) * u per slot (elements 2i, 2i+1)
  unsigned long long* sflag;    // [Is/16] call tag << 32 once a shared tile is published
  unsigned long long* scnt;     // [Is/16] (call tag << 32) | K-parts of a shared tile finished
  // plain data, read only after its flag or counter says it is current
  uint16_t* hs;                 // [N, Is] bf16 of gate * SiLU(g) * u (shared expert)
  float* shpart;                // [Is/16, sh_parts, 256] K-part partial sums of shared tiles
  float* oacc;                  // [H, N rounded up to even] FP32 output accumulator (zeroed each call)
  // geometry
  int stages;                   // weight ring depth (kSkStages)
  int sh_parts;                 // K-parts of one shared gate/up tile
  int off_ring, off_aux, off_x16, off_tab, off_split, smem_bytes;
  unsigned long long timeout_ns;
};

// Layers and token counts the stream kernel runs; fills the shared-memory
// layout.  False if the shape is outside what it takes.
bool plan_stream(StreamParams& p, int smem_budget, int grid);
cudaError_t launch_stream(const StreamParams& p, int grid, cudaStream_t stream);
cudaError_t stream_set_smem(int smem_bytes);

// ------------------------------------------------------------ grouped path
// Many-token forward (N * top_k beyond kMaxSlots, or from 128 for large FP4
// experts; moe_api.cu grouped_path): per-expert token groups on
// the tensor cores (grouped_kernel.cu).
constexpr int kGTileTok = 32;   // positions per token tile (MMA N <= 32)

struct GroupedParams {
  int N, H, inter, E, k, scoring, norm;
  float rsf;
  int fmt;
  int route_only;
  const uint16_t* x;        // [N, H] bf16
  const uint16_t* router;   // [E, H] bf16, or E2M1 codes [E, H/2] (router_fmt 1)
  int router_fmt;           // 0 = BF16 router, 1 = NVFP4 router
  const uint8_t* router_s;  // NVFP4 router: E4M3 scales [E, H/16]
  const float* router_s2;   // NVFP4 router: scale2 (one float) or null
  const float* bias;        // [E] or null
  int32_t* topk_idx;        // [N, k] or null
  float* topk_w;
  uint16_t* out;            // [N, H] bf16
  // workspace
  float* logits;            // [N, E]
  int* xexp;                // [N]   x = xg * 2^xexp
  int* sel_e;               // [S]   per (token, slot)
  float* sel_w;
  int* tiles;               // [T][3] expert, first position, positions
  int* ntiles;              // [1]
  int* pos_of;              // [S]   expert-sorted position of slot s
  int* tok_of;              // [S]   token of position
  float* w_of;              // [S]   routing weight of position
  int* bexp;                // [S]   exponent of xg rows
  int* hexp;                // [S]   exponent of h16 rows
  uint16_t* xg;             // [S, H] f16
  float* hbuf;              // [S, max(inter, H)] FP32: h, later y
  uint16_t* h16;            // [S, inter] f16
};

struct GemmParams {
  CUtensorMap tmA[2];       // FP4 rows [E*rows, K/2] bytes: box 64 B x 128 rows, 64-byte swizzle
  CUtensorMap tmB;          // f16 rows [S, 2K] bytes: box 128 B x 64 rows, 128-byte swizzle
  const uint8_t* sc[2];     // block scales [E, rows, K/gs]
  const float* s2[2];       // per-expert scale2 (NVFP4) or null
  const int* tiles;
  const int* ntiles;
  const int* bexp;          // per position: exponent of the B row
  const float* wpos;        // per position routing weight (one-projection GEMM)
  float* out;               // [S, rows] FP32
  uint32_t* err;            // workspace error word
  int rows, K, sr;
  int nstages, nscbuf, stage_bytes, sc_bytes, off_sc, off_bar;
  unsigned long long timeout_ns;
};

// Ring and scale-buffer layout of a grouped GEMM; returns its shared-memory
// bytes (0 if it does not fit in `smem_budget`).
int grouped_plan_gemm(GemmParams& g, int nproj, int smem_budget);
cudaError_t grouped_set_smem(int smem_bytes);
cudaError_t launch_grouped(const GroupedParams& gp, GemmParams gu, GemmParams gd, int grid,
                           int smem_gu, int smem_gd, cudaStream_t st);

// Fills p.geo / ring / smem layout from the layer shape; returns false if
// the shape does not fit the kernel's shared-memory budget.
bool plan_decode(Params& p, int smem_budget, int grid);

// Shared memory the decode kernel may use on this device.
int decode_smem_budget(int device);

// Number of CTAs the decode kernel runs with on `device` (one per SM); also
// raises the kernels' dynamic shared-memory limit to `smem_bytes`.
int decode_grid(int device, int smem_bytes);

// Enqueue the fused decode kernel; returns a CUDA error code.
cudaError_t launch_decode(const Params& p, int grid, cudaStream_t stream);

}  // namespace moe
