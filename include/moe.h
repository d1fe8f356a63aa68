/*
 * moe.h — C ABI of the GB300 (sm_103a) fused Mixture-of-Experts layer.
 *
 * The layer computes, for every token t of a batch,
 *
 *   out[t] = sum_j  w[t,j] * W2[e_j] * ( SiLU(x_t . Wgate[e_j]^T) (.) (x_t . Wup[e_j]^T) ),
 *   e_j = topk_ids[t,j],  Wgate[e] = W13[e, 0:I, :],  Wup[e] = W13[e, I:2I, :],
 *
 * as the pipeline that the "HPC-Ops × SGLang" post (LMSYS blog, section "MoE:
 * reducing the overhead around small expert GEMMs") describes: a routing/index
 * build, a Gate-Up GEMM that reads token rows through the index, a fused
 * SiLU-and-mul (+ FP8 requantisation), a Down GEMM, and a top-k weighted
 * reduction back to token order, chained with Programmatic Dependent Launch.
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers owned by the caller; tensors are
 *     dense and row-major.  The library never allocates, frees or synchronises
 *     inside these calls (the one set-up exception is noted where it applies).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Host-side argument checks happen before anything is launched and return
 *     a moe_status other than MOE_OK; nothing is enqueued in that case.
 *   - `dev_status` (nullable) is a device int32 that kernels OR bit flags into:
 *     bit (1 << MOE_ERR_EXPERT_ID) when a top-k id lies outside [0, E) (that
 *     assignment is dropped and contributes 0), bit (1 << MOE_ERR_TIMEOUT) when
 *     a bounded on-chip wait gave up.  moe_align / moe_forward clear it to 0 at
 *     the start of their first kernel.  Read it after your own synchronisation.
 *   - A launch error reported by the CUDA runtime maps to MOE_ERR_CUDA.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

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

typedef enum {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,        /* null pointer or bad enum value */
  MOE_ERR_SHAPE = 2,      /* unsupported or inconsistent sizes */
  MOE_ERR_DTYPE = 3,      /* unsupported mode / output dtype */
  MOE_ERR_ALIGN = 4,      /* pointer not 16-byte aligned */
  MOE_ERR_WORKSPACE = 5,  /* workspace too small */
  MOE_ERR_EXPERT_ID = 6,  /* device flag: an id outside [0, E) was dropped */
  MOE_ERR_TIMEOUT = 7,    /* device flag: a bounded wait gave up */
  MOE_ERR_CUDA = 8        /* CUDA runtime / driver error */
} moe_status;

/* Precision of a layer call.  MOE_BF16: bf16 weights and activations.
 * MOE_FP8_W8A8: e4m3 weights with fp32 128x128 block scales and e4m3
 * activations (per token / row, per 128 channels).  MOE_W8A16: e4m3 weights
 * with fp32 128x128 block scales and bf16 activations (HPC-Ops × SGLang,
 * operator table, row MoE); the weights are dequantised to bf16 on chip
 * (code * scale, round to nearest even) and the layer runs as MOE_BF16. */
typedef enum { MOE_BF16 = 0, MOE_FP8_W8A8 = 1, MOE_W8A16 = 2 } moe_mode;
typedef enum { MOE_OUT_F32 = 0, MOE_OUT_BF16 = 1 } moe_out;
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;

/* Problem sizes.  T tokens, hidden size H, intermediate size I, E experts,
 * top-k = k.  block_m is the row-tile height of the index and of both expert
 * GEMMs (the token tile): 0 lets the planner choose, otherwise one of
 * 16, 32, 64, 128, 256 (FP8: at most 128).
 * Supported: T >= 1, 1 <= k <= E <= 512, H % 128 == 0, I % 64 == 0
 * (FP8: I % 128 == 0), T*k < 2^31. */
typedef struct {
  int32_t T, H, I, E, k;
  int32_t block_m;
  int32_t mode;       /* moe_mode */
  int32_t out_dtype;  /* moe_out */
} moe_shape;

/* The routing index ("routing and index build", HPC-Ops × SGLang, section MoE).
 * Every field is a caller-owned device buffer.  With a = t*k + j the flat
 * assignment number, Tk = T*k, bm = block_m:
 *   counts[E]        assignments per expert (invalid ids not counted)
 *   offsets[E+1]     exclusive prefix of counts rounded up to multiples of bm
 *   sorted_ids[rows_cap]   expert e's interval [offsets[e], offsets[e+1])
 *                    holds its assignments a in ascending order, then the
 *                    sentinel Tk; every row from offsets[E] on holds Tk
 *   tile_expert[tiles_cap] expert of row tile q (rows q*bm .. q*bm+bm-1), -1
 *                    for q >= num_tiles
 *   tiles[tiles_cap][4]    task map {expert, row_start, rows_valid, 0};
 *                    {-1, q*bm, 0, 0} for q >= num_tiles
 *   inv_pos[Tk]      row that holds assignment a, -1 if its id was invalid
 *   num_tiles[1]     offsets[E] / bm
 * with tiles_cap = ceil(Tk/bm) + min(E, Tk) and rows_cap = tiles_cap*bm. */
typedef struct {
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted_ids;
  int32_t* tile_expert;
  int32_t* tiles;
  int32_t* inv_pos;
  int32_t* num_tiles;
} moe_index;

/* FP8 block scales (FP8 mode only): one fp32 per 128x128 weight block, so that
 * W13 ~= e4m3(W13q) * w13_scale[e][row/128][col/128]
 * ("block_shape [128, 128]", SGLang MoE Triton tuning guide, section 4.1). */
typedef struct {
  const float* w13_scale;  /* [E][2I/128][H/128] */
  const float* w2_scale;   /* [E][H/128][I/128]  */
} moe_scales;

/* Options of moe_forward_ex (zero-initialised = defaults of moe_forward).
 * Stage events: with the shared-memory index there is no align stage, and
 * where the index launch also quantises x (see separate_quant) no x-quant
 * stage (their two events are recorded back to back). */
typedef struct {
  int32_t disable_pdl;      /* 1: plain stream order instead of PDL chaining */
  int32_t split_gateup;     /* 0: planner; else forced split-K count, Gate-Up */
  int32_t split_down;       /* 0: planner; else forced split-K count, Down    */
  int32_t grid_ctas;        /* 0: planner; else CTAs of the persistent GEMMs  */
  /* Optional cudaEvent_t handles recorded on `stream` before stage s
   * (0 align, 1 x-quant, 2 Gate-Up, 3 act, 4 Down, 5 combine) and after the
   * last one (index 6).  NULL entries are skipped.  Recording events between
   * stages serialises them (PDL overlap is lost); use for profiling only. */
  void* stage_events[8];
  /* 1: run SiLU-and-mul as its own stage even where the plan fuses it into
   * the Gate-Up epilogue (BF16 layer with an unsplit Gate-Up), and read the
   * Gate-Up's gate and up sums there even where the plan has the Gate-Up
   * epilogue store SiLU(gate)*up (FP8 layer, unsplit 128-row Gate-Up: see
   * moe_workspace_layout.g_act_rows).  Results are the same either way. */
  int32_t separate_act;
  /* Every GEMM CTA rebuilds the routing index from the top-k ids in its
   * shared memory (T*k <= 4096 and room next to the pipeline), instead of
   * the separate index kernel; the Gate-Up writes the index out.
   * 1: on where it fits; -1: off; 0: planner (on where it fits for BF16
   * layers with at most 16 experts, index and weight experts counted;
   * never with moe_forward_routed).  Other values: MOE_ERR_ARG. */
  int32_t smem_index;
  /* 1: one 128-row weight tile per GEMM work unit even for large token tiles
   * (where the plan pairs two to halve the token-tile traffic per MMA). */
  int32_t single_weight_tile;
  /* Shared experts (SGLang's shared-expert fusion, which DeepSeek-V3, GLM4-MoE
   * and Llama 4 layers use): w13 / w2 (and FP8 scales) hold E routed experts
   * followed by num_shared_experts experts that every token selects with
   * weight shared_expert_weight (0 is read as 1.0); they become extra
   * assignments of the index (slots k.. of each token), so the grouped GEMMs
   * run them with the routed ones.  0 = none; at most 8. */
  int32_t num_shared_experts;
  float shared_expert_weight;
  /* Expert parallelism, local part: the E routed experts held here are the
   * global ids [ep_first_expert, ep_first_expert + E) of ep_num_experts; an
   * assignment to another valid id is dropped without a flag (another rank
   * holds that expert), ids outside [0, ep_num_experts) are invalid (dropped
   * and flagged).  The output is this rank's partial sum.  0 = off. */
  int32_t ep_first_expert;
  int32_t ep_num_experts;
  /* moe_forward_routed: how the router's GEMM, top-k, the FP8 quantisation
   * of x and the routing index run.  1: as one cooperative launch (the
   * router GEMM on the tensor cores, then, after a grid barrier, each CTA's
   * block of tokens: top-k and per-expert counts, with x-quant on the CTAs
   * the GEMM leaves free, then, after a second barrier, its block's rows of
   * the index), preceded by an 8-byte memset of its barrier counters.
   * 0 (default) or -1: as separate PDL-chained kernels (router GEMM, top-k,
   * then the index and x-quant: one launch where one CTA builds the index,
   * see separate_quant), measured faster on the Zipf-routed Qwen3-shaped
   * FP8 layer at every token count tried.  Bit-identical results. */
  int32_t fuse_routing;
  /* Order in which each persistent GEMM walks its work units (weight tile x
   * split x token tile).  0: planner.  1: weight-tile-major (the units of
   * one weight tile over all token tiles are consecutive).  2: token-tile-
   * major (the units of one token tile are consecutive, so an expert's few
   * token tiles read each weight tile at about the same time and the second
   * read hits L2).  The planner takes 2 when an expert's expected token
   * tiles times its units per token tile fit one wave of CTAs, else 1.
   * Results do not depend on it. */
  int32_t unit_order;
  /* Testing aid for the timeout path.  0 (default): the pipeline waits of the
   * expert GEMMs (operands landed, stage free, accumulator ready) give up
   * after 2 s.  A positive value sets that limit in nanoseconds (and those
   * waits then poll without blocking), so that a test can make them give up;
   * 1 makes a wait give up unless its barrier is already complete when first
   * tested.  The kernel then flags MOE_ERR_TIMEOUT in dev_status, lets its
   * own copies and MMAs finish, frees its tensor memory and returns, and the
   * call's output is undefined.  The waits for the kernel's own copies and
   * MMAs before it exits keep the 2-s limit. */
  int32_t pipeline_wait_ns;
  /* Coalesced token tiles for small row tiles (block_m 16 or 32).  The index
   * still pads each expert to block_m rows, but the expert GEMMs take an
   * expert's rows in tiles of up to C consecutive rows (a work list written
   * next to the task map), so an expert holding many rows (skewed routing)
   * has its weight tiles streamed once per C rows instead of once per
   * block_m, while a tile with few rows still loads and multiplies only
   * those (rounded up to 16).  0: planner; -1: off; 32 or 64: C, used where
   * C > block_m (not for MOE_W8A16).  Other values: MOE_ERR_ARG.  Results do
   * not depend on it. */
  int32_t coalesce_rows;
  /* Layers whose index has 256-row tiles (the planner's choice for BF16
   * layers with 128 or more rows per active expert): 128 makes the Down GEMM
   * take each expert's rows in tiles of up to 128 (a work list over the same
   * index) with the 128-row tile instead of the 256-row token-major one;
   * -1 keeps the 256-row tiles; 0: planner (128-row tiles from 256 rows per
   * active expert on average).  Other values: MOE_ERR_ARG.  Results do not
   * depend on it. */
  int32_t down_tile_rows;
  /* FP8 layers whose index is built by one CTA (T*k <= 2048, no shared-
   * memory index): the plan quantises x on the index launch's other blocks,
   * with per-token scales the Gate-Up looks up through the index
   * (moe_workspace_layout.xs_by_token).  1: quantise x in its own kernel,
   * which also writes the scales per index row.  Results are the same. */
  int32_t separate_quant;
} moe_forward_opts;

/* Options of moe_align_ex: the same shared-expert and expert-parallel mapping
 * of topk_ids onto the experts of the index as moe_forward_opts. */
typedef struct {
  int32_t num_shared_experts;
  int32_t ep_first_expert;
  int32_t ep_num_experts;
} moe_align_opts;

/* Where moe_forward keeps its intermediates inside the caller's workspace
 * (byte offsets from the workspace base) and the plan it runs. */
typedef struct {
  int32_t block_m, tiles_cap, rows_cap;
  int32_t split_gateup, split_down;    /* split-K counts S1, S2 */
  int32_t grid_gateup, grid_down;      /* persistent CTAs per GEMM */
  int32_t fused_act;   /* 1: SiLU-and-mul runs in the Gate-Up epilogue (no G) */
  int32_t smem_index;  /* 1: GEMM CTAs rebuild the index in shared memory; the
                          Gate-Up writes it out (no separate index kernel) */
  int32_t weight_tiles_per_unit;  /* Gate-Up | Down << 8 (1 or 2 each) */
  int32_t route_fused;  /* moe_forward_routed: router top-k, x-quant and index in one grid */
  int32_t unit_order;   /* Gate-Up | Down << 8: 1 weight-tile-major, 2 token-tile-major */
  size_t off_counts, off_offsets, off_sorted_ids, off_tile_expert, off_tiles,
      off_inv_pos, off_num_tiles;
  size_t off_index_scratch; /* per-chunk histograms of the split index build */
  size_t off_xq;   /* FP8: e4m3 x            [T][H]                         */
  size_t off_xs;   /* FP8: fp32 x scales     [T][H/128]                     */
  size_t off_xs_rows; /* FP8: the same scales in index-row order [rows_cap][H/128]
                         (0 bytes when xs_by_token) */
  size_t off_g;    /* fp32 Gate-Up partials  [S1][rows_cap][2I] (0 bytes when fused_act),
                      or fp32 SiLU(gate)*up rows [rows_cap][I] when g_act_rows */
  size_t off_a;    /* activation: bf16 [rows_cap][I] or e4m3 [rows_cap][I]  */
  size_t off_as;   /* FP8: fp32 act scales   [rows_cap][I/128]              */
  size_t off_y;    /* Down output rows (sorted): fp32 partials [S2][rows_cap][H], or
                      bf16 [rows_cap][H] when y_bf16 (S2 = 1) */
  size_t off_router;        /* moe_forward_routed: router GEMM partial sums   */
  size_t off_route_counter; /* fused routing: two grid-barrier counters (8 bytes) */
  size_t total_bytes;
  size_t off_route_hist;    /* fused routing: per-CTA expert counts           */
  int32_t coalesce_rows;    /* Gate-Up: C of the work list it takes, 0 for the task map */
  size_t off_work_tiles;    /* work list: int32 [work_cap][4] {expert, first row, rows, 0} */
  size_t off_num_work_tiles;  /* its length (int32) */
  int32_t y_bf16;           /* 1: the Down GEMM is unsplit and stores bf16 rows at off_y */
  int32_t down_tile_rows;   /* Down: C of the work list it takes, 0 for the task map */
  int32_t work_cap;         /* entries of the work list (0 when there is none) */
  int32_t g_act_rows;       /* 1: the Gate-Up epilogue stores SiLU(gate)*up in fp32 at off_g
                               and the activation stage only quantises it (FP8 layer whose
                               Gate-Up runs unsplit on 128-row token tiles) */
  int32_t xs_by_token;      /* FP8: 1 when the Gate-Up reads the x scales per token (off_xs)
                               and off_xs_rows is not written */
} moe_workspace_layout;

/* tiles_cap of the index for these sizes (0 on invalid arguments). */
MOE_API size_t moe_index_tiles_cap(int32_t T, int32_t k, int32_t E, int32_t block_m);

/* Resolve the plan moe_forward(_ex) will run for `shape` (opts nullable) and
 * the layout of its workspace.  Pure host computation. */
MOE_API moe_status moe_plan(const moe_shape* shape, const moe_forward_opts* opts,
                    moe_workspace_layout* layout);

/* Workspace bytes moe_forward(_ex) needs (0 on invalid arguments). */
MOE_API size_t moe_workspace_bytes(const moe_shape* shape, const moe_forward_opts* opts);

/* Routing and index build ("routing and index build", HPC-Ops × SGLang,
 * section MoE): a shared-memory counting pass and scan that place every
 * assignment a = t*k + j of topk_ids[T][k] (int32) into its expert's
 * contiguous interval, stable in a, with no global atomics on the ordering
 * path; also writes the per-tile task map.  Layout of every output: moe_index.
 * block_m must be one of 16, 32, 64, 128, 256.  Invalid ids are dropped and
 * flagged in dev_status.  Errors: MOE_ERR_ARG (null idx field / topk_ids),
 * MOE_ERR_SHAPE (sizes), MOE_ERR_CUDA. */
MOE_API moe_status moe_align(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                     int32_t block_m, const moe_index* idx, int32_t* dev_status,
                     void* stream);

/* moe_align with shared experts and / or the expert-parallel local mapping
 * (opts nullable = moe_align).  The index then covers T*(k + n_shared)
 * assignments a = t*(k + n_shared) + j over E + n_shared experts (shared
 * expert s of token t is slot k + s, expert E + s); size its buffers with
 * moe_index_tiles_cap(T, k + n_shared, E + n_shared, block_m).  Mapped ids
 * are staged on chip: T*(k + n_shared) <= 32768, else MOE_ERR_SHAPE.  Remote
 * ids (expert parallelism) get inv_pos -1 like invalid ones but no flag. */
MOE_API moe_status moe_align_ex(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                        int32_t block_m, const moe_align_opts* opts, const moe_index* idx,
                        int32_t* dev_status, void* stream);

/* The whole layer.  Inputs:
 *   x        bf16 [T][H]
 *   w13      bf16 [E][2I][H] (FP8: e4m3 bytes), rows 0..I-1 gate, I..2I-1 up
 *   w2       bf16 [E][H][I]  (FP8: e4m3 bytes)
 *   topk_ids int32 [T][k];  topk_w fp32 [T][k] (used as given)
 *   scales   FP8 only (NULL in BF16 mode)
 *   out      [T][H], fp32 or bf16 per shape->out_dtype
 *   workspace, ws_bytes  >= moe_workspace_bytes(shape, NULL), 256-byte aligned
 * FP8 mode quantises x per token per 128 channels (s = amax/448, 1 if amax is
 * 0; q = e4m3 RNE-satfinite(x/s)) and the activation per row per 128 channels
 * by the same rule.  Stages: align, [x-quant], Gate-Up, act, Down, combine,
 * launched on `stream` with PDL.  Errors: MOE_ERR_ARG, MOE_ERR_SHAPE,
 * MOE_ERR_DTYPE, MOE_ERR_ALIGN, MOE_ERR_WORKSPACE, MOE_ERR_CUDA.
 * The first call on a device (per weight-pointer set) encodes TMA descriptors
 * on the host; nothing is allocated. */
MOE_API moe_status moe_forward(const moe_shape* shape, const void* x, const void* w13,
                       const void* w2, const int32_t* topk_ids,
                       const float* topk_w, const moe_scales* scales, void* out,
                       void* workspace, size_t ws_bytes, int32_t* dev_status,
                       void* stream);

/* moe_forward with options (opts nullable = defaults).  The workspace must be
 * sized with the same opts. */
MOE_API moe_status moe_forward_ex(const moe_shape* shape, const void* x,
                          const void* w13, const void* w2,
                          const int32_t* topk_ids, const float* topk_w,
                          const moe_scales* scales, void* out, void* workspace,
                          size_t ws_bytes, int32_t* dev_status, void* stream,
                          const moe_forward_opts* opts);

/* Top-k weighted reduction back to token order (HPC-Ops × SGLang, section MoE,
 * "PDL-chained stages": the final top-k weighted reduce):
 *   out[t][h] = sum_{j=0..k-1, ascending} topk_w[t][j] *
 *               sum_{s=0..splits-1, ascending} y[s][inv_pos[t*k+j]][h]
 * in fp32, assignments with inv_pos = -1 contributing 0; no atomics, so the
 * result is bitwise reproducible.  y is fp32 [splits][rows_cap][H] in sorted
 * (expert-grouped) row order.  out is [T][H] fp32 or bf16 (shape->out_dtype);
 * only shape->T, H, k, out_dtype are read.  Errors: MOE_ERR_ARG,
 * MOE_ERR_SHAPE, MOE_ERR_ALIGN, MOE_ERR_CUDA. */
MOE_API moe_status moe_combine(const moe_shape* shape, int32_t splits, int32_t rows_cap,
                       const float* y, const int32_t* inv_pos,
                       const float* topk_w, void* out, void* stream);

/* The layer with its router in the path (HPC-Ops × SGLang, section "Router
 * GEMM" feeding section "MoE"): the two-bf16 router GEMM over hi_lo (from
 * moe_router_prepare) scores x, its top-k becomes the layer's routing, and the
 * layer runs as in moe_forward — one chain of launches on `stream`, whose
 * front (router GEMM, top-k, FP8 quantisation of x, routing index) is four
 * PDL-chained kernels or, on request, one cooperative grid
 * (moe_forward_opts.fuse_routing).  Outputs besides `out`: scores fp32 [T][E],
 * topk_ids int32 [T][k], topk_w fp32 [T][k] (caller-owned).  score_fn and
 * scale as in moe_router_topk; router shapes as moe_router_workspace_bytes
 * accepts (E a multiple of 64, k <= 32).  Not combined with shared experts,
 * expert parallelism or the shared-memory index (MOE_ERR_SHAPE).  The
 * workspace is sized by moe_routed_workspace_bytes / moe_plan_routed (the
 * router's partial sums and, fused, the barrier counters and per-CTA expert
 * counts are added). */
MOE_API moe_status moe_plan_routed(const moe_shape* shape, const moe_forward_opts* opts,
                           moe_workspace_layout* layout);
MOE_API size_t moe_routed_workspace_bytes(const moe_shape* shape, const moe_forward_opts* opts);
MOE_API moe_status moe_forward_routed(const moe_shape* shape, const void* x, const void* hi_lo,
                              int32_t score_fn, float scale, const void* w13, const void* w2,
                              const moe_scales* scales, float* scores, int32_t* topk_ids,
                              float* topk_w, void* out, void* workspace, size_t ws_bytes,
                              int32_t* dev_status, void* stream, const moe_forward_opts* opts);

/* Router weight preparation ("a precision-aware BF16 formulation", HPC-Ops ×
 * SGLang, section Router GEMM): from fp32 wr[E][H] writes bf16
 * hi_lo[2E][H]: rows 0..E-1 hi = wr truncated to bf16, rows E..2E-1
 * lo = bf16_rne((wr - hi) * 256).  Run once per weight set (untimed prep).
 * Errors: MOE_ERR_ARG, MOE_ERR_SHAPE, MOE_ERR_ALIGN, MOE_ERR_CUDA. */
MOE_API moe_status moe_router_prepare(const float* wr, int32_t E, int32_t H,
                              void* hi_lo, void* stream);

/* Workspace bytes moe_router_topk needs (0 on invalid arguments). */
MOE_API size_t moe_router_workspace_bytes(int32_t T, int32_t H, int32_t E);

/* Router GEMM + top-k: scores[t][e] = sum_h x[t][h]*hi[e][h]
 *   + (sum_h x[t][h]*lo[e][h]) / 256, fp32 accumulation on the tensor cores,
 * written fp32 [T][E]; then p = softmax over e (score_fn 0) or sigmoid
 * (score_fn 1); the k largest scores (ties -> lower e) give topk_ids int32
 * [T][k] (descending score) and topk_w fp32 [T][k] = scale * p_j / sum p_sel.
 * x bf16 [T][H]; H % 128 == 0, 1 <= k <= E, E % 64 == 0, E <= 512.
 * Errors: MOE_ERR_ARG, MOE_ERR_SHAPE, MOE_ERR_ALIGN, MOE_ERR_WORKSPACE,
 * MOE_ERR_CUDA. */
MOE_API moe_status moe_router_topk(const void* x, const void* hi_lo, int32_t T,
                           int32_t H, int32_t E, int32_t k, int32_t score_fn,
                           float scale, float* scores, int32_t* topk_ids,
                           float* topk_w, void* workspace, size_t ws_bytes,
                           void* stream);

/* Largest workspace moe_forward_static can serve (128 MiB).  With the plans
 * of this version that covers every T up to 768 for the Mixtral-shaped bf16
 * layer, up to 912 for the Qwen3-30B-A3B-shaped layer and up to 20 for the
 * DeepSeek-V3-shaped FP8 layer; moe_workspace_bytes(shape, NULL) tells for
 * any shape. */
#define MOE_STATIC_SCRATCH_BYTES ((size_t)128 << 20)

/* moe_forward without a workspace argument, for callers that cannot allocate
 * device memory: serving engines that reserve all device memory at start-up
 * and forbid later allocation, and plain-C hosts with no device allocator of
 * their own.  No counterpart on the pages: it is an interface convenience of
 * this library.
 *   The intermediates live in one file-scope device array of
 *   MOE_STATIC_SCRATCH_BYTES.  The call itself allocates nothing (no
 *   cudaMalloc / cudaFree, no allocating library routine), but under the CUDA
 *   runtime's lazy module loading (its default) the array is reserved on a
 *   device by the first moe_forward_static call there, and then held until
 *   the process exits.  Make that first call on each device before reserving
 *   the rest of device memory, and before any stream capture: it looks up the
 *   array's device address with that device current.  A failed lookup returns
 *   MOE_ERR_CUDA and is retried by the next call.
 *   All calls share the array and it keeps the last call's contents (nothing
 *   in it needs to start at zero): calls that overlap on the GPU race and must
 *   be serialised by the caller.
 * Arguments, layouts and device-status behaviour are those of moe_forward.
 * Errors: those of moe_forward; MOE_ERR_WORKSPACE when the shape needs more
 * than MOE_STATIC_SCRATCH_BYTES (moe_workspace_bytes(shape, NULL) tells). */
MOE_API moe_status moe_forward_static(const moe_shape* shape, const void* x,
                                      const void* w13, const void* w2,
                                      const int32_t* topk_ids, const float* topk_w,
                                      const moe_scales* scales, void* out,
                                      int32_t* dev_status, void* stream);

/* Static description of a status code. */
MOE_API const char* moe_status_str(int32_t status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
