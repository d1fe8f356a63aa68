// internal.h — declarations shared by the translation units of the library
// (host side).  Not part of the public C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

// Which rows feed the MMA's token operand.
enum BSource : int {
  kGather = 0,  // rows of x picked through sorted_ids (Gate-Up), gate/up paired
  kDirect = 1,  // rows row_start.. of a row tile (Down reads the activation)
  kDense = 2,   // rows 0..dense_rows-1 tiled by BN (router GEMM)
};

// How the layer's assignments map onto the experts of the index (and of the
// weight tensors).  Token t has kk = k + n_shared assignments: slots j < k are
// its routed ids topk_ids[t][j], slots k..kk-1 the shared experts E..E+n_shared-1,
// which every token selects (SGLang's shared-expert fusion: the shared expert
// becomes one more expert of the grouped GEMM).  Expert parallelism: the E
// routed experts held here are the global ids [e0, e0 + E) of Eg; a routed id
// of another rank's range is dropped without a flag (that rank computes it);
// ids outside [0, Eg) (outside [0, E) without expert parallelism) are invalid.
struct IdMap {
  int k;    // routed slots per token (columns of topk_ids)
  int kk;   // assignments per token: k + shared experts
  int E;    // routed experts held here
  int e0;   // global id of the first of them
  int Eg;   // routed experts in all; 0: no expert parallelism
  __host__ __device__ bool plain() const { return kk == k && Eg == 0; }
};

struct GemmParams {
  int M;             // output columns: 2I (Gate-Up), H (Down), 2E (router)
  int K;             // reduction length in elements
  int I;             // Gate-Up pairing offset (up rows start at I)
  int m_tiles;       // 128-row weight tiles per expert
  int splits;        // split-K count
  int kt_per_split;  // K tiles (128 bytes of K each) per split
  int kt_total;      // K tiles in total
  int tile_major;    // unit order: 0 weight-tile-major, 1 token-tile-major
  const int32_t* tiles;      // [tiles_cap][4] task map (gather / direct)
  const int32_t* num_tiles;  // device scalar (gather / direct)
  const int32_t* sorted_ids; // gather: row -> assignment
  const void* b_rows;        // gather: token rows (x or its e4m3 copy), row-major
  int b_row_bytes;           // gather: bytes per token row
  int topk;                  // gather: token = assignment / topk
  int sentinel;              // gather: T*k marks padding rows
  int dense_rows;            // dense: number of rows
  const float* w_scale;      // FP8: [E][M/128][K/128]
  const float* b_scale;      // FP8: token-operand scales by index row [rows_cap][K/128]
  float* out;                // [splits][rows_cap][M] fp32 partial sums
  void* act_out;             // Gate-Up, bf16, one split: SiLU(g)*u as bf16 [rows_cap][I]
                             // instead of the partial sums
  int g_act;                 // Gate-Up, FP8 128-row token-major tile, one split: SiLU(g)*u
                             // as fp32 rows [rows_cap][I] in `out` instead of the sums
  int rows_cap;              // rows of one split slice of `out` (and of the index)
  int32_t* dev_status;
  // Shared-memory index mode: every CTA rebuilds the routing index from the
  // top-k ids in its prologue instead of reading tiles / sorted_ids.
  int smem_index;
  const int32_t* topk_ids;   // [T][topk], an input of the layer call
  int T, E, tiles_cap;       // E: experts of the index (routed here + shared)
  IdMap idmap;               // topk_ids -> index experts (shared-memory index)
  int write_index;           // CTA 0 also writes the index to `index_out` and the
  struct {                   // expert-id status bit to dev_status
    int32_t *counts, *offsets, *sorted_ids, *tile_expert, *tiles, *inv_pos, *num_tiles;
  } index_out;
  int clear_status;          // first kernel of the call: CTA 0 zeroes dev_status at start
  int early_weights;         // contiguous token operand: stream weights before the wait
  uint64_t pipe_wait_ns;     // limit of the pipeline waits (0: kWaitLimitNs); drains keep
                             // the full limit
  // Coalesced work list (gather / direct operands): the index pads experts
  // to index_bm rows, and the GEMM's token tiles are the work list's tiles of
  // up to `coalesce` (<= BN) consecutive rows of one expert, each entry
  // carrying its first row (tiles / num_tiles then point at the work list).
  // A direct token operand is loaded as ceil(rows / index_bm) boxes of
  // index_bm rows (the map's box).  0: off (tile q is rows q*BN.., a box of
  // BN rows).
  int coalesce;
  int index_bm;              // rows per index tile (0: BN)
  int list_cap;              // entries of the list at `tiles` (0: tiles_cap; the work
                             // list of smaller tiles than the index's holds more)
  // Unsplit GEMM (splits == 1), no fused activation: the output rows are
  // stored as bf16 [rows_cap][M] instead of fp32 partials.
  int out_bf16;
  int scale_by_token;        // FP8 gathered operand: b_scale rows are tokens
};

// Bytes of the shared-memory index of one GEMM CTA (shared-memory index mode).
size_t gemm_index_smem_bytes(int nwarps, int E, int tk, int rows_cap, int tiles_cap);

// Shared memory of one GEMM instantiation without the index, and its warps.
size_t gemm_smem_bytes(int fp8, int bn, int bsrc);
int gemm_warps(int fp8, int bn, int bsrc);
constexpr size_t kMaxGemmSmem = 227 * 1024;

// Launch the persistent GEMM (defined per mode in k_gemm_{bf16,fp8}.cu).
// `me` weight tiles per work unit (1, or 2 for bf16 with bn 128 / 256);
// p.m_tiles then counts groups of `me` tiles.
cudaError_t launch_gemm_bf16(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                             const CUtensorMap& tmA, const CUtensorMap& tmB,
                             const GemmParams& p, int me = 1);
cudaError_t launch_gemm_fp8(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                            const CUtensorMap& tmA, const CUtensorMap& tmB,
                            const GemmParams& p);

// w8a16: FP8 weights (tmA over e4m3 bytes, 64-byte boxes, no swizzle) and
// bf16 token rows; the epilogue is the bf16 GEMM's (k_gemm_w8.cu).
cudaError_t launch_gemm_w8(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                           const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p);

// Index build, pointwise stages (k_align.cu, k_pointwise.cu).
struct IndexPtrs {
  int32_t *counts, *offsets, *sorted_ids, *tile_expert, *tiles, *inv_pos, *num_tiles;
  // Optional (moe_forward with coalesced units): the work list of tiles of up
  // to `coalesce` rows, {expert, first row, rows, 0} x work_cap, and its length.
  int32_t *work_tiles = nullptr, *num_work_tiles = nullptr;
  int coalesce = 0;
  int work_cap = 0;
};
// k and E below count assignments per token and experts of the index (map.kk
// and map.E + shared experts); `map` turns topk_ids into index experts.
// `clear`: the kernel is the call's first and zeroes dev_status before any
// kernel of the call can set a bit (later kernels only OR bits in).
cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int bm, int tiles_cap,
                         const IndexPtrs& idx, int32_t* dev_status, cudaStream_t st,
                         bool pdl, const IdMap& map, bool clear);
// FP8: the same index (block 0) and, on the launch's other blocks, the e4m3
// codes xq [T][H] and per-token scales xs [T][H/128] of x (bf16 [T][H]).
cudaError_t launch_align_quant(const int32_t* ids, int T, int k, int E, int bm, int tiles_cap,
                               const IndexPtrs& idx, int32_t* dev_status, cudaStream_t st,
                               bool pdl, const IdMap& map, bool clear, const void* x, int H,
                               uint8_t* xq, float* xs);
// The same index built by three kernels over chunks of assignments (count,
// scan, scatter); `scratch` holds align_split_scratch_words(T, k, E) ints.
size_t align_split_scratch_words(int T, int k, int E);
cudaError_t launch_align_split(const int32_t* ids, int T, int k, int E, int bm, int tiles_cap,
                               const IndexPtrs& idx, int32_t* scratch, int32_t* dev_status,
                               cudaStream_t st, bool pdl, const IdMap& map, bool clear);
cudaError_t launch_quant_x(const void* x, int T, int H, int k, const int32_t* inv_pos,
                           uint8_t* xq, float* xs, float* xs_rows, int rows_cap, cudaStream_t st,
                           bool pdl);
// (inv_pos / xs_rows may be null: then only the per-token scales are written)
// G: Gate-Up partial sums [splits][rows_cap][2I]; splits = 0: G holds the
// rows of SiLU(gate)*up [rows_cap][I] already (FP8 only), which are only
// quantised.
cudaError_t launch_act(int fp8, const float* G, int splits, int rows_cap, int I,
                       const int32_t* sorted_ids, int sentinel, void* A, float* As,
                       cudaStream_t st, bool pdl);
// k assignments per token, the first k_routed weighted by topk_w[t][j], the
// others (shared experts) by w_shared.  Y: fp32 partials [splits][rows_cap][H],
// or with y_bf16 the bf16 rows [rows_cap][H] of an unsplit Down GEMM.
cudaError_t launch_combine(const void* Y, int y_bf16, int splits, int rows_cap, int H,
                           const int32_t* inv_pos, const float* topk_w, int T, int k,
                           int k_routed, float w_shared, void* out, int out_bf16,
                           cudaStream_t st, bool pdl);
cudaError_t launch_router_prepare(const float* wr, int E, int H, void* hi_lo,
                                  cudaStream_t st);

// The in-path router GEMM, its top-k, the FP8 x-quant and the routing index
// in one cooperative launch (k_route.cu).  The router GEMM's GemmParams are
// passed beside these.
struct RouteFrontParams {
  const float* P;            // router GEMM split-K partials [splits][rows_cap_r][2E]
  int splits, rows_cap_r, T, E, k, score_fn;
  float scale;
  float* scores;             // [T][E]
  int32_t* ids;              // [T][k]
  float* w;                  // [T][k]
  const void* x;             // bf16 [T][H]; xq null: no quantisation
  int H;
  uint8_t* xq;               // e4m3 [T][H]
  float* xs;                 // [T][H/128]
  int Ei, bm, tiles_cap;     // index: experts, row tile, tiles
  IndexPtrs idx;
  int32_t* dev_status;
  int owners, tpc;           // CTAs that own tokens, and tokens per owner
  int gemm_ctas;             // CTAs running router-GEMM units (the others quantise x)
  int32_t* hist;             // [owners][Ei] per-owner expert counts
  unsigned int* bar;         // two grid-barrier counters, zero at launch
};
size_t route_front_smem_bytes(int bn, int tpc, int k, int Ei);
cudaError_t launch_route_front(int bn, int grid, cudaStream_t st, const CUtensorMap& tmW,
                               const CUtensorMap& tmX, const GemmParams& gp,
                               const RouteFrontParams& q);
cudaError_t launch_router_topk(const float* P, int splits, int rows_cap, int T, int E,
                               int k, int score_fn, float scale, float* scores,
                               int32_t* ids, float* w, cudaStream_t st, bool pdl);

// Launch helper: plain or PDL-chained launch with dynamic shared memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
