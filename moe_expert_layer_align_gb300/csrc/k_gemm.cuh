// k_gemm.cuh — persistent grouped expert GEMM on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM, operands staged by TMA / cp.async).
//
// Role in the layer (HPC-Ops × SGLang, section "MoE", fused pipeline): the
// "Gate-Up GEMM reads the original token rows through the routing index" and
// the Down GEMM is "the same persistent task-map expert GEMM".  The same
// kernel also runs the router's two-bf16 GEMM (section "Router GEMM").  For
// the bf16 layer with an unsplit Gate-Up, the epilogue also applies the
// SiLU-and-mul of section "MoE", "Gate-Up and activation" and writes the
// activation Down reads, so no separate activation stage runs.
//
// Orientation ("swap-AB"): the MMA's M side is 128 weight rows, the N side
// (BN = block_m) is the token tile.  A decode-sized expert group of a few
// tokens then costs a narrow N, not a padded 128-row M.  FP8 with 128-row
// token tiles is the exception: it runs token-major (kTokM below), which
// makes the block-scale promotion per-thread constant.
//
// For weight tile mt, split ks and row tile q (one work unit), with e the
// tile's expert:
//   out[ks][row0 + n][col(m)] = sum_{k in split ks} W[e][row(m)][k] * B[n][k]
// where B[n] is x[sorted_ids[row0+n] / topk] (gather), row row0+n of the
// activation (direct) or row q*BN+n of x (dense).  Gate-Up pairs the tile per
// 32-lane TMEM quadrant q: lanes 32q..32q+15 hold gate rows mt*64+16q.. and
// lanes 32q+16..32q+31 the matching up rows I+mt*64+16q.., so each gate/up
// pair meets inside one warp (a shuffle apart).  Split-K partial sums are
// written in fp32 and reduced, in a fixed order, by the next stage (act or
// combine): nothing is accumulated with atomics.
//
// FP8 (e4m3, kind::f8f6f4): every 128-wide K block is its own MMA group into
// one of up to 8 TMEM buffers; the epilogue warps read it and add
// partial * w_scale[e][row/128][kb] * b_scale[row or token][kb] into fp32
// registers (block scales are fp32, so the product cannot be folded into the
// MMA).  Work units are walked weight-tile-major or token-tile-major, as the
// planner chooses (make_unit).
//
// Index modes.  With few assignments every CTA rebuilds the routing index in
// its own shared memory from the top-k ids (index_build.cuh) — an input of
// the layer call, so this needs no wait on the previous stage; CTA 0 of the
// Gate-Up also writes the index out for the later stages.  No separate index
// kernel runs, the Gate-Up streams weights as soon as it starts, and the Down
// GEMM streams its first weight stages before the previous stage has
// finished.  With many assignments an index kernel runs first and CTAs read
// the task map from global memory.
//
// Warp roles: warp 0 issues the TMA loads (weights; the token tile too when
// its rows are contiguous), warp 1 (one thread) issues MMAs, the epilogue
// warps (4, or 8 for FP8 with 64/128-row tiles) drain TMEM, and for the
// gathered token operand the last 1-2 warps copy the token rows with 16-byte
// cp.async into the 128-byte-swizzled layout, each thread arriving on the
// stage barrier when its copies land.  TMA's four-row gather alone (one op
// per ~40 ns) capped the prefill Gate-Up at a third of the rate of a dense
// load of the same bytes; for 128-row bf16 tiles the TMA warp gathers 32 of
// the rows that way next to the cp.async warps.  With the accumulator in TMEM
// instead of registers this split costs no registers, so the Hopper argument
// for one warp group doing everything ("occupancy first, no warp
// specialisation") does not carry over.  Every wait is bounded
// (GemmParams::pipe_wait_ns, kWaitLimitNs by default); on a timeout the
// kernel ORs kStatusTimeout into dev_status and raises a CTA-wide abort flag
// that every other wait also watches, so all roles leave their loops; then
// the TMA warp waits for its own copies to land, the gather threads for
// theirs, the MMA thread for its MMAs, and TMEM is freed.  Waits of warps
// that go on to warp-collective instructions (tcgen05.ld, __syncwarp) are
// voted across the warp, so its lanes never part ways.
#pragma once
#include <cuda_bf16.h>

#include "index_build.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kTileM = 128;                 // weight rows per tile (MMA M)
constexpr int kKBytes = 128;                // K bytes per pipeline stage
constexpr int kABytes = kTileM * kKBytes;   // 16 KB weight tile per stage

__host__ __device__ constexpr int stages_for(int fp8, int bn, int me) {
  return me == 1 ? (bn <= 64 ? 8 : bn == 128 ? (fp8 ? 5 : 6) : 4)
                 : (196608 / (me * kABytes + bn * kKBytes) < 8 ? 196608 / (me * kABytes + bn * kKBytes)
                                                               : 8);
}

// ME weight tiles per work unit: ME = 2 halves the token-tile traffic per
// MMA for large (prefill) tiles, where L2 bandwidth, not HBM, is the limit.
template <int FP8, int BN, int BSRC = kDirect, int ME = 1>
struct GemmShape {
  static constexpr int kStages = stages_for(FP8, BN, ME);
  static constexpr int kAStage = ME * kABytes;
  // Epilogue warps: four (one per TMEM lane quadrant), or eight for FP8
  // with wide token tiles, where the per-K-block promotion is the busiest
  // role; the second warp of a quadrant then takes the upper half of the
  // columns.
  // bf16 with 256-row token tiles and two weight tiles per unit runs token-
  // major as well: the two 128-row halves of the token tile are the M sides
  // of two MMAs against one N = 256 operand made of both weight tiles, i.e. a
  // 256 x 256 tile per CTA staging 64 MACs per operand byte (the 128-row
  // tiles' 2 x 128 x 128 stage holds 43, and their rate is what the L2-to-SM
  // bandwidth allows).  The halves' fp32 accumulators fill the 512 TMEM
  // columns, so there is one set, drained and released per half by four
  // epilogue warps each; a TMEM lane is a token, so each thread writes its
  // token's output row with 16-byte stores.
  static constexpr bool kTok2 = !FP8 && BN == 256 && ME == 2 && BSRC != kDense;
  static constexpr int kEpiWarps = ((FP8 && BN >= 64) || kTok2) ? 8 : 4;   // 16 measured slower (spills)
  // FP8 with 128-row token tiles runs token-major: the token tile is the
  // MMA's M side and the weight tile its N side.  A TMEM lane is then one
  // token, and both block scales of its K-block partial are per-thread
  // constants (the token's, and the weight block's: one for Down, gate and
  // up for Gate-Up), so the promotion is one packed FMA per two values with
  // no per-column scale loads.  (Swap-AB needs a per-column token scale.)
  static constexpr bool kTokM = FP8 && BN == 128;
  // FP8 16..64-row tiles: ring stage i and accumulator buffer i advance in
  // lockstep (8 each), so the accumulator-ready commit of a K block also
  // releases its stage (the producer and gather warps wait on it) and the
  // MMA thread commits once per K block, not twice (DeepSeek-shaped layer at
  // T=64: 1476 -> 1453 us).
  static constexpr bool kShareRel = FP8 && BN <= 64;
  static constexpr int kEpiThreads = 32 * kEpiWarps;
  static constexpr int kRoleThreads = 64 + kEpiThreads;   // + TMA and MMA warps
  // token-row gather warps (gathered operand only) and block size
  static constexpr int kGatherWarps = BSRC == kGather ? (BN >= 256 ? 4 : BN >= 64 ? 2 : 1) : 0;
  static constexpr int kGatherThreads = 32 * kGatherWarps;
  static constexpr int kThreads = kRoleThreads + kGatherThreads;
  static constexpr int kWarps = kThreads / 32;
  // Prefill tiles (bf16): the TMA warp also gathers the first kTmaRows token
  // rows of every stage with the TMA's four-row gather, next to the cp.async
  // warps' share — two gather engines instead of one.
  static constexpr int kTmaRows = (BSRC == kGather && BN >= 128 && !FP8) ? 32 : 0;
  static constexpr int kRowsPerGatherThread =
      kGatherWarps ? (BN - kTmaRows) / (4 * kGatherWarps) : 1;
  static constexpr int kBBytes = BN * kKBytes;
  // TMEM accumulator buffers (each ME x BN columns): two per-unit buffers
  // for bf16 where they fit; for FP8 every 128-wide K block is its own
  // buffer, so keep up to 8 in flight (the MMA would otherwise wait on the
  // epilogue's promotion every other K block).
  // (kTok2: the two token halves, each with its own full / empty barriers.)
  static constexpr int kAccBufs =
      kTok2 ? 2 : FP8 ? (512 / BN < 8 ? 512 / BN : 8) : (512 / (ME * BN) < 2 ? 1 : 2);
  static constexpr int kTmemCols =
      kTok2 ? 512 : (kAccBufs * ME * BN < 32) ? 32 : kAccBufs * ME * BN;
  static constexpr int kElemsPerStage = FP8 ? 128 : 64;
  static constexpr uint32_t kIdesc =
      kTok2 ? mma_idesc(1u, kTileM, ME * kTileM) : mma_idesc(FP8 ? 0u : 1u, kTileM, BN);
  static constexpr int kOffB = kStages * kAStage;
  static constexpr int kOffBar = kOffB + kStages * kBBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;  // + drain
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  // FP8: the token-operand scales of one K block, double-buffered per
  // epilogue warp: [kEpiWarps][2][its BN * 4 / kEpiWarps columns]
  static constexpr int kOffScale = (kOffMisc + 16 + 15) & ~15;
  static constexpr int kOffIdx = kOffScale + (FP8 ? 8 * BN * 4 : 0);  // shared-memory index
  static constexpr size_t kSmemBytes = 1024 + kOffIdx;             // without the index
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 M=128 needs N % 16 == 0");
  static_assert(ME == 1 || !FP8, "FP8 promotion keeps one weight tile per unit");
  static_assert(!kShareRel || kStages == kAccBufs, "shared release needs lockstep rings");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                "tcgen05.alloc takes a power of two from 32 to 512 columns");
};

// Shared-memory index: build scratch, staged ids, sorted rows, task map.
struct SmemIndex {
  IndexScratch sc;
  int32_t* ids;    // [T*k]
  int32_t* rows;   // [rows_cap]: assignment per sorted row, T*k on padding
  int4* tiles;     // [tiles_cap]
  __host__ __device__ static size_t words_before_tiles(int nwarps, int E, int tk, int rows_cap) {
    return (IndexScratch::words(nwarps, E) + tk + rows_cap + 3) & ~static_cast<size_t>(3);
  }
  __host__ __device__ static size_t bytes(int nwarps, int E, int tk, int rows_cap, int tiles_cap) {
    return 4 * words_before_tiles(nwarps, E, tk, rows_cap) + 16 * static_cast<size_t>(tiles_cap);
  }
  __device__ void carve(int32_t* base, int nwarps, int E, int tk, int rows_cap, int remote) {
    sc.carve(base, nwarps, E, remote);
    ids = base + IndexScratch::words(nwarps, E);
    rows = ids + tk;
    tiles = reinterpret_cast<int4*>(base + words_before_tiles(nwarps, E, tk, rows_cap));
  }
};

struct WorkUnit {
  int mt, ks, e, row0, rows, kt0, kt1;
};

// Unit u = ((mt * splits + ks) * num_tiles + q), weight-tile-major:
// consecutive units share a weight tile; or, token-tile-major,
// u = (q * m_tiles + mt) * splits + ks: consecutive units share a token tile,
// and the few token tiles of an expert reach each of its weight tiles within
// one wave of CTAs (the later reads hit L2).  The task-map entry is the only
// memory read, so roles load the next unit's entry while they work on the
// current one.
template <int BN, int BSRC>
__device__ __forceinline__ int4 load_tile(int q, const GemmParams& p, const int4* smem_tiles) {
  if (BSRC == kDense) return make_int4(0, q * BN, min(BN, p.dense_rows - q * BN), 0);
  // L2-coherent load: the Down GEMM may read the task map before its PDL wait
  const int4 t = smem_tiles ? smem_tiles[q] : __ldcg(reinterpret_cast<const int4*>(p.tiles) + q);
  // Every address below derives from this entry: row 0 of tile q is q*BN
  // by construction (a work-list entry carries its own, checked to lie in
  // [0, rows_cap - rows]), and an entry that is not a well-formed one (a
  // workspace overwritten between the stages) becomes an empty tile of
  // expert 0 rather than an out-of-range access.
  if (p.coalesce == 0) {
    const bool ok = t.x >= 0 && t.x < p.E && t.z >= 0 && t.z <= BN;
    return make_int4(ok ? t.x : 0, q * BN, ok ? t.z : 0, 0);
  }
  const bool ok = t.x >= 0 && t.x < p.E && t.z >= 0 && t.z <= BN && t.y >= 0 &&
                  t.y <= p.rows_cap - t.z;
  return ok ? make_int4(t.x, t.y, t.z, 0) : make_int4(0, 0, 0, 0);
}

// Token of sorted row `a`'s assignment, or -1 for padding and any value
// outside [0, T*k).
__device__ __forceinline__ int assignment_token(int a, const GemmParams& p) {
  return static_cast<unsigned>(a) < static_cast<unsigned>(p.T * p.topk) ? a / p.topk : -1;
}

__device__ __forceinline__ int unit_tile(int u, int num_tiles, const GemmParams& p) {
  return p.tile_major ? u / (p.m_tiles * p.splits) : u % num_tiles;
}

__device__ __forceinline__ WorkUnit make_unit(int u, int num_tiles, int4 t, const GemmParams& p) {
  WorkUnit w;
  const int r = p.tile_major ? u % (p.m_tiles * p.splits) : u / num_tiles;
  w.ks = r % p.splits;
  w.mt = r / p.splits;
  w.e = t.x;
  w.row0 = t.y;
  w.rows = t.z;
  w.kt0 = w.ks * p.kt_per_split;
  w.kt1 = min(p.kt_total, w.kt0 + p.kt_per_split);
  return w;
}

// Iterates a CTA's units with the next task-map entry prefetched.
template <int BN, int BSRC>
struct UnitIter {
  int u, units, num_tiles;
  const int4* smem_tiles;
  int4 next;
  __device__ __forceinline__ UnitIter(int units_, int num_tiles_, const GemmParams& p,
                                      const int4* st)
      : u(blockIdx.x), units(units_), num_tiles(num_tiles_), smem_tiles(st) {
    if (u < units) next = load_tile<BN, BSRC>(unit_tile(u, num_tiles, p), p, smem_tiles);
  }
  __device__ __forceinline__ bool valid() const { return u < units; }
  // The current unit; starts the load of the one after it.
  __device__ __forceinline__ WorkUnit take(const GemmParams& p) {
    const int4 t = next;
    const int un = u + gridDim.x;
    if (un < units) next = load_tile<BN, BSRC>(unit_tile(un, num_tiles, p), p, smem_tiles);
    return make_unit(u, num_tiles, t, p);
  }
  __device__ __forceinline__ void advance() { u += gridDim.x; }
  __device__ __forceinline__ bool has_next() const { return u + static_cast<int>(gridDim.x) < units; }
};

// Sixteen fp32 values (raw bits) as two 16-byte stores of bf16 (dst 16-byte
// aligned).
__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const uint32_t* v) {
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162 b2 =
        __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  d[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

__device__ __forceinline__ void report_timeout(const GemmParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  if (p.dev_status) atomicOr(p.dev_status, kStatusTimeout);
}

// The persistent GEMM as run by one CTA of S::kThreads threads with the
// dynamic shared memory at smem_raw: the body of moe_gemm_kernel, and the
// first phase of the fused routing kernel (k_route.cu), which goes on with
// the same CTAs after it returns.
template <int FP8, int BN, int BSRC, int ME>
__device__ __forceinline__ void gemm_cta(const CUtensorMap& tmA, const CUtensorMap& tmB,
                                         const GemmParams& p, uint8_t* smem_raw) {
  using S = GemmShape<FP8, BN, BSRC, ME>;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + S::kOffB;
  const uint32_t bar_full = sA + S::kOffBar;
  const uint32_t bar_empty = bar_full + 8 * S::kStages;
  const uint32_t bar_accf = bar_empty + 8 * S::kStages;
  const uint32_t bar_acce = bar_accf + 8 * S::kAccBufs;
  const uint32_t bar_drain = bar_acce + 8 * S::kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 4);
  volatile int* issued_slot = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 8);
  float* sx_buf = reinterpret_cast<float*>(smem + S::kOffScale);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tk = p.T * p.topk;
  // Pipeline waits: bounded by pipe_wait_ns and left early once another role
  // raised the abort flag.  warp_wait votes across the warp (a lane that saw
  // the abort flag counts as failed), so all its lanes take the same branch.
  const uint64_t wait_ns = p.pipe_wait_ns ? p.pipe_wait_ns : kWaitLimitNs;
  auto thread_wait = [&](uint32_t bar, uint32_t par) {
    return mbar_wait_pipe(bar, par, wait_ns, abort_flag);
  };
  auto warp_wait = [&](uint32_t bar, uint32_t par) {
    const bool r = mbar_wait_pipe(bar, par, wait_ns, abort_flag) && *abort_flag == 0;
    return __all_sync(0xffffffffu, r);
  };
  auto warp_aborted = [&]() { return __any_sync(0xffffffffu, *abort_flag != 0); };

  if (threadIdx.x == 0) {
    // First kernel of the call: clear the status word before any bit is set.
    // (A timeout bit of another CTA comes at least kWaitLimitNs after the
    // grid started; CTA 0's own expert-id bit is ORed in after the prologue
    // barrier, which orders it after this store.)
    if (p.clear_status && p.dev_status && blockIdx.x == 0) *p.dev_status = 0;
    for (int s = 0; s < S::kStages; ++s) {
      // the TMA thread's expect-tx arrival, plus one per gather thread
      mbar_init(bar_full + 8 * s, 1 + S::kGatherThreads);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < S::kAccBufs; ++b) {
      mbar_init(bar_accf + 8 * b, 1);
      // one arrival per epilogue warp (kTok2: per warp of that token half)
      mbar_init(bar_acce + 8 * b, S::kTok2 ? S::kEpiWarps / 2 : S::kEpiWarps);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), S::kTmemCols);
    tmem_relinquish();
  }

  SmemIndex si;
  const bool smem_idx = BSRC != kDense && p.smem_index;
  const int ibm = p.index_bm ? p.index_bm : BN;   // rows per index tile
  const int lcap = p.list_cap ? p.list_cap : p.tiles_cap;   // entries of this GEMM's list
  if (smem_idx) {
    // The top-k ids are an input of the call: complete before its first
    // kernel started, so they are read without waiting on the predecessor.
    si.carve(reinterpret_cast<int32_t*>(smem + S::kOffIdx), S::kWarps, p.E, tk, p.rows_cap,
             p.idmap.Eg != 0);
    for (int i = threadIdx.x; i < tk; i += S::kThreads) si.ids[i] = mapped_id(p.topk_ids, i, p.idmap);
    index_count_and_scan(si.ids, tk, p.E, ibm, si.sc, p.coalesce);
    index_scatter(si.ids, tk, p.E, si.sc, [&](int pos, int a) { si.rows[pos] = a; },
                  [](int) {});
    index_pads(p.E, p.rows_cap, si.sc, [&](int pos) { si.rows[pos] = tk; });
    // this CTA's task map: the work list with coalesced units
    for (int q = threadIdx.x; q < lcap; q += S::kThreads)
      si.tiles[q] = p.coalesce ? index_work_tile(q, p.E, p.coalesce, si.sc)
                               : index_tile(q, p.E, ibm, si.sc);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int num_tiles;
  const int4* smem_tiles = nullptr;
  // Early start: the roles wait on the previous stage only where they read
  // its output.  Gate-Up with the shared-memory index; Down whenever its
  // index was written at least two stages back (the Gate-Up waited for it
  // before letting this grid launch).
  const bool early = smem_idx || (BSRC == kDirect && p.early_weights);
  if (smem_idx) {
    num_tiles = min(p.coalesce ? si.sc.coffs[p.E] : si.sc.offs[p.E] / ibm, lcap);
    smem_tiles = si.tiles;
  } else {
    if (!early) pdl_wait();
    num_tiles = (BSRC == kDense) ? (p.dense_rows + BN - 1) / BN
                                 : min(max(__ldcg(p.num_tiles), 0), lcap);
  }
  pdl_launch_dependents();   // dependents read nothing of ours before their own wait
  const int units = num_tiles * p.m_tiles * p.splits;
  // assignment held by sorted row `pos`
  auto row_assign = [&](int pos) -> int {
    return smem_idx ? si.rows[pos] : __ldcg(p.sorted_ids + pos);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // With the shared-memory index and a contiguous token operand (Down), the
    // first kStages weight tiles are requested before waiting on the stage
    // that writes the token rows; their token loads follow the wait.
    int stage = 0;
    uint32_t phase = 0;
    long issued = 0;
    bool ok = true;
    // Contiguous token operand: one box of BN rows, or with the work list
    // (coalesce) ceil(rows / box) boxes of the index's box rows, so that a
    // tile with few valid rows loads few rows.
    const bool b_boxes = BSRC == kDirect && p.coalesce != 0;
    const int box = b_boxes ? min(ibm, BN) : BN;
    auto b_box_count = [&](const WorkUnit& w) {
      return b_boxes ? min(BN / box, (w.rows + box - 1) / box) : 1;
    };
    auto load_b = [&](uint32_t dst, uint32_t bar, int kc, int row0, int nbox) {
      for (int b = 0; b < nbox; ++b)
        tma_load_2d(dst + b * box * kKBytes, &tmB, bar, kc, row0 + b * box);
    };
    int tma_tok[S::kTmaRows > 0 ? S::kTmaRows : 1];   // token rows this warp gathers (lane 0)
    bool b_now = !(early && BSRC == kDirect);
    int deferred = 0;
    auto flush_deferred = [&]() {
      pdl_wait();
      int i = 0;
      for (UnitIter<BN, BSRC> it(units, num_tiles, p, smem_tiles); i < deferred && it.valid();
           it.advance()) {
        const WorkUnit w = it.take(p);
        const int nbox = b_box_count(w);
        for (int kt = w.kt0; kt < w.kt1 && i < deferred; ++kt, ++i)
          if (lane == 0)
            load_b(sB + i * S::kBBytes, bar_full + 8 * i, kt * S::kElemsPerStage, w.row0, nbox);
      }
      __syncwarp();
      b_now = true;
    };
    for (UnitIter<BN, BSRC> it(units, num_tiles, p, smem_tiles); ok && it.valid(); it.advance()) {
      if (warp_aborted()) break;
      const WorkUnit w = it.take(p);
      const int nbox = b_box_count(w);
      const uint32_t bytes =
          S::kAStage + (BSRC == kGather ? static_cast<uint32_t>(S::kTmaRows * kKBytes)
                                        : static_cast<uint32_t>(nbox * box * kKBytes));
      if constexpr (S::kTmaRows > 0) {
        // lane l looks up row l's token; padding rows read token 0 (their
        // columns are never stored)
        const int tl = lane < w.rows ? assignment_token(row_assign(w.row0 + lane), p) : -1;
        const int tok = tl < 0 ? 0 : tl;
#pragma unroll
        for (int j = 0; j < S::kTmaRows; ++j) tma_tok[j] = __shfl_sync(0xffffffffu, tok, j);
      }
      for (int kt = w.kt0; kt < w.kt1; ++kt) {
        if (!warp_wait((S::kShareRel ? bar_accf : bar_empty) + 8 * stage, phase ^ 1u)) {
          report_timeout(p, abort_flag);
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = bar_full + 8 * stage;
          const uint32_t a_dst = sA + stage * S::kAStage;
          const int kc = kt * S::kElemsPerStage;
          mbar_arrive_expect_tx(full, bytes);
#pragma unroll
          for (int me = 0; me < ME; ++me) {
            const int mt = w.mt * ME + me;
            if (BSRC == kGather)
              // one box of the 5-D view (K, 16 rows, gate|up, 16-row group,
              // expert): smem rows 32q..32q+15 gate rows, 32q+16.. up rows
              tma_load_5d(a_dst + me * kABytes, &tmA, full, kc, 0, 0, mt * 4, w.e);
            else
              tma_load_3d(a_dst + me * kABytes, &tmA, full, kc, mt * kTileM, w.e);
          }
          if (BSRC != kGather && b_now) load_b(sB + stage * S::kBBytes, full, kc, w.row0, nbox);
          if constexpr (S::kTmaRows > 0) {
#pragma unroll
            for (int g = 0; g < S::kTmaRows / 4; ++g)
              tma_gather4(sB + stage * S::kBBytes + g * 4 * kKBytes, &tmB, full, kc,
                          tma_tok[4 * g], tma_tok[4 * g + 1], tma_tok[4 * g + 2],
                          tma_tok[4 * g + 3]);
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == S::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (!b_now && ++deferred == S::kStages) flush_deferred();
      }
    }
    if (!b_now) flush_deferred();   // fewer stages than the ring holds
    if constexpr (S::kGatherThreads > 0) {
      // The gather threads make up the arrivals they skipped on stages we
      // issued (after an abort), so that the drain below can complete.
      if (lane == 0) *issued_slot = static_cast<int>(issued);
      named_barrier_sync(1, 32 + S::kGatherThreads);
    }
    if (lane == 0) {
      // Let our own copies land before the CTA can exit (after a normal run
      // every one of them has already been waited for by the MMA thread).
      // Long limit and no abort check: this is the drain.
      const long first = issued > S::kStages ? issued - S::kStages : 0;
      for (long i = first; i < issued; ++i)
        mbar_wait(bar_full + 8 * static_cast<int>(i % S::kStages),
                  static_cast<uint32_t>((i / S::kStages) & 1));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int ab = 0;
      uint32_t aph = 0;
      bool ok = true;
      for (UnitIter<BN, BSRC> it(units, num_tiles, p, smem_tiles); ok && it.valid(); it.advance()) {
        if (*abort_flag) break;
        const WorkUnit w = it.take(p);
        if constexpr (S::kTok2) {
          // Both token halves of the previous unit drained, then per stage
          // the 4 K steps of each half that holds valid rows (a half of
          // padding rows only is not computed).
          if (!thread_wait(bar_acce, aph ^ 1u) || !thread_wait(bar_acce + 8, aph ^ 1u)) {
            report_timeout(p, abort_flag);
            break;
          }
          tc_fence_after();
          const int halves = w.rows > kTileM ? 2 : 1;
          for (int kt = w.kt0; kt < w.kt1; ++kt) {
            if (!thread_wait(bar_full + 8 * stage, phase)) {
              report_timeout(p, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            if (BSRC == kGather) fence_proxy_async_smem();
            const uint64_t wdesc = smem_desc_sw128(sA + stage * S::kAStage);  // 2 x 128 weight rows
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (h < halves) {
                const uint64_t tdesc =
                    smem_desc_sw128(sB + stage * S::kBBytes + h * kTileM * kKBytes);
                const uint32_t d = tmem_base + static_cast<uint32_t>(h * ME * kTileM);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  mma_bf16(d, tdesc + 2 * k, wdesc + 2 * k, S::kIdesc, (kt > w.kt0 || k > 0));
              }
            }
            tc_commit(bar_empty + 8 * stage);
            if (++stage == S::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) {
            tc_commit(bar_accf);
            tc_commit(bar_accf + 8);
            aph ^= 1u;
          }
          continue;
        }
        // The MMA's N is the tile's valid rows rounded up to 16: columns of
        // padding rows are never computed (nor stored), so a wide token tile
        // costs a narrow one's MMA time when few of its rows are valid.
        // (Token-major tiles keep the full 128-row M: M is 64 or 128.)
        const int n_eff = S::kTokM ? BN : min(BN, max(16, (w.rows + 15) & ~15));
        const uint32_t idesc = (S::kIdesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(n_eff >> 3) << 17);
        if (!FP8) {
          if (!thread_wait(bar_acce + 8 * ab, aph ^ 1u)) {
            report_timeout(p, abort_flag);
            break;
          }
          tc_fence_after();
        }
        for (int kt = w.kt0; kt < w.kt1; ++kt) {
          if (FP8) {
            if (!thread_wait(bar_acce + 8 * ab, aph ^ 1u)) {
              report_timeout(p, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
          }
          if (!thread_wait(bar_full + 8 * stage, phase)) {
            report_timeout(p, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          // token rows written by cp.async (generic proxy) are read by the MMA
          // through the async proxy
          if (BSRC == kGather) fence_proxy_async_smem();
          const uint64_t bdesc = smem_desc_sw128(sB + stage * S::kBBytes);
#pragma unroll
          for (int me = 0; me < ME; ++me) {
            const uint32_t d = tmem_base + static_cast<uint32_t>((ab * ME + me) * BN);
            const uint64_t adesc = smem_desc_sw128(sA + stage * S::kAStage + me * kABytes);
#pragma unroll
            for (int k = 0; k < 4; ++k) {  // 4 MMAs of 32 bytes of K each
              const uint32_t acc = FP8 ? (k > 0) : (kt > w.kt0 || k > 0);
              if (S::kTokM)   // tokens are the M side, weight rows the N side
                mma_e4m3(d, bdesc + 2 * k, adesc + 2 * k, idesc, acc);
              else if (FP8)
                mma_e4m3(d, adesc + 2 * k, bdesc + 2 * k, idesc, acc);
              else
                mma_bf16(d, adesc + 2 * k, bdesc + 2 * k, idesc, acc);
            }
          }
          if (!S::kShareRel) tc_commit(bar_empty + 8 * stage);
          if (++stage == S::kStages) {
            stage = 0;
            phase ^= 1u;
          }
          if (FP8) {
            tc_commit(bar_accf + 8 * ab);
            if (++ab == S::kAccBufs) {
              ab = 0;
              aph ^= 1u;
            }
          }
        }
        if (!FP8 && ok) {
          tc_commit(bar_accf + 8 * ab);
          if (++ab == S::kAccBufs) {
            ab = 0;
            aph ^= 1u;
          }
        }
      }
      // Wait for our own MMAs before TMEM is freed (always: another role may
      // have given up after this thread issued its last MMA).  Long limit.
      tc_commit(bar_drain);
      mbar_wait(bar_drain, 0);
    }
    __syncwarp();
  } else if (warp < S::kRoleThreads / 32) {
    // ------------------------------------------------------------ epilogue
    if (early) pdl_wait();   // reads scales, writes outputs the chain reads
    if (smem_idx && p.write_index && blockIdx.x == 0) {
      // The later stages read the index from global memory.
      const int et = threadIdx.x - 64;
      constexpr int kET = S::kEpiThreads;
      for (int e = et; e < p.E; e += kET) p.index_out.counts[e] = si.sc.tot[e];
      for (int e = et; e <= p.E; e += kET) p.index_out.offsets[e] = si.sc.offs[e];
      for (int pos = et; pos < p.rows_cap; pos += kET) {
        const int a = si.rows[pos];
        p.index_out.sorted_ids[pos] = a;
        if (a < tk) p.index_out.inv_pos[a] = pos;
      }
      for (int a = et; a < tk; a += kET) {
        const int e = si.ids[a];
        if (e < 0 || e >= p.E) p.index_out.inv_pos[a] = -1;
      }
      for (int q = et; q < p.tiles_cap; q += kET) {
        const int4 t = p.coalesce ? index_tile(q, p.E, ibm, si.sc) : si.tiles[q];
        p.index_out.tile_expert[q] = t.x;
        reinterpret_cast<int4*>(p.index_out.tiles)[q] = t;
      }
      if (et == 0) {
        *p.index_out.num_tiles = si.sc.offs[p.E] / ibm;
        if (p.dev_status && *si.sc.flag) atomicOr(p.dev_status, kStatusExpertId);
      }
    }
    const int qd = warp & 3;          // TMEM lane quadrant this warp may read
    const int r = qd * 32 + lane;     // row of the 128-row weight tile
    // column range of this warp: all BN columns, or one half of them when
    // two warps share the quadrant (FP8 with eight epilogue warps)
    constexpr int kWarpCols = BN / (S::kEpiWarps / 4);
    const int c_base = ((warp - 2) >> 2) * kWarpCols;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(qd * 32) << 16);
    int ab = 0;
    uint32_t aph = 0;
    for (UnitIter<BN, BSRC> it(units, num_tiles, p, smem_tiles); it.valid(); it.advance()) {
      const WorkUnit w = it.take(p);
      if constexpr (S::kTok2) {
        // Token half h, lanes qd*32.. of it: lane n of the accumulator is row
        // h*128 + n of the token tile; column j is weight row j of the unit's
        // two tiles (tile j/128; Gate-Up: rows 32q..32q+15 of a tile gate,
        // 32q+16.. up, as the weight map stages them).
        const int h = (warp - 2) >> 2;
        const int n = h * kTileM + qd * 32 + lane;
        if (!warp_wait(bar_accf + 8 * h, aph)) {
          report_timeout(p, abort_flag);
          break;
        }
        tc_fence_after();
        if (h * kTileM + qd * 32 < w.rows) {   // warp-uniform: the warp holds a valid row
          const uint32_t tb = t_lane + static_cast<uint32_t>(h * ME * kTileM);
          const bool live = n < w.rows;
          if (BSRC == kGather && p.act_out != nullptr) {
            // SiLU(gate) * up of 16 channels per (tile, quadrant group), as
            // two 16-byte stores of bf16 into the token's activation row.
            // This epilogue runs between units (one accumulator set), so
            // SiLU uses the fast exponential and division intrinsics
            // (relative error ~1e-6, far below the bf16 rounding of the
            // result; a very negative gate still gives 0) instead of expf
            // and an IEEE division: the epilogue's 128 SiLUs per thread and
            // unit are otherwise ~10 % of the unit's MMA time.
            __nv_bfloat16* arow = static_cast<__nv_bfloat16*>(p.act_out) +
                                  static_cast<size_t>(w.row0 + n) * p.I;
#pragma unroll 1
            for (int g = 0; g < ME * 4; ++g) {
              const int me = g >> 2, q = g & 3;
              uint32_t gv[16], uv[16];
              tmem_ld16(tb + static_cast<uint32_t>(me * kTileM + 32 * q), gv);
              tmem_ld16(tb + static_cast<uint32_t>(me * kTileM + 32 * q + 16), uv);
              tmem_ld_wait();
              tmem_ld_bind(gv);
              tmem_ld_bind(uv);
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float g0 = __uint_as_float(gv[2 * i]), g1 = __uint_as_float(gv[2 * i + 1]);
                const float a0 = __fdividef(g0, 1.0f + __expf(-g0)) * __uint_as_float(uv[2 * i]);
                const float a1 = __fdividef(g1, 1.0f + __expf(-g1)) * __uint_as_float(uv[2 * i + 1]);
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(a0, a1);
                pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              if (live) {
                uint4* dst = reinterpret_cast<uint4*>(arow + (w.mt * ME + me) * 64 + 16 * q);
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
              }
            }
          } else {
            float* orow =
                p.out + (static_cast<size_t>(w.ks) * p.rows_cap + w.row0 + n) * p.M;
#pragma unroll 1
            for (int c = 0; c < ME * kTileM / 16; ++c) {
              uint32_t v[16];
              tmem_ld16(tb + static_cast<uint32_t>(c * 16), v);
              tmem_ld_wait();
              tmem_ld_bind(v);
              const int me = c >> 3, j0 = (c & 7) * 16;
              int col0 = (w.mt * ME + me) * kTileM + j0;
              if (BSRC == kGather) {
                const int feat = (w.mt * ME + me) * 64 + 16 * (j0 >> 5);
                col0 = (j0 & 31) < 16 ? feat : p.I + feat;
              }
              if (live && col0 + 16 <= p.M) {
                if (p.out_bf16) {
                  store_bf16x16(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                    static_cast<size_t>(w.row0 + n) * p.M + col0, v);
                } else {
                  float4* dst = reinterpret_cast<float4*>(orow + col0);
#pragma unroll
                  for (int q4 = 0; q4 < 4; ++q4)
                    dst[q4] = make_float4(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1]),
                                          __uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3]));
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acce + 8 * h);
        aph ^= 1u;
        continue;
      }
      if (!FP8) {
        if (!warp_wait(bar_accf + 8 * ab, aph)) {
          report_timeout(p, abort_flag);
          break;
        }
        tc_fence_after();
        const bool fuse = BSRC == kGather && p.act_out != nullptr;
#pragma unroll 1
        for (int me = 0; me < ME; ++me) {
        const int mt = w.mt * ME + me;
        int col;
        bool col_ok = true;
        const int feat = mt * 64 + qd * 16 + (lane & 15);  // Gate-Up: this lane's channel
        if (BSRC == kGather) {
          col = lane < 16 ? feat : p.I + feat;
        } else {
          col = mt * kTileM + r;
          col_ok = col < p.M;
        }
        float* outp = p.out + (static_cast<size_t>(w.ks) * p.rows_cap + w.row0) * p.M + col;
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) {
          if (c * 16 < w.rows) {
            uint32_t v[16];
            tmem_ld16(t_lane + static_cast<uint32_t>((ab * ME + me) * BN + c * 16), v);
            tmem_ld_wait();
            if (fuse) {
              // lanes 0..15 hold gate, 16..31 the matching up: swap halves, then
              // lanes 0..15 finish columns 0..7 of the chunk, lanes 16..31 8..15.
              const bool lo = lane < 16;
              __nv_bfloat16* arow = static_cast<__nv_bfloat16*>(p.act_out) +
                                    static_cast<size_t>(w.row0) * p.I + feat;
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const float mine_a = __uint_as_float(v[jj]);
                const float mine_b = __uint_as_float(v[8 + jj]);
                const float peer_a = __shfl_xor_sync(0xffffffffu, mine_a, 16);
                const float peer_b = __shfl_xor_sync(0xffffffffu, mine_b, 16);
                const float g = lo ? mine_a : peer_b;
                const float u = lo ? peer_a : mine_b;
                const int n = c * 16 + (lo ? jj : 8 + jj);
                if (n < w.rows)
                  arow[static_cast<size_t>(n) * p.I] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * u);
              }
            } else if (p.out_bf16) {
              __nv_bfloat16* outb = reinterpret_cast<__nv_bfloat16*>(p.out) +
                                    static_cast<size_t>(w.row0) * p.M + col;
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = c * 16 + j;
                if (n < w.rows && col_ok)
                  outb[static_cast<size_t>(n) * p.M] = __float2bfloat16_rn(__uint_as_float(v[j]));
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = c * 16 + j;
                if (n < w.rows && col_ok) outp[static_cast<size_t>(n) * p.M] = __uint_as_float(v[j]);
              }
            }
          }
        }
        }  // me
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acce + 8 * ab);
        if (++ab == S::kAccBufs) {
          ab = 0;
          aph ^= 1u;
        }
      } else if constexpr (S::kTokM) {
        // Token-major FP8 tile: lane n of the accumulator is token row n of
        // the tile, column j weight row j of the 128-row tile (Gate-Up: rows
        // 32q..32q+15 gate, 32q+16..32q+31 up, as the weight map stages
        // them).  Per K block a thread needs its token's scale and one
        // weight-block scale per 16 columns, all fetched three blocks ahead.
        const int n = qd * 32 + lane;
        const bool live = qd * 32 < w.rows;   // warp-uniform: any valid row
        const int KB = p.kt_total;
        int srow = -1;
        if (n < w.rows)
          srow = p.scale_by_token ? assignment_token(row_assign(w.row0 + n), p) : w.row0 + n;
        const float* bsp = srow >= 0 ? p.b_scale + static_cast<size_t>(srow) * KB : nullptr;
        const size_t wblk = static_cast<size_t>(w.e) * (p.M >> 7);
        const float* wsg = p.w_scale +
            (wblk + (BSRC == kGather ? (w.mt * 64) >> 7 : w.mt)) * KB;   // gate (or only)
        const float* wsu = p.w_scale +
            (wblk + (BSRC == kGather ? (p.I + w.mt * 64) >> 7 : w.mt)) * KB;   // up
        auto sx_at = [&](int kt) { return (bsp && kt < w.kt1) ? __ldg(bsp + kt) : 0.f; };
        auto sg_at = [&](int kt) { return kt < w.kt1 ? __ldg(wsg + kt) : 0.f; };
        auto su_at = [&](int kt) { return kt < w.kt1 ? __ldg(wsu + kt) : 0.f; };
        float sx0 = sx_at(w.kt0), sx1 = sx_at(w.kt0 + 1), sx2 = sx_at(w.kt0 + 2);
        float sg0 = sg_at(w.kt0), sg1 = sg_at(w.kt0 + 1), sg2 = sg_at(w.kt0 + 2);
        float su0 = su_at(w.kt0), su1 = su_at(w.kt0 + 1), su2 = su_at(w.kt0 + 2);
        uint64_t acc2[kWarpCols / 2];
#pragma unroll
        for (int j = 0; j < kWarpCols / 2; ++j) acc2[j] = 0ull;
        bool ok = true;
        for (int kt = w.kt0; kt < w.kt1; ++kt) {
          const float sg = sx0 * sg0, su = sx0 * su0;
          sx0 = sx1, sx1 = sx2, sx2 = sx_at(kt + 3);
          sg0 = sg1, sg1 = sg2, sg2 = sg_at(kt + 3);
          su0 = su1, su1 = su2, su2 = su_at(kt + 3);
          if (!warp_wait(bar_accf + 8 * ab, aph)) {
            report_timeout(p, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          if (live) {
            uint32_t v[kWarpCols / 16][16];
#pragma unroll
            for (int g = 0; g < kWarpCols / 16; ++g)
              tmem_ld16(t_lane + static_cast<uint32_t>(ab * BN + c_base + g * 16), v[g]);
            tmem_ld_wait();
            const uint64_t s_g = pack_f32x2(sg, sg), s_u = pack_f32x2(su, su);
#pragma unroll
            for (int g = 0; g < kWarpCols / 16; ++g) {
              tmem_ld_bind(v[g]);
              const bool gate = BSRC != kGather || (((c_base + g * 16) & 31) < 16);
              const uint64_t sc = gate ? s_g : s_u;
#pragma unroll
              for (int h = 0; h < 8; ++h)
                acc2[g * 8 + h] = fma_f32x2(pack_u32x2(v[g][2 * h], v[g][2 * h + 1]), sc,
                                            acc2[g * 8 + h]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acce + 8 * ab);
          if (++ab == S::kAccBufs) {
            ab = 0;
            aph ^= 1u;
          }
        }
        if (!ok) break;
        if (BSRC == kGather && p.g_act) {
          // SiLU(gate)*up: column group g (16 gate rows) and g + 1 (the up
          // rows of the same 16 channels) give 16 values of the token's row
          // of I, stored as fp32 (the activation stage quantises them).
          static_assert(kWarpCols % 32 == 0, "a warp's columns hold whole gate/up pairs");
          if (n < w.rows) {
            float* arow = p.out + static_cast<size_t>(w.row0 + n) * p.I;
#pragma unroll
            for (int g = 0; g < kWarpCols / 16; g += 2) {
              const int feat = w.mt * 64 + 16 * ((c_base + g * 16) >> 5);
              if (feat + 16 <= p.I) {
                float av[16];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  float g0, g1, u0, u1;
                  unpack_f32x2(acc2[g * 8 + q], g0, g1);
                  unpack_f32x2(acc2[(g + 1) * 8 + q], u0, u1);
                  av[2 * q] = silu_mul_fast(g0, u0);
                  av[2 * q + 1] = silu_mul_fast(g1, u1);
                }
                float4* dst = reinterpret_cast<float4*>(arow + feat);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  dst[q] = make_float4(av[4 * q], av[4 * q + 1], av[4 * q + 2], av[4 * q + 3]);
              }
            }
          }
        } else if (n < w.rows) {
          float* orow = p.out + (static_cast<size_t>(w.ks) * p.rows_cap + w.row0 + n) * p.M;
#pragma unroll
          for (int g = 0; g < kWarpCols / 16; ++g) {
            const int j0 = c_base + g * 16;
            int col0 = w.mt * kTileM + j0;
            if (BSRC == kGather) {
              const int feat = w.mt * 64 + 16 * (j0 >> 5);
              col0 = (j0 & 31) < 16 ? feat : p.I + feat;
            }
            if (col0 + 16 <= p.M) {
              uint32_t vv[16];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                float a, b;
                unpack_f32x2(acc2[g * 8 + q], a, b);
                vv[2 * q] = __float_as_uint(a);
                vv[2 * q + 1] = __float_as_uint(b);
              }
              if (p.out_bf16) {
                store_bf16x16(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                  static_cast<size_t>(w.row0 + n) * p.M + col0, vv);
              } else {
                float4* dst = reinterpret_cast<float4*>(orow + col0);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  dst[q] = make_float4(__uint_as_float(vv[4 * q]), __uint_as_float(vv[4 * q + 1]),
                                       __uint_as_float(vv[4 * q + 2]), __uint_as_float(vv[4 * q + 3]));
              }
            }
          }
        }
      } else {
        const int feat = w.mt * 64 + qd * 16 + (lane & 15);  // Gate-Up: this lane's channel
        int col;
        bool col_ok = true;
        if (BSRC == kGather) {
          col = lane < 16 ? feat : p.I + feat;
        } else {
          col = w.mt * kTileM + r;
          col_ok = col < p.M;
        }
        float* outp = p.out + (static_cast<size_t>(w.ks) * p.rows_cap + w.row0) * p.M + col;
        // The token-operand scale of column n is the same for every row, so
        // each epilogue warp stages its own columns' scales in its own
        // shared-memory slots once per K block (lane j loads column
        // c_base + j) and reads them back as broadcast 16-byte loads; a
        // __syncwarp publishes them, so the warps never wait on one another
        // (a block-wide barrier per K block cost 4-8 % of the FP8 decode
        // GEMMs).  The slot written is never the one being read.
        const int KB = p.kt_total;
        float* sxw = sx_buf + (warp - 2) * 2 * kWarpCols;
        const int jc = c_base + lane;   // this lane's column
        int srow = -1;
        if (lane < kWarpCols && jc < w.rows)
          srow = p.scale_by_token ? assignment_token(row_assign(w.row0 + jc), p) : w.row0 + jc;
        const float* bsp = srow >= 0 ? p.b_scale + static_cast<size_t>(srow) * KB : nullptr;
        const int blk = (BSRC == kGather) ? ((lane < 16 ? w.mt * 64 : p.I + w.mt * 64) >> 7) : w.mt;
        const float* wsp = p.w_scale + (static_cast<size_t>(w.e) * (p.M >> 7) + blk) * KB;
        // Scales are fetched two K blocks ahead of their use: the epilogue is
        // the busy role here, so a load issued in the block that needs it
        // would put its latency on the critical path.
        auto sx_at = [&](int kt) { return (bsp && kt < w.kt1) ? __ldg(bsp + kt) : 0.f; };
        auto sw_at = [&](int kt) { return kt < w.kt1 ? __ldg(wsp + kt) : 0.f; };
        if (lane < kWarpCols) sxw[lane] = sx_at(w.kt0);
        float sx_n1 = sx_at(w.kt0 + 1), sx_n2 = sx_at(w.kt0 + 2);
        float sw_0 = sw_at(w.kt0), sw_1 = sw_at(w.kt0 + 1), sw_2 = sw_at(w.kt0 + 2);
        __syncwarp();
        // this warp's columns c_base.. in packed pairs (fma.rn.f32x2: two
        // fp32 FMAs, each rounded as fmaf)
        uint64_t acc2[kWarpCols / 2];
#pragma unroll
        for (int j = 0; j < kWarpCols / 2; ++j) acc2[j] = 0ull;
        const int wrows = w.rows - c_base;   // valid columns from c_base on
        bool ok = true;
        int cur = 0;
        for (int kt = w.kt0; kt < w.kt1; ++kt) {
          const float sw = sw_0;
          sw_0 = sw_1;
          sw_1 = sw_2;
          sw_2 = sw_at(kt + 3);
          const float sx_stage = sx_n1;   // published below for kt + 1
          sx_n1 = sx_n2;
          sx_n2 = sx_at(kt + 3);
          if (!warp_wait(bar_accf + 8 * ab, aph)) {
            report_timeout(p, abort_flag);
            ok = false;
          }
          if (ok) {
            tc_fence_after();
            const float* sxb = sxw + cur * kWarpCols;   // this warp's columns
            const uint64_t sw2 = pack_f32x2(sw, sw);
            // TMEM reads two 16-column chunks at a time, one wait per pair
            constexpr int kLdBatch = kWarpCols / 16 < 2 ? kWarpCols / 16 : 2;
#pragma unroll
            for (int c0 = 0; c0 < kWarpCols / 16; c0 += kLdBatch) {
              if (c0 * 16 < wrows) {
                uint32_t v[kLdBatch][16];
#pragma unroll
                for (int g = 0; g < kLdBatch; ++g)
                  if ((c0 + g) * 16 < wrows)
                    tmem_ld16(t_lane + static_cast<uint32_t>(ab * BN + c_base + (c0 + g) * 16),
                              v[g]);
                tmem_ld_wait();
#pragma unroll
                for (int g = 0; g < kLdBatch; ++g) {
                  if ((c0 + g) * 16 >= wrows) continue;
                  tmem_ld_bind(v[g]);
                  const int c = c0 + g;
#pragma unroll
                  for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 s4 =
                        *reinterpret_cast<const float4*>(sxb + c * 16 + 4 * q4);
                    const int h = (c * 16 + 4 * q4) / 2;
                    const uint64_t s01 = mul_f32x2(pack_f32x2(s4.x, s4.y), sw2);
                    const uint64_t s23 = mul_f32x2(pack_f32x2(s4.z, s4.w), sw2);
                    acc2[h] = fma_f32x2(pack_u32x2(v[g][4 * q4 + 0], v[g][4 * q4 + 1]), s01, acc2[h]);
                    acc2[h + 1] =
                        fma_f32x2(pack_u32x2(v[g][4 * q4 + 2], v[g][4 * q4 + 3]), s23, acc2[h + 1]);
                  }
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acce + 8 * ab);
            if (++ab == S::kAccBufs) {
              ab = 0;
              aph ^= 1u;
            }
          }
          cur ^= 1;
          if (lane < kWarpCols) sxw[cur * kWarpCols + lane] = sx_stage;
          __syncwarp();
          if (!ok) break;
        }
        if (!ok) break;
        __nv_bfloat16* outb = reinterpret_cast<__nv_bfloat16*>(p.out) +
                              static_cast<size_t>(w.row0) * p.M + col;
#pragma unroll
        for (int h = 0; h < kWarpCols / 2; ++h) {
          float a0, a1;
          unpack_f32x2(acc2[h], a0, a1);
          const int n = c_base + 2 * h;
          if (p.out_bf16) {
            if (n < w.rows && col_ok) outb[static_cast<size_t>(n) * p.M] = __float2bfloat16_rn(a0);
            if (n + 1 < w.rows && col_ok)
              outb[static_cast<size_t>(n + 1) * p.M] = __float2bfloat16_rn(a1);
          } else {
            if (n < w.rows && col_ok) outp[static_cast<size_t>(n) * p.M] = a0;
            if (n + 1 < w.rows && col_ok) outp[static_cast<size_t>(n + 1) * p.M] = a1;
          }
        }
      }
    }
  } else if (BSRC == kGather) {
    // ------------------------------------------------------------ token gather
    // Thread t copies 16-byte chunk c = t % 8 of rows n = t/8 + 4*NG*i; a
    // warp instruction covers four whole 128-byte rows.  Padding rows are not
    // copied: their MMA columns are never stored.
    constexpr int kR = S::kRowsPerGatherThread;
    constexpr int kRowStep = 4 * (S::kGatherWarps > 0 ? S::kGatherWarps : 1);
    const int t = threadIdx.x - S::kRoleThreads;
    const int c = t & 7;
    const int r0 = t >> 3;
    const uint8_t* rows = static_cast<const uint8_t*>(p.b_rows) + c * 16;
    if (early) pdl_wait();   // the token rows may come from the previous stage
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int tok[kR];
    bool tok_ready = false;       // tok[] already holds the current unit's rows
    long garr = 0;                // stages this thread has arrived on
    for (UnitIter<BN, BSRC> it(units, num_tiles, p, smem_tiles); ok && it.valid(); it.advance()) {
      if (*abort_flag) break;
      const WorkUnit w = it.take(p);
      if (!tok_ready) {
#pragma unroll
        for (int i = 0; i < kR; ++i) {
          const int n = S::kTmaRows + r0 + kRowStep * i;
          tok[i] = n < w.rows ? assignment_token(row_assign(w.row0 + n), p) : -1;
        }
      }
      // The next unit's rows are looked up in two steps spread over this
      // unit's first stages (its task-map entry, then its sorted rows), so
      // neither dependent load stalls the copies of the current unit.
      int tok_next[kR];
      tok_ready = false;
      const int nk = w.kt1 - w.kt0;
      const int step_a = nk > 1 ? 1 : 0;           // sorted-row loads issued
      const int step_b = nk > 2 ? 2 : nk - 1;      // turned into token rows
      for (int kt = w.kt0; kt < w.kt1; ++kt) {
        if (!thread_wait((S::kShareRel ? bar_accf : bar_empty) + 8 * stage, phase ^ 1u)) {
          report_timeout(p, abort_flag);
          ok = false;
          break;
        }
        const uint32_t b_dst = sB + stage * S::kBBytes;
        const uint8_t* src = rows + static_cast<size_t>(kt) * kKBytes;
#pragma unroll
        for (int i = 0; i < kR; ++i) {
          const int n = S::kTmaRows + r0 + kRowStep * i;
          if (tok[i] >= 0)
            cp_async_16(b_dst + n * kKBytes + ((c ^ (n & 7)) << 4),
                        src + static_cast<size_t>(tok[i]) * p.b_row_bytes);
        }
        cp_async_arrive_noinc(bar_full + 8 * stage);
        ++garr;
        if (++stage == S::kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (it.has_next()) {
          const int i_kt = kt - w.kt0;
          if (i_kt == step_a) {
            const int4 tn = it.next;
#pragma unroll
            for (int i = 0; i < kR; ++i) {
              const int n = S::kTmaRows + r0 + kRowStep * i;
              tok_next[i] = n < tn.z ? row_assign(tn.y + n) : -1;   // assignment for now
            }
          }
          if (i_kt == step_b) {
#pragma unroll
            for (int i = 0; i < kR; ++i)
              tok_next[i] = tok_next[i] >= 0 ? assignment_token(tok_next[i], p) : -1;
            tok_ready = true;
          }
        }
      }
      if (tok_ready) {
#pragma unroll
        for (int i = 0; i < kR; ++i) tok[i] = tok_next[i];
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy outlives the CTA
    // Stages the TMA warp issued but this thread skipped (it gave up first):
    // arrive on them so that their phases, and the TMA warp's drain, can
    // complete.  Stage i's previous phase (i - kStages) needs no arrival of
    // ours any more (every thread arrived on it before the TMA warp could
    // reissue the stage), so wait for it to complete before arriving.
    named_barrier_sync(1, 32 + S::kGatherThreads);
    const long issued_total = *issued_slot;
    for (long i = garr; i < issued_total; ++i) {
      const int s = static_cast<int>(i % S::kStages);
      if (i >= S::kStages)
        mbar_wait(bar_full + 8 * s, static_cast<uint32_t>(((i - S::kStages) / S::kStages) & 1));
      mbar_arrive(bar_full + 8 * s);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
}

template <int FP8, int BN, int BSRC, int ME>
__global__ void __launch_bounds__(GemmShape<FP8, BN, BSRC, ME>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  gemm_cta<FP8, BN, BSRC, ME>(tmA, tmB, p, smem_raw);
}

template <int FP8, int BN, int BSRC, int ME = 1>
cudaError_t launch_gemm_inst(int grid, cudaStream_t st, bool pdl, const CUtensorMap& a,
                             const CUtensorMap& b, const GemmParams& p) {
  using S = GemmShape<FP8, BN, BSRC, ME>;
  auto kern = moe_gemm_kernel<FP8, BN, BSRC, ME>;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !configured[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kMaxGemmSmem));
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  size_t smem = S::kSmemBytes;
  if (BSRC != kDense && p.smem_index)
    smem += SmemIndex::bytes(S::kWarps, p.E, p.T * p.topk, p.rows_cap,
                             p.list_cap ? p.list_cap : p.tiles_cap);
  if (smem > kMaxGemmSmem) return cudaErrorInvalidValue;
  return launch_kernel(kern, dim3(grid), dim3(S::kThreads), smem, st, pdl, a, b, p);
}

template <int FP8, int BSRC>
cudaError_t launch_gemm_bn(int bn, int grid, cudaStream_t st, bool pdl, const CUtensorMap& a,
                           const CUtensorMap& b, const GemmParams& p, int me = 1) {
  if (me == 2) {
    if constexpr (!FP8) {
      if (bn == 128) return launch_gemm_inst<FP8, 128, BSRC, 2>(grid, st, pdl, a, b, p);
      if (bn == 256) return launch_gemm_inst<FP8, 256, BSRC, 2>(grid, st, pdl, a, b, p);
    }
    return cudaErrorInvalidValue;
  }
  switch (bn) {
    case 16: return launch_gemm_inst<FP8, 16, BSRC>(grid, st, pdl, a, b, p);
    case 32: return launch_gemm_inst<FP8, 32, BSRC>(grid, st, pdl, a, b, p);
    case 64: return launch_gemm_inst<FP8, 64, BSRC>(grid, st, pdl, a, b, p);
    case 128: return launch_gemm_inst<FP8, 128, BSRC>(grid, st, pdl, a, b, p);
    case 256:
      if constexpr (!FP8) return launch_gemm_inst<FP8, 256, BSRC>(grid, st, pdl, a, b, p);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
