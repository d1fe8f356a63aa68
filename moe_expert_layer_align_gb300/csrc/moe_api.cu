// moe_api.cu — the C ABI (include/moe.h): argument checks, the planner that
// picks the row tile and split-K counts, workspace layout, TMA descriptors,
// and the PDL-chained launch of the stages.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {
namespace {

// The split-K choice is planned for this many persistent CTAs so that the
// plan, and with it the workspace size, is a function of the shape alone.
constexpr int kPlanCtas = 152;
constexpr int kMaxSplits = 32;
// Largest T*k for which GEMM CTAs rebuild the routing index themselves.
constexpr int kSmemIndexMaxAssignments = 4096;
// Above this many assignments the index is built over chunks by several CTAs.
constexpr int kSplitIndexMinAssignments = 2048;
// Coalesced work list the planner uses over 16- and 32-row index tiles
// (0: none).
constexpr int kPlanCoalesce = 0;
// 256-row token tiles: the planner gives the Down GEMM 128-row tiles of a
// work list where an active expert holds at least this many rows on average.
constexpr int kPlanDownSplitMinRows = 256;
// Router GEMM split-K count bound: one top-k warp per token sums at most 4
// partials at once; the block top-k (few tokens) up to 32.
constexpr int kRouterMaxSplitsHost = 4;
constexpr int kRouterMaxSplitsWide = 32;
constexpr int kRouterWideMaxT = 256;

enum {
  kOffCounts, kOffOffsets, kOffSorted, kOffTileExpert, kOffTiles, kOffInvPos, kOffNumTiles,
  kOffIdxScratch, kOffXq, kOffXs, kOffXsRows, kOffG, kOffA, kOffAs, kOffY, kOffRouterP,
  kOffCounter, kOffRouteHist, kOffWorkTiles, kOffNumWorkTiles, kNumOff
};

struct Plan {
  // k, E: assignments per token and experts of the index and the weights
  // (routed + shared); the IdMap maps topk_ids onto them.
  int T, H, I, E, k, bm, fp8, out_bf16;
  int co;                  // work list written by the index: tiles of up to co rows (0: none)
  int co1, co2;            // work-list tile rows each GEMM takes (0: the task map)
  int bn1, bn2;            // token rows of each GEMM kernel's tile
  int y16;                 // unsplit Down: bf16 output rows (else fp32 partials)
  int bn;                  // token rows of the GEMM kernels' tile: co, else bm
  int w8;                  // w8a16: e4m3 weights dequantised on chip, bf16 activations
  IdMap map;
  float w_shared;
  int tiles_cap, rows_cap;
  int work_cap;            // work-list entries (tiles of co rows; co < bm needs more)
  int s1, kts1, kt1, mt1;  // Gate-Up: splits, k-tiles per split, k-tiles, weight tiles
  int s2, kts2, kt2, mt2;  // Down
  int me1, me2;            // weight tiles per work unit (2: large token tiles, bf16)
  int fused_act;           // SiLU-and-mul in the Gate-Up epilogue
  int g_act;               // the Gate-Up epilogue stores SiLU(gate)*up in fp32 (FP8)
  int ord1, ord2;          // unit order per GEMM: 1 weight-tile-major, 2 token-tile-major
  int smem_index;          // GEMM CTAs rebuild the index in shared memory
  int align_quant;         // FP8: x-quant on the one-CTA index kernel's other blocks
  int xs_by_token;         // FP8: the Gate-Up reads x scales per token (no per-row copy)
  size_t off[kNumOff];
  int split_index;         // index built by the count / scan / scatter kernels
  size_t total;
  // in-path router (moe_forward_routed)
  int routed;
  int route_fused;         // router GEMM, top-k, x-quant and index in one launch
  int rp_bn, rp_rows_cap, rp_splits, rp_kts, rp_kt, rp_mt;
  size_t rp_bytes;
  int rp_owners_cap;       // fused routing: most token-owning CTAs (histogram rows)
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool valid_bm(int bm, int fp8) {
  return bm == 16 || bm == 32 || bm == 64 || bm == 128 || (bm == 256 && !fp8);
}

int64_t tiles_cap_of(int64_t T, int64_t k, int64_t E, int64_t bm) {
  const int64_t tk = T * k;
  return (tk + bm - 1) / bm + std::min(E, tk);
}

// Row tile: the smallest of 16..128 that holds 1.5x the mean rows of an
// active expert, so that most experts occupy one tile.
// FP8 takes 128 where this gives 64: 128-row FP8 tiles run token-major with
// per-thread block scales, cheaper to promote than the swap-AB 64-row tile
// (DeepSeek-shaped layer at T=1024: 2.23 ms against 2.47 ms).
// bf16 takes 256 where an active expert holds 128 rows or more on average and
// both GEMMs pair two weight tiles per unit (`pair`): the token-major tile
// (one or two 128-row token halves against one N = 256 operand of both
// weight tiles) stages 64 MACs per operand byte with two halves against the
// 128-row tiles' 43, and issues half as many MMAs per stage even with one
// (Mixtral-shaped layer at T=2048: 1366 -> 1248 us; T=512, 128 rows per
// expert: 576 -> 527 us; Qwen3-shaped T=4096, 256 +- 16 rows: 445 -> 422 us;
// at 64 rows, Qwen3-shaped T=1024, it measured 279 -> 284 us).
// Mean rows of an active expert: T*k assignments over the experts that
// uniform routing is expected to reach.
double mean_rows(int T, int k, int E) {
  const double tk = static_cast<double>(T) * k;
  const double active = E * (1.0 - std::pow(1.0 - static_cast<double>(k) / E, T));
  return tk / std::max(1.0, std::min(active, tk));
}

int auto_bm(int T, int k, int E, int fp8, bool pair) {
  const double mean = mean_rows(T, k, E);
  if (!fp8 && pair && mean >= 128) return 256;
  const int cap = 128;
  int bm = 16;
  while (bm < cap && bm < 1.5 * mean) bm *= 2;
  return (fp8 && bm == 64) ? 128 : bm;
}

// Expected number of row tiles under uniform routing (a planning estimate;
// the kernels read the true count from the index).
int est_tiles(int T, int k, int E, int bm, int tiles_cap) {
  const double tk = static_cast<double>(T) * k;
  const double active = E * (1.0 - std::pow(1.0 - static_cast<double>(k) / E, T));
  const double per = tk / std::max(1.0, active);
  const double est = std::max(1.0, active) * std::ceil(per / bm);
  return static_cast<int>(std::min<double>(tiles_cap, std::max(1.0, std::round(est))));
}

// Unit order of a GEMM with mk units per token tile (weight tiles x
// splits).  Token-tile-major keeps all units of a token tile together; an
// expert's token tiles then reach each of its weight tiles mk units apart,
// within one wave of CTAs when (its token tiles) x mk <= the CTAs, so the
// later reads of the weight tile hit L2 (measured on the Qwen3-shaped
// layer at T=4096: Down 179 -> 137 us; DeepSeek-shaped FP8 at T=4096: Down
// 1.53 -> 1.18 ms).  Otherwise (Mixtral-shaped prefill: four token tiles
// per expert, 112 units each) weight-tile-major keeps the token tiles of a
// weight tile adjacent instead (Gate-Up at T=2048: 891 us against 1078).
// The expert's token tiles are estimated under uniform routing with two
// standard deviations of headroom for the ragged last tile.
int unit_order(int T, int k, int E, int bm, int mk) {
  const double tk = static_cast<double>(T) * k;
  const double active = E * (1.0 - std::pow(1.0 - static_cast<double>(k) / E, T));
  const double per = tk / std::max(1.0, active);
  const double tiles = std::ceil((per + 2.0 * std::sqrt(per)) / bm);
  return tiles * mk <= kPlanCtas ? 2 : 1;
}

// Split-K count minimising (waves of units) x (k-tiles per unit) plus the
// cost of writing and re-reading fp32 partial rows, in k-tile units.
// Fixed cost of a bf16 work unit in pipeline stages (its pipeline fill and
// drain and its epilogue), charged per wave in choose_split.  Without it the
// planner split the Mixtral-shaped Down (K = 14336) 7 ways at T=16..64 and
// 16 ways at T=4: now 4 and 7 (T=64 457 -> 449 us, T=4 353 -> 339 us); the
// Qwen3-shaped Down drops its split at T=4 and 8 (84.5 -> 80.4 us, 109.1 ->
// 105.6 us).  FP8 and w8a16 units, whose per-K-block work is heavier, keep
// the plain count: their split Gate-Ups at DeepSeek-shaped T=1 and 4
// measured 2.5-4.5 % faster than the unsplit ones this cost would choose.
constexpr double kPlanUnitCost = 4.0;

void choose_split(int m_tiles, int kt_total, int tiles, int bn, int* s_out, int* kts_out,
                  int max_splits = kMaxSplits, bool large_tiles_unsplit = true,
                  double unit_cost = 0.0) {
  double best = 1e300;
  int bs = 1, bk = kt_total;
  // Large token tiles: unsplit.  Every split adds a full fp32 partial slice
  // of the rows, written here and re-read by the reduction, where an
  // unsplit GEMM stores bf16 rows; with those, one split measured best even
  // where it leaves SMs idle (Mixtral-shaped Down at T=512, 128 units for
  // 152 SMs: 507 us per layer against 521 / 525 / 536 us with 2 / 3 / 4
  // splits; T=2048: 1117 against 1125 / 1153; Qwen3- and DeepSeek-shaped
  // prefill: 1 by 2-50 %).  (Before the bf16 rows, 3 splits were 10 % faster
  // than 1 on that Down GEMM.)  The router GEMM writes fp32 partials either
  // way and has only 2E/128 weight tiles, so it keeps the split search.
  if (bn >= 128 && large_tiles_unsplit) {
    *s_out = 1;
    *kts_out = kt_total;
    return;
  }
  for (int s = 1; s <= std::min(max_splits, kt_total); ++s) {
    const int kts = (kt_total + s - 1) / s;
    const int se = (kt_total + kts - 1) / kts;
    if (se != s) continue;            // same as a smaller count
    if (s > 1 && kts < 4) break;      // keep the pipeline at least 4 stages deep
    const double units = static_cast<double>(m_tiles) * se * tiles;
    const double grid = std::min<double>(kPlanCtas, units);
    const double waves = std::ceil(units / grid);
    const double extra = se > 1 ? 0.5 * units * bn / 16.0 / kPlanCtas : 0.0;
    const double cost = waves * (kts + unit_cost) + extra;
    if (cost < best - 1e-9) {
      best = cost;
      bs = se;
      bk = kts;
    }
  }
  *s_out = bs;
  *kts_out = bk;
}

moe_status check_shape(const moe_shape* s) {
  if (!s) return MOE_ERR_ARG;
  if (s->mode != MOE_BF16 && s->mode != MOE_FP8_W8A8 && s->mode != MOE_W8A16)
    return MOE_ERR_DTYPE;
  if (s->out_dtype != MOE_OUT_F32 && s->out_dtype != MOE_OUT_BF16) return MOE_ERR_DTYPE;
  const int fp8 = s->mode == MOE_FP8_W8A8;
  const int w8 = s->mode == MOE_W8A16;
  if (w8 && (s->H % 128 || s->I % 128 || s->block_m == 256)) return MOE_ERR_SHAPE;
  if (s->T < 1 || s->H < 128 || s->I < 64 || s->E < 1 || s->E > 512 || s->k < 1 || s->k > s->E)
    return MOE_ERR_SHAPE;
  if (s->H % 128 || s->I % (fp8 ? 128 : 64)) return MOE_ERR_SHAPE;
  if (static_cast<int64_t>(s->T) * s->k >= (int64_t(1) << 31) / 2) return MOE_ERR_SHAPE;
  if (s->block_m != 0 && !valid_bm(s->block_m, fp8)) return MOE_ERR_SHAPE;
  return MOE_OK;
}

// Router plan: row tile, split-K count and workspace for the partial sums.
struct RouterPlan {
  int bn, rows_cap, splits, kts, kt, mt;
  size_t bytes;
};
bool router_plan(int T, int H, int E, RouterPlan* r, bool fused_front = false);

// Shared experts and the expert-parallel range (moe_forward_opts /
// moe_align_opts) as an IdMap; MOE_ERR_SHAPE on inconsistent values.
moe_status make_idmap(int k, int E, int n_shared, int e0, int Eg, IdMap* m) {
  if (n_shared < 0 || n_shared > 8 || E + n_shared > 512) return MOE_ERR_SHAPE;
  if (Eg < 0 || (Eg > 0 && (e0 < 0 || e0 + E > Eg)) || (Eg == 0 && e0 != 0)) return MOE_ERR_SHAPE;
  m->k = k;
  m->kk = k + n_shared;
  m->E = E;
  m->e0 = Eg > 0 ? e0 : 0;
  m->Eg = Eg;
  return MOE_OK;
}

moe_status make_plan(const moe_shape* s, const moe_forward_opts* o, Plan* p, bool routed = false) {
  moe_status st = check_shape(s);
  if (st != MOE_OK) return st;
  std::memset(p, 0, sizeof(*p));
  if (routed) {
    // the router's ids arrive in-chain: the shared-memory index (which reads
    // them before waiting on the previous stage) is off, and the id mapping
    // variants are not combined with the in-path router
    RouterPlan r;
    const bool fused = o && o->fuse_routing == 1 && !o->num_shared_experts && !o->ep_num_experts;
    if (!router_plan(s->T, s->H, s->E, &r, fused) || s->k > 32) return MOE_ERR_SHAPE;
    if (o && (o->smem_index == 1 || o->num_shared_experts || o->ep_num_experts)) return MOE_ERR_SHAPE;
    p->routed = 1;
    p->rp_bn = r.bn, p->rp_rows_cap = r.rows_cap, p->rp_splits = r.splits, p->rp_kts = r.kts;
    p->rp_kt = r.kt, p->rp_mt = r.mt, p->rp_bytes = r.bytes;
  }
  const int n_shared = o ? o->num_shared_experts : 0;
  st = make_idmap(s->k, s->E, n_shared, o ? o->ep_first_expert : 0, o ? o->ep_num_experts : 0,
                  &p->map);
  if (st != MOE_OK) return st;
  if (static_cast<int64_t>(s->T) * p->map.kk >= (int64_t(1) << 31) / 2) return MOE_ERR_SHAPE;
  p->w_shared = (o && o->shared_expert_weight != 0.f) ? o->shared_expert_weight : 1.0f;
  p->T = s->T, p->H = s->H, p->I = s->I;
  p->E = s->E + n_shared;   // experts in the weights and the index
  p->k = p->map.kk;         // assignments per token
  p->fp8 = s->mode == MOE_FP8_W8A8;
  p->w8 = s->mode == MOE_W8A16;
  p->out_bf16 = s->out_dtype == MOE_OUT_BF16;
  const bool pair = !p->fp8 && !p->w8 && !(o && o->single_weight_tile) &&
                    (s->I / 64) % 2 == 0 && (s->H / 128) % 2 == 0;
  p->bm = s->block_m ? s->block_m : auto_bm(p->T, p->k, p->E, p->fp8, pair);
  // Coalesced work list over a 16- or 32-row index.
  if (o && !(o->coalesce_rows == 0 || o->coalesce_rows == -1 || o->coalesce_rows == 32 ||
             o->coalesce_rows == 64))
    return MOE_ERR_ARG;
  {
    const int want = o ? o->coalesce_rows : 0;
    const int c = want == 0 ? kPlanCoalesce : want;
    p->co = (c > p->bm && !p->w8) ? c : 0;
  }
  p->co1 = p->co2 = p->co;
  // 256-row token-major tiles: the Down GEMM may instead take the experts'
  // rows in tiles of up to 128 (a work list over the same index) with the
  // 128-row swap-AB tile and its two accumulator sets, whose epilogue
  // overlaps the next unit's MMAs.  The planner does so from 256 rows per
  // active expert (Qwen3-shaped T=4096: 404 -> 394 us; Mixtral-shaped
  // T=2048, 512 rows: 1144 -> 1104 us); at 128 rows the 256 x 256 tile is
  // faster (Qwen3-shaped T=2048: 296 against 302 us; Mixtral-shaped T=512:
  // 509 against 568 us).
  if (o && !(o->down_tile_rows == 0 || o->down_tile_rows == -1 || o->down_tile_rows == 128))
    return MOE_ERR_ARG;
  if (p->bm == 256) {
    const int want = o ? o->down_tile_rows : 0;
    const bool split =
        want == 128 || (want == 0 && mean_rows(p->T, p->k, p->E) >= kPlanDownSplitMinRows);
    if (split) p->co = p->co2 = 128;
  }
  p->bn1 = p->co1 ? p->co1 : p->bm;
  p->bn2 = p->co2 ? p->co2 : p->bm;
  const int64_t tc = tiles_cap_of(p->T, p->k, p->E, p->bm);
  if (tc * p->bm >= (int64_t(1) << 31) / 2) return MOE_ERR_SHAPE;
  p->tiles_cap = static_cast<int>(tc);
  p->rows_cap = static_cast<int>(tc * p->bm);
  // a work list of tiles smaller than the index's holds up to this many
  p->work_cap = p->co ? static_cast<int>(tiles_cap_of(p->T, p->k, p->E, std::min(p->co, p->bm)))
                      : 0;
  const int kstage = (p->fp8 || p->w8) ? 128 : 64;   // K elements per pipeline stage
  p->kt1 = s->H / kstage;
  p->mt1 = s->I / 64;
  p->kt2 = s->I / kstage;
  p->mt2 = s->H / 128;
  // Large token tiles (prefill) are L2-bandwidth bound with one 128-row
  // weight tile per unit: pair two weight tiles per unit there.
  p->me1 = (!p->fp8 && !p->w8 && p->bm >= 128 && p->mt1 % 2 == 0 &&
             !(o && o->single_weight_tile)) ? 2 : 1;
  p->me2 = (!p->fp8 && !p->w8 && p->bm >= 128 && p->mt2 % 2 == 0 &&
             !(o && o->single_weight_tile)) ? 2 : 1;
  const int est = est_tiles(p->T, p->k, p->E, p->bm, p->tiles_cap);
  const double unit_cost = (p->fp8 || p->w8) ? 0.0 : kPlanUnitCost;
  if (!p->fp8 && !(o && o->separate_act)) {
    // bf16 activations: an unsplit Gate-Up applies SiLU-and-mul in its
    // epilogue; measured faster than any split (whose partials then need the
    // separate activation stage) at every decode size tried
    p->s1 = 1;
    p->kts1 = p->kt1;
  } else {
    choose_split(p->mt1 / p->me1, p->kt1, est, p->bm, &p->s1, &p->kts1, kMaxSplits, true,
                 unit_cost);
  }
  choose_split(p->mt2 / p->me2, p->kt2, est, p->bm, &p->s2, &p->kts2, kMaxSplits, true,
               unit_cost);
  if (o && o->split_gateup > 0) {
    p->kts1 = (p->kt1 + o->split_gateup - 1) / o->split_gateup;
    p->s1 = (p->kt1 + p->kts1 - 1) / p->kts1;
  }
  if (o && o->split_down > 0) {
    p->kts2 = (p->kt2 + o->split_down - 1) / o->split_down;
    p->s2 = (p->kt2 + p->kts2 - 1) / p->kts2;
  }
  p->fused_act = !p->fp8 && p->s1 == 1 && !(o && o->separate_act);
  // FP8, unsplit 128-row (token-major) Gate-Up: each epilogue thread holds
  // its token's gate and up sums of the same channels, so it stores
  // SiLU(gate)*up, I fp32 values a row instead of 2I, and the activation
  // stage only quantises (DeepSeek-shaped T=4096: 268 MB less written and
  // read back).  The quantisation needs all 128 channels of a group, which
  // span two units, so it stays a separate stage.
  p->g_act = p->fp8 && p->bn1 == 128 && p->s1 == 1 && !(o && o->separate_act);
  // An unsplit Down GEMM stores its rows in bf16 (the combine's input), half
  // the bytes of fp32 partials written and read back (prefill: 268 MB of
  // fp32 rows at the Qwen3-shaped T=4096)
  p->y16 = p->s2 == 1 && !p->w8;
  if (o && (o->unit_order < 0 || o->unit_order > 2)) return MOE_ERR_ARG;
  if (o && o->pipeline_wait_ns < 0) return MOE_ERR_ARG;
  if (o && o->unit_order) {
    p->ord1 = p->ord2 = o->unit_order;
  } else {
    p->ord1 = unit_order(p->T, p->k, p->E, p->bm, p->mt1 / p->me1 * p->s1);
    p->ord2 = unit_order(p->T, p->k, p->E, p->bm, p->mt2 / p->me2 * p->s2);
  }
  // Every GEMM CTA rebuilds the index from the top-k ids in shared memory
  // (no index kernel) on request, or by default for bf16 layers with at most
  // 16 experts, where the per-CTA build is short (tiny 8-expert layer at
  // T=8: 23.1 -> 21.0 us; with 128 experts it measured slower), when it fits
  // next to the pipeline.
  {
    if (o && (o->smem_index < -1 || o->smem_index > 1)) return MOE_ERR_ARG;
    const int want = o ? o->smem_index : 0;
    const bool auto_on = want == 0 && !routed && !p->fp8 && !p->w8 && p->E <= 16;
    const int tk = p->T * p->k;
    bool fits = tk <= kSmemIndexMaxAssignments && (want == 1 || auto_on) && !p->w8;
    for (int bsrc : {static_cast<int>(kGather), static_cast<int>(kDirect)}) {
      const int bn = bsrc == kGather ? p->bn1 : p->bn2;
      const int lcap = (bsrc == kGather ? p->co1 : p->co2) ? p->work_cap : p->tiles_cap;
      const size_t need = gemm_smem_bytes(p->fp8, bn, bsrc) +
                          gemm_index_smem_bytes(gemm_warps(p->fp8, bn, bsrc), p->E, tk, p->rows_cap,
                                                lcap);
      if (need > kMaxGemmSmem) fits = false;
    }
    p->smem_index = fits;
  }
  // many assignments: build the index over chunks, one CTA each
  p->split_index = !p->smem_index && static_cast<int64_t>(p->T) * p->k > kSplitIndexMinAssignments;
  // in-path router: its GEMM, top-k, x-quant and index in one cooperative
  // launch on request (fuse_routing 1).  The planner (0) and -1 keep the
  // separate PDL-chained kernels: measured faster on the Zipf-routed layer
  // (T=4: 54.7 against 62.0 us; T=64: 97.1 against 104.8 us), because PDL
  // hides each separate kernel's launch behind its predecessor while the
  // single grid pays its memset, its two grid barriers and a longer tail.
  if (o && (o->fuse_routing < -1 || o->fuse_routing > 1)) return MOE_ERR_ARG;
  p->route_fused = p->routed && p->map.plain() && o && o->fuse_routing == 1;
  // FP8 with a one-CTA index kernel: the x-quant runs on the same launch's
  // other blocks (one launch fewer in front of the Gate-Up), with per-token
  // scales that the Gate-Up looks up through the index.
  p->align_quant = p->fp8 && !p->route_fused && !p->split_index && !p->smem_index &&
                   !(o && o->separate_quant);
  p->xs_by_token = p->fp8 && (p->smem_index || p->route_fused || p->align_quant);
  p->rp_owners_cap = std::min((p->T + 5) / 6, kPlanCtas);
  // workspace layout
  const size_t tk = static_cast<size_t>(p->T) * p->k;
  const size_t rc = p->rows_cap;
  const size_t sizes[kNumOff] = {
      4u * p->E,
      4u * (p->E + 1),
      4 * rc,
      4u * p->tiles_cap,
      16u * p->tiles_cap,
      4 * tk,
      4,
      p->split_index ? 4 * align_split_scratch_words(p->T, p->k, p->E) : 0,
      p->fp8 ? static_cast<size_t>(s->T) * s->H : 0,
      p->fp8 ? 4 * static_cast<size_t>(s->T) * (s->H / 128) : 0,
      p->fp8 && !p->xs_by_token ? 4 * rc * (s->H / 128) : 0,
      p->fused_act ? 0 : p->g_act ? 4 * rc * s->I : 4 * static_cast<size_t>(p->s1) * rc * 2 * s->I,
      rc * s->I * (p->fp8 ? 1 : 2),
      p->fp8 ? 4 * rc * (s->I / 128) : 0,
      (p->y16 ? 2 : 4 * static_cast<size_t>(p->s2)) * rc * s->H,
      p->routed ? p->rp_bytes : 0,
      p->route_fused ? 8u : 0u,
      p->route_fused ? 4 * static_cast<size_t>(p->rp_owners_cap) * p->E : 0,
      16u * p->work_cap,
      p->co ? 4u : 0u,
  };
  size_t cur = 0;
  for (int i = 0; i < kNumOff; ++i) {
    p->off[i] = cur;
    cur = align_up(cur + sizes[i], 256);
  }
  p->total = cur;
  return MOE_OK;
}

void fill_layout(const Plan& p, moe_workspace_layout* L) {
  std::memset(L, 0, sizeof(*L));
  L->block_m = p.bm;
  L->tiles_cap = p.tiles_cap;
  L->rows_cap = p.rows_cap;
  L->split_gateup = p.s1;
  L->split_down = p.s2;
  L->grid_gateup = kPlanCtas;
  L->grid_down = kPlanCtas;
  L->fused_act = p.fused_act;
  L->g_act_rows = p.g_act;
  L->xs_by_token = p.xs_by_token;
  L->smem_index = p.smem_index;
  L->weight_tiles_per_unit = p.me1 | (p.me2 << 8);
  L->off_counts = p.off[kOffCounts];
  L->off_offsets = p.off[kOffOffsets];
  L->off_sorted_ids = p.off[kOffSorted];
  L->off_tile_expert = p.off[kOffTileExpert];
  L->off_tiles = p.off[kOffTiles];
  L->off_inv_pos = p.off[kOffInvPos];
  L->off_num_tiles = p.off[kOffNumTiles];
  L->route_fused = p.route_fused;
  L->unit_order = p.ord1 | (p.ord2 << 8);
  L->off_router = p.off[kOffRouterP];
  L->off_route_counter = p.off[kOffCounter];
  L->off_route_hist = p.off[kOffRouteHist];
  L->off_index_scratch = p.off[kOffIdxScratch];
  L->off_xq = p.off[kOffXq];
  L->off_xs = p.off[kOffXs];
  L->off_xs_rows = p.off[kOffXsRows];
  L->off_g = p.off[kOffG];
  L->off_a = p.off[kOffA];
  L->off_as = p.off[kOffAs];
  L->off_y = p.off[kOffY];
  L->total_bytes = p.total;
  L->coalesce_rows = p.co1;
  L->down_tile_rows = p.co2;
  L->work_cap = p.work_cap;
  L->y_bf16 = p.y16;
  L->off_work_tiles = p.off[kOffWorkTiles];
  L->off_num_work_tiles = p.off[kOffNumWorkTiles];
}

// ---------------------------------------------------------------- devices
int device_sms() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return kPlanCtas;
  if (!sms[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = kPlanCtas;
    sms[dev] = v;
  }
  return sms[dev];
}

// ---------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D K-major map [rows][cols] of `esize`-byte elements, box {128 bytes of
// K, box_rows}, 128-byte swizzle.
bool make_map_2d(CUtensorMap* m, const void* base, int esize, uint64_t cols, uint64_t rows,
                 uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * esize};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D K-major map [experts][rows][cols], box {128 bytes of K, box_rows, 1}.
bool make_map_3d(CUtensorMap* m, const void* base, int esize, uint64_t cols, uint64_t rows,
                 uint64_t experts, uint32_t box_rows, bool raw64 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cols, rows, experts};
  const cuuint64_t strides[2] = {cols * esize, cols * rows * esize};
  // raw64: 64-byte rows with the 64-byte swizzle (e4m3 weight stages of the
  // w8a16 GEMM, read a row per converter thread)
  const cuuint32_t box[3] = {static_cast<cuuint32_t>((raw64 ? 64 : 128) / esize), box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            raw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Gate-Up weights W13 [experts][2I][cols] as the 5-D view
// (cols, 16 rows, gate|up, I/16 row groups, experts): one box of
// {128 bytes, 16, 2, 4, 1} brings 64 gate rows and their 64 up rows,
// interleaved 16 by 16, in a single copy.
bool make_map_gateup(CUtensorMap* m, const void* base, int esize, uint64_t cols, uint64_t I,
                     uint64_t experts, bool raw64 = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t row = cols * esize;
  const cuuint64_t dims[5] = {cols, 16, 2, I / 16, experts};
  const cuuint64_t strides[4] = {row, I * row, 16 * row, 2 * I * row};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>((raw64 ? 64 : 128) / esize), 16, 2, 4, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            raw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Stage events.  Under stream capture a plain record only orders work inside
// the graph; the external flag makes it a real timestamp node.
void record(const moe_forward_opts* o, int i, cudaStream_t st) {
  if (!o || !o->stage_events[i]) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  cudaEventRecordWithFlags(static_cast<cudaEvent_t>(o->stage_events[i]), st,
                           cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                               : cudaEventRecordDefault);
}

cudaError_t launch_gemm(int fp8, int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                        const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                        int me = 1) {
  return fp8 ? launch_gemm_fp8(bn, bsrc, grid, st, pdl, a, b, p)
             : launch_gemm_bf16(bn, bsrc, grid, st, pdl, a, b, p, me);
}

// The router GEMM over [hi; lo] (2E rows, K = H) for T tokens.  Few tokens
// leave most SMs idle at the split counts one top-k warp can sum at once, so
// with few token tiles the split may go up to 32, which the top-k kernel
// then reduces with a block of eight warps per token (router table shape,
// K = 4096, N = 192 experts: 12 CTAs streaming 256 KB each at one token);
// the fused routing front sums in one warp per token and keeps at most four.
bool router_plan(int T, int H, int E, RouterPlan* r, bool fused_front) {
  if (T < 1 || H < 128 || H % 128 || E < 64 || E > 512 || E % 64) return false;
  r->bn = T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128;
  r->rows_cap = (T + r->bn - 1) / r->bn * r->bn;
  r->kt = H / 64;
  r->mt = 2 * E / 128;
  const int tiles = r->rows_cap / r->bn;
  const bool wide = !fused_front && T <= kRouterWideMaxT;
  choose_split(r->mt, r->kt, tiles, r->bn, &r->splits, &r->kts,
               wide ? kRouterMaxSplitsWide : kRouterMaxSplitsHost, false);
  r->bytes = 4ull * r->splits * r->rows_cap * 2 * E;
  return true;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_index_tiles_cap(int32_t T, int32_t k, int32_t E, int32_t block_m) {
  if (T < 1 || k < 1 || E < 1 || block_m < 1) return 0;
  return static_cast<size_t>(tiles_cap_of(T, k, E, block_m));
}

moe_status moe_plan(const moe_shape* shape, const moe_forward_opts* opts,
                    moe_workspace_layout* layout) {
  if (!layout) return MOE_ERR_ARG;
  Plan p;
  const moe_status st = make_plan(shape, opts, &p);
  if (st != MOE_OK) return st;
  fill_layout(p, layout);
  return MOE_OK;
}

size_t moe_workspace_bytes(const moe_shape* shape, const moe_forward_opts* opts) {
  Plan p;
  return make_plan(shape, opts, &p) == MOE_OK ? p.total : 0;
}

moe_status moe_align(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E, int32_t block_m,
                     const moe_index* idx, int32_t* dev_status, void* stream) {
  if (!topk_ids || !idx || !idx->counts || !idx->offsets || !idx->sorted_ids ||
      !idx->tile_expert || !idx->tiles || !idx->inv_pos || !idx->num_tiles)
    return MOE_ERR_ARG;
  if (T < 1 || k < 1 || E < 1 || E > 512 || k > E || !valid_bm(block_m, 0))
    return MOE_ERR_SHAPE;
  if (static_cast<int64_t>(T) * k >= (int64_t(1) << 31) / 2) return MOE_ERR_SHAPE;
  if (!aligned(idx->tiles, 16)) return MOE_ERR_ALIGN;
  IndexPtrs ip{idx->counts, idx->offsets, idx->sorted_ids, idx->tile_expert,
               idx->tiles,  idx->inv_pos,  idx->num_tiles};
  const int tc = static_cast<int>(tiles_cap_of(T, k, E, block_m));
  IdMap plain{k, k, E, 0, 0};
  return cuda_status(launch_align(topk_ids, T, k, E, block_m, tc, ip, dev_status,
                                  static_cast<cudaStream_t>(stream), false, plain, true));
}

moe_status moe_align_ex(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E, int32_t block_m,
                        const moe_align_opts* opts, const moe_index* idx, int32_t* dev_status,
                        void* stream) {
  if (!opts) return moe_align(topk_ids, T, k, E, block_m, idx, dev_status, stream);
  if (!topk_ids || !idx || !idx->counts || !idx->offsets || !idx->sorted_ids ||
      !idx->tile_expert || !idx->tiles || !idx->inv_pos || !idx->num_tiles)
    return MOE_ERR_ARG;
  if (T < 1 || k < 1 || E < 1 || E > 512 || k > E || !valid_bm(block_m, 0))
    return MOE_ERR_SHAPE;
  IdMap m;
  moe_status st = make_idmap(k, E, opts->num_shared_experts, opts->ep_first_expert,
                             opts->ep_num_experts, &m);
  if (st != MOE_OK) return st;
  const int64_t tk = static_cast<int64_t>(T) * m.kk;
  if (!m.plain() && tk > 32768) return MOE_ERR_SHAPE;   // mapped ids are staged on chip
  if (tk >= (int64_t(1) << 31) / 2) return MOE_ERR_SHAPE;
  if (!aligned(idx->tiles, 16)) return MOE_ERR_ALIGN;
  IndexPtrs ip{idx->counts, idx->offsets, idx->sorted_ids, idx->tile_expert,
               idx->tiles,  idx->inv_pos,  idx->num_tiles};
  const int Ei = E + opts->num_shared_experts;
  const int tc = static_cast<int>(tiles_cap_of(T, m.kk, Ei, block_m));
  return cuda_status(launch_align(topk_ids, T, m.kk, Ei, block_m, tc, ip, dev_status,
                                  static_cast<cudaStream_t>(stream), false, m, true));
}

}  // extern "C"

namespace moe {
namespace {

// The in-path router of a moe_forward_routed call.
struct RouteCall {
  const void* hi_lo;
  int score_fn;
  float scale;
  float* scores;
};

moe_status forward_impl(const Plan& p, const void* x, const void* w13, const void* w2,
                        const int32_t* topk_ids, const float* topk_w, const moe_scales* scales,
                        void* out, void* workspace, size_t ws_bytes, int32_t* dev_status,
                        void* stream, const moe_forward_opts* opts, const RouteCall* rc) {
  if (!x || !w13 || !w2 || !topk_ids || !topk_w || !out || !workspace) return MOE_ERR_ARG;
  if ((p.fp8 || p.w8) && (!scales || !scales->w13_scale || !scales->w2_scale)) return MOE_ERR_ARG;
  if (!aligned(x, 16) || !aligned(w13, 16) || !aligned(w2, 16) || !aligned(out, 16) ||
      !aligned(topk_ids, 4) || !aligned(topk_w, 4) || !aligned(workspace, 256))
    return MOE_ERR_ALIGN;
  if ((p.fp8 || p.w8) && (!aligned(scales->w13_scale, 4) || !aligned(scales->w2_scale, 4)))
    return MOE_ERR_ALIGN;
  if (ws_bytes < p.total) return MOE_ERR_WORKSPACE;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool pdl = !(opts && opts->disable_pdl);
  const uint64_t wait_ns =
      (opts && opts->pipeline_wait_ns > 0) ? static_cast<uint64_t>(opts->pipeline_wait_ns) : 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto at = [&](int i) { return ws + p.off[i]; };
  IndexPtrs ip{reinterpret_cast<int32_t*>(at(kOffCounts)),     reinterpret_cast<int32_t*>(at(kOffOffsets)),
               reinterpret_cast<int32_t*>(at(kOffSorted)),     reinterpret_cast<int32_t*>(at(kOffTileExpert)),
               reinterpret_cast<int32_t*>(at(kOffTiles)),      reinterpret_cast<int32_t*>(at(kOffInvPos)),
               reinterpret_cast<int32_t*>(at(kOffNumTiles))};
  if (p.co) {
    ip.work_tiles = reinterpret_cast<int32_t*>(at(kOffWorkTiles));
    ip.num_work_tiles = reinterpret_cast<int32_t*>(at(kOffNumWorkTiles));
    ip.coalesce = p.co;
    ip.work_cap = p.work_cap;
  }
  uint8_t* xq = at(kOffXq);
  float* xs = reinterpret_cast<float*>(at(kOffXs));
  float* xs_rows = reinterpret_cast<float*>(at(kOffXsRows));
  float* G = reinterpret_cast<float*>(at(kOffG));
  void* A = at(kOffA);
  float* As = reinterpret_cast<float*>(at(kOffAs));
  float* Y = reinterpret_cast<float*>(at(kOffY));
  const int esize = p.fp8 ? 1 : 2;              // activation bytes
  const int wsize = (p.fp8 || p.w8) ? 1 : 2;    // weight bytes
  const int tk = p.T * p.k;

  CUtensorMap tmW13, tmX, tmW2, tmA;
  if (!make_map_gateup(&tmW13, w13, wsize, p.H, p.I, p.E, p.w8) ||
      !make_map_2d(&tmX, p.fp8 ? static_cast<const void*>(xq) : x, esize, p.H, p.T, 1) ||
      !make_map_3d(&tmW2, w2, wsize, p.I, p.H, p.E, 128, p.w8) ||
      !make_map_2d(&tmA, A, esize, p.I, p.rows_cap, p.co2 ? std::min(p.bm, p.bn2) : p.bm))
    return MOE_ERR_CUDA;

  const int sms = device_sms();
  const int grid_cap = opts && opts->grid_ctas > 0 ? opts->grid_ctas : sms;
  cudaError_t e;

  // The first launch of the call waits for all earlier work on the stream
  // (no PDL attribute); later launches overlap their predecessor's tail.
  bool first = true;
  auto chain = [&]() {
    const bool r = first ? false : pdl;
    first = false;
    return r;
  };

  if (rc) {
    // router GEMM over [hi; lo] (dense token rows)
    record(opts, 7, s);
    CUtensorMap tmR, tmXr;
    if (!make_map_3d(&tmR, rc->hi_lo, 2, p.H, 2ull * p.map.E, 1, 128) ||
        !make_map_2d(&tmXr, x, 2, p.H, p.T, p.rp_bn))
      return MOE_ERR_CUDA;
    GemmParams gr = {};
    gr.M = 2 * p.map.E;
    gr.K = p.H;
    gr.m_tiles = p.rp_mt;
    gr.splits = p.rp_splits;
    gr.kt_per_split = p.rp_kts;
    gr.kt_total = p.rp_kt;
    gr.dense_rows = p.T;
    gr.out = reinterpret_cast<float*>(at(kOffRouterP));
    gr.rows_cap = p.rp_rows_cap;
    gr.dev_status = dev_status;
    gr.clear_status = 1;   // the call's first kernel
    gr.pipe_wait_ns = wait_ns;
    const int units_r = p.rp_mt * p.rp_splits * (p.rp_rows_cap / p.rp_bn);
    if (p.route_fused) {
      // one cooperative grid: the router GEMM, then the top-k / x-quant /
      // index phases on owner CTAs of tpc tokens each
      // a token per warp of an owner (six warps), more where the owners would
      // outnumber the SMs; the grid also covers the x-quant at eight
      // 128-channel groups per warp
      const int tpc = std::max(6, (p.T + std::min(sms, p.rp_owners_cap) - 1) /
                                      std::min(sms, p.rp_owners_cap));
      RouteFrontParams q = {};
      q.P = gr.out;
      q.splits = p.rp_splits;
      q.rows_cap_r = p.rp_rows_cap;
      q.T = p.T;
      q.E = p.map.E;
      q.k = p.k;
      q.score_fn = rc->score_fn;
      q.scale = rc->scale;
      q.scores = rc->scores;
      q.ids = const_cast<int32_t*>(topk_ids);
      q.w = const_cast<float*>(topk_w);
      q.x = x;
      q.H = p.H;
      q.xq = p.fp8 ? xq : nullptr;
      q.xs = xs;
      q.Ei = p.E;
      q.bm = p.bm;
      q.tiles_cap = p.tiles_cap;
      q.idx = ip;
      q.dev_status = dev_status;
      q.tpc = tpc;
      q.owners = (p.T + tpc - 1) / tpc;
      q.hist = reinterpret_cast<int32_t*>(at(kOffRouteHist));
      q.bar = reinterpret_cast<unsigned int*>(at(kOffCounter));
      if (cudaMemsetAsync(q.bar, 0, 8, s) != cudaSuccess) return MOE_ERR_CUDA;
      first = false;   // the memset orders the grid after earlier work on the stream
      const int quant_ctas = p.fp8 ? (p.T * (p.H / 128) + 47) / 48 : 0;
      const int grid = std::min(sms, std::max(units_r + quant_ctas, q.owners));
      q.gemm_ctas = std::min(units_r, grid);
      e = launch_route_front(p.rp_bn, grid, s, tmR, tmXr, gr, q);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      record(opts, 0, s);
    } else {
      e = launch_gemm_bf16(p.rp_bn, kDense, std::min(sms, units_r), s, chain(), tmR, tmXr, gr);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      record(opts, 0, s);
      e = launch_router_topk(reinterpret_cast<const float*>(at(kOffRouterP)), p.rp_splits,
                             p.rp_rows_cap, p.T, p.map.E, p.k, rc->score_fn, rc->scale,
                             rc->scores, const_cast<int32_t*>(topk_ids),
                             const_cast<float*>(topk_w), s, chain());
      if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
  } else {
    record(opts, 0, s);
  }
  if (p.route_fused) {
    // routing index and x-quant done by the fused routing kernel
  } else if (p.split_index) {
    e = launch_align_split(topk_ids, p.T, p.k, p.E, p.bm, p.tiles_cap, ip,
                           reinterpret_cast<int32_t*>(at(kOffIdxScratch)), dev_status, s, chain(),
                           p.map, rc == nullptr);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else if (p.align_quant) {
    e = launch_align_quant(topk_ids, p.T, p.k, p.E, p.bm, p.tiles_cap, ip, dev_status, s,
                           chain(), p.map, rc == nullptr, x, p.H, xq, xs);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else if (!p.smem_index) {
    e = launch_align(topk_ids, p.T, p.k, p.E, p.bm, p.tiles_cap, ip, dev_status, s, chain(),
                     p.map, rc == nullptr);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }

  record(opts, 1, s);
  if (p.fp8 && !p.route_fused && !p.align_quant) {
    // with the shared-memory index the scales stay per token (the Gate-Up
    // epilogue looks tokens up in its own index)
    e = launch_quant_x(x, p.T, p.H, p.k, p.smem_index ? nullptr : ip.inv_pos, xq, xs,
                       p.smem_index ? nullptr : xs_rows, p.rows_cap, s, chain());
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }

  record(opts, 2, s);
  GemmParams g1 = {};
  g1.M = 2 * p.I;
  g1.K = p.H;
  g1.I = p.I;
  g1.m_tiles = p.mt1 / p.me1;
  g1.splits = p.s1;
  g1.kt_per_split = p.kts1;
  g1.kt_total = p.kt1;
  g1.tile_major = p.ord1 == 2;
  g1.tiles = p.co1 ? ip.work_tiles : ip.tiles;
  g1.num_tiles = p.co1 ? ip.num_work_tiles : ip.num_tiles;
  g1.coalesce = p.co1;
  g1.index_bm = p.bm;
  g1.sorted_ids = ip.sorted_ids;
  g1.b_rows = p.fp8 ? static_cast<const void*>(xq) : x;
  g1.b_row_bytes = p.H * esize;
  g1.topk = p.k;
  g1.sentinel = tk;
  g1.w_scale = (p.fp8 || p.w8) ? scales->w13_scale : nullptr;
  // per-token scales where no index-ordered copy was written
  g1.b_scale = p.fp8 ? (p.xs_by_token ? xs : xs_rows) : nullptr;
  g1.scale_by_token = p.xs_by_token;
  g1.smem_index = p.smem_index;
  g1.topk_ids = topk_ids;
  g1.T = p.T;
  g1.E = p.E;
  g1.idmap = p.map;
  g1.tiles_cap = p.tiles_cap;
  g1.list_cap = p.co1 ? p.work_cap : p.tiles_cap;
  g1.write_index = p.smem_index;
  g1.clear_status = p.smem_index && rc == nullptr;   // the Gate-Up is the call's first kernel
  g1.index_out = {ip.counts, ip.offsets, ip.sorted_ids, ip.tile_expert, ip.tiles, ip.inv_pos,
                  ip.num_tiles};
  g1.out = G;
  g1.act_out = p.fused_act ? A : nullptr;
  g1.g_act = p.g_act;
  g1.rows_cap = p.rows_cap;
  g1.dev_status = dev_status;
  g1.pipe_wait_ns = wait_ns;
  const int units1 = g1.m_tiles * p.s1 * g1.list_cap;
  e = p.w8 ? launch_gemm_w8(p.bm, kGather, std::min(grid_cap, units1), s, chain(), tmW13, tmX, g1)
           : launch_gemm(p.fp8, p.bn1, kGather, std::min(grid_cap, units1), s, chain(), tmW13,
                         tmX, g1, p.me1);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  record(opts, 3, s);
  if (!p.fused_act) {
    e = launch_act(p.fp8, G, p.g_act ? 0 : p.s1, p.rows_cap, p.I, ip.sorted_ids, tk, A, As, s,
                   pdl);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }

  record(opts, 4, s);
  GemmParams g2 = {};
  g2.M = p.H;
  g2.K = p.I;
  g2.I = 0;
  g2.m_tiles = p.mt2 / p.me2;
  g2.splits = p.s2;
  g2.kt_per_split = p.kts2;
  g2.kt_total = p.kt2;
  g2.tile_major = p.ord2 == 2;
  g2.tiles = p.co2 ? ip.work_tiles : ip.tiles;
  g2.num_tiles = p.co2 ? ip.num_work_tiles : ip.num_tiles;
  g2.coalesce = p.co2;
  g2.index_bm = p.bm;
  g2.sorted_ids = ip.sorted_ids;
  g2.topk = p.k;
  g2.sentinel = tk;
  g2.w_scale = (p.fp8 || p.w8) ? scales->w2_scale : nullptr;
  g2.b_scale = p.fp8 ? As : nullptr;
  g2.smem_index = p.smem_index;
  g2.topk_ids = topk_ids;
  g2.T = p.T;
  g2.E = p.E;
  g2.idmap = p.map;
  g2.tiles_cap = p.tiles_cap;
  g2.list_cap = p.co2 ? p.work_cap : p.tiles_cap;
  g2.early_weights = 1;   // the index is complete before this grid launches
  g2.out = Y;
  g2.out_bf16 = p.y16;
  g2.rows_cap = p.rows_cap;
  g2.dev_status = dev_status;
  g2.pipe_wait_ns = wait_ns;
  const int units2 = g2.m_tiles * p.s2 * g2.list_cap;
  e = p.w8 ? launch_gemm_w8(p.bm, kDirect, std::min(grid_cap, units2), s, pdl, tmW2, tmA, g2)
           : launch_gemm(p.fp8, p.bn2, kDirect, std::min(grid_cap, units2), s, pdl, tmW2, tmA, g2,
                         p.me2);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  record(opts, 5, s);
  e = launch_combine(Y, p.y16, p.s2, p.rows_cap, p.H, ip.inv_pos, topk_w, p.T, p.k, p.map.k, p.w_shared,
                     out, p.out_bf16, s,
                     pdl);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  record(opts, 6, s);
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_forward_ex(const moe_shape* shape, const void* x, const void* w13, const void* w2,
                          const int32_t* topk_ids, const float* topk_w, const moe_scales* scales,
                          void* out, void* workspace, size_t ws_bytes, int32_t* dev_status,
                          void* stream, const moe_forward_opts* opts) {
  Plan p;
  moe_status st = make_plan(shape, opts, &p);
  if (st != MOE_OK) return st;
  return forward_impl(p, x, w13, w2, topk_ids, topk_w, scales, out, workspace, ws_bytes,
                      dev_status, stream, opts, nullptr);
}

moe_status moe_plan_routed(const moe_shape* shape, const moe_forward_opts* opts,
                           moe_workspace_layout* layout) {
  if (!layout) return MOE_ERR_ARG;
  Plan p;
  moe_status st = make_plan(shape, opts, &p, true);
  if (st != MOE_OK) return st;
  fill_layout(p, layout);
  return MOE_OK;
}

size_t moe_routed_workspace_bytes(const moe_shape* shape, const moe_forward_opts* opts) {
  Plan p;
  return make_plan(shape, opts, &p, true) == MOE_OK ? p.total : 0;
}

moe_status moe_forward_routed(const moe_shape* shape, const void* x, const void* hi_lo,
                              int32_t score_fn, float scale, const void* w13, const void* w2,
                              const moe_scales* scales, float* scores, int32_t* topk_ids,
                              float* topk_w, void* out, void* workspace, size_t ws_bytes,
                              int32_t* dev_status, void* stream, const moe_forward_opts* opts) {
  Plan p;
  moe_status st = make_plan(shape, opts, &p, true);
  if (st != MOE_OK) return st;
  if (!hi_lo || !scores) return MOE_ERR_ARG;
  if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_ARG;
  if (!aligned(hi_lo, 16) || !aligned(scores, 4)) return MOE_ERR_ALIGN;
  RouteCall rc{hi_lo, score_fn, scale, scores};
  return forward_impl(p, x, w13, w2, topk_ids, topk_w, scales, out, workspace, ws_bytes,
                      dev_status, stream, opts, &rc);
}

moe_status moe_forward(const moe_shape* shape, const void* x, const void* w13, const void* w2,
                       const int32_t* topk_ids, const float* topk_w, const moe_scales* scales,
                       void* out, void* workspace, size_t ws_bytes, int32_t* dev_status,
                       void* stream) {
  return moe_forward_ex(shape, x, w13, w2, topk_ids, topk_w, scales, out, workspace, ws_bytes,
                        dev_status, stream, nullptr);
}

moe_status moe_combine(const moe_shape* shape, int32_t splits, int32_t rows_cap, const float* y,
                       const int32_t* inv_pos, const float* topk_w, void* out, void* stream) {
  if (!shape || !y || !inv_pos || !topk_w || !out) return MOE_ERR_ARG;
  if (shape->out_dtype != MOE_OUT_F32 && shape->out_dtype != MOE_OUT_BF16) return MOE_ERR_DTYPE;
  if (shape->T < 1 || shape->k < 1 || shape->H < 4 || shape->H % 4 || splits < 1 || rows_cap < 1)
    return MOE_ERR_SHAPE;
  if (!aligned(y, 16) || !aligned(out, 16)) return MOE_ERR_ALIGN;
  return cuda_status(launch_combine(y, 0, splits, rows_cap, shape->H, inv_pos, topk_w, shape->T,
                                    shape->k, shape->k, 1.0f, out,
                                    shape->out_dtype == MOE_OUT_BF16,
                                    static_cast<cudaStream_t>(stream), false));
}

moe_status moe_router_prepare(const float* wr, int32_t E, int32_t H, void* hi_lo, void* stream) {
  if (!wr || !hi_lo) return MOE_ERR_ARG;
  if (E < 1 || H < 1) return MOE_ERR_SHAPE;
  if (!aligned(hi_lo, 2) || !aligned(wr, 4)) return MOE_ERR_ALIGN;
  return cuda_status(launch_router_prepare(wr, E, H, hi_lo, static_cast<cudaStream_t>(stream)));
}

size_t moe_router_workspace_bytes(int32_t T, int32_t H, int32_t E) {
  RouterPlan r;
  return router_plan(T, H, E, &r) ? r.bytes : 0;
}

moe_status moe_router_topk(const void* x, const void* hi_lo, int32_t T, int32_t H, int32_t E,
                           int32_t k, int32_t score_fn, float scale, float* scores,
                           int32_t* topk_ids, float* topk_w, void* workspace, size_t ws_bytes,
                           void* stream) {
  if (!x || !hi_lo || !scores || !topk_ids || !topk_w || !workspace) return MOE_ERR_ARG;
  if (score_fn != MOE_SCORE_SOFTMAX && score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_ARG;
  RouterPlan r;
  if (!router_plan(T, H, E, &r) || k < 1 || k > E || k > 32) return MOE_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(hi_lo, 16) || !aligned(workspace, 16)) return MOE_ERR_ALIGN;
  if (ws_bytes < r.bytes) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUtensorMap tmW, tmX;
  if (!make_map_3d(&tmW, hi_lo, 2, H, 2ull * E, 1, 128) ||
      !make_map_2d(&tmX, x, 2, H, T, r.bn))
    return MOE_ERR_CUDA;
  GemmParams g = {};
  g.M = 2 * E;
  g.K = H;
  g.m_tiles = r.mt;
  g.splits = r.splits;
  g.kt_per_split = r.kts;
  g.kt_total = r.kt;
  g.dense_rows = T;
  g.out = static_cast<float*>(workspace);
  g.rows_cap = r.rows_cap;
  const int units = r.mt * r.splits * (r.rows_cap / r.bn);
  cudaError_t e = launch_gemm_bf16(r.bn, kDense, std::min(device_sms(), units), s, false, tmW,
                                   tmX, g);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return cuda_status(launch_router_topk(static_cast<const float*>(workspace), r.splits, r.rows_cap,
                                        T, E, k, score_fn, scale, scores, topk_ids, topk_w, s,
                                        true));
}

const char* moe_status_str(int32_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument (null pointer or bad enum)";
    case MOE_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case MOE_ERR_DTYPE: return "unsupported mode or output dtype";
    case MOE_ERR_ALIGN: return "pointer not suitably aligned";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_EXPERT_ID: return "an expert id outside [0, E) was dropped";
    case MOE_ERR_TIMEOUT: return "a bounded on-chip wait gave up";
    case MOE_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

}  // extern "C"
