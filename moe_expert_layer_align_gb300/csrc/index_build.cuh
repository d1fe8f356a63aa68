// index_build.cuh — the routing and index build as block-level device code.
//
// HPC-Ops × SGLang, section "MoE", fused pipeline, "routing and index build":
// a shared-memory counting pass arranges token-expert assignments into
// contiguous per-expert intervals without global atomics and emits the tile
// task map the persistent expert GEMM consumes.
//
// One thread block builds the whole index.  Warp w of the block owns the
// contiguous slice [w*seg, (w+1)*seg) of the flat assignments a = t*k + j and
// walks it in rounds of 32 (one assignment per lane):
//   1. count: a ballot per key bit groups a round's lanes by expert and the
//      group's lowest lane adds the group size to cnt[w][e] (one writer per
//      address, no atomics);
//   2. scan: per expert an exclusive prefix of cnt[.][e] over the warps gives
//      each warp's base inside the expert; a warp scan of the counts rounded
//      up to block_m gives offsets[];
//   3. scatter: the same rounds again; an assignment's row is
//      offsets[e] + base[w][e] + (lanes of its group below it).
// Slices ascend in a, rounds run in order and ranks inside a round follow the
// lane, so each interval lists its assignments in ascending a: the result is
// unique and deterministic.  The caller chooses where rows and tiles go (the
// align kernel writes global memory; the GEMM's prologue, shared memory).
#pragma once
#include <cstdint>

#include <climits>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

// Index expert of assignment a under `m` (IdMap): a routed expert (0..E-1),
// a shared one (E..), -1 for an invalid id, or kRemoteId for a valid id of
// another rank's experts (dropped without a flag).
constexpr int kRemoteId = INT_MIN;
__device__ __forceinline__ int mapped_id(const int32_t* ids, int a, const IdMap& m) {
  if (m.plain()) return ids[a];
  const int t = a / m.kk, j = a - t * m.kk;
  if (j >= m.k) return m.E + (j - m.k);
  const int e = ids[static_cast<size_t>(t) * m.k + j];
  if (m.Eg == 0) return (e >= 0 && e < m.E) ? e : -1;
  if (e < 0 || e >= m.Eg) return -1;
  return (e >= m.e0 && e < m.e0 + m.E) ? e - m.e0 : kRemoteId;
}

__device__ __forceinline__ int lanemask_lt() {
  int m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Lanes of the warp whose key equals this lane's, from one ballot per key
// bit (ANDing each bit's agreement mask).  Keys are in [0, 2^bits); a lane
// with an invalid id passes key = 2^bits, so `bits + 1` bits are compared.
// (One vote per bit instead of __match_any_sync, whose cost grows with the
// number of distinct keys in the warp.)
__device__ __forceinline__ unsigned peer_mask(int key, int bits) {
  unsigned mask = 0xffffffffu;
  for (int b = 0; b <= bits; ++b) {
    const bool set = (key >> b) & 1;
    const unsigned v = __ballot_sync(0xffffffffu, set);
    mask &= set ? v : ~v;
  }
  return mask;
}

__device__ __forceinline__ int key_bits(int E) {
  int b = 0;
  while ((1 << b) < E) ++b;
  return b;
}

// Shared-memory scratch of one index build.
struct IndexScratch {
  int32_t* cnt;    // [nwarps][E]: per-warp counts, then per-warp bases
  int32_t* offs;   // [E + 1]: padded offsets
  int32_t* tot;    // [E]: per-expert counts
  int32_t* flag;   // [1]: an invalid id was seen
  int32_t* wsum;   // [2][33]: per-warp sums of the two offset scans, then their totals
  int32_t* coffs;  // [E + 1]: work-list offsets (coalesced tiles before each expert)
  int remote_ok;   // kRemoteId entries are another rank's: dropped, not flagged
  static __host__ __device__ constexpr size_t words(int nwarps, int E) {
    return static_cast<size_t>(nwarps) * E + (E + 1) + E + 1 + 66 + (E + 1);
  }
  __device__ void carve(int32_t* base, int nwarps, int E, int remote = 0) {
    remote_ok = remote;
    cnt = base;
    offs = cnt + nwarps * E;
    tot = offs + E + 1;
    flag = tot + E;
    wsum = flag + 1;
    coffs = wsum + 66;
  }
};

// Warps that take part in counting and scattering: one per 32 assignments,
// at most the block's.  A small batch then zeroes and scans a short count
// table instead of the whole block's (the segments, and with them the
// result, are the same function of tk and this count in both passes).
__device__ __forceinline__ int index_warps(int tk) {
  const int nwarps = blockDim.x >> 5;
  const int need = (tk + 31) / 32;
  return need < 1 ? 1 : (need < nwarps ? need : nwarps);
}

// Inclusive warp scan of v.
__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

// offs[0..E] = exclusive prefix of tot[] rounded up to multiples of bm (a
// power of two, as the host checks): one expert per thread, a shuffle scan
// per warp and one over the warps' sums, blockDim.x experts at a time.  (A
// single warp walking the experts with divisions took ~2-4 us for 128
// experts.)  With coalesce C > 0 (a power of two) the same pass also gives
// coffs[0..E], the exclusive prefix of ceil(tot / C): the work-list tiles of
// up to C rows before each expert (index_work_tile).  Ends with a block
// barrier.
__device__ __forceinline__ void index_scan_offsets(int E, int bm, const IndexScratch& sc,
                                                   int C = 0) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31, nw = nthreads >> 5;
  const int mask = bm - 1;
  const int cs = C > 0 ? __ffs(C) - 1 : 0;
  int carry = 0, ccarry = 0;   // padded rows (work tiles) of the experts before this round's
  for (int e0 = 0; e0 < E; e0 += nthreads) {
    const int e = e0 + tid;
    const int t = e < E ? sc.tot[e] : 0;
    const int v = (t + mask) & ~mask;
    const int cv = C > 0 ? (t + C - 1) >> cs : 0;
    const int incl = warp_incl_scan(v, lane);
    const int cincl = C > 0 ? warp_incl_scan(cv, lane) : 0;
    if (lane == 31) {
      sc.wsum[warp] = incl;
      sc.wsum[33 + warp] = cincl;
    }
    __syncthreads();
    if (warp == 0) {
      const int x = lane < nw ? sc.wsum[lane] : 0;
      const int xi = warp_incl_scan(x, lane);
      const int cx = lane < nw ? sc.wsum[33 + lane] : 0;
      const int cxi = C > 0 ? warp_incl_scan(cx, lane) : 0;
      if (lane < nw) {              // exclusive warp bases
        sc.wsum[lane] = xi - x;
        sc.wsum[33 + lane] = cxi - cx;
      }
      if (lane == 31) {             // this round's totals
        sc.wsum[32] = xi;
        sc.wsum[65] = cxi;
      }
    }
    __syncthreads();
    if (e < E) {
      sc.offs[e] = carry + sc.wsum[warp] + incl - v;
      if (C > 0) sc.coffs[e] = ccarry + sc.wsum[33 + warp] + cincl - cv;
    }
    carry += sc.wsum[32];
    ccarry += sc.wsum[65];
    __syncthreads();   // wsum is rewritten by the next round
  }
  if (tid == 0) {
    sc.offs[E] = carry;
    if (C > 0) sc.coffs[E] = ccarry;
  }
  __syncthreads();
}

// Steps 1-2: counts, per-warp bases and padded offsets (and with C > 0 the
// work-list offsets), all in `sc`.  `src` holds the T*k ids (shared or global
// memory).  Ends with a block barrier.
__device__ __forceinline__ void index_count_and_scan(const int32_t* src, int tk, int E, int bm,
                                                     const IndexScratch& sc, int C = 0) {
  const int tid = threadIdx.x, nthreads = blockDim.x, nwarps = index_warps(tk);
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < nwarps * E; i += nthreads) sc.cnt[i] = 0;
  if (tid == 0) *sc.flag = 0;
  __syncthreads();
  const int seg = (tk + nwarps - 1) / nwarps;
  const int beg = min(tk, warp * seg);
  const int end = min(tk, beg + seg);
  const int bits = key_bits(E);
  for (int base = beg; base < end; base += 32) {
    const int a = base + lane;
    const bool in = a < end;
    const int e = in ? src[a] : -1;
    const bool valid = in && e >= 0 && e < E;
    if (in && !valid && !(sc.remote_ok && e == kRemoteId)) *sc.flag = 1;
    const unsigned grp = peer_mask(valid ? e : (1 << bits), bits);
    if (valid && lane == __ffs(grp) - 1) sc.cnt[warp * E + e] += __popc(grp);
    __syncwarp();
  }
  __syncthreads();
  for (int e = tid; e < E; e += nthreads) {
    int run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const int c = sc.cnt[w * E + e];
      sc.cnt[w * E + e] = run;
      run += c;
    }
    sc.tot[e] = run;
  }
  __syncthreads();
  index_scan_offsets(E, bm, sc, C);
}

// Step 3: every valid assignment a goes to row(pos, a); an invalid one to
// invalid(a).  Uses and advances the per-warp bases in sc.cnt.  No barrier.
template <class RowFn, class InvalidFn>
__device__ __forceinline__ void index_scatter(const int32_t* src, int tk, int E,
                                              const IndexScratch& sc, RowFn row,
                                              InvalidFn invalid) {
  const int tid = threadIdx.x, nwarps = index_warps(tk);
  const int warp = tid >> 5, lane = tid & 31;
  const int seg = (tk + nwarps - 1) / nwarps;
  const int beg = min(tk, warp * seg);
  const int end = min(tk, beg + seg);
  const int bits = key_bits(E);
  for (int base = beg; base < end; base += 32) {
    const int a = base + lane;
    const bool in = a < end;
    const int e = in ? src[a] : -1;
    const bool valid = in && e >= 0 && e < E;
    const unsigned grp = peer_mask(valid ? e : (1 << bits), bits);
    if (valid)
      row(sc.offs[e] + sc.cnt[warp * E + e] + __popc(grp & lanemask_lt()), a);
    else if (in)
      invalid(a);
    __syncwarp();
    if (valid && lane == __ffs(grp) - 1) sc.cnt[warp * E + e] += __popc(grp);
    __syncwarp();
  }
}

// Padding rows of every expert interval (fewer than bm each), a warp per
// expert with its lanes on consecutive rows, then the tail [offs[E],
// rows_end).  (A thread per expert wrote its padding row by row: with
// 256-row tiles up to 255 stores each, 32 scattered rows per warp store —
// 13 us of the index scan kernel at the Qwen3-shaped T=4096.)
template <class PadFn>
__device__ __forceinline__ void index_pads(int E, int rows_end, const IndexScratch& sc, PadFn pad) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int lane = tid & 31, nwarps = nthreads >> 5;
  for (int e = tid >> 5; e < E; e += nwarps)
    for (int pos = sc.offs[e] + sc.tot[e] + lane; pos < sc.offs[e + 1]; pos += 32) pad(pos);
  for (int pos = sc.offs[E] + tid; pos < rows_end; pos += nthreads) pad(pos);
}

// Task-map entry of row tile q: {expert, row_start, rows_valid, 0}, or
// {-1, q*bm, 0, 0} past the last tile.
__device__ __forceinline__ int4 index_tile(int q, int E, int bm, const IndexScratch& sc) {
  const int row0 = q * bm;
  if (row0 >= sc.offs[E]) return make_int4(-1, row0, 0, 0);
  int lo = 0, hi = E - 1;   // largest e with offs[e] <= row0 (a non-empty expert)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sc.offs[mid] <= row0) lo = mid; else hi = mid - 1;
  }
  return make_int4(lo, row0, min(bm, sc.offs[lo] + sc.tot[lo] - row0), 0);
}

// Work-list entry q with coalesce C (after index_scan_offsets(.., C)): the
// expert's rows in tiles of up to C consecutive rows from its first, so a
// hot expert's weight tiles are streamed once per C rows rather than once
// per bm; {expert, first row, rows, 0}, or {-1, 0, 0, 0} past the last
// (coffs[E] entries).
__device__ __forceinline__ int4 index_work_tile(int q, int E, int C, const IndexScratch& sc) {
  if (q >= sc.coffs[E]) return make_int4(-1, 0, 0, 0);
  int lo = 0, hi = E - 1;   // largest e with coffs[e] <= q (an expert with rows)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sc.coffs[mid] <= q) lo = mid; else hi = mid - 1;
  }
  const int j = (q - sc.coffs[lo]) * C;   // rows of the expert before this tile
  return make_int4(lo, sc.offs[lo] + j, min(C, sc.tot[lo] - j), 0);
}

// The task map (tile_expert, tiles, num_tiles: tiles of bm rows) and, where
// idx.work_tiles is set, the work list of tiles of up to C rows, written by
// the block's threads from `sc`.  No barrier.
__device__ __forceinline__ void index_write_tiles(int E, int bm, int tiles_cap, int C,
                                                  const IndexScratch& sc, const IndexPtrs& idx) {
  const int tid = threadIdx.x, nthreads = blockDim.x;
  if (tid == 0) *idx.num_tiles = sc.offs[E] / bm;
  for (int q = tid; q < tiles_cap; q += nthreads) {
    const int4 t = index_tile(q, E, bm, sc);
    idx.tile_expert[q] = t.x;
    reinterpret_cast<int4*>(idx.tiles)[q] = t;
  }
  if (C > 0 && idx.work_tiles) {
    if (tid == 0) *idx.num_work_tiles = sc.coffs[E];
    for (int q = tid; q < idx.work_cap; q += nthreads)
      reinterpret_cast<int4*>(idx.work_tiles)[q] = index_work_tile(q, E, C, sc);
  }
}

}  // namespace moe
