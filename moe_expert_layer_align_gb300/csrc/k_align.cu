// k_align.cu — routing and index build as its own kernel (one CTA of 1024
// threads), used when the batch has too many assignments for every GEMM CTA
// to rebuild the index in shared memory.  The algorithm is index_build.cuh's
// (HPC-Ops × SGLang, section "MoE", fused pipeline, "routing and index
// build"); here rows, inverse positions and the task map go to global memory.
#include <cuda_bf16.h>
#include <cstdint>

#include "index_build.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {

// Block size of the one-CTA build and of the scan kernel.  (128 or 256
// threads for small batches measured slower: the per-expert loops get longer
// than the barriers get cheaper.)
constexpr int kAlignThreads = 1024;
constexpr int kAlignMaxStagedIds = 32768;  // ids staged in shared memory up to this many

// Batches of at most 32 assignments with plain ids and no work list: one
// warp holds every assignment, so the counting, ranking and offset passes of
// index_build.cuh (and their block barriers) reduce to warp votes.  The warp
// lists the active experts (at most 32) with their counts and padded offsets
// in shared memory and writes the assignments' rows; after one barrier every
// thread writes its share of counts, offsets, padding rows and the task map
// from that list.  The index is the one index_build.cuh builds: rows of an
// expert in ascending assignment order, offsets the exclusive prefix of the
// counts rounded up to bm (a power of two), invalid ids dropped and flagged.
// (At T*k = 8 and 128 experts the block passes took ~9k cycles after the
// ids arrived, mostly barrier and shared-memory latency chains.)
constexpr int kAlignSmallMax = 32;

__device__ __forceinline__ void align_small(const int32_t* __restrict__ ids, int tk, int E,
                                            int bm, int tiles_cap, const IndexPtrs& idx,
                                            int32_t* dev_status, int clear_status, int32_t* sm) {
  // sm: [0, 32) expert, [32, 64) count, [64, 96) padded offset of the active
  // experts; [96] how many; [97] padded total; [98] an invalid id was seen
  const int tid = threadIdx.x, lane = tid & 31;
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0 && dev_status && clear_status) *dev_status = 0;
  if (tid < 32) {
    // every lane loads (a valid address), then selects: a load under a
    // condition left the warp diverged, and each of the votes and shuffles
    // below then waited for it to reconverge (~300 cycles each at T*k = 8)
    const bool in = lane < tk;
    const int loaded = __ldg(ids + (in ? lane : 0));
    const int e = in ? loaded : -1;
    __syncwarp();
    const bool valid = in && e >= 0 && e < E;
    const int bits = key_bits(E);
    const unsigned grp = peer_mask(valid ? e : (1 << bits), bits);
    const bool leader = valid && lane == __ffs(grp) - 1;
    const int cnt = __popc(grp);
    const int padded = leader ? (cnt + bm - 1) & ~(bm - 1) : 0;
    // padded offset of this lane's expert: the padded counts of the smaller
    // active experts (one leader lane each)
    int off = 0;
    for (int j = 0; j < 32; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      const int pj = __shfl_sync(0xffffffffu, padded, j);
      if (pj > 0 && ej < e) off += pj;
    }
    int total = padded;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) total += __shfl_xor_sync(0xffffffffu, total, d);
    const unsigned leaders = __ballot_sync(0xffffffffu, leader);
    const bool bad = __any_sync(0xffffffffu, in && !valid);
    if (leader) {
      const int s = __popc(leaders & lanemask_lt());
      sm[s] = e;
      sm[32 + s] = cnt;
      sm[64 + s] = off;
    }
    if (lane == 0) {
      sm[96] = __popc(leaders);
      sm[97] = total;
      sm[98] = bad ? 1 : 0;
    }
    if (valid) {
      const int pos = off + __popc(grp & lanemask_lt());
      idx.sorted_ids[pos] = lane;
      idx.inv_pos[lane] = pos;
    } else if (in) {
      idx.inv_pos[lane] = -1;
    }
  }
  __syncthreads();
  const int na = sm[96], total = sm[97];
  for (int e = tid; e <= E; e += blockDim.x) {
    int c = 0, o = 0;
    for (int s = 0; s < na; ++s) {
      const int es = sm[s], cs = sm[32 + s];
      if (es == e) c = cs;
      if (es < e) o += (cs + bm - 1) & ~(bm - 1);
    }
    if (e < E) idx.counts[e] = c;
    idx.offsets[e] = o;   // e == E: the padded total
  }
  const int rows_end = tiles_cap * bm;
  for (int r = tid; r < rows_end; r += blockDim.x) {   // rows that hold no assignment
    bool held = false;
    for (int s = 0; s < na; ++s) {
      const int o = sm[64 + s];
      held = held || (r >= o && r < o + sm[32 + s]);
    }
    if (!held) idx.sorted_ids[r] = tk;
  }
  if (tid == 0) *idx.num_tiles = total / bm;
  for (int q = tid; q < tiles_cap; q += blockDim.x) {
    const int row0 = q * bm;
    int4 t = make_int4(-1, row0, 0, 0);
    for (int s = 0; s < na; ++s) {
      const int o = sm[64 + s], c = sm[32 + s];
      if (row0 >= o && row0 < o + ((c + bm - 1) & ~(bm - 1)))
        t = make_int4(sm[s], row0, min(bm, o + c - row0), 0);
    }
    idx.tile_expert[q] = t.x;
    reinterpret_cast<int4*>(idx.tiles)[q] = t;
  }
  if (tid == 0 && sm[98] && dev_status) atomicOr(dev_status, kStatusExpertId);
}

// The whole index by one block (the block's threads and dynamic shared
// memory).
__device__ __forceinline__ void align_block(const int32_t* __restrict__ ids, int T, int k, int E,
                                            int bm, int tiles_cap, const IndexPtrs& idx,
                                            int32_t* dev_status, int stage_ids, const IdMap& map,
                                            int clear_status, int32_t* sm) {
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  IndexScratch sc;
  sc.carve(sm, nwarps, E, map.Eg != 0);
  // [T*k] staged ids (optional), 16-byte aligned for vector stores
  int32_t* sids = sm + ((IndexScratch::words(nwarps, E) + 3) & ~static_cast<size_t>(3));

  const int tid = threadIdx.x;
  const int tk = T * k;
  if (tk <= kAlignSmallMax && map.plain() && idx.coalesce == 0) {
    align_small(ids, tk, E, bm, tiles_cap, idx, dev_status, clear_status, sm);
    return;
  }

  pdl_wait();
  pdl_launch_dependents();

  if (tid == 0 && dev_status && clear_status) *dev_status = 0;
  if (stage_ids && !map.plain()) {
    // shared experts / expert parallelism: stage the index experts
    for (int i = tid; i < tk; i += nthreads) sids[i] = mapped_id(ids, i, map);
  } else if (stage_ids) {
    // 16-byte loads, several in flight per thread (one dependent load per
    // iteration made this loop the kernel's cost at 32K assignments)
    const int n4 = (reinterpret_cast<uintptr_t>(ids) & 15) ? 0 : tk / 4;
    const int4* ids4 = reinterpret_cast<const int4*>(ids);
    int4* s4 = reinterpret_cast<int4*>(sids);
#pragma unroll 8
    for (int i = tid; i < n4; i += nthreads) s4[i] = __ldg(ids4 + i);
    for (int i = 4 * n4 + tid; i < tk; i += nthreads) sids[i] = __ldg(ids + i);
  }
  const int32_t* src = stage_ids ? sids : ids;

  index_count_and_scan(src, tk, E, bm, sc, idx.coalesce);
  for (int e = tid; e < E; e += nthreads) idx.counts[e] = sc.tot[e];
  for (int e = tid; e <= E; e += nthreads) idx.offsets[e] = sc.offs[e];
  index_scatter(
      src, tk, E, sc,
      [&](int pos, int a) {
        idx.sorted_ids[pos] = a;
        idx.inv_pos[a] = pos;
      },
      [&](int a) { idx.inv_pos[a] = -1; });
  index_pads(E, tiles_cap * bm, sc, [&](int pos) { idx.sorted_ids[pos] = tk; });
  index_write_tiles(E, bm, tiles_cap, idx.coalesce, sc, idx);
  __syncthreads();
  if (tid == 0 && *sc.flag && dev_status) atomicOr(dev_status, kStatusExpertId);
}

__global__ void __launch_bounds__(kAlignThreads)
    moe_align_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int bm, int tiles_cap,
                     IndexPtrs idx, int32_t* dev_status, int stage_ids, IdMap map,
                     int clear_status) {
  extern __shared__ int32_t sm[];
  align_block(ids, T, k, E, bm, tiles_cap, idx, dev_status, stage_ids, map, clear_status, sm);
}

// FP8 layers: block 0 builds the index as moe_align_kernel does, the other
// blocks quantise x meanwhile (HPC-Ops × SGLang, section "MoE": per token and
// 128-channel group, s = amax/448, e4m3 codes), four groups per warp at a
// time.  Neither needs the other, so one launch replaces two dependent ones
// in front of the Gate-Up.  The scales stay per token (xs): the Gate-Up
// looks each index row's token up in the index instead of reading a copy of
// the scales per index row, which would need the index first.
__global__ void __launch_bounds__(kAlignThreads)
    moe_align_quant_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int bm,
                           int tiles_cap, IndexPtrs idx, int32_t* dev_status, int stage_ids,
                           IdMap map, int clear_status, const __nv_bfloat16* __restrict__ x,
                           int H, uint8_t* __restrict__ xq, float* __restrict__ xs) {
  extern __shared__ int32_t sm[];
  if (blockIdx.x == 0) {
    align_block(ids, T, k, E, bm, tiles_cap, idx, dev_status, stage_ids, map, clear_status, sm);
    return;
  }
  pdl_wait();
  pdl_launch_dependents();
  constexpr int kWarps = kAlignThreads / 32;
  const int G = H / 128, items = T * G;
  const int nw = (gridDim.x - 1) * kWarps;
  for (int i0 = (blockIdx.x - 1) * kWarps + (threadIdx.x >> 5); i0 < items; i0 += 4 * nw) {
    int tt[4], gg[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + j * nw;
      tt[j] = i < items ? i / G : -1;
      gg[j] = i < items ? i % G : 0;
    }
    quant_x_groups4_warp(x, tt, gg, H, xq, xs);
  }
}

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int bm, int tiles_cap,
                         const IndexPtrs& idx, int32_t* dev_status, cudaStream_t st, bool pdl,
                         const IdMap& map, bool clear) {
  const int tk = T * k;
  const int stage_ids = tk <= kAlignMaxStagedIds ? 1 : 0;
  if (!stage_ids && !map.plain()) return cudaErrorInvalidValue;   // mapped ids are staged
  const int threads = kAlignThreads;
  const size_t smem =
      sizeof(int32_t) * (((IndexScratch::words(threads / 32, E) + 3) & ~static_cast<size_t>(3)) +
                         (stage_ids ? tk : 0));
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !configured[dev]) {
    err = cudaFuncSetAttribute(moe_align_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               227 * 1024);
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  return launch_kernel(moe_align_kernel, dim3(1), dim3(threads), smem, st, pdl, ids, T, k, E,
                       bm, tiles_cap, idx, dev_status, stage_ids, map, clear ? 1 : 0);
}

cudaError_t launch_align_quant(const int32_t* ids, int T, int k, int E, int bm, int tiles_cap,
                               const IndexPtrs& idx, int32_t* dev_status, cudaStream_t st,
                               bool pdl, const IdMap& map, bool clear, const void* x, int H,
                               uint8_t* xq, float* xs) {
  const int tk = T * k;
  const int stage_ids = tk <= kAlignMaxStagedIds ? 1 : 0;
  if (!stage_ids && !map.plain()) return cudaErrorInvalidValue;   // mapped ids are staged
  if (H % 128 != 0) return cudaErrorInvalidValue;
  const int threads = kAlignThreads;
  const size_t smem =
      sizeof(int32_t) * (((IndexScratch::words(threads / 32, E) + 3) & ~static_cast<size_t>(3)) +
                         (stage_ids ? tk : 0));
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !configured[dev]) {
    err = cudaFuncSetAttribute(moe_align_quant_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // quant blocks: a warp per four groups, at most two per SM (the warps loop)
  const int items = T * (H / 128);
  const int want = (items + 4 * (threads / 32) - 1) / (4 * (threads / 32));
  const int nq = want < 2 * sms ? want : 2 * sms;
  return launch_kernel(moe_align_quant_kernel, dim3(1 + (nq > 0 ? nq : 1)), dim3(threads), smem,
                       st, pdl, ids, T, k, E, bm, tiles_cap, idx, dev_status, stage_ids, map,
                       clear ? 1 : 0, static_cast<const __nv_bfloat16*>(x), H, xq, xs);
}

// ---------------------------------------------------------------- split build
// For many assignments the same algorithm runs over chunks of kChunk
// assignments, one CTA each, so that no single SM walks them all:
//   count:   per-CTA expert histogram of its chunk (hist[b][e]);
//   scan:    one CTA turns hist into per-CTA bases (exclusive prefix over b,
//            in place), totals, padded offsets, padding and the task map;
//   scatter: each CTA re-ranks its chunk and writes its assignments at
//            offsets[e] + base[b][e] + (rank inside the chunk).
// Chunks ascend in a and the in-chunk ranks are the block algorithm's, so
// the result equals the single-CTA build's.
constexpr int kChunk = 1024;
constexpr int kSplitThreads = 256;
constexpr int kSplitWarps = kSplitThreads / 32;

__host__ __device__ inline size_t chunk_smem_words(int E) {
  return ((IndexScratch::words(kSplitWarps, E) + 3) & ~static_cast<size_t>(3)) + kChunk;
}

__device__ __forceinline__ int stage_chunk(const int32_t* ids, int tk, int32_t* chunk,
                                           const IdMap& map) {
  const int a0 = blockIdx.x * kChunk;
  const int n = min(kChunk, tk - a0);
  if (map.plain())
    for (int i = threadIdx.x; i < n; i += kSplitThreads) chunk[i] = __ldg(ids + a0 + i);
  else
    for (int i = threadIdx.x; i < n; i += kSplitThreads) chunk[i] = mapped_id(ids, a0 + i, map);
  return n;
}

__global__ void __launch_bounds__(kSplitThreads)
    moe_align_count_kernel(const int32_t* __restrict__ ids, int tk, int E, int bm,
                           int32_t* __restrict__ hist, int32_t* __restrict__ flags, IdMap map,
                           int32_t* dev_status, int clear_status) {
  extern __shared__ int32_t sm[];
  IndexScratch sc;
  sc.carve(sm, kSplitWarps, E, map.Eg != 0);
  int32_t* chunk = sm + (chunk_smem_words(E) - kChunk);
  pdl_wait();
  pdl_launch_dependents();
  if (clear_status && dev_status && blockIdx.x == 0 && threadIdx.x == 0) *dev_status = 0;
  const int n = stage_chunk(ids, tk, chunk, map);
  index_count_and_scan(chunk, n, E, bm, sc);
  for (int e = threadIdx.x; e < E; e += kSplitThreads)
    hist[static_cast<size_t>(blockIdx.x) * E + e] = sc.tot[e];
  if (threadIdx.x == 0) flags[blockIdx.x] = *sc.flag;
}

__global__ void __launch_bounds__(kAlignThreads)
    moe_align_scan_kernel(int32_t* __restrict__ hist, const int32_t* __restrict__ flags, int nb,
                          int tk, int E, int bm, int tiles_cap, IndexPtrs idx,
                          int32_t* dev_status) {
  extern __shared__ int32_t sm[];
  IndexScratch sc;
  sc.carve(sm, 1, E);   // tot and offs only
  const int tid = threadIdx.x;
  pdl_wait();
  pdl_launch_dependents();
  // Per expert, the exclusive prefix over the chunks.  Each batch's counts
  // are all loaded before its bases are stored: a load-store-load walk put
  // one L2 round trip per chunk on the critical path (13.9 us at 32 chunks).
  constexpr int kScanBatch = 16;
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += kScanBatch) {
      int c[kScanBatch];
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j)
        c[j] = b0 + j < nb ? hist[static_cast<size_t>(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kScanBatch; ++j) {
        if (b0 + j < nb) hist[static_cast<size_t>(b0 + j) * E + e] = run;
        run += c[j];
      }
    }
    sc.tot[e] = run;
    idx.counts[e] = run;
  }
  __syncthreads();
  index_scan_offsets(E, bm, sc, idx.coalesce);
  for (int e = tid; e <= E; e += kAlignThreads) idx.offsets[e] = sc.offs[e];
  index_pads(E, tiles_cap * bm, sc, [&](int pos) { idx.sorted_ids[pos] = tk; });
  index_write_tiles(E, bm, tiles_cap, idx.coalesce, sc, idx);
  if (tid == 0 && dev_status) {
    int any = 0;
    for (int b = 0; b < nb; ++b) any |= flags[b];
    if (any) atomicOr(dev_status, kStatusExpertId);
  }
}

__global__ void __launch_bounds__(kSplitThreads)
    moe_align_scatter_kernel(const int32_t* __restrict__ ids, int tk, int E, int bm,
                             const int32_t* __restrict__ base, IndexPtrs idx, IdMap map) {
  extern __shared__ int32_t sm[];
  IndexScratch sc;
  sc.carve(sm, kSplitWarps, E, map.Eg != 0);
  int32_t* chunk = sm + (chunk_smem_words(E) - kChunk);
  pdl_wait();
  pdl_launch_dependents();
  const int n = stage_chunk(ids, tk, chunk, map);
  index_count_and_scan(chunk, n, E, bm, sc);   // in-chunk per-warp bases
  for (int e = threadIdx.x; e < E; e += kSplitThreads)
    sc.offs[e] = idx.offsets[e] + base[static_cast<size_t>(blockIdx.x) * E + e];
  __syncthreads();
  const int a0 = blockIdx.x * kChunk;
  index_scatter(
      chunk, n, E, sc,
      [&](int pos, int a) {
        idx.sorted_ids[pos] = a0 + a;
        idx.inv_pos[a0 + a] = pos;
      },
      [&](int a) { idx.inv_pos[a0 + a] = -1; });
}

size_t align_split_scratch_words(int T, int k, int E) {
  const int nb = (T * k + kChunk - 1) / kChunk;
  return static_cast<size_t>(nb) * E + nb;
}

cudaError_t launch_align_split(const int32_t* ids, int T, int k, int E, int bm, int tiles_cap,
                               const IndexPtrs& idx, int32_t* scratch, int32_t* dev_status,
                               cudaStream_t st, bool pdl, const IdMap& map, bool clear) {
  const int tk = T * k;
  const int nb = (tk + kChunk - 1) / kChunk;
  int32_t* hist = scratch;
  int32_t* flags = scratch + static_cast<size_t>(nb) * E;
  const size_t chunk_smem = 4 * chunk_smem_words(E);
  cudaError_t e = launch_kernel(moe_align_count_kernel, dim3(nb), dim3(kSplitThreads), chunk_smem,
                                st, pdl, ids, tk, E, bm, hist, flags, map, dev_status,
                                clear ? 1 : 0);
  if (e != cudaSuccess) return e;
  e = launch_kernel(moe_align_scan_kernel, dim3(1), dim3(kAlignThreads),
                    4 * IndexScratch::words(1, E), st, true, hist,
                    static_cast<const int32_t*>(flags), nb, tk, E, bm, tiles_cap, idx, dev_status);
  if (e != cudaSuccess) return e;
  return launch_kernel(moe_align_scatter_kernel, dim3(nb), dim3(kSplitThreads), chunk_smem, st,
                       true, ids, tk, E, bm, static_cast<const int32_t*>(hist), idx, map);
}

}  // namespace moe
