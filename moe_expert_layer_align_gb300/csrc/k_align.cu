// k_align.cu — routing and index build.
//
// HPC-Ops × SGLang, section "MoE", fused pipeline, "routing and index build":
// starting from the selected top-k expert ids, a shared-memory counting pass
// arranges token-expert assignments into contiguous per-expert output
// intervals, which relieves global atomic pressure, and emits the routing
// index and the per-tile task map that the persistent expert GEMM consumes.
//
// One CTA of 1024 threads (32 warps).  Warp w owns the contiguous slice
// [w*seg, (w+1)*seg) of the flat assignments a = t*k + j and walks it in
// rounds of 32 consecutive assignments, one per lane:
//   1. count: __match_any_sync groups the lanes of a round by expert; the
//      group's lowest lane adds the group size to cnt[w][e] (shared memory,
//      one writer per address, no atomics);
//   2. scan: per expert, an exclusive prefix of cnt[.][e] over warps gives
//      each warp's base inside the expert; a block scan of the padded counts
//      gives offsets[];
//   3. scatter: the same rounds again; an assignment's row is
//      offsets[e] + base[w][e] + (lanes of its group below it), after which
//      the group's lowest lane advances base[w][e].
// Slices are ascending in a, rounds are in order and ranks inside a round
// follow the lane, so every expert's interval holds its assignments in
// ascending a: the result is unique and deterministic.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kAlignMaxStagedIds = 32768;  // ids staged in shared memory up to this many

__device__ __forceinline__ int lanemask_lt() {
  int m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__global__ void __launch_bounds__(kAlignThreads)
    moe_align_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int bm, int tiles_cap,
                     IndexPtrs idx, int32_t* dev_status, int stage_ids) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                             // [32][E]: counts, then bases
  int32_t* offs = cnt + kAlignWarps * E;         // [E + 1]
  int32_t* tot = offs + E + 1;                   // [E] per-expert totals
  int32_t* wsum = tot + E;                       // [32] scan scratch
  int32_t* flag = wsum + kAlignWarps;            // [1] invalid-id seen
  int32_t* sids = flag + 1;                      // [T*k] staged ids (optional)

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tk = T * k;

  pdl_wait();
  pdl_launch_dependents();

  if (tid == 0) {
    *flag = 0;
    if (dev_status) *dev_status = 0;
  }
  for (int i = tid; i < kAlignWarps * E; i += kAlignThreads) cnt[i] = 0;
  if (stage_ids)
    for (int i = tid; i < tk; i += kAlignThreads) sids[i] = __ldg(ids + i);
  __syncthreads();
  const int32_t* src = stage_ids ? sids : ids;

  const int seg = (tk + kAlignWarps - 1) / kAlignWarps;
  const int beg = min(tk, warp * seg);
  const int end = min(tk, beg + seg);

  // 1. count per (warp, expert)
  for (int base = beg; base < end; base += 32) {
    const int a = base + lane;
    const bool in = a < end;
    const int e = in ? src[a] : -1;
    const bool valid = in && e >= 0 && e < E;
    if (in && !valid) *flag = 1;
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid && lane == __ffs(grp) - 1) cnt[warp * E + e] += __popc(grp);
    __syncwarp();
  }
  __syncthreads();

  // 2a. per expert: exclusive prefix over warps, total, padded size
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = 0;
    for (int w = 0; w < kAlignWarps; ++w) {
      const int c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
    tot[e] = run;
    idx.counts[e] = run;
  }
  __syncthreads();

  // 2b. block scan of padded sizes over experts (E <= 1024): offs[e+1]
  {
    const int v = (tid < E) ? ((tot[tid] + bm - 1) / bm) * bm : 0;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int s = wsum[lane];
      int si = s;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, si, d);
        if (lane >= d) si += o;
      }
      wsum[lane] = si - s;  // exclusive prefix of warp sums
    }
    __syncthreads();
    if (tid < E) offs[tid + 1] = incl + wsum[warp];
    if (tid == 0) offs[0] = 0;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += kAlignThreads) idx.offsets[e] = offs[e];

  // 3. scatter in ascending a
  for (int base = beg; base < end; base += 32) {
    const int a = base + lane;
    const bool in = a < end;
    const int e = in ? src[a] : -1;
    const bool valid = in && e >= 0 && e < E;
    const unsigned grp = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid) {
      const int pos = offs[e] + cnt[warp * E + e] + __popc(grp & lanemask_lt());
      idx.sorted_ids[pos] = a;
      idx.inv_pos[a] = pos;
    } else if (in) {
      idx.inv_pos[a] = -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(grp) - 1) cnt[warp * E + e] += __popc(grp);
    __syncwarp();
  }

  // 4. padding rows (disjoint from step 3's rows): the sentinel T*k
  const int rows_cap = tiles_cap * bm;
  for (int e = warp; e < E; e += kAlignWarps)
    for (int pos = offs[e] + tot[e] + lane; pos < offs[e + 1]; pos += 32)
      idx.sorted_ids[pos] = tk;
  for (int pos = offs[E] + tid; pos < rows_cap; pos += kAlignThreads) idx.sorted_ids[pos] = tk;

  // 5. task map
  const int num_tiles = offs[E] / bm;
  if (tid == 0) *idx.num_tiles = num_tiles;
  for (int q = tid; q < tiles_cap; q += kAlignThreads) {
    const int row0 = q * bm;
    int4 t;
    if (q < num_tiles) {
      // largest e with offs[e] <= row0 (that expert is non-empty)
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= row0) lo = mid; else hi = mid - 1;
      }
      t = make_int4(lo, row0, min(bm, offs[lo] + tot[lo] - row0), 0);
    } else {
      t = make_int4(-1, row0, 0, 0);
    }
    idx.tile_expert[q] = t.x;
    reinterpret_cast<int4*>(idx.tiles)[q] = t;
  }
  __syncthreads();
  if (tid == 0 && *flag && dev_status) atomicOr(dev_status, kStatusExpertId);
}

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int bm, int tiles_cap,
                         const IndexPtrs& idx, int32_t* dev_status, cudaStream_t st, bool pdl) {
  const int tk = T * k;
  const int stage_ids = tk <= kAlignMaxStagedIds ? 1 : 0;
  const size_t smem =
      sizeof(int32_t) * (static_cast<size_t>(kAlignWarps) * E + (E + 1) + E + kAlignWarps + 1 +
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
  return launch_kernel(moe_align_kernel, dim3(1), dim3(kAlignThreads), smem, st, pdl, ids, T, k, E,
                       bm, tiles_cap, idx, dev_status, stage_ids);
}

}  // namespace moe
