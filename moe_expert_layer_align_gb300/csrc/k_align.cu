// k_align.cu — routing and index build as its own kernel (one CTA of 1024
// threads), used when the batch has too many assignments for every GEMM CTA
// to rebuild the index in shared memory.  The algorithm is index_build.cuh's
// (HPC-Ops × SGLang, section "MoE", fused pipeline, "routing and index
// build"); here rows, inverse positions and the task map go to global memory.
#include <cstdint>

#include "index_build.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kAlignMaxStagedIds = 32768;  // ids staged in shared memory up to this many

__global__ void __launch_bounds__(kAlignThreads)
    moe_align_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int bm, int tiles_cap,
                     IndexPtrs idx, int32_t* dev_status, int stage_ids) {
  extern __shared__ int32_t sm[];
  IndexScratch sc;
  sc.carve(sm, kAlignWarps, E);
  int32_t* sids = sm + IndexScratch::words(kAlignWarps, E);   // [T*k] staged ids (optional)

  const int tid = threadIdx.x;
  const int tk = T * k;

  pdl_wait();
  pdl_launch_dependents();

  if (tid == 0 && dev_status) *dev_status = 0;
  if (stage_ids)
    for (int i = tid; i < tk; i += kAlignThreads) sids[i] = __ldg(ids + i);
  const int32_t* src = stage_ids ? sids : ids;

  index_count_and_scan(src, tk, E, bm, sc);
  for (int e = tid; e < E; e += kAlignThreads) idx.counts[e] = sc.tot[e];
  for (int e = tid; e <= E; e += kAlignThreads) idx.offsets[e] = sc.offs[e];
  index_scatter(
      src, tk, E, sc,
      [&](int pos, int a) {
        idx.sorted_ids[pos] = a;
        idx.inv_pos[a] = pos;
      },
      [&](int a) { idx.inv_pos[a] = -1; });
  index_pads(E, tiles_cap * bm, sc, [&](int pos) { idx.sorted_ids[pos] = tk; });
  if (tid == 0) *idx.num_tiles = sc.offs[E] / bm;
  for (int q = tid; q < tiles_cap; q += kAlignThreads) {
    const int4 t = index_tile(q, E, bm, sc);
    idx.tile_expert[q] = t.x;
    reinterpret_cast<int4*>(idx.tiles)[q] = t;
  }
  __syncthreads();
  if (tid == 0 && *sc.flag && dev_status) atomicOr(dev_status, kStatusExpertId);
}

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int bm, int tiles_cap,
                         const IndexPtrs& idx, int32_t* dev_status, cudaStream_t st, bool pdl) {
  const int tk = T * k;
  const int stage_ids = tk <= kAlignMaxStagedIds ? 1 : 0;
  const size_t smem =
      sizeof(int32_t) * (IndexScratch::words(kAlignWarps, E) + (stage_ids ? tk : 0));
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
