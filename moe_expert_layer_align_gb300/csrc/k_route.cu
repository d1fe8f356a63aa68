// k_route.cu — the in-path router's top-k, the FP8 quantisation of x and the
// routing index in one launch.
//
// HPC-Ops × SGLang: section "Router GEMM" (two-bf16 scores, top-k) feeds
// section "MoE", "routing and index build".  Run as separate kernels these
// are three launches of a few microseconds each in front of a decode-sized
// layer; here one grid does all three:
//   * CTA b owns tokens 4b..4b+3: warp w < 4 reduces the router GEMM's
//     split-K partials of token 4b+w into scores, selects the top-k and
//     writes ids and weights, while warp 4+w (FP8 layer) quantises the
//     token's row of x;
//   * every CTA takes a ticket when its warps are done; the CTA that draws
//     the last ticket builds the index from all tokens' ids with the block
//     algorithm of index_build.cuh.  Nothing waits on another CTA: the last
//     one simply starts after the others have published their ids.
// The ticket counter is zeroed by the router GEMM at its start (one launch
// earlier in the same chain), so each call starts from zero.
#include <cuda_bf16.h>
#include <cstdint>

#include "index_build.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {

constexpr int kRouteTokens = 4;                     // tokens per CTA
constexpr int kRouteThreads = 64 * kRouteTokens;    // a top-k and a quant warp each
constexpr int kRouteWarps = kRouteThreads / 32;

__global__ void __launch_bounds__(kRouteThreads) moe_route_index_kernel(RouteIndexParams q) {
  extern __shared__ int32_t sm[];
  __shared__ int s_last;
  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_wait();                 // the router GEMM's partials (and the zeroed counter)
  pdl_launch_dependents();
  const int t = blockIdx.x * kRouteTokens + (warp % kRouteTokens);
  if (t < q.T) {
    if (warp < kRouteTokens)
      router_topk_warp(q.P, q.splits, q.rows_cap_r, t, q.E, q.k, q.score_fn, q.scale, q.scores,
                       q.ids, q.w);
    else if (q.xq != nullptr)
#pragma unroll 4
      for (int g = 0; g < q.H / 128; ++g)
        quant_x_group_warp(static_cast<const __nv_bfloat16*>(q.x), t, g, q.H, q.xq, q.xs);
  }
  // Publish this CTA's ids, then take a ticket.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(q.counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();            // the other CTAs' ids are visible from here on

  IndexScratch sc;
  sc.carve(sm, kRouteWarps, q.Ei, 0);
  int32_t* sids = sm + ((IndexScratch::words(kRouteWarps, q.Ei) + 3) & ~static_cast<size_t>(3));
  const int tk = q.T * q.k;
  // ids written by other CTAs of this grid: read through L2 (ld.global.cg)
  for (int a = tid; a < tk; a += kRouteThreads) sids[a] = __ldcg(q.ids + a);
  index_count_and_scan(sids, tk, q.Ei, q.bm, sc);
  const IndexPtrs& idx = q.idx;
  for (int e = tid; e < q.Ei; e += kRouteThreads) idx.counts[e] = sc.tot[e];
  for (int e = tid; e <= q.Ei; e += kRouteThreads) idx.offsets[e] = sc.offs[e];
  index_scatter(
      sids, tk, q.Ei, sc,
      [&](int pos, int a) {
        idx.sorted_ids[pos] = a;
        idx.inv_pos[a] = pos;
      },
      [&](int a) { idx.inv_pos[a] = -1; });
  index_pads(q.Ei, q.tiles_cap * q.bm, sc, [&](int pos) { idx.sorted_ids[pos] = tk; });
  if (tid == 0) *idx.num_tiles = sc.offs[q.Ei] / q.bm;
  for (int i = tid; i < q.tiles_cap; i += kRouteThreads) {
    const int4 tile = index_tile(i, q.Ei, q.bm, sc);
    idx.tile_expert[i] = tile.x;
    reinterpret_cast<int4*>(idx.tiles)[i] = tile;
  }
  __syncthreads();
  if (tid == 0 && q.dev_status && *sc.flag) atomicOr(q.dev_status, kStatusExpertId);
}

size_t route_index_smem_bytes(int T, int k, int Ei) {
  return sizeof(int32_t) *
         (((IndexScratch::words(kRouteWarps, Ei) + 3) & ~static_cast<size_t>(3)) +
          static_cast<size_t>(T) * k);
}

cudaError_t launch_route_index(const RouteIndexParams& q, cudaStream_t st, bool pdl) {
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !configured[dev]) {
    err = cudaFuncSetAttribute(moe_route_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               128 * 1024);
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  const int grid = (q.T + kRouteTokens - 1) / kRouteTokens;
  return launch_kernel(moe_route_index_kernel, dim3(grid), dim3(kRouteThreads),
                       route_index_smem_bytes(q.T, q.k, q.Ei), st, pdl, q);
}

}  // namespace moe
