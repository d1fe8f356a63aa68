// k_route.cu — the in-path router GEMM, its top-k, the FP8 quantisation of x
// and the routing index in one launch.
//
// HPC-Ops × SGLang: section "Router GEMM" (the two-bf16 scores, top-k) feeds
// section "MoE", "routing and index build".  As separate kernels these are
// four dependent launches of a few microseconds each in front of a
// decode-sized layer; here one cooperative grid (every CTA resident, so CTAs
// may wait on one another) runs them as three phases with a grid barrier
// between them:
//   1. the router GEMM over [hi; lo] on the tensor cores, exactly as
//      moe_gemm_kernel runs it (gemm_cta, dense token rows, split-K partials
//      into the workspace), on as many CTAs as it has work units;
//      The CTAs beyond the GEMM's meanwhile quantise x's 128-channel groups
//      (FP8 layers), which needs no routing;
//   2. "owner" CTA c takes tokens [c*tpc, (c+1)*tpc): a warp per token sums
//      the partials into scores and selects the top-k (route_common.cuh), and
//      the block algorithm of index_build.cuh counts the block's assignments
//      per expert and ranks them (stable, by assignment) — its histogram goes
//      to the workspace;
//   3. every owner reads all histograms: the experts' totals give the padded
//      offsets, the histograms of the owners before it give its bases, and
//      it writes its assignments' rows; owner 0 also writes counts, offsets,
//      padding, the task map and the tile count.
// Owners' token blocks ascend, and ranks inside a block are the block
// algorithm's, so the index is the one moe_align builds from the same ids.
// The grid barrier waits are bounded (kWaitLimitNs); one that gives up sets
// the timeout bit and the CTA skips the remaining phases.  Its two counters
// are zeroed on the stream before every launch.
#include <cuda_bf16.h>
#include <cstdint>

#include "k_gemm.cuh"
#include "route_common.cuh"

namespace moe {

// Grid-wide barrier of a cooperative launch: arrive on *ctr, then wait
// (bounded) until n CTAs have.  Returns false, with the timeout bit set, if
// the wait gave up.
__device__ __forceinline__ bool grid_barrier(unsigned int* ctr, unsigned int n,
                                             int32_t* dev_status, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();   // this CTA's writes before its arrival, device-wide
    atomicAdd(ctr, 1u);
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
      if (v >= n) break;
      if ((i & 63u) == 0u && global_timer_ns() - t0 > kWaitLimitNs) {
        ok = 0;
        if (dev_status) atomicOr(dev_status, kStatusTimeout);
        break;
      }
    }
    __threadfence();
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

template <int BN>
__global__ void __launch_bounds__(GemmShape<0, BN, kDense>::kThreads, 1)
    moe_route_front_kernel(const __grid_constant__ CUtensorMap tmW,
                           const __grid_constant__ CUtensorMap tmX, const GemmParams gp,
                           const RouteFrontParams q) {
  using S = GemmShape<0, BN, kDense>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_flag;

  constexpr int kThreads = S::kThreads;
  constexpr int kWarps = kThreads / 32;
  const int tid = threadIdx.x, warp = tid >> 5;

  // 1. router GEMM partial sums (P = gp.out) on the first q.gemm_ctas CTAs;
  // the others meanwhile quantise x (FP8 layers; it needs no routing), four
  // 128-channel groups per warp at a time
  gemm_cta<0, BN, kDense, 1>(tmW, tmX, gp, smem_raw);
  if (q.xq != nullptr && (static_cast<int>(blockIdx.x) >= q.gemm_ctas ||
                          static_cast<int>(gridDim.x) <= q.gemm_ctas)) {
    const int G = q.H / 128, items = q.T * G;
    const int qc0 = static_cast<int>(gridDim.x) > q.gemm_ctas ? q.gemm_ctas : 0;
    const int nw = (gridDim.x - qc0) * kWarps;
    for (int i0 = (blockIdx.x - qc0) * kWarps + warp; i0 < items; i0 += 4 * nw) {
      int tt[4], gg[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j * nw;
        tt[j] = i < items ? i / G : -1;
        gg[j] = i < items ? i % G : 0;
      }
      quant_x_groups4_warp(static_cast<const __nv_bfloat16*>(q.x), tt, gg, q.H, q.xq, q.xs);
    }
  }
  if (!grid_barrier(q.bar, gridDim.x, q.dev_status, &s_flag)) return;

  const int c = blockIdx.x;
  const bool owner = c < q.owners;
  // shared memory of phase 1 is free again: index scratch, the block's ids,
  // the experts' bases
  int32_t* sm = reinterpret_cast<int32_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~static_cast<uintptr_t>(15));
  IndexScratch sc;
  sc.carve(sm, kWarps, q.Ei, 0);
  int32_t* chunk = sm + ((IndexScratch::words(kWarps, q.Ei) + 3) & ~static_cast<size_t>(3));
  int32_t* bse = chunk + q.tpc * q.k;
  const int t0 = c * q.tpc, t1 = min(q.T, t0 + q.tpc);
  const int a0 = t0 * q.k;
  const int n = owner ? max(0, t1 - t0) * q.k : 0;

  // 2. top-k and the block's per-expert counts
  if (owner) {
    for (int t = t0 + warp; t < t1; t += kWarps)
      router_topk_warp<true>(q.P, q.splits, q.rows_cap_r, t, q.E, q.k, q.score_fn, q.scale,
                             q.scores, q.ids, q.w, chunk + (t - t0) * q.k);
    __syncthreads();
    index_count_and_scan(chunk, n, q.Ei, q.bm, sc);   // per-warp bases, block totals
    for (int e = tid; e < q.Ei; e += kThreads)
      q.hist[static_cast<size_t>(c) * q.Ei + e] = sc.tot[e];
  }
  if (!grid_barrier(q.bar + 1, gridDim.x, q.dev_status, &s_flag) || !owner) return;

  // 3. totals, offsets, this block's bases; then its rows
  for (int e = tid; e < q.Ei; e += kThreads) {
    int base = 0, tot = 0;
    for (int b0 = 0; b0 < q.owners; b0 += 8) {   // eight loads in flight at a time
      int h[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        h[j] = b0 + j < q.owners ? __ldcg(q.hist + static_cast<size_t>(b0 + j) * q.Ei + e) : 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        base += b0 + j < c ? h[j] : 0;
        tot += h[j];
      }
    }
    sc.tot[e] = tot;
    bse[e] = base;
  }
  __syncthreads();
  index_scan_offsets(q.Ei, q.bm, sc, q.idx.coalesce);   // sc.offs: the layer's padded offsets
  const IndexPtrs& idx = q.idx;
  const int tk = q.T * q.k;
  if (c == 0) {
    for (int e = tid; e < q.Ei; e += kThreads) idx.counts[e] = sc.tot[e];
    for (int e = tid; e <= q.Ei; e += kThreads) idx.offsets[e] = sc.offs[e];
    index_pads(q.Ei, q.tiles_cap * q.bm, sc, [&](int pos) { idx.sorted_ids[pos] = tk; });
    index_write_tiles(q.Ei, q.bm, q.tiles_cap, idx.coalesce, sc, idx);
  }
  __syncthreads();
  for (int e = tid; e < q.Ei; e += kThreads) sc.offs[e] += bse[e];
  __syncthreads();
  index_scatter(
      chunk, n, q.Ei, sc,
      [&](int pos, int a) {
        idx.sorted_ids[pos] = a0 + a;
        idx.inv_pos[a0 + a] = pos;
      },
      [&](int a) { idx.inv_pos[a0 + a] = -1; });
}

size_t route_front_smem_bytes(int bn, int tpc, int k, int Ei) {
  const size_t idx = 16 + sizeof(int32_t) *
      (((IndexScratch::words(6, Ei) + 3) & ~static_cast<size_t>(3)) +
       static_cast<size_t>(tpc) * k + Ei);
  size_t gemm = 0;
  switch (bn) {
    case 16: gemm = GemmShape<0, 16, kDense>::kSmemBytes; break;
    case 32: gemm = GemmShape<0, 32, kDense>::kSmemBytes; break;
    case 64: gemm = GemmShape<0, 64, kDense>::kSmemBytes; break;
    default: gemm = GemmShape<0, 128, kDense>::kSmemBytes; break;
  }
  return gemm > idx ? gemm : idx;
}

template <int BN>
cudaError_t launch_route_front_bn(int grid, cudaStream_t st, const CUtensorMap& tmW,
                                  const CUtensorMap& tmX, const GemmParams& gp,
                                  const RouteFrontParams& q) {
  static_assert(GemmShape<0, BN, kDense>::kThreads / 32 == 6, "phase 2-3 sized for 6 warps");
  auto kern = moe_route_front_kernel<BN>;
  // dynamic shared memory up to the per-block limit less room for the
  // kernel's static shared memory (the barrier flag)
  constexpr size_t kDynMax = kMaxGemmSmem - 1024;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !configured[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kDynMax));
    if (err != cudaSuccess) return err;
    configured[dev] = 1;
  }
  const size_t smem = route_front_smem_bytes(BN, q.tpc, q.k, q.Ei);
  if (smem > kDynMax) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(GemmShape<0, BN, kDense>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: they wait on one another
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmW, tmX, gp, q);
}

cudaError_t launch_route_front(int bn, int grid, cudaStream_t st, const CUtensorMap& tmW,
                               const CUtensorMap& tmX, const GemmParams& gp,
                               const RouteFrontParams& q) {
  switch (bn) {
    case 16: return launch_route_front_bn<16>(grid, st, tmW, tmX, gp, q);
    case 32: return launch_route_front_bn<32>(grid, st, tmW, tmX, gp, q);
    case 64: return launch_route_front_bn<64>(grid, st, tmW, tmX, gp, q);
    case 128: return launch_route_front_bn<128>(grid, st, tmW, tmX, gp, q);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
