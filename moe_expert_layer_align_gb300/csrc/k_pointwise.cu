// k_pointwise.cu — the bandwidth-bound stages around the expert GEMMs:
// activation quantisation, the fused SiLU-and-mul (+ FP8 requantisation),
// the top-k weighted combine, and the router's weight split and top-k.
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "route_common.cuh"

namespace moe {

// ---------------------------------------------------------------- x quant
// x bf16 [T][H] -> xq e4m3 [T][H], xs [T][H/128].  The scales are also
// written to the index rows that hold the token's assignments
// (xs_rows[inv_pos[t*k+j]]), so the Gate-Up epilogue reads them by row
// without going through the index.
//
// Block (t, b) quantises eight group pairs of token t, one per warp: each
// half-warp one 128-channel group with eight channels per lane (one 16-byte
// load, one 8-byte store); the token's index rows are staged once per block.
constexpr int kQuantThreads = 256;
constexpr int kQuantMaxK = 64;   // index rows of a token staged in shared memory

__global__ void __launch_bounds__(kQuantThreads) moe_quant_x_kernel(
    const __nv_bfloat16* __restrict__ x, int T, int H, int k, const int32_t* __restrict__ inv_pos,
    uint8_t* __restrict__ xq, float* __restrict__ xs, float* __restrict__ xs_rows, int rows_cap) {
  __shared__ int s_pos[kQuantMaxK];
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int G = H / 128;
  const bool staged = inv_pos != nullptr && k <= kQuantMaxK;
  if (staged) {
    for (int j = threadIdx.x; j < k; j += kQuantThreads)
      s_pos[j] = __ldg(inv_pos + static_cast<size_t>(t) * k + j);
    __syncthreads();
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = lane & 15;
  const int gp = blockIdx.y * (kQuantThreads / 32) + warp;
  if (2 * gp < G) {
    const int g = 2 * gp + (lane >> 4);
    const bool on = g < G;   // an odd G leaves the last pair's upper half idle
    const size_t base = static_cast<size_t>(t) * H + g * 128 + hl * 8;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (on) raw = __ldg(reinterpret_cast<const uint4*>(x + base));
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w4[i]);
      v[2 * i] = __low2float(b);
      v[2 * i + 1] = __high2float(b);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int d = 8; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float sc = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
    uint32_t q[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint16_t lo = cvt_e4m3x2(__fdiv_rn(v[4 * i + 1], sc), __fdiv_rn(v[4 * i], sc));
      const uint16_t hi = cvt_e4m3x2(__fdiv_rn(v[4 * i + 3], sc), __fdiv_rn(v[4 * i + 2], sc));
      q[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    if (!on) return;
    *reinterpret_cast<uint2*>(xq + base) = make_uint2(q[0], q[1]);
    if (hl == 0) xs[static_cast<size_t>(t) * G + g] = sc;
    if (inv_pos != nullptr)
      for (int j = hl; j < k; j += 16) {
        const int pos = staged ? s_pos[j] : __ldg(inv_pos + static_cast<size_t>(t) * k + j);
        if (static_cast<unsigned>(pos) < static_cast<unsigned>(rows_cap))
          xs_rows[static_cast<size_t>(pos) * G + g] = sc;
      }
  }
}

cudaError_t launch_quant_x(const void* x, int T, int H, int k, const int32_t* inv_pos,
                           uint8_t* xq, float* xs, float* xs_rows, int rows_cap, cudaStream_t st,
                           bool pdl) {
  const int pairs = (H / 128 + 1) / 2;
  const dim3 grid(T, (pairs + kQuantThreads / 32 - 1) / (kQuantThreads / 32));
  return launch_kernel(moe_quant_x_kernel, grid, dim3(kQuantThreads), 0, st, pdl,
                       static_cast<const __nv_bfloat16*>(x), T, H, k, inv_pos, xq, xs, xs_rows,
                       rows_cap);
}

// ---------------------------------------------------------------- act
// HPC-Ops × SGLang, section "MoE", "Gate-Up and activation": SiLU-and-mul and
// FP8 requantisation run as one fused kernel whose output Down reads as is.
// For each index row p that holds an assignment:
//   g = sum_s G[s][p][i], u = sum_s G[s][p][I + i] (split-K partials in order)
//   a = SiLU(g) * u = g / (1 + exp(-g)) * u
// BF16: A[p][i] = bf16(a).  FP8: per 128 channels s = amax/448, codes e4m3.
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

constexpr int kActThreads = 256;

template <int FP8>
__global__ void __launch_bounds__(kActThreads)
    moe_act_kernel(const float* __restrict__ G, int splits, int rows_cap, int I,
                   const int32_t* __restrict__ sorted_ids, int sentinel, void* __restrict__ A,
                   float* __restrict__ As) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t two_i = 2 * static_cast<size_t>(I);
  const size_t slice = static_cast<size_t>(rows_cap) * two_i;
  // Block-strided over index rows, thread-strided over 4-channel groups.  In
  // FP8 mode a warp covers one whole 128-channel group per iteration (the
  // loop bound is warp-uniform because I % 128 == 0).
  for (int p = blockIdx.x; p < rows_cap; p += gridDim.x) {
    if (__ldg(sorted_ids + p) >= sentinel) continue;  // padding row (block-uniform)
    const float* row = G + static_cast<size_t>(p) * two_i;
    for (int i = threadIdx.x * 4; i < I; i += kActThreads * 4) {
      float4 g = __ldg(reinterpret_cast<const float4*>(row + i));
      float4 u = __ldg(reinterpret_cast<const float4*>(row + I + i));
#pragma unroll 4
      for (int s = 1; s < splits; ++s) {
        const float4 gs = __ldg(reinterpret_cast<const float4*>(row + s * slice + i));
        const float4 us = __ldg(reinterpret_cast<const float4*>(row + s * slice + I + i));
        g.x += gs.x; g.y += gs.y; g.z += gs.z; g.w += gs.w;
        u.x += us.x; u.y += us.y; u.z += us.z; u.w += us.w;
      }
      float v[4] = {silu_mul(g.x, u.x), silu_mul(g.y, u.y), silu_mul(g.z, u.z),
                    silu_mul(g.w, u.w)};
      if (FP8) {
        float sc;
        const uint32_t q = quant_group4(v, &sc);
        uint8_t* Aq = static_cast<uint8_t*>(A);
        *reinterpret_cast<uint32_t*>(Aq + static_cast<size_t>(p) * I + i) = q;
        if ((threadIdx.x & 31) == 0) As[static_cast<size_t>(p) * (I / 128) + i / 128] = sc;
      } else {
        __nv_bfloat16* Ab = static_cast<__nv_bfloat16*>(A) + static_cast<size_t>(p) * I + i;
        __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t*>(&lo);
        packed.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(Ab) = packed;
      }
    }
  }
}

cudaError_t launch_act(int fp8, const float* G, int splits, int rows_cap, int I,
                       const int32_t* sorted_ids, int sentinel, void* A, float* As,
                       cudaStream_t st, bool pdl) {
  // A few resident blocks per SM walk all rows: launching one block per
  // (row, column chunk) spent most of the stage scheduling blocks of padding.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = rows_cap < 4 * sms ? rows_cap : 4 * sms;
  if (fp8)
    return launch_kernel(moe_act_kernel<1>, dim3(grid), dim3(kActThreads), 0, st, pdl, G, splits,
                         rows_cap, I, sorted_ids, sentinel, A, As);
  return launch_kernel(moe_act_kernel<0>, dim3(grid), dim3(kActThreads), 0, st, pdl, G, splits,
                       rows_cap, I, sorted_ids, sentinel, A, As);
}

// ---------------------------------------------------------------- combine
// HPC-Ops × SGLang, section "MoE", "PDL-chained stages": the final top-k
// weighted reduction restores expert outputs to token order.
//   out[t][h] = sum_{j ascending} w[t][j] * sum_{s ascending} Y[s][inv_pos[t*k+j]][h]
// fp32, fixed order, no atomics.
constexpr int kCombineBatch = 8;   // assignments whose rows are loaded together

__global__ void __launch_bounds__(128)
    moe_combine_kernel(const float* __restrict__ Y, int splits, int rows_cap, int H,
                       const int32_t* __restrict__ inv_pos, const float* __restrict__ topk_w,
                       int T, int k, int k_routed, float w_shared, void* __restrict__ out,
                       int out_bf16) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int h = (blockIdx.y * 128 + threadIdx.x) * 4;
  if (h >= H) return;
  const size_t slice = static_cast<size_t>(rows_cap) * H;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < k; j0 += kCombineBatch) {
    // Issue every row load of the batch before reducing: the reduction order
    // (splits ascending, then j ascending) is unchanged.
    int pos[kCombineBatch];
    float w[kCombineBatch];
    float4 y[kCombineBatch];
#pragma unroll
    for (int b = 0; b < kCombineBatch; ++b) {
      const int j = j0 + b;
      pos[b] = j < k ? __ldg(inv_pos + static_cast<size_t>(t) * k + j) : -1;
      if (pos[b] >= rows_cap) pos[b] = -1;   // only rows of the index are read
      // routed slots weigh topk_w[t][j]; the shared experts' slots w_shared
      w[b] = j < k_routed ? __ldg(topk_w + static_cast<size_t>(t) * k_routed + j)
                          : (j < k ? w_shared : 0.f);
    }
#pragma unroll
    for (int b = 0; b < kCombineBatch; ++b)
      y[b] = pos[b] >= 0 ? __ldg(reinterpret_cast<const float4*>(Y + static_cast<size_t>(pos[b]) * H + h))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int s = 1; s < splits; ++s) {
#pragma unroll
      for (int b = 0; b < kCombineBatch; ++b) {
        if (pos[b] < 0) continue;
        const float4 ys = __ldg(reinterpret_cast<const float4*>(
            Y + s * slice + static_cast<size_t>(pos[b]) * H + h));
        y[b].x += ys.x; y[b].y += ys.y; y[b].z += ys.z; y[b].w += ys.w;
      }
    }
#pragma unroll
    for (int b = 0; b < kCombineBatch; ++b) {
      if (pos[b] < 0) continue;   // dropped assignment contributes 0
      acc.x = fmaf(w[b], y[b].x, acc.x);
      acc.y = fmaf(w[b], y[b].y, acc.y);
      acc.z = fmaf(w[b], y[b].z, acc.z);
      acc.w = fmaf(w[b], y[b].w, acc.w);
    }
  }
  const size_t o = static_cast<size_t>(t) * H + h;
  if (out_bf16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + o) = packed;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + o) = acc;
  }
}

cudaError_t launch_combine(const float* Y, int splits, int rows_cap, int H, const int32_t* inv_pos,
                           const float* topk_w, int T, int k,
                           int k_routed, float w_shared, void* out, int out_bf16,
                           cudaStream_t st, bool pdl) {
  const dim3 grid(T, (H / 4 + 127) / 128);
  return launch_kernel(moe_combine_kernel, grid, dim3(128), 0, st, pdl, Y, splits, rows_cap, H,
                       inv_pos, topk_w, T, k, k_routed, w_shared, out, out_bf16);
}

// ---------------------------------------------------------------- router
// HPC-Ops × SGLang, section "Router GEMM", "a precision-aware BF16
// formulation": the fp32 weight is split into two bf16 parts, the high part
// by plain truncation and the low part from the residual scaled by 256, so
// that W ~= hi + lo/256 and the router GEMM runs as two bf16 GEMMs.
__global__ void moe_router_prepare_kernel(const float* __restrict__ wr, size_t n,
                                          __nv_bfloat16* __restrict__ hi_lo) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float w = wr[i];
    const uint32_t bits = __float_as_uint(w) & 0xFFFF0000u;   // truncation
    const float hi = __uint_as_float(bits);
    const float lo = (w - hi) * 256.0f;                        // exact
    hi_lo[i] = __ushort_as_bfloat16(static_cast<unsigned short>(bits >> 16));
    hi_lo[n + i] = __float2bfloat16_rn(lo);
  }
}

cudaError_t launch_router_prepare(const float* wr, int E, int H, void* hi_lo, cudaStream_t st) {
  const size_t n = static_cast<size_t>(E) * H;
  const int blocks = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  moe_router_prepare_kernel<<<blocks, 256, 0, st>>>(wr, n, static_cast<__nv_bfloat16*>(hi_lo));
  return cudaGetLastError();
}

// One warp per token (router_topk_warp).

__global__ void __launch_bounds__(128)
    moe_router_topk_kernel(const float* __restrict__ P, int splits, int rows_cap, int T, int E,
                           int k, int score_fn, float scale, float* __restrict__ scores,
                           int32_t* __restrict__ ids, float* __restrict__ w) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t < T) router_topk_warp(P, splits, rows_cap, t, E, k, score_fn, scale, scores, ids, w);
}

cudaError_t launch_router_topk(const float* P, int splits, int rows_cap, int T, int E, int k,
                               int score_fn, float scale, float* scores, int32_t* ids, float* w,
                               cudaStream_t st, bool pdl) {
  return launch_kernel(moe_router_topk_kernel, dim3((T + 3) / 4), dim3(128), 0, st, pdl, P, splits,
                       rows_cap, T, E, k, score_fn, scale, scores, ids, w);
}

}  // namespace moe
