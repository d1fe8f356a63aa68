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
// FP8 with no splits: the unsplit token-major Gate-Up stored a itself
// (G = [rows_cap][I], the same silu_mul_fast), so only the quantisation runs.
// SiLU with the fast exponential and division intrinsics (relative error
// ~1e-6, far below the bf16 rounding of a bf16 result and the e4m3 step of
// an FP8 one), as in the GEMM epilogues: with expf and an IEEE division the
// kernel was compute-bound (DeepSeek-shaped T=4096: 165 us for 670 MB of
// traffic).

constexpr int kActThreads = 256;

// Each block iteration takes R = max(1, 256 / (I/8)) index rows; thread t
// owns channels 8c..8c+7 of row t / (I/8), c = t % (I/8) (more chunks than
// threads: c = t, t + 256, ...), and loads its eight gate and eight up
// values of every split as four 16-byte loads.  Padding rows are skipped
// with one load.  In FP8 mode a half-warp covers one 128-channel group of
// one row (I % 128 == 0, so 16 aligned lanes share row and group).
template <int FP8>
__global__ void __launch_bounds__(kActThreads, 4)
    moe_act_kernel(const float* __restrict__ G, int splits, int rows_cap, int I,
                   const int32_t* __restrict__ sorted_ids, int sentinel, void* __restrict__ A,
                   float* __restrict__ As) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t two_i = 2 * static_cast<size_t>(I);
  const size_t slice = static_cast<size_t>(rows_cap) * two_i;
  const int chunks = I / 8;
  const bool wide = chunks >= kActThreads;
  const int rows_per = wide ? 1 : kActThreads / chunks;
  const int my_row = wide ? 0 : threadIdx.x / chunks;
  const int c_first = wide ? threadIdx.x : threadIdx.x % chunks;
  const int c_step = wide ? kActThreads : chunks;
  const int lane = threadIdx.x & 31;
  const uint32_t half_mask = lane < 16 ? 0x0000ffffu : 0xffff0000u;
  if (my_row >= rows_per) return;   // threads past rows_per whole rows
  // The next row's sorted id is loaded while this row is processed, so an
  // iteration waits on one load latency (the row's), not two.
  const int stride = gridDim.x * rows_per;
  int p = blockIdx.x * rows_per + my_row;
  int sid = p < rows_cap ? __ldg(sorted_ids + p) : sentinel;
  for (; p < rows_cap; p += stride) {
    const int sid_next = p + stride < rows_cap ? __ldg(sorted_ids + p + stride) : sentinel;
    const bool padding = sid >= sentinel;
    sid = sid_next;
    if (padding) continue;
    const float* row = G + static_cast<size_t>(p) * (splits ? two_i : static_cast<size_t>(I));
    for (int c = c_first; c < chunks; c += c_step) {
      const int i = 8 * c;
      float v[8];
      if (FP8 && splits == 0) {   // SiLU(gate)*up stored by the Gate-Up epilogue
        const float4 a0 = __ldg(reinterpret_cast<const float4*>(row + i));
        const float4 a1 = __ldg(reinterpret_cast<const float4*>(row + i + 4));
        v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
        v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
      } else {
        float g[8], u[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = u[j] = 0.f;
#pragma unroll 4
        for (int sp = 0; sp < splits; ++sp) {
          const float* r = row + sp * slice + i;
          const float4 g0 = __ldg(reinterpret_cast<const float4*>(r));
          const float4 g1 = __ldg(reinterpret_cast<const float4*>(r + 4));
          const float4 u0 = __ldg(reinterpret_cast<const float4*>(r + I));
          const float4 u1 = __ldg(reinterpret_cast<const float4*>(r + I + 4));
          g[0] += g0.x; g[1] += g0.y; g[2] += g0.z; g[3] += g0.w;
          g[4] += g1.x; g[5] += g1.y; g[6] += g1.z; g[7] += g1.w;
          u[0] += u0.x; u[1] += u0.y; u[2] += u0.z; u[3] += u0.w;
          u[4] += u1.x; u[5] += u1.y; u[6] += u1.z; u[7] += u1.w;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = silu_mul_fast(g[j], u[j]);
      }
      if (FP8) {
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
#pragma unroll
        for (int d = 8; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(half_mask, amax, d));
        const float sc = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
        uint32_t q[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint16_t lo = cvt_e4m3x2(__fdiv_rn(v[4 * h + 1], sc), __fdiv_rn(v[4 * h], sc));
          const uint16_t hi = cvt_e4m3x2(__fdiv_rn(v[4 * h + 3], sc), __fdiv_rn(v[4 * h + 2], sc));
          q[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        uint8_t* Aq = static_cast<uint8_t*>(A);
        *reinterpret_cast<uint2*>(Aq + static_cast<size_t>(p) * I + i) = make_uint2(q[0], q[1]);
        if ((lane & 15) == 0) As[static_cast<size_t>(p) * (I / 128) + i / 128] = sc;
      } else {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * h], v[2 * h + 1]);
          w[h] = *reinterpret_cast<uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(A) + static_cast<size_t>(p) * I + i) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

cudaError_t launch_act(int fp8, const float* G, int splits, int rows_cap, int I,
                       const int32_t* sorted_ids, int sentinel, void* A, float* As,
                       cudaStream_t st, bool pdl) {
  // Up to eight resident blocks of 256 threads per SM walk all index rows:
  // one block per (row, column chunk) spent most of the stage scheduling
  // blocks of padding.
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int chunks = I / 8;
  const int rows_per = chunks >= kActThreads ? 1 : kActThreads / chunks;
  const int want = (rows_cap + rows_per - 1) / rows_per;
  const int grid = want < 8 * sms ? want : 8 * sms;
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
// kCols output columns per thread (one or two 16-byte loads a row) and kBatch
// assignments whose rows are loaded together: wide (8, 4) where the blocks
// fill the GPU, narrow (4, 8) for few tokens, where more, shorter blocks
// and all of a token's rows in flight at once cut the latency.
constexpr int kCombineThreads = 256;

// Four consecutive values of Y (fp32 partials, or bf16 rows of an unsplit
// Down GEMM) as a float4.
__device__ __forceinline__ float4 load_y4(const float* Y, size_t off) {
  return __ldg(reinterpret_cast<const float4*>(Y + off));
}
__device__ __forceinline__ float4 load_y4(const __nv_bfloat16* Y, size_t off) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(Y + off));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <int kCols, int kBatch, typename TY>
__global__ void __launch_bounds__(kCombineThreads)
    moe_combine_kernel(const TY* __restrict__ Y, int splits, int rows_cap, int H,
                       const int32_t* __restrict__ inv_pos, const float* __restrict__ topk_w,
                       int T, int k, int k_routed, float w_shared, void* __restrict__ out,
                       int out_bf16) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  constexpr int kQ = kCols / 4;
  const int h = (blockIdx.y * kCombineThreads + threadIdx.x) * kCols;
  if (h >= H) return;
  const size_t slice = static_cast<size_t>(rows_cap) * H;
  // H % 4 == 0: the second four columns exist unless this is a 4-column tail
  const bool q1 = kQ > 1 && h + 4 < H;
  float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  for (int j0 = 0; j0 < k; j0 += kBatch) {
    // Issue every row load of the batch before reducing: the reduction order
    // (splits ascending, then j ascending) is unchanged.
    int pos[kBatch];
    float w[kBatch];
    float4 y[kBatch][kQ];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int j = j0 + b;
      pos[b] = j < k ? __ldg(inv_pos + static_cast<size_t>(t) * k + j) : -1;
      if (pos[b] >= rows_cap) pos[b] = -1;   // only rows of the index are read
      // routed slots weigh topk_w[t][j]; the shared experts' slots w_shared
      w[b] = j < k_routed ? __ldg(topk_w + static_cast<size_t>(t) * k_routed + j)
                          : (j < k ? w_shared : 0.f);
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
#pragma unroll
      for (int q = 0; q < kQ; ++q)
        y[b][q] = (pos[b] >= 0 && (q == 0 || q1))
                      ? load_y4(Y, static_cast<size_t>(pos[b]) * H + h + 4 * q)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
    for (int s = 1; s < splits; ++s) {
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (pos[b] < 0) continue;
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
          if (q == 1 && !q1) continue;
          const float4 ys = load_y4(Y, s * slice + static_cast<size_t>(pos[b]) * H + h + 4 * q);
          y[b][q].x += ys.x; y[b][q].y += ys.y; y[b][q].z += ys.z; y[b][q].w += ys.w;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (pos[b] < 0) continue;   // dropped assignment contributes 0
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        acc[q].x = fmaf(w[b], y[b][q].x, acc[q].x);
        acc[q].y = fmaf(w[b], y[b][q].y, acc[q].y);
        acc[q].z = fmaf(w[b], y[b][q].z, acc[q].z);
        acc[q].w = fmaf(w[b], y[b][q].w, acc[q].w);
      }
    }
  }
  // 8-byte (bf16) or 16-byte (fp32) stores per four columns: t * H is only a
  // multiple of 4
  const size_t o = static_cast<size_t>(t) * H + h;
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
    if (q == 1 && !q1) break;
    if (out_bf16) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc[q].x, acc[q].y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc[q].z, acc[q].w);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + o + 4 * q) =
          make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + o + 4 * q) = acc[q];
    }
  }
}

// Unsplit Down GEMM (bf16 rows, one per assignment): a thread takes eight
// columns, one 16-byte load per row, and has all of a token's (up to eight)
// rows in flight as raw bf16 before reducing them in j order — one index
// load and one row load latency per token instead of two each for batches of
// four (the fp32 kernel converts rows on load and keeps float4s, twice the
// registers per row).
constexpr int kCombineRows = 8;
__global__ void __launch_bounds__(kCombineThreads)
    moe_combine_rows_kernel(const __nv_bfloat16* __restrict__ Y, int rows_cap, int H,
                            const int32_t* __restrict__ inv_pos, const float* __restrict__ topk_w,
                            int T, int k, int k_routed, float w_shared, void* __restrict__ out,
                            int out_bf16) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x;
  const int h = (blockIdx.y * kCombineThreads + threadIdx.x) * 8;
  if (h >= H) return;   // H % 8 == 0
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < k; j0 += kCombineRows) {
    int pos[kCombineRows];
    float w[kCombineRows];
    uint4 raw[kCombineRows];
#pragma unroll
    for (int b = 0; b < kCombineRows; ++b) {
      const int j = j0 + b;
      pos[b] = j < k ? __ldg(inv_pos + static_cast<size_t>(t) * k + j) : -1;
      if (pos[b] >= rows_cap) pos[b] = -1;   // only rows of the index are read
      w[b] = j < k_routed ? __ldg(topk_w + static_cast<size_t>(t) * k_routed + j)
                          : (j < k ? w_shared : 0.f);
    }
#pragma unroll
    for (int b = 0; b < kCombineRows; ++b)
      raw[b] = pos[b] >= 0
                   ? __ldg(reinterpret_cast<const uint4*>(Y + static_cast<size_t>(pos[b]) * H + h))
                   : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int b = 0; b < kCombineRows; ++b) {
      if (pos[b] < 0) continue;   // dropped assignment contributes 0
      const uint32_t u[4] = {raw[b].x, raw[b].y, raw[b].z, raw[b].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
        acc[2 * i] = fmaf(w[b], f.x, acc[2 * i]);
        acc[2 * i + 1] = fmaf(w[b], f.y, acc[2 * i + 1]);
      }
    }
  }
  const size_t o = static_cast<size_t>(t) * H + h;   // a multiple of 8
  if (out_bf16) {
    uint32_t pk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + o) =
        make_uint4(pk[0], pk[1], pk[2], pk[3]);
  } else {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
    d[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    d[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

template <typename TY>
cudaError_t launch_combine_t(const TY* Y, int splits, int rows_cap, int H,
                             const int32_t* inv_pos, const float* topk_w, int T, int k,
                             int k_routed, float w_shared, void* out, int out_bf16,
                             cudaStream_t st, bool pdl) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int wide_blocks = T * ((H + 8 * kCombineThreads - 1) / (8 * kCombineThreads));
  if (wide_blocks >= 4 * sms) {
    const dim3 grid(T, (H + 8 * kCombineThreads - 1) / (8 * kCombineThreads));
    return launch_kernel(moe_combine_kernel<8, 4, TY>, grid, dim3(kCombineThreads), 0, st, pdl,
                         Y, splits, rows_cap, H, inv_pos, topk_w, T, k, k_routed, w_shared, out,
                         out_bf16);
  }
  const dim3 grid(T, (H + 4 * kCombineThreads - 1) / (4 * kCombineThreads));
  return launch_kernel(moe_combine_kernel<4, 8, TY>, grid, dim3(kCombineThreads), 0, st, pdl, Y,
                       splits, rows_cap, H, inv_pos, topk_w, T, k, k_routed, w_shared, out,
                       out_bf16);
}

cudaError_t launch_combine(const void* Y, int y_bf16, int splits, int rows_cap, int H,
                           const int32_t* inv_pos, const float* topk_w, int T, int k,
                           int k_routed, float w_shared, void* out, int out_bf16,
                           cudaStream_t st, bool pdl) {
  if (y_bf16) {
    const dim3 grid(T, (H + 8 * kCombineThreads - 1) / (8 * kCombineThreads));
    return launch_kernel(moe_combine_rows_kernel, grid, dim3(kCombineThreads), 0, st, pdl,
                         static_cast<const __nv_bfloat16*>(Y), rows_cap, H, inv_pos, topk_w, T,
                         k, k_routed, w_shared, out, out_bf16);
  }
  return launch_combine_t(static_cast<const float*>(Y), splits, rows_cap, H, inv_pos, topk_w, T,
                          k, k_routed, w_shared, out, out_bf16, st, pdl);
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

// Many split-K partials (few tokens, the router GEMM spread over many CTAs):
// a block of eight warps per token.  Warp g loads the partials of splits
// [g*G, (g+1)*G) (G = ceil(splits / 8) <= 4) all at once and sums them in
// split order; warp 0 adds the eight group sums in group order, then selects.
// (One warp looping over 32 splits would wait for eight L2 round trips.)
constexpr int kTopkGroups = 8;
template <int kPer>
__global__ void __launch_bounds__(32 * kTopkGroups)
    moe_router_topk_block_kernel(const float* __restrict__ P, int splits, int rows_cap, int T,
                                 int E, int k, int score_fn, float scale,
                                 float* __restrict__ scores, int32_t* __restrict__ ids,
                                 float* __restrict__ w) {
  __shared__ float part[kTopkGroups][2][32 * kPer];
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x, g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t slice = static_cast<size_t>(rows_cap) * 2 * E;
  const float* row = P + static_cast<size_t>(t) * 2 * E;
  const int G = (splits + kTopkGroups - 1) / kTopkGroups;
  float ph[kRouterMaxSplits][kPer], pl[kRouterMaxSplits][kPer];
#pragma unroll
  for (int j = 0; j < kRouterMaxSplits; ++j)
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int sp = g * G + j, e = lane + 32 * i;
      const bool in = j < G && sp < splits && e < E;
      ph[j][i] = in ? __ldg(row + sp * slice + e) : 0.f;
      pl[j][i] = in ? __ldg(row + sp * slice + E + e) : 0.f;
    }
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    float hi = ph[0][i], lo = pl[0][i];
#pragma unroll
    for (int j = 1; j < kRouterMaxSplits; ++j) {
      hi += ph[j][i];
      lo += pl[j][i];
    }
    part[g][0][lane + 32 * i] = hi;
    part[g][1][lane + 32 * i] = lo;
  }
  __syncthreads();
  if (g != 0) return;
  float s[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    if (e < E) {
      float hi = part[0][0][e], lo = part[0][1][e];
#pragma unroll
      for (int q = 1; q < kTopkGroups; ++q) {
        hi += part[q][0][e];
        lo += part[q][1][e];
      }
      v = hi + lo * (1.0f / 256.0f);
      scores[static_cast<size_t>(t) * E + e] = v;
    }
    s[i] = v;
  }
  router_select_warp<kPer>(s, t, E, k, score_fn, scale, ids, w, nullptr);
}

cudaError_t launch_router_topk(const float* P, int splits, int rows_cap, int T, int E, int k,
                               int score_fn, float scale, float* scores, int32_t* ids, float* w,
                               cudaStream_t st, bool pdl) {
  if (splits > kRouterMaxSplits) {
    if (splits > kRouterMaxSplits * kTopkGroups) return cudaErrorInvalidValue;
    if (E <= 128)
      return launch_kernel(moe_router_topk_block_kernel<4>, dim3(T), dim3(32 * kTopkGroups), 0,
                           st, pdl, P, splits, rows_cap, T, E, k, score_fn, scale, scores, ids,
                           w);
    if (E <= 256)
      return launch_kernel(moe_router_topk_block_kernel<8>, dim3(T), dim3(32 * kTopkGroups), 0,
                           st, pdl, P, splits, rows_cap, T, E, k, score_fn, scale, scores, ids,
                           w);
    return launch_kernel(moe_router_topk_block_kernel<kRouterMaxE / 32>, dim3(T),
                         dim3(32 * kTopkGroups), 0, st, pdl, P, splits, rows_cap, T, E, k,
                         score_fn, scale, scores, ids, w);
  }
  return launch_kernel(moe_router_topk_kernel, dim3((T + 3) / 4), dim3(128), 0, st, pdl, P, splits,
                       rows_cap, T, E, k, score_fn, scale, scores, ids, w);
}

}  // namespace moe
