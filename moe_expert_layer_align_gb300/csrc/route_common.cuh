// route_common.cuh — warp-level routines shared by the stand-alone router /
// quantisation kernels and the fused routing + index kernel.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace moe {

// FP8 rule for one group of 128 channels held 4 per lane by a warp:
// s = amax/448 (1 when amax is 0); q = e4m3 RNE-satfinite(v / s) (IEEE fp32
// division).  Returns the 4 codes packed little-endian; writes s via *scale.
__device__ __forceinline__ uint32_t quant_group4(const float (&v)[4], float* scale) {
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
  const float s = (amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f);
  *scale = s;
  const uint16_t lo = cvt_e4m3x2(__fdiv_rn(v[1], s), __fdiv_rn(v[0], s));
  const uint16_t hi = cvt_e4m3x2(__fdiv_rn(v[3], s), __fdiv_rn(v[2], s));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// x quantisation of token t, group g of 128 channels, by one warp: codes to
// xq[t][g*128..], the scale to xs[t][g].  Returns the scale.
__device__ __forceinline__ float quant_x_group_warp(const __nv_bfloat16* __restrict__ x, int t,
                                                    int g, int H, uint8_t* __restrict__ xq,
                                                    float* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  const size_t base = static_cast<size_t>(t) * H + g * 128 + lane * 4;
  const uint2 raw = *reinterpret_cast<const uint2*>(x + base);
  const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
  const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
  float v[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
  float s;
  const uint32_t q = quant_group4(v, &s);
  *reinterpret_cast<uint32_t*>(xq + base) = q;
  if (lane == 0) xs[static_cast<size_t>(t) * (H / 128) + g] = s;
  return s;
}

// x quantisation of up to four (token, group) items by one warp, every row
// load issued before the first is used (items with t < 0 are skipped).
__device__ __forceinline__ void quant_x_groups4_warp(const __nv_bfloat16* __restrict__ x,
                                                     const int (&t)[4], const int (&g)[4],
                                                     int H, uint8_t* __restrict__ xq,
                                                     float* __restrict__ xs) {
  const int lane = threadIdx.x & 31;
  uint2 raw[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    raw[j] = t[j] >= 0 ? *reinterpret_cast<const uint2*>(
                             x + static_cast<size_t>(t[j]) * H + g[j] * 128 + lane * 4)
                       : make_uint2(0u, 0u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (t[j] < 0) continue;
    const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw[j].x);
    const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw[j].y);
    float v[4] = {__low2float(p0), __high2float(p0), __low2float(p1), __high2float(p1)};
    float s;
    const uint32_t q = quant_group4(v, &s);
    const size_t base = static_cast<size_t>(t[j]) * H + g[j] * 128 + lane * 4;
    *reinterpret_cast<uint32_t*>(xq + base) = q;
    if (lane == 0) xs[static_cast<size_t>(t[j]) * (H / 128) + g[j]] = s;
  }
}

// Router scores and top-k of token t by one warp (HPC-Ops × SGLang, section
// "Router GEMM"): the split-K partials of the two GEMMs (P[s][t][0..E) = x.hi,
// P[s][t][E..2E) = x.lo) give score = acc_hi + acc_lo/256; softmax (or
// sigmoid); k rounds of warp arg-max over the raw scores (ties to the lower
// id); weights renormalised over the selected ids, times `scale`.
constexpr int kRouterMaxE = 512;
constexpr int kRouterMaxSplits = 4;   // router GEMM split-K partials per score

// Softmax (or sigmoid) and top-k of token t from its raw scores, lane l
// holding experts l + 32 i in s[i] (-inf beyond E); one warp.
template <int kPer>
__device__ __forceinline__ void router_select_warp(float (&s)[kPer], int t, int E, int k,
                                                   int score_fn, float scale,
                                                   int32_t* __restrict__ ids,
                                                   float* __restrict__ w, int32_t* ids_out);

// kPer score slots per lane (E <= 32 * kPer).  kL2: the partials were written
// by other CTAs of the same grid, so they are read through L2 (ld.global.cg)
// rather than the non-coherent path.  ids_out (nullable): the selected ids
// are also written there, ids_out[j] for j < k.
template <int kPer, bool kL2>
__device__ __forceinline__ void router_topk_warp_t(const float* __restrict__ P, int splits,
                                                   int rows_cap, int t, int E, int k,
                                                   int score_fn, float scale,
                                                   float* __restrict__ scores,
                                                   int32_t* __restrict__ ids,
                                                   float* __restrict__ w, int32_t* ids_out) {
  const int lane = threadIdx.x & 31;
  auto ld = [](const float* a) { return kL2 ? __ldcg(a) : __ldg(a); };
  float s[kPer];
  const size_t slice = static_cast<size_t>(rows_cap) * 2 * E;
  const int per = (E + 31) / 32;   // slots this warp really uses
  const float* row = P + static_cast<size_t>(t) * 2 * E;
  if (kPer <= 8 && splits <= kRouterMaxSplits) {
    // every partial of this lane's slots is loaded before any is summed (one
    // L2 round trip, not one per slot and split); sums run in split order
    float ph[kRouterMaxSplits][kPer], pl[kRouterMaxSplits][kPer];
#pragma unroll
    for (int sp = 0; sp < kRouterMaxSplits; ++sp)
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        const bool in = sp < splits && i < per && e < E;
        ph[sp][i] = in ? ld(row + sp * slice + e) : 0.f;
        pl[sp][i] = in ? ld(row + sp * slice + E + e) : 0.f;
      }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      float v = -INFINITY;
      if (i < per && e < E) {
        float hi = ph[0][i], lo = pl[0][i];
#pragma unroll
        for (int sp = 1; sp < kRouterMaxSplits; ++sp)
          if (sp < splits) {
            hi += ph[sp][i];
            lo += pl[sp][i];
          }
        v = hi + lo * (1.0f / 256.0f);
        scores[static_cast<size_t>(t) * E + e] = v;
      }
      s[i] = v;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      float v = -INFINITY;
      if (i < per && e < E) {
        float hi = ld(row + e), lo = ld(row + E + e);
#pragma unroll 4
        for (int sp = 1; sp < splits; ++sp) {
          hi += ld(row + sp * slice + e);
          lo += ld(row + sp * slice + E + e);
        }
        v = hi + lo * (1.0f / 256.0f);
        scores[static_cast<size_t>(t) * E + e] = v;
      }
      s[i] = v;
    }
  }
  router_select_warp<kPer>(s, t, E, k, score_fn, scale, ids, w, ids_out);
}

template <int kPer>
__device__ __forceinline__ void router_select_warp(float (&s)[kPer], int t, int E, int k,
                                                   int score_fn, float scale,
                                                   int32_t* __restrict__ ids,
                                                   float* __restrict__ w, int32_t* ids_out) {
  const int lane = threadIdx.x & 31;
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) mx = fmaxf(mx, s[i]);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
  float prob[kPer];
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane + 32 * i;
    float pv = 0.f;
    if (e < E) pv = score_fn == 0 ? expf(s[i] - mx) : 1.0f / (1.0f + expf(-s[i]));
    prob[i] = pv;
    z += pv;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) z += __shfl_xor_sync(0xffffffffu, z, d);
  float psel = 0.f, my_p = 0.f;
  int my_id = -1;
  for (int j = 0; j < k; ++j) {
    // this lane's best (first of equal values: e ascends with i) ...
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = lane + 32 * i;
      if (e < E && s[i] > bv) {
        bv = s[i];
        bi = e;
      }
    }
    // ... then the warp's: the largest value (as an order-preserving
    // unsigned key; -0 counts as +0, as in a float compare), and among the
    // lanes holding it the lowest id
    const uint32_t bits = __float_as_uint(bv == 0.f ? 0.f : bv);
    const uint32_t key = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    bi = static_cast<int>(
        __reduce_min_sync(0xffffffffu, key == kmax ? static_cast<uint32_t>(bi) : 0xffffffffu));
    // owner lane removes the winner and reports its probability
    float pw = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (lane + 32 * i == bi) {
        pw = score_fn == 0 ? prob[i] / z : prob[i];
        s[i] = -INFINITY;
      }
    const int owner = bi & 31;
    pw = __shfl_sync(0xffffffffu, pw, owner);
    psel += pw;
    if (lane == j) {
      my_id = bi;
      my_p = pw;
    }
  }
  if (lane < k) {
    ids[static_cast<size_t>(t) * k + lane] = my_id;
    if (ids_out != nullptr) ids_out[lane] = my_id;
    w[static_cast<size_t>(t) * k + lane] = scale * (my_p / psel);
  }
}

template <bool kL2 = false>
__device__ __forceinline__ void router_topk_warp(const float* __restrict__ P, int splits,
                                                 int rows_cap, int t, int E, int k, int score_fn,
                                                 float scale, float* __restrict__ scores,
                                                 int32_t* __restrict__ ids,
                                                 float* __restrict__ w,
                                                 int32_t* ids_out = nullptr) {
  if (E <= 128)
    router_topk_warp_t<4, kL2>(P, splits, rows_cap, t, E, k, score_fn, scale, scores, ids, w,
                               ids_out);
  else if (E <= 256)
    router_topk_warp_t<8, kL2>(P, splits, rows_cap, t, E, k, score_fn, scale, scores, ids, w,
                               ids_out);
  else
    router_topk_warp_t<kRouterMaxE / 32, kL2>(P, splits, rows_cap, t, E, k, score_fn, scale,
                                              scores, ids, w, ids_out);
}

}  // namespace moe
