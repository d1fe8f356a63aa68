/*
 * moe_oracle.c — plain, slow CPU oracle of the fused MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline / reference legs of bench.py may load this library.  The product
 * path (the CUDA library and its Python binding) never calls it, and this file
 * shares no code, header, table or constant with the CUDA sources.
 *
 * What it computes, and from which passage:
 *   - oracle_align: the routing index of the "routing and index build" step
 *     (HPC-Ops × SGLang, section "MoE", fused pipeline, routing and index
 *     build): assignments a = t*k + j grouped into contiguous per-expert
 *     intervals.  Written as its plain definition (count, pad, prefix, place in
 *     ascending a) — no counting-pass mechanics.
 *   - oracle_e4m3_encode / _decode: the OCP FP8 E4M3 ("e4m3fn") format: bias 7,
 *     3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448.
 *     Encoding rounds to nearest, ties to even, and saturates to +-448.
 *   - oracle_quant_group: the per-token-per-128-channel rule used for FP8
 *     activations (s = amax/448, 1 if amax == 0; q = e4m3(v/s)) in fp32, the
 *     precision the kernel takes the decision in.
 *   - oracle_moe_bf16 / oracle_moe_fp8 / oracle_moe_w8a16: the layer as the conventional unfused
 *     path states it (HPC-Ops × SGLang, section "MoE", paragraph on the
 *     conventional path: route, Gate-Up, activation (+quant), Down, top-k
 *     weighted reduce), per token, in fp64.  FP8 operands are dequantised
 *     exactly (e4m3 value * fp32 scale in fp64); the activation requantisation
 *     decision is taken on the fp32 rounding of the fp64 activation.
 *   - oracle_router_split / oracle_router_scores / oracle_router_topk: the
 *     router of HPC-Ops × SGLang, section "Router GEMM", "a precision-aware
 *     BF16 formulation": hi = bf16 truncation of W, lo = bf16 RNE of
 *     (W - hi) * 256; reference scores in fp64 from the fp32 weights; softmax
 *     or sigmoid, top-k with ties to the lower expert id, renormalised.
 *
 * Pins: every function here is checked by tests/test_oracle_*.py against
 * closed forms, invariants, brute force on tiny inputs and library routines
 * (torch's e4m3 / bf16 casts, numpy's fp64 matmul).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- numbers */

/* bf16 bit pattern -> value (exact: bf16 is the top half of an fp32). */
static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }

/* fp32 -> bf16 bit pattern, round to nearest, ties to even, on the bit
 * pattern: keep the upper 16 bits, add one when the dropped lower 16 bits
 * exceed half, or equal half with an odd kept part.  (Finite inputs.) */
uint16_t oracle_bf16_rne(float v) {
  uint32_t u;
  memcpy(&u, &v, sizeof u);
  uint32_t upper = u >> 16, lower = u & 0xFFFFu;
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return (uint16_t)upper;
}

/* fp32 -> bf16 bit pattern by truncation (drop the lower 16 bits). */
uint16_t oracle_bf16_trunc(float v) {
  uint32_t u;
  memcpy(&u, &v, sizeof u);
  return (uint16_t)(u >> 16);
}

/* E4M3 code -> value.  Exponent field 0: subnormal m * 2^-9.  Otherwise
 * (1 + m/8) * 2^(e-7) = (8 + m) * 2^(e-10).  e = 15, m = 7 is NaN. */
double oracle_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

/* value -> E4M3 code, round to nearest even, saturating at +-448. */
uint8_t oracle_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* 448 = 1.75 * 2^8 */
  if (a < ldexp(1.0, -6)) {
    /* subnormal spacing 2^-9; n = 8 is the smallest normal 2^-6 = code 0x08 */
    double n = nearbyint(a / ldexp(1.0, -9));
    return (uint8_t)(sign | (uint8_t)n);
  }
  int ex;
  frexp(a, &ex);       /* a = f * 2^ex, f in [0.5, 1) */
  int E = ex - 1;      /* a in [2^E, 2^(E+1)), E in [-6, 8] */
  double n = nearbyint(a / ldexp(1.0, E - 3)); /* in [8, 16] */
  if (n >= 16.0) {
    E += 1;
    n = 8.0;
  }
  /* a < 448 keeps (E, n) at or below (8, 14): never the NaN pattern */
  return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | ((int)n - 8)));
}

/* Array forms of the four conversions above (element by element). */
void oracle_e4m3_encode_n(const float* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}
void oracle_e4m3_decode_n(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}
void oracle_bf16_rne_n(const float* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne(v[i]);
}
void oracle_bf16_trunc_n(const float* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_trunc(v[i]);
}

/* Quantise n values with one scale: s = amax/448 (1 when amax is 0), q[i] =
 * e4m3(v[i] / s).  All arithmetic in fp32 (the kernel's precision). */
void oracle_quant_group(const float* v, int n, uint8_t* q, float* scale) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > amax) amax = a;
  }
  float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
  for (int i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(v[i] / s);
  *scale = s;
}

/* x bf16 [T][H] -> xq e4m3 [T][H], xs fp32 [T][H/128] (per token, per 128
 * channels).  H % 128 == 0. */
void oracle_quant_x(int T, int H, const uint16_t* x, uint8_t* xq, float* xs) {
  float buf[128];
  for (int t = 0; t < T; ++t)
    for (int g = 0; g < H / 128; ++g) {
      for (int i = 0; i < 128; ++i)
        buf[i] = (float)bf16_value(x[(size_t)t * H + g * 128 + i]);
      oracle_quant_group(buf, 128, xq + (size_t)t * H + g * 128,
                         xs + (size_t)t * (H / 128) + g);
    }
}

/* ---------------------------------------------------------------- index */

int64_t oracle_tiles_cap(int T, int k, int E, int bm) {
  int64_t tk = (int64_t)T * k;
  return (tk + bm - 1) / bm + (E < tk ? E : tk);
}

/* The routing index.  Returns the number of invalid ids (dropped).
 * Output sizes: counts[E], offsets[E+1], sorted_ids[tiles_cap*bm],
 * tile_expert[tiles_cap], tiles[tiles_cap*4], inv_pos[T*k], num_tiles[1]. */
int oracle_align(const int32_t* ids, int T, int k, int E, int bm,
                 int32_t* counts, int32_t* offsets, int32_t* sorted_ids,
                 int32_t* tile_expert, int32_t* tiles, int32_t* inv_pos,
                 int32_t* num_tiles) {
  int64_t tk = (int64_t)T * k;
  int64_t tiles_cap = oracle_tiles_cap(T, k, E, bm);
  int64_t rows_cap = tiles_cap * bm;
  int invalid = 0;

  /* 1. count assignments per expert */
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < tk; ++a) {
    int e = ids[a];
    if (e >= 0 && e < E)
      counts[e] += 1;
    else
      invalid += 1;
  }
  /* 2. pad each count up to a multiple of bm; exclusive prefix */
  offsets[0] = 0;
  for (int e = 0; e < E; ++e)
    offsets[e + 1] = offsets[e] + ((counts[e] + bm - 1) / bm) * bm;
  /* 3. every row starts as the sentinel Tk */
  for (int64_t p = 0; p < rows_cap; ++p) sorted_ids[p] = (int32_t)tk;
  /* 4. place assignments in ascending a inside their expert's interval */
  int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
  for (int e = 0; e < E; ++e) cursor[e] = offsets[e];
  for (int64_t a = 0; a < tk; ++a) {
    int e = ids[a];
    if (e >= 0 && e < E) {
      sorted_ids[cursor[e]] = (int32_t)a;
      inv_pos[a] = cursor[e];
      cursor[e] += 1;
    } else {
      inv_pos[a] = -1;
    }
  }
  free(cursor);
  /* 5. task map: one entry per row tile */
  int32_t nt = offsets[E] / bm;
  *num_tiles = nt;
  for (int64_t q = 0; q < tiles_cap; ++q) {
    int32_t row0 = (int32_t)(q * bm);
    if (q < nt) {
      int e = 0;
      while (!(offsets[e] <= row0 && row0 < offsets[e + 1])) ++e;
      int32_t valid = offsets[e] + counts[e] - row0;
      if (valid > bm) valid = bm;
      tile_expert[q] = e;
      tiles[4 * q + 0] = e;
      tiles[4 * q + 1] = row0;
      tiles[4 * q + 2] = valid;
      tiles[4 * q + 3] = 0;
    } else {
      tile_expert[q] = -1;
      tiles[4 * q + 0] = -1;
      tiles[4 * q + 1] = row0;
      tiles[4 * q + 2] = 0;
      tiles[4 * q + 3] = 0;
    }
  }
  return invalid;
}

/* ---------------------------------------------------------------- layer */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* BF16 layer, fp64 arithmetic, for the n_sel tokens listed in sel[].
 * x bf16 [T][H]; w13 bf16 [E][2I][H]; w2 bf16 [E][H][I]; ids int32 [T][k];
 * w fp32 [T][k]; out fp64 [n_sel][H]. */
void oracle_moe_bf16(int T, int H, int I, int E, int k, const uint16_t* x,
                     const uint16_t* w13, const uint16_t* w2,
                     const int32_t* ids, const float* w, const int32_t* sel,
                     int n_sel, double* out) {
  (void)T;
  double* xt = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  double* act = (double*)malloc(sizeof(double) * (size_t)I);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int si = 0; si < n_sel; ++si) {
    int t = sel[si];
    double* o = out + (size_t)si * H;
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    for (int h = 0; h < H; ++h) xt[h] = bf16_value(x[(size_t)t * H + h]);
    for (int j = 0; j < k; ++j) {
      int e = ids[(size_t)t * k + j];
      if (e < 0 || e >= E) continue; /* dropped assignment contributes 0 */
      const uint16_t* wg = w13 + (size_t)e * 2 * I * H;
      const uint16_t* wu = wg + (size_t)I * H;
      const uint16_t* wd = w2 + (size_t)e * H * I;
#pragma omp parallel for schedule(static)
      for (int i = 0; i < I; ++i) {
        double sg = 0.0, su = 0.0;
        for (int h = 0; h < H; ++h) {
          sg += xt[h] * bf16_value(wg[(size_t)i * H + h]);
          su += xt[h] * bf16_value(wu[(size_t)i * H + h]);
        }
        g[i] = sg;
        u[i] = su;
      }
      for (int i = 0; i < I; ++i) act[i] = silu(g[i]) * u[i];
#pragma omp parallel for schedule(static)
      for (int h = 0; h < H; ++h) {
        double s = 0.0;
        for (int i = 0; i < I; ++i) s += act[i] * bf16_value(wd[(size_t)h * I + i]);
        y[h] = s;
      }
      double wj = (double)w[(size_t)t * k + j];
      for (int h = 0; h < H; ++h) o[h] += wj * y[h];
    }
  }
  free(xt);
  free(g);
  free(u);
  free(act);
  free(y);
}

/* FP8 w8a8 layer.  xq e4m3 [T][H] with xs [T][H/128] (from oracle_quant_x);
 * w13q e4m3 [E][2I][H] with w13s [E][2I/128][H/128]; w2q e4m3 [E][H][I] with
 * w2s [E][H/128][I/128].  The activation is requantised per 128 channels with
 * oracle_quant_group on its fp32 rounding, then dequantised exactly.
 * If act_q / act_s are non-NULL they receive, per selected token and slot j,
 * the activation codes [n_sel][k][I] and scales [n_sel][k][I/128]. */
/* w8a16 layer (the HPC-Ops MoE precision, operator table: "BF16 hidden
 * states; FP8 E4M3 expert weights"): bf16 x as is, weights e4m3 with one fp32
 * scale per 128x128 block dequantised exactly (e4m3_value(q) * scale, in
 * fp64); the activation is not quantised.  Same step order and conventions
 * as oracle_moe_bf16. */
void oracle_moe_w8a16(int T, int H, int I, int E, int k, const uint16_t* x,
                      const uint8_t* w13q, const float* w13s, const uint8_t* w2q,
                      const float* w2s, const int32_t* ids, const float* w,
                      const int32_t* sel, int n_sel, double* out) {
  (void)T;
  const int HB = H / 128, IB = I / 128;
  double* xt = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  double* act = (double*)malloc(sizeof(double) * (size_t)I);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int si = 0; si < n_sel; ++si) {
    int t = sel[si];
    double* o = out + (size_t)si * H;
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    for (int h = 0; h < H; ++h) xt[h] = bf16_value(x[(size_t)t * H + h]);
    for (int j = 0; j < k; ++j) {
      int e = ids[(size_t)t * k + j];
      if (e < 0 || e >= E) continue; /* dropped assignment contributes 0 */
      const uint8_t* q13 = w13q + (size_t)e * 2 * I * H;
      const float* s13 = w13s + (size_t)e * (2 * I / 128) * HB;
      const uint8_t* q2 = w2q + (size_t)e * H * I;
      const float* s2 = w2s + (size_t)e * (H / 128) * IB;
#pragma omp parallel for schedule(static)
      for (int i = 0; i < I; ++i) {
        double sg = 0.0, su = 0.0;
        const int ru = I + i;   /* up row */
        for (int h = 0; h < H; ++h) {
          const double wg = oracle_e4m3_decode(q13[(size_t)i * H + h]) *
                            (double)s13[(size_t)(i / 128) * HB + h / 128];
          const double wu = oracle_e4m3_decode(q13[(size_t)ru * H + h]) *
                            (double)s13[(size_t)(ru / 128) * HB + h / 128];
          sg += xt[h] * wg;
          su += xt[h] * wu;
        }
        g[i] = sg;
        u[i] = su;
      }
      for (int i = 0; i < I; ++i) act[i] = silu(g[i]) * u[i];
#pragma omp parallel for schedule(static)
      for (int h = 0; h < H; ++h) {
        double s = 0.0;
        for (int i = 0; i < I; ++i)
          s += act[i] * oracle_e4m3_decode(q2[(size_t)h * I + i]) *
               (double)s2[(size_t)(h / 128) * IB + i / 128];
        y[h] = s;
      }
      double wj = (double)w[(size_t)t * k + j];
      for (int h = 0; h < H; ++h) o[h] += wj * y[h];
    }
  }
  free(xt);
  free(g);
  free(u);
  free(act);
  free(y);
}

void oracle_moe_fp8(int T, int H, int I, int E, int k, const uint8_t* xq,
                    const float* xs, const uint8_t* w13q, const float* w13s,
                    const uint8_t* w2q, const float* w2s, const int32_t* ids,
                    const float* w, const int32_t* sel, int n_sel, double* out,
                    uint8_t* act_q, float* act_s) {
  (void)T;
  const int HB = H / 128, IB = I / 128;
  double* xt = (double*)malloc(sizeof(double) * (size_t)H);
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  float* a32 = (float*)malloc(sizeof(float) * (size_t)I);
  uint8_t* aq = (uint8_t*)malloc((size_t)I);
  float* as = (float*)malloc(sizeof(float) * (size_t)(IB > 0 ? IB : 1));
  double* ad = (double*)malloc(sizeof(double) * (size_t)I);
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int si = 0; si < n_sel; ++si) {
    int t = sel[si];
    double* o = out + (size_t)si * H;
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    for (int h = 0; h < H; ++h)
      xt[h] = oracle_e4m3_decode(xq[(size_t)t * H + h]) * (double)xs[(size_t)t * HB + h / 128];
    for (int j = 0; j < k; ++j) {
      int e = ids[(size_t)t * k + j];
      if (e < 0 || e >= E) continue;
      const uint8_t* wg = w13q + (size_t)e * 2 * I * H;
      const uint8_t* wu = wg + (size_t)I * H;
      const float* sg_ = w13s + (size_t)e * (2 * I / 128) * HB;
      const uint8_t* wd = w2q + (size_t)e * H * I;
      const float* sd_ = w2s + (size_t)e * HB * IB;
#pragma omp parallel for schedule(static)
      for (int i = 0; i < I; ++i) {
        double accg = 0.0, accu = 0.0;
        for (int h = 0; h < H; ++h) {
          double wgv = oracle_e4m3_decode(wg[(size_t)i * H + h]) *
                       (double)sg_[(size_t)(i / 128) * HB + h / 128];
          double wuv = oracle_e4m3_decode(wu[(size_t)i * H + h]) *
                       (double)sg_[(size_t)((I + i) / 128) * HB + h / 128];
          accg += xt[h] * wgv;
          accu += xt[h] * wuv;
        }
        g[i] = accg;
        u[i] = accu;
      }
      for (int i = 0; i < I; ++i) a32[i] = (float)(silu(g[i]) * u[i]);
      for (int b = 0; b < IB; ++b) oracle_quant_group(a32 + b * 128, 128, aq + b * 128, as + b);
      for (int i = 0; i < I; ++i) ad[i] = oracle_e4m3_decode(aq[i]) * (double)as[i / 128];
      if (act_q) memcpy(act_q + ((size_t)si * k + j) * I, aq, (size_t)I);
      if (act_s) memcpy(act_s + ((size_t)si * k + j) * IB, as, sizeof(float) * (size_t)IB);
#pragma omp parallel for schedule(static)
      for (int h = 0; h < H; ++h) {
        double s = 0.0;
        for (int i = 0; i < I; ++i)
          s += ad[i] * oracle_e4m3_decode(wd[(size_t)h * I + i]) *
               (double)sd_[(size_t)(h / 128) * IB + i / 128];
        y[h] = s;
      }
      double wj = (double)w[(size_t)t * k + j];
      for (int h = 0; h < H; ++h) o[h] += wj * y[h];
    }
  }
  free(xt);
  free(g);
  free(u);
  free(a32);
  free(aq);
  free(as);
  free(ad);
  free(y);
}

/* ---------------------------------------------------------------- router */

/* hi = bf16 truncation of W, lo = bf16 RNE of (W - hi) * 256.  W - hi is the
 * dropped low mantissa part of W, exact in fp32; the *256 is exact too. */
void oracle_router_split(const float* wr, int64_t n, uint16_t* hi, uint16_t* lo) {
  for (int64_t i = 0; i < n; ++i) {
    uint16_t h = oracle_bf16_trunc(wr[i]);
    float hv = (float)bf16_value(h);
    float r = (wr[i] - hv) * 256.0f;
    hi[i] = h;
    lo[i] = oracle_bf16_rne(r);
  }
}

/* Reference router scores in fp64 from bf16 x [T][H] and the fp32 weights
 * wr [E][H]: scores[t][e] = sum_h x[t][h] * wr[e][h]. */
void oracle_router_scores(int T, int H, int E, const uint16_t* x,
                          const float* wr, double* scores) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double s = 0.0;
      for (int h = 0; h < H; ++h)
        s += bf16_value(x[(size_t)t * H + h]) * (double)wr[(size_t)e * H + h];
      scores[(size_t)t * E + e] = s;
    }
}

/* Top-k over the scores of each token (largest first, ties to the lower id);
 * p = softmax over all E (score_fn 0) or sigmoid (score_fn 1);
 * w_j = scale * p_j / sum of p over the selected ids. */
void oracle_router_topk(int T, int E, int k, const double* scores,
                        int score_fn, double scale, int32_t* ids, double* w) {
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  char* taken = (char*)malloc((size_t)E);
  for (int t = 0; t < T; ++t) {
    const double* s = scores + (size_t)t * E;
    if (score_fn == 0) {
      double m = s[0];
      for (int e = 1; e < E; ++e)
        if (s[e] > m) m = s[e];
      double z = 0.0;
      for (int e = 0; e < E; ++e) {
        p[e] = exp(s[e] - m);
        z += p[e];
      }
      for (int e = 0; e < E; ++e) p[e] /= z;
    } else {
      for (int e = 0; e < E; ++e) p[e] = 1.0 / (1.0 + exp(-s[e]));
    }
    memset(taken, 0, (size_t)E);
    double psum = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || s[e] > s[best])) best = e;
      taken[best] = 1;
      ids[(size_t)t * k + j] = best;
      psum += p[best];
    }
    for (int j = 0; j < k; ++j)
      w[(size_t)t * k + j] = scale * p[ids[(size_t)t * k + j]] / psum;
  }
  free(p);
  free(taken);
}
