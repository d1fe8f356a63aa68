// k_gemm_w8.cuh — the expert GEMM with FP8 weights and bf16 activations
// (w8a16: HPC-Ops × SGLang, operator table, row MoE: "BF16 hidden states;
// FP8 E4M3 expert weights").
//
// The weights stream from HBM as e4m3 bytes (half the bytes of bf16) with one
// fp32 scale per 128x128 block.  tcgen05's kind::f16 MMA needs both operands
// bf16, so converter warps turn every weight stage into a bf16 tile — e4m3 to
// fp16 (exact), to fp32 (exact), times the block scale, to bf16 (round to
// nearest even) — and the MMA, the epilogue (with the fused SiLU-and-mul) and
// the token operand are those of the bf16 layer.  The converted tile goes to
// tensor memory, as the MMA's A operand (a weight row per TMEM lane, two bf16
// of K per column): a converter thread owns one weight row, reads its e4m3
// bytes from shared memory and writes the row's bf16 values with one
// tcgen05.st.  (Converting into shared memory instead put the bf16 tile's
// write and the MMA's read of it — 64 KB per 16 KB stage — on the shared
// memory the TMA and the gathered token rows also use.)
//
// A stage is one 128-wide K block (one block scale).  Two rings: R raw slots
// (the e4m3 weight stage as two 64-wide halves of 128 rows x 64 bytes, one TMA
// box each with the 64-byte swizzle, so that the 32 rows a converter warp
// reads fall in different banks, plus for the Down GEMM its token rows as two
// 64-wide bf16 sub-tiles) filled by TMA, and C converted slots: 64 TMEM
// columns of A each (plus for the Gate-Up GEMM the gathered token rows as two
// 64-wide sub-tiles in shared memory).  The MMA issues eight instructions per
// stage.  A Gate-Up raw slot is released by the converter warps once they have
// read it; a Down raw slot, whose token rows the MMA reads, when that MMA
// completes; a converted slot likewise.  The raw ring is as deep as shared
// memory allows because in the decode regime the weight stream is what the
// kernel waits on.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "k_gemm.cuh"

namespace moe {

constexpr int kW8RawHalf = kTileM * 64;  // one 64-wide K half of a stage, 64-byte rows
constexpr int kW8RawA = 2 * kW8RawHalf;  // e4m3 weight stage: 128 rows x 128 K
constexpr int kW8Budget = 214 * 1024;    // both rings

// converted slots: A operands in tensor memory (64 columns each, next to the
// accumulators), plus shared memory for the Gate-Up's gathered token rows
__host__ __device__ constexpr int w8_conv_slots(int bn) { return bn <= 64 ? 4 : 2; }
__host__ __device__ constexpr int w8_conv_slot_bytes(int bn, int bsrc) {
  return bsrc == kGather ? 2 * bn * kKBytes : 0;
}
__host__ __device__ constexpr int w8_raw_slot_bytes(int bn, int bsrc) {
  return kW8RawA + (bsrc == kDirect ? 2 * bn * kKBytes : 0);
}
__host__ __device__ constexpr int w8_raw_slots(int bn, int bsrc) {
  return ((kW8Budget - w8_conv_slots(bn) * w8_conv_slot_bytes(bn, bsrc)) /
              w8_raw_slot_bytes(bn, bsrc) < 16)
             ? (kW8Budget - w8_conv_slots(bn) * w8_conv_slot_bytes(bn, bsrc)) /
                   w8_raw_slot_bytes(bn, bsrc)
             : 16;
}

template <int BN, int BSRC>
struct W8Shape {
  static constexpr int kBBytes = BN * kKBytes;            // one 64-wide token sub-tile
  static constexpr int kRawB = BSRC == kDirect ? 2 * kBBytes : 0;   // token rows (Down)
  static constexpr int kRawSlot = w8_raw_slot_bytes(BN, BSRC);
  static constexpr int kConvSlot = w8_conv_slot_bytes(BN, BSRC);   // Gate-Up token rows
  static constexpr int kRawSlots = w8_raw_slots(BN, BSRC);
  static constexpr int kConvSlots = w8_conv_slots(BN);
  static constexpr int kEpiWarps = 4;
  // two converter warps per scheduler for decode tiles: one alone is
  // latency-bound on the conversion chain
  static constexpr int kConvWarps = BN <= 64 ? 8 : 4;
  static constexpr int kRoleThreads = 64 + 32 * kEpiWarps;        // TMA, MMA, epilogue
  static constexpr int kConvThreads = 32 * kConvWarps;
  static constexpr int kGatherWarps = BSRC == kGather ? (BN >= 128 ? 2 : 1) : 0;
  static constexpr int kGatherThreads = 32 * kGatherWarps;
  static constexpr int kGatherBase = kRoleThreads + kConvThreads;
  static constexpr int kThreads = kGatherBase + kGatherThreads;
  static constexpr int kWarps = kThreads / 32;
  static constexpr int kRowsPerGatherThread = kGatherWarps ? BN / (4 * kGatherWarps) : 1;
  static constexpr int kAccBufs = (512 / BN < 2) ? 1 : 2;
  static constexpr int kACol0 = kAccBufs * BN;   // TMEM column of converted slot 0
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kIdesc = mma_idesc(1u, kTileM, BN);   // bf16 x bf16 -> fp32
  static constexpr int kOffConv = kRawSlots * kRawSlot;
  static constexpr int kOffBar = kOffConv + kConvSlots * kConvSlot;
  static constexpr int kNumBars = 2 * kRawSlots + 2 * kConvSlots + 2 * kAccBufs + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr size_t kSmemBytes = 1024 + ((kOffMisc + 16 + 15) & ~15);
  static_assert(kRawSlot % 1024 == 0 && kConvSlot % 1024 == 0, "slots keep 1024-byte alignment");
  static_assert(kACol0 + kConvSlots * 64 <= kTmemCols, "accumulators and A slots fit TMEM");
  static_assert(kConvWarps == 4 || kConvWarps == 8, "converter warps cover the four lane quadrants");
  static_assert(kRawSlots >= 3, "raw ring too shallow");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                "tcgen05.alloc takes a power of two from 32 to 512 columns");
};

// 16 e4m3 codes -> 16 bf16 values of code * scale (fp32 product, RNE to bf16):
// e4m3 pairs to fp16 pairs (exact), to fp32 (exact), one multiply, cvt.rn to
// bf16.  (Building the fp32 values by bit placement instead — an e4m3 byte in
// an fp32's low exponent bits is its value times 2^-120 — measured slower on
// the DeepSeek-shaped layer: 4.0 ms against 3.1 ms at T=64.)
__device__ __forceinline__ void dequant16_bf16(const uint4 raw, float scale, uint4& lo, uint4& hi) {
  const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint16_t pair = static_cast<uint16_t>(in[i] >> (16 * h));
      uint32_t f16x2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(f16x2) : "h"(pair));
      const __half2 hv = *reinterpret_cast<const __half2*>(&f16x2);
      const float a = __low2float(hv) * scale;    // the lower code of the pair
      const float b = __high2float(hv) * scale;
      const __nv_bfloat162 bv = __floats2bfloat162_rn(a, b);
      out[2 * i + h] = *reinterpret_cast<const uint32_t*>(&bv);
    }
  }
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
}

template <int BN, int BSRC>
__global__ void __launch_bounds__(W8Shape<BN, BSRC>::kThreads, 1)
    moe_gemm_w8_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using S = W8Shape<BN, BSRC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sRaw = smem_u32(smem);
  const uint32_t sConv = sRaw + S::kOffConv;
  const uint32_t bar_rfull = sRaw + S::kOffBar;
  const uint32_t bar_rempty = bar_rfull + 8 * S::kRawSlots;
  const uint32_t bar_cfull = bar_rempty + 8 * S::kRawSlots;
  const uint32_t bar_cempty = bar_cfull + 8 * S::kConvSlots;
  const uint32_t bar_accf = bar_cempty + 8 * S::kConvSlots;
  const uint32_t bar_acce = bar_accf + 8 * S::kAccBufs;
  const uint32_t bar_drain = bar_acce + 8 * S::kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Pipeline waits as in moe_gemm_kernel: bounded, left early once another
  // role gave up, and voted across the warp where warp-collective
  // instructions follow.
  const uint64_t wait_ns = p.pipe_wait_ns ? p.pipe_wait_ns : kWaitLimitNs;
  auto thread_wait = [&](uint32_t bar, uint32_t par) {
    return mbar_wait_pipe(bar, par, wait_ns, abort_flag);
  };
  auto warp_wait = [&](uint32_t bar, uint32_t par) {
    const bool r = mbar_wait_pipe(bar, par, wait_ns, abort_flag) && *abort_flag == 0;
    return __all_sync(0xffffffffu, r);
  };
  auto warp_aborted = [&]() { return __any_sync(0xffffffffu, *abort_flag != 0); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S::kRawSlots; ++s) {
      mbar_init(bar_rfull + 8 * s, 1);      // the TMA thread's expect-tx arrival
      // Gate-Up: each converter warp once it has read the slot; Down (whose
      // token rows the MMA reads from it): the MMA's commit
      mbar_init(bar_rempty + 8 * s, BSRC == kGather ? S::kConvWarps : 1);
    }
    for (int s = 0; s < S::kConvSlots; ++s) {
      mbar_init(bar_cfull + 8 * s, S::kConvThreads + S::kGatherThreads);
      mbar_init(bar_cempty + 8 * s, 1);
    }
    for (int b = 0; b < S::kAccBufs; ++b) {
      mbar_init(bar_accf + 8 * b, 1);
      mbar_init(bar_acce + 8 * b, S::kEpiWarps);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), S::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  pdl_wait();   // the index, the token rows and (Down) the activation come from earlier stages
  const int num_tiles = min(max(__ldcg(p.num_tiles), 0), p.tiles_cap);
  pdl_launch_dependents();
  const int units = num_tiles * p.m_tiles * p.splits;
  auto row_assign = [&](int pos) -> int { return __ldcg(p.sorted_ids + pos); };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int slot = 0;
    uint32_t phase = 0;
    long issued = 0;
    bool ok = true;
    constexpr uint32_t bytes = kW8RawA + S::kRawB;
    for (UnitIter<BN, BSRC> it(units, num_tiles, p, nullptr); ok && it.valid(); it.advance()) {
      if (warp_aborted()) break;
      const WorkUnit w = it.take(p);
      for (int kt = w.kt0; kt < w.kt1; ++kt) {
        if (!warp_wait(bar_rempty + 8 * slot, phase ^ 1u)) {
          report_timeout(p, abort_flag);
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = bar_rfull + 8 * slot;
          const uint32_t dst = sRaw + slot * S::kRawSlot;
          const int kc = kt * 128;   // e4m3: elements are bytes
          mbar_arrive_expect_tx(full, bytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (BSRC == kGather)
              tma_load_5d(dst + h * kW8RawHalf, &tmA, full, kc + 64 * h, 0, 0, w.mt * 4, w.e);
            else
              tma_load_3d(dst + h * kW8RawHalf, &tmA, full, kc + 64 * h, w.mt * kTileM, w.e);
            if (BSRC != kGather)
              tma_load_2d(dst + kW8RawA + h * S::kBBytes, &tmB, full, kc + 64 * h, w.row0);
          }
        }
        __syncwarp();
        ++issued;
        if (++slot == S::kRawSlots) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0) {
      // drain: our own copies land before the CTA can exit (long limit)
      const long first = issued > S::kRawSlots ? issued - S::kRawSlots : 0;
      for (long i = first; i < issued; ++i)
        mbar_wait(bar_rfull + 8 * static_cast<int>(i % S::kRawSlots),
                  static_cast<uint32_t>((i / S::kRawSlots) & 1));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int rs = 0, cs = 0, ab = 0;
      uint32_t cph = 0, aph = 0;
      bool ok = true;
      for (UnitIter<BN, BSRC> it(units, num_tiles, p, nullptr); ok && it.valid(); it.advance()) {
        if (*abort_flag) break;
        const WorkUnit w = it.take(p);
        const int n_eff = min(BN, max(16, (w.rows + 15) & ~15));
        const uint32_t idesc =
            (S::kIdesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(n_eff >> 3) << 17);
        if (!thread_wait(bar_acce + 8 * ab, aph ^ 1u)) {
          report_timeout(p, abort_flag);
          break;
        }
        tc_fence_after();
        for (int kt = w.kt0; kt < w.kt1; ++kt) {
          if (!thread_wait(bar_cfull + 8 * cs, cph)) {
            report_timeout(p, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();   // the converted A slot: tcgen05.st of other threads
          if (BSRC == kGather) fence_proxy_async_smem();   // gathered rows: generic-proxy writes
          const uint32_t conv = sConv + cs * S::kConvSlot;
          const uint32_t d = tmem_base + static_cast<uint32_t>(ab * BN);
          const uint32_t a_tm = tmem_base + static_cast<uint32_t>(S::kACol0 + cs * 64);
#pragma unroll
          for (int h = 0; h < 2; ++h) {   // the stage's two 64-wide halves of K
            const uint64_t bdesc = smem_desc_sw128(
                BSRC == kGather ? conv + h * S::kBBytes
                                : sRaw + rs * S::kRawSlot + kW8RawA + h * S::kBBytes);
#pragma unroll
            for (int k = 0; k < 4; ++k)   // 16 of K: 8 columns of A
              mma_bf16_tmem_a(d, a_tm + static_cast<uint32_t>(h * 32 + k * 8), bdesc + 2 * k,
                              idesc, (kt > w.kt0 || h > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(bar_cempty + 8 * cs);
          if (BSRC != kGather) tc_commit(bar_rempty + 8 * rs);
          if (++cs == S::kConvSlots) {
            cs = 0;
            cph ^= 1u;
          }
          if (++rs == S::kRawSlots) rs = 0;
        }
        if (ok) {
          tc_commit(bar_accf + 8 * ab);
          if (++ab == S::kAccBufs) {
            ab = 0;
            aph ^= 1u;
          }
        }
      }
      // always: another role may give up after our last MMA (long limit)
      tc_commit(bar_drain);
      mbar_wait(bar_drain, 0);
    }
    __syncwarp();
  } else if (warp < S::kRoleThreads / 32) {
    // ------------------------------------------------------------ epilogue (bf16)
    const int qd = warp & 3;
    const int r = qd * 32 + lane;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(qd * 32) << 16);
    int ab = 0;
    uint32_t aph = 0;
    for (UnitIter<BN, BSRC> it(units, num_tiles, p, nullptr); it.valid(); it.advance()) {
      const WorkUnit w = it.take(p);
      if (!warp_wait(bar_accf + 8 * ab, aph)) {
        report_timeout(p, abort_flag);
        break;
      }
      tc_fence_after();
      const bool fuse = BSRC == kGather && p.act_out != nullptr;
      const int feat = w.mt * 64 + qd * 16 + (lane & 15);   // Gate-Up: this lane's channel
      int col;
      bool col_ok = true;
      if (BSRC == kGather) {
        col = lane < 16 ? feat : p.I + feat;
      } else {
        col = w.mt * kTileM + r;
        col_ok = col < p.M;
      }
      float* outp = p.out + (static_cast<size_t>(w.ks) * p.rows_cap + w.row0) * p.M + col;
#pragma unroll
      for (int c = 0; c < BN / 16; ++c) {
        if (c * 16 < w.rows) {
          uint32_t v[16];
          tmem_ld16(t_lane + static_cast<uint32_t>(ab * BN + c * 16), v);
          tmem_ld_wait();
          tmem_ld_bind(v);
          if (fuse) {
            // lanes 0..15 hold gate, 16..31 the matching up: as in the bf16 GEMM
            const bool lo = lane < 16;
            __nv_bfloat16* arow = static_cast<__nv_bfloat16*>(p.act_out) +
                                  static_cast<size_t>(w.row0) * p.I + feat;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const float mine_a = __uint_as_float(v[jj]);
              const float mine_b = __uint_as_float(v[8 + jj]);
              const float peer_a = __shfl_xor_sync(0xffffffffu, mine_a, 16);
              const float peer_b = __shfl_xor_sync(0xffffffffu, mine_b, 16);
              const float g = lo ? mine_a : peer_b;
              const float u = lo ? peer_a : mine_b;
              const int n = c * 16 + (lo ? jj : 8 + jj);
              if (n < w.rows)
                arow[static_cast<size_t>(n) * p.I] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = c * 16 + j;
              if (n < w.rows && col_ok) outp[static_cast<size_t>(n) * p.M] = __uint_as_float(v[j]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acce + 8 * ab);
      if (++ab == S::kAccBufs) {
        ab = 0;
        aph ^= 1u;
      }
    }
  } else if (warp < S::kGatherBase / 32) {
    // ------------------------------------------------------------ converters
    // Lane l of a converter warp owns weight row r = 32 (warp % 4) + l of the
    // stage's 128-row tile (the TMEM lanes this warp may write) and converts
    // K half(s) kh of it: 64 e4m3 bytes, four 16-byte chunks read from the
    // 64-byte-swizzled raw half (chunk c of row r sits at c ^ ((r >> 1) & 3),
    // so a warp's 32 rows spread over eight bank groups), into 32 columns of
    // packed bf16 written with one tcgen05.st.  Eight warps: one K half each
    // (two warps per lane quadrant); four: both halves.  A row's block scale
    // is Down's, or (Gate-Up: rows 16..31 of each 32-row group are up rows)
    // the gate or up scale.
    constexpr int kHalves = S::kConvWarps == 8 ? 1 : 2;
    const int cw = warp - S::kRoleThreads / 32;   // converter warp 0..kConvWarps-1
    const int quad = warp & 3;
    const int kh0 = S::kConvWarps == 8 ? (cw >> 2) : 0;
    const int r = quad * 32 + lane;
    const int rsw = (r >> 1) & 3;
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
    const bool up_rows = BSRC == kGather && lane >= 16;
    const int t = threadIdx.x - S::kRoleThreads;
    const int KB = p.kt_total;      // 128-wide K blocks = stages
    int rs = 0, cs = 0;
    uint32_t rph = 0, cph = 0;
    bool ok = true;
    for (UnitIter<BN, BSRC> it(units, num_tiles, p, nullptr); ok && it.valid(); it.advance()) {
      if (warp_aborted()) break;
      const WorkUnit w = it.take(p);
      const int row = BSRC == kGather ? (up_rows ? p.I + w.mt * 64 : w.mt * 64) : w.mt * kTileM;
      const float* wsp = p.w_scale + (static_cast<size_t>(w.e) * (p.M >> 7) + (row >> 7)) * KB;
      float sc_next = __ldg(wsp + w.kt0);
      for (int kt = w.kt0; kt < w.kt1; ++kt) {
        const float sc = sc_next;
        if (kt + 1 < w.kt1) sc_next = __ldg(wsp + kt + 1);
        // both slots ready, one vote for the two waits
        const bool ready = mbar_wait_pipe(bar_rfull + 8 * rs, rph, wait_ns, abort_flag) &&
                           mbar_wait_pipe(bar_cempty + 8 * cs, cph ^ 1u, wait_ns, abort_flag) &&
                           *abort_flag == 0;
        if (!__all_sync(0xffffffffu, ready)) {
          report_timeout(p, abort_flag);
          ok = false;
          break;
        }
        const uint8_t* raw = smem + rs * S::kRawSlot + r * 64;
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
          const int kh = kh0 + hh;
          uint32_t col[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 q =
                *reinterpret_cast<const uint4*>(raw + kh * kW8RawHalf + ((c ^ rsw) << 4));
            uint4 lo, hi;
            dequant16_bf16(q, sc, lo, hi);
            col[8 * c + 0] = lo.x, col[8 * c + 1] = lo.y, col[8 * c + 2] = lo.z, col[8 * c + 3] = lo.w;
            col[8 * c + 4] = hi.x, col[8 * c + 5] = hi.y, col[8 * c + 6] = hi.z, col[8 * c + 7] = hi.w;
          }
          tmem_st32(t_row + static_cast<uint32_t>(S::kACol0 + cs * 64 + kh * 32), col);
        }
        tmem_st_wait();
        tc_fence_before();   // the MMA thread reads the slot after its wait
        mbar_arrive(bar_cfull + 8 * cs);
        if (BSRC == kGather) {
          // this warp's reads of the raw slot are done (their values were used)
          __syncwarp();
          if ((t & 31) == 0) mbar_arrive(bar_rempty + 8 * rs);
        }
        if (++rs == S::kRawSlots) {
          rs = 0;
          rph ^= 1u;
        }
        if (++cs == S::kConvSlots) {
          cs = 0;
          cph ^= 1u;
        }
      }
    }
  } else if (BSRC == kGather) {
    // ------------------------------------------------------------ token gather
    // As in the bf16 GEMM, into the converted slot's token area.
    constexpr int kR = S::kRowsPerGatherThread;
    constexpr int kRowStep = 4 * (S::kGatherWarps > 0 ? S::kGatherWarps : 1);
    const int t = threadIdx.x - S::kGatherBase;
    const int c = t & 7;
    const int r0 = t >> 3;
    const uint8_t* rows = static_cast<const uint8_t*>(p.b_rows) + c * 16;
    int cs = 0;
    uint32_t cph = 0;
    bool ok = true;
    for (UnitIter<BN, BSRC> it(units, num_tiles, p, nullptr); ok && it.valid(); it.advance()) {
      if (*abort_flag) break;
      const WorkUnit w = it.take(p);
      int tok[kR];
#pragma unroll
      for (int i = 0; i < kR; ++i) {
        const int n = r0 + kRowStep * i;
        tok[i] = n < w.rows ? assignment_token(row_assign(w.row0 + n), p) : -1;
      }
      for (int kt = w.kt0; kt < w.kt1; ++kt) {
        if (!thread_wait(bar_cempty + 8 * cs, cph ^ 1u)) {
          report_timeout(p, abort_flag);
          ok = false;
          break;
        }
        // the stage's 128 K of each row: two 128-byte halves, one per sub-tile
        const uint32_t b_dst = sConv + cs * S::kConvSlot;
        const uint8_t* src = rows + static_cast<size_t>(kt) * 2 * kKBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < kR; ++i) {
            const int n = r0 + kRowStep * i;
            if (tok[i] >= 0)
              cp_async_16(b_dst + h * S::kBBytes + n * kKBytes + ((c ^ (n & 7)) << 4),
                          src + h * kKBytes + static_cast<size_t>(tok[i]) * p.b_row_bytes);
          }
        cp_async_arrive_noinc(bar_cfull + 8 * cs);
        if (++cs == S::kConvSlots) {
          cs = 0;
          cph ^= 1u;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::kTmemCols);
  }
}

template <int BN, int BSRC>
cudaError_t launch_gemm_w8_inst(int grid, cudaStream_t st, bool pdl, const CUtensorMap& a,
                                const CUtensorMap& b, const GemmParams& p) {
  using S = W8Shape<BN, BSRC>;
  auto kern = moe_gemm_w8_kernel<BN, BSRC>;
  static int configured[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(S::kSmemBytes));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  return launch_kernel(kern, dim3(grid), dim3(S::kThreads), S::kSmemBytes, st, pdl, a, b, p);
}

}  // namespace moe
