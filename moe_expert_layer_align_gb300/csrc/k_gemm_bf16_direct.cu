// k_gemm_bf16_direct.cu — bf16 (kind::f16) Down GEMM instantiations (token
// operand = contiguous activation rows of a tile).
#include "k_gemm.cuh"

namespace moe {

cudaError_t launch_gemm_bf16_gather_dense(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                                          const CUtensorMap& a, const CUtensorMap& b,
                                          const GemmParams& p, int me);

cudaError_t launch_gemm_bf16(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                             const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                             int me) {
  if (bsrc == kDirect) return launch_gemm_bn<0, kDirect>(bn, grid, st, pdl, a, b, p, me);
  return launch_gemm_bf16_gather_dense(bn, bsrc, grid, st, pdl, a, b, p, me);
}

template <int FP8, int BSRC>
size_t smem_bytes_bn(int bn) {
  switch (bn) {
    case 16: return GemmShape<FP8, 16, BSRC>::kSmemBytes;
    case 32: return GemmShape<FP8, 32, BSRC>::kSmemBytes;
    case 64: return GemmShape<FP8, 64, BSRC>::kSmemBytes;
    case 128: return GemmShape<FP8, 128, BSRC>::kSmemBytes;
    case 256: return FP8 ? 0 : GemmShape<0, 256, BSRC>::kSmemBytes;
    default: return 0;
  }
}

size_t gemm_smem_bytes(int fp8, int bn, int bsrc) {
  if (bsrc == kGather) return fp8 ? smem_bytes_bn<1, kGather>(bn) : smem_bytes_bn<0, kGather>(bn);
  return fp8 ? smem_bytes_bn<1, kDirect>(bn) : smem_bytes_bn<0, kDirect>(bn);
}

template <int FP8>
int gemm_warps_t(int bn, int bsrc) {
  switch (bn) {
    case 16: return bsrc == kGather ? GemmShape<FP8, 16, kGather>::kWarps : GemmShape<FP8, 16, kDirect>::kWarps;
    case 32: return bsrc == kGather ? GemmShape<FP8, 32, kGather>::kWarps : GemmShape<FP8, 32, kDirect>::kWarps;
    case 64: return bsrc == kGather ? GemmShape<FP8, 64, kGather>::kWarps : GemmShape<FP8, 64, kDirect>::kWarps;
    case 128: return bsrc == kGather ? GemmShape<FP8, 128, kGather>::kWarps : GemmShape<FP8, 128, kDirect>::kWarps;
    default: return bsrc == kGather ? GemmShape<FP8, 256, kGather>::kWarps : GemmShape<FP8, 256, kDirect>::kWarps;
  }
}

int gemm_warps(int fp8, int bn, int bsrc) {
  return fp8 ? gemm_warps_t<1>(bn, bsrc) : gemm_warps_t<0>(bn, bsrc);
}

size_t gemm_index_smem_bytes(int nwarps, int E, int tk, int rows_cap, int tiles_cap) {
  return SmemIndex::bytes(nwarps, E, tk, rows_cap, tiles_cap);
}

}  // namespace moe
