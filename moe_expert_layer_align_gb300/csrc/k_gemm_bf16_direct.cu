// k_gemm_bf16_direct.cu — bf16 (kind::f16) Down GEMM instantiations (token
// operand = contiguous activation rows of a tile).
#include "k_gemm.cuh"

namespace moe {

cudaError_t launch_gemm_bf16_gather_dense(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                                          const CUtensorMap& a, const CUtensorMap& b,
                                          const GemmParams& p);

cudaError_t launch_gemm_bf16(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                             const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p) {
  if (bsrc == kDirect) return launch_gemm_bn<0, kDirect>(bn, grid, st, pdl, a, b, p);
  return launch_gemm_bf16_gather_dense(bn, bsrc, grid, st, pdl, a, b, p);
}

int gemm_stages(int fp8, int bn) { return stages_for(fp8, bn); }

size_t gemm_smem_bytes(int fp8, int bn, int) {
  switch (bn) {
    case 16: return fp8 ? GemmShape<1, 16>::kSmemBytes : GemmShape<0, 16>::kSmemBytes;
    case 32: return fp8 ? GemmShape<1, 32>::kSmemBytes : GemmShape<0, 32>::kSmemBytes;
    case 64: return fp8 ? GemmShape<1, 64>::kSmemBytes : GemmShape<0, 64>::kSmemBytes;
    case 128: return fp8 ? GemmShape<1, 128>::kSmemBytes : GemmShape<0, 128>::kSmemBytes;
    case 256: return GemmShape<0, 256>::kSmemBytes;
    default: return 0;
  }
}

}  // namespace moe
