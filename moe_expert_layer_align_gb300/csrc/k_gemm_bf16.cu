// k_gemm_bf16.cu — bf16 (kind::f16) instantiations of the expert GEMM:
// Gate-Up (gathered token rows) and router (dense rows).
#include "k_gemm.cuh"

namespace moe {

cudaError_t launch_gemm_bf16_gather_dense(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                                          const CUtensorMap& a, const CUtensorMap& b,
                                          const GemmParams& p, int me) {
  if (bsrc == kGather) return launch_gemm_bn<0, kGather>(bn, grid, st, pdl, a, b, p, me);
  if (bsrc == kDense) return launch_gemm_bn<0, kDense>(bn, grid, st, pdl, a, b, p);
  return cudaErrorInvalidValue;
}

}  // namespace moe
