// k_gemm_fp8.cu — e4m3 (kind::f8f6f4) instantiations of the expert GEMM with
// per-128 block-scale promotion: Gate-Up (gathered rows) and Down (direct).
#include "k_gemm.cuh"

namespace moe {

cudaError_t launch_gemm_fp8(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                            const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p) {
  if (bsrc == kGather) return launch_gemm_bn<1, kGather>(bn, grid, st, pdl, a, b, p);
  if (bsrc == kDirect) return launch_gemm_bn<1, kDirect>(bn, grid, st, pdl, a, b, p);
  return cudaErrorInvalidValue;
}

}  // namespace moe
