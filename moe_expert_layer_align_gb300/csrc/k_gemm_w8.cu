// k_gemm_w8.cu — instantiations of the w8a16 expert GEMM (FP8 weights, bf16
// activations): Gate-Up (gathered token rows) and Down (contiguous rows).
#include "k_gemm_w8.cuh"

namespace moe {

template <int BSRC>
cudaError_t launch_w8_bn(int bn, int grid, cudaStream_t st, bool pdl, const CUtensorMap& a,
                         const CUtensorMap& b, const GemmParams& p) {
  switch (bn) {
    case 16: return launch_gemm_w8_inst<16, BSRC>(grid, st, pdl, a, b, p);
    case 32: return launch_gemm_w8_inst<32, BSRC>(grid, st, pdl, a, b, p);
    case 64: return launch_gemm_w8_inst<64, BSRC>(grid, st, pdl, a, b, p);
    case 128: return launch_gemm_w8_inst<128, BSRC>(grid, st, pdl, a, b, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_w8(int bn, int bsrc, int grid, cudaStream_t st, bool pdl,
                           const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p) {
  if (bsrc == kGather) return launch_w8_bn<kGather>(bn, grid, st, pdl, tmA, tmB, p);
  if (bsrc == kDirect) return launch_w8_bn<kDirect>(bn, grid, st, pdl, tmA, tmB, p);
  return cudaErrorInvalidValue;
}

}  // namespace moe
