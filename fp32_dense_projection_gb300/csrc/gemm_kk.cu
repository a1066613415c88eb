// Instantiations of the BF16 GEMM for the forward: K-major A (X or dY), K-major B (W).
// One translation unit per operand-major combination so the builds run in parallel.
#include "gemm_kernel.cuh"

namespace dp {

cudaError_t launch_gemm_kk(int bn, const GemmLaunch& l, cudaStream_t stream) {
  switch (bn) {
    case 64:
      return launch_gemm_t<64, false, false>(l, stream);
    case 128:
      return launch_gemm_t<128, false, false>(l, stream);
    case 256:
      return launch_gemm_t<256, false, false>(l, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t set_attributes_kk() {
  cudaError_t e = set_attr_t<64, false, false>();
  if (e == cudaSuccess) e = set_attr_t<128, false, false>();
  if (e == cudaSuccess) e = set_attr_t<256, false, false>();
  return e;
}

}  // namespace dp
