// Instantiations of the GEMM for the input gradient: K-major A (dY), MN-major B (W).
// One translation unit per operand-major combination so the builds run in parallel.
// BF16 operands: single-CTA tiles 128 x {64, 128, 256}, CTA-pair tiles 256 x {128, 256}.
// (The router's input gradient runs these BF16 kernels on its concatenated hi/lo operands.)
#include "gemm_kernel.cuh"

namespace dp {

cudaError_t launch_gemm_km(int bn, const GemmLaunch& l, cudaStream_t stream) {
  if (l.x3) return cudaErrorInvalidValue;  // the router's input gradient runs the plain BF16 kernel
  if (l.pair) {
    switch (bn) {
      case 128:
        return launch_gemm_t<128, false, true, true>(l, stream);
      case 256:
        return launch_gemm_t<256, false, true, true>(l, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 64:
      return launch_gemm_t<64, false, true, false>(l, stream);
    case 128:
      return launch_gemm_t<128, false, true, false>(l, stream);
    case 256:
      return launch_gemm_t<256, false, true, false>(l, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t set_attributes_km() {
  cudaError_t e = set_attr_t<64, false, true, false>();
  if (e == cudaSuccess) e = set_attr_t<128, false, true, false>();
  if (e == cudaSuccess) e = set_attr_t<256, false, true, false>();
  if (e == cudaSuccess) e = set_attr_t<128, false, true, true>();
  if (e == cudaSuccess) e = set_attr_t<256, false, true, true>();
  return e;
}

int max_clusters_km(int bn, int cluster, int grid) {
  switch (bn) {
    case 64:
      return max_active_clusters_t<64, false, true, false>(cluster, grid);
    case 128:
      return max_active_clusters_t<128, false, true, false>(cluster, grid);
    case 256:
      return max_active_clusters_t<256, false, true, false>(cluster, grid);
    default:
      return 0;
  }
}

}  // namespace dp
