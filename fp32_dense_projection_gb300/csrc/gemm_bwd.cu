// Instantiations of the co-scheduled backward launch: the input gradient (K-major
// A = dY, MN-major B = W) and the weight gradient (MN-major A and B) of one layer
// as one persistent grid over both problems' tiles.  Tiles 128 x {128, 256} (one
// CTA) and 256 x {128, 256} (a CTA pair); both problems keep whole K per tile.
#include "gemm_kernel.cuh"

namespace dp {

cudaError_t launch_gemm_bwd(int bn, bool pair, const GemmLaunch& l, cudaStream_t stream) {
  if (pair) {
    switch (bn) {
      case 128:
        return launch_gemm_t<128, false, true, true, false, true>(l, stream);
      case 256:
        return launch_gemm_t<256, false, true, true, false, true>(l, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 128:
      return launch_gemm_t<128, false, true, false, false, true>(l, stream);
    case 256:
      return launch_gemm_t<256, false, true, false, false, true>(l, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t set_attributes_bwd() {
  cudaError_t e = set_attr_t<128, false, true, false, false, true>();
  if (e == cudaSuccess) e = set_attr_t<256, false, true, false, false, true>();
  if (e == cudaSuccess) e = set_attr_t<128, false, true, true, false, true>();
  if (e == cudaSuccess) e = set_attr_t<256, false, true, true, false, true>();
  return e;
}

}  // namespace dp
