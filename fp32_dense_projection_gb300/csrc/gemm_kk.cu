// Instantiations of the GEMM for the forward: K-major A (X or dY), K-major B (W).
// One translation unit per operand-major combination so the builds run in parallel.
// BF16 operands: single-CTA tiles 128 x {64, 128, 256}, CTA-pair tiles 256 x {128, 256}.
// Router BF16x3 forward (FP32 X split in the kernel, W from pre-split planes):
// single-CTA tiles 128 x {64, 128, 256}, CTA-pair tiles 256 x {128, 256}.
#include "gemm_kernel.cuh"

namespace dp {

cudaError_t launch_gemm_kk(int bn, const GemmLaunch& l, cudaStream_t stream) {
  if (l.x3 && l.pair) {
    switch (bn) {
      case 128:
        return launch_gemm_t<128, false, false, true, true>(l, stream);
      case 256:
        return launch_gemm_t<256, false, false, true, true>(l, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  if (l.x3) {
    switch (bn) {
      case 64:
        return launch_gemm_t<64, false, false, false, true>(l, stream);
      case 128:
        return launch_gemm_t<128, false, false, false, true>(l, stream);
      case 256:
        return launch_gemm_t<256, false, false, false, true>(l, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  if (l.pair) {
    switch (bn) {
      case 128:
        return launch_gemm_t<128, false, false, true>(l, stream);
      case 256:
        return launch_gemm_t<256, false, false, true>(l, stream);
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 64:
      return launch_gemm_t<64, false, false, false>(l, stream);
    case 128:
      return launch_gemm_t<128, false, false, false>(l, stream);
    case 256:
      return launch_gemm_t<256, false, false, false>(l, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t set_attributes_kk() {
  cudaError_t e = set_attr_t<64, false, false, false>();
  if (e == cudaSuccess) e = set_attr_t<128, false, false, false>();
  if (e == cudaSuccess) e = set_attr_t<256, false, false, false>();
  if (e == cudaSuccess) e = set_attr_t<128, false, false, true>();
  if (e == cudaSuccess) e = set_attr_t<256, false, false, true>();
  if (e == cudaSuccess) e = set_attr_t<64, false, false, false, true>();
  if (e == cudaSuccess) e = set_attr_t<128, false, false, false, true>();
  if (e == cudaSuccess) e = set_attr_t<256, false, false, false, true>();
  if (e == cudaSuccess) e = set_attr_t<128, false, false, true, true>();
  if (e == cudaSuccess) e = set_attr_t<256, false, false, true, true>();
  return e;
}

int max_clusters_kk(int bn, bool x3, int cluster, int grid) {
  switch (bn) {
    case 64:
      return x3 ? max_active_clusters_t<64, false, false, false, true>(cluster, grid)
                : max_active_clusters_t<64, false, false, false>(cluster, grid);
    case 128:
      return x3 ? max_active_clusters_t<128, false, false, false, true>(cluster, grid)
                : max_active_clusters_t<128, false, false, false>(cluster, grid);
    case 256:
      return x3 ? max_active_clusters_t<256, false, false, false, true>(cluster, grid)
                : max_active_clusters_t<256, false, false, false>(cluster, grid);
    default:
      return 0;
  }
}

}  // namespace dp
