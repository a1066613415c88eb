// BF16x3 operand split for the FP32 router GEMMs: x -> hi = RNE_bf16(x),
// lo = RNE_bf16(x - hi) (x - hi is exact in FP32), written as bf16 segments.
//
// The router's GEMMs emulate an FP32 product with three bf16 products,
// hi_a*hi_b + hi_a*lo_b + lo_a*hi_b (FlashInfer page "cache the router entry
// points' calls ...": the router GEMM through BF16x3 emulation, with an exact
// BF16x3 split).  The streamed operand is split inside the GEMM; the operand that
// every row tile reuses is split here once per call, so the GEMM does not redo
// the same split for each tile.  Two layouts are written:
//   planes       segment 0 = hi, segment 1 = lo, each a [rows][ldo] matrix
//                (forward: W; weight gradient: dY);
//   concatenated three segments per row or per matrix, so that one plain BF16
//                contraction over 3x the length sums lo*hi + hi*lo + hi*hi
//                (input gradient: dY as [lo | hi | hi] columns, W as [hi; lo; hi] rows).
// Each thread converts four consecutive FP32 values (one 16-byte load) and writes
// four bf16 per segment (8-byte stores); the pass is HBM-bound.
#include <algorithm>

#include "gemm_kernel.cuh"

namespace dp {

namespace {

struct SplitJobs {
  SplitJob job[2];
  int64_t quads[2];  // four-element groups of each job
  int njobs;
};

__global__ void __launch_bounds__(256) split_x3_kernel(const __grid_constant__ SplitJobs jobs) {
  const int64_t total = jobs.quads[0] + (jobs.njobs > 1 ? jobs.quads[1] : 0);
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
    const int j = i < jobs.quads[0] ? 0 : 1;
    const SplitJob& s = jobs.job[j];
    const int64_t q = j == 0 ? i : i - jobs.quads[0];
    const int64_t per_row = s.cols / 4;
    const int64_t r = q / per_row;
    const int64_t c = (q - r * per_row) * 4;
    const float4 x = __ldg(reinterpret_cast<const float4*>(s.x + r * s.ldx + c));
    const uint32_t h01 = pack_bf16x2(x.x, x.y), h23 = pack_bf16x2(x.z, x.w);
    const uint32_t l01 = pack_bf16x2(x.x - __uint_as_float(h01 << 16), x.y - __uint_as_float(h01 & 0xFFFF0000u));
    const uint32_t l23 = pack_bf16x2(x.z - __uint_as_float(h23 << 16), x.w - __uint_as_float(h23 & 0xFFFF0000u));
    const uint2 hi = make_uint2(h01, h23), lo = make_uint2(l01, l23);
    uint16_t* o = s.out + r * s.ldo + c;
    for (int seg = 0; seg < s.nseg; ++seg)
      *reinterpret_cast<uint2*>(o + seg * s.seg_stride) = ((s.lo_mask >> seg) & 1u) ? lo : hi;
  }
}

}  // namespace

cudaError_t launch_split_x3(const SplitJob* jobs, int njobs, int sm_count, cudaStream_t stream) {
  if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
  SplitJobs p = {};
  int64_t total = 0;
  for (int j = 0; j < njobs; ++j) {
    const SplitJob& s = jobs[j];
    // 16-byte loads and 8-byte stores: every row, column group and segment start aligned
    if (s.cols % 4 != 0 || s.ldx % 4 != 0 || s.ldo % 4 != 0 || s.seg_stride % 4 != 0 ||
        (reinterpret_cast<uintptr_t>(s.x) & 15u) != 0 || (reinterpret_cast<uintptr_t>(s.out) & 7u) != 0 ||
        s.nseg < 1 || s.nseg > 3)
      return cudaErrorInvalidValue;
    p.job[j] = s;
    p.quads[j] = s.rows * (s.cols / 4);
    total += p.quads[j];
  }
  p.njobs = njobs;
  if (total == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(sm_count) * 8);
  split_x3_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dp
