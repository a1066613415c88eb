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
// A quad of four consecutive FP32 values (one 16-byte load) becomes four bf16 per
// segment (8-byte stores); the pass is HBM-bound.
#include <algorithm>

#include "gemm_kernel.cuh"

namespace dp {

namespace {

struct SplitJobs {
  SplitJob job[2];
  int64_t quads[2];  // four-element groups of each job
  int njobs;
  ZeroJob zero;      // FP32 matrix to zero-fill (out null: none)
  int64_t zquads;    // its four-element groups
};

// Each thread converts four quads spaced one grid apart, all four loads issued
// before any store; row and column of a quad come from a 32-bit division when the
// job is small enough (always, for the router's sizes).
constexpr int kSplitThreads = 256;
constexpr int kSplitQuads = 4;

__device__ __forceinline__ void locate(const SplitJobs& jobs, uint64_t i, const SplitJob** s, int64_t* r,
                                       int64_t* c) {
  const int j = i < static_cast<uint64_t>(jobs.quads[0]) ? 0 : 1;
  *s = &jobs.job[j];
  const uint64_t q = j == 0 ? i : i - static_cast<uint64_t>(jobs.quads[0]);
  const uint64_t per_row = static_cast<uint64_t>((*s)->cols / 4);
  uint64_t row;
  if (q < (1ull << 32) && per_row < (1ull << 32))
    row = static_cast<uint32_t>(q) / static_cast<uint32_t>(per_row);
  else
    row = q / per_row;
  *r = static_cast<int64_t>(row);
  *c = static_cast<int64_t>(q - row * per_row) * 4;
}

__global__ void __launch_bounds__(kSplitThreads) split_x3_kernel(const __grid_constant__ SplitJobs jobs) {
  // Launched as a programmatic dependent of the kernel before it (so its launch overlaps
  // that kernel's tail): it reads nothing until that kernel is done, and only then lets
  // the GEMM launch, whose staging loads of its FP32 operand start before the GEMM's own
  // wait -- by then every kernel before this one has completed.
  pdl_wait();
  pdl_launch_dependents();  // the GEMM may start staging its other operand meanwhile
  // the zero fill of a non-deterministic call's output, one float4 per thread and step
  const uint64_t gstep = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < static_cast<uint64_t>(jobs.zquads); i += gstep) {
    const uint64_t per_row = static_cast<uint64_t>(jobs.zero.cols / 4);
    const uint64_t r = i / per_row, q = i - r * per_row;
    *reinterpret_cast<float4*>(jobs.zero.out + r * jobs.zero.ld + 4 * q) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const uint64_t total =
      static_cast<uint64_t>(jobs.quads[0]) + (jobs.njobs > 1 ? static_cast<uint64_t>(jobs.quads[1]) : 0);
  const uint64_t step = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i0 = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total;
       i0 += kSplitQuads * step) {
    float4 x[kSplitQuads];
    const SplitJob* sj[kSplitQuads];
    int64_t r[kSplitQuads], c[kSplitQuads];
#pragma unroll
    for (int k = 0; k < kSplitQuads; ++k) {
      const uint64_t i = i0 + k * step;
      if (i < total) {
        locate(jobs, i, &sj[k], &r[k], &c[k]);
        x[k] = __ldg(reinterpret_cast<const float4*>(sj[k]->x + r[k] * sj[k]->ldx + c[k]));
      }
    }
#pragma unroll
    for (int k = 0; k < kSplitQuads; ++k) {
      if (i0 + k * step >= total) continue;
      const uint32_t h01 = pack_bf16x2(x[k].x, x[k].y), h23 = pack_bf16x2(x[k].z, x[k].w);
      const uint32_t l01 =
          pack_bf16x2(x[k].x - __uint_as_float(h01 << 16), x[k].y - __uint_as_float(h01 & 0xFFFF0000u));
      const uint32_t l23 =
          pack_bf16x2(x[k].z - __uint_as_float(h23 << 16), x[k].w - __uint_as_float(h23 & 0xFFFF0000u));
      const uint2 hi = make_uint2(h01, h23), lo = make_uint2(l01, l23);
      uint16_t* o = sj[k]->out + r[k] * sj[k]->ldo + c[k];
      for (int seg = 0; seg < sj[k]->nseg; ++seg)
        *reinterpret_cast<uint2*>(o + seg * sj[k]->seg_stride) = ((sj[k]->lo_mask >> seg) & 1u) ? lo : hi;
    }
  }
}

}  // namespace

cudaError_t launch_split_x3(const SplitJob* jobs, int njobs, int sm_count, cudaStream_t stream,
                            const ZeroJob* zero) {
  if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
  SplitJobs p = {};
  if (zero && zero->rows > 0) {
    if (zero->cols % 4 != 0 || zero->ld % 4 != 0 || (reinterpret_cast<uintptr_t>(zero->out) & 15u) != 0)
      return cudaErrorInvalidValue;
    p.zero = *zero;
    p.zquads = zero->rows * (zero->cols / 4);
  }
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
  if (total == 0 && p.zquads == 0) return cudaSuccess;
  const int64_t per_block = kSplitThreads * kSplitQuads;
  const int64_t work = std::max<int64_t>(total, p.zquads);
  const int64_t blocks = std::min<int64_t>((work + per_block - 1) / per_block, static_cast<int64_t>(sm_count) * 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kSplitThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_x3_kernel, p);
}

cudaError_t set_attributes_split() {
  // the same shared-memory carveout as the GEMM kernels, so switching between them
  // does not reconfigure the SMs
  return cudaFuncSetAttribute(split_x3_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              cudaSharedmemCarveoutMaxShared);
}

}  // namespace dp
