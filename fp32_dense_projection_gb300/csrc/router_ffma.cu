// Small-T FP32 router program: a SIMT FP32 FFMA GEMM with a deterministic split of
// the contraction across the CTAs of a thread-block cluster.
//
// At a few dozen to a few hundred tokens the router's three GEMMs (hidden H ->
// 256 experts) are too small for the tensor-core BF16x3 program's three kernels
// (operand split, GEMM, ordered reduction) to pay: each leaves most of its time
// in launch and pipeline latency.  The pages record that at T = 64 and 256 plain
// FP32 library GEMMs beat the deterministic BF16x3 router (FlashInfer page
// "cache the router entry points' calls ...", SOTA rows at T 64 / 256).  This
// program computes the same contractions directly in FP32 on the CUDA cores, in
// one launch, with no workspace:
//
//   D[m][n] = sum_k A(m, k) * B(n, k)   (FP32 operands, FP32 fused multiply-adds)
//
// Tiling.  A cluster of S CTAs owns one 64 x BN output tile; CTA s of the cluster
// sums the contraction chunks [s * C / S, (s + 1) * C / S) of the C chunks of
// 16 * KG elements.  Inside the CTA the 256 threads form KG contraction groups of
// BN threads; group g takes the elements [16 g, 16 g + 16) of every chunk, and each
// thread accumulates an 8 x 8 block of the tile (16 floats read from shared memory
// per 64 FMAs, so the FMA pipe, not shared-memory bandwidth, sets the pace).
//
// Order of the sums (fixed, so the output is bitwise repeatable): each thread
// accumulates its k in ascending order with one FMA per product; the CTA adds its
// KG group partials in group order; rank r of the cluster adds the S CTA partials
// of its rows in rank order, read from the other CTAs' shared memory.
//
// Operands arrive through cp.async (16-byte copies, zero fill outside the
// matrices) into a two-stage shared-memory ring.  K-major tiles are stored as
// [row][k] with rows padded by 4 floats and read as float4 along k; MN-major
// tiles as [k][row] and read as float4 along the rows; each layout gives its
// thread a row mapping (strided for [row][k], consecutive for [k][row]) under
// which the float4 reads of a warp do not conflict on banks.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_kernel.cuh"

namespace dp {

namespace {

constexpr int kFfmaThreads = 256;
constexpr int kFfmaBM = 64;

template <int BN, bool A_MN, bool B_MN>
struct FfmaCfg {
  static constexpr int BM = kFfmaBM;
  static constexpr int COLS = BN / 8;      // column slots of a group's 8 x COLS thread grid
  static constexpr int TG = 8 * COLS;      // threads of one contraction group (an 8 x 8 block each)
  static constexpr int KG = kFfmaThreads / TG;
  static constexpr int KS = 16;            // contraction elements of a group per stage
  static constexpr int BKS = KS * KG;      // contraction elements per stage
  static_assert(BKS == ffma_stage_k(BN), "stage length");
  // floats per row of each smem tile, and per tile
  static constexpr int A_LD = A_MN ? BM : BKS + 4;
  static constexpr int B_LD = B_MN ? BN : BKS + 4;
  static constexpr int A_FLOATS = A_MN ? BKS * BM : BM * (BKS + 4);
  static constexpr int B_FLOATS = B_MN ? BKS * BN : BN * (BKS + 4);
  static constexpr int STAGE_FLOATS = A_FLOATS + B_FLOATS;
  // stages in flight: as many as fit in 168 KB, 2 to 8 (the loads come from L2 or
  // DRAM with microseconds of latency)
  static constexpr int STAGES_FIT = (168 * 1024) / (STAGE_FLOATS * 4);
  static constexpr int STAGES = STAGES_FIT < 2 ? 2 : (STAGES_FIT > 8 ? 8 : STAGES_FIT);
  static constexpr int RED_FLOATS = BM * BN;  // the CTA's partial tile (read by the cluster)
  static constexpr int SMEM_BYTES = (STAGES * STAGE_FLOATS + RED_FLOATS) * 4;
  static_assert(kFfmaThreads % TG == 0 && KG >= 1, "thread groups");
  static_assert(KG * BM * BN <= STAGES * STAGE_FLOATS, "group partials fit in the stage buffers");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Copy the chunk [k0, k0 + BKS) of the tile's operand rows [r0, r0 + ROWS) into smem.
// K-major: global [rows][k] -> smem [row][LD]; MN-major: global [k][rows] -> smem [k][ROWS].
template <int ROWS, int BKS, int LD, bool MN>
__device__ __forceinline__ void load_tile(uint32_t dst, const float* src, int64_t ld, int64_t rows, int64_t kdim,
                                          int64_t r0, int64_t k0) {
  if (!MN) {
    constexpr int per_row = BKS / 4;
    for (int c = static_cast<int>(threadIdx.x); c < ROWS * per_row; c += kFfmaThreads) {
      const int r = c / per_row, q = c - r * per_row;
      const int64_t gr = r0 + r, gk = k0 + 4 * q;
      const bool ok = gr < rows && gk < kdim;
      cp_async16(dst + 4u * static_cast<uint32_t>(r * LD + 4 * q), ok ? src + gr * ld + gk : src, ok);
    }
  } else {
    constexpr int per_k = ROWS / 4;
    for (int c = static_cast<int>(threadIdx.x); c < BKS * per_k; c += kFfmaThreads) {
      const int k = c / per_k, q = c - k * per_k;
      const int64_t gk = k0 + k, gr = r0 + 4 * q;
      const bool ok = gk < kdim && gr < rows;
      cp_async16(dst + 4u * static_cast<uint32_t>(k * ROWS + 4 * q), ok ? src + gk * ld + gr : src, ok);
    }
  }
}

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kFfmaThreads, 1) router_ffma_kernel(const __grid_constant__ FfmaArgs args) {
  using C = FfmaCfg<BN, A_MN, B_MN>;
  extern __shared__ __align__(16) float fsm[];
  const uint32_t sbase = smem_addr(fsm);
  float* red = fsm + C::STAGES * C::STAGE_FLOATS;

  const int S = args.splits;
  const int s = S > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int tile = static_cast<int>(blockIdx.x) / S;
  const int tm = tile / args.tiles_n, tn = tile - tm * args.tiles_n;
  const int64_t m0 = static_cast<int64_t>(tm) * C::BM, n0 = static_cast<int64_t>(tn) * BN;
  const int c0 = static_cast<int>(static_cast<int64_t>(s) * args.kchunks / S);
  const int c1 = static_cast<int>(static_cast<int64_t>(s + 1) * args.kchunks / S);

  // (launched as a programmatic dependent of the kernel before it on the stream: its
  // setup overlaps that kernel's tail, and nothing is read before that kernel is done)
  pdl_wait();
  const int tid = static_cast<int>(threadIdx.x);
  const int g = tid / C::TG, t = tid - g * C::TG;
  const int ty = t / C::COLS, tx = t - ty * C::COLS;
  // this thread's 8 rows and 8 columns of the tile: from a [row][k] tile rows ty + 8i
  // (the float4 reads along k of 8 neighbouring threads hit different banks); from a
  // [k][row] tile two runs of 4, 4ty.. and 32 + 4ty.. (neighbouring threads read
  // consecutive 16-byte pieces)
  int mrow[8], ncol[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    mrow[i] = A_MN ? (i < 4 ? 4 * ty + i : C::BM / 2 + 4 * ty + i - 4) : ty + 8 * i;
    ncol[i] = B_MN ? (i < 4 ? 4 * tx + i : BN / 2 + 4 * tx + i - 4) : tx + C::COLS * i;
  }
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  auto stage_load = [&](int chunk, int buf) {
    const uint32_t sa = sbase + 4u * static_cast<uint32_t>(buf * C::STAGE_FLOATS);
    const int64_t k0 = static_cast<int64_t>(chunk) * C::BKS;
    load_tile<C::BM, C::BKS, C::A_LD, A_MN>(sa, args.a, args.lda, args.gm, args.gk, m0, k0);
    load_tile<BN, C::BKS, C::B_LD, B_MN>(sa + 4u * C::A_FLOATS, args.b, args.ldb, args.gn, args.gk, n0, k0);
  };

  // STAGES - 1 chunks in flight ahead of the one being summed (one commit group per
  // chunk slot, empty past the end, so the wait counts stay uniform)
#pragma unroll
  for (int i = 0; i < C::STAGES - 1; ++i) {
    if (c0 + i < c1) stage_load(c0 + i, i);
    cp_async_commit();
  }
  for (int c = c0; c < c1; ++c) {
    const int buf = (c - c0) % C::STAGES;
    cp_async_wait<C::STAGES - 2>();  // chunk c has landed (for this thread's copies)
    __syncthreads();                 // ... for every thread's; and buffer c - 1 is free
    if (c + C::STAGES - 1 < c1) stage_load(c + C::STAGES - 1, (c - c0 + C::STAGES - 1) % C::STAGES);
    cp_async_commit();
    const float* As = fsm + buf * C::STAGE_FLOATS;
    const float* Bs = As + C::A_FLOATS;
    const int kg = C::KS * g;  // this group's elements of the chunk
#pragma unroll 1
    for (int kk = 0; kk < C::KS; kk += 4) {
      float a[8][4], b[8][4];  // [row or column][k]
      if (!A_MN) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v = *reinterpret_cast<const float4*>(As + mrow[i] * C::A_LD + kg + kk);
          a[i][0] = v.x, a[i][1] = v.y, a[i][2] = v.z, a[i][3] = v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float4 v = *reinterpret_cast<const float4*>(As + (kg + kk + k) * C::BM + mrow[4 * h]);
            a[4 * h][k] = v.x, a[4 * h + 1][k] = v.y, a[4 * h + 2][k] = v.z, a[4 * h + 3][k] = v.w;
          }
      }
      if (!B_MN) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 v = *reinterpret_cast<const float4*>(Bs + ncol[j] * C::B_LD + kg + kk);
          b[j][0] = v.x, b[j][1] = v.y, b[j][2] = v.z, b[j][3] = v.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float4 v = *reinterpret_cast<const float4*>(Bs + (kg + kk + k) * BN + ncol[4 * h]);
            b[4 * h][k] = v.x, b[4 * h + 1][k] = v.y, b[4 * h + 2][k] = v.z, b[4 * h + 3][k] = v.w;
          }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i][k], b[j][k], acc[i][j]);
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // every copy landed and every read of the stage buffers done

  // group partials -> the stage buffers (free now) -> the CTA partial, groups in order
  float* part = fsm;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) part[(g * C::BM + mrow[i]) * BN + ncol[j]] = acc[i][j];
  __syncthreads();
  for (int e = tid; e < C::BM * BN; e += kFfmaThreads) {
    float v = part[e];
#pragma unroll
    for (int q = 1; q < C::KG; ++q) v += part[q * C::BM * BN + e];
    red[e] = v;
  }

  if (S == 1) {
    __syncthreads();
    for (int e = tid; e < C::BM * BN; e += kFfmaThreads) {
      const int r = e / BN, col = e - r * BN;
      if (m0 + r < args.gm && n0 + col < args.gn) args.out[(m0 + r) * args.ldo + n0 + col] = red[e];
    }
    return;
  }
  // the cluster's CTA partials, rank order; rank s writes rows [s*BM/S, (s+1)*BM/S)
  cluster_sync();
  const int r0 = s * C::BM / S, r1 = (s + 1) * C::BM / S;
  const uint32_t red_addr = smem_addr(red);
  for (int e = r0 * BN + tid; e < r1 * BN; e += kFfmaThreads) {
    float v = ld_cluster_f32(map_shared_rank(red_addr + 4u * e, 0));
    for (int q = 1; q < S; ++q) v += ld_cluster_f32(map_shared_rank(red_addr + 4u * e, q));
    const int r = e / BN, col = e - r * BN;
    if (m0 + r < args.gm && n0 + col < args.gn) args.out[(m0 + r) * args.ldo + n0 + col] = v;
  }
  cluster_sync();  // no CTA leaves while the others read its partial
}

template <int BN, bool A_MN, bool B_MN>
cudaError_t launch_t(const FfmaArgs& a, cudaStream_t stream) {
  using C = FfmaCfg<BN, A_MN, B_MN>;
  cudaLaunchConfig_t cfg = {};
  const int tiles = static_cast<int>(((a.gm + C::BM - 1) / C::BM) * a.tiles_n);
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * a.splits), 1, 1);
  cfg.blockDim = dim3(kFfmaThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (a.splits > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(a.splits);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, router_ffma_kernel<BN, A_MN, B_MN>, a);
}

template <int BN, bool A_MN, bool B_MN>
cudaError_t set_attr_ffma() {
  return cudaFuncSetAttribute(router_ffma_kernel<BN, A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              FfmaCfg<BN, A_MN, B_MN>::SMEM_BYTES);
}

template <bool A_MN, bool B_MN>
cudaError_t launch_view_ffma(int bn, const FfmaArgs& a, cudaStream_t stream) {
  switch (bn) {
    case 32:
      return launch_t<32, A_MN, B_MN>(a, stream);
    case 64:
      return launch_t<64, A_MN, B_MN>(a, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

template <bool A_MN, bool B_MN>
cudaError_t set_view_ffma() {
  cudaError_t e = set_attr_ffma<32, A_MN, B_MN>();
  if (e == cudaSuccess) e = set_attr_ffma<64, A_MN, B_MN>();
  return e;
}

}  // namespace

cudaError_t launch_router_ffma(int bn, bool a_mn, bool b_mn, const FfmaArgs& a, cudaStream_t stream) {
  if (a.splits < 1 || a.splits > 8 || a.kchunks < 1) return cudaErrorInvalidValue;
  if (!a_mn && !b_mn) return launch_view_ffma<false, false>(bn, a, stream);
  if (!a_mn && b_mn) return launch_view_ffma<false, true>(bn, a, stream);
  if (a_mn && b_mn) return launch_view_ffma<true, true>(bn, a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t set_attributes_ffma() {
  cudaError_t e = set_view_ffma<false, false>();
  if (e == cudaSuccess) e = set_view_ffma<false, true>();
  if (e == cudaSuccess) e = set_view_ffma<true, true>();
  return e;
}

}  // namespace dp
