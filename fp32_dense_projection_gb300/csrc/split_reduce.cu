// Ordered reduction of split partial tiles.
//
// A plan that splits a tile's contraction into `splits` contiguous ranges has the
// GEMM write one FP32 partial tile per range.  This kernel, launched right behind
// the GEMM on the same stream, adds them for every output element in ascending
// range order (p_0 + p_1 + ... + p_{S-1}, FP32) and rounds the sum once to the
// output type.  The order depends on nothing but the plan, so the result is
// bitwise repeatable (FlashInfer page "... restore the K1 weight-gradient routes
// ...": deterministic weight gradients over a fixed split of the 64-token blocks).
// Every slice of every tile is summed by its own CTA, so the sum costs about one
// round trip to L2 instead of S of them in a single CTA.  It is launched as a
// programmatic dependent of the GEMM: its launch overlaps the GEMM's tail and
// griddepcontrol.wait holds it until the partials are complete and visible.
#include "gemm_kernel.cuh"

namespace dp {

namespace {

struct ReduceArgs {
  GemmArgs g;              // output, partial buffer and the tile raster of the GEMM
  int32_t bn;              // tile width: a partial tile is 128 x bn FP32 per slot
  int32_t tile_rows;       // rows of an output tile (256 for a CTA pair)
  int32_t slots_per_tile;  // partial slots per tile (one per CTA of the tile)
  int32_t chunks;          // 32-column chunks per tile
};

// One CTA of four warps per (slot, 32-column chunk); warp w sums rows
// [32w, 32w + 32) of the slot.  Partial layout: [slot][split][bn/4][128] float4.
// Lane layout: for the row-major output value i of a lane is row 4i + lane/8,
// float4 chunk lane%8, so each store instruction writes four whole 128-byte row
// segments; for the transposed store (swapped weight gradient) it is row `lane`,
// chunk i, so consecutive lanes write consecutive elements of each output row.
__global__ void __launch_bounds__(128) split_reduce_kernel(const __grid_constant__ ReduceArgs ra) {
  pdl_wait();  // the GEMM's partials are complete and visible
  const GemmArgs& a = ra.g;
  const int chunk = static_cast<int>(blockIdx.x) % ra.chunks;
  const int slot = static_cast<int>(blockIdx.x) / ra.chunks;
  const int ptile = slot / ra.slots_per_tile, rank = slot - ptile * ra.slots_per_tile;
  int tm, tn;
  tile_coords(a, a.full_units + ptile, &tm, &tn);
  const int warp = static_cast<int>(threadIdx.x) >> 5, lane = static_cast<int>(threadIdx.x) & 31;
  const int64_t m0 = static_cast<int64_t>(tm) * ra.tile_rows + rank * kBlockM + warp * 32;
  const int64_t col = static_cast<int64_t>(tn) * ra.bn + chunk * 32;
  if (m0 >= a.gm || col >= a.gn) return;
  const bool tr = a.out_trans != 0;
  const int r0 = tr ? lane : (lane >> 3), dr = tr ? 0 : 4;
  const int c0 = tr ? 0 : (lane & 7), dc = tr ? 1 : 0;
  const int istep = dc * kBlockM + dr;  // float4 distance between a lane's values i and i + 1
  const int64_t rows_left = a.gm - m0;
  const size_t pstride = static_cast<size_t>(kBlockM) * ra.bn / 4;  // float4 per partial tile
  // (rows past the output's end hold no partials; their sums are never stored)
  const float4* src = a.partials + static_cast<size_t>(slot) * a.splits * pstride +
                      static_cast<size_t>(chunk) * 8 * kBlockM + warp * 32 + c0 * kBlockM + r0;
  float4 acc[8];
  // splits in ascending order, four in flight at a time
  for (int sp = 0; sp < a.splits; sp += 4) {
    float4 x[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (sp + k < a.splits)
#pragma unroll
        for (int i = 0; i < 8; ++i) x[k][i] = __ldcg(src + (sp + k) * pstride + i * istep);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (sp + k < a.splits)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (sp + k == 0) {
            acc[i] = x[k][i];
          } else {
            acc[i].x += x[k][i].x;
            acc[i].y += x[k][i].y;
            acc[i].z += x[k][i].z;
            acc[i].w += x[k][i].w;
          }
        }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = r0 + i * dr;
    const int64_t cc = col + 4 * (c0 + i * dc);
    if (r >= rows_left || cc >= a.gn) continue;
    if (tr) {
      const float e[4] = {acc[i].x, acc[i].y, acc[i].z, acc[i].w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int64_t o = (cc + t) * a.ldo + m0 + r;
        if (a.out_f32)
          static_cast<float*>(a.out)[o] = e[t];
        else
          static_cast<uint16_t*>(a.out)[o] = static_cast<uint16_t>(pack_bf16x2(e[t], 0.0f) & 0xFFFFu);
      }
    } else if (a.out_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(a.out) + (m0 + r) * a.ldo + cc) = acc[i];
    } else {
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + (m0 + r) * a.ldo + cc) =
          make_uint2(pack_bf16x2(acc[i].x, acc[i].y), pack_bf16x2(acc[i].z, acc[i].w));
    }
  }
}

}  // namespace

cudaError_t launch_split_reduce(const GemmLaunch& l, int bn, bool pair, int64_t split_tiles, cudaStream_t stream) {
  ReduceArgs ra;
  ra.g = l.args;
  ra.bn = bn;
  ra.tile_rows = pair ? 2 * kBlockM : kBlockM;
  ra.slots_per_tile = pair ? 2 : 1;
  ra.chunks = bn / 32;
  const int64_t blocks = split_tiles * ra.slots_per_tile * ra.chunks;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_reduce_kernel, ra);
}

}  // namespace dp
