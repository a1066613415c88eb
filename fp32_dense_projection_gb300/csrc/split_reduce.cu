// Ordered reduction of split partial tiles.
//
// A plan that splits a tile's contraction into `splits` contiguous ranges has the
// GEMM write one FP32 partial tile per range (a stream-K plan: one per slot whose
// block range cuts the tile, however many that is for each tile).  This kernel, launched right behind
// the GEMM on the same stream, adds them for every output element in ascending
// range order (p_0 + p_1 + ... + p_{S-1}, FP32) and rounds the sum once to the
// output type.  The order depends on nothing but the plan, so the result is
// bitwise repeatable (FlashInfer page "... restore the K1 weight-gradient routes
// ...": deterministic weight gradients over a fixed split of the 64-token blocks).
// Every float4 of every split tile (transposed output: every four rows of one) has
// its own thread, which issues the loads of all its splits at once (or in batches
// of 8 or 16), so the sum costs about one round trip to L2.  It is
// launched as a programmatic dependent of the GEMM: its launch overlaps the GEMM's
// tail and griddepcontrol.wait holds it until the partials are complete and
// visible.
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

// Row-major output: one thread per float4 of the split tiles.  Thread t of the (slot,
// 32-column chunk) handles row t % 128 and float4 column t / 128 of the chunk, so a
// warp's loads are 512 contiguous bytes of each partial, and loads all splits (8 or
// 16 at a time) before adding them in order; it stores its 4 values as one 16-byte
// store (or 8 bytes of bf16).  Transposed output (the swapped weight gradient): one
// thread per 4 rows of a float4 column (thread t: rows 4(t % 32) .. +3, float4 column
// t / 32), which it writes as one 16-byte (8-byte) store per output column, next to
// its neighbouring lanes' rows.  Partial layout: [slot][split][bn/4][128] float4.
constexpr int kReduceThreads = 128;
constexpr int kReduceBatchTrans = 4;  // (four rows each: 16 float4 loads in flight)

// TRANS: the transposed output (a.out_trans).  BATCH: row-major partials loaded at a
// time, 8 for plans of at most 8 splits and 16 above (measured on GB300: 8 is 1-2 us
// faster for the 7- and 8-way thin weight-gradient sums at T = 65537, 16 is 2-3 us
// faster for the router forward's 16- and 19-way sums).  Each combination is its own
// instantiation, so none carries the registers of a larger one.
template <bool TRANS, int BATCH>
__global__ void __launch_bounds__(kReduceThreads) split_reduce_kernel(const __grid_constant__ ReduceArgs ra) {
  pdl_wait();  // the GEMM's partials are complete and visible
  const GemmArgs& a = ra.g;
  // CTAs per (slot, chunk): 1024 float4, one or four per thread
  const int per_slice = (TRANS ? kBlockM * 8 / 4 : kBlockM * 8) / kReduceThreads;
  const int cta = static_cast<int>(blockIdx.x);
  const int slice = cta / per_slice;
  const int t = (cta - slice * per_slice) * kReduceThreads + static_cast<int>(threadIdx.x);  // 0..1023 (255)
  const int chunk = slice % ra.chunks;
  const int slot = slice / ra.chunks;
  const int ptile = slot / ra.slots_per_tile, rank = slot - ptile * ra.slots_per_tile;
  // partials to add: the plan's split count, or for a stream-K plan the number of
  // slots whose block ranges touch this tile (one: the GEMM stored the tile whole)
  int nparts = a.splits;
  if (a.sk_slots > 0) {
    const int64_t t0 = static_cast<int64_t>(ptile) * a.nkb;
    nparts = sk_slot_of(a, t0 + a.nkb - 1) - sk_slot_of(a, t0) + 1;
    if (nparts < 2) return;
  }
  int bt, tm, tn;
  tile_coords(a, a.full_units + ptile, &bt, &tm, &tn);
  void* out = out_at(a, bt);
  // row of the slot (the first of four: transposed output), float4 column in the chunk
  const int row = TRANS ? 4 * (t & 31) : t & (kBlockM - 1), j = TRANS ? t >> 5 : t >> 7;
  const int64_t m = static_cast<int64_t>(tm) * ra.tile_rows + rank * kBlockM + row;
  const int64_t col = static_cast<int64_t>(tn) * ra.bn + chunk * 32 + 4 * j;
  if (m >= a.gm || col >= a.gn) return;  // (transposed: gm and gn are multiples of 4)
  const size_t pstride = static_cast<size_t>(kBlockM) * ra.bn / 4;  // float4 per partial tile
  const float4* src = a.partials + static_cast<size_t>(slot) * a.splits * pstride +
                      static_cast<size_t>(chunk * 8 + j) * kBlockM + row;
  if constexpr (TRANS) {
    float4 acc[4];
    for (int s0 = 0; s0 < nparts; s0 += kReduceBatchTrans) {
      float4 x[kReduceBatchTrans][4];
#pragma unroll
      for (int k = 0; k < kReduceBatchTrans; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (s0 + k < nparts) x[k][i] = __ldcg(src + static_cast<size_t>(s0 + k) * pstride + i);
#pragma unroll
      for (int k = 0; k < kReduceBatchTrans; ++k)
        if (s0 + k < nparts)
#pragma unroll
          for (int i = 0; i < 4; ++i) sum_step(acc[i], x[k][i], s0 + k == 0);
    }
    store_trans4x4(a, out, m, col, acc);
    return;
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // splits in ascending order: acc = p_0, then acc += p_s
  for (int s0 = 0; s0 < nparts; s0 += BATCH) {
    float4 x[BATCH];
#pragma unroll
    for (int k = 0; k < BATCH; ++k)
      if (s0 + k < nparts) x[k] = __ldcg(src + static_cast<size_t>(s0 + k) * pstride);
#pragma unroll
    for (int k = 0; k < BATCH; ++k)
      if (s0 + k < nparts) sum_step(acc, x[k], s0 + k == 0);
  }
  if (a.out_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + m * a.ldo + col) = acc;
  } else {
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + m * a.ldo + col) =
        make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
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
  const int64_t blocks = split_tiles * ra.slots_per_tile * ra.chunks *
                        ((l.args.out_trans ? kBlockM * 8 / 4 : kBlockM * 8) / kReduceThreads);
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kReduceThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (l.args.out_trans) return cudaLaunchKernelEx(&cfg, split_reduce_kernel<true, 8>, ra);
  return l.args.splits > 8 ? cudaLaunchKernelEx(&cfg, split_reduce_kernel<false, 16>, ra)
                           : cudaLaunchKernelEx(&cfg, split_reduce_kernel<false, 8>, ra);
}

cudaError_t set_attributes_reduce() {
  // the same shared-memory carveout as the GEMM kernels, so switching between them
  // does not reconfigure the SMs
  cudaError_t e = cudaFuncSetAttribute(split_reduce_kernel<false, 8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(split_reduce_kernel<false, 16>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(split_reduce_kernel<true, 8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

}  // namespace dp
