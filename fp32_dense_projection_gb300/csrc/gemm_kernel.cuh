// Persistent, warp-specialised BF16 GEMM for sm_103a:
//     D[m][n] = sum_k A(m, k) * B(n, k)      (FP32 accumulation in TMEM)
//
// One CTA per SM walks a static list of work units (output tile x contraction
// split).  Roles inside the CTA (256 threads; the router's BF16x3 mode adds the
// converter warps 2, 3, 8, 9 and, on single CTAs, warp 10):
//   warp 0      TMA producer: loads 128x64 A and BNx64 B bf16 tiles (128-byte
//               swizzle) into a shared-memory ring of STAGES block slots, one
//               or two contraction blocks per ring stage (GemmArgs::kps);
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer (M=128,
//               N=BN, K=16 per instruction), accumulating into one of two TMEM
//               accumulators so the epilogue of a tile overlaps the next tile's
//               main loop;
//   warp 2      BF16 mode: the loads of B (warp 0 then loads only A);
//   warp 10     BF16x3 on single CTAs: the loads of B's bf16 planes (warp 0 then loads
//               only A's FP32 staging tiles);
//   warps 4..7  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//               32*(w%4)...), BF16 round-to-nearest-even or FP32, staged in
//               shared memory and written by TMA stores or 16-byte stores; for
//               split units, FP32 partial tiles in the workspace, summed in
//               ascending split order by the tile's cluster after the main loop
//               (cluster_fixup_sum) or by the reduction kernel (split_reduce.cu).
//
// Operand "majorness" is a template parameter.  A K-major operand is a row-major
// [rows][contraction] matrix (one TMA box of 64 contraction elements x rows);
// an MN-major operand is a row-major [contraction][rows] matrix (boxes of 64
// rows-direction elements x 64 contraction rows, placed 8 KB apart).  The
// forward pass uses K-major A and B, the input gradient K-major A and MN-major B,
// and the weight gradient MN-major A and B (FlashInfer page
// "perf(cake_dense_projection_det_gemm): plan the 4096 -> 12288 input gradient
// ...", PR body: "forward (K-major B)" and "input-gradient (MN-major B)" forms;
// page "... restore the K1 weight-gradient routes ...": wgrad over 64-token K
// blocks).  Ragged edges come from TMA zero fill on loads and bounds checks on
// stores, so a partial 64-token block adds exactly its valid tokens.
//
// Every barrier wait is bounded (see mbar_wait): on a timeout the kernel records
// a fault bit, unwinds, waits (bounded) for its own TMA loads and MMAs, and frees
// its TMEM, so a broken pipeline cannot hang the GPU.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "planner.h"
#include "ptx.cuh"

namespace dp {

struct GemmArgs {
  int64_t gm, gn;      // output rows and columns of the contraction view
  int32_t nkb;         // 64-wide contraction blocks in total
  int32_t splits;      // contraction splits of each split tile
  int32_t full_units;  // units [0, full_units) are whole-K tiles; the rest split `splits` ways
  int32_t tiles_m, tiles_n;
  int32_t group;       // raster group width, in tiles of the grouped raster dimension
  int32_t raster_m;    // 1: row tiles fastest inside a group (B column blocks shared)
  int32_t units;       // full_units + (tiles - full_units) * splits
  int32_t batch;       // independent GEMMs sharing the plan (tiles of batch b follow those of b - 1)
  int32_t tiles_per_batch;  // tiles_m * tiles_n
  int64_t out_bstride; // output elements between consecutive batches
  void* out;
  int64_t ldo;         // output leading dimension (elements)
  int32_t out_f32;     // 1: FP32 output, 0: BF16 output
  int32_t out_trans;   // 1: D[m][n] is stored at out[n * ldo + m] (swapped weight gradient)
  // MN-major operands whose tensor map is 3-D, [column group][contraction row][128 B]:
  // the groups of a tile arrive in one load instead of one load per group
  int32_t a3d, b3d;
  // A read MN-major (the template's A_MN, except in a co-scheduled launch, whose two
  // problems may differ)
  int32_t a_mn;
  // > 1: launched as clusters of `splits` CTAs, one split tile per cluster and one
  // unit per CTA; the cluster sums its partials itself after the main loop
  int32_t cluster_fixup;
  // > 0: a stream-K plan.  The sk_slots persistent slots (CTAs, or pairs) share the
  // sk_work = tiles * nkb contraction blocks evenly: slot c takes the blocks
  // [c * sk_work / sk_slots, (c + 1) * sk_work / sk_slots) of the tile-major order.
  // A tile cut by a slot boundary is summed in pieces, one per slot that touches it
  // (piece s of the tile from the s-th such slot, in block order), each an FP32
  // partial in slot s of the tile's `splits` partial slots; whole tiles are stored.
  int32_t sk_slots;
  int64_t sk_work;
  // 1 (non-deterministic plans, FP32 output): split units add their FP32 partial
  // into the output, which the launch zero-filled, with atomic adds; no partials
  // and no reduction.  The order of the adds, and so the last bits, vary by run.
  int32_t atomic;
  // contraction blocks per stage of the operand ring (1 or 2; 1 for BF16x3 and
  // co-scheduled launches): a stage's loads complete on one barrier, and an SM's
  // TMA streams from DRAM at about one stage per round trip slot whatever the
  // stage's size, so streaming plans carry two blocks per stage
  int32_t kps;
  // bit 0 (A) / bit 1 (B): the operand's bytes are read once by the whole launch (one
  // column tile reads all of A, or one row tile all of B; split units read disjoint
  // contraction ranges), so its TMA loads carry an L2 evict-first policy and the
  // stream replaces its own lines instead of the rest of the L2 (single-CTA tiles)
  int32_t evict_first;
  // 1: the epilogue warps stage TMA stores in one block each even where two exist
  // (comparisons of the two)
  int32_t epi_single;
  float4* partials;    // split partial tiles: [split tile slot][split][BN/4][128] float4
  uint32_t* fault;     // device status word
  uint64_t wait_ns;    // limit of every barrier wait (ns); past it the kernel records a fault and unwinds
  // tma_store = 1: whole-tile results leave through TMA stores instead of the
  // epilogue warps' own stores, with tmO the output as a TMA map ([batch][gm][gn],
  // leading dimension ldo; boxes of 32 rows x 128 bytes (32 FP32 or 64 BF16
  // columns) with the 128-byte swizzle the epilogue stages them in)
  int32_t tma_store;
  // tma_store2 = 1 (FP32 output of one problem, a whole number of 32-column blocks
  // wide): two staged 32 x 32 blocks leave in one TMA store, through tmO2, the output as
  // [32-column block][row][32] with the same swizzle
  int32_t tma_store2;
  CUtensorMap tmO;
  CUtensorMap tmO2;
};

// X3: the FP32 router's BF16x3 mode.  A stage of the MMA ring then holds the bf16
// hi and lo halves of a 32-wide contraction block of each operand
// ([A_hi | A_lo | B_hi | B_lo]).  A's halves are written by converter warps from an
// FP32 staging tile that TMA loads into a separate, one-stage-deeper ring; B's
// halves are loaded by TMA from two bf16 planes split before the launch.  With
// PAIR, each CTA of the pair splits its own 128 rows of A and loads half of B, and
// both CTAs' converters arrive on the leader's full barrier.
template <int BN, bool PAIR = false, bool X3 = false>
struct TileCfg {
  static constexpr int BM = kBlockM;             // accumulator rows per CTA
  static constexpr int TM = PAIR ? 2 * BM : BM;  // output tile rows (a CTA pair splits them)
  static constexpr int BNH = PAIR ? BN / 2 : BN; // B rows each CTA loads
  static constexpr int BK = X3 ? kRouterBlockK : kBlockK;
  static constexpr int STAGES = X3 ? stages_x3(BN, PAIR) : stages_for(BN, PAIR);
  static constexpr int SSTAGES = X3 ? staging_stages_x3(BN, PAIR) : 0;  // FP32 staging ring (X3)
  static constexpr int A_HALF = BM * BK * 2;     // one bf16 copy of the A tile
  static constexpr int B_HALF = BNH * BK * 2;
  // (X3 on a single CTA: A's halves in tensor memory, none in the stage)
  static constexpr int A_BYTES = X3 ? (PAIR ? 2 * A_HALF : 0) : A_HALF;
  static constexpr int B_BYTES = X3 ? 2 * B_HALF : B_HALF;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SA_BYTES = X3 ? BM * BK * 4 : 0;  // one FP32 staging tile of A (X3)
  // X3 on single CTAs: the converter warps write A's bf16 hi and lo halves into tensor
  // memory (32 columns per ring stage: hi in the first 16, lo in the next 16, two bf16 per
  // 32-bit column, row = lane) and the MMAs read A from there, which takes A's writes and
  // its three reads per slice off the shared-memory port (CTA pairs keep A in shared memory)
  static constexpr bool A_TMEM = X3 && !PAIR;
  static_assert(!X3 || A_TMEM == (A_BYTES == 0), "BF16x3 stage layout");
  // accumulators: two (a unit's epilogue overlaps the next unit's main loop), or one where
  // the A stages would not fit beside two (256-wide BF16x3 tiles)
  static constexpr int NACC = (A_TMEM && 2 * BN + STAGES * 32 > 512) ? 1 : 2;
  static constexpr int A_TMEM_COL = NACC * BN;  // first column of the A stages
  static constexpr int TMEM_NEED = NACC * BN + (A_TMEM ? STAGES * 32 : 0);
  static constexpr int TMEM_COLS = TMEM_NEED <= 32    ? 32
                                   : TMEM_NEED <= 64  ? 64
                                   : TMEM_NEED <= 128 ? 128
                                   : TMEM_NEED <= 256 ? 256
                                                      : 512;
  static_assert(TMEM_NEED <= 512, "tensor memory");
  // Output staging blocks per epilogue warp (4 KB each: a 32 x 32 FP32 block, or two 32 x
  // 32 BF16 blocks): two, so a warp stages its next block while the TMA store of the
  // previous one still reads shared memory; one in BF16x3 mode, whose rings leave no room.
  static constexpr int EPI_BUFS = X3 ? 1 : 2;
  static constexpr int EPI_BYTES = 4 * 4096 * EPI_BUFS;
  // X3: four converter warps (2, 3, 8, 9: one per SM sub-partition) split A
  static constexpr int CONV_WARPS = X3 ? 4 : 0;
  // B's loads have their own producer thread (lane 0 of warp B_WARP_ID): warp 2, idle
  // otherwise, in BF16 mode; an eleventh warp for BF16x3 on single CTAs, so the thread
  // that loads A's FP32 staging tiles and the one that loads B each wait on one ring.
  // (One thread serving both took ~1000 cycles per 32-wide BF16x3 block for two barrier
  // tests, two expect-tx arrivals and three TMA issues, against ~770 cycles of MMAs.)
  // BF16x3 pairs keep one producer thread.
  static constexpr bool B_WARP = !(X3 && PAIR);
  static constexpr int B_WARP_ID = X3 ? 10 : 2;
  static constexpr int THREADS = X3 ? (B_WARP ? 352 : 320) : 256;
  static_assert(X3 || (B_WARP && B_WARP_ID == 2), "BF16 mode: warp 2 loads B");
  // full, empty, tmem_full x2, tmem_empty x2, drain (+ staging full / empty for X3)
  static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * SSTAGES;
  static constexpr int SMEM_BYTES =
      1024 + STAGES * STAGE_BYTES + SSTAGES * SA_BYTES + EPI_BYTES + NUM_BARS * 8 + 64;
  static_assert(BN == 64 || BN == 128 || BN == 256, "tile width");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(STAGE_BYTES % 1024 == 0 && SA_BYTES % 1024 == 0, "swizzle alignment");
  static_assert(!X3 || (STAGE_BYTES == x3_stage_bytes(BN, PAIR) && SA_BYTES == kX3StagingBytes), "planner sizes");
};

// Work unit u -> output tile, contraction range and, for split units, the split
// index and the split tile's slot in the partial/counter arrays.
//   u <  full_units: whole-K unit of tile u (all nkb blocks, one accumulator)
//   u >= full_units: v = u - full_units; tile full_units + v / splits, split v % splits,
//                    blocks [s*nkb/splits, (s+1)*nkb/splits)
// A plan either splits every tile (full_units = 0), none (units = full_units), or
// only the tiles of the last partial wave.  Tiles are rastered in groups of
// `group` tiles along one dimension with that dimension fastest, so the CTAs
// running at one time share operand blocks in L2: by default groups of output
// columns (A row-blocks shared); with raster_m, groups of output rows (B
// column-blocks shared), which the planner picks when B is the larger operand.
struct Unit {
  int b;         // batch
  int tm, tn;    // output tile coordinates
  int s;         // split index (0 for whole-K units)
  int ptile;     // index of a split tile among the split tiles (its partials' slot)
  int kb0, kb1;  // contraction blocks [kb0, kb1)
  bool split;    // partial result: summed by the ordered reduction kernel
};

// Output tile index -> (batch, row tile, column tile); within a batch the tiles
// follow the grouped raster.
__device__ __forceinline__ void tile_coords(const GemmArgs& a, int tile, int* b, int* tm, int* tn) {
  *b = tile / a.tiles_per_batch;
  tile -= *b * a.tiles_per_batch;
  const int fast_tiles = a.raster_m ? a.tiles_m : a.tiles_n;  // dimension grouped, fastest
  const int slow_tiles = a.raster_m ? a.tiles_n : a.tiles_m;
  const int per_group = a.group * slow_tiles;
  const int g = tile / per_group;
  const int first = g * a.group;
  const int width = min(a.group, fast_tiles - first);
  const int local = tile - g * per_group;
  const int fast = first + local % width;
  const int slow = local / width;
  *tm = a.raster_m ? fast : slow;
  *tn = a.raster_m ? slow : fast;
}

__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, int u) {
  Unit r;
  int tile;
  if (u < a.full_units) {
    tile = u;
    r.s = 0;
    r.ptile = 0;
    r.kb0 = 0;
    r.kb1 = a.nkb;
    r.split = false;
  } else {
    const int v = u - a.full_units;
    const int q = v / a.splits;
    r.s = v - q * a.splits;
    r.ptile = q;
    tile = a.full_units + q;
    r.kb0 = static_cast<int>(static_cast<int64_t>(r.s) * a.nkb / a.splits);
    r.kb1 = static_cast<int>(static_cast<int64_t>(r.s + 1) * a.nkb / a.splits);
    r.split = a.splits > 1;
  }
  tile_coords(a, tile, &r.b, &r.tm, &r.tn);
  return r;
}

// Stream-K plans: the first block of slot c's range, the slot whose range holds
// block x, and the j-th piece of slot c's range (false past its end).
__device__ __forceinline__ int64_t sk_begin(const GemmArgs& a, int64_t c) { return c * a.sk_work / a.sk_slots; }
__device__ __forceinline__ int sk_slot_of(const GemmArgs& a, int64_t x) {
  int64_t c = x * a.sk_slots / a.sk_work;
  while (c + 1 < a.sk_slots && sk_begin(a, c + 1) <= x) ++c;
  while (c > 0 && sk_begin(a, c) > x) --c;
  return static_cast<int>(c);
}
__device__ __forceinline__ bool sk_piece(const GemmArgs& a, int c, int j, Unit* w) {
  const int64_t b = sk_begin(a, c), e = sk_begin(a, c + 1);
  const int64_t tile = b / a.nkb + j, t0 = tile * a.nkb;
  if (b >= e || t0 >= e) return false;
  w->kb0 = static_cast<int>((b > t0 ? b : t0) - t0);
  w->kb1 = static_cast<int>((e < t0 + a.nkb ? e : t0 + a.nkb) - t0);
  w->split = !(w->kb0 == 0 && w->kb1 == a.nkb);
  w->s = c - sk_slot_of(a, t0);  // the tile's first piece comes from the slot holding its block 0
  w->ptile = static_cast<int>(tile);
  tile_coords(a, static_cast<int>(tile), &w->b, &w->tm, &w->tn);
  return true;
}

// Output of batch b.
__device__ __forceinline__ void* out_at(const GemmArgs& a, int b) {
  return static_cast<char*>(a.out) + static_cast<int64_t>(b) * a.out_bstride * (a.out_f32 ? 4 : 2);
}

// The second problem of a co-scheduled launch (DUAL): its tensor maps and
// arguments.  Its units follow the first problem's in the launch's unit list, so
// the persistent CTAs that finish the first problem's tiles go on with the second's
// (the input and weight gradients of one layer in one launch: B is MN-major in
// both, A is K-major in the input gradient and MN-major in the weight gradient).
template <bool DUAL>
struct SecondProblem {
  int32_t none;
};
template <>
struct SecondProblem<true> {
  CUtensorMap tmA, tmB;
  GemmArgs args;
};

// One unit of the launch: its problem's arguments and maps, and its index there.
struct UnitRef {
  const GemmArgs* a;
  const CUtensorMap* mA;
  const CUtensorMap* mB;
  int u;
};

__device__ __forceinline__ int second_units(const SecondProblem<false>&) { return 0; }
__device__ __forceinline__ int second_units(const SecondProblem<true>& s) { return s.args.units; }
__device__ __forceinline__ void prefetch_second(const SecondProblem<false>&) {}
__device__ __forceinline__ void prefetch_second(const SecondProblem<true>& s) {
  tma_prefetch_map(&s.tmA);
  tma_prefetch_map(&s.tmB);
}
__device__ __forceinline__ UnitRef unit_ref(int u, const GemmArgs& a0, const CUtensorMap& mA, const CUtensorMap& mB,
                                            const SecondProblem<false>&) {
  return {&a0, &mA, &mB, u};
}
__device__ __forceinline__ UnitRef unit_ref(int u, const GemmArgs& a0, const CUtensorMap& mA, const CUtensorMap& mB,
                                            const SecondProblem<true>& s) {
  if (u < a0.units) return {&a0, &mA, &mB, u};
  return {&s.args, &s.tmA, &s.tmB, u - a0.units};
}

// The k-th unit of the CTA (or pair) in slot `slot`: units slot, slot + step, ... of
// the launch's list, or the pieces of the slot's block range in a stream-K plan.
// False past the last one.
template <bool DUAL>
__device__ __forceinline__ bool slot_unit(int k, int slot, int step, int total, const GemmArgs& args,
                                          const CUtensorMap& mA, const CUtensorMap& mB,
                                          const SecondProblem<DUAL>& sec, UnitRef* ur, Unit* w) {
  if (!DUAL && args.sk_slots > 0) {
    *ur = {&args, &mA, &mB, 0};
    return sk_piece(args, slot, k, w);
  }
  const int u = slot + k * step;
  if (u >= total) return false;
  *ur = unit_ref(u, args, mA, mB, sec);
  *w = decode_unit(DUAL ? *ur->a : args, ur->u);
  return true;
}

// Store 32 FP32 accumulator values (one row segment) as BF16 or FP32.  add (FP32
// output of a non-deterministic split unit): add them into the output atomically.
__device__ __forceinline__ void store_row32(const GemmArgs& a, void* out, int64_t m, int64_t col0,
                                            const float (&v)[32], bool add = false) {
  if (m >= a.gm) return;
  if (a.out_trans) {
    // D[m][n] goes to out[n][m]: the 32 lanes of a warp hold 32 consecutive m, so
    // each of these stores writes 32 consecutive output elements.
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (col0 + j >= a.gn) break;
      const int64_t o = (col0 + j) * a.ldo + m;
      if (add)
        red_add_f32(static_cast<float*>(out) + o, v[j]);
      else if (a.out_f32)
        static_cast<float*>(out)[o] = v[j];
      else
        static_cast<uint16_t*>(out)[o] = static_cast<uint16_t>(pack_bf16x2(v[j], 0.0f) & 0xFFFFu);
    }
    return;
  }
  if (a.out_f32) {
    float* dst = static_cast<float*>(out) + m * a.ldo + col0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (col0 + 4 * j < a.gn)
        *reinterpret_cast<float4*>(dst + 4 * j) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  } else {
    uint16_t* dst = static_cast<uint16_t*>(out) + m * a.ldo + col0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (col0 + 8 * j < a.gn) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
        w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
        w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
        w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
        *reinterpret_cast<uint4*>(dst + 8 * j) = w;
      }
  }
}

// Store a 32 x 32 block of the output, called by a whole warp: lane i holds the
// 32 values of row m0 + i, columns [col0, col0 + 32).  stage_block32 puts the block
// in the warp's 4 KB of shared memory (16-byte chunks XOR-swizzled by row, so
// neither the row-wise writes nor the column-wise reads conflict on banks);
// flush_block32 reads it back by columns and writes 16-byte stores of which each
// instruction covers whole 128-byte (FP32) or 64-byte (BF16) row segments, instead
// of one 16-byte piece of 32 different rows.  (The transposed store of the swapped
// weight gradient is already coalesced and goes straight out.)
__device__ __forceinline__ void stage_block32(const GemmArgs& a, uint32_t buf, int lane, const float (&v)[32]) {
  __syncwarp();  // the previous block's reads of buf are done
  if (a.out_f32) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_u4(buf + lane * 128 + ((j ^ (lane & 7)) << 4),
                   make_uint4(__float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                              __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3])));
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      st_shared_u4(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4),
                   make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                              pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7])));
  }
  __syncwarp();
}

// BF16 half h (columns [32h, 32h + 32)) of a 32 x 64 block staged for a TMA store:
// rows of 128 bytes, 16-byte chunk j of row r at chunk j ^ (r % 8) (the 128-byte
// swizzle of the output map).  Lane i holds row i.
__device__ __forceinline__ void stage_half64_bf16(uint32_t buf, int lane, int h, const float (&v)[32]) {
  __syncwarp();  // the block's previous reader is done (and half 0 is written before half 1)
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_u4(buf + lane * 128 + (((4 * h + j) ^ (lane & 7)) << 4),
                 make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                            pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7])));
  __syncwarp();
}

__device__ __forceinline__ void flush_block32(const GemmArgs& a, void* out, uint32_t buf, int lane, int64_t m0,
                                              int64_t col0, bool add = false) {
  const int64_t rows_left = a.gm - m0;
  if (a.out_f32) {
    const int ch = lane & 7, r0 = lane >> 3;
    const bool col_ok = col0 + 4 * ch < a.gn;
    float* p = static_cast<float*>(out) + (m0 + r0) * a.ldo + col0 + 4 * ch;
    const int64_t step = 4 * a.ldo;
#pragma unroll
    for (int i = 0; i < 8; ++i, p += step) {
      const int r = 4 * i + r0;
      const uint4 x = ld_shared_u4(buf + r * 128 + ((ch ^ (r & 7)) << 4));
      if (col_ok && r < rows_left) {
        if (add)
          red_add_v4_f32(p, x);
        else
          *reinterpret_cast<uint4*>(p) = x;
      }
    }
  } else {
    const int ch = lane & 3, r0 = lane >> 2;
    const bool col_ok = col0 + 8 * ch < a.gn;
    uint16_t* p = static_cast<uint16_t*>(out) + (m0 + r0) * a.ldo + col0 + 8 * ch;
    const int64_t step = 8 * a.ldo;
#pragma unroll
    for (int i = 0; i < 4; ++i, p += step) {
      const int r = 8 * i + r0;
      const uint4 x = ld_shared_u4(buf + r * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
      if (col_ok && r < rows_left) *reinterpret_cast<uint4*>(p) = x;
    }
  }
}

// (add: a non-deterministic split unit's FP32 partial, added into the zero-filled
// output with atomic adds: 16-byte vector adds of whole 128-byte row segments, or
// for the transposed output coalesced scalar adds)
__device__ __forceinline__ void store_block32(const GemmArgs& a, void* out, uint32_t buf, int lane, int64_t m0,
                                              int64_t col0, const float (&v)[32], bool add = false) {
  if (a.out_trans) {
    store_row32(a, out, m0 + lane, col0, v, add);
    return;
  }
  stage_block32(a, buf, lane, v);
  flush_block32(a, out, buf, lane, m0, col0, add);
}

// Four output rows of a transposed store: D[m..m+3][col..col+3] (acc[i] = row m+i,
// columns col..col+3) go to out[(col+t)*ldo + m .. m+3], one 16-byte (FP32) or 8-byte
// (BF16) store per column.  m is a multiple of 4 and ldo, the output's base and its
// batch stride are 16-byte multiples, so every store is aligned.
__device__ __forceinline__ void store_trans4x4(const GemmArgs& a, void* out, int64_t m, int64_t col,
                                               const float4 (&acc)[4]) {
  const float c[4][4] = {{acc[0].x, acc[1].x, acc[2].x, acc[3].x},
                         {acc[0].y, acc[1].y, acc[2].y, acc[3].y},
                         {acc[0].z, acc[1].z, acc[2].z, acc[3].z},
                         {acc[0].w, acc[1].w, acc[2].w, acc[3].w}};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int64_t o = (col + t) * a.ldo + m;
    if (a.out_f32)
      *reinterpret_cast<float4*>(static_cast<float*>(out) + o) = make_float4(c[t][0], c[t][1], c[t][2], c[t][3]);
    else
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + o) =
          make_uint2(pack_bf16x2(c[t][0], c[t][1]), pack_bf16x2(c[t][2], c[t][3]));
  }
}

// acc = x (k == 0) or acc += x: the ordered sum's step.
__device__ __forceinline__ void sum_step(float4& acc, const float4& x, bool first) {
  if (first) {
    acc = x;
  } else {
    acc.x += x.x;
    acc.y += x.y;
    acc.z += x.z;
    acc.w += x.w;
  }
}

// In-kernel ordered sum for cluster plans: the S CTAs of a cluster computed the S
// splits of one tile (CTA rank r = split r, one unit each) and wrote their FP32
// partials.  After a cluster barrier (release / acquire, so every partial is
// visible), CTA r sums its rows of the tile, [4*floor(32r/S), 4*floor(32(r+1)/S)),
// over all S partials in ascending split order and rounds once: the same arithmetic
// as the reduction kernel, so the two give the same bits.  Row-major output: one
// float4 per step, consecutive threads on consecutive rows (512-byte partial reads).
// Transposed output (the swapped weight gradient): four rows per step, so each output
// column gets one 8- or 16-byte store instead of four element stores.
template <int BN>
__device__ __forceinline__ void cluster_fixup_sum(const GemmArgs& a, int nthreads) {
  __threadfence();
  cluster_sync();
  const int S = a.splits;
  const int u = static_cast<int>(blockIdx.x);  // this CTA's only unit
  const Unit w = decode_unit(a, u);
  const int r0 = 4 * (w.s * (kBlockM / 4) / S), r1 = 4 * ((w.s + 1) * (kBlockM / 4) / S), rows = r1 - r0;
  const int64_t m_tile = static_cast<int64_t>(w.tm) * kBlockM, n0 = static_cast<int64_t>(w.tn) * BN;
  const size_t pstride = static_cast<size_t>(kBlockM) * BN / 4;
  const float4* p0 = a.partials + static_cast<size_t>(w.ptile) * S * pstride;
  void* out = out_at(a, w.b);
  if (a.out_trans) {
    const int groups = rows / 4, total = groups * (BN / 4);
    for (int e = static_cast<int>(threadIdx.x); e < total; e += nthreads) {
      const int j4 = e / groups, row = r0 + 4 * (e - j4 * groups);
      const int64_t m = m_tile + row, col = n0 + 4 * j4;
      if (m >= a.gm || col >= a.gn) continue;  // (gm and gn are multiples of 4)
      const float4* src = p0 + static_cast<size_t>(j4) * kBlockM + row;
      float4 acc[4];
#pragma unroll
      for (int k0 = 0; k0 < 8; k0 += 4) {  // four splits' loads in flight at a time
        if (k0 >= S) break;
        float4 x[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (k0 + k < S) x[k][i] = __ldcg(src + (k0 + k) * pstride + i);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k0 + k < S)
#pragma unroll
            for (int i = 0; i < 4; ++i) sum_step(acc[i], x[k][i], k0 + k == 0);
      }
      store_trans4x4(a, out, m, col, acc);
    }
    return;
  }
  const int total = rows * (BN / 4);
  for (int e = static_cast<int>(threadIdx.x); e < total; e += nthreads) {
    const int j4 = e / rows, row = r0 + (e - j4 * rows);
    const int64_t m = m_tile + row, col = n0 + 4 * j4;
    if (m >= a.gm || col >= a.gn) continue;
    const float4* src = p0 + static_cast<size_t>(j4) * kBlockM + row;
    float4 x[8];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < S) x[k] = __ldcg(src + k * pstride);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < S) sum_step(acc, x[k], k == 0);
    if (a.out_f32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + m * a.ldo + col) = acc;
    } else {
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + m * a.ldo + col) =
          make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  }
}

// DUAL: a co-scheduled launch of two problems with MN-major B (see SecondProblem);
// each unit's A majorness comes from its problem's arguments.
template <int BN, bool A_MN, bool B_MN, bool PAIR, bool X3, bool DUAL>
__global__ void __launch_bounds__(TileCfg<BN, PAIR, X3>::THREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ GemmArgs args,
                     const __grid_constant__ SecondProblem<DUAL> second) {
  using C = TileCfg<BN, PAIR, X3>;
  static_assert(!DUAL || (B_MN && !X3), "co-scheduled problems: BF16, MN-major B");
  constexpr int STAGES = C::STAGES;
  constexpr int SSTAGES = C::SSTAGES;
  constexpr uint32_t IDESC = idesc_bf16_f32(C::TM, BN, A_MN, B_MN);
  constexpr uint32_t IDESC_AMN = idesc_bf16_f32(C::TM, BN, true, B_MN);  // (DUAL: MN-major A)
  constexpr uint32_t IDESC_TS = idesc_bf16_f32(C::TM, BN, false, B_MN);  // (A in tensor memory: K-major)
  const int total_units = args.units + second_units(second);
  // With PAIR, a cluster of two CTAs computes one TM x BN tile: rank r loads A rows
  // [r*128, r*128+128) and B rows [r*BN/2, (r+1)*BN/2) of the tile into the same
  // shared-memory offsets, the leader (rank 0) issues the 2-CTA MMAs, and rank r's
  // TMEM receives accumulator rows [r*128, r*128+128).
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int unit_step = PAIR ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle wants 1024-byte alignment
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sbase = base + STAGES * C::STAGE_BYTES;  // FP32 staging ring (X3)
  const uint32_t ebase = sbase + SSTAGES * C::SA_BYTES;   // epilogue output blocks
  const uint32_t bar0 = ebase + C::EPI_BYTES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + STAGES * C::STAGE_BYTES + SSTAGES * C::SA_BYTES +
                                                    C::EPI_BYTES + C::NUM_BARS * 8);
  volatile uint32_t* flag_wait = tmem_slot + 2;  // [2], double-buffered by unit parity

  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  auto sfull_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 5 + s); };             // X3 staging landed
  auto sempty_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 5 + SSTAGES + s); };  // X3 staging read

  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
  const int lane = static_cast<int>(threadIdx.x) & 31;
  if (threadIdx.x == 0) {  // descriptors on their way while the CTA sets up
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    if (X3) tma_prefetch_map(&tmB2);
    prefetch_second(second);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // X3: the B loads' arrival and one per converter warp; for a pair, the leader's
      // also takes one forwarded arrival from the peer, whose own full barriers only
      // collect its converters
      // (BF16: one expect-tx arrival from each of the A and B producer threads)
      mbar_init(full_bar(s), !X3 ? 2 : (PAIR && rank != 0) ? C::CONV_WARPS : 1 + C::CONV_WARPS + (PAIR ? 1 : 0));
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < SSTAGES; ++s) {
      mbar_init(sfull_bar(s), 1);
      mbar_init(sempty_bar(s), C::CONV_WARPS);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), PAIR ? 8 : 4);  // one arrival per epilogue warp (of both CTAs)
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(smem_addr(tmem_slot), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR)
    cluster_sync();  // both CTAs' barriers are initialised before either signals the other
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0 || (C::B_WARP && warp == C::B_WARP_ID)) {
    // ------------------------------------------------------------ producer(s)
    if (lane == 0) {
      int stage = 0, sstage = 0;
      uint32_t phase = 0, sphase = 0;
      const uint64_t pol_ef = l2_policy_evict_first();  // (for operands read once: evict_first)
      // per-stage bit masks of issued loads and their phases, for the final drain
      uint32_t issued = 0, issued_phase = 0, sissued = 0, sissued_phase = 0;
      bool ok = true;
      if (X3) {
        // Two cursors walk the same (unit, k-block) sequence: the FP32 staging loads
        // of A run ahead as far as the staging ring allows (DRAM latency), B's bf16
        // hi/lo loads as far as the MMA ring allows; neither waits for the other.
        // (each cursor walks this slot's units -- or, for a stream-K plan, the pieces of
        // its block range -- in order; k is the index in that list)
        struct Cursor {
          int k, kb, kb1, tm, tn;
          bool done;
        };
        auto seek = [&](Cursor& c, int k) {
          for (c.k = k;; ++c.k) {
            UnitRef ur;
            Unit w;
            if (!slot_unit(c.k, unit0, unit_step, total_units, args, tmA, tmB, second, &ur, &w)) {
              c.done = true;
              return;
            }
            c.kb = w.kb0;
            c.kb1 = w.kb1;
            c.tm = w.tm;
            c.tn = w.tn;
            c.done = false;
            if (c.kb < c.kb1) return;
          }
        };
        auto next = [&](Cursor& c) {
          if (++c.kb == c.kb1) seek(c, c.k + 1);
        };
        Cursor xc, bc, fc;
        seek(xc, 0);
        seek(bc, 0);
        seek(fc, 0);
        // (with B_WARP: warp 0 walks A's cursor only, warp B_WARP_ID B's only, and each
        // tests its one barrier with try_wait, which may suspend the thread briefly,
        // instead of test_wait's pure poll)
        if (C::B_WARP) {
          if (warp == 0)
            bc.done = true;
          else
            xc.done = true;
        }
        auto poll = [&](uint32_t bar, uint32_t parity) {
          return C::B_WARP ? mbar_test(bar, parity) : mbar_peek(bar, parity);
        };
        // (a pair's peer: one arrival on the leader's full barrier per stage, once this
        // CTA's converters have filled it)
        const bool forward = PAIR && rank != 0;
        int fstage = 0;
        uint32_t fphase = 0;
        if (!forward) fc.done = true;
        uint32_t idle = 0;
        uint64_t t_idle = 0;
        // The staging ring is filled first: A (FP32, the caller's) does not depend on
        // the split kernel, so its loads overlap that kernel's tail.
        bool b_ready = false;
        int issued_x = 0;
        while (!xc.done || !bc.done || !fc.done) {
          if (xc.done) issued_x = SSTAGES;  // (fewer blocks than staging slots)
          bool progressed = false;
          if (!xc.done && poll(sempty_bar(sstage), sphase ^ 1u)) {
            const uint32_t xa = sbase + sstage * C::SA_BYTES;
            const uint32_t xf = sfull_bar(sstage);
            const int a_row0 = xc.tm * C::TM + static_cast<int>(rank) * C::BM;
            mbar_expect_tx(xf, C::SA_BYTES);
            const bool ha = !PAIR && (args.evict_first & 1);
            auto sload2 = [&](uint32_t dst, int32_t x, int32_t y) {
              if (ha)
                tma_load_2d_hint(dst, &tmA, xf, x, y, pol_ef);
              else
                tma_load_2d(dst, &tmA, xf, x, y);
            };
            if (A_MN && args.a3d) {
              if (ha)
                tma_load_3d_hint(xa, &tmA, xf, 0, xc.kb * C::BK, a_row0 / 32, pol_ef);
              else
                tma_load_3d(xa, &tmA, xf, 0, xc.kb * C::BK, a_row0 / 32);
            } else if (A_MN) {
#pragma unroll
              for (int j = 0; j < C::BM / 32; ++j) sload2(xa + 4096 * j, a_row0 + 32 * j, xc.kb * C::BK);
            } else {
              sload2(xa, xc.kb * C::BK, a_row0);
            }
            sissued |= 1u << sstage;
            sissued_phase = (sissued_phase & ~(1u << sstage)) | (sphase << sstage);
            if (++sstage == SSTAGES) {
              sstage = 0;
              sphase ^= 1u;
            }
            next(xc);
            ++issued_x;
            progressed = true;
          }
          if (!bc.done && !b_ready && issued_x >= SSTAGES) {
            pdl_wait();  // B's planes come from the split kernel launched before this grid
            b_ready = true;
          }
          if (b_ready && !bc.done &&
              (PAIR ? mbar_peek_cluster(empty_bar(stage), phase ^ 1u) : poll(empty_bar(stage), phase ^ 1u))) {
            const uint32_t sb = base + stage * C::STAGE_BYTES + C::A_BYTES;
            // a pair's B loads all complete on the leader's full barrier
            const uint32_t fb = PAIR ? map_shared_rank(full_bar(stage), 0) : full_bar(stage);
            const int b_row0 = bc.tn * BN + static_cast<int>(rank) * C::BNH;
            if (rank == 0) mbar_expect_tx(full_bar(stage), (PAIR ? 2 : 1) * C::B_BYTES);
            const bool hb = !PAIR && (args.evict_first & 2);
            auto load2 = [&](uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y) {
              if (PAIR)
                tma_load_2d_pair(dst, map, fb, x, y);
              else if (hb)
                tma_load_2d_hint(dst, map, fb, x, y, pol_ef);
              else
                tma_load_2d(dst, map, fb, x, y);
            };
            auto load3 = [&](uint32_t dst, const CUtensorMap* map, int32_t y, int32_t z) {
              if (PAIR)
                tma_load_3d_pair(dst, map, fb, 0, y, z);
              else if (hb)
                tma_load_3d_hint(dst, map, fb, 0, y, z, pol_ef);
              else
                tma_load_3d(dst, map, fb, 0, y, z);
            };
            if (B_MN && args.b3d) {
              // 64-column groups of 32 contraction rows (4 KB each, 128-byte swizzle)
              load3(sb, &tmB, bc.kb * C::BK, b_row0 / 64);
              load3(sb + C::B_HALF, &tmB2, bc.kb * C::BK, b_row0 / 64);
            } else if (B_MN) {
#pragma unroll
              for (int j = 0; j < C::BNH / 64; ++j) {
                load2(sb + 4096 * j, &tmB, b_row0 + 64 * j, bc.kb * C::BK);
                load2(sb + C::B_HALF + 4096 * j, &tmB2, b_row0 + 64 * j, bc.kb * C::BK);
              }
            } else {
              // rows of 32 contraction elements (64 bytes, 64-byte swizzle)
              load2(sb, &tmB, bc.kb * C::BK, b_row0);
              load2(sb + C::B_HALF, &tmB2, bc.kb * C::BK, b_row0);
            }
            issued |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            next(bc);
            progressed = true;
          }
          if (!fc.done && mbar_peek(full_bar(fstage), fphase)) {
            mbar_arrive_cluster(map_shared_rank(full_bar(fstage), 0));
            if (++fstage == STAGES) {
              fstage = 0;
              fphase ^= 1u;
            }
            next(fc);
            progressed = true;
          }
          // bounded: give up once neither ring has moved for the wait limit
          if (progressed) {
            idle = 0;
          } else if ((++idle & 255u) == 1u) {
            const uint64_t now = globaltimer_ns();
            if (idle == 1u) {
              t_idle = now;
            } else if (now - t_idle > args.wait_ns) {
              atomicOr(args.fault, kFaultProducerWait);
              ok = false;
              break;
            }
          }
        }
      }
      if (!X3) pdl_wait();  // the previous kernel on the stream (launched as its dependent) is done
      // (BF16: warp 0 loads A, warp B_WARP_ID loads B, each counting its own bytes)
      const bool load_a = warp == 0, load_b = warp != 0;
      const int kps = (X3 || args.kps != 2) ? 1 : 2;
      const int nst = STAGES / kps;  // stages of the ring, kps block slots each
      for (int k = 0; !X3 && ok; ++k) {
        UnitRef ur;
        Unit w;
        if (!slot_unit(k, unit0, unit_step, total_units, args, tmA, tmB, second, &ur, &w)) break;
        // (one problem: the kernel's own parameters, read from the parameter space)
        const GemmArgs& ga = DUAL ? *ur.a : args;
        const CUtensorMap* mapA = DUAL ? ur.mA : &tmA;
        const CUtensorMap* mapB = DUAL ? ur.mB : &tmB;
        const bool a_mn = DUAL ? ga.a_mn != 0 : A_MN;
        const int a_row0 = w.tm * C::TM + static_cast<int>(rank) * C::BM;
        const int b_row0 = w.tn * BN + static_cast<int>(rank) * C::BNH;
        for (int kbs = w.kb0; kbs < w.kb1; kbs += kps) {
          const int nb = min(kps, w.kb1 - kbs);  // blocks in this stage
          if (!mbar_wait<PAIR>(empty_bar(stage), phase ^ 1u, args.wait_ns)) {
            atomicOr(args.fault, kFaultProducerWait);
            ok = false;
            break;
          }
          // a pair's loads all complete on the leader's full barrier
          const uint32_t fb = PAIR ? map_shared_rank(full_bar(stage), 0) : full_bar(stage);
          if (rank == 0)
            mbar_expect_tx(full_bar(stage),
                           (PAIR ? 2 : 1) * nb * ((load_a ? C::A_BYTES : 0) + (load_b ? C::B_BYTES : 0)));
          // (batched plans: every map has a trailing batch dimension; `hint`: the operand
          // is read once by the launch, loaded with the evict-first policy)
          auto load = [&](uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, bool hint) {
            if (ga.batch > 1) {
              if (PAIR)
                tma_load_3d_pair(dst, map, fb, x, y, w.b);
              else if (hint)
                tma_load_3d_hint(dst, map, fb, x, y, w.b, pol_ef);
              else
                tma_load_3d(dst, map, fb, x, y, w.b);
            } else if (PAIR) {
              tma_load_2d_pair(dst, map, fb, x, y);
            } else if (hint) {
              tma_load_2d_hint(dst, map, fb, x, y, pol_ef);
            } else {
              tma_load_2d(dst, map, fb, x, y);
            }
          };
          auto load3 = [&](uint32_t dst, const CUtensorMap* map, int32_t y, int32_t z, bool hint) {
            if (PAIR)
              tma_load_3d_pair(dst, map, fb, 0, y, z);
            else if (hint)
              tma_load_3d_hint(dst, map, fb, 0, y, z, pol_ef);
            else
              tma_load_3d(dst, map, fb, 0, y, z);
          };
          const bool ha = (ga.evict_first & 1) != 0, hb = (ga.evict_first & 2) != 0;
          for (int j = 0; j < nb; ++j) {
            const int kb = kbs + j;
            const uint32_t sa = base + (stage * kps + j) * C::STAGE_BYTES;
            const uint32_t sb = sa + C::A_BYTES;
            // MN-major: 64-column groups of 64 contraction rows (8 KB each)
            if (!load_a) {
            } else if (a_mn && ga.a3d) {
              load3(sa, mapA, kb * C::BK, a_row0 / 64, ha);
            } else if (a_mn) {
              load(sa, mapA, a_row0, kb * C::BK, ha);
              load(sa + 8192, mapA, a_row0 + 64, kb * C::BK, ha);
            } else {
              load(sa, mapA, kb * C::BK, a_row0, ha);
            }
            if (!load_b) {
            } else if (B_MN && ga.b3d) {
              load3(sb, mapB, kb * C::BK, b_row0 / 64, hb);
            } else if (B_MN) {
#pragma unroll
              for (int g = 0; g < C::BNH / 64; ++g) load(sb + 8192 * g, mapB, b_row0 + 64 * g, kb * C::BK, hb);
            } else {
              load(sb, mapB, kb * C::BK, b_row0, hb);
            }
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // The grid launched after this one on the stream (the split reduction, or the
      // next call's kernel) may start its launch once every CTA has issued its last
      // loads: early enough to hide that launch behind this grid's last MMAs and
      // epilogue, late enough that its CTAs do not sit on this grid's SMs for the
      // whole main loop (measured on GB300 against a trigger right after setup: the
      // T = 64 forward 10.2 -> 9.7 us, fwd + fwd + bwd at T = 1024, 4096 -> 1024,
      // 71.1 -> 67.4 us; the large calls unchanged).  (With B_WARP: the thread that
      // loads B, whose loads come last.)
      if (!C::B_WARP || warp != 0) pdl_launch_dependents();
      // Every load this thread issued has landed before the CTA may exit: on the
      // stage's full barrier, or for a pair (whose loads complete on the leader's
      // barrier) on the empty barrier the leader's MMAs release after reading it.
      // (X3: the staging tiles on their own full barriers.)
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u) {
          const uint32_t par = (issued_phase >> s) & 1u;
          const bool landed = PAIR ? mbar_wait<true>(empty_bar(s), par, args.wait_ns)
                                   : mbar_wait(full_bar(s), par, args.wait_ns);
          if (!landed) atomicOr(args.fault, kFaultDrainWait);
        }
      for (int s = 0; s < SSTAGES; ++s)
        if ((sissued >> s) & 1u) {
          if (!mbar_wait(sfull_bar(s), (sissued_phase >> s) & 1u, args.wait_ns)) atomicOr(args.fault, kFaultDrainWait);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      const int kps = (X3 || args.kps != 2) ? 1 : 2;
      const int nst = STAGES / kps;
      for (int k = 0; ok; ++k, ++local) {
        UnitRef ur;
        Unit w;
        if (!slot_unit(k, unit0, unit_step, total_units, args, tmA, tmB, second, &ur, &w)) break;
        const bool a_mn = DUAL ? ur.a->a_mn != 0 : A_MN;  // (one problem: the template's)
        const uint32_t idesc = (DUAL && a_mn) ? IDESC_AMN : IDESC;
        const int kb0 = w.kb0, kb1 = w.kb1;
        const int acc = C::NACC == 2 ? (local & 1) : 0;
        const uint32_t aph = C::NACC == 2 ? ((local >> 1) & 1) : (local & 1);
        if (!mbar_wait<PAIR>(tempty_bar(acc), aph ^ 1u, args.wait_ns)) {
          atomicOr(args.fault, kFaultMmaWait);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kbs = kb0; kbs < kb1; kbs += kps) {
          if (!mbar_wait<PAIR>(full_bar(stage), phase, args.wait_ns)) {
            atomicOr(args.fault, kFaultMmaWait);
            ok = false;
            break;
          }
          tc_fence_after();
          const int nb = min(kps, kb1 - kbs);
          for (int j = 0; j < nb; ++j) {
            const int kb = kbs + j;
            const uint32_t sa = base + (stage * kps + j) * C::STAGE_BYTES;
            const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
            for (int kk = 0; kk < C::BK / 16; ++kk) {
              if (X3) {
                // bf16 hi/lo tiles, 32 contraction elements: K-major rows are 64 bytes
                // (64-byte swizzle, 8-row groups 512 B apart, step 32 B per 16 elements);
                // MN-major tiles keep 128-byte rows (64-element groups 4 KB apart).
                auto d_a = [&](uint32_t t) {
                  return A_MN ? sdesc(t + kk * 2048, 4096, 1024, 2) : sdesc(t + kk * 32, 16, 512, 4);
                };
                auto d_b = [&](uint32_t t) {
                  return B_MN ? sdesc(t + kk * 2048, 4096, 1024, 2) : sdesc(t + kk * 32, 16, 512, 4);
                };
                if constexpr (C::A_TMEM) {
                  // A's halves of this stage in tensor memory: hi in columns [0, 16), lo in
                  // [16, 32); 8 columns (16 contraction elements) per MMA
                  const uint32_t a_t = tmem_base + static_cast<uint32_t>(C::A_TMEM_COL + stage * 32 + kk * 8);
                  const uint64_t b_hi = d_b(sb), b_lo = d_b(sb + C::B_HALF);
                  mma_bf16_ts(d_tmem, a_t + 16, b_hi, IDESC_TS, (kb > kb0 || kk > 0) ? 1u : 0u);
                  mma_bf16_ts(d_tmem, a_t, b_lo, IDESC_TS, 1u);
                  mma_bf16_ts(d_tmem, a_t, b_hi, IDESC_TS, 1u);
                  continue;
                }
                const uint64_t a_hi = d_a(sa), a_lo = d_a(sa + C::A_HALF);
                const uint64_t b_hi = d_b(sb), b_lo = d_b(sb + C::B_HALF);
                // x*w ~ lo_x*hi_w + hi_x*lo_w + hi_x*hi_w (lo*lo dropped), small terms first
                if (PAIR) {
                  mma_bf16_pair(d_tmem, a_lo, b_hi, IDESC, (kb > kb0 || kk > 0) ? 1u : 0u);
                  mma_bf16_pair(d_tmem, a_hi, b_lo, IDESC, 1u);
                  mma_bf16_pair(d_tmem, a_hi, b_hi, IDESC, 1u);
                } else {
                  mma_bf16(d_tmem, a_lo, b_hi, IDESC, (kb > kb0 || kk > 0) ? 1u : 0u);
                  mma_bf16(d_tmem, a_hi, b_lo, IDESC, 1u);
                  mma_bf16(d_tmem, a_hi, b_hi, IDESC, 1u);
                }
                continue;
              }
              // K-major: step 16 elements (32 bytes) along the swizzled row;
              // MN-major: step 16 contraction rows (16 x 128 bytes).
              const uint64_t ad = a_mn ? sdesc_sw128(sa + kk * 2048, 8192, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? sdesc_sw128(sb + kk * 2048, 8192, 1024) : sdesc_sw128(sb + kk * 32, 16, 1024);
              if (PAIR)
                mma_bf16_pair(d_tmem, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
              else
                mma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
            }
          }
          // frees the stage (in both CTAs of a pair) once these MMAs have read it
          if (PAIR)
            mma_commit_pair_multicast(empty_bar(stage), 0x3);
          else
            mma_commit(empty_bar(stage));
          if (++stage == nst) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator complete (in both CTAs' TMEM for a pair)
        if (PAIR)
          mma_commit_pair_multicast(tfull_bar(acc), 0x3);
        else
          mma_commit(tfull_bar(acc));
      }
      // Every MMA this thread issued has finished before TMEM is freed.
      if (PAIR)
        mma_commit_pair(drain_bar);
      else
        mma_commit(drain_bar);
      if (!mbar_wait(drain_bar, 0, args.wait_ns)) atomicOr(args.fault, kFaultDrainWait);
    }
  } else if (X3 && (warp == 2 || warp == 3 || warp == 8 || warp == 9)) {
    // ------------------------------------------------------------ converter (X3)
    // Turns each FP32 staging tile of A into the bf16 hi/lo A tiles of an MMA stage:
    // hi = RNE(x), lo = RNE(x - hi) (x - hi is exact), written in the tensor core's
    // swizzled layout.  A task is one 16-byte bf16 chunk (8 elements) of A, read
    // from two 16-byte FP32 chunks:
    //   K-major: FP32 rows of 128 B (128-byte swizzle) -> bf16 rows of 64 B
    //            (64-byte swizzle); chunk c of row r <- FP32 chunks 2c, 2c+1 of row r;
    //   MN-major: FP32 boxes of 32 elements x 32 contraction rows (4 KB, 128-byte
    //            swizzle) -> bf16 groups of 64 elements x 32 rows (4 KB, 128-byte
    //            swizzle).
    // The 512 tasks of a stage are dealt round-robin to the 128 converter threads;
    // their shared-memory offsets do not depend on the stage, so they are computed
    // once, and each thread loads all of its chunks before converting any.
    // Single CTAs (A_TMEM) write the halves into tensor memory instead: thread i of
    // warp w converts row 32 (w % 4) + i (the TMEM lane quarter warp w may access) and
    // stores its 32 hi and 32 lo values as two 16-column rows of the stage's columns.
    if constexpr (C::A_TMEM) {
      const int sub = warp & 3;
      const int r = sub * 32 + lane;  // row of A == TMEM lane
      const uint32_t trow = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + static_cast<uint32_t>(C::A_TMEM_COL);
      // this thread's FP32 row in a staging tile -- K-major: 8 16-byte chunks of row r,
      // chunk j at j ^ (r % 8); MN-major: element (k, r) of the 32 x 32 box r / 32, at row
      // k, 16-byte chunk (r % 32) / 4 ^ (k % 8), word r % 4
      const uint32_t kmaj_row = static_cast<uint32_t>(r) * 128u;
      const uint32_t mn_col = static_cast<uint32_t>(r >> 5) * 4096u + static_cast<uint32_t>(r & 3) * 4u;
      const int mn_c4 = (r & 31) >> 2;
      int stage = 0, sstage = 0;
      uint32_t phase = 0, sphase = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        UnitRef ur;
        Unit w;
        if (!slot_unit(k, unit0, unit_step, total_units, args, tmA, tmB, second, &ur, &w)) break;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          // every lane waits itself; the warp leaves together if any wait gives up
          const bool mine = mbar_wait(sfull_bar(sstage), sphase, args.wait_ns) &&
                             mbar_wait(empty_bar(stage), phase ^ 1u, args.wait_ns);
          if (!__all_sync(0xffffffffu, mine)) {
            if (lane == 0) atomicOr(args.fault, kFaultProducerWait);
            ok = false;
            break;
          }
          const uint32_t xs = sbase + sstage * C::SA_BYTES;
          float4 v[8];
          if (A_MN) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              float e[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int kk = 4 * j + q;
                e[q] = ld_shared_f32(xs + mn_col + kk * 128 + ((mn_c4 ^ (kk & 7)) << 4));
              }
              v[j] = make_float4(e[0], e[1], e[2], e[3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = ld_shared_f4(xs + kmaj_row + ((j ^ (r & 7)) << 4));
          }
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 h, l;
            split8_bf16x3(v[2 * j], v[2 * j + 1], h, l);
            hi[4 * j] = h.x, hi[4 * j + 1] = h.y, hi[4 * j + 2] = h.z, hi[4 * j + 3] = h.w;
            lo[4 * j] = l.x, lo[4 * j + 1] = l.y, lo[4 * j + 2] = l.z, lo[4 * j + 3] = l.w;
          }
          const uint32_t ta = trow + static_cast<uint32_t>(stage * 32);
          tmem_st_32x32b_x16(ta, hi);
          tmem_st_32x32b_x16(ta + 16, lo);
          tmem_wait_st();     // the halves are in tensor memory
          tc_fence_before();  // ... before the arrival that lets the MMAs read them
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(sempty_bar(sstage));  // staging tile may be reloaded
            mbar_arrive(full_bar(stage));     // this warp's quarter of A is ready
          }
          if (++sstage == SSTAGES) {
            sstage = 0;
            sphase ^= 1u;
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else {
    constexpr int NCT = (X3 ? C::CONV_WARPS : 4) * 32;  // (the branch only runs with X3)
    constexpr int kTasks = 512 / NCT;
    static_assert(512 % NCT == 0, "converter tasks");
    const int ctid = (warp < 4 ? warp - 2 : warp - 6) * 32 + lane;
    uint32_t src0[kTasks], src1[kTasks], dsto[kTasks];
#pragma unroll
    for (int b = 0; b < kTasks; ++b) {
      const int t = ctid + NCT * b;
      if (A_MN) {
        const int k = t >> 4, q = t & 15;  // contraction row, chunk along the 128 rows
        const int g = q >> 3, c = q & 7;
        const uint32_t row = (2 * g + (c >> 2)) * 4096 + k * 128;
        const int j0 = 2 * (c & 3);
        src0[b] = row + ((j0 ^ (k & 7)) << 4);
        src1[b] = row + (((j0 + 1) ^ (k & 7)) << 4);
        dsto[b] = g * 4096 + k * 128 + ((c ^ (k & 7)) << 4);
      } else {
        const int r = t >> 2, c = t & 3;
        src0[b] = r * 128 + (((2 * c) ^ (r & 7)) << 4);
        src1[b] = r * 128 + (((2 * c + 1) ^ (r & 7)) << 4);
        dsto[b] = r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
      }
    }
    int stage = 0, sstage = 0;
    uint32_t phase = 0, sphase = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      UnitRef ur;
      Unit w;
      if (!slot_unit(k, unit0, unit_step, total_units, args, tmA, tmB, second, &ur, &w)) break;
      for (int kb = w.kb0; kb < w.kb1; ++kb) {
        // every lane waits itself; the warp leaves together if any wait gives up
        const bool mine = mbar_wait(sfull_bar(sstage), sphase, args.wait_ns) &&
                           mbar_wait<PAIR>(empty_bar(stage), phase ^ 1u, args.wait_ns);
        if (!__all_sync(0xffffffffu, mine)) {
          if (lane == 0) atomicOr(args.fault, kFaultProducerWait);
          ok = false;
          break;
        }
        const uint32_t xs = sbase + sstage * C::SA_BYTES;
        const uint32_t ah = base + stage * C::STAGE_BYTES, al = ah + C::A_HALF;
        float4 x0[kTasks], x1[kTasks];
#pragma unroll
        for (int b = 0; b < kTasks; ++b) {
          x0[b] = ld_shared_f4(xs + src0[b]);
          x1[b] = ld_shared_f4(xs + src1[b]);
        }
#pragma unroll
        for (int b = 0; b < kTasks; ++b) {
          uint4 h, l;
          split8_bf16x3(x0[b], x1[b], h, l);
          st_shared_u4(ah + dsto[b], h);
          st_shared_u4(al + dsto[b], l);
        }
        fence_proxy_async_shared();  // the tensor core reads what this thread wrote
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(sempty_bar(sstage));  // staging tile may be reloaded
          // A half of the bf16 stage ready (a pair's peer forwards it to the leader)
          mbar_arrive(full_bar(stage));
        }
        if (++sstage == SSTAGES) {
          sstage = 0;
          sphase ^= 1u;
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    }  // (A in shared memory)
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM sub-partition this warp may read
    const int row = q * 32 + lane;   // accumulator row == TMEM lane
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t ebuf = ebase + q * (4096 * C::EPI_BUFS);  // this warp's output block(s)
    // TMA-store staging: the block the next store stages in (alternating when there are
    // two), and whether the most recent bulk store, from the other block, may still be
    // reading it
    int sbuf = 0;
    bool store_pending = false;
    const bool leader = threadIdx.x == 128;
    int local = 0;
    // the epilogue warps (of both CTAs of a pair) release the accumulator on the
    // leader's barrier, once their tensor-memory reads have completed (tmem_wait_ld)
    auto release_acc = [&](int a) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_remote(map_shared_rank(tempty_bar(a), 0));
        else
          mbar_arrive(tempty_bar(a));
      }
    };
    for (int k = 0;; ++k, ++local) {
      UnitRef ur;
      Unit w;
      if (!slot_unit(k, unit0, unit_step, total_units, args, tmA, tmB, second, &ur, &w)) break;
      const GemmArgs& ga = DUAL ? *ur.a : args;  // (one problem: the kernel's own parameters)
      const int tm = w.tm, tn = w.tn;
      const int slot = w.ptile * (PAIR ? 2 : 1) + static_cast<int>(rank);  // this CTA's partial slot
      const int acc = C::NACC == 2 ? (local & 1) : 0;
      const uint32_t aph = C::NACC == 2 ? ((local >> 1) & 1) : (local & 1);
      // One thread waits; the outcome reaches the other 127 through a named barrier,
      // so all of them leave together if the wait gives up.
      if (leader) {
        const bool ready = mbar_wait<PAIR>(tfull_bar(acc), aph, args.wait_ns);
        if (!ready) atomicOr(args.fault, kFaultEpilogueWait);
        flag_wait[local & 1] = ready ? 1u : 0u;
      }
      named_sync(1, 128);
      if (flag_wait[local & 1] == 0u) break;
      tc_fence_after();
      const int64_t m = static_cast<int64_t>(tm) * C::TM + static_cast<int64_t>(rank) * C::BM + row;
      const int64_t m0 = m - lane;  // row of lane 0
      void* outb = out_at(ga, w.b);
      const int64_t n0 = static_cast<int64_t>(tn) * BN;
      const uint32_t tcol = lane_addr + static_cast<uint32_t>(acc * BN);
      if ((!w.split && !ga.tma_store) || (w.split && ga.atomic)) {
        // (the warp's own stores; a split unit here is a non-deterministic plan's, added
        // into the zero-filled output.  Its staging waits for earlier bulk stores to
        // have read the block.)
        if (ga.tma_store && lane == 0) bulk_wait_group_read0();
        store_pending = false;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tcol + c * 32, r);
          tmem_wait_ld();
          if (c == BN / 32 - 1) release_acc(acc);  // accumulator may be reused
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          store_block32(ga, outb, ebuf, lane, m0, n0 + c * 32, v, w.split);
        }
      } else if (C::EPI_BUFS == 2 && !w.split && ga.tma_store2 && !ga.epi_single) {
        // FP32 through the [32-column block][row][32] view: both staging blocks of the warp,
        // side by side, leave as one 3-D box (8 KB per TMA store: issuing a store took
        // ~280-800 cycles of the ~900 a 4 KB block cost); they are restaged once that
        // store has read them
#pragma unroll 1
        for (int c = 0; c < BN / 32; c += 2) {
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(tcol + c * 32, r0);
          tmem_ld_32x32b_x32(tcol + (c + 1) * 32, r1);
          tmem_wait_ld();
          if (c + 2 == BN / 32) release_acc(acc);  // accumulator may be reused
          if (lane == 0) bulk_wait_group_read0();
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r0[j]);
          stage_block32(ga, ebuf, lane, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r1[j]);
          stage_block32(ga, ebuf + 4096u, lane, v);
          fence_proxy_async_shared();
          __syncwarp();
          const int32_t z = static_cast<int32_t>((n0 + c * 32) / 32), y = static_cast<int32_t>(m0);
          if (lane == 0 && y < ga.gm && static_cast<int64_t>(z) * 32 < ga.gn) {
            tma_store_3d(&ga.tmO2, ebuf, 0, y, z);
            bulk_commit_group();
          }
        }
        // (a store from both blocks may be in flight: the next staging waits for it)
        store_pending = false;
        sbuf = 0;
      } else if (!w.split) {
        // Stage and hand to TMA (which clips rows >= gm, columns >= gn) 4 KB at a
        // time: an FP32 32 x 32 block, or two BF16 32 x 32 blocks side by side (32
        // rows of 128 bytes).  A staging block is rewritten only once the bulk store
        // that last used it has read it: with two blocks, every store but the most
        // recent (which used the other block) has; with one, every store.
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tcol + c * 32, r);
          tmem_wait_ld();
          if (c == BN / 32 - 1) release_acc(acc);  // accumulator may be reused
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          const int h = ga.out_f32 ? 0 : (c & 1);
          const uint32_t sb = ebuf + static_cast<uint32_t>(sbuf) * 4096u;
          if (h == 0 && lane == 0) {
            if (C::EPI_BUFS == 2 && !ga.epi_single && store_pending)
              bulk_wait_group_read1();
            else
              bulk_wait_group_read0();
          }
          if (ga.out_f32)
            stage_block32(ga, sb, lane, v);
          else
            stage_half64_bf16(sb, lane, h, v);
          if (ga.out_f32 || h == 1) {
            fence_proxy_async_shared();
            __syncwarp();
            const int32_t x = static_cast<int32_t>(n0 + (c - h) * 32), y = static_cast<int32_t>(m0);
            const bool inside = x < ga.gn && y < ga.gm;  // (blocks wholly outside: nothing to store)
            if (lane == 0 && inside) {
              if (ga.batch > 1)
                tma_store_3d(&ga.tmO, sb, x, y, w.b);
              else
                tma_store_2d(&ga.tmO, sb, x, y);
              bulk_commit_group();
            }
            store_pending = inside;
            if (C::EPI_BUFS == 2 && !ga.epi_single) sbuf ^= 1;
          }
        }
      } else {
        // FP32 partial of this split, laid out [BN/4][128] float4 so a warp's
        // 32 rows write 512 contiguous bytes.
        float4* part = ga.partials + (static_cast<size_t>(slot) * ga.splits + w.s) * (C::BM * BN / 4);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tcol + c * 32, r);
          tmem_wait_ld();
          if (c == BN / 32 - 1) release_acc(acc);
          if (m < ga.gm) {  // padding rows of a thin tile are never read back
#pragma unroll
            for (int j = 0; j < 8; ++j)
              __stcg(&part[(c * 8 + j) * C::BM + row],
                     make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                 __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])));
          }
        }
      }
    }
    // this warp's bulk stores have completed before the CTA (and its shared memory) goes
    if (lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncwarp();
  if (PAIR)
    cluster_sync();  // neither CTA leaves while the leader's MMAs may still use the peer
  else
    __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
  if (!PAIR && !DUAL && args.cluster_fixup > 1) cluster_fixup_sum<BN>(args, C::THREADS);
}

// Host-side launch of one instantiation (defined in the per-view .cu files).
struct GemmLaunch {
  CUtensorMap tmA, tmB;
  CUtensorMap tmB2;  // X3: B's bf16 lo plane (tmB is the hi plane); otherwise unused
  GemmArgs args;
  SecondProblem<true> second;  // co-scheduled launches: the second problem
  int grid;   // CTAs (twice the number of pairs for a paired plan)
  bool pair;  // clusters of two CTAs share each tile
  bool x3;    // router BF16x3 mode: FP32 A split in the kernel, B from pre-split planes
  bool pdl;   // launched as a programmatic dependent of the previous kernel on the stream
};

// Clusters of `cluster` single-CTA tiles of width bn that run at once (0 if none).
int max_clusters_kk(int bn, bool x3, int cluster, int grid);
int max_clusters_km(int bn, int cluster, int grid);
int max_clusters_mm(int bn, bool x3, int cluster, int grid);
cudaError_t launch_gemm_kk(int bn, const GemmLaunch& l, cudaStream_t stream);  // forward
cudaError_t launch_gemm_km(int bn, const GemmLaunch& l, cudaStream_t stream);  // input gradient
cudaError_t launch_gemm_mm(int bn, const GemmLaunch& l, cudaStream_t stream);  // weight gradient
// Input gradient and weight gradient co-scheduled in one launch (gemm_bwd.cu):
// l.args / l.tmA / l.tmB the problem whose units come first, l.second the other.
cudaError_t launch_gemm_bwd(int bn, bool pair, const GemmLaunch& l, cudaStream_t stream);
cudaError_t set_attributes_bwd();
// Router operand split: the bf16 hi/lo copies the BF16x3 GEMMs read (split_x3.cu).
struct SplitJob {
  const float* x;       // FP32 [rows][cols], leading dimension ldx (multiple of 4)
  uint16_t* out;        // segment s of row r starts at out + s * seg_stride + r * ldo
  int64_t rows, cols, ldx, ldo, seg_stride;
  int32_t nseg;         // 2 or 3 segments
  uint32_t lo_mask;     // bit s set: segment s holds lo = RNE(x - hi), else hi = RNE(x)
};
// (zero, if not null: also zero-fill that FP32 [rows][cols] matrix, leading
// dimension ld, in the same launch: the output of a non-deterministic router call)
struct ZeroJob {
  float* out;
  int64_t rows, cols, ld;
};
cudaError_t launch_split_x3(const SplitJob* jobs, int njobs, int sm_count, cudaStream_t stream,
                            const ZeroJob* zero = nullptr);
// Small-T FP32 router program (router_ffma.cu): D[m][n] = sum_k A(m, k) B(n, k) on
// FP32 operands with FP32 FMAs; 64 x bn tiles (bn 16 / 32 / 64), each tile's
// contraction split over a cluster of `splits` CTAs (<= 8) whose partials are
// summed in rank order.  K-major operands are [rows][k] matrices, MN-major ones
// [k][rows] (leading dimensions in elements, multiples of 4, 16-byte aligned).
struct FfmaArgs {
  const float* a;
  const float* b;
  float* out;          // [gm][gn], leading dimension ldo
  int64_t lda, ldb, ldo;
  int64_t gm, gn, gk;
  int32_t tiles_n;     // ceil(gn / bn)
  int32_t splits;      // CTAs per tile (cluster size)
  int32_t kchunks;     // ceil(gk / (4096 / bn)): contraction chunks of one stage
};
constexpr int ffma_stage_k(int bn) { return 4096 / bn; }  // 16 elements x (256 / bn) contraction groups
cudaError_t launch_router_ffma(int bn, bool a_mn, bool b_mn, const FfmaArgs& a, cudaStream_t stream);
cudaError_t set_attributes_ffma();
// Ordered sum of the split partials a GEMM launch wrote (split_reduce.cu): for each
// split tile, partials s = 0..splits-1 added in that order in FP32, rounded once.
cudaError_t launch_split_reduce(const GemmLaunch& l, int bn, bool pair, int64_t split_tiles, cudaStream_t stream);
// Shared-memory carveout of the split and reduction kernels (set once per device).
cudaError_t set_attributes_split();
cudaError_t set_attributes_reduce();
// Dynamic shared memory limits of each instantiation, on the current device.
cudaError_t set_attributes_kk();
cudaError_t set_attributes_km();
cudaError_t set_attributes_mm();

inline SecondProblem<false> second_of(const GemmLaunch&, std::false_type) { return SecondProblem<false>{0}; }
inline const SecondProblem<true>& second_of(const GemmLaunch& l, std::true_type) { return l.second; }

template <int BN, bool A_MN, bool B_MN, bool PAIR, bool X3 = false, bool DUAL = false>
cudaError_t launch_gemm_t(const GemmLaunch& l, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(l.grid), 1, 1);
  cfg.blockDim = dim3(TileCfg<BN, PAIR, X3>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = TileCfg<BN, PAIR, X3>::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  const int cluster = PAIR ? 2 : (l.args.cluster_fixup > 1 ? l.args.cluster_fixup : 1);
  if (cluster > 1) {  // CTA pairs, or the split CTAs of a tile for an in-cluster sum
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (l.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, gemm_bf16_kernel<BN, A_MN, B_MN, PAIR, X3, DUAL>, l.tmA, l.tmB, l.tmB2, l.args,
                            second_of(l, std::integral_constant<bool, DUAL>()));
}

// How many clusters of `cluster` CTAs of this instantiation the device runs at once
// (clusters live inside one GPC, so this can be fewer than SMs / cluster).
template <int BN, bool A_MN, bool B_MN, bool PAIR, bool X3 = false>
int max_active_clusters_t(int cluster, int grid) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(TileCfg<BN, PAIR, X3>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = TileCfg<BN, PAIR, X3>::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_bf16_kernel<BN, A_MN, B_MN, PAIR, X3, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();  // clear: treated as "no cluster plan"
    return 0;
  }
  return n;
}

template <int BN, bool A_MN, bool B_MN, bool PAIR, bool X3 = false, bool DUAL = false>
cudaError_t set_attr_t() {
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel<BN, A_MN, B_MN, PAIR, X3, DUAL>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, TileCfg<BN, PAIR, X3>::SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_bf16_kernel<BN, A_MN, B_MN, PAIR, X3, DUAL>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  return e;
}

}  // namespace dp
