// Per-shape planner: a pure function of (op, T, N, K, output dtype, SM count).
//
// Every operation is mapped onto one contraction view
//     D[m][n] = sum_{k < gk} A(m, k) * B(n, k),      m < gm, n < gn,
// tiled into 128 x block_n output tiles, each tile's k-blocks (64 wide) split
// into `splits` contiguous ranges.  Because the plan depends only on the shape
// and the SM count, every launch of a shape uses the same partition, which is
// what makes the outputs bitwise repeatable.
#pragma once

#include <cstddef>
#include <cstdint>

namespace dp {

enum Op : int {
  kOpFwd = 0,
  kOpDgrad = 1,
  kOpWgrad = 2,
  kOpRouterFwd = 3,
  kOpRouterDgrad = 4,
  kOpRouterWgrad = 5,
};

constexpr int kBlockM = 128;
constexpr int kBlockK = 64;
// Most split tiles (tiles whose contraction is split, times CTAs per tile) a plan
// takes by choice: splits beyond what the accumulation bound below requires are
// considered only up to this many, which bounds the workspace their FP32 partials
// take.  (The bound itself always holds: a larger shape with a long contraction
// gets the splits the bound needs and a workspace to match.)
constexpr int kMaxSplitTiles = 4096;
// Longest contraction one TMEM accumulator sums, in 64-wide blocks (16384 tokens).
// The tensor core rounds each FP32 accumulate toward zero, so the error of a
// running sum grows with its length; at 32768 tokens per accumulator a BF16
// output of the 65537-token weight gradient fell outside the pages' budget.
// Longer contractions are always split (fixed partition, partials summed in
// order), whatever the shape.
constexpr int kMaxAccumBlocks = 256;

struct Plan {
  int op = 0;
  int64_t T = 0, N = 0, K = 0;
  int out_f32 = 0;
  // contraction view
  int64_t gm = 0, gn = 0, gk = 0;
  bool a_mn = false, b_mn = false;
  // weight gradient computed as D[k][n] = sum_t X[t][k] dY[t][n] (A = X, B = dY) and
  // stored transposed into dW[n][k]: thin N becomes the MMA's N, K fills the tile rows
  bool swap = false;
  bool raster_m = false;  // raster groups of row tiles, rows fastest (B the larger operand, or B > L2 / 2)
  bool pair = false;      // tiles of 256 rows computed by a cluster of two CTAs (bm = 256)
  bool out_trans = false; // D[m][n] stored at out[n][m]
  int64_t batch = 1;      // independent GEMMs; tiles of batch b follow those of batch b - 1
  bool w_kn = false;      // W / dW stored [K][N]
  // tiling
  int bm = kBlockM, bn = 256, bk = kBlockK, stages = 4, splits = 1, group = 16, grid = 0;
  int64_t tiles_m = 0, tiles_n = 0, nkb = 0, units = 0;
  int64_t tiles = 0;      // batch * tiles_m * tiles_n
  // units [0, full_units) are whole-K tiles; the remaining tiles are split
  // `splits` ways (all tiles when full_units = 0, the last partial wave otherwise)
  int64_t full_units = 0;
  // workspace layout (byte offsets from the workspace base): split partials, then
  // the router's split operands
  size_t off_partials = 0, bytes_partials = 0;
  // router: bf16 hi/lo copies of the FP32 operands the kernel reads pre-split
  // (forward: W; weight gradient: dY; input gradient: both, in concatenated form)
  size_t off_split_a = 0, bytes_split_a = 0;
  size_t off_split_b = 0, bytes_split_b = 0;
  int64_t ld_split_a = 0, ld_split_b = 0;  // their leading dimensions (elements)
  size_t ws_bytes = 0;
  double model_ns = 0.0;  // the cost model's estimate for the chosen plan
  // Router only: the SIMT FP32 program (64 x bn tiles, each tile's contraction split
  // over a cluster of `splits` CTAs) instead of the tensor-core BF16x3 program; its
  // view is the plain contraction (input gradient over N, weight gradient unswapped),
  // nkb counts its contraction chunks of bk = 4096 / bn elements.
  bool ffma = false;
  // Stream-K: the grid's slots share the tiles' blocks evenly (slot c takes blocks
  // [c W / G, (c + 1) W / G) of the tile-major order, W = tiles * nkb); a tile cut by
  // slot boundaries is summed in pieces, up to `splits` of them, whose FP32 partials
  // the reduction adds in block order.  units = the pieces of all slots.
  bool stream_k = false;
  // Non-deterministic (deterministic = 0, FP32 output): the split units add their FP32
  // partials into the zero-filled output with atomic adds (no partials, no reduction).
  bool atomic = false;
  // Contraction blocks per stage of the operand ring (1 or 2): each stage's loads
  // complete on one barrier, and one SM's TMA streams from DRAM at about one stage
  // per barrier round trip whatever the stage's size (measured on GB300), so plans
  // that stream their operands from DRAM move two blocks per stage (half as many
  // stages).  BF16x3 plans keep one.
  int kps = 1;
};

// Shared-memory pipeline depth: as many stages of a 128 x 64 A tile plus a b_rows
// x 64 B tile (bf16) as fit in 192 KB, at most 8.  b_rows is the tile width, or
// half of it when a CTA pair shares the tile (each CTA holds half of B).
constexpr int stages_for_rows(int b_rows) {
  return (192 * 1024) / (kBlockM * kBlockK * 2 + b_rows * kBlockK * 2) < 8
             ? (192 * 1024) / (kBlockM * kBlockK * 2 + b_rows * kBlockK * 2)
             : 8;
}
constexpr int stages_for(int bn, bool pair = false) { return stages_for_rows(pair ? bn / 2 : bn); }

// The FP32 router's BF16x3 GEMM (forward and weight gradient) streams 32-wide
// contraction blocks.  The streamed FP32 operand A is loaded by TMA into a staging
// ring (128 x 32 FP32 = 16 KB per stage) and split into bf16 hi/lo by converter
// warps; the reused operand B arrives already split, as two bf16 planes.  On a single
// CTA the converters write A's halves into tensor memory, so a stage of the MMA ring
// holds [B_hi | B_lo] (bn x 32 x 2 x 2 bytes): 3 stages for 256-wide tiles, 4 for
// narrower ones; the staging ring of A's DRAM stream takes the rest of 208 KB (7, 9 and
// 11 slots for 256-, 128- and 64-wide tiles).  (Measured on GB300 against 3 + 4 slots and
// against 4 + 5: the same time within 2%.)  A CTA pair keeps A in shared memory: a stage holds
// [A_hi | A_lo | B_hi | B_lo] (half of B's rows) and the staging ring is one stage
// deeper than the MMA ring.
constexpr int kRouterBlockK = 32;
constexpr int kX3StagingBytes = kBlockM * kRouterBlockK * 4;
constexpr int kX3RingBytes = 208 * 1024;
constexpr int x3_stage_bytes(int bn, bool pair = false) {
  return pair ? (kBlockM + bn / 2) * kRouterBlockK * 4 : bn * kRouterBlockK * 4;
}
constexpr int stages_x3(int bn, bool pair = false) {
  return pair ? ((kX3RingBytes - kX3StagingBytes) / (x3_stage_bytes(bn, pair) + kX3StagingBytes) < 6
                     ? (kX3RingBytes - kX3StagingBytes) / (x3_stage_bytes(bn, pair) + kX3StagingBytes)
                     : 6)
              : (bn >= 256 ? 3 : 4);
}
constexpr int staging_stages_x3(int bn, bool pair = false) {
  return pair ? stages_x3(bn, pair) + 1
              : (kX3RingBytes - stages_x3(bn, pair) * x3_stage_bytes(bn, pair)) / kX3StagingBytes;
}

// Overrides of the planner's choices, for tests and tuning (all unset in normal
// use): > 0 forces the tile width / uniform split count / last-wave split count;
// >= 0 forces the weight-gradient orientation (swap) or single-CTA (0) versus
// CTA-pair (1) tiles.
struct Overrides {
  int bn = 0;
  int splits = 0;
  int tail_splits = 0;
  int swap = -1;
  int pair = -1;
  // backward pass: 0 two launches; 1 one co-scheduled launch (if any tiling admits it),
  // 2 / 3 the same with the weight / input gradient's units first
  int fuse = -1;
  int ffma = -1;  // router: 0 tensor-core BF16x3 program, 1 SIMT FP32 program
  int stream_k = -1;  // 0 never, 1 only stream-K candidates (where the shape admits one)
  int atomic = -1;    // non-deterministic calls: 0 ordered split sums, 1 atomic ones (where admitted)
  int kps = 0;        // > 0: contraction blocks per ring stage (1 or 2; BF16 plans only)
  int group = 0;      // > 0: raster group width in tiles
  int raster_m = -1;  // >= 0: raster groups of row tiles (1) or of column tiles (0)
};

// Fill `plan`; returns false if the arguments cannot be planned (negative sizes,
// sm_count < 1, unknown op, or overrides that admit no plan).
// batch > 1: `batch` independent GEMMs of this shape in one launch (BF16 ops);
// w_kn: W (and dW) stored [K][N] rather than [N][K].
// deterministic = false admits the atomic split sums (FP32 outputs of single-problem
// calls), where the model finds them faster than the ordered sum.
bool make_plan(int op, int64_t T, int64_t N, int64_t K, int out_f32, int sm_count, Plan* plan,
               const Overrides& overrides = Overrides(), int64_t batch = 1, bool w_kn = false,
               bool deterministic = true);

// The backward pass of one layer: the input gradient and the weight gradient of
// the same dY.  Either the two single-op plans, run one after the other, or one
// co-scheduled launch: both problems tiled alike with whole K per tile, their units
// in one list dealt to the same persistent CTAs, so the CTAs that run out of one
// problem's tiles go on with the other's instead of waiting for a second launch.
struct BwdPlan {
  bool fused = false;        // one co-scheduled launch
  bool wgrad_first = false;  // fused: the weight gradient's units come first in the list
  Plan dgrad, wgrad;         // fused: whole-K plans of one tiling; else the single-op plans
  int grid = 0;              // fused: CTAs of the launch
  int kps = 1;               // fused: contraction blocks per ring stage (both problems)
  double model_ns = 0.0;     // the chosen form's modelled duration
  double separate_ns = 0.0;  // the two single-op launches' modelled duration
  size_t ws_bytes = 0;       // workspace (the two single-op calls share one)
};
bool make_plan_bwd(int64_t T, int64_t N, int64_t K, int dx_f32, int dw_f32, int sm_count, BwdPlan* plan,
                   const Overrides& overrides = Overrides());

}  // namespace dp
