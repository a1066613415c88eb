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
// The first kCounterBytes of every non-empty workspace hold the split arrival
// counters (one uint32 per output tile of a split plan).  Nothing else is ever
// written there, so one zero-filled workspace can serve every op in turn: each
// split launch returns its counters to zero.
constexpr int kMaxSplitTiles = 4096;
// Longest contraction one TMEM accumulator sums, in 64-wide blocks (16384 tokens).
// The tensor core rounds each FP32 accumulate toward zero, so the error of a
// running sum grows with its length; at 32768 tokens per accumulator a BF16
// output of the 65537-token weight gradient fell outside the pages' budget.
// Longer contractions are split (fixed partition, partials summed in order).
constexpr int kMaxAccumBlocks = 256;
constexpr size_t kCounterBytes = kMaxSplitTiles * sizeof(uint32_t);

struct Plan {
  int op = 0;
  int64_t T = 0, N = 0, K = 0;
  int out_f32 = 0;
  // contraction view
  int64_t gm = 0, gn = 0, gk = 0;
  bool a_mn = false, b_mn = false;
  // tiling
  int bm = kBlockM, bn = 256, bk = kBlockK, stages = 4, splits = 1, group = 16, grid = 0;
  int64_t tiles_m = 0, tiles_n = 0, nkb = 0, units = 0;
  // units [0, full_units) are whole-K tiles; the remaining tiles are split
  // `splits` ways (all tiles when full_units = 0, the last partial wave otherwise)
  int64_t full_units = 0;
  // workspace layout (byte offsets from the workspace base): counters first, in
  // a fixed region of kCounterBytes, then split partials, then router operands
  size_t off_counters = 0, bytes_counters = 0;
  size_t off_partials = 0, bytes_partials = 0;
  size_t off_router_a = 0, bytes_router_a = 0;
  size_t off_router_b = 0, bytes_router_b = 0;
  size_t ws_bytes = 0;
};

// Shared-memory pipeline depth for a tile width: as many 128 x 64 + bn x 64 bf16
// stages as fit in 192 KB (4 for bn = 256, 6 for 128, 8 for 64).
constexpr int stages_for(int bn) {
  return (192 * 1024) / (kBlockM * kBlockK * 2 + bn * kBlockK * 2) < 8
             ? (192 * 1024) / (kBlockM * kBlockK * 2 + bn * kBlockK * 2)
             : 8;
}

// Fill `plan`; returns false if the arguments cannot be planned (negative sizes,
// sm_count < 1, unknown op).  `force_bn` / `force_splits` > 0 override the
// planner's choice (used by tests and tuning).
bool make_plan(int op, int64_t T, int64_t N, int64_t K, int out_f32, int sm_count, Plan* plan,
               int force_bn = 0, int force_splits = 0);

}  // namespace dp
