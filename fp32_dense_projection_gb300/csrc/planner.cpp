// Per-shape planner (pure host code, no CUDA calls).
//
// The pages' deterministic package maps (arch, SM count, shape, T) to a program
// through a table of measured row rules and keeps "the K split of the row's
// previous plan (whole K per output tile)" so outputs stay bitwise identical
// (FlashInfer page "perf(cake_dense_projection_det_gemm): plan the 4096 -> 12288
// input gradient ...", PR body).  This planner replaces the table with a small
// analytic cost model over the same decisions: output tile width, the number of
// contraction splits (1 = whole K per tile), the raster group (16 output-column
// tiles, as the pages' column-grouped raster), and a persistent grid no larger
// than the SM count read at run time.
#include "planner.h"

#include <algorithm>

namespace dp {

namespace {

constexpr double kFlopPerNsPerSm = 12500.0;  // dense BF16 tensor rate per SM
constexpr double kL2BytesPerNsPerSm = 110.0;  // operand bytes an SM pulls from L2
constexpr double kHbmBytesPerNs = 6500.0;     // whole-GPU DRAM bandwidth
constexpr double kSmDramBytesPerNs = 64.0;    // most DRAM bandwidth one SM's TMA stream sustains
constexpr double kUnitOverheadNs = 600.0;     // prologue / epilogue drain per unit

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

struct View {
  int64_t gm, gn, gk;
  bool a_mn, b_mn;
  int a_elem, b_elem;  // bytes per element as streamed by the GEMM (bf16 = 2)
};

bool make_view(int op, int64_t T, int64_t N, int64_t K, View* v) {
  switch (op) {
    case kOpFwd:  // Y[T,N] = X[T,K] W[N,K]^T : A = X (K-major), B = W (K-major)
      *v = {T, N, K, false, false, 2, 2};
      return true;
    case kOpDgrad:  // dX[T,K] = dY[T,N] W[N,K] : A = dY (K-major), B = W (MN-major)
      *v = {T, K, N, false, true, 2, 2};
      return true;
    case kOpWgrad:  // dW[N,K] = dY[T,N]^T X[T,K] : A = dY (MN-major), B = X (MN-major)
      *v = {N, K, T, true, true, 2, 2};
      return true;
    // Router: the same views with the contraction tripled (hi|hi|lo against hi|lo|hi).
    case kOpRouterFwd:
      *v = {T, N, 3 * K, false, false, 2, 2};
      return true;
    case kOpRouterDgrad:
      *v = {T, K, 3 * N, false, true, 2, 2};
      return true;
    case kOpRouterWgrad:
      *v = {N, K, 3 * T, true, true, 2, 2};
      return true;
    default:
      return false;
  }
}

// Modelled time (ns) of one unit that sums `kb` contraction blocks of a
// 128 x bn tile.  Operand bytes come from L2 at a per-SM rate, but no faster in
// total than the unique bytes can come from DRAM with `active` SMs pulling; a
// split unit also writes and re-reads an FP32 partial tile.
double unit_ns(const View& v, int bn, int64_t kb, bool split, int64_t active, double reuse, int out_bytes) {
  const double a_rows = static_cast<double>(std::min<int64_t>(kBlockM, v.gm));
  const double b_rows = static_cast<double>(std::min<int64_t>(bn, v.gn));
  const double bytes_per_kb = (a_rows * v.a_elem + b_rows * v.b_elem) * kBlockK;
  const double flop_per_kb = 2.0 * kBlockM * bn * kBlockK;
  const double t_mma = kb * flop_per_kb / kFlopPerNsPerSm;
  const double per_sm_bw =
      std::min(kSmDramBytesPerNs, kHbmBytesPerNs / static_cast<double>(std::max<int64_t>(1, active)));
  const double bw = 1.0 / ((1.0 / reuse) / per_sm_bw + (1.0 - 1.0 / reuse) / kL2BytesPerNsPerSm);
  const double t_load = kb * bytes_per_kb / bw;
  const double tile_bytes = static_cast<double>(kBlockM) * bn;
  double t_epi = tile_bytes * out_bytes / per_sm_bw;
  if (split) t_epi += tile_bytes * 4.0 * 2.0 / per_sm_bw;  // partial out + last-arriver read share
  return std::max(t_mma, t_load) + t_epi + kUnitOverheadNs;
}

// Modelled time of a plan: `full` whole-K units followed by (tiles - full) tiles
// split `splits` ways, run by min(units, sm) persistent CTAs.
double model_ns(const View& v, int bn, int64_t full, int64_t splits, int sm, int out_bytes) {
  const int64_t tiles = ceil_div(v.gm, kBlockM) * ceil_div(v.gn, bn);
  const int64_t nkb = std::max<int64_t>(1, ceil_div(v.gk, kBlockK));
  const int64_t split_units = (tiles - full) * splits;
  const int64_t units = full + split_units;
  const int64_t active = std::min<int64_t>(units, sm);
  const double bytes_per_kb = (static_cast<double>(std::min<int64_t>(kBlockM, v.gm)) * v.a_elem +
                               static_cast<double>(std::min<int64_t>(bn, v.gn)) * v.b_elem) *
                              kBlockK;
  const double loaded = static_cast<double>(tiles) * nkb * bytes_per_kb;
  const double unique = static_cast<double>(v.gm * v.a_elem + v.gn * v.b_elem) * v.gk;
  const double reuse = std::max(1.0, loaded / std::max(1.0, unique));
  double t = 0.0;
  if (full > 0) t += static_cast<double>(ceil_div(full, sm)) * unit_ns(v, bn, nkb, false, active, reuse, out_bytes);
  if (split_units > 0)  // full is 0 or a whole number of waves when any tile is split
    t += static_cast<double>(ceil_div(split_units, sm)) *
         unit_ns(v, bn, ceil_div(nkb, splits), splits > 1, active, reuse, out_bytes);
  return t;
}

}  // namespace

bool make_plan(int op, int64_t T, int64_t N, int64_t K, int out_f32, int sm, Plan* p, int force_bn,
               int force_splits) {
  if (!p || sm < 1 || T < 0 || N < 1 || K < 1) return false;
  View v;
  if (!make_view(op, T, N, K, &v)) return false;
  Plan plan;
  plan.op = op;
  plan.T = T;
  plan.N = N;
  plan.K = K;
  plan.out_f32 = (op >= kOpRouterFwd) ? 1 : (out_f32 ? 1 : 0);
  plan.gm = v.gm;
  plan.gn = v.gn;
  plan.gk = v.gk;
  plan.a_mn = v.a_mn;
  plan.b_mn = v.b_mn;
  plan.nkb = ceil_div(v.gk, kBlockK);
  const int out_bytes = plan.out_f32 ? 4 : 2;

  int best_bn = 256;
  int64_t best_s = 1, best_full = 0;
  if (v.gm > 0 && plan.nkb > 0) {
    double best_t = 0.0;
    bool have = false;
    auto consider = [&](int bn, int64_t full, int64_t s, double t) {
      // prefer fewer split units and wider tiles on near-ties (less partial traffic)
      if (!have || t < best_t * 0.97) {
        have = true;
        best_t = t;
        best_bn = bn;
        best_s = s;
        best_full = full;
      }
    };
    for (int bn : {256, 128, 64}) {
      if (force_bn > 0 && bn != force_bn) continue;
      if (force_bn <= 0 && bn > 64 && v.gn <= bn / 2) continue;  // tile would be mostly empty
      const int64_t tiles = ceil_div(v.gm, kBlockM) * ceil_div(v.gn, bn);
      // bounded accumulation length, unless the tiles are too many to split at all
      // (then whole K per tile: a longer running sum, the only case without the bound)
      const int64_t min_s = tiles > kMaxSplitTiles ? 1 : ceil_div(plan.nkb, kMaxAccumBlocks);
      const int64_t max_s = std::max<int64_t>(min_s, std::min<int64_t>(plan.nkb, 64));
      // every tile split the same way (s = 1: whole K per tile)
      for (int64_t s = min_s; s <= max_s; ++s) {
        if (force_splits > 0 && s != std::min<int64_t>(force_splits, plan.nkb)) continue;
        if (force_splits <= 0 && s > min_s && tiles * s > 4LL * sm) break;  // splitting beyond 4 waves never pays
        if (s > 1 && tiles > kMaxSplitTiles) break;                         // one counter per tile
        consider(bn, s == 1 ? tiles : 0, s, model_ns(v, bn, s == 1 ? tiles : 0, s, sm, out_bytes));
      }
      // whole-K tiles for the full waves, the last partial wave's tiles split
      if (min_s == 1 && force_splits <= 0 && tiles > sm && tiles % sm != 0) {
        const int64_t full = tiles / sm * sm;
        const int64_t tail = tiles - full;
        if (tail <= kMaxSplitTiles) {
          for (int64_t s = 2; s <= std::min<int64_t>(plan.nkb, 16); ++s)
            consider(bn, full, s, model_ns(v, bn, full, s, sm, out_bytes));
        }
      }
    }
    if (!have) return false;
  }
  plan.bn = best_bn;
  plan.splits = static_cast<int>(best_s);
  plan.stages = stages_for(plan.bn);
  plan.tiles_m = ceil_div(v.gm, kBlockM);
  plan.tiles_n = ceil_div(v.gn, plan.bn);
  plan.full_units = best_full;
  plan.units = best_full + (plan.tiles_m * plan.tiles_n - best_full) * plan.splits;
  plan.group = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(16, plan.tiles_n)));
  plan.grid = static_cast<int>(std::min<int64_t>(plan.units, sm));

  // workspace layout: [counters | split partials | router A' | router B']
  size_t off = kCounterBytes;
  const int64_t tiles = plan.tiles_m * plan.tiles_n;
  const bool router_copies = op >= kOpRouterFwd && v.gm > 0;
  if (plan.splits > 1 || router_copies) {
    plan.off_counters = 0;
    plan.bytes_counters = kCounterBytes;
  }
  if (plan.splits > 1) {
    plan.off_partials = off;
    plan.bytes_partials =
        static_cast<size_t>(tiles - plan.full_units) * plan.splits * kBlockM * plan.bn * sizeof(float);
    off += plan.bytes_partials;
  }
  if (router_copies) {
    // hi/lo bf16 copies of both operands, concatenated along the contraction
    int64_t a_elems = 0, b_elems = 0;
    if (op == kOpRouterFwd) {
      a_elems = T * 3 * K;
      b_elems = N * 3 * K;
    } else if (op == kOpRouterDgrad) {
      a_elems = T * 3 * N;
      b_elems = 3 * N * K;
    } else {
      a_elems = 3 * T * N;
      b_elems = 3 * T * K;
    }
    off = round_up(off, 1024);
    plan.off_router_a = off;
    plan.bytes_router_a = static_cast<size_t>(a_elems) * 2;
    off = round_up(off + plan.bytes_router_a, 1024);
    plan.off_router_b = off;
    plan.bytes_router_b = static_cast<size_t>(b_elems) * 2;
    off += plan.bytes_router_b;
  }
  plan.ws_bytes = (plan.splits > 1 || router_copies) ? round_up(off, 256) : 0;
  *p = plan;
  return true;
}

}  // namespace dp
