// Per-shape planner (pure host code, no CUDA calls).
//
// The pages' deterministic package maps (arch, SM count, shape, T) to a program
// through a table of measured row rules and keeps whole K per output tile so
// outputs stay bitwise identical (FlashInfer page
// "perf(cake_dense_projection_det_gemm): plan the 4096 -> 12288 input gradient
// ...", PR body).  This planner replaces the table with a small analytic cost
// model over the same decisions: tile shape (one CTA or a CTA pair, output tile
// width), the contraction split (whole K per tile, every tile split, or only the
// last partial wave's tiles), the weight gradient's orientation and a persistent
// grid no larger than the SM count read at run time; and, by rules measured on
// GB300, the raster order (groups of 16 tiles as the pages' column-grouped raster,
// or groups of row tiles sized to the L2 when B is large) and the contraction
// blocks per ring stage.  The plan is a pure function of its arguments, so every
// launch of a shape partitions every tile's contraction the same way.
#include "planner.h"

#include <algorithm>
#include <vector>

namespace dp {

namespace {

// Rates calibrated on GB300 measurements of this kernel (cold L2).
constexpr double kFlopPerNsPerSm = 12500.0;   // dense BF16 tensor rate per SM
constexpr double kL2BytesPerNsPerSm = 160.0;  // operand bytes an SM pulls when they hit in L2
constexpr double kHbmBytesPerNs = 5500.0;     // whole-GPU DRAM streaming rate
constexpr double kSmDramBytesPerNs = 45.0;    // most DRAM bandwidth one SM's TMA stream sustains
constexpr double kReduceNs = 2000.0;          // the split reduction kernel's launch and one L2 round trip
constexpr double kClusterSumNs = 1500.0;      // in-cluster sum (one unit per CTA, clusters of <= 4 run at once)
constexpr int kClusterSumMax = 4;             // largest cluster the device is assumed to co-schedule for it
constexpr double kReduceBytesPerNs = 4000.0;  // partial bytes it sums per ns (whole GPU, L2-resident)
constexpr double kPairGain = 0.93;            // a CTA pair reads half of B per SM: less shared-memory traffic
constexpr double kNarrowB = 1.35;             // tiles whose B slice per CTA is 64 columns (128 x 64, or a pair's
                                              // 256 x 128) run their main loop this much slower than the rates say
constexpr double kX3SplitPerNs = 20.0;        // FP32 values one SM's converter warps split into bf16 hi/lo
constexpr double kX3BlockNs = 450.0;          // least time of one 32-wide BF16x3 block (shared-memory traffic)
// ... in units of >= 8 blocks on tiles of <= 128 columns: forced-plan sweeps of the router at
// T = 64-4031 (CUPTI span, cold L2) put their blocks at ~650 ns (T = 1024: forward 128 x 128 x
// 8 splits 22.5 us against 128 x 256 x 16 splits 20.9 us; weight gradient 128 x 128 x 2
// splits 23.4 us against 128 x 256 x 4 splits 20.2 us, where the rates above predicted the
// opposite); in shorter units the fixed costs hide the difference (T = 64 forward: 128 x 128
// and 128 x 256 tiles of 4 blocks within 3%)
constexpr double kX3NarrowBlockNs = 650.0;
constexpr int kX3NarrowMinBlocks = 8;
constexpr bool kAutoPair = true;              // CTA-pair tiles chosen automatically (else only when forced)
// The epilogue of one unit (TMEM -> registers -> shared -> global), per CTA: a fixed
// cost (a CTA pair's two epilogues release one accumulator together: more), and the
// output bytes at its store rate.  It overlaps the next unit's main loop, so it only
// shows when it is the longer of the two (short contractions: measured on batched
// per-head GEMMs with 2 contraction blocks per tile).
constexpr double kEpiNs = 670.0;
constexpr double kEpiPairNs = 1420.0;
constexpr double kEpiBytesPerNs = 37.0;
// A CTA pair's MMA waits for both CTAs' operand stages, so a load-bound pair runs at
// its slower CTA's pace (measured on the batched per-head shapes: pairs 1.2x slower)
constexpr double kPairLoadPenalty = 1.2;
constexpr double kLaunchNs = 3000.0;
constexpr double kL2Bytes = 129e6;     // GB300 L2
constexpr double kL2Resident = 104e6;  // what a raster group's reused operand slabs may occupy of it          // a launch's fixed cost: setup, first loads, last tile's epilogue
// Non-deterministic atomic split sums: the zero fill's fixed cost (a memset node
// before the GEMM; for the router, a job of its operand-split kernel, nearly free),
// and the rate of FP32 atomic adds into L2
constexpr double kZeroMemsetNs = 2500.0;
constexpr double kZeroInSplitNs = 300.0;
constexpr double kAtomicBytesPerNs = 3000.0;
// SIMT FP32 router program, measured on GB300: FMAs one SM sustains (~51% of 4 x 32
// lanes at ~1.9 GHz: its shared-memory reads match the FMA pipe's rate), the
// launch's fixed cost, each wave's fixed cost (first loads from DRAM, the group and
// cluster sums, the store), and CTAs per SM (its ~150 KB of shared memory: one)
constexpr double kFfmaPerNsPerSm = 125.0;
constexpr double kFfmaFixedNs = 1500.0;
constexpr double kFfmaWaveNs = 3000.0;
constexpr double kFfmaClusterNs = 1000.0;
constexpr int kFfmaCtasPerSm = 1;
constexpr double kFuseGain = 0.97;            // co-schedule the backward pass only for >= 3% modelled gain
// what a launch of the backward pass costs beyond its modelled work, in a sequence of
// calls (measured: two calls 24.1 us vs one co-scheduled launch 19.2 us at T = 1024,
// 4096 -> 1024, where the model's work differs by ~1 us)
constexpr double kBwdLaunchNs = 5000.0;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Contraction blocks per ring stage.  One SM's TMA completes about one stage's
// loads per barrier round trip, whatever the stage's size, so two blocks per stage
// (half as many stages) speed up both the short latency-bound calls and the
// tensor-bound ones whose operands come from L2 (measured on GB300: -10% at
// T = 64 and 1025, -5% for the 4096 -> 12288 forward at T = 16384).  Long DRAM
// streams (units of >= 48 blocks, at most three per SM) keep single-block stages:
// they need the deeper ring (+2-5% with two blocks per stage at T = 16173 and
// 65537) unless their ring has eight block slots (four two-block stages).  Only
// even ring depths split into two-block stages.
bool long_stream(int64_t kb_unit, int64_t units, int64_t slots) { return kb_unit >= 48 && units <= 3 * slots; }
int blocks_per_stage(int stages, int64_t kb_unit, int64_t units, int64_t slots, int forced) {
  if (stages % 2 != 0) return 1;
  if (forced == 1 || forced == 2) return forced;
  return (stages < 8 && long_stream(kb_unit, units, slots)) ? 1 : 2;
}
int64_t ffma_stage_k_host(int bn) { return 4096 / bn; }  // contraction elements per stage of the SIMT program
size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

struct View {
  int64_t gm, gn, gk;
  bool a_mn, b_mn;
  int a_elem, b_elem;  // bytes per element as streamed by the GEMM (bf16 = 2, fp32 = 4)
  int terms = 1;       // MMAs per contraction element (3 for the router's BF16x3)
  int bk = kBlockK;    // contraction block (32 for the router's fused split)
  int64_t batch = 1;   // independent GEMMs of this view
  bool zero_in_split = false;  // router: its operand-split kernel can zero-fill the output
};

// w_kn: the weight (and the weight gradient) stored [K][N] instead of [N][K] (the
// batched entry points' weight layout); it flips the majorness of W's view.
bool make_view(int op, int64_t T, int64_t N, int64_t K, View* v, bool w_kn = false) {
  switch (op) {
    case kOpFwd:  // Y[T,N] = X[T,K] W[N,K]^T : A = X (K-major), B = W (K-major; MN-major if W is [K][N])
      *v = {T, N, K, false, w_kn, 2, 2};
      return true;
    case kOpDgrad:  // dX[T,K] = dY[T,N] W[N,K] : A = dY (K-major), B = W (MN-major; K-major if W is [K][N])
      *v = {T, K, N, false, !w_kn, 2, 2};
      return true;
    case kOpWgrad:  // dW[N,K] = dY[T,N]^T X[T,K] : A = dY (MN-major), B = X (MN-major)
      *v = {N, K, T, true, true, 2, 2};
      return true;
    // Router forward: A = X (FP32, split into bf16 hi/lo in the kernel), B = W's
    // bf16 hi and lo planes (split once per call); three MMAs per 32-wide block.
    case kOpRouterFwd:
      *v = {T, N, K, false, false, 4, 4, 3, kRouterBlockK};
      return true;
    // Router input gradient: the plain BF16 view over the concatenated operands
    // dY' = [lo | hi | hi] (T x 3N) and W' = [hi; lo; hi] (3N x K).
    case kOpRouterDgrad:
      *v = {T, K, 3 * N, false, true, 2, 2};
      return true;
    // Router weight gradient, always swapped: dW^T[K,N] = X^T dY with A = X (FP32,
    // MN-major, split in the kernel) and B = dY's bf16 hi/lo planes (MN-major),
    // stored transposed; X streams through the SMs once when N fits one tile.
    case kOpRouterWgrad:
      *v = {K, N, T, true, true, 4, 4, 3, kRouterBlockK};
      return true;
    default:
      return false;
  }
}

// A tiling: tile = rows x bn, rows = 128 (one CTA) or 256 (a CTA pair).
struct Tiling {
  int bn;
  bool pair;
  int64_t rows() const { return pair ? 2 * kBlockM : kBlockM; }
};

// Modelled time (ns) of one unit that sums `kb` contraction blocks of a tile,
// per SM.  Operand bytes come at a rate between the per-SM DRAM share and the L2
// rate, weighted by how often the plan re-reads each operand byte (`reuse`); the
// output or the FP32 partial is written at the per-SM DRAM share.
double unit_ns(const View& v, const Tiling& t, int64_t kb, bool split, int64_t active_sms, double reuse,
               int out_bytes) {
  const double a_rows = static_cast<double>(std::min<int64_t>(kBlockM, v.gm));
  const double b_rows = static_cast<double>(std::min<int64_t>(t.bn, v.gn)) / (t.pair ? 2.0 : 1.0);
  const double bytes_per_kb = (a_rows * v.a_elem + b_rows * v.b_elem) * v.bk;
  const double flop_per_kb = 2.0 * kBlockM * t.bn * v.bk * v.terms;  // per SM, tensor-pipe work
  const double narrow = (t.pair ? t.bn / 2 : t.bn) == 64 ? kNarrowB : 1.0;
  const double t_mma = kb * flop_per_kb / kFlopPerNsPerSm * (t.pair ? kPairGain : 1.0) * narrow;
  // BF16x3: the converter warps split every A element of the block
  const double x3_block = (t.bn >= 256 || kb < kX3NarrowMinBlocks) ? kX3BlockNs : kX3NarrowBlockNs;
  const double t_split = v.terms > 1 ? kb * std::max(kBlockM * v.bk / kX3SplitPerNs, x3_block) : 0.0;
  const double dram =
      std::min(kSmDramBytesPerNs, kHbmBytesPerNs / static_cast<double>(std::max<int64_t>(1, active_sms)));
  const double bw = 1.0 / ((1.0 / reuse) / dram + (1.0 - 1.0 / reuse) * narrow / kL2BytesPerNsPerSm);
  const double t_load = kb * bytes_per_kb / bw * (t.pair ? kPairLoadPenalty : 1.0);
  const double out_tile = a_rows * static_cast<double>(std::min<int64_t>(t.bn, v.gn)) * (split ? 4.0 : out_bytes);
  const double t_main = std::max(std::max(t_mma, t_load), t_split) + out_tile / dram;
  const double t_epi = (t.pair ? kEpiPairNs : kEpiNs) + out_tile / kEpiBytesPerNs;
  return std::max(t_main, t_epi);
}

// How many times the tiles load each unique operand byte (at least 1).
double reuse_of(const View& v, const Tiling& t) {
  const int64_t tiles = v.batch * ceil_div(v.gm, t.rows()) * ceil_div(v.gn, t.bn);
  const int64_t nkb = std::max<int64_t>(1, ceil_div(v.gk, v.bk));
  const double a_rows = static_cast<double>(std::min<int64_t>(t.rows(), v.gm));
  const double b_rows = static_cast<double>(std::min<int64_t>(t.bn, v.gn));
  const double loaded = static_cast<double>(tiles) * nkb * (a_rows * v.a_elem + b_rows * v.b_elem) * v.bk;
  const double unique = static_cast<double>(v.batch) * (v.gm * v.a_elem + v.gn * v.b_elem) * v.gk;
  return std::max(1.0, loaded / std::max(1.0, unique));
}

// Modelled time of a plan: `full` whole-K units followed by (tiles - full) tiles
// split `splits` ways, run by min(units, slots) persistent CTAs (or pairs); never
// faster than the unique operand bytes cross from DRAM; split plans add the
// reduction kernel that sums the partials.
// atomic_ok: the split sums may be atomic adds (taken if modelled faster, or always
// with force_atomic); *atomic reports the choice.
double model_ns(const View& v, const Tiling& t, int64_t full, int64_t splits, int sm, int out_bytes,
                bool atomic_ok = false, bool* atomic = nullptr, bool force_atomic = false) {
  const int64_t slots = t.pair ? sm / 2 : sm;
  const int64_t tiles = v.batch * ceil_div(v.gm, t.rows()) * ceil_div(v.gn, t.bn);
  const int64_t nkb = std::max<int64_t>(1, ceil_div(v.gk, v.bk));
  const int64_t split_units = (tiles - full) * splits;
  const int64_t units = full + split_units;
  const int64_t active_sms = std::min<int64_t>(units, slots) * (t.pair ? 2 : 1);
  const double a_rows = static_cast<double>(std::min<int64_t>(t.rows(), v.gm));
  const double reuse = reuse_of(v, t);
  const double unique = static_cast<double>(v.batch) * (v.gm * v.a_elem + v.gn * v.b_elem) * v.gk;
  double time = 0.0;
  if (full > 0)
    time += static_cast<double>(ceil_div(full, slots)) * unit_ns(v, t, nkb, false, active_sms, reuse, out_bytes);
  if (split_units > 0)  // full is 0 or a whole number of waves when any tile is split
    time += static_cast<double>(ceil_div(split_units, slots)) *
            unit_ns(v, t, ceil_div(nkb, splits), splits > 1, active_sms, reuse, out_bytes);
  const double t_dram = (unique + static_cast<double>(v.batch) * v.gm * v.gn * out_bytes) / kHbmBytesPerNs;
  time = std::max(time, t_dram);
  if (atomic) *atomic = false;
  if (splits > 1 && split_units > 0) {  // every split tile's partials, summed in split order
    // by the GEMM's own clusters (single-CTA tiles, every tile split, one unit per
    // CTA) or else by the reduction kernel
    const bool in_cluster = !t.pair && full == 0 && splits <= kClusterSumMax && units <= slots;
    const double partial_bytes = static_cast<double>(tiles - full) * (t.pair ? 2 : 1) * splits *
                                 std::min<double>(kBlockM, a_rows) *
                                 static_cast<double>(std::min<int64_t>(t.bn, v.gn)) * 4.0;
    const double ordered = (in_cluster ? kClusterSumNs : kReduceNs) + partial_bytes / kReduceBytesPerNs;
    // or, non-deterministic: atomic adds into the output after a zero fill of all of it
    const double added = (v.zero_in_split ? kZeroInSplitNs : kZeroMemsetNs) + partial_bytes / kAtomicBytesPerNs +
                         static_cast<double>(v.batch) * v.gm * v.gn * 4.0 / kHbmBytesPerNs;
    if (atomic_ok && (force_atomic || added < ordered)) {
      time += added;
      if (atomic) *atomic = true;
    } else {
      time += ordered;
    }
  }
  return time;
}

struct Choice {
  bool have = false;
  double t = 0.0;
  Tiling tiling = {256, false};
  int64_t splits = 1, full = 0;
  bool stream_k = false;
  bool atomic = false;
};

// Stream-K pieces: the slots' block ranges [c W / G, (c + 1) W / G) over the tiles'
// nkb blocks each; per tile, how many slots' ranges touch it.  Returns the most
// pieces of one tile and the total (pieces[] optional).
int64_t stream_k_pieces(int64_t tiles, int64_t nkb, int64_t slots, int64_t* total) {
  const int64_t work = tiles * nkb;
  std::vector<int64_t> pieces(static_cast<size_t>(tiles), 0);
  for (int64_t c = 0; c < slots; ++c) {
    const int64_t b = c * work / slots, e = (c + 1) * work / slots;
    if (b >= e) continue;
    for (int64_t t = b / nkb; t <= (e - 1) / nkb; ++t) ++pieces[static_cast<size_t>(t)];
  }
  int64_t most = 0, sum = 0;
  for (int64_t p : pieces) {
    most = std::max(most, p);
    sum += p;
  }
  if (total) *total = sum;
  return most;
}

// Modelled time of a stream-K plan: every slot sums ceil(W / G) blocks (the pieces of
// one or two tiles) and writes up to two FP32 partial tiles; then the reduction
// kernel adds the cut tiles' pieces.
double stream_k_model_ns(const View& v, const Tiling& t, int64_t tiles, int64_t nkb, int sm, int out_bytes) {
  const int64_t slots = t.pair ? sm / 2 : sm;
  const int64_t per_slot = ceil_div(tiles * nkb, slots);
  const int64_t active_sms = slots * (t.pair ? 2 : 1);
  const double reuse = reuse_of(v, t);
  const double a_rows = static_cast<double>(std::min<int64_t>(kBlockM, v.gm));
  const double partial = a_rows * static_cast<double>(std::min<int64_t>(t.bn, v.gn)) * 4.0;
  const double dram = std::min(kSmDramBytesPerNs, kHbmBytesPerNs / static_cast<double>(active_sms));
  double time = unit_ns(v, t, per_slot, true, active_sms, reuse, out_bytes) + partial / dram;
  const double unique = static_cast<double>(v.batch) * (v.gm * v.a_elem + v.gn * v.b_elem) * v.gk;
  time = std::max(time, (unique + static_cast<double>(v.batch) * v.gm * v.gn * out_bytes) / kHbmBytesPerNs);
  return time + kReduceNs + 2.0 * slots * (t.pair ? 2 : 1) * partial / kReduceBytesPerNs;
}

// Best (tiling, split count, whole-K prefix) for one contraction view.
void search(const View& v, int64_t nkb, int sm, int out_bytes, const Overrides& o, Choice* best,
            bool atomic_ok = false) {
  bool atomic = false;  // (set by the last model_ns call: its split sums are atomic)
  auto consider = [&](const Tiling& t, int64_t full, int64_t s, double time, bool sk = false) {
    // prefer earlier candidates (single CTA, wider tiles, fewer splits) on near-ties
    if (!best->have || time < best->t * 0.99) {
      best->have = true;
      best->t = time;
      best->tiling = t;
      best->splits = s;
      best->full = full;
      best->stream_k = sk;
      best->atomic = !sk && atomic;
    }
  };
  for (int pair = 0; pair < 2; ++pair) {
    if (o.pair >= 0 && pair != o.pair) continue;
    if (pair && !kAutoPair && o.pair != 1) continue;
    if (pair && (sm < 2 || v.gm <= kBlockM)) continue;  // a pair needs two row blocks of work
    if (pair && v.terms > 1 && o.pair != 1) continue;  // BF16x3 pairs only when forced (measured slower)
    const int64_t slots = pair ? sm / 2 : sm;
    for (int bn : {256, 128, 64}) {
      if (pair && bn < 128) continue;  // each CTA of a pair holds bn / 2 >= 64 columns of B
      if (o.bn > 0 && bn != o.bn) continue;
      if (o.bn <= 0 && bn > 64 && v.gn <= bn / 2) continue;  // tile would be mostly empty
      const Tiling t = {bn, pair != 0};
      const int64_t tiles = v.batch * ceil_div(v.gm, t.rows()) * ceil_div(v.gn, bn);
      const int64_t cta_tiles = tiles * (pair ? 2 : 1);  // partial slots: one per CTA tile
      // bounded accumulation length: every accumulator sums at most max_blocks blocks, so
      // a longer contraction is always split (kMaxAccumBlocks counts 64-element blocks of
      // one MMA each; BF16x3 accumulates three per element)
      const int64_t max_blocks = kMaxAccumBlocks * kBlockK / (v.bk * v.terms);
      const int64_t min_s = ceil_div(nkb, max_blocks);
      const int64_t max_s = std::max<int64_t>(min_s, std::min<int64_t>(nkb, 64));
      // every tile split the same way (s = 1: whole K per tile)
      for (int64_t s = min_s; s <= max_s && o.tail_splits <= 0 && o.stream_k != 1; ++s) {
        if (o.splits > 0 && s != std::min<int64_t>(o.splits, nkb)) continue;
        if (o.splits <= 0 && s > min_s && tiles * s > 4LL * slots) break;  // beyond 4 waves never pays
        // more splits than the bound needs only while the partials stay within
        // kMaxSplitTiles tiles' worth of workspace
        if (s > std::max<int64_t>(1, min_s) && cta_tiles > kMaxSplitTiles) break;
        consider(t, s == 1 ? tiles : 0, s,
                 model_ns(v, t, s == 1 ? tiles : 0, s, sm, out_bytes, atomic_ok, &atomic, o.atomic == 1));
      }
      // Stream-K, for tile counts that fit in one wave: every slot takes an even share
      // of all tiles' blocks, so no SM idles while others finish a wider split.  (More
      // tiles keep the raster-ordered waves, whose neighbouring tiles share operands in
      // L2.)  Each piece stays within the accumulation bound; one problem per launch,
      // single-CTA tiles for BF16x3 (whose pairs are not used).
      const int64_t per_slot = ceil_div(tiles * nkb, slots);
      if (o.stream_k != 0 && (v.terms == 1 || !pair) && v.batch == 1 && o.splits <= 0 && o.tail_splits <= 0 &&
          tiles <= slots && tiles * nkb >= 2 * slots && std::min(per_slot, nkb) <= max_blocks) {
        const int64_t most = stream_k_pieces(tiles, nkb, slots, nullptr);
        if (most >= 2 && cta_tiles * most <= kMaxSplitTiles) {
          consider(t, 0, most, stream_k_model_ns(v, t, tiles, nkb, sm, out_bytes), true);
        }
      }
      // whole-K tiles for the full waves, the last partial wave's tiles split
      if (o.stream_k != 1 && min_s == 1 && o.splits <= 0 && tiles > slots && tiles % slots != 0) {
        const int64_t full = tiles / slots * slots;
        if ((tiles - full) * (pair ? 2 : 1) <= kMaxSplitTiles) {
          for (int64_t s = 2; s <= std::min<int64_t>(nkb, 16); ++s)
            if (o.tail_splits <= 0 || s == o.tail_splits)
              consider(t, full, s, model_ns(v, t, full, s, sm, out_bytes, atomic_ok, &atomic, o.atomic == 1));
        }
      }
    }
  }
}

// The router's plain FP32 contraction views for the SIMT program:
//   forward      D = Y[T][N]:   A = X [T][K] (K-major),  B = W [N][K] (K-major)
//   input grad.  D = dX[T][K]:  A = dY [T][N] (K-major), B = W [N][K] (MN-major), over N
//   weight grad. D = dW[N][K]:  A = dY [T][N] (MN-major), B = X [T][K] (MN-major), over T
View ffma_view(int op, int64_t T, int64_t N, int64_t K) {
  if (op == kOpRouterFwd) return {T, N, K, false, false, 4, 4};
  if (op == kOpRouterDgrad) return {T, K, N, false, true, 4, 4};
  return {N, K, T, true, true, 4, 4};
}

// Modelled time of the SIMT program for tile width bn and `splits` CTAs per tile:
// the CTAs run in waves of kFfmaCtasPerSm per SM sharing its FMA rate; each CTA's
// FMAs, or its operand bytes at the L2 / DRAM mix of unit_ns, whichever is longer.
double ffma_model_ns(const View& v, int bn, int splits, int sm) {
  const int64_t bk = ffma_stage_k_host(bn);
  const int64_t tiles = ceil_div(v.gm, 64) * ceil_div(v.gn, bn);
  const int64_t chunks = std::max<int64_t>(1, ceil_div(v.gk, bk));
  const int64_t ctas = tiles * splits;
  const int64_t per_sm = std::min<int64_t>(kFfmaCtasPerSm, ceil_div(ctas, sm));
  // clusters of 8 of these CTAs (~150 KB of shared memory each) run 8 at a time
  const int64_t resident = splits > 4 ? std::min<int64_t>(sm, 64) : static_cast<int64_t>(sm) * per_sm;
  const int64_t waves = ceil_div(ctas, resident);
  const double k_slice = static_cast<double>(ceil_div(chunks, splits) * bk);
  const double t_fma = 64.0 * bn * k_slice * per_sm / kFfmaPerNsPerSm;
  const double loaded = static_cast<double>(ctas) * (64 + bn) * k_slice * 4;
  const double unique = (static_cast<double>(v.gm) + v.gn) * v.gk * 4;
  const double reuse = std::max(1.0, loaded / std::max(1.0, unique));
  const double active = static_cast<double>(std::min<int64_t>(ctas, sm));
  const double dram = std::min(kSmDramBytesPerNs, kHbmBytesPerNs / active);
  const double bw = 1.0 / ((1.0 / reuse) / dram + (1.0 - 1.0 / reuse) / kL2BytesPerNsPerSm);
  const double t_load = (64 + bn) * k_slice * 4 * per_sm / bw;
  const double out_bytes = static_cast<double>(v.gm) * v.gn * 4;
  const double t_cluster = splits > 1 ? kFfmaClusterNs : 0.0;  // the partials' sum across the cluster
  return kFfmaFixedNs + static_cast<double>(waves) * (kFfmaWaveNs + t_cluster + std::max(t_fma, t_load)) +
         out_bytes / kHbmBytesPerNs;
}

// Modelled time of one co-scheduled launch: the whole-K units of `first`, then
// those of `second` (same tiling), dealt round-robin to the persistent CTAs (unit
// u to CTA slot u mod slots, as the kernel walks them); the busiest slot sets the
// time, never below the DRAM time of both problems' unique bytes.
double fused_model_ns(const Plan& first, const Plan& second, int sm) {
  const Tiling t = {first.bn, first.pair};
  const int64_t slots = t.pair ? sm / 2 : sm;
  const int64_t units = first.units + second.units;
  const int64_t active_sms = std::min<int64_t>(units, slots) * (t.pair ? 2 : 1);
  double dram_bytes = 0.0;
  auto unit_time = [&](const Plan& p) {
    const View v = {p.gm, p.gn, p.gk, p.a_mn, p.b_mn, 2, 2};
    const int out_bytes = p.out_f32 ? 4 : 2;
    dram_bytes += (v.gm * v.a_elem + v.gn * v.b_elem) * static_cast<double>(v.gk) +
                  static_cast<double>(v.gm) * v.gn * out_bytes;
    return unit_ns(v, t, std::max<int64_t>(1, p.nkb), false, active_sms, reuse_of(v, t), out_bytes);
  };
  const double t1 = unit_time(first), t2 = unit_time(second);
  std::vector<double> slot(static_cast<size_t>(slots), 0.0);
  for (int64_t u = 0; u < units; ++u) slot[static_cast<size_t>(u % slots)] += u < first.units ? t1 : t2;
  const double busiest = *std::max_element(slot.begin(), slot.end());
  return std::max(busiest, dram_bytes / kHbmBytesPerNs);
}

}  // namespace

bool make_plan(int op, int64_t T, int64_t N, int64_t K, int out_f32, int sm, Plan* p, const Overrides& o,
               int64_t batch, bool w_kn, bool deterministic) {
  if (!p || sm < 1 || T < 0 || N < 1 || K < 1 || batch < 1) return false;
  if ((batch > 1 || w_kn) && op >= kOpRouterFwd) return false;  // batched forms: BF16 ops only
  View v;
  if (!make_view(op, T, N, K, &v, w_kn)) return false;
  v.batch = batch;
  v.zero_in_split = op >= kOpRouterFwd;
  Plan plan;
  plan.batch = batch;
  plan.w_kn = w_kn;
  plan.op = op;
  plan.T = T;
  plan.N = N;
  plan.K = K;
  plan.out_f32 = (op >= kOpRouterFwd) ? 1 : (out_f32 ? 1 : 0);
  plan.swap = op == kOpRouterWgrad;  // the router's weight gradient is always computed transposed
  plan.a_mn = v.a_mn;
  plan.b_mn = v.b_mn;
  plan.nkb = ceil_div(v.gk, v.bk);
  plan.bk = v.bk;
  const int out_bytes = plan.out_f32 ? 4 : 2;

  Choice c;
  c.have = true;  // empty problems: any tiling, no work units
  if (v.gm > 0 && plan.nkb > 0) {
    c.have = false;
    // (the orientation override applies to the BF16 weight gradient only; a router
    // plan forced onto the SIMT program takes its tile and split overrides there)
    Overrides ot = o;
    if (op >= kOpRouterFwd && o.ffma == 1) ot.bn = ot.splits = ot.tail_splits = 0;
    // (atomic split sums: FP32 outputs of single-problem calls that need not be
    // bitwise repeatable)
    const bool atomic_ok = !deterministic && out_bytes == 4 && batch == 1 && o.atomic != 0;
    if (op != kOpWgrad || o.swap != 1) search(v, plan.nkb, sm, out_bytes, ot, &c, atomic_ok);
    if (op == kOpWgrad && o.swap != 0) {
      // thin outputs: let K fill the 128-row tile side and N be the MMA's N
      View sv = {K, N, T, true, true, 2, 2};
      sv.batch = batch;
      Choice cs;
      search(sv, plan.nkb, sm, out_bytes, o, &cs, atomic_ok);
      // Thin N (<= 64) streamed over a long contraction: the swapped 128 x 64 tiles
      // (eight block slots, two blocks per stage) stream X faster than tiles with N
      // as their 128 rows, half of them padding, in six or four slots (measured
      // 35.3 -> 32.4 us at T = 16173, 4096 -> 64, and 45.2 -> 39.5 us at 5120 -> 48);
      // the rates of the model do not tell them apart, so this is a rule, taken
      // where the swapped plan models within 10%
      const int64_t s_tiles = ceil_div(sv.gm, kBlockM) * ceil_div(sv.gn, cs.tiling.bn);
      const int64_t s_units = cs.full + (s_tiles - cs.full) * cs.splits;
      const bool thin_stream = cs.have && !cs.tiling.pair && cs.tiling.bn == 64 && !cs.stream_k && N <= 64 &&
                               long_stream(cs.full > 0 ? plan.nkb : ceil_div(plan.nkb, cs.splits), s_units, sm);
      if (cs.have && (!c.have || cs.t < c.t * 0.97 || o.swap == 1 || (thin_stream && cs.t < c.t * 1.10))) {
        c = cs;
        plan.swap = true;
        v = sv;
      }
    }
    if (!c.have) return false;
  }
  plan.gm = v.gm;
  plan.gn = v.gn;
  plan.gk = v.gk;
  plan.model_ns = c.have ? c.t : 0.0;
  plan.pair = c.tiling.pair;
  plan.bm = static_cast<int>(c.tiling.rows());
  plan.bn = c.tiling.bn;
  plan.splits = static_cast<int>(c.splits);
  plan.stream_k = c.stream_k;
  plan.atomic = c.atomic && c.splits > 1;
  plan.stages = v.terms > 1 ? stages_x3(plan.bn, plan.pair) : stages_for(plan.bn, plan.pair);
  plan.tiles_m = ceil_div(v.gm, plan.bm);
  plan.tiles_n = ceil_div(v.gn, plan.bn);
  plan.tiles = batch * plan.tiles_m * plan.tiles_n;
  const int64_t tiles = plan.tiles;
  plan.full_units = (v.gm > 0 && plan.nkb > 0) ? c.full : tiles;
  plan.units = plan.full_units + (tiles - plan.full_units) * plan.splits;
  const int64_t slots_all = plan.pair ? sm / 2 : sm;
  if (plan.stream_k) {  // units: every piece of every slot's block range
    stream_k_pieces(tiles, plan.nkb, slots_all, &plan.units);
    plan.full_units = 0;
  }
  // Group along the dimension whose operand is larger, so the tiles that share
  // its blocks run in the same wave and it crosses from DRAM about once.
  plan.raster_m = o.raster_m >= 0 ? o.raster_m != 0 : v.gn > v.gm;
  int group = 16;
  // When B is large too (more than half the L2), groups of row tiles instead, as wide as
  // their A slabs fit in ~104 MB of the L2: each group's A stays resident while B streams
  // through it once per group (measured on GB300 at 4096 -> 12288, T = 16384: forward
  // 843 -> 830 us, input gradient 893 -> 871, weight gradient 880 -> 869 with groups of 8;
  // shapes whose B fits keep the rule above, measured equal or better).
  const double b_bytes = static_cast<double>(batch) * v.gn * v.gk * v.b_elem;
  if (o.raster_m < 0 && b_bytes > kL2Bytes / 2) {
    plan.raster_m = true;
    const double slab = static_cast<double>(plan.bm) * v.gk * v.a_elem;
    while (group > 1 && group * slab > kL2Resident) group /= 2;
  }
  plan.group = static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>(o.group > 0 ? o.group : group, plan.raster_m ? plan.tiles_m : plan.tiles_n)));
  // (stream-K: every slot, each with its share of the blocks)
  plan.grid = static_cast<int>((plan.stream_k ? slots_all : std::min<int64_t>(plan.units, slots_all)) *
                               (plan.pair ? 2 : 1));
  // (BF16x3 keeps one block per stage: its converter warps fill the stages block by block)
  const int64_t kb_unit = plan.full_units > 0 ? plan.nkb : ceil_div(plan.nkb, plan.splits);
  plan.kps = v.terms == 1 ? blocks_per_stage(plan.stages, kb_unit, plan.units, slots_all, o.kps) : 1;

  // workspace layout: [split partials | router's pre-split operands]
  size_t off = 0;
  if (plan.splits > 1 && !plan.atomic) {
    // one FP32 partial per split of every split tile, per CTA of the tile
    plan.off_partials = off;
    plan.bytes_partials = static_cast<size_t>(tiles - plan.full_units) * (plan.pair ? 2 : 1) * plan.splits *
                          kBlockM * plan.bn * sizeof(float);
    off += plan.bytes_partials;
  }
  const bool router = op >= kOpRouterFwd;
  if (router && T > 0) {
    auto region = [&](size_t bytes, size_t* at) {
      off = round_up(off, 256);
      *at = off;
      off += bytes;
      return bytes;
    };
    const size_t e = sizeof(uint16_t);
    if (op == kOpRouterFwd) {  // W: hi and lo planes [N][K]
      plan.ld_split_b = static_cast<int64_t>(round_up(K, 8));
      plan.bytes_split_b = region(2 * static_cast<size_t>(N) * plan.ld_split_b * e, &plan.off_split_b);
    } else if (op == kOpRouterWgrad) {  // dY: hi and lo planes [T][N]
      plan.ld_split_b = static_cast<int64_t>(round_up(N, 8));
      plan.bytes_split_b = region(2 * static_cast<size_t>(T) * plan.ld_split_b * e, &plan.off_split_b);
    } else {  // dY' [T][3N] and W' [3N][K]
      plan.ld_split_a = static_cast<int64_t>(round_up(3 * N, 8));
      plan.bytes_split_a = region(static_cast<size_t>(T) * plan.ld_split_a * e, &plan.off_split_a);
      plan.ld_split_b = static_cast<int64_t>(round_up(K, 8));
      plan.bytes_split_b = region(3 * static_cast<size_t>(N) * plan.ld_split_b * e, &plan.off_split_b);
    }
  }
  plan.ws_bytes = ((plan.splits > 1 && !plan.atomic) || (router && T > 0)) ? round_up(off, 256) : 0;
  // D[m][n] goes out transposed for the swapped weight gradient, unless the weight
  // gradient is itself stored [K][N] (then the unswapped one is transposed instead)
  plan.out_trans = (op == kOpWgrad || op == kOpRouterWgrad) && (plan.swap != w_kn);

  // Router: the SIMT FP32 program instead, when it models faster than the BF16x3
  // program plus that program's operand-split kernel (one more launch and a pass
  // over the reused operand).
  if (router && T > 0 && o.ffma != 0) {
    const View fv = ffma_view(op, T, N, K);
    double best = 0.0;
    int best_bn = 0, best_s = 0;
    for (int bn : {64, 32}) {
      if (o.bn > 0 && bn != o.bn) continue;
      const int64_t chunks = std::max<int64_t>(1, ceil_div(fv.gk, ffma_stage_k_host(bn)));
      for (int sp = 1; sp <= 8; ++sp) {
        if (o.splits > 0 && sp != o.splits) continue;
        if (sp > chunks) break;
        const double t = ffma_model_ns(fv, bn, sp, sm);
        if (best_bn == 0 || t < best * 0.99) {
          best = t;
          best_bn = bn;
          best_s = sp;
        }
      }
    }
    // (the BF16x3 program: its GEMM's launch, plus the split kernel's pass over the
    // reused operand, reading FP32 and writing bf16 hi / lo, and the half of that
    // kernel's launch which the GEMM, its programmatic dependent, does not overlap)
    const double split_pass = kLaunchNs / 2 + static_cast<double>(plan.bytes_split_a + plan.bytes_split_b) * 3.0 /
                                                  kHbmBytesPerNs;
    if (best_bn > 0 && (o.ffma == 1 || best < plan.model_ns + kLaunchNs + split_pass)) {
      Plan f;
      f.op = op;
      f.T = T;
      f.N = N;
      f.K = K;
      f.out_f32 = 1;
      f.ffma = true;
      f.gm = fv.gm;
      f.gn = fv.gn;
      f.gk = fv.gk;
      f.a_mn = fv.a_mn;
      f.b_mn = fv.b_mn;
      f.bm = 64;
      f.bn = best_bn;
      f.bk = static_cast<int>(ffma_stage_k_host(best_bn));
      f.stages = 2;
      f.splits = best_s;
      f.group = 1;
      f.tiles_m = ceil_div(fv.gm, 64);
      f.tiles_n = ceil_div(fv.gn, best_bn);
      f.tiles = f.tiles_m * f.tiles_n;
      f.nkb = std::max<int64_t>(1, ceil_div(fv.gk, f.bk));
      f.units = f.tiles * best_s;
      f.full_units = best_s == 1 ? f.tiles : 0;
      f.grid = static_cast<int>(std::min<int64_t>(f.units, 0x7FFFFFFF));
      f.model_ns = best;
      plan = f;
    }
  }
  *p = plan;
  return true;
}

bool make_plan_bwd(int64_t T, int64_t N, int64_t K, int dx_f32, int dw_f32, int sm, BwdPlan* out,
                   const Overrides& o) {
  if (!out || sm < 1) return false;
  BwdPlan r;
  if (!make_plan(kOpDgrad, T, N, K, dx_f32, sm, &r.dgrad, o) || !make_plan(kOpWgrad, T, N, K, dw_f32, sm, &r.wgrad, o))
    return false;
  r.separate_ns = r.dgrad.model_ns + r.wgrad.model_ns + 2 * kBwdLaunchNs;
  r.model_ns = r.separate_ns;
  r.ws_bytes = std::max(r.dgrad.ws_bytes, r.wgrad.ws_bytes);
  // Co-scheduled candidates: one tiling for both problems, whole K per tile (no
  // workspace, and the same per-tile sums as whole-K single-op plans), either
  // problem's units first.
  if (T > 0 && o.fuse != 0 && o.splits <= 1 && o.tail_splits <= 0) {
    bool have = false;
    BwdPlan best;
    for (int pair = 0; pair < 2; ++pair) {
      if (o.pair >= 0 && pair != o.pair) continue;
      for (int bn : {256, 128}) {
        if (o.bn > 0 && bn != o.bn) continue;
        Overrides f = o;
        f.pair = pair;
        f.bn = bn;
        f.splits = 1;
        f.tail_splits = 0;
        Plan d, w;
        if (!make_plan(kOpDgrad, T, N, K, dx_f32, sm, &d, f) || !make_plan(kOpWgrad, T, N, K, dw_f32, sm, &w, f))
          continue;
        if (d.splits != 1 || w.splits != 1 || d.units < 1 || w.units < 1) continue;
        for (int wf = 0; wf < 2; ++wf) {
          if (o.fuse >= 2 && wf != (o.fuse == 2 ? 1 : 0)) continue;
          const double t = fused_model_ns(wf ? w : d, wf ? d : w, sm) + kBwdLaunchNs;
          if (!have || t < best.model_ns) {
            have = true;
            best.fused = true;
            best.wgrad_first = wf != 0;
            best.dgrad = d;
            best.wgrad = w;
            best.model_ns = t;
            const int64_t slots = pair ? sm / 2 : sm;
            best.grid = static_cast<int>(std::min<int64_t>(d.units + w.units, slots) * (pair ? 2 : 1));
            // (one ring for both problems' units)
            best.kps = blocks_per_stage(d.stages, std::max(d.nkb, w.nkb), d.units + w.units, slots, o.kps);
          }
        }
      }
    }
    if (have && (o.fuse >= 1 || best.model_ns < kFuseGain * r.separate_ns)) {
      best.separate_ns = r.separate_ns;
      best.ws_bytes = 0;
      r = best;
    }
  }
  *out = r;
  return true;
}

}  // namespace dp
