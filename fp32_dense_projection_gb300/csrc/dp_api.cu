// C ABI of the dense projection GEMM library (declared in include/dp_gemm.h):
// argument checks, the planner call, TMA tensor-map encoding, the BF16x3 operand
// split of the router, and the kernel launches.  Nothing here allocates device
// memory or synchronises, except the explicit debug read-out dp_device_error().
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "dp_gemm.h"
#include "gemm_kernel.cuh"
#include "planner.h"

namespace {

using namespace dp;

// Device status word: kernels OR fault bits into it when a bounded wait gives up.
__device__ uint32_t g_fault_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool initialised = false;
  dp_status status = DP_OK;
  int sm_count = 0;
  uint32_t* fault = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

dp_status init_device(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return DP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& d = g_devices[dev];
  if (!d.initialised) {
    int major = 0, minor = 0, sm = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return DP_ERR_LAUNCH;
    }
    d.sm_count = sm;
    if (major != 10 || minor != 3) {
      d.status = DP_ERR_ARCH;  // the library carries sm_103a code only
    } else {
      int cur = -1;
      if (cudaGetDevice(&cur) != cudaSuccess) return DP_ERR_LAUNCH;
      if (cur != dev && cudaSetDevice(dev) != cudaSuccess) return DP_ERR_LAUNCH;
      void* fault = nullptr;
      cudaError_t e = set_attributes_kk();
      if (e == cudaSuccess) e = set_attributes_km();
      if (e == cudaSuccess) e = set_attributes_mm();
      if (e == cudaSuccess) e = set_attributes_bwd();
      if (e == cudaSuccess) e = set_attributes_ffma();
      if (e == cudaSuccess) e = set_attributes_split();
      if (e == cudaSuccess) e = set_attributes_reduce();
      if (e == cudaSuccess) e = cudaGetSymbolAddress(&fault, g_fault_word);
      if (cur != dev) cudaSetDevice(cur);
      if (e != cudaSuccess) return DP_ERR_LAUNCH;
      d.fault = static_cast<uint32_t*>(fault);
      d.status = DP_OK;
    }
    d.initialised = true;
  }
  *out = &d;
  return d.status;
}

dp_status current_device(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DP_ERR_LAUNCH;
  return init_device(dev, out);
}

// ------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Map over a row-major [rows][cols] matrix (leading dimension ld elements) of bf16
// (box = box_rows x 64 columns) or FP32 (box = box_rows x 32 columns): 128-byte
// box rows, 128-byte swizzle, zero fill outside the matrix.
// batch > 1: a third dimension of `batch` matrices `bstride` elements apart (box 1).
bool encode_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows,
                bool f32, uint32_t box_cols, CUtensorMapSwizzle swizzle, int64_t batch = 1, int64_t bstride = 0) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int es = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * es, static_cast<cuuint64_t>(bstride) * es};
  const cuuint32_t box[3] = {box_cols ? box_cols : (f32 ? 32u : 64u), box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, batch > 1 ? 3 : 2,
            const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the same matrix for MN-major tiles: dimensions (inner, rows,
// cols / inner) with strides (ld, inner) elements, box (inner, box_rows, groups):
// a tile of `groups` column groups of `inner` columns arrives as [group][row][inner]
// (the layout the kernel's MN-major tiles use) in one load.  Only for cols a
// multiple of inner, so every group lies inside the rows.
bool encode_map3(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, uint32_t inner,
                 uint32_t box_rows, uint32_t groups, bool f32) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || cols % inner != 0) return false;
  const int es = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {inner, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / inner)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * es, static_cast<cuuint64_t>(inner) * es};
  const cuuint32_t box[3] = {inner, box_rows, groups};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host-path caches.  A training or serving loop calls the same shapes on the same
// buffers again and again; the plan (a pure function of the shape) and the tensor
// maps (a pure function of pointer, shape, stride and box) are kept per thread in
// small direct-mapped tables, so a repeated call skips the planner's search and
// the driver's map encoding.  (FlashInfer page "cache the router entry points'
// calls by their own tensors": the pages cache the router entry points' host work
// per call signature for the same reason.)
struct MapKey {
  const void* ptr;
  int64_t rows, cols, ld, batch, bstride;
  uint32_t box_rows, box_cols;
  int f32, swizzle;
  uint32_t groups;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && ld == o.ld && box_rows == o.box_rows &&
           box_cols == o.box_cols && f32 == o.f32 && swizzle == o.swizzle && groups == o.groups &&
           batch == o.batch && bstride == o.bstride;
  }
};

uint64_t mix(uint64_t h, uint64_t v) {
  h ^= v + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
  return h;
}

constexpr int kMapCacheSize = 256;  // entries per thread (power of two)
constexpr int kPlanCacheSize = 64;

struct MapEntry {
  bool valid = false;
  MapKey key;
  CUtensorMap map;
};
thread_local MapEntry t_maps[kMapCacheSize];

// groups > 0: the 3-D map of encode_map3 with inner = box_cols (or 64 / 32 columns).
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows,
              bool f32 = false, uint32_t box_cols = 0, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
              uint32_t groups = 0, int64_t batch = 1, int64_t bstride = 0) {
  const MapKey k = {ptr, rows, cols, ld, batch, bstride, box_rows, box_cols, f32 ? 1 : 0, static_cast<int>(swizzle),
                    groups};
  uint64_t h = mix(mix(mix(reinterpret_cast<uintptr_t>(ptr), static_cast<uint64_t>(rows)), static_cast<uint64_t>(cols)),
                   static_cast<uint64_t>(ld));
  h = mix(mix(h, box_rows | (static_cast<uint64_t>(box_cols) << 32)),
          static_cast<uint64_t>(k.f32 * 16 + k.swizzle) | (static_cast<uint64_t>(groups) << 8));
  h = mix(mix(h, static_cast<uint64_t>(batch)), static_cast<uint64_t>(bstride));
  MapEntry& e = t_maps[h & (kMapCacheSize - 1)];
  if (e.valid && e.key == k) {
    *map = e.map;
    return true;
  }
  const bool ok = groups > 0 ? encode_map3(map, ptr, rows, cols, ld, box_cols ? box_cols : (f32 ? 32u : 64u), box_rows,
                                            groups, f32)
                             : encode_map(map, ptr, rows, cols, ld, box_rows, f32, box_cols, swizzle, batch, bstride);
  if (!ok) return false;
  e.valid = true;
  e.key = k;
  e.map = *map;
  return true;
}

// ------------------------------------------------------------ argument checks

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A row-major rows x cols operand with leading dimension ld (0 = cols).
dp_status check_matrix(const void* p, int64_t rows, int64_t cols, int64_t* ld, int esize) {
  if (*ld == 0) *ld = cols;
  if (*ld < cols) return DP_ERR_INVALID_ARG;
  if (rows > 0 && p == nullptr) return DP_ERR_INVALID_ARG;
  if (!aligned16(p)) return DP_ERR_ALIGNMENT;
  if ((*ld * esize) % 16 != 0) return DP_ERR_ALIGNMENT;
  if (*ld > (int64_t{1} << 36)) return DP_ERR_UNSUPPORTED;
  return DP_OK;
}

// Tuning and test overrides come from the environment only in a process started
// with DP_TUNING set (read once, at the first call that plans).  Then every call
// reads the DP_FORCE_* variables again, so a test or a sweep can change them
// between calls; otherwise no call reads the environment, and the plan caches
// see the planner's own choices only.
bool tuning_enabled() {
  static const bool on = std::getenv("DP_TUNING") != nullptr;
  return on;
}

// An override's value, or `unset` if the variable is absent or tuning is off.
int env_int(const char* name, int unset) {
  if (!tuning_enabled()) return unset;
  const char* v = std::getenv(name);
  return v ? std::atoi(v) : unset;
}

// Plan overrides (with DP_TUNING only): DP_FORCE_BN, DP_FORCE_SPLITS,
// DP_FORCE_TAIL_SPLITS, DP_FORCE_KPS, DP_FORCE_GROUP (> 0 forces),
// DP_FORCE_RASTER_M and DP_FORCE_SWAP (0 or 1: raster groups of row tiles, the
// weight-gradient orientation), DP_FORCE_PAIR (0 or 1: single-CTA or CTA-pair
// tiles), DP_FORCE_FUSE, DP_FORCE_FFMA, DP_FORCE_STREAM_K and DP_FORCE_ATOMIC (0
// or 1).  Two more are read where the launch is prepared: DP_FORCE_CLUSTER_SUM=0
// (split sums in the reduction kernel, never in the GEMM's clusters) and
// DP_FORCE_TMA_STORE (0 / 1: the epilogue's TMA stores off / on everywhere).
Overrides env_overrides() {
  Overrides o;
  if (!tuning_enabled()) return o;
  o.bn = env_int("DP_FORCE_BN", 0);
  o.splits = env_int("DP_FORCE_SPLITS", 0);
  o.tail_splits = env_int("DP_FORCE_TAIL_SPLITS", 0);
  o.swap = env_int("DP_FORCE_SWAP", -1);
  o.pair = env_int("DP_FORCE_PAIR", -1);
  o.fuse = env_int("DP_FORCE_FUSE", -1);
  o.ffma = env_int("DP_FORCE_FFMA", -1);
  o.stream_k = env_int("DP_FORCE_STREAM_K", -1);
  o.atomic = env_int("DP_FORCE_ATOMIC", -1);
  o.kps = env_int("DP_FORCE_KPS", 0);
  o.group = env_int("DP_FORCE_GROUP", 0);
  o.raster_m = env_int("DP_FORCE_RASTER_M", -1);
  return o;
}

struct PlanEntry {
  bool valid = false;
  int op, out_f32, sm, w_kn, det;
  int64_t T, N, K, batch;
  Overrides o;
  Plan plan;
};
thread_local PlanEntry t_plans[kPlanCacheSize];

bool plan_for(int op, int64_t T, int64_t N, int64_t K, int out_f32, int sm, Plan* plan, int64_t batch = 1,
              int w_kn = 0, int deterministic = 1) {
  deterministic = deterministic ? 1 : 0;
  const Overrides o = env_overrides();
  uint64_t h = mix(mix(mix(static_cast<uint64_t>(op), static_cast<uint64_t>(T)), static_cast<uint64_t>(N)),
                   static_cast<uint64_t>(K));
  h = mix(mix(h, static_cast<uint64_t>(out_f32 * 4096 + sm)),
          static_cast<uint64_t>(o.bn) * 131 + static_cast<uint64_t>(o.splits) * 17 + o.tail_splits * 7 +
              (o.swap + 1) * 3 + (o.pair + 1) + static_cast<uint64_t>(o.ffma + 1) * 7919 +
              static_cast<uint64_t>(o.stream_k + 1) * 104729 + static_cast<uint64_t>(o.atomic + 1) * 1299709 +
              static_cast<uint64_t>(o.kps) * 15485863 + static_cast<uint64_t>(o.group) * 32452843 +
              static_cast<uint64_t>(o.raster_m + 1) * 49979687);
  h = mix(h, static_cast<uint64_t>(batch) * 4 + static_cast<uint64_t>(w_kn) * 2 + static_cast<uint64_t>(deterministic));
  PlanEntry& e = t_plans[h & (kPlanCacheSize - 1)];
  if (e.valid && e.op == op && e.T == T && e.N == N && e.K == K && e.out_f32 == out_f32 && e.sm == sm &&
      e.batch == batch && e.w_kn == w_kn && e.det == deterministic && e.o.bn == o.bn && e.o.splits == o.splits &&
      e.o.tail_splits == o.tail_splits && e.o.swap == o.swap && e.o.pair == o.pair && e.o.ffma == o.ffma &&
      e.o.stream_k == o.stream_k && e.o.atomic == o.atomic && e.o.kps == o.kps && e.o.group == o.group &&
      e.o.raster_m == o.raster_m) {
    *plan = e.plan;
    return true;
  }
  if (!make_plan(op, T, N, K, out_f32, sm, plan, o, batch, w_kn != 0, deterministic != 0)) return false;
  e.det = deterministic;
  e.batch = batch;
  e.w_kn = w_kn;
  e.valid = true;
  e.op = op;
  e.T = T;
  e.N = N;
  e.K = K;
  e.out_f32 = out_f32;
  e.sm = sm;
  e.o = o;
  e.plan = *plan;
  return true;
}

dp_status check_sizes(int64_t T, int64_t N, int64_t K, int op) {
  if (T < 0 || N < 1 || K < 1) return DP_ERR_INVALID_ARG;
  if (N % 8 != 0 || K % 8 != 0) return DP_ERR_UNSUPPORTED;
  const int64_t lim = 0x7FFFFFFF;
  (void)op;
  if (T > lim || N > lim || K > lim) return DP_ERR_UNSUPPORTED;
  return DP_OK;
}

// ------------------------------------------------------------ one GEMM launch

// In-cluster sum of split partials: for plans of single-CTA tiles that split every
// tile S <= 8 ways with one unit per CTA, the GEMM runs as clusters of S CTAs and
// each cluster sums its tile's partials after the main loop (no second kernel).
// Used only if the device runs all those clusters at once (clusters live inside one
// GPC); otherwise the reduction kernel does the same sum.  Both give the same bits.
struct ClusterKey {
  int dev, view, bn, x3, size;
};
std::mutex g_cluster_mutex;
std::vector<std::pair<ClusterKey, int>> g_cluster_capacity;

int cluster_fixup(const Plan& p, bool x3, const DeviceState& dev) {
  if (p.pair || p.stream_k || p.atomic || p.splits < 2 || p.splits > 8 || p.full_units != 0 || p.units != p.grid)
    return 0;
  if (env_int("DP_FORCE_CLUSTER_SUM", 1) == 0) return 0;  // always the reduction kernel (tests)
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return 0;
  const int view = p.a_mn ? 2 : (p.b_mn ? 1 : 0);
  const ClusterKey k = {cur, view, p.bn, x3 ? 1 : 0, p.splits};
  int cap = -1;
  {
    std::lock_guard<std::mutex> lock(g_cluster_mutex);
    for (const auto& kv : g_cluster_capacity)
      if (kv.first.dev == k.dev && kv.first.view == k.view && kv.first.bn == k.bn && kv.first.x3 == k.x3 &&
          kv.first.size == k.size)
        cap = kv.second;
    if (cap < 0) {
      const int grid = dev.sm_count - dev.sm_count % p.splits;
      cap = view == 0 ? max_clusters_kk(p.bn, x3, p.splits, grid)
                      : (view == 1 ? (x3 ? 0 : max_clusters_km(p.bn, p.splits, grid))
                                   : max_clusters_mm(p.bn, x3, p.splits, grid));
      g_cluster_capacity.push_back({k, cap});
    }
  }
  return static_cast<int64_t>(cap) * p.splits >= p.grid ? p.splits : 0;
}

// A: operand (m, k) -- K-major: [gm][gk] matrix; MN-major: [gk][gm] matrix.
// B: operand (n, k) -- K-major: [gn][gk] matrix; MN-major: [gk][gn] matrix.
// Router BF16x3 plans (x3): A is FP32, B and B_lo are B's bf16 hi and lo planes.
// Batched plans: bsa / bsb / bso are the elements between consecutive batches of
// A, B and the output.
// prepare_view fills a launch (tensor maps and kernel arguments) without enqueueing it.
dp_status prepare_view(const Plan& p, const DeviceState& dev, const void* A, int64_t lda, const void* B,
                       int64_t ldb, const void* B_lo, void* out, int64_t ldo, void* ws, int64_t bsa, int64_t bsb,
                       int64_t bso, GemmLaunch* launch) {
  if (p.units > 0x7FFFFFFF || p.tiles > 0x7FFFFFFF || p.nkb > 0x7FFFFFFF || p.batch > 0xFFFFFF)
    return DP_ERR_UNSUPPORTED;
  GemmLaunch& l = *launch;
  std::memset(&l, 0, sizeof(l));
  const bool x3 = p.op == kOpRouterFwd || p.op == kOpRouterWgrad;
  // Boxes: K-major operands one box of bk contraction columns x tile rows; MN-major
  // operands boxes of 64 (bf16) or 32 (FP32) tile columns x bk contraction rows.
  const uint32_t kb_rows = static_cast<uint32_t>(p.bk);
  const uint32_t b_rows = static_cast<uint32_t>(p.pair ? p.bn / 2 : p.bn);
  // MN-major tiles load as one 3-D box when the matrix's columns are whole groups
  const uint32_t a_inner = x3 ? 32u : 64u;
  const int64_t nb = p.batch;
  const bool a3d = p.a_mn && p.gm % a_inner == 0 && nb == 1;
  const bool b3d = p.b_mn && p.gn % 64 == 0 && nb == 1;
  const uint32_t a_groups = a3d ? kBlockM / a_inner : 0u, b_groups = b3d ? b_rows / 64 : 0u;
  const auto sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
  const bool ok_a = p.a_mn ? make_map(&l.tmA, A, p.gk, p.gm, lda, kb_rows, x3, 0, sw128, a_groups, nb, bsa)
                           : make_map(&l.tmA, A, p.gm, p.gk, lda, kBlockM, x3, 0, sw128, 0, nb, bsa);
  bool ok_b;
  if (!x3) {
    ok_b = p.b_mn ? make_map(&l.tmB, B, p.gk, p.gn, ldb, kb_rows, false, 0, sw128, b_groups, nb, bsb)
                  : make_map(&l.tmB, B, p.gn, p.gk, ldb, b_rows, false, 0, sw128, 0, nb, bsb);
    l.tmB2 = l.tmB;
  } else if (p.b_mn) {  // 64-column groups of 32 rows, 128-byte swizzle
    ok_b = make_map(&l.tmB, B, p.gk, p.gn, ldb, kb_rows, false, 0, CU_TENSOR_MAP_SWIZZLE_128B, b_groups) &&
           make_map(&l.tmB2, B_lo, p.gk, p.gn, ldb, kb_rows, false, 0, CU_TENSOR_MAP_SWIZZLE_128B, b_groups);
  } else {  // rows of 32 contraction elements (64 bytes), 64-byte swizzle
    ok_b = make_map(&l.tmB, B, p.gn, p.gk, ldb, b_rows, false, kb_rows, CU_TENSOR_MAP_SWIZZLE_64B) &&
           make_map(&l.tmB2, B_lo, p.gn, p.gk, ldb, b_rows, false, kb_rows, CU_TENSOR_MAP_SWIZZLE_64B);
  }
  if (!ok_a || !ok_b) return DP_ERR_LAUNCH;
  GemmArgs& a = l.args;
  a.gm = p.gm;
  a.gn = p.gn;
  a.nkb = static_cast<int32_t>(p.nkb);
  a.splits = p.splits;
  a.full_units = static_cast<int32_t>(p.full_units);
  a.tiles_m = static_cast<int32_t>(p.tiles_m);
  a.tiles_n = static_cast<int32_t>(p.tiles_n);
  a.group = p.group;
  a.raster_m = p.raster_m ? 1 : 0;
  a.units = static_cast<int32_t>(p.units);
  a.batch = static_cast<int32_t>(nb);
  a.tiles_per_batch = static_cast<int32_t>(p.tiles_m * p.tiles_n);
  a.out_bstride = bso;
  a.out = out;
  a.ldo = ldo;
  a.out_f32 = p.out_f32;
  a.out_trans = p.out_trans ? 1 : 0;
  a.a3d = a3d ? 1 : 0;
  a.b3d = b3d ? 1 : 0;
  a.a_mn = p.a_mn ? 1 : 0;
  a.sk_slots = p.stream_k ? p.grid / (p.pair ? 2 : 1) : 0;
  a.atomic = p.atomic ? 1 : 0;
  a.sk_work = p.tiles * p.nkb;
  a.cluster_fixup = cluster_fixup(p, x3, dev);
  a.kps = (!x3 && p.kps == 2 && p.stages % 2 == 0) ? 2 : 1;
  // An operand that one column tile (A) or one row tile (B) reads in full is read once
  // by the launch (split units read disjoint contraction ranges): its loads take the L2
  // evict-first policy, so the stream recycles its own lines and leaves the rest of the
  // L2 (the other operand, split partials, and dirty lines a previous kernel left, whose
  // write-back would share DRAM with the stream) in place.  Single-CTA tiles only.
  // DP_FORCE_EVICT_FIRST=0 turns it off (comparisons).
  a.evict_first = (p.pair || env_int("DP_FORCE_EVICT_FIRST", 1) == 0)
                      ? 0
                      : ((p.tiles_n == 1 ? 1 : 0) | (p.tiles_m == 1 ? 2 : 0));
  // Whole-tile results leave through TMA stores of the epilogue's staged blocks:
  // FP32 outputs always, BF16 outputs of units of >= 8 contraction blocks (measured on
  // GB300: -4 to -15% for FP32-output calls whose epilogue is their bound, <= 1% either
  // way for the long BF16 ones, 2-4% slower for BF16 units of 2 blocks).  The
  // transposed store of the swapped weight gradient keeps its own path;
  // DP_FORCE_TMA_STORE=0 / 1 turns them off / on everywhere else (tests, comparisons).
  const int ts = env_int("DP_FORCE_TMA_STORE", -1);
  const int64_t kb_unit = p.full_units > 0 ? p.nkb : (p.nkb + p.splits - 1) / p.splits;
  const bool want_tma_store = ts >= 0 ? ts != 0 : (p.out_f32 != 0 || kb_unit >= 8);
  a.tma_store = (!p.out_trans && p.gm > 0 && want_tma_store &&
                 make_map(&a.tmO, out, p.gm, p.gn, ldo, 32, p.out_f32 != 0, p.out_f32 ? 32 : 64,
                          CU_TENSOR_MAP_SWIZZLE_128B, 0, nb, bso))
                    ? 1
                    : 0;
  // BF16-mode FP32 whole tiles of one problem whose width is a whole number of 32-column
  // blocks store two staged blocks (the epilogue warp's two) per TMA store through a
  // [block][row][32] view of the output (a box cannot clip inside a block, hence the
  // width rule), when a CTA has several tiles, whose epilogue then paces it (measured on
  // GB300: router input gradient T = 16384 90.9 -> 86.6 us; a CTA with one tile waits for
  // both blocks at once and gains nothing).  DP_FORCE_STORE2=0: one block per store.
  const bool several_tiles = p.units > p.grid / (p.pair ? 2 : 1);
  a.tma_store2 = (!x3 && a.tma_store && p.out_f32 && nb == 1 && p.gn % 32 == 0 && several_tiles &&
                  env_int("DP_FORCE_STORE2", 1) != 0 &&
                  make_map(&a.tmO2, out, p.gm, p.gn, ldo, 32, true, 32, CU_TENSOR_MAP_SWIZZLE_128B, 2))
                     ? 1
                     : 0;
  a.epi_single = env_int("DP_FORCE_EPI_SINGLE", 0) != 0 ? 1 : 0;  // (comparisons)
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.partials = p.splits > 1 ? reinterpret_cast<float4*>(w + p.off_partials) : nullptr;
  a.fault = dev.fault;
  a.wait_ns = kWaitLimitNs;
  l.grid = p.grid;
  l.pair = p.pair;
  l.x3 = x3;
  // Every GEMM launches as a programmatic dependent of the kernel before it on the
  // stream: its setup (barriers, TMEM, descriptor prefetch) overlaps that kernel's
  // tail, and its producer waits (griddepcontrol.wait) before its first load, so
  // every global access of the GEMM follows the predecessor's completion.  (The
  // router's FP32 staging loads start before that wait: their predecessor is the
  // same call's split kernel, which writes only the workspace.)
  l.pdl = true;
  return DP_OK;
}

dp_status launch_view(const Plan& p, const DeviceState& dev, const void* A, int64_t lda, const void* B,
                      int64_t ldb, const void* B_lo, void* out, int64_t ldo, void* ws, cudaStream_t stream,
                      int64_t bsa = 0, int64_t bsb = 0, int64_t bso = 0) {
  GemmLaunch l;
  const dp_status st = prepare_view(p, dev, A, lda, B, ldb, B_lo, out, ldo, ws, bsa, bsb, bso, &l);
  if (st != DP_OK) return st;
  const GemmArgs& a = l.args;
  cudaError_t e = cudaErrorInvalidValue;
  if (!p.a_mn && !p.b_mn)
    e = launch_gemm_kk(p.bn, l, stream);
  else if (!p.a_mn && p.b_mn)
    e = launch_gemm_km(p.bn, l, stream);
  else if (p.a_mn && p.b_mn)
    e = launch_gemm_mm(p.bn, l, stream);
  // split tiles: the ordered sum of their partials, queued behind the GEMM (unless
  // the GEMM's clusters sum them themselves)
  const int64_t split_tiles = p.tiles - p.full_units;
  if (e == cudaSuccess && p.splits > 1 && split_tiles > 0 && a.cluster_fixup <= 1 && !p.atomic)
    e = launch_split_reduce(l, p.bn, p.pair, split_tiles, stream);
  return e == cudaSuccess ? DP_OK : DP_ERR_LAUNCH;
}

dp_status zero_output(void* out, int64_t rows, int64_t cols, int64_t ld, int esize, cudaStream_t stream) {
  if (rows == 0) return DP_OK;
  const cudaError_t e = cudaMemset2DAsync(out, static_cast<size_t>(ld) * esize, 0, static_cast<size_t>(cols) * esize,
                                          static_cast<size_t>(rows), stream);
  return e == cudaSuccess ? DP_OK : DP_ERR_LAUNCH;
}

// Shapes of the three operands of each op: a [ra][ca], b [rb][cb], out [ro][co].
void op_shapes(int op, int64_t T, int64_t N, int64_t K, int64_t* ra, int64_t* ca, int64_t* rb, int64_t* cb,
               int64_t* ro, int64_t* co) {
  switch (op % 3) {
    case kOpFwd:  // X[T][K], W[N][K] -> Y[T][N]
      *ra = T, *ca = K, *rb = N, *cb = K, *ro = T, *co = N;
      break;
    case kOpDgrad:  // dY[T][N], W[N][K] -> dX[T][K]
      *ra = T, *ca = N, *rb = N, *cb = K, *ro = T, *co = K;
      break;
    default:  // dY[T][N], X[T][K] -> dW[N][K]
      *ra = T, *ca = N, *rb = T, *cb = K, *ro = N, *co = K;
      break;
  }
}

dp_status run_op(int op, const void* a, int64_t lda, const void* b, int64_t ldb, void* out, int64_t ldo, int64_t T,
                 int64_t N, int64_t K, int out_f32, void* ws, size_t ws_bytes, cudaStream_t stream,
                 int deterministic = 1) {
  const bool router = op >= kOpRouterFwd;
  if (!router && out_f32 != DP_OUT_BF16 && out_f32 != DP_OUT_F32) return DP_ERR_INVALID_ARG;
  dp_status st = check_sizes(T, N, K, op);
  if (st != DP_OK) return st;
  int64_t ra, ca, rb, cb, ro, co;
  op_shapes(op, T, N, K, &ra, &ca, &rb, &cb, &ro, &co);
  const int in_size = router ? 4 : 2;
  const int out_size = (router || out_f32) ? 4 : 2;
  if ((st = check_matrix(a, ra, ca, &lda, in_size)) != DP_OK) return st;
  if ((st = check_matrix(b, rb, cb, &ldb, in_size)) != DP_OK) return st;
  if ((st = check_matrix(out, ro, co, &ldo, out_size)) != DP_OK) return st;
  if (out == nullptr && ro > 0) return DP_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != DP_OK) return st;

  if (T == 0) {  // empty token set: nothing to compute, the weight gradient is zero
    if (op % 3 == kOpWgrad) return zero_output(out, ro, co, ldo, out_size, stream);
    return DP_OK;
  }
  Plan p;
  if (!plan_for(op, T, N, K, out_size == 4 ? 1 : 0, dev->sm_count, &p, 1, 0, deterministic))
    return DP_ERR_INVALID_ARG;
  if (p.ws_bytes > 0 && (ws == nullptr || ws_bytes < p.ws_bytes)) return DP_ERR_WORKSPACE;
  if (p.ws_bytes > 0 && !aligned16(ws)) return DP_ERR_ALIGNMENT;

  if (!router) {
    // non-deterministic split sums add into the output: zero it first
    if (p.atomic && (st = zero_output(out, ro, co, ldo, 4, stream)) != DP_OK) return st;
    if (p.swap) return launch_view(p, *dev, b, ldb, a, lda, nullptr, out, ldo, ws, stream);  // A = X, B = dY
    return launch_view(p, *dev, a, lda, b, ldb, nullptr, out, ldo, ws, stream);
  }

  // Router, small T: the SIMT FP32 program, one launch on the caller's operands.
  if (p.ffma) {
    FfmaArgs fa;
    std::memset(&fa, 0, sizeof(fa));
    fa.a = static_cast<const float*>(a);
    fa.b = static_cast<const float*>(b);
    fa.out = static_cast<float*>(out);
    fa.lda = lda;
    fa.ldb = ldb;
    fa.ldo = ldo;
    fa.gm = p.gm;
    fa.gn = p.gn;
    fa.gk = p.gk;
    fa.tiles_n = static_cast<int32_t>(p.tiles_n);
    fa.splits = p.splits;
    fa.kchunks = static_cast<int32_t>(p.nkb);
    if (p.units > 0x7FFFFFFF || p.nkb > 0x7FFFFFFF) return DP_ERR_UNSUPPORTED;
    return launch_router_ffma(p.bn, p.a_mn, p.b_mn, fa, stream) == cudaSuccess ? DP_OK : DP_ERR_LAUNCH;
  }

  // Router (BF16x3).  The operand that every row tile reuses is split into bf16
  // hi/lo once here; the streamed FP32 operand is split inside the GEMM.
  uint8_t* w = static_cast<uint8_t*>(ws);
  uint16_t* sa = reinterpret_cast<uint16_t*>(w + p.off_split_a);
  uint16_t* sb = reinterpret_cast<uint16_t*>(w + p.off_split_b);
  SplitJob jobs[2];
  int njobs = 1;
  std::memset(jobs, 0, sizeof(jobs));
  if (op == kOpRouterFwd) {  // W [N][K] -> hi, lo planes
    jobs[0] = {static_cast<const float*>(b), sb, N, K, ldb, p.ld_split_b, N * p.ld_split_b, 2, 0x2u};
  } else if (op == kOpRouterWgrad) {  // dY [T][N] -> hi, lo planes
    jobs[0] = {static_cast<const float*>(a), sb, T, N, lda, p.ld_split_b, T * p.ld_split_b, 2, 0x2u};
  } else {  // dY' = [lo | hi | hi] (T x 3N), W' = [hi; lo; hi] (3N x K)
    jobs[0] = {static_cast<const float*>(a), sa, T, N, lda, p.ld_split_a, N, 3, 0x1u};
    jobs[1] = {static_cast<const float*>(b), sb, N, K, ldb, p.ld_split_b, N * p.ld_split_b, 3, 0x2u};
    njobs = 2;
  }
  // (non-deterministic split sums add into the output: the split kernel zeroes it too)
  ZeroJob zero = {static_cast<float*>(out), ro, co, ldo};
  if (launch_split_x3(jobs, njobs, dev->sm_count, stream, p.atomic ? &zero : nullptr) != cudaSuccess)
    return DP_ERR_LAUNCH;
  if (op == kOpRouterFwd)  // A = X (FP32), B = W planes
    return launch_view(p, *dev, a, lda, sb, p.ld_split_b, sb + N * p.ld_split_b, out, ldo, ws, stream);
  if (op == kOpRouterWgrad)  // dW^T = X^T dY: A = X (FP32), B = dY planes; stored transposed
    return launch_view(p, *dev, b, ldb, sb, p.ld_split_b, sb + T * p.ld_split_b, out, ldo, ws, stream);
  return launch_view(p, *dev, sa, p.ld_split_a, sb, p.ld_split_b, nullptr, out, ldo, ws, stream);
}

void fill_info(const Plan& p, int64_t T, dp_plan_info* info) {
  std::memset(info, 0, sizeof(*info));
  info->block_m = p.bm;
  info->block_n = p.bn;
  info->block_k = p.bk;
  info->stages = p.stages;
  info->splits = p.splits;
  info->raster_group = p.group;
  info->grid = p.grid;
  info->a_mn_major = p.a_mn ? 1 : 0;
  info->b_mn_major = p.b_mn ? 1 : 0;
  info->swap_ab = p.swap ? 1 : 0;
  info->cta_pair = p.pair ? 1 : 0;
  info->raster_rows = p.raster_m ? 1 : 0;
  info->gemm_m = p.gm;
  info->gemm_n = p.gn;
  info->gemm_k = p.gk;
  info->tiles_m = p.tiles_m;
  info->tiles_n = p.tiles_n;
  info->k_blocks = p.nkb;
  info->units = p.units;
  info->full_units = p.full_units;
  info->workspace_bytes = T == 0 ? 0 : p.ws_bytes;
  info->batch = p.batch;
  info->weight_kn = p.w_kn ? 1 : 0;
  info->tiles = p.tiles;
  info->program = p.ffma ? 1 : 0;
  info->stream_k = p.stream_k ? 1 : 0;
  info->atomic = p.atomic ? 1 : 0;
  info->blocks_per_stage = p.kps;
  info->model_us = p.model_ns * 1e-3;
  info->cluster_sum = -1;  // (known for the current device only: set by the plan queries)
}

// The in-cluster sum of a plan on the current device (dp_plan_info::cluster_sum).
int32_t cluster_sum_here(const Plan& p) {
  DeviceState* ds = nullptr;
  if (current_device(&ds) != DP_OK) return -1;  // (current_device sets the kernels' attributes)
  return p.ffma ? 0 : cluster_fixup(p, p.op == kOpRouterFwd || p.op == kOpRouterWgrad, *ds);
}

// Batched BF16 ops: B independent problems in one launch.  Operand / output matrix
// b starts b * bs elements after matrix 0 (bs = 0: rows * ld, packed).  w_kn: W and
// dW are [K][N] matrices instead of [N][K].
dp_status run_batched(int op, const void* a, int64_t lda, int64_t bsa, const void* b, int64_t ldb, int64_t bsb,
                      void* out, int64_t ldo, int64_t bso, int w_kn, int64_t B, int64_t T, int64_t N, int64_t K,
                      int out_f32, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (op < kOpFwd || op > kOpWgrad) return DP_ERR_INVALID_ARG;
  if (out_f32 != DP_OUT_BF16 && out_f32 != DP_OUT_F32) return DP_ERR_INVALID_ARG;
  if ((w_kn != 0 && w_kn != 1) || B < 0 || bsa < 0 || bsb < 0 || bso < 0) return DP_ERR_INVALID_ARG;
  dp_status st = check_sizes(T, N, K, op);
  if (st != DP_OK) return st;
  if (B > 0xFFFFFF) return DP_ERR_UNSUPPORTED;
  if (B == 0) return DP_OK;
  int64_t ra, ca, rb, cb, ro, co;
  op_shapes(op, T, N, K, &ra, &ca, &rb, &cb, &ro, &co);
  if (w_kn) {  // W (fwd, dgrad) or dW (wgrad) stored [K][N]
    if (op == kOpWgrad)
      std::swap(ro, co);
    else
      std::swap(rb, cb);
  }
  const int out_size = out_f32 ? 4 : 2;
  if ((st = check_matrix(a, ra, ca, &lda, 2)) != DP_OK) return st;
  if ((st = check_matrix(b, rb, cb, &ldb, 2)) != DP_OK) return st;
  if ((st = check_matrix(out, ro, co, &ldo, out_size)) != DP_OK) return st;
  if (out == nullptr && ro > 0) return DP_ERR_INVALID_ARG;
  if (bsa == 0) bsa = ra * lda;
  if (bsb == 0) bsb = rb * ldb;
  if (bso == 0) bso = ro * ldo;
  if ((bsa * 2) % 16 != 0 || (bsb * 2) % 16 != 0 || (bso * out_size) % 16 != 0) return DP_ERR_ALIGNMENT;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != DP_OK) return st;
  if (T == 0) {
    if (op != kOpWgrad) return DP_OK;
    for (int64_t i = 0; i < B; ++i)
      if ((st = zero_output(static_cast<char*>(out) + i * bso * out_size, ro, co, ldo, out_size, stream)) != DP_OK)
        return st;
    return DP_OK;
  }
  Plan p;
  if (!plan_for(op, T, N, K, out_f32, dev->sm_count, &p, B, w_kn)) return DP_ERR_INVALID_ARG;
  if (p.ws_bytes > 0 && (ws == nullptr || ws_bytes < p.ws_bytes)) return DP_ERR_WORKSPACE;
  if (p.ws_bytes > 0 && !aligned16(ws)) return DP_ERR_ALIGNMENT;
  if (op == kOpWgrad && p.swap)  // A = X, B = dY
    return launch_view(p, *dev, b, ldb, a, lda, nullptr, out, ldo, ws, stream, bsb, bsa, bso);
  return launch_view(p, *dev, a, lda, b, ldb, nullptr, out, ldo, ws, stream, bsa, bsb, bso);
}

// ------------------------------------------------------------ backward pass


struct BwdEntry {
  bool valid = false;
  int64_t T, N, K;
  int dx_f32, dw_f32, sm;
  Overrides o;
  BwdPlan plan;
};
thread_local BwdEntry t_bwd_plans[16];

bool bwd_plan_for(int64_t T, int64_t N, int64_t K, int dx_f32, int dw_f32, int sm, BwdPlan* plan) {
  const Overrides o = env_overrides();
  uint64_t h = mix(mix(mix(static_cast<uint64_t>(T), static_cast<uint64_t>(N)), static_cast<uint64_t>(K)),
                   static_cast<uint64_t>(dx_f32 * 2 + dw_f32) * 4096 + static_cast<uint64_t>(sm));
  h = mix(h, static_cast<uint64_t>(o.bn) * 131 + static_cast<uint64_t>(o.splits) * 17 + o.tail_splits * 7 +
                 (o.swap + 1) * 3 + (o.pair + 1) + static_cast<uint64_t>(o.fuse + 1) * 1000003 +
                 static_cast<uint64_t>(o.stream_k + 1) * 104729 + static_cast<uint64_t>(o.kps) * 15485863 +
                 static_cast<uint64_t>(o.group) * 32452843 + static_cast<uint64_t>(o.raster_m + 1) * 49979687);
  BwdEntry& e = t_bwd_plans[h & 15];
  if (e.valid && e.T == T && e.N == N && e.K == K && e.dx_f32 == dx_f32 && e.dw_f32 == dw_f32 && e.sm == sm &&
      e.o.bn == o.bn && e.o.splits == o.splits && e.o.tail_splits == o.tail_splits && e.o.swap == o.swap &&
      e.o.pair == o.pair && e.o.fuse == o.fuse && e.o.stream_k == o.stream_k && e.o.ffma == o.ffma &&
      e.o.atomic == o.atomic && e.o.kps == o.kps && e.o.group == o.group && e.o.raster_m == o.raster_m) {
    *plan = e.plan;
    return true;
  }
  if (!make_plan_bwd(T, N, K, dx_f32, dw_f32, sm, plan, o)) return false;
  e.valid = true;
  e.T = T;
  e.N = N;
  e.K = K;
  e.dx_f32 = dx_f32;
  e.dw_f32 = dw_f32;
  e.sm = sm;
  e.o = o;
  e.plan = *plan;
  return true;
}

// dX = dY W and dW = dY^T X: either the two single-op calls one after the other, or
// one co-scheduled launch over both problems' whole-K tiles.
dp_status run_bwd(const void* dY, int64_t ldg, const void* X, int64_t ldx, const void* W, int64_t ldw, void* dX,
                  int64_t ld_dx, int dx_f32, void* dW, int64_t ld_dw, int dw_f32, int64_t T, int64_t N, int64_t K,
                  void* ws, size_t ws_bytes, cudaStream_t stream, int deterministic) {
  if ((dx_f32 != DP_OUT_BF16 && dx_f32 != DP_OUT_F32) || (dw_f32 != DP_OUT_BF16 && dw_f32 != DP_OUT_F32))
    return DP_ERR_INVALID_ARG;
  dp_status st = check_sizes(T, N, K, kOpDgrad);
  if (st != DP_OK) return st;
  if ((st = check_matrix(dY, T, N, &ldg, 2)) != DP_OK) return st;
  if ((st = check_matrix(X, T, K, &ldx, 2)) != DP_OK) return st;
  if ((st = check_matrix(W, N, K, &ldw, 2)) != DP_OK) return st;
  if ((st = check_matrix(dX, T, K, &ld_dx, dx_f32 ? 4 : 2)) != DP_OK) return st;
  if ((st = check_matrix(dW, N, K, &ld_dw, dw_f32 ? 4 : 2)) != DP_OK) return st;
  if (dW == nullptr || (dX == nullptr && T > 0) || W == nullptr) return DP_ERR_INVALID_ARG;
  DeviceState* dev = nullptr;
  if ((st = current_device(&dev)) != DP_OK) return st;
  BwdPlan bp;
  if (!bwd_plan_for(T, N, K, dx_f32, dw_f32, dev->sm_count, &bp)) return DP_ERR_INVALID_ARG;
  if (bp.ws_bytes > 0 && T > 0 && (ws == nullptr || ws_bytes < bp.ws_bytes)) return DP_ERR_WORKSPACE;
  if (bp.ws_bytes > 0 && T > 0 && !aligned16(ws)) return DP_ERR_ALIGNMENT;
  if (!bp.fused) {
    st = run_op(kOpDgrad, dY, ldg, W, ldw, dX, ld_dx, T, N, K, dx_f32, ws, ws_bytes, stream, deterministic);
    if (st != DP_OK) return st;
    return run_op(kOpWgrad, dY, ldg, X, ldx, dW, ld_dw, T, N, K, dw_f32, ws, ws_bytes, stream, deterministic);
  }
  GemmLaunch ld, lw;
  st = prepare_view(bp.dgrad, *dev, dY, ldg, W, ldw, nullptr, dX, ld_dx, nullptr, 0, 0, 0, &ld);
  if (st != DP_OK) return st;
  st = bp.wgrad.swap ? prepare_view(bp.wgrad, *dev, X, ldx, dY, ldg, nullptr, dW, ld_dw, nullptr, 0, 0, 0, &lw)
                     : prepare_view(bp.wgrad, *dev, dY, ldg, X, ldx, nullptr, dW, ld_dw, nullptr, 0, 0, 0, &lw);
  if (st != DP_OK) return st;
  GemmLaunch& first = bp.wgrad_first ? lw : ld;
  const GemmLaunch& second = bp.wgrad_first ? ld : lw;
  first.second.tmA = second.tmA;
  first.second.tmB = second.tmB;
  first.second.args = second.args;
  first.args.kps = first.second.args.kps = bp.kps;  // (the two problems share one ring)
  first.grid = bp.grid;
  return launch_gemm_bwd(bp.dgrad.bn, bp.dgrad.pair, first, stream) == cudaSuccess ? DP_OK : DP_ERR_LAUNCH;
}

void fill_bwd_info(const BwdPlan& bp, int64_t T, dp_bwd_plan_info* info) {
  std::memset(info, 0, sizeof(*info));
  info->fused = bp.fused ? 1 : 0;
  info->wgrad_first = bp.wgrad_first ? 1 : 0;
  info->grid = bp.fused ? bp.grid : 0;
  info->blocks_per_stage = bp.fused ? bp.kps : 0;
  info->model_us = bp.model_ns * 1e-3;
  info->separate_us = bp.separate_ns * 1e-3;
  info->workspace_bytes = T == 0 ? 0 : bp.ws_bytes;
  fill_info(bp.dgrad, T, &info->dgrad);
  fill_info(bp.wgrad, T, &info->wgrad);
}

// The bounded wait on its own: one CTA whose first thread waits, through the same
// mbar_wait the GEMM's roles use, on a shared-memory barrier of arrival count 1 --
// one that nothing arrives on, or (arrive != 0) one it has just arrived on itself.
// A wait that gives up after limit_ns records kFaultProbeWait in the status word
// and the kernel returns; it holds no TMEM and issues no copies, so it ends either way.
__global__ void wait_probe_kernel(uint32_t* fault, uint64_t limit_ns, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (arrive) mbar_arrive(b);
    if (!mbar_wait(b, 0, limit_ns)) atomicOr(fault, kFaultProbeWait);
  }
}

}  // namespace

// =================================================================== C ABI

extern "C" {

dp_status dp_gemm_fwd_ex(const void* X, int64_t ldx, const void* W, int64_t ldw, void* Y, int64_t ldy, int64_t T,
                         int64_t N, int64_t K, dp_out_dtype out, int deterministic, void* workspace,
                         size_t workspace_bytes, dp_stream stream) {
  return run_op(kOpFwd, X, ldx, W, ldw, Y, ldy, T, N, K, static_cast<int>(out), workspace, workspace_bytes,
                static_cast<cudaStream_t>(stream), deterministic);
}

dp_status dp_gemm_fwd(const void* X, const void* W, void* Y, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                      int deterministic, void* workspace, size_t workspace_bytes, dp_stream stream) {
  return dp_gemm_fwd_ex(X, 0, W, 0, Y, 0, T, N, K, out, deterministic, workspace, workspace_bytes, stream);
}

dp_status dp_gemm_dgrad_ex(const void* dY, int64_t ldg, const void* W, int64_t ldw, void* dX, int64_t ldx, int64_t T,
                           int64_t N, int64_t K, dp_out_dtype out, int deterministic, void* workspace,
                           size_t workspace_bytes, dp_stream stream) {
  return run_op(kOpDgrad, dY, ldg, W, ldw, dX, ldx, T, N, K, static_cast<int>(out), workspace, workspace_bytes,
                static_cast<cudaStream_t>(stream), deterministic);
}

dp_status dp_gemm_dgrad(const void* dY, const void* W, void* dX, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                        int deterministic, void* workspace, size_t workspace_bytes, dp_stream stream) {
  return dp_gemm_dgrad_ex(dY, 0, W, 0, dX, 0, T, N, K, out, deterministic, workspace, workspace_bytes, stream);
}

dp_status dp_gemm_wgrad_ex(const void* dY, int64_t ldg, const void* X, int64_t ldx, void* dW, int64_t ldw, int64_t T,
                           int64_t N, int64_t K, dp_out_dtype out, int deterministic, void* workspace,
                           size_t workspace_bytes, dp_stream stream) {
  return run_op(kOpWgrad, dY, ldg, X, ldx, dW, ldw, T, N, K, static_cast<int>(out), workspace, workspace_bytes,
                static_cast<cudaStream_t>(stream), deterministic);
}

dp_status dp_gemm_wgrad(const void* dY, const void* X, void* dW, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                        int deterministic, void* workspace, size_t workspace_bytes, dp_stream stream) {
  return dp_gemm_wgrad_ex(dY, 0, X, 0, dW, 0, T, N, K, out, deterministic, workspace, workspace_bytes, stream);
}

dp_status router_fwd_ex(const float* X, int64_t ldx, const float* W, int64_t ldw, float* Y, int64_t ldy, int64_t T,
                        int64_t N, int64_t K, int deterministic, void* workspace, size_t workspace_bytes,
                        dp_stream stream) {
  return run_op(kOpRouterFwd, X, ldx, W, ldw, Y, ldy, T, N, K, 1, workspace, workspace_bytes,
                static_cast<cudaStream_t>(stream), deterministic);
}

dp_status router_fwd(const float* X, const float* W, float* Y, int64_t T, int64_t N, int64_t K, int deterministic,
                     void* workspace, size_t workspace_bytes, dp_stream stream) {
  return router_fwd_ex(X, 0, W, 0, Y, 0, T, N, K, deterministic, workspace, workspace_bytes, stream);
}

dp_status router_dgrad_ex(const float* dY, int64_t ldg, const float* W, int64_t ldw, float* dX, int64_t ldx,
                          int64_t T, int64_t N, int64_t K, int deterministic, void* workspace,
                          size_t workspace_bytes, dp_stream stream) {
  return run_op(kOpRouterDgrad, dY, ldg, W, ldw, dX, ldx, T, N, K, 1, workspace, workspace_bytes,
                static_cast<cudaStream_t>(stream), deterministic);
}

dp_status router_dgrad(const float* dY, const float* W, float* dX, int64_t T, int64_t N, int64_t K,
                       int deterministic, void* workspace, size_t workspace_bytes, dp_stream stream) {
  return router_dgrad_ex(dY, 0, W, 0, dX, 0, T, N, K, deterministic, workspace, workspace_bytes, stream);
}

dp_status router_wgrad_ex(const float* dY, int64_t ldg, const float* X, int64_t ldx, float* dW, int64_t ldw,
                          int64_t T, int64_t N, int64_t K, int deterministic, void* workspace,
                          size_t workspace_bytes, dp_stream stream) {
  return run_op(kOpRouterWgrad, dY, ldg, X, ldx, dW, ldw, T, N, K, 1, workspace, workspace_bytes,
                static_cast<cudaStream_t>(stream), deterministic);
}

dp_status router_wgrad(const float* dY, const float* X, float* dW, int64_t T, int64_t N, int64_t K,
                       int deterministic, void* workspace, size_t workspace_bytes, dp_stream stream) {
  return router_wgrad_ex(dY, 0, X, 0, dW, 0, T, N, K, deterministic, workspace, workspace_bytes, stream);
}

dp_status dp_plan_query(dp_op op, int64_t T, int64_t N, int64_t K, dp_out_dtype out, int sm_count,
                        dp_plan_info* info) {
  return dp_plan_query_ex(op, T, N, K, out, 1, sm_count, info);
}

dp_status dp_plan_query_ex(dp_op op, int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                           int sm_count, dp_plan_info* info) {
  if (!info || static_cast<int>(op) < 0 || static_cast<int>(op) > kOpRouterWgrad) return DP_ERR_INVALID_ARG;
  const dp_status st = check_sizes(T, N, K, static_cast<int>(op));
  if (st != DP_OK) return st;
  const bool this_device = sm_count <= 0;
  if (sm_count <= 0) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DP_ERR_LAUNCH;
  }
  const bool router = static_cast<int>(op) >= kOpRouterFwd;
  Plan p;
  if (!plan_for(static_cast<int>(op), T, N, K, (router || out == DP_OUT_F32) ? 1 : 0, sm_count, &p, 1, 0,
                deterministic))
    return DP_ERR_INVALID_ARG;
  fill_info(p, T, info);
  if (this_device) info->cluster_sum = cluster_sum_here(p);
  return DP_OK;
}

dp_status dp_gemm_fwd_batched(const void* X, int64_t ldx, int64_t bsx, const void* W, int64_t ldw, int64_t bsw,
                              int weight_kn, void* Y, int64_t ldy, int64_t bsy, int64_t B, int64_t T, int64_t N,
                              int64_t K, dp_out_dtype out, int deterministic, void* workspace,
                              size_t workspace_bytes, dp_stream stream) {
  (void)deterministic;
  return run_batched(kOpFwd, X, ldx, bsx, W, ldw, bsw, Y, ldy, bsy, weight_kn, B, T, N, K, static_cast<int>(out),
                     workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

dp_status dp_gemm_dgrad_batched(const void* dY, int64_t ldg, int64_t bsg, const void* W, int64_t ldw, int64_t bsw,
                                int weight_kn, void* dX, int64_t ldx, int64_t bsx, int64_t B, int64_t T, int64_t N,
                                int64_t K, dp_out_dtype out, int deterministic, void* workspace,
                                size_t workspace_bytes, dp_stream stream) {
  (void)deterministic;
  return run_batched(kOpDgrad, dY, ldg, bsg, W, ldw, bsw, dX, ldx, bsx, weight_kn, B, T, N, K,
                     static_cast<int>(out), workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

dp_status dp_gemm_wgrad_batched(const void* dY, int64_t ldg, int64_t bsg, const void* X, int64_t ldx, int64_t bsx,
                                void* dW, int64_t ldw, int64_t bsw, int weight_kn, int64_t B, int64_t T, int64_t N,
                                int64_t K, dp_out_dtype out, int deterministic, void* workspace,
                                size_t workspace_bytes, dp_stream stream) {
  (void)deterministic;
  return run_batched(kOpWgrad, dY, ldg, bsg, X, ldx, bsx, dW, ldw, bsw, weight_kn, B, T, N, K,
                     static_cast<int>(out), workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

dp_status dp_plan_query_batched(dp_op op, int64_t B, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                                int weight_kn, int sm_count, dp_plan_info* info) {
  if (!info || static_cast<int>(op) < 0 || static_cast<int>(op) > kOpWgrad) return DP_ERR_INVALID_ARG;
  if (B < 1 || (weight_kn != 0 && weight_kn != 1)) return DP_ERR_INVALID_ARG;
  if (B > 0xFFFFFF) return DP_ERR_UNSUPPORTED;
  const dp_status st = check_sizes(T, N, K, static_cast<int>(op));
  if (st != DP_OK) return st;
  const bool this_device = sm_count <= 0;
  if (sm_count <= 0) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DP_ERR_LAUNCH;
  }
  Plan p;
  if (!plan_for(static_cast<int>(op), T, N, K, out == DP_OUT_F32 ? 1 : 0, sm_count, &p, B, weight_kn))
    return DP_ERR_INVALID_ARG;
  fill_info(p, T, info);
  if (this_device) info->cluster_sum = cluster_sum_here(p);
  return DP_OK;
}

dp_status dp_workspace_size_batched(dp_op op, int64_t B, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                                    int weight_kn, int sm_count, size_t* bytes) {
  if (!bytes) return DP_ERR_INVALID_ARG;
  dp_plan_info info;
  const dp_status st = dp_plan_query_batched(op, B, T, N, K, out, weight_kn, sm_count, &info);
  if (st != DP_OK) return st;
  *bytes = static_cast<size_t>(info.workspace_bytes);
  return DP_OK;
}

dp_status dp_workspace_size(dp_op op, int64_t T, int64_t N, int64_t K, dp_out_dtype out, int sm_count,
                            size_t* bytes) {
  if (!bytes) return DP_ERR_INVALID_ARG;
  dp_plan_info info;
  const dp_status st = dp_plan_query(op, T, N, K, out, sm_count, &info);
  if (st != DP_OK) return st;
  *bytes = static_cast<size_t>(info.workspace_bytes);
  return DP_OK;
}

dp_status dp_gemm_bwd(const void* dY, int64_t ldg, const void* X, int64_t ldx, const void* W, int64_t ldw, void* dX,
                      int64_t ld_dx, dp_out_dtype out_dx, void* dW, int64_t ld_dw, dp_out_dtype out_dw, int64_t T,
                      int64_t N, int64_t K, int deterministic, void* workspace, size_t workspace_bytes,
                      dp_stream stream) {
  return run_bwd(dY, ldg, X, ldx, W, ldw, dX, ld_dx, static_cast<int>(out_dx), dW, ld_dw, static_cast<int>(out_dw),
                 T, N, K, workspace, workspace_bytes, static_cast<cudaStream_t>(stream), deterministic);
}

dp_status dp_plan_query_bwd(int64_t T, int64_t N, int64_t K, dp_out_dtype out_dx, dp_out_dtype out_dw, int sm_count,
                            dp_bwd_plan_info* info) {
  if (!info || (out_dx != DP_OUT_BF16 && out_dx != DP_OUT_F32) || (out_dw != DP_OUT_BF16 && out_dw != DP_OUT_F32))
    return DP_ERR_INVALID_ARG;
  const dp_status st = check_sizes(T, N, K, kOpDgrad);
  if (st != DP_OK) return st;
  const bool this_device = sm_count <= 0;
  if (sm_count <= 0) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DP_ERR_LAUNCH;
  }
  BwdPlan bp;
  if (!bwd_plan_for(T, N, K, out_dx == DP_OUT_F32 ? 1 : 0, out_dw == DP_OUT_F32 ? 1 : 0, sm_count, &bp))
    return DP_ERR_INVALID_ARG;
  fill_bwd_info(bp, T, info);
  if (this_device) {  // (a co-scheduled launch keeps whole K per tile: no split sums)
    info->dgrad.cluster_sum = cluster_sum_here(bp.dgrad);
    info->wgrad.cluster_sum = cluster_sum_here(bp.wgrad);
  }
  return DP_OK;
}

dp_status dp_workspace_size_bwd(int64_t T, int64_t N, int64_t K, dp_out_dtype out_dx, dp_out_dtype out_dw,
                                int sm_count, size_t* bytes) {
  if (!bytes) return DP_ERR_INVALID_ARG;
  dp_bwd_plan_info info;
  const dp_status st = dp_plan_query_bwd(T, N, K, out_dx, out_dw, sm_count, &info);
  if (st != DP_OK) return st;
  *bytes = static_cast<size_t>(info.workspace_bytes);
  return DP_OK;
}

dp_status dp_init(int device) {
  if (device < 0 && cudaGetDevice(&device) != cudaSuccess) return DP_ERR_LAUNCH;
  DeviceState* d = nullptr;
  return init_device(device, &d);
}

dp_status dp_device_error(int clear) {
  DeviceState* d = nullptr;
  dp_status st = current_device(&d);
  if (st != DP_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return DP_ERR_LAUNCH;
  uint32_t word = 0;
  if (cudaMemcpyFromSymbol(&word, g_fault_word, sizeof(word)) != cudaSuccess) return DP_ERR_LAUNCH;
  if (clear) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(zero)) != cudaSuccess) return DP_ERR_LAUNCH;
  }
  return word ? DP_ERR_TIMEOUT : DP_OK;
}

dp_status dp_wait_probe(uint64_t limit_ns, int arrive, dp_stream stream) {
  if (limit_ns < 1000 || limit_ns > kWaitLimitNs) return DP_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  const dp_status st = current_device(&d);
  if (st != DP_OK) return st;
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(d->fault, limit_ns, arrive ? 1 : 0);
  return cudaGetLastError() == cudaSuccess ? DP_OK : DP_ERR_LAUNCH;
}

const char* dp_status_string(dp_status status) {
  switch (status) {
    case DP_OK:
      return "ok";
    case DP_ERR_INVALID_ARG:
      return "invalid argument";
    case DP_ERR_ALIGNMENT:
      return "pointer or row stride not 16-byte aligned";
    case DP_ERR_UNSUPPORTED:
      return "unsupported size (N and K must be multiples of 8; sizes below 2^31)";
    case DP_ERR_WORKSPACE:
      return "workspace missing or smaller than dp_workspace_size()";
    case DP_ERR_ARCH:
      return "current device is not sm_103a (compute capability 10.3)";
    case DP_ERR_LAUNCH:
      return "a CUDA call failed while enqueueing";
    case DP_ERR_TIMEOUT:
      return "a kernel gave up waiting on a barrier";
    default:
      return "unknown status";
  }
}

int dp_version(void) { return 130; }

}  // extern "C"
