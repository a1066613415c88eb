/*
 * dp_gemm.h -- C ABI of the GB300 (sm_103a) dense projection GEMM library.
 *
 * The library computes the projection GEMMs of one training step of a linear
 * layer Y = X W^T, as described on the FlashInfer pull-request pages about the
 * "Cake" dense projection GEMM packages:
 *
 *   forward          Y[T,N]  = X[T,K] . W[N,K]^T           (K-major B)
 *   input gradient   dX[T,K] = dY[T,N] . W[N,K]            (MN-major B)
 *   weight gradient  dW[N,K] = dY[T,N]^T . X[T,K]          (contraction over the
 *                                                           T tokens, 64-token blocks)
 *   router           the same three contractions on FP32 operands (hidden H -> 256
 *                    experts) computed through BF16x3 emulation.
 *
 * Page references used below:
 *   [det-dgrad]  "perf(cake_dense_projection_det_gemm): plan the 4096 -> 12288
 *                input gradient with the row-half-release program at T-exact keys",
 *                PR body: forward (K-major B) and input-gradient (MN-major B) forms;
 *                whole K per output tile keeps outputs bitwise identical.
 *   [k1-wgrad]   "perf(cake_dense_projection_gemm): restore the K1 weight-gradient
 *                routes that meet the deterministic package's absolute FP64 budgets",
 *                PR body: K1 has BF16 or FP32 output; wgrad contracts over 64-token
 *                K blocks with one or two K splits; the FP64 error budgets.
 *   [router]     "perf(cake_dense_projection_gemm): cache the router entry points'
 *                calls by their own tensors", summary: FP32 router [T,H] x [256,H]^T,
 *                BF16x3 emulation, router_forward / router_dgrad / router_wgrad,
 *                deterministic=True is the default.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  All matrix pointers are DEVICE pointers on the current CUDA device,
 *   row-major, 16-byte aligned.  BF16 operands are passed as raw 16-bit patterns
 *   (`const void*`).  Leading dimensions (`ld*`, in elements) give the distance
 *   between consecutive rows; 0 means "contiguous" (the row length).  Every
 *   leading dimension times the element size must be a multiple of 16 bytes, and
 *   the row lengths N and K must be multiples of 8 (16-byte rows).  An output
 *   with a padded leading dimension is written only in its first N (or K) columns.
 * Ownership.  The caller owns every buffer, the workspace and the stream.  The
 *   library never allocates device memory, never synchronises and never frees.
 * Workspace.  `workspace` is caller-provided device memory of at least
 *   dp_workspace_size(...) bytes (may be NULL when that size is 0).  It is
 *   scratch: FP32 partial tiles of split contractions and the router's bf16
 *   hi/lo operand copies, written before they are read within the call, so it
 *   needs no initial value.  One workspace must not be used by two calls that may
 *   run concurrently.
 * Launches.  Each call enqueues one GEMM kernel; a plan that splits contractions
 *   adds the kernel that sums the partials, and a router call adds the kernel
 *   that splits its reused FP32 operand into bf16 hi/lo before the GEMM (a router
 *   call on the small-T SIMT program is that one kernel alone; a non-deterministic
 *   plan adds a memset of its FP32 output instead of the reduction).  The GEMM
 *   and the reduction launch as programmatic dependents of the kernel before them
 *   on the stream: their setup overlaps that kernel's tail, and they wait for its
 *   completion before touching global memory, so stream order between calls (one
 *   call reading what the previous one wrote, or overwriting what it read) holds
 *   as for ordinary launches.
 * Stream.  `stream` is a cudaStream_t (NULL = legacy default stream).  All work
 *   is enqueued on it; calls return before the GPU finishes.  Calls are legal
 *   inside CUDA stream capture after the first call on the device (which sets
 *   kernel attributes; dp_init() does it explicitly).
 * Determinism.  With deterministic != 0 (the default of the pages' entry points)
 *   every output is bitwise reproducible for the same inputs, shapes, strides and
 *   SM count: each output tile's contraction is split into a fixed partition
 *   chosen by a pure planner, and split partials are summed in split order.
 *   deterministic = 0 (the pages' non-deterministic package) admits, for FP32
 *   outputs of single-problem calls, plans whose split units add their FP32
 *   partials into the output with atomic adds after a zero fill of the output
 *   (a memset node, or a job of the router's split kernel): no partial workspace
 *   and no reduction kernel, at the cost of run-to-run variation in the last bits
 *   (the adds' order).  The planner takes it only where its model finds it
 *   faster; BF16 outputs, batched calls and plans without split tiles stay
 *   deterministic either way.
 * Errors.  Arguments are checked before anything is enqueued; a non-DP_OK status
 *   means nothing was launched (except DP_ERR_LAUNCH, reported by CUDA after the
 *   attempt).  No exception crosses the ABI.
 * Empty input.  T == 0 is legal: forward and input gradient enqueue nothing; the
 *   weight gradient writes zeros (the sum over an empty token set).
 */
#ifndef DP_GEMM_H
#define DP_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dp_status {
    DP_OK = 0,
    DP_ERR_INVALID_ARG = 1,   /* null pointer, negative size, ld smaller than the row */
    DP_ERR_ALIGNMENT = 2,     /* pointer or row stride not 16-byte aligned */
    DP_ERR_UNSUPPORTED = 3,   /* N or K not a multiple of 8, or a size beyond 2^31-1 */
    DP_ERR_WORKSPACE = 4,     /* workspace NULL or smaller than dp_workspace_size() */
    DP_ERR_ARCH = 5,          /* current device is not compute capability 10.3 (sm_103a) */
    DP_ERR_LAUNCH = 6,        /* a CUDA call failed while enqueueing */
    DP_ERR_TIMEOUT = 7        /* a kernel gave up waiting on one of its barriers (debug read-out) */
} dp_status;

typedef enum dp_out_dtype {
    DP_OUT_BF16 = 0,          /* FP32 accumulator rounded once to bf16, nearest-even */
    DP_OUT_F32 = 1            /* FP32 accumulator stored as is */
} dp_out_dtype;

typedef enum dp_op {
    DP_OP_FWD = 0,
    DP_OP_DGRAD = 1,
    DP_OP_WGRAD = 2,
    DP_OP_ROUTER_FWD = 3,
    DP_OP_ROUTER_DGRAD = 4,
    DP_OP_ROUTER_WGRAD = 5
} dp_op;

/* A cudaStream_t, passed as a plain pointer. */
typedef void* dp_stream;

/* ------------------------------------------------------------------ BF16 ops */

/* Forward, [det-dgrad] "forward (K-major B) form":
 *   Y[t][n] = sum_k X[t][k] * W[n][k]
 * X: T x K bf16 (ldx), W: N x K bf16 (ldw), Y: T x N (ldy) in `out` precision.
 * FP32 accumulation; rows t >= T are never written. */
dp_status dp_gemm_fwd(const void* X, const void* W, void* Y,
                      int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                      void* workspace, size_t workspace_bytes, dp_stream stream);
dp_status dp_gemm_fwd_ex(const void* X, int64_t ldx, const void* W, int64_t ldw,
                         void* Y, int64_t ldy,
                         int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                         void* workspace, size_t workspace_bytes, dp_stream stream);

/* Input gradient, [det-dgrad] "input-gradient (MN-major B) form":
 *   dX[t][k] = sum_n dY[t][n] * W[n][k]
 * dY: T x N bf16 (ldg), W: N x K bf16 (ldw; read with the contraction N as its
 * outer, MN-major dimension), dX: T x K (ldx) in `out` precision. */
dp_status dp_gemm_dgrad(const void* dY, const void* W, void* dX,
                        int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                        void* workspace, size_t workspace_bytes, dp_stream stream);
dp_status dp_gemm_dgrad_ex(const void* dY, int64_t ldg, const void* W, int64_t ldw,
                           void* dX, int64_t ldx,
                           int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                           void* workspace, size_t workspace_bytes, dp_stream stream);

/* Weight gradient, [k1-wgrad] (contraction over the tokens in 64-token K blocks):
 *   dW[n][k] = sum_t dY[t][n] * X[t][k]
 * dY: T x N bf16 (ldg), X: T x K bf16 (ldx), dW: N x K (ldw) in `out` precision.
 * The token blocks of one output tile are summed by one CTA in order, or, for
 * thin outputs, split into S contiguous block ranges whose FP32 partials are
 * added in ascending split order before the single output rounding. */
dp_status dp_gemm_wgrad(const void* dY, const void* X, void* dW,
                        int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                        void* workspace, size_t workspace_bytes, dp_stream stream);
dp_status dp_gemm_wgrad_ex(const void* dY, int64_t ldg, const void* X, int64_t ldx,
                           void* dW, int64_t ldw,
                           int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                           void* workspace, size_t workspace_bytes, dp_stream stream);

/* Weight gradient for callers that cannot allocate device memory.  The pages have
 * no counterpart of this entry point; it exists for this library's users.
 * Some callers cannot pass a workspace: a serving runtime that reserves all device
 * memory at start-up, or a plugin whose host forbids cudaMalloc on its hot path
 * because it can synchronise the device.  This call computes exactly what
 * dp_gemm_wgrad_ex computes (same plan, same kernels, same bits) but keeps its
 * split partials in a 64 MiB scratch array built into the library,
 * which every GPU that loads the library holds until the process exits.  The
 * caller still passes dY, X and dW.  Arguments and errors as dp_gemm_wgrad_ex;
 * a shape whose plan needs more than 64 MiB of scratch returns DP_ERR_WORKSPACE
 * (dp_workspace_size(DP_OP_WGRAD, ...) tells beforehand).  The first call on each
 * device looks up the array's device address (with that device current).  Every
 * call shares the one array; calls that overlap on the GPU
 * (different streams or threads) race on it and must be serialised by the caller.  No cudaMalloc,
 * cudaFree or allocating library routine is called. */
dp_status dp_gemm_wgrad_noalloc(const void* dY, int64_t ldg, const void* X, int64_t ldx,
                                void* dW, int64_t ldw,
                                int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                                dp_stream stream);

/* ------------------------------------------------------------ batched BF16 ops */
/* Batched projection GEMMs: B independent problems of one shape in one launch,
 * as the pages' integration runs its per-head projections ("one batched BF16 GEMM
 * over strided views, forward and both gradients", with a weight layout option).
 * Problem b reads X_b = X + b*bsx (and so on for every operand and output, in
 * elements; a batch stride of 0 means packed, rows * ld).  Batch strides may be
 * smaller than a row (per-head slices of a [T][H][D] tensor: ld = H*D, bs = D);
 * they must keep 16-byte alignment.  weight_kn = 0: W_b and dW_b are [N][K]
 * matrices as in the single-problem calls; 1: they are [K][N].  One plan covers
 * the B * tiles_m * tiles_n tiles in one persistent launch (its tile shape and
 * splits are chosen for the whole batch, so they can differ from a single
 * problem's); every problem's tiles use the same fixed contraction partition and
 * summation order, so the outputs are deterministic (whatever `deterministic`). */
dp_status dp_gemm_fwd_batched(const void* X, int64_t ldx, int64_t bsx, const void* W, int64_t ldw, int64_t bsw,
                              int weight_kn, void* Y, int64_t ldy, int64_t bsy,
                              int64_t B, int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                              void* workspace, size_t workspace_bytes, dp_stream stream);
dp_status dp_gemm_dgrad_batched(const void* dY, int64_t ldg, int64_t bsg, const void* W, int64_t ldw, int64_t bsw,
                                int weight_kn, void* dX, int64_t ldx, int64_t bsx,
                                int64_t B, int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                                void* workspace, size_t workspace_bytes, dp_stream stream);
dp_status dp_gemm_wgrad_batched(const void* dY, int64_t ldg, int64_t bsg, const void* X, int64_t ldx, int64_t bsx,
                                void* dW, int64_t ldw, int64_t bsw, int weight_kn,
                                int64_t B, int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                                void* workspace, size_t workspace_bytes, dp_stream stream);

/* -------------------------------------------------------- backward pass (BF16) */
/* Input gradient and weight gradient of one layer from the same dY (the pages'
 * "bwd" op is dgrad + wgrad, [router] benchmark rows):
 *   dX[t][k] = sum_n dY[t][n] * W[n][k]      (as dp_gemm_dgrad_ex)
 *   dW[n][k] = sum_t dY[t][n] * X[t][k]      (as dp_gemm_wgrad_ex)
 * with their own output precisions and leading dimensions.  The planner picks one
 * of two forms (dp_plan_query_bwd reports which):
 *   - the two single-op calls, one after the other on `stream`, sharing the
 *     workspace (bitwise the same as calling dp_gemm_dgrad_ex, dp_gemm_wgrad_ex);
 *   - one co-scheduled launch: both problems tiled alike (one tile shape) with
 *     whole K per tile, their tiles in one list dealt to one persistent grid, so
 *     the SMs left idle by one problem's last wave run the other's tiles.  Needs
 *     no workspace.  Every output element is the same whole-K sum a whole-K
 *     single-op plan computes.
 * Chosen when the cost model expects the co-scheduled launch to be at least 3%
 * faster (small and mid-size T, where each single-op launch leaves SMs idle);
 * DP_FORCE_FUSE (with DP_TUNING, see below) overrides (0: two calls; 1:
 * co-scheduled; 2 / 3: co-scheduled with the weight / input gradient's tiles
 * first).  dX and dW must not overlap
 * dY, X or W.
 * Arguments and errors as the single-op calls; workspace: dp_workspace_size_bwd. */
dp_status dp_gemm_bwd(const void* dY, int64_t ldg, const void* X, int64_t ldx, const void* W, int64_t ldw,
                      void* dX, int64_t ld_dx, dp_out_dtype out_dx, void* dW, int64_t ld_dw, dp_out_dtype out_dw,
                      int64_t T, int64_t N, int64_t K, int deterministic,
                      void* workspace, size_t workspace_bytes, dp_stream stream);

/* ----------------------------------------------------------------- router ops */
/* [router]: FP32 operands and FP32 output; N is the expert count (256 on the
 * pages) and K the hidden size.  Each FP32 operand value x is split into bf16
 * hi = RNE(x) and lo = RNE(x - hi); every product a*b is formed as
 * hi_a*hi_b + hi_a*lo_b + lo_a*hi_b on the BF16 tensor cores with FP32
 * accumulation (lo_a*lo_b is dropped).  The operand the whole output reuses (W,
 * or dY for the weight gradient; both for the input gradient) is split once per
 * call into bf16 copies in the workspace; the streamed FP32 operand is split
 * inside the GEMM.  The weight gradient is computed as dW^T = X^T dY and stored
 * transposed.
 * Small T (a few hundred tokens or fewer, as the planner's cost model decides;
 * dp_plan_info.program reports it): a SIMT FP32 program instead -- the plain
 * FP32 contraction with FP32 fused multiply-adds on the CUDA cores, in one launch
 * and without workspace, each output tile's contraction split over the CTAs of a
 * thread-block cluster whose partials are summed in a fixed order (so the output
 * is bitwise repeatable; its error is the FP32 rounding of the sum, below the
 * BF16x3 program's).  DP_FORCE_FFMA=0 / 1 (with DP_TUNING, see below) forces
 * either program (1: where the forced tile width and split count, if any, fit the
 * shape). */

/* Router forward: Y[t][n] = sum_k X[t][k] * W[n][k];  X: T x K, W: N x K, Y: T x N. */
dp_status router_fwd(const float* X, const float* W, float* Y,
                     int64_t T, int64_t N, int64_t K, int deterministic,
                     void* workspace, size_t workspace_bytes, dp_stream stream);
dp_status router_fwd_ex(const float* X, int64_t ldx, const float* W, int64_t ldw,
                        float* Y, int64_t ldy, int64_t T, int64_t N, int64_t K, int deterministic,
                        void* workspace, size_t workspace_bytes, dp_stream stream);

/* Router input gradient: dX[t][k] = sum_n dY[t][n] * W[n][k];  dY: T x N, dX: T x K. */
dp_status router_dgrad(const float* dY, const float* W, float* dX,
                       int64_t T, int64_t N, int64_t K, int deterministic,
                       void* workspace, size_t workspace_bytes, dp_stream stream);
dp_status router_dgrad_ex(const float* dY, int64_t ldg, const float* W, int64_t ldw,
                          float* dX, int64_t ldx, int64_t T, int64_t N, int64_t K, int deterministic,
                          void* workspace, size_t workspace_bytes, dp_stream stream);

/* Router weight gradient: dW[n][k] = sum_t dY[t][n] * X[t][k];  dW: N x K. */
dp_status router_wgrad(const float* dY, const float* X, float* dW,
                       int64_t T, int64_t N, int64_t K, int deterministic,
                       void* workspace, size_t workspace_bytes, dp_stream stream);
dp_status router_wgrad_ex(const float* dY, int64_t ldg, const float* X, int64_t ldx,
                          float* dW, int64_t ldw, int64_t T, int64_t N, int64_t K, int deterministic,
                          void* workspace, size_t workspace_bytes, dp_stream stream);

/* ------------------------------------------------------------ planning, misc */
/* Tuning and test overrides.  They are read from the environment only in a
 * process that has DP_TUNING set when the library first plans a call; such a
 * process reads them again on every call (so a test can change them between
 * calls).  Without DP_TUNING no call reads the environment.  The variables:
 * DP_FORCE_BN (64 / 128 / 256), DP_FORCE_SPLITS (uniform split count),
 * DP_FORCE_TAIL_SPLITS (split only the last partial wave, this many ways),
 * DP_FORCE_SWAP (0 / 1: BF16 weight-gradient orientation), DP_FORCE_PAIR (0 / 1:
 * single-CTA or CTA-pair tiles), DP_FORCE_CLUSTER_SUM=0 (sum split partials in
 * the reduction kernel instead of inside the GEMM's clusters; the two give the
 * same bits), DP_FORCE_TMA_STORE (0 / 1: the epilogue's whole-tile TMA stores off
 * / on for every non-transposed output; both store paths give the same bits),
 * DP_FORCE_STORE2=0 (FP32 whole tiles store one 32 x 32 block per TMA store
 * instead of two; the same bits), DP_FORCE_EPI_SINGLE=1 (one TMA-store staging
 * block per epilogue warp instead of two; the same bits), DP_FORCE_EVICT_FIRST=0
 * (no L2 evict-first policy on the operand a launch reads once; the same bits),
 * DP_FORCE_FUSE (0 / 1 / 2 / 3: dp_gemm_bwd as two calls or as one co-scheduled
 * launch, see dp_gemm_bwd), DP_FORCE_STREAM_K (0: never; 1: a stream-K plan where
 * the shape admits one), DP_FORCE_ATOMIC (calls with deterministic = 0: 0 ordered
 * split sums, 1 atomic ones wherever admitted), DP_FORCE_KPS (1 / 2 contraction
 * blocks per ring stage; BF16x3 plans keep 1), DP_FORCE_FFMA (0 / 1: the router's
 * BF16x3 or SIMT program), DP_FORCE_GROUP (raster group width in tiles) and
 * DP_FORCE_RASTER_M (1: groups of row tiles, 0: of column tiles).
 * A forced plan is still deterministic and keeps the accumulation-length bound. */

/* The plan the library uses for one call.  The planner is a pure function of
 * (op, T, N, K, out, sm_count), so a workspace sized here fits the call. */
typedef struct dp_plan_info {
    int32_t block_m;          /* output tile rows (128, or 256 for a CTA pair) */
    int32_t block_n;          /* output tile columns (64, 128 or 256) */
    int32_t block_k;          /* contraction block (64 elements = 64 tokens for wgrad; 32 for
                                 the router's forward and weight gradient) */
    int32_t stages;           /* shared-memory pipeline depth */
    int32_t splits;           /* contraction splits per output tile (1 = whole K per tile) */
    int32_t raster_group;     /* tiles per raster group (columns, or rows if raster_rows) */
    int32_t grid;             /* persistent CTAs launched (<= sm_count; even for a pair) */
    int32_t a_mn_major;       /* A operand read MN-major (1) or K-major (0) */
    int32_t b_mn_major;       /* B operand read MN-major (1) or K-major (0) */
    int32_t swap_ab;          /* weight gradient as dW^T = X^T dY (thin N as the MMA's N),
                                 stored transposed into dW */
    int32_t cta_pair;         /* 1: tiles of 256 rows shared by a cluster of two CTAs */
    int32_t raster_rows;      /* 1: raster groups of row tiles, rows fastest (B is the larger
                                 operand, or more than half the L2) */
    int32_t stream_k;         /* 1: the grid's slots share all tiles' contraction blocks evenly
                                 (slot c takes blocks [c W / grid_slots, (c + 1) W / grid_slots)
                                 of the tile-major order, W = tiles * k_blocks); a tile cut by
                                 slot boundaries is summed from up to `splits` pieces in block
                                 order; units counts the pieces */
    int64_t gemm_m;           /* output rows of the contraction */
    int64_t gemm_n;           /* output columns */
    int64_t gemm_k;           /* contraction length (3N for the router's input gradient,
                                 which contracts concatenated [lo|hi|hi] x [hi;lo;hi] copies) */
    int64_t tiles_m;
    int64_t tiles_n;
    int64_t k_blocks;         /* ceil(gemm_k / block_k) */
    int64_t units;            /* full_units + (tiles_m * tiles_n - full_units) * splits */
    int64_t full_units;       /* leading whole-K units; the remaining tiles are split */
    uint64_t workspace_bytes; /* == dp_workspace_size() */
    double model_us;          /* the planner's modelled duration of the call (diagnostic) */
    int64_t batch;            /* independent problems in the launch (1 except batched calls) */
    int64_t tiles;            /* batch * tiles_m * tiles_n */
    int32_t weight_kn;        /* batched calls: W / dW stored [K][N] */
    int32_t program;          /* router: 0 tensor-core BF16x3 program, 1 SIMT FP32 program
                                 (64 x block_n tiles, `splits` CTAs per tile, block_k
                                 contraction elements per stage); BF16 ops: 0 */
    int32_t atomic;           /* 1: split units add into the zero-filled FP32 output with
                                 atomic adds (deterministic = 0 only) */
    int32_t blocks_per_stage; /* contraction blocks per stage of the operand ring (1 or 2: a
                                 stage's loads complete on one barrier, so streaming plans
                                 carry two blocks per stage in half as many stages) */
    int32_t cluster_sum;      /* split plans with one unit per CTA: the tile's `splits` CTAs
                                 run as one thread-block cluster and sum their partials
                                 themselves after the main loop, with no reduction kernel
                                 (the cluster size, 2..8).  0: the reduction kernel sums the
                                 split partials, or the plan has none.  It depends on how
                                 many such clusters the device runs at once, so it is known
                                 only for the current device (sm_count <= 0); -1 otherwise */
} dp_plan_info;

/* Fill `info` with the plan for a call on a GPU with `sm_count` SMs
 * (sm_count <= 0: query the current device).  Pure host function. */
dp_status dp_plan_query(dp_op op, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                        int sm_count, dp_plan_info* info);
/* The same for a call with the given `deterministic` flag (dp_plan_query is
 * deterministic = 1).  A non-deterministic plan needs no more workspace than the
 * deterministic one of the same call. */
dp_status dp_plan_query_ex(dp_op op, int64_t T, int64_t N, int64_t K, dp_out_dtype out, int deterministic,
                           int sm_count, dp_plan_info* info);
/* The same for a batched BF16 call (op DP_OP_FWD / DGRAD / WGRAD, B >= 1). */
dp_status dp_plan_query_batched(dp_op op, int64_t B, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                                int weight_kn, int sm_count, dp_plan_info* info);

/* The backward pass's plan: the form chosen and the plan of each problem (for the
 * co-scheduled launch, whole-K plans of one tile shape; grid is the launch's). */
typedef struct dp_bwd_plan_info {
    int32_t fused;            /* 1: one co-scheduled launch; 0: two single-op calls */
    int32_t wgrad_first;      /* co-scheduled: the weight gradient's tiles are dealt first */
    int32_t grid;             /* co-scheduled: persistent CTAs of the launch (else 0) */
    int32_t blocks_per_stage; /* co-scheduled: contraction blocks per ring stage, for both
                                 problems (else 0; each call's own is in dgrad / wgrad) */
    double model_us;          /* modelled duration of the chosen form */
    double separate_us;       /* modelled duration of the two single-op calls */
    uint64_t workspace_bytes; /* == dp_workspace_size_bwd() */
    dp_plan_info dgrad;       /* input-gradient problem */
    dp_plan_info wgrad;       /* weight-gradient problem */
} dp_bwd_plan_info;
dp_status dp_plan_query_bwd(int64_t T, int64_t N, int64_t K, dp_out_dtype out_dx, dp_out_dtype out_dw,
                            int sm_count, dp_bwd_plan_info* info);

/* Workspace bytes a call needs (see dp_plan_query for sm_count). */
dp_status dp_workspace_size(dp_op op, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                            int sm_count, size_t* bytes);
dp_status dp_workspace_size_batched(dp_op op, int64_t B, int64_t T, int64_t N, int64_t K, dp_out_dtype out,
                                    int weight_kn, int sm_count, size_t* bytes);
dp_status dp_workspace_size_bwd(int64_t T, int64_t N, int64_t K, dp_out_dtype out_dx, dp_out_dtype out_dw,
                                int sm_count, size_t* bytes);

/* Check the device's architecture and set kernel attributes on `device`
 * (the current device if < 0).  Optional: the first call on a device does it. */
dp_status dp_init(int device);

/* Debug read-out: synchronise the current device and report whether any kernel
 * of this library gave up waiting (DP_ERR_TIMEOUT) since the last clear.
 * `clear` != 0 resets the flag.  Not for use inside stream capture. */
dp_status dp_device_error(int clear);

/* Test entry for the kernels' bounded waits (the failure-detection path).  Every
 * barrier wait in this library's kernels gives up after a time limit that is a
 * launch argument (2 s in the calls above), records the fault in the device status
 * word that dp_device_error() reports as DP_ERR_TIMEOUT, and lets the kernel
 * unwind and return instead of hanging the GPU.  This call enqueues on `stream` one
 * CTA that waits through that same bounded wait, with limit `limit_ns`
 * (1e3 .. 2e9 ns, else DP_ERR_INVALID_ARG), on a shared-memory barrier that nothing
 * arrives on (arrive = 0: the wait runs out and the kernel records the timeout) or
 * that the waiting thread arrived on first (arrive != 0: it returns at once and
 * records nothing).  The kernel holds no TMEM and issues no copies, so it ends
 * either way and the stream stays usable.  No counterpart on the pages: it exists
 * so the timeout path can be tested on a GPU without faulting or hanging one. */
dp_status dp_wait_probe(uint64_t limit_ns, int arrive, dp_stream stream);

/* Static description of a status code. */
const char* dp_status_string(dp_status status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int dp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DP_GEMM_H */
