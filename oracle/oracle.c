/*
 * FP64 oracle for the dense projection GEMM family.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only in the seeded input tensors they both read.
 *
 * What it computes is the plain definition of each contraction, widened
 * exactly to FP64 and summed in natural index order.  The pages describe three
 * operations of a projection layer Y = X W^T and one FP32 router GEMM:
 *
 *   forward          Y[t][n]  = sum_k X[t][k]  * W[n][k]      (X: T x K, W: N x K)
 *   input gradient  dX[t][k]  = sum_n dY[t][n] * W[n][k]      (dY: T x N)
 *   weight gradient dW[n][k]  = sum_t dY[t][n] * X[t][k]      (sum over the T tokens)
 *
 * Sources (FlashInfer pull-request pages on the "Cake" dense projection GEMMs):
 *   - "perf(cake_dense_projection_det_gemm): plan the 4096 -> 12288 input
 *     gradient with the row-half-release program at T-exact keys", body:
 *     the forward form takes a K-major B, the input gradient an MN-major B.
 *   - "perf(cake_dense_projection_gemm): restore the K1 weight-gradient routes
 *     ...", body: the weight gradient contracts over the tokens in 64-token K
 *     blocks; BF16 or FP32 output; the FP64 error budgets.
 *   - "perf(cake_dense_projection_gemm): cache the router entry points' calls by
 *     their own tensors", summary: router GEMM [T,H] x [256,H]^T with FP32
 *     inputs and outputs, computed through BF16x3 emulation.
 *
 * The 64-token blocking of the weight gradient is a partition of the sum over
 * t; zeros past the last token add nothing, so the definition here sums every
 * token once, in order.
 *
 * BF16x3 (router): each FP32 operand x is split into bf16 hi = RNE(x) and
 * lo = RNE(x - hi); the product x*w is replaced by hi_x*hi_w + hi_x*lo_w +
 * lo_x*hi_w (lo_x*lo_w dropped).  The pages name the method ("BF16x3
 * emulation", "exact BF16x3 split") but not its rounding or term list; this
 * file takes round-to-nearest-even for both halves and the three-term list.
 * Each bf16 x bf16 product is exact in FP64 (8 + 8 significant bits).
 *
 * Parity pins (tests/test_oracle_pins.py) hold this file to brute force over
 * Python integers, the adjoint identity, hi-only exactness of BF16x3, closed
 * forms of the split, and IEEE round-to-nearest-even fixtures.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (contraction off so
 * that no fused multiply-add changes a rounding on any host).
 */
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- scalar conversions ------------------------------------------------- */

/* bfloat16 is the upper half of an IEEE binary32: widening is exact. */
static double bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary32 -> bfloat16, round to nearest, ties to even, by integer bits.
 * Adding 0x7FFF plus the lowest kept bit and truncating rounds to nearest with
 * ties going to the even neighbour; a carry out of the fraction moves to the
 * next binade and, past the largest finite value, to infinity, as IEEE
 * rounding requires.  NaN keeps its sign and becomes a quiet NaN. */
uint16_t oracle_f32_to_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7FFFu + keep_lsb;
    return (uint16_t)(u >> 16);
}

double oracle_bf16_to_f64(uint16_t b) { return bf16_to_f64(b); }

/* BF16x3 split of n FP32 values: hi = RNE(x), lo = RNE(x - hi).  x - hi is
 * formed in FP64, where it is exact, then narrowed to binary32, which is exact
 * as well (it has at most 24 significant bits). */
void oracle_split_bf16x3(const float* x, uint16_t* hi, uint16_t* lo, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        uint16_t h = oracle_f32_to_bf16_rne(x[i]);
        float rest = (float)((double)x[i] - bf16_to_f64(h));
        hi[i] = h;
        lo[i] = oracle_f32_to_bf16_rne(rest);
    }
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- one output element per operation ----------------------------------- */
/* Row-major, contiguous operands.  Each function is the definition, term by
 * term, in natural index order. */

/* forward, BF16 operands: Y[t][n] = sum_k X[t][k] * W[n][k] */
static double fwd_elem_bf16(const uint16_t* X, const uint16_t* W,
                            int64_t K, int64_t t, int64_t n)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
        s += bf16_to_f64(X[t * K + k]) * bf16_to_f64(W[n * K + k]);
    return s;
}

/* input gradient, BF16 operands: dX[t][k] = sum_n dY[t][n] * W[n][k] */
static double dgrad_elem_bf16(const uint16_t* dY, const uint16_t* W,
                              int64_t N, int64_t K, int64_t t, int64_t k)
{
    double s = 0.0;
    for (int64_t n = 0; n < N; ++n)
        s += bf16_to_f64(dY[t * N + n]) * bf16_to_f64(W[n * K + k]);
    return s;
}

/* weight gradient, BF16 operands: dW[n][k] = sum_t dY[t][n] * X[t][k] */
static double wgrad_elem_bf16(const uint16_t* dY, const uint16_t* X,
                              int64_t T, int64_t N, int64_t K, int64_t n, int64_t k)
{
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t)
        s += bf16_to_f64(dY[t * N + n]) * bf16_to_f64(X[t * K + k]);
    return s;
}

/* the same three definitions on FP32 operands (router, plain FP64 reference) */
static double fwd_elem_f32(const float* X, const float* W,
                           int64_t K, int64_t t, int64_t n)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
        s += (double)X[t * K + k] * (double)W[n * K + k];
    return s;
}

static double dgrad_elem_f32(const float* dY, const float* W,
                             int64_t N, int64_t K, int64_t t, int64_t k)
{
    double s = 0.0;
    for (int64_t n = 0; n < N; ++n)
        s += (double)dY[t * N + n] * (double)W[n * K + k];
    return s;
}

static double wgrad_elem_f32(const float* dY, const float* X,
                             int64_t T, int64_t N, int64_t K, int64_t n, int64_t k)
{
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t)
        s += (double)dY[t * N + n] * (double)X[t * K + k];
    return s;
}

/* BF16x3 restatement: operands already split into (hi, lo) bf16 halves.
 * product(a, b) ~ a_hi*b_hi + a_hi*b_lo + a_lo*b_hi, summed in FP64. */
static double x3(uint16_t ah, uint16_t al, uint16_t bh, uint16_t bl)
{
    double a_hi = bf16_to_f64(ah), a_lo = bf16_to_f64(al);
    double b_hi = bf16_to_f64(bh), b_lo = bf16_to_f64(bl);
    return a_hi * b_hi + a_hi * b_lo + a_lo * b_hi;
}

static double fwd_elem_x3(const uint16_t* Xh, const uint16_t* Xl,
                          const uint16_t* Wh, const uint16_t* Wl,
                          int64_t K, int64_t t, int64_t n)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
        s += x3(Xh[t * K + k], Xl[t * K + k], Wh[n * K + k], Wl[n * K + k]);
    return s;
}

static double dgrad_elem_x3(const uint16_t* Gh, const uint16_t* Gl,
                            const uint16_t* Wh, const uint16_t* Wl,
                            int64_t N, int64_t K, int64_t t, int64_t k)
{
    double s = 0.0;
    for (int64_t n = 0; n < N; ++n)
        s += x3(Gh[t * N + n], Gl[t * N + n], Wh[n * K + k], Wl[n * K + k]);
    return s;
}

static double wgrad_elem_x3(const uint16_t* Gh, const uint16_t* Gl,
                            const uint16_t* Xh, const uint16_t* Xl,
                            int64_t T, int64_t N, int64_t K, int64_t n, int64_t k)
{
    double s = 0.0;
    for (int64_t t = 0; t < T; ++t)
        s += x3(Gh[t * N + n], Gl[t * N + n], Xh[t * K + k], Xl[t * K + k]);
    return s;
}

/* ---- full outputs --------------------------------------------------------- */
/* Row loop parallel over threads; every element is still one ordered sum. */

void oracle_fwd_bf16(const uint16_t* X, const uint16_t* W, double* Y,
                     int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n)
            Y[t * N + n] = fwd_elem_bf16(X, W, K, t, n);
}

void oracle_dgrad_bf16(const uint16_t* dY, const uint16_t* W, double* dX,
                       int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k)
            dX[t * K + k] = dgrad_elem_bf16(dY, W, N, K, t, k);
}

void oracle_wgrad_bf16(const uint16_t* dY, const uint16_t* X, double* dW,
                       int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            dW[n * K + k] = wgrad_elem_bf16(dY, X, T, N, K, n, k);
}

void oracle_fwd_f32(const float* X, const float* W, double* Y,
                    int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n)
            Y[t * N + n] = fwd_elem_f32(X, W, K, t, n);
}

void oracle_dgrad_f32(const float* dY, const float* W, double* dX,
                      int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k)
            dX[t * K + k] = dgrad_elem_f32(dY, W, N, K, t, k);
}

void oracle_wgrad_f32(const float* dY, const float* X, double* dW,
                      int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            dW[n * K + k] = wgrad_elem_f32(dY, X, T, N, K, n, k);
}

void oracle_fwd_x3(const uint16_t* Xh, const uint16_t* Xl,
                   const uint16_t* Wh, const uint16_t* Wl, double* Y,
                   int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n)
            Y[t * N + n] = fwd_elem_x3(Xh, Xl, Wh, Wl, K, t, n);
}

void oracle_dgrad_x3(const uint16_t* Gh, const uint16_t* Gl,
                     const uint16_t* Wh, const uint16_t* Wl, double* dX,
                     int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t k = 0; k < K; ++k)
            dX[t * K + k] = dgrad_elem_x3(Gh, Gl, Wh, Wl, N, K, t, k);
}

void oracle_wgrad_x3(const uint16_t* Gh, const uint16_t* Gl,
                     const uint16_t* Xh, const uint16_t* Xl, double* dW,
                     int64_t T, int64_t N, int64_t K)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            dW[n * K + k] = wgrad_elem_x3(Gh, Gl, Xh, Xl, T, N, K, n, k);
}

/* ---- sampled outputs ------------------------------------------------------ */
/* out[i] = the element (r[i], c[i]) of the full output, for outputs too large
 * to form whole.  (r, c) is (t, n) for forward, (t, k) for the input gradient
 * and (n, k) for the weight gradient. */

void oracle_fwd_bf16_at(const uint16_t* X, const uint16_t* W, int64_t T, int64_t N, int64_t K,
                        const int64_t* r, const int64_t* c, int64_t count, double* out)
{
    (void)T; (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = fwd_elem_bf16(X, W, K, r[i], c[i]);
}

void oracle_dgrad_bf16_at(const uint16_t* dY, const uint16_t* W, int64_t T, int64_t N, int64_t K,
                          const int64_t* r, const int64_t* c, int64_t count, double* out)
{
    (void)T;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = dgrad_elem_bf16(dY, W, N, K, r[i], c[i]);
}

void oracle_wgrad_bf16_at(const uint16_t* dY, const uint16_t* X, int64_t T, int64_t N, int64_t K,
                          const int64_t* r, const int64_t* c, int64_t count, double* out)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = wgrad_elem_bf16(dY, X, T, N, K, r[i], c[i]);
}

void oracle_fwd_f32_at(const float* X, const float* W, int64_t T, int64_t N, int64_t K,
                       const int64_t* r, const int64_t* c, int64_t count, double* out)
{
    (void)T; (void)N;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = fwd_elem_f32(X, W, K, r[i], c[i]);
}

void oracle_dgrad_f32_at(const float* dY, const float* W, int64_t T, int64_t N, int64_t K,
                         const int64_t* r, const int64_t* c, int64_t count, double* out)
{
    (void)T;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = dgrad_elem_f32(dY, W, N, K, r[i], c[i]);
}

void oracle_wgrad_f32_at(const float* dY, const float* X, int64_t T, int64_t N, int64_t K,
                         const int64_t* r, const int64_t* c, int64_t count, double* out)
{
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < count; ++i)
        out[i] = wgrad_elem_f32(dY, X, T, N, K, r[i], c[i]);
}
