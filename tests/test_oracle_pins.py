"""Pins that hold the FP64 oracle to something other than itself.

Each check below is chosen so that a plausible slip in ``oracle/oracle.c`` -- a
transposed operand, a wrong index or sign, a dropped BF16x3 term, a wrong
rounding -- fails at least one of them:

  * brute force against exact Python-integer triple loops (layout, indexing,
    sign, transposition of all three operations, bf16 and fp32 inputs);
  * the adjoint identity <dY, X W^T> = <dY W, X> = <dY^T X, W> (pairs the two
    gradients with the forward);
  * special cases: identity weights, one-hot gradients;
  * BF16x3: hand-worked split and product fixtures, exactness on hi-only inputs,
    the split's error bound, and the three-term error bound against FP64;
  * round-to-nearest-even fixtures from the binary32/bfloat16 formats and
    agreement with torch's bf16 cast (a library routine).

Definitions follow the FlashInfer pages on the Cake dense projection GEMMs:
forward with K-major B and input gradient with MN-major B ("plan the 4096 ->
12288 input gradient ...", body), weight gradient over the tokens ("restore
the K1 weight-gradient routes ...", body), router via BF16x3 ("cache the
router entry points' calls by their own tensors", summary).
"""
import os
import struct

import numpy as np
import pytest
import torch

import oracle
from fp32_dense_projection_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def _f32_from_bits(h: str) -> np.float32:
    return np.frombuffer(struct.pack("<I", int(h, 16)), dtype=np.float32)[0]


# ------------------------------------------------------------- brute force

def _int_matmul(A, B):
    """Exact integer product of Python-int nested lists: C[i][j] = sum_p A[i][p] B[p][j]."""
    n, p, m = len(A), len(B), len(B[0])
    return [[sum(A[i][q] * B[q][j] for q in range(p)) for j in range(m)] for i in range(n)]


def _T(A):
    return [list(r) for r in zip(*A)]


def _as_int(t: torch.Tensor):
    return t.to(torch.int64).tolist()


SHAPES = [(1, 1, 1), (2, 3, 5), (5, 3, 7), (17, 8, 65), (3, 17, 2), (65, 5, 3), (1, 129, 2)]


@pytest.mark.parametrize("T,N,K", SHAPES)
def test_brute_force_integer_bf16(T, N, K):
    c = inputs.integer_case(T, N, K, seed=T * 100 + N * 10 + K)
    X, W, dY = _as_int(c["X"]), _as_int(c["W"]), _as_int(c["dY"])
    Y = _int_matmul(X, _T(W))          # Y[t][n] = sum_k X[t][k] W[n][k]
    dX = _int_matmul(dY, W)            # dX[t][k] = sum_n dY[t][n] W[n][k]
    dW = _int_matmul(_T(dY), X)        # dW[n][k] = sum_t dY[t][n] X[t][k]
    assert np.array_equal(oracle.fwd_bf16(c["X"], c["W"]), np.array(Y, np.float64))
    assert np.array_equal(oracle.dgrad_bf16(c["dY"], c["W"]), np.array(dX, np.float64))
    assert np.array_equal(oracle.wgrad_bf16(c["dY"], c["X"]), np.array(dW, np.float64))


@pytest.mark.parametrize("T,N,K", SHAPES[:5])
def test_brute_force_integer_f32_and_x3(T, N, K):
    c = inputs.integer_case(T, N, K, seed=7 + T + N + K, dtype=torch.float32)
    X, W, dY = _as_int(c["X"]), _as_int(c["W"]), _as_int(c["dY"])
    Y = np.array(_int_matmul(X, _T(W)), np.float64)
    dX = np.array(_int_matmul(dY, W), np.float64)
    dW = np.array(_int_matmul(_T(dY), X), np.float64)
    assert np.array_equal(oracle.fwd_f32(c["X"], c["W"]), Y)
    assert np.array_equal(oracle.dgrad_f32(c["dY"], c["W"]), dX)
    assert np.array_equal(oracle.wgrad_f32(c["dY"], c["X"]), dW)
    # integers in [-3, 3] are bf16-exact, so the BF16x3 split has lo = 0
    assert np.array_equal(oracle.fwd_bf16x3(c["X"], c["W"]), Y)
    assert np.array_equal(oracle.dgrad_bf16x3(c["dY"], c["W"]), dX)
    assert np.array_equal(oracle.wgrad_bf16x3(c["dY"], c["X"]), dW)


def test_sampled_matches_full():
    T, N, K = 33, 24, 40
    c = inputs.dense_projection(T, N, K, seed=3)
    rng = np.random.default_rng(0)
    for fn_full, fn_at, a, b, shape in (
        (oracle.fwd_bf16, oracle.fwd_bf16_at, c["X"], c["W"], (T, N)),
        (oracle.dgrad_bf16, oracle.dgrad_bf16_at, c["dY"], c["W"], (T, K)),
        (oracle.wgrad_bf16, oracle.wgrad_bf16_at, c["dY"], c["X"], (N, K)),
    ):
        full = fn_full(a, b)
        r = rng.integers(0, shape[0], 50)
        cc = rng.integers(0, shape[1], 50)
        assert np.array_equal(fn_at(a, b, r, cc), full[r, cc])
    cf = inputs.router(T, K, seed=3, experts=N)
    for fn_full, fn_at, a, b, shape in (
        (oracle.fwd_f32, oracle.fwd_f32_at, cf["X"], cf["W"], (T, N)),
        (oracle.dgrad_f32, oracle.dgrad_f32_at, cf["dY"], cf["W"], (T, K)),
        (oracle.wgrad_f32, oracle.wgrad_f32_at, cf["dY"], cf["X"], (N, K)),
    ):
        full = fn_full(a, b)
        r = rng.integers(0, shape[0], 50)
        cc = rng.integers(0, shape[1], 50)
        assert np.array_equal(fn_at(a, b, r, cc), full[r, cc])


# ---------------------------------------------------------- adjoint identity

def _inner(a, b):
    return float(np.sum(np.asarray(a, np.float64) * np.asarray(b, np.float64)))


@pytest.mark.parametrize("T,N,K", [(7, 5, 3), (64, 24, 40), (65, 16, 129)])
def test_adjoint_identity_bf16(T, N, K):
    c = inputs.dense_projection(T, N, K, seed=11)
    X = oracle.bf16_to_f64(c["X"])
    W = oracle.bf16_to_f64(c["W"])
    dY = oracle.bf16_to_f64(c["dY"])
    a = _inner(dY, oracle.fwd_bf16(c["X"], c["W"]))
    b = _inner(oracle.dgrad_bf16(c["dY"], c["W"]), X)
    d = _inner(oracle.wgrad_bf16(c["dY"], c["X"]), W)
    # all three equal sum_{t,n,k} dY[t,n] X[t,k] W[n,k]; they differ only by FP64 rounding in
    # different summation orders, bounded by (T + N + K) * 2^-53 * sum |dY| |X| |W|
    mag = float(np.sum(np.abs(dY) * (np.abs(X) @ np.abs(W).T)))
    tol = (T + N + K) * 2.0**-53 * mag
    assert abs(a - b) <= tol
    assert abs(a - d) <= tol


def test_adjoint_identity_integer_exact():
    T, N, K = 13, 11, 9
    c = inputs.integer_case(T, N, K, seed=5)
    X = oracle.bf16_to_f64(c["X"])
    W = oracle.bf16_to_f64(c["W"])
    dY = oracle.bf16_to_f64(c["dY"])
    a = _inner(dY, oracle.fwd_bf16(c["X"], c["W"]))
    b = _inner(oracle.dgrad_bf16(c["dY"], c["W"]), X)
    d = _inner(oracle.wgrad_bf16(c["dY"], c["X"]), W)
    assert a == b == d


def test_adjoint_identity_f32():
    T, N, K = 31, 16, 48
    c = inputs.router(T, K, seed=2, experts=N)
    a = _inner(c["dY"].numpy(), oracle.fwd_f32(c["X"], c["W"]))
    b = _inner(oracle.dgrad_f32(c["dY"], c["W"]), c["X"].numpy())
    d = _inner(oracle.wgrad_f32(c["dY"], c["X"]), c["W"].numpy())
    assert abs(a - b) <= 1e-10 * (abs(a) + 1)
    assert abs(a - d) <= 1e-10 * (abs(a) + 1)


# ------------------------------------------------------------ special cases

def test_identity_weight():
    T, K = 9, 16
    X = inputs.normal((T, K), seed=1, role=inputs.ROLE_X)
    eye = torch.eye(K, dtype=torch.bfloat16)
    assert np.array_equal(oracle.fwd_bf16(X, eye), oracle.bf16_to_f64(X))
    # dgrad with W = I returns dY
    assert np.array_equal(oracle.dgrad_bf16(X, eye), oracle.bf16_to_f64(X))


def test_one_hot_gradient_selects_rows():
    T, N, K = 12, 5, 8
    X = inputs.normal((T, K), seed=4, role=inputs.ROLE_X)
    W = inputs.normal((N, K), seed=4, role=inputs.ROLE_W)
    pick = [(3 * t + 1) % N for t in range(T)]
    dY = torch.zeros(T, N, dtype=torch.bfloat16)
    for t, p in enumerate(pick):
        dY[t, p] = 1.0
    Xd = oracle.bf16_to_f64(X)
    Wd = oracle.bf16_to_f64(W)
    # input gradient: row t of dX is row pick[t] of W
    assert np.array_equal(oracle.dgrad_bf16(dY, W), Wd[pick])
    # weight gradient: row n of dW is the sum of the X rows routed to n, in token order
    dW = oracle.wgrad_bf16(dY, X)
    for n in range(N):
        s = np.zeros(K)
        for t in range(T):
            if pick[t] == n:
                s = s + Xd[t]
        assert np.array_equal(dW[n], s)


def test_empty_token_count():
    X = torch.zeros(0, 16, dtype=torch.bfloat16)
    dY = torch.zeros(0, 8, dtype=torch.bfloat16)
    W = inputs.normal((8, 16), seed=0, role=inputs.ROLE_W)
    assert oracle.fwd_bf16(X, W).shape == (0, 8)
    assert oracle.dgrad_bf16(dY, W).shape == (0, 16)
    assert np.array_equal(oracle.wgrad_bf16(dY, X), np.zeros((8, 16)))


# ------------------------------------------------------------------- rounding

def test_rne_golden():
    for fbits, want, *_ in _rows("bf16_rne.txt"):
        x = _f32_from_bits(fbits)
        got = int(oracle.f32_to_bf16(np.array([x], np.float32))[0])
        assert got == int(want, 16), (fbits, hex(got), want)


def test_rne_matches_torch_cast():
    rng = np.random.default_rng(123)
    u = rng.integers(0, 2**32, 200_000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    got = oracle.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_widen_is_exact():
    b = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    w = oracle.bf16_to_f64(b)
    f = (b.astype(np.uint32) << 16).view(np.float32)
    fin = np.isfinite(f)
    assert np.array_equal(w[fin], f[fin].astype(np.float64))


# -------------------------------------------------------------------- BF16x3

def test_split_golden():
    for xb, hb, lb, *_ in _rows("bf16x3_split.txt"):
        x = np.array([_f32_from_bits(xb)], np.float32)
        hi, lo = oracle.split_bf16x3(x)
        assert (int(hi[0]), int(lo[0])) == (int(hb, 16), int(lb, 16)), xb


def test_product_golden():
    for xb, wb, exact, x3, *_ in _rows("bf16x3_products.txt"):
        X = np.array([[_f32_from_bits(xb)]], np.float32)
        W = np.array([[_f32_from_bits(wb)]], np.float32)
        assert oracle.fwd_f32(X, W)[0, 0] == float(exact)
        assert oracle.fwd_bf16x3(X, W)[0, 0] == float(x3)
        # the same single product through the two gradient forms
        assert oracle.dgrad_bf16x3(X, W)[0, 0] == float(x3)
        assert oracle.wgrad_bf16x3(X, W)[0, 0] == float(x3)


def test_split_error_bound():
    # |x - hi| <= 2^-8 |x| (RNE to 8 significant bits); |x - hi - lo| <= 2^-16 |x|
    x = inputs.normal((100_000,), seed=9, role=1, dtype=torch.float32).numpy()
    x = np.concatenate([x, x * 1e-20, x * 1e20])
    hi, lo = oracle.split_bf16x3(x)
    h = oracle.bf16_to_f64(hi)
    l_ = oracle.bf16_to_f64(lo)
    xd = x.astype(np.float64)
    assert np.all(np.abs(xd - h) <= 2.0**-8 * np.abs(xd))
    assert np.all(np.abs(xd - h - l_) <= 2.0**-16 * np.abs(xd))
    # hi is the nearest bf16: neither neighbour is strictly closer
    for d in (-1, 1):
        nb = oracle.bf16_to_f64((hi.astype(np.int32) + d).astype(np.uint16))
        ok = np.isfinite(nb) & (np.sign(nb) == np.sign(h))
        assert np.all(np.abs(xd - h)[ok] <= np.abs(xd - nb)[ok])


def test_hi_only_inputs_are_exact():
    # FP32 inputs that are bf16-representable give lo = 0: BF16x3 == plain FP64, bitwise
    T, N, K = 40, 24, 72
    c = inputs.router(T, K, seed=21, experts=N)
    X = c["X"].to(torch.bfloat16).float()
    W = c["W"].to(torch.bfloat16).float()
    dY = c["dY"].to(torch.bfloat16).float()
    assert np.array_equal(oracle.fwd_bf16x3(X, W), oracle.fwd_f32(X, W))
    assert np.array_equal(oracle.dgrad_bf16x3(dY, W), oracle.dgrad_f32(dY, W))
    assert np.array_equal(oracle.wgrad_bf16x3(dY, X), oracle.wgrad_f32(dY, X))


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_bf16x3_error_bound(op):
    # x = hi + lo + e, |e| <= 2^-16|x|, |lo| <= 2^-8|x|(1+2^-8): per product the dropped part is
    # below 3.1 * 2^-16 |x||w|.  A dropped hi*lo or lo*hi term (about 2^-8 |x||w|) breaks this.
    T, N, K = 24, 16, 80
    c = inputs.router(T, K, seed=33, experts=N)
    X, W, dY = c["X"].numpy(), c["W"].numpy(), c["dY"].numpy()
    f = {"fwd": (oracle.fwd_bf16x3, oracle.fwd_f32, np.abs(X).astype(np.float64) @ np.abs(W).T.astype(np.float64), X, W),
         "dgrad": (oracle.dgrad_bf16x3, oracle.dgrad_f32, np.abs(dY).astype(np.float64) @ np.abs(W).astype(np.float64), dY, W),
         "wgrad": (oracle.wgrad_bf16x3, oracle.wgrad_f32, np.abs(dY).T.astype(np.float64) @ np.abs(X).astype(np.float64), dY, X)}[op]
    x3, exact, mag, a, b = f
    err = np.abs(x3(a, b) - exact(a, b))
    assert np.all(err <= 3.1 * 2.0**-16 * mag + 1e-300)
    # and the emulation is not trivially exact: the dropped lo*lo term is visible
    assert err.max() > 0
    # a two-term variant (hi*hi + hi*lo) would miss by about 2^-9 |x||w|: far above the bound
    assert 3.1 * 2.0**-16 < 2.0**-10
