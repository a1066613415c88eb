"""GPU parity: every op through the C ABI against the FP64 oracle.

* exact integer cases (bitwise equal to the oracle), over ragged T and several tiles;
* the dense projection 4096 -> 1024 at T = 64, ten seeds, BF16 and FP32 output;
* the FP32 router 4096 -> 256 experts at T in {64, 256, 1024}, ten seeds;
* the thin-N weight gradients at odd 64-token block counts, BF16 and FP32 output
  (T = 1025 in full, T = 16173 sampled; the full-size shapes are in
  test_gpu_full_size.py).

Budgets (FlashInfer page "perf(cake_dense_projection_gemm): restore the K1
weight-gradient routes ...", PR body): BF16 output atol = rtol = 1e-2 with zero
violations; FP32 output rel_fro <= 5e-5 and max_abs <= 1e-3 * max|ref|.
"""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
from fp32_dense_projection_gb300 import inputs
from budgets import f32_errors
from gpu_common import (DEV, as_f64, assert_budget, bf16_min_slack, full_ref, gpu, no_device_fault, operands,
                        out_shape, record_margin, sample_points, sampled_ref, stratified_points)

pytestmark = pytest.mark.gpu


def to_dev(c):
    return {k: v.to(DEV) for k, v in c.items()}


# ------------------------------------------------------------ exact integers

TS = [1, 2, 3, 5, 17, 64, 65, 129]
NK = [(8, 16), (24, 64), (136, 8), (64, 136), (256, 200)]


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("N,K", NK)
@pytest.mark.parametrize("T", TS)
def test_integer_exact(op, T, N, K):
    # FP32 output: values in [-3, 3] keep every partial sum an exact integer.
    c = inputs.integer_case(T, N, K, seed=T + N + K)
    a, b = operands(op, c)
    ref = full_ref(op, a, b)
    d = to_dev(c)
    got = as_f64(gpu(op, *operands(op, d), out_dtype=torch.float32))
    assert np.array_equal(got, ref), (op, T, N, K, np.abs(got - ref).max())
    # BF16 output: values in [-1, 1] keep |sums| <= 256, exact in bf16.
    c = inputs.integer_case(T, N, K, seed=1 + T + N + K, lo=-1, hi=1)
    a, b = operands(op, c)
    ref = full_ref(op, a, b)
    d = to_dev(c)
    got = as_f64(gpu(op, *operands(op, d), out_dtype=torch.bfloat16))
    assert np.array_equal(got, ref), (op, T, N, K)


@pytest.mark.parametrize("op", ["router_fwd", "router_dgrad", "router_wgrad"])
@pytest.mark.parametrize("T,N,K", [(1, 8, 8), (17, 16, 72), (65, 256, 128), (129, 24, 264)])
def test_router_integer_exact(op, T, N, K):
    # integers are bf16-exact: lo = 0 and the BF16x3 result equals the exact sum
    c = inputs.integer_case(T, N, K, seed=3 * T + N, dtype=torch.float32)
    a, b = operands(op, c)
    ref = full_ref(op, a, b)
    got = as_f64(gpu(op, *operands(op, to_dev(c))))
    assert np.array_equal(got, ref), (op, T, N, K)


# ------------------------------------------ dense projection 4096 -> 1024, T = 64

@pytest.mark.parametrize("seed", range(10))
def test_dense_projection_t64(seed):
    T, N, K = 64, 1024, 4096
    c = inputs.dense_projection(T, N, K, seed=seed)
    d = to_dev(c)
    for op in ("fwd", "dgrad", "wgrad"):
        ref = full_ref(op, *operands(op, c))
        for out_dtype, name in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
            got = as_f64(gpu(op, *operands(op, d), out_dtype=out_dtype))
            record_margin(margin_cell("dense_t64", op, T, seed, name, got, ref))
            assert_budget(got, ref, name, f"{op} {name} seed {seed}")
    no_device_fault()


def margin_cell(cell, op, T, seed, out, got, ref):
    """Every element checked: the BF16 output's smallest slack to atol + rtol * |ref|, or
    the FP32 output's rel_fro and max_abs as fractions of their budgets."""
    d = {"cell": cell, "op": op, "T": T, "seed": seed, "out": out, "points": int(np.asarray(ref).size)}
    if out == "bf16":
        d["min_slack"] = bf16_min_slack(got, ref)
    else:
        rel, mx, mref = f32_errors(got, ref)
        d.update({"f32_rel_fro": rel, "f32_rel_fro_over_budget": rel / 5e-5, "f32_max_abs_over_budget": mx / (1e-3 * mref)})
    return d


# ---------------------------------------------------- FP32 router 4096 -> 256

@pytest.mark.parametrize("T", [64, 256, 1024])
@pytest.mark.parametrize("seed", range(10))
def test_router(T, seed):
    K, E = 4096, 256
    c = inputs.router(T, K, seed=seed, experts=E)
    d = to_dev(c)
    for op in ("router_fwd", "router_dgrad", "router_wgrad"):
        ref = full_ref(op, *operands(op, c))
        got = as_f64(gpu(op, *operands(op, d)))
        record_margin(margin_cell("router", op, T, seed, "f32", got, ref))
        assert_budget(got, ref, "f32", f"{op} T={T} seed {seed}")
    no_device_fault()


def test_router_other_hidden_sizes():
    for K in (5120, 6144):
        c = inputs.router(256, K, seed=5)
        d = to_dev(c)
        for op in ("router_fwd", "router_dgrad", "router_wgrad"):
            ref = full_ref(op, *operands(op, c))
            assert_budget(as_f64(gpu(op, *operands(op, d))), ref, "f32", f"{op} H={K}")


# The wide projection 4096 -> 12288 at its full sizes, and the thin weight gradient at
# T = 65537, are in test_gpu_full_size.py (ten seeds, tile-stratified samples,
# bitwise repeats and graph replay).

# ------------------------------------------------ thin-N weight gradient

THIN = [(4096, 64), (4096, 128), (4096, 512), (5120, 48), (5120, 64)]


@pytest.mark.parametrize("K,N", THIN)
def test_thin_wgrad_t1025_full(K, N):
    T = 1025
    c = inputs.thin_wgrad(T, N, K, seed=1)
    ref = full_ref("wgrad", c["dY"], c["X"])
    d = to_dev(c)
    for out_dtype, name in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
        got = as_f64(dp.dp_gemm_wgrad(d["dY"], d["X"], out_dtype=out_dtype))
        assert_budget(got, ref, name, f"wgrad {K}->{N} T={T} {name}")


@pytest.mark.parametrize("K,N", THIN)
def test_thin_wgrad_t16173_sampled(K, N):
    # eight elements in every 128 x 128 block, 1024 random ones and one full row and
    # column, into NaN-filled outputs (an unwritten element fails)
    T = 16173
    c = inputs.thin_wgrad(T, N, K, seed=2)
    d = to_dev(c)
    rng = np.random.default_rng(T + K + N)
    r1, c1 = stratified_points((N, K), rng)
    r2, c2 = sample_points((N, K), rng, n_random=1024, full_rows=1, full_cols=1)
    rows, cols = np.concatenate([r1, r2]), np.concatenate([c1, c2])
    ref = sampled_ref("wgrad", c["dY"], c["X"], rows, cols)
    ri, ci = torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)
    for out_dtype, name in ((torch.float32, "f32"), (torch.bfloat16, "bf16")):
        got = torch.full((N, K), float("nan"), dtype=out_dtype, device=DEV)
        dp.dp_gemm_wgrad(d["dY"], d["X"], out=got, out_dtype=out_dtype)
        g = got.float()[ri, ci].double().cpu().numpy()
        assert_budget(g, ref, name, f"wgrad {K}->{N} T={T} {name}")
        assert torch.isfinite(got).all()
    no_device_fault()


# ------------------------------------- split tail: whole-K full waves + split last wave

TAIL_CASES = [("fwd", 2048, 2560, 2048), ("dgrad", 2048, 2048, 2560), ("wgrad", 4096, 2048, 2560)]


@pytest.mark.parametrize("op,T,N,K", TAIL_CASES)
def test_split_tail_plan(op, T, N, K):
    p = dp.plan(op, T, N, K)
    tiles = p["tiles_m"] * p["tiles_n"]
    if not (0 < p["full_units"] < tiles):
        pytest.skip(f"plan on this device has no split tail: {p}")
    c = inputs.dense_projection(T, N, K, seed=8)
    d = to_dev(c)
    a, b = operands(op, c)
    got32 = gpu(op, *operands(op, d), out_dtype=torch.float32)
    got16 = gpu(op, *operands(op, d), out_dtype=torch.bfloat16)
    R, C = got32.shape
    rng = np.random.default_rng(1)
    # the tail tiles are the last ones in raster order: check the last tile row in full
    last = np.arange(max(0, R - 128), R)
    rows = np.concatenate([np.repeat(last, C), rng.integers(0, R, 4096)])
    cols = np.concatenate([np.tile(np.arange(C), last.size), rng.integers(0, C, 4096)])
    ref = sampled_ref(op, a, b, rows, cols)
    ri, ci = torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)
    assert_budget(got32[ri, ci].double().cpu().numpy(), ref, "f32", f"{op} split tail f32")
    assert_budget(got16.float()[ri, ci].double().cpu().numpy(), ref, "bf16", f"{op} split tail bf16")
    for _ in range(3):
        again = gpu(op, *operands(op, d), out_dtype=torch.float32)
        assert torch.equal(again.view(torch.int32), got32.view(torch.int32))
    no_device_fault()


@pytest.mark.parametrize("swap", [0, 1])
@pytest.mark.parametrize("T,K,N", [(1025, 4096, 64), (1025, 5120, 48), (4100, 4096, 128), (300, 1024, 200)])
def test_thin_wgrad_both_orientations(monkeypatch, swap, T, K, N):
    # dW = dY^T X (tile rows over N) and dW^T = X^T dY stored transposed (tile rows over K)
    monkeypatch.setenv("DP_FORCE_SWAP", str(swap))
    p = dp.plan("wgrad", T, N, K)
    assert p["swap_ab"] == swap
    c = inputs.thin_wgrad(T, N, K, seed=4)
    ref = full_ref("wgrad", c["dY"], c["X"])
    d = to_dev(c)
    for out_dtype, name in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
        wide = torch.full((N, K + 16), float("nan"), dtype=out_dtype, device=DEV)
        view = wide[:, 8:8 + K]
        dp.dp_gemm_wgrad(d["dY"], d["X"], out=view, out_dtype=out_dtype)
        assert_budget(as_f64(view), ref, name, f"wgrad swap={swap} {K}->{N} T={T} {name}")
        assert torch.isnan(wide[:, :8].float()).all() and torch.isnan(wide[:, 8 + K:].float()).all()
    no_device_fault()


# --------------------------------- CTA-pair tiles (256 rows over a cluster of two CTAs)

PAIR_SHAPES = [("fwd", 257, 256, 192), ("fwd", 600, 384, 512), ("dgrad", 300, 136, 256), ("dgrad", 513, 512, 384),
               ("wgrad", 129, 264, 512), ("wgrad", 1000, 512, 256)]


@pytest.mark.parametrize("op,T,N,K", PAIR_SHAPES)
@pytest.mark.parametrize("bn", [128, 256])
def test_pair_integer_exact(monkeypatch, op, T, N, K, bn):
    monkeypatch.setenv("DP_FORCE_PAIR", "1")
    monkeypatch.setenv("DP_FORCE_BN", str(bn))
    monkeypatch.setenv("DP_FORCE_SWAP", "0")
    p = dp.plan(op, T, N, K)
    if not p["cta_pair"]:
        pytest.skip(f"no pair plan for this shape: {p}")
    c = inputs.integer_case(T, N, K, seed=T + N + K + bn)
    ref = full_ref(op, *operands(op, c))
    got = as_f64(gpu(op, *operands(op, to_dev(c)), out_dtype=torch.float32))
    assert np.array_equal(got, ref), (op, T, N, K, bn, p)
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K", [("router_fwd", 257, 256, 192), ("router_fwd", 600, 136, 520),
                                      ("router_wgrad", 300, 256, 264), ("router_wgrad", 77, 136, 520)])
@pytest.mark.parametrize("bn", [128, 256])
def test_router_pair_integer_exact(monkeypatch, op, T, N, K, bn):
    # BF16x3 over CTA pairs: each CTA splits its own 128 rows of A, B comes in halves
    monkeypatch.setenv("DP_FORCE_PAIR", "1")
    monkeypatch.setenv("DP_FORCE_BN", str(bn))
    p = dp.plan(op, T, N, K)
    if not p["cta_pair"]:
        pytest.skip(f"no pair plan for this shape: {p}")
    c = inputs.integer_case(T, N, K, seed=T + N + K + bn, dtype=torch.float32)
    a, b = operands(op, c)
    ref = full_ref(op, a, b)
    got = as_f64(gpu(op, *operands(op, to_dev(c))))
    assert np.array_equal(got, ref), (op, T, N, K, bn, p)
    no_device_fault()


@pytest.mark.parametrize("op", ["router_fwd", "router_wgrad"])
@pytest.mark.parametrize("T,splits", [(1024, 0), (1024, 4), (4031, 0)])
def test_router_pair_budget(monkeypatch, op, T, splits):
    monkeypatch.setenv("DP_FORCE_PAIR", "1")
    monkeypatch.setenv("DP_FORCE_BN", "256")
    if splits:
        monkeypatch.setenv("DP_FORCE_SPLITS", str(splits))
    p = dp.plan(op, T, 256, 4096)
    assert p["cta_pair"], p
    c = inputs.router(T, 4096, seed=T + splits, experts=256)
    ref = full_ref(op, *operands(op, c))
    got = as_f64(gpu(op, *operands(op, to_dev(c))))
    assert_budget(got, ref, "f32", f"pair {op} T={T} {p['splits']} splits")
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K,tail", [("fwd", 2048, 2560, 2048, 2), ("dgrad", 2048, 2048, 2560, 3),
                                           ("wgrad", 4096, 2048, 2560, 0), ("wgrad", 16173, 512, 1024, 0)])
def test_pair_split_plans(monkeypatch, op, T, N, K, tail):
    # pairs with split tails or split-everything plans: ordered reduction per CTA half
    monkeypatch.setenv("DP_FORCE_PAIR", "1")
    if tail:
        monkeypatch.setenv("DP_FORCE_TAIL_SPLITS", str(tail))
    p = dp.plan(op, T, N, K)
    assert p["cta_pair"] and p["splits"] > 1, p
    c = inputs.dense_projection(T, N, K, seed=9)
    d = to_dev(c)
    got = gpu(op, *operands(op, d), out_dtype=torch.float32)
    R, C = got.shape
    rng = np.random.default_rng(3)
    last = np.arange(max(0, R - 256), R)
    rows = np.concatenate([np.repeat(last, C), rng.integers(0, R, 4096)])
    cols = np.concatenate([np.tile(np.arange(C), last.size), rng.integers(0, C, 4096)])
    ref = sampled_ref(op, *operands(op, c), rows, cols)
    ri, ci = torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)
    assert_budget(got[ri, ci].double().cpu().numpy(), ref, "f32", f"pair {op} {p}")
    again = gpu(op, *operands(op, d), out_dtype=torch.float32)
    assert torch.equal(again.view(torch.int32), got.view(torch.int32))
    no_device_fault()
