"""Full-size runs of the workloads' own shapes through the C ABI, as the benchmark
launches them (the planner's default plans):

* bitwise determinism: ten eager calls and one CUDA-graph replay, each into an
  output pre-filled with NaN, give the first call's bits exactly -- the wide
  projection 4096 -> 12288 at T = 16384 and the ragged 16231 (whose input and
  weight gradients split their last partial wave), and the thin weight gradients
  4096 -> 64 and 5120 -> 48 at T = 65537 (eight-way token splits), BF16 and FP32
  output;
* tile-stratified parity against the FP64 oracle: eight random elements in every
  128 x 128 block of the output, the last row and column in full, and (seed 0 of
  the wide projection) every element of the last tile in the grid's order, of the
  first split tile and of the bottom-right tile; a NaN left anywhere fails;
* ten seeds per configuration, each seed's margin to the budget recorded
  (``record_margin``; DP_MARGINS_OUT collects them as JSON lines).

Budgets (FlashInfer page "perf(cake_dense_projection_gemm): restore the K1
weight-gradient routes ...", PR body): BF16 output atol = rtol = 1e-2 with zero
violations; FP32 output rel_fro <= 5e-5 and max_abs <= 1e-3 * max|ref|.  That page's
accuracy sweep records that its deterministic program misses the BF16 budget for
some seeds at T around 47k-65k; the margins recorded here show how far each cell stays from it.
"""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
from budgets import f32_errors
from fp32_dense_projection_gb300 import inputs
from gpu_common import (DEV, assert_budget, bf16_min_slack, gpu, no_device_fault, operands, plan_tile_points,
                        raster_tile, record_margin, sampled_ref, stratified_points)

pytestmark = pytest.mark.gpu

WIDE_N, WIDE_K = 12288, 4096
WIDE_T = (16384, 16231)
THIN = [(4096, 64), (4096, 128), (4096, 512), (5120, 48), (5120, 64)]
THIN_BITWISE = ((4096, 64), (5120, 48))
NAN = float("nan")


def to_dev(c):
    return {k: v.to(DEV) for k, v in c.items()}


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def determinism(call, shape, dtype):
    """call(out) writes the op into `out`.  Ten eager calls and one CUDA-graph replay,
    each into a NaN-filled output, must write every element and give the same bits.
    Returns the first call's output."""
    out = torch.full(shape, NAN, dtype=dtype, device=DEV)
    call(out)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all(), "an output element was left unwritten (NaN)"
    first = out.clone()
    for i in range(9):
        out.fill_(NAN)
        call(out)
        assert torch.equal(bits(out), bits(first)), f"eager call {i + 2} differs from the first"
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(out)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(out)
    out.fill_(NAN)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bits(out), bits(first)), "CUDA-graph replay differs from the eager call"
    del g
    return first


def edge_points(shape):
    R, C = shape
    return [(np.full(C, R - 1), np.arange(C)), (np.arange(R), np.full(R, C - 1))]


def gather(out: torch.Tensor, rows, cols) -> np.ndarray:
    ri, ci = torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)
    return out.float()[ri, ci].double().cpu().numpy()


def cat(points):
    return (np.concatenate([p[0] for p in points]).astype(np.int64),
            np.concatenate([p[1] for p in points]).astype(np.int64))


# ------------------------------------------------- wide projection 4096 -> 12288

def wide_shape(op, T):
    return {"fwd": (T, WIDE_N), "dgrad": (T, WIDE_K), "wgrad": (WIDE_N, WIDE_K)}[op]


@pytest.fixture(scope="module", params=WIDE_T)
def wide_seed0(request):
    T = request.param
    c = inputs.dense_projection(T, WIDE_N, WIDE_K, seed=0, w_scale=1.0 / 64)
    return T, c, to_dev(c)


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_wide_projection_bitwise_and_every_tile(wide_seed0, op):
    T, c, d = wide_seed0
    a, b = operands(op, d)
    p = dp.plan(op, T, WIDE_N, WIDE_K)
    ws = torch.empty(max(1, p["workspace_bytes"]), dtype=torch.uint8, device=DEV)
    shape = wide_shape(op, T)
    out = determinism(lambda o: gpu(op, a, b, out=o, out_dtype=torch.bfloat16, workspace=ws), shape,
                      torch.bfloat16)
    rng = np.random.default_rng(1000 + T + len(op))
    pts = [stratified_points(shape, rng)] + edge_points(shape)
    tiles = {raster_tile(p, p["tiles"] - 1), (p["tiles_m"] - 1, p["tiles_n"] - 1)}
    if p["full_units"] < p["tiles"]:  # the plan splits its last partial wave: its first split tile
        tiles.add(raster_tile(p, p["full_units"]))
    pts += [plan_tile_points(p, tm, tn, shape) for tm, tn in sorted(tiles)]
    rows, cols = cat(pts)
    ref = sampled_ref(op, *operands(op, c), rows, cols)
    got = gather(out, rows, cols)
    record_margin({"cell": "wide", "op": op, "T": T, "seed": 0, "out": "bf16", "points": int(rows.size),
                   "min_slack": bf16_min_slack(got, ref), "split_tiles": p["tiles"] - p["full_units"],
                   "splits": p["splits"]})
    assert_budget(got, ref, "bf16", f"{op} T={T} seed 0")
    no_device_fault()


@pytest.mark.parametrize("T", WIDE_T)
@pytest.mark.parametrize("seed", range(1, 10))
def test_wide_projection_seeds(T, seed):
    c = inputs.dense_projection(T, WIDE_N, WIDE_K, seed=seed, w_scale=1.0 / 64)
    d = to_dev(c)
    for op in ("fwd", "dgrad", "wgrad"):
        shape = wide_shape(op, T)
        out = torch.full(shape, NAN, dtype=torch.bfloat16, device=DEV)
        gpu(op, *operands(op, d), out=out, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), f"{op}: an output element was left unwritten"
        rows, cols = cat([stratified_points(shape, np.random.default_rng(seed * 7 + len(op)))] + edge_points(shape))
        ref = sampled_ref(op, *operands(op, c), rows, cols)
        got = gather(out, rows, cols)
        record_margin({"cell": "wide", "op": op, "T": T, "seed": seed, "out": "bf16", "points": int(rows.size),
                       "min_slack": bf16_min_slack(got, ref)})
        assert_budget(got, ref, "bf16", f"{op} T={T} seed {seed}")
        del out
    no_device_fault()


# --------------------------------------- thin-N weight gradient at T = 65537 tokens

@pytest.mark.parametrize("seed", range(10))
def test_thin_wgrad_t65537_seeds(seed):
    """Five (K, N) shapes, BF16 and FP32 output.  Checked elements: eight per 128 x 128
    block, 1024 random ones, the last row and column, and -- where the BF16 budget is
    tightest, at the smallest |dW| -- the output's smallest elements by magnitude."""
    T = 65537
    X_K, X, X_cpu = None, None, None
    for K, N in THIN:
        if X_K != K:  # X depends on (T, K, seed) only: drawn once for the shapes sharing K
            X_K, X, X_cpu = K, None, None
            X_cpu = inputs.normal((T, K), seed, inputs.ROLE_X)  # the thin_wgrad recipe's X
            X = X_cpu.to(DEV)
        dY_cpu = inputs.normal((T, N), seed, inputs.ROLE_DY)
        dY = dY_cpu.to(DEV)
        p = dp.plan("wgrad", T, N, K)
        ws = torch.empty(max(1, p["workspace_bytes"]), dtype=torch.uint8, device=DEV)
        outs = {}
        for dtype in (torch.bfloat16, torch.float32):
            def call(o, dtype=dtype):
                dp.dp_gemm_wgrad(dY, X, out=o, out_dtype=dtype, workspace=ws)
            if seed == 0 and (K, N) in THIN_BITWISE:
                outs[dtype] = determinism(call, (N, K), dtype)
            else:
                o = torch.full((N, K), NAN, dtype=dtype, device=DEV)
                call(o)
                torch.cuda.synchronize()
                assert torch.isfinite(o).all(), f"{K}->{N} {dtype}: an output element was left unwritten"
                outs[dtype] = o
        rng = np.random.default_rng(seed * 31 + K + N)
        unbiased = cat([stratified_points((N, K), rng), (rng.integers(0, N, 1024), rng.integers(0, K, 1024))]
                       + edge_points((N, K)))
        nsmall = min(4096, N * K // 64)
        small = torch.topk(outs[torch.bfloat16].float().abs().reshape(-1), nsmall, largest=False).indices.cpu().numpy()
        rows, cols = cat([unbiased, (small // K, small % K)])
        n_unb = unbiased[0].size
        ref = sampled_ref("wgrad", dY_cpu, X_cpu, rows, cols)
        g16 = gather(outs[torch.bfloat16], rows, cols)
        g32 = gather(outs[torch.float32], rows, cols)
        rel, mx, _ = f32_errors(g32[:n_unb], ref[:n_unb])
        mx_all = float(np.abs(g32 - ref).max())
        max_ref = float(np.abs(ref[:n_unb]).max())
        record_margin({"cell": "thin", "K": K, "N": N, "T": T, "seed": seed, "splits": p["splits"],
                       "points": int(rows.size), "bf16_min_slack": bf16_min_slack(g16, ref),
                       "f32_rel_fro": rel, "f32_max_abs_over_budget": mx_all / (1e-3 * max_ref)})
        assert_budget(g16, ref, "bf16", f"wgrad {K}->{N} T={T} seed {seed} bf16")
        assert rel <= 5e-5 and mx_all <= 1e-3 * max_ref, (K, N, seed, rel, mx_all, max_ref)
        del outs, dY, ws
    del X, X_cpu
    no_device_fault()
