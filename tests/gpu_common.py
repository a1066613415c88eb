"""Helpers shared by the GPU parity tests: run an op through the C ABI binding,
compute the FP64 oracle (whole or sampled), and apply the pages' budgets."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import fp32_dense_projection_gb300 as dp
import oracle
from budgets import check

DEV = torch.device("cuda", 0)

# op -> (GPU entry point, full oracle, sampled oracle, FP32-operand flag)
OPS = {
    "fwd": (dp.dp_gemm_fwd, oracle.fwd_bf16, oracle.fwd_bf16_at, False),
    "dgrad": (dp.dp_gemm_dgrad, oracle.dgrad_bf16, oracle.dgrad_bf16_at, False),
    "wgrad": (dp.dp_gemm_wgrad, oracle.wgrad_bf16, oracle.wgrad_bf16_at, False),
    "router_fwd": (dp.router_fwd, oracle.fwd_f32, oracle.fwd_f32_at, True),
    "router_dgrad": (dp.router_dgrad, oracle.dgrad_f32, oracle.dgrad_f32_at, True),
    "router_wgrad": (dp.router_wgrad, oracle.wgrad_f32, oracle.wgrad_f32_at, True),
}


def operands(op: str, c: dict):
    """The (a, b) operand pair of an op from a dict holding X, W, dY."""
    base = op.replace("router_", "")
    if base == "fwd":
        return c["X"], c["W"]
    if base == "dgrad":
        return c["dY"], c["W"]
    return c["dY"], c["X"]


def out_shape(op: str, c: dict):
    T = c["X"].shape[0] if "X" in c else c["dY"].shape[0]
    base = op.replace("router_", "")
    if base == "fwd":
        return T, c["W"].shape[0]
    if base == "dgrad":
        return T, c["W"].shape[1]
    return c["dY"].shape[1], c["X"].shape[1]


def gpu(op: str, a, b, out_dtype=torch.bfloat16, **kw):
    fn = OPS[op][0]
    if op.startswith("router"):
        return fn(a, b, **kw)
    return fn(a, b, out_dtype=out_dtype, **kw)


def full_ref(op: str, a_cpu, b_cpu) -> np.ndarray:
    return OPS[op][1](a_cpu, b_cpu)


def sample_points(shape, rng, n_random=2048, full_rows=2, full_cols=2):
    R, C = shape
    rows = [rng.integers(0, R, n_random)]
    cols = [rng.integers(0, C, n_random)]
    for r in rng.integers(0, R, full_rows):
        rows.append(np.full(C, r))
        cols.append(np.arange(C))
    for cc in rng.integers(0, C, full_cols):
        rows.append(np.arange(R))
        cols.append(np.full(R, cc))
    # the last row and column always: the ragged tail of the tiling
    rows += [np.full(C, R - 1), np.arange(R)]
    cols += [np.arange(C), np.full(R, C - 1)]
    return np.concatenate(rows).astype(np.int64), np.concatenate(cols).astype(np.int64)


def sampled_ref(op: str, a_cpu, b_cpu, rows, cols) -> np.ndarray:
    return OPS[op][2](a_cpu, b_cpu, rows, cols)


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.double().cpu().numpy()


def assert_budget(got, ref, out_dtype: str, what: str = ""):
    ok, msg = check(got, ref, out_dtype)
    assert ok, f"{what}: {msg}"
    return msg


def no_device_fault():
    assert dp.device_error(clear=True) == 0, "a kernel reported a barrier timeout"


def stratified_points(shape, rng, tile=128, per=8):
    """`per` random points in every tile x tile block of an R x C output (the blocks of
    the last row and column clipped to the matrix), block by block."""
    R, C = shape
    tr, tc = -(-R // tile), -(-C // tile)
    bi = np.repeat(np.arange(tr), tc * per)
    bj = np.tile(np.repeat(np.arange(tc), per), tr)
    r0, c0 = bi * tile, bj * tile
    rh, ch = np.minimum(tile, R - r0), np.minimum(tile, C - c0)
    rows = r0 + np.floor(rng.random(bi.size) * rh).astype(np.int64)
    cols = c0 + np.floor(rng.random(bj.size) * ch).astype(np.int64)
    return rows, cols


def block_points(r0, r1, c0, c1):
    """Every element of rows [r0, r1) x columns [c0, c1)."""
    rr, cc = np.meshgrid(np.arange(r0, r1), np.arange(c0, c1), indexing="ij")
    return rr.reshape(-1).astype(np.int64), cc.reshape(-1).astype(np.int64)


def raster_tile(p: dict, tile: int):
    """Output-view coordinates (row tile, column tile) of the plan's tile number `tile`
    in the order the persistent grid takes them: groups of `raster_group` tiles along
    the rows (raster_rows) or the columns, that dimension fastest."""
    tm_n, tn_n, group = p["tiles_m"], p["tiles_n"], p["raster_group"]
    fast_n, slow_n = (tm_n, tn_n) if p["raster_rows"] else (tn_n, tm_n)
    per_group = group * slow_n
    g = tile // per_group
    first = g * group
    width = min(group, fast_n - first)
    local = tile - g * per_group
    fast, slow = first + local % width, local // width
    return (fast, slow) if p["raster_rows"] else (slow, fast)


def plan_tile_points(p: dict, tm: int, tn: int, out_shape):
    """Every output element of the plan's tile (tm, tn), in the output's own indices
    (the swapped weight gradient's view is the transposed output)."""
    r0, c0 = tm * p["block_m"], tn * p["block_n"]
    r1, c1 = min(p["gemm_m"], r0 + p["block_m"]), min(p["gemm_n"], c0 + p["block_n"])
    rows, cols = block_points(r0, r1, c0, c1)
    if p["swap_ab"]:
        rows, cols = cols, rows
    assert rows.max() < out_shape[0] and cols.max() < out_shape[1]
    return rows, cols


def bf16_min_slack(got, ref) -> float:
    """Smallest margin to the BF16 budget over the checked elements:
    min(atol + rtol * |ref| - |got - ref|); negative means a violation."""
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    return float(np.min(1e-2 + 1e-2 * np.abs(r) - np.abs(g - r)))


def record_margin(cell: dict):
    """Print one accuracy cell and, if DP_MARGINS_OUT names a file, append it there as a
    JSON line (the per-seed margin tables are built from these)."""
    line = json.dumps(cell, sort_keys=True)
    print(line)
    path = os.environ.get("DP_MARGINS_OUT")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")
