"""Helpers shared by the GPU parity tests: run an op through the C ABI binding,
compute the FP64 oracle (whole or sampled), and apply the pages' budgets."""
from __future__ import annotations

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
