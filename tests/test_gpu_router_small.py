"""The FP32 router's small-T SIMT program (FP32 FMAs on the CUDA cores, one launch,
each output tile's contraction split over a thread-block cluster and summed in rank
order) against the FP64 oracle: forward, input gradient and weight gradient, every
tile width and cluster size, ragged token counts, exact on integer inputs,
bitwise repeatable and the same under CUDA-graph replay.

The pages record that at T = 64 and 256 plain FP32 GEMMs beat the deterministic
BF16x3 router (FlashInfer page "cache the router entry points' calls ...", SOTA
rows); the SIMT program is this library's FP32 path for that regime."""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
import oracle
from fp32_dense_projection_gb300 import inputs
from gpu_common import DEV, as_f64, assert_budget, no_device_fault
from budgets import f32_errors

pytestmark = pytest.mark.gpu

FN = {"router_fwd": dp.router_fwd, "router_dgrad": dp.router_dgrad, "router_wgrad": dp.router_wgrad}
REF = {"router_fwd": oracle.fwd_f32, "router_dgrad": oracle.dgrad_f32, "router_wgrad": oracle.wgrad_f32}


def operands(op, c):
    return {"router_fwd": (c["X"], c["W"]), "router_dgrad": (c["dY"], c["W"]),
            "router_wgrad": (c["dY"], c["X"])}[op]


def force(monkeypatch, bn=None, splits=None):
    monkeypatch.setenv("DP_FORCE_FFMA", "1")
    if bn:
        monkeypatch.setenv("DP_FORCE_BN", str(bn))
    if splits:
        monkeypatch.setenv("DP_FORCE_SPLITS", str(splits))


@pytest.mark.parametrize("op", list(FN))
@pytest.mark.parametrize("T,N,K", [(64, 256, 4096), (1, 256, 4096), (37, 256, 5120), (200, 136, 1032)])
def test_simt_router_budget(monkeypatch, op, T, N, K):
    # FP32 sums: far inside the FP32 budget, and inside the pages' 2e-6 library bar
    force(monkeypatch)
    p = dp.plan(op, T, N, K)
    assert p["program"] == 1 and p["workspace_bytes"] == 0
    c = inputs.router(T, K, seed=T + K, experts=N)
    a, b = operands(op, c)
    got = FN[op](a.to(DEV), b.to(DEV))
    ref = REF[op](a, b)
    assert_budget(as_f64(got), ref, "f32", f"{op} T={T} simt")
    rel, _, _ = f32_errors(as_f64(got), ref)
    assert rel <= 2e-6, rel
    no_device_fault()


# (each shape's contraction has at least 8 stage chunks, so every cluster size applies)
INT_SHAPES = {"router_fwd": (77, 200, 2056), "router_dgrad": (77, 1032, 520), "router_wgrad": (1000, 200, 520)}


@pytest.mark.parametrize("op", list(FN))
@pytest.mark.parametrize("bn", [32, 64])
@pytest.mark.parametrize("splits", [1, 2, 3, 8])
def test_simt_router_integer_exact(monkeypatch, op, bn, splits):
    # small-integer operands: every sum is exact in FP32, whatever the tile width,
    # cluster size and group split; the ragged T and N edges are exact too
    T, N, K = INT_SHAPES[op]
    force(monkeypatch, bn, splits)
    p = dp.plan(op, T, N, K)
    assert (p["program"], p["block_n"], p["splits"]) == (1, bn, splits)
    c = inputs.integer_case(T, N, K, seed=bn + splits, dtype=torch.float32)
    a, b = operands(op, c)
    got = FN[op](a.to(DEV), b.to(DEV))
    assert np.array_equal(as_f64(got), REF[op](a, b)), (op, bn, splits)
    no_device_fault()


def test_simt_router_repeats_and_replays(monkeypatch):
    T, N, K = 64, 256, 4096
    force(monkeypatch, 32, 8)
    c = {k: v.to(DEV) for k, v in inputs.router(T, K, seed=3).items()}
    outs = {op: torch.empty(*((T, N) if op == "router_fwd" else (T, K) if op == "router_dgrad" else (N, K)),
                            device=DEV) for op in FN}
    for op in FN:
        FN[op](*operands(op, c), out=outs[op])
    torch.cuda.synchronize()
    ref = {op: o.clone() for op, o in outs.items()}
    for _ in range(4):
        for op in FN:
            FN[op](*operands(op, c), out=outs[op])
            assert torch.equal(outs[op].view(torch.int32), ref[op].view(torch.int32)), op
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for op in FN:
            FN[op](*operands(op, c), out=outs[op])
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for op in FN:
            FN[op](*operands(op, c), out=outs[op])
    for o in outs.values():
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    for op in FN:
        assert torch.equal(outs[op].view(torch.int32), ref[op].view(torch.int32)), op
    no_device_fault()


def test_simt_router_padded_output(monkeypatch):
    T, N, K = 50, 256, 1024
    force(monkeypatch, 64, 2)
    c = inputs.integer_case(T, N, K, seed=4, dtype=torch.float32)
    buf = torch.full((T, K + 12), 5.0, device=DEV)
    dp.router_dgrad(c["dY"].to(DEV), c["W"].to(DEV), out=buf[:, :K])
    assert np.array_equal(as_f64(buf[:, :K]), oracle.dgrad_f32(c["dY"], c["W"]))
    assert bool((buf[:, K:] == 5).all())
    no_device_fault()


def test_both_router_programs_agree_within_budget():
    # at T = 64 the planner's choice and the other program meet the same budget
    T, N, K = 64, 256, 4096
    c = inputs.router(T, K, seed=8)
    for op in FN:
        a, b = operands(op, c)
        ref = REF[op](a, b)
        got = FN[op](a.to(DEV), b.to(DEV))
        assert_budget(as_f64(got), ref, "f32", f"{op} planner's program")
    no_device_fault()
