"""Calls with deterministic = 0: FP32 outputs whose split units add their partials
into the zero-filled output with atomic adds (the pages' non-deterministic package:
zero fill, then FP32 atomics), against the FP64 oracle.  Exact on integer inputs
(integer sums do not depend on the order of the adds), within the FP32 budget on
the pages' distributions, correct over a dirty output buffer and under CUDA-graph
replay; BF16 outputs keep the deterministic plans and bits."""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
import oracle
from fp32_dense_projection_gb300 import inputs
from gpu_common import DEV, as_f64, assert_budget, full_ref, no_device_fault, operands

pytestmark = pytest.mark.gpu

FN = {"fwd": dp.dp_gemm_fwd, "dgrad": dp.dp_gemm_dgrad, "wgrad": dp.dp_gemm_wgrad,
      "router_fwd": dp.router_fwd, "router_dgrad": dp.router_dgrad, "router_wgrad": dp.router_wgrad}


def call(op, a, b, **kw):
    if op.startswith("router"):
        return FN[op](a, b, deterministic=False, **kw)
    return FN[op](a, b, out_dtype=torch.float32, deterministic=False, **kw)


# (op, T, N, K, forced splits, forced orientation / pair)
CASES = [("fwd", 64, 1024, 4096, None, {}), ("dgrad", 200, 512, 2048, 3, {}), ("wgrad", 3000, 64, 1024, 4, {"DP_FORCE_SWAP": "1"}),
         ("wgrad", 3000, 136, 1024, 3, {"DP_FORCE_SWAP": "0"}), ("fwd", 1000, 512, 2048, 2, {"DP_FORCE_PAIR": "1"}),
         ("router_fwd", 64, 256, 4096, None, {}), ("router_wgrad", 1024, 256, 1024, 2, {}),
         ("router_dgrad", 300, 256, 1024, 2, {"DP_FORCE_FFMA": "0"})]


def setup(monkeypatch, splits, extra):
    monkeypatch.setenv("DP_FORCE_ATOMIC", "1")
    if splits:
        monkeypatch.setenv("DP_FORCE_SPLITS", str(splits))
    for k, v in extra.items():
        monkeypatch.setenv(k, v)


@pytest.mark.parametrize("op,T,N,K,splits,extra", CASES)
def test_atomic_integer_exact(monkeypatch, op, T, N, K, splits, extra):
    setup(monkeypatch, splits, extra)
    p = dp.plan(op, T, N, K, out_f32=True, deterministic=False)
    assert p["atomic"] == 1 and p["splits"] > 1, p
    # no partial workspace (the router's keeps its split operands)
    assert op.startswith("router") or p["workspace_bytes"] == 0
    c = inputs.integer_case(T, N, K, seed=T + N, dtype=torch.float32 if op.startswith("router") else torch.bfloat16)
    a, b = operands(op, c)
    ref = full_ref(op, a, b)
    shape = ref.shape
    out = torch.full(shape, 123.0, device=DEV)  # dirty: the call zero-fills it
    got = call(op, a.to(DEV), b.to(DEV), out=out)
    assert np.array_equal(as_f64(got), ref), op
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K,splits,extra", CASES)
def test_atomic_budget(monkeypatch, op, T, N, K, splits, extra):
    setup(monkeypatch, splits, extra)
    c = (inputs.router(T, K, seed=5, experts=N) if op.startswith("router")
         else inputs.dense_projection(T, N, K, seed=5))
    a, b = operands(op, c)
    got = call(op, a.to(DEV), b.to(DEV))
    assert_budget(as_f64(got), full_ref(op, a, b), "f32", f"{op} atomic")
    no_device_fault()


def test_atomic_graph_replay(monkeypatch):
    setup(monkeypatch, 4, {})
    T, N, K = 2000, 64, 1024
    c = inputs.integer_case(T, N, K, seed=2)
    dY, X = c["dY"].to(DEV), c["X"].to(DEV)
    assert dp.plan("wgrad", T, N, K, out_f32=True, deterministic=False)["atomic"] == 1
    out = torch.empty(N, K, device=DEV)
    call("wgrad", dY, X, out=out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call("wgrad", dY, X, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call("wgrad", dY, X, out=out)
    ref = oracle.wgrad_bf16(c["dY"], c["X"])
    for _ in range(3):
        out.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(as_f64(out), ref)
    no_device_fault()


def test_bf16_output_stays_deterministic():
    T, N, K = 64, 1024, 4096
    assert dp.plan("fwd", T, N, K, deterministic=False)["atomic"] == 0
    c = {k: v.to(DEV) for k, v in inputs.dense_projection(T, N, K, seed=1).items()}
    a = dp.dp_gemm_fwd(c["X"], c["W"], deterministic=False)
    b = dp.dp_gemm_fwd(c["X"], c["W"], deterministic=True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    no_device_fault()
