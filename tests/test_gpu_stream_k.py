"""Stream-K plans (the grid's slots share all tiles' contraction blocks evenly; a
tile cut by slot boundaries is summed from its pieces' FP32 partials in block
order) against the FP64 oracle: exact on integer inputs for every op, tile shape
and weight-gradient orientation, within the pages' budgets on their
distributions, bitwise repeatable and the same under CUDA-graph replay."""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
import oracle
from fp32_dense_projection_gb300 import inputs
from gpu_common import DEV, as_f64, assert_budget, full_ref, gpu, no_device_fault, operands

pytestmark = pytest.mark.gpu

CASES = [("wgrad", 1025, 64, 4096), ("wgrad", 4100, 128, 1024), ("wgrad", 2000, 200, 520),
         ("fwd", 300, 512, 2048), ("dgrad", 300, 2048, 512), ("fwd", 1000, 136, 4096)]


def force(monkeypatch, pair=None, bn=None, swap=None):
    monkeypatch.setenv("DP_FORCE_STREAM_K", "1")
    for k, v in (("DP_FORCE_PAIR", pair), ("DP_FORCE_BN", bn), ("DP_FORCE_SWAP", swap)):
        if v is not None:
            monkeypatch.setenv(k, str(v))


def stream_k_plan(op, T, N, K, f32=False):
    try:
        p = dp.plan(op, T, N, K, out_f32=f32)
    except dp.DPError:
        return None
    return p if p["stream_k"] else None


@pytest.mark.parametrize("op,T,N,K", CASES)
@pytest.mark.parametrize("pair,bn", [(0, 64), (0, 128), (0, 256), (1, 128), (1, 256)])
def test_stream_k_integer_exact(monkeypatch, op, T, N, K, pair, bn):
    force(monkeypatch, pair, bn)
    p = stream_k_plan(op, T, N, K, True)
    if p is None:
        pytest.skip("no stream-K plan of this tile shape for the shape")
    assert p["splits"] >= 2 and p["workspace_bytes"] > 0 and p["grid"] % (2 if pair else 1) == 0
    c = inputs.integer_case(T, N, K, seed=T + bn + pair)
    a, b = operands(op, c)
    got = gpu(op, a.to(DEV), b.to(DEV), out_dtype=torch.float32)
    assert np.array_equal(as_f64(got), full_ref(op, a, b)), (op, T, N, K, pair, bn)
    no_device_fault()


@pytest.mark.parametrize("swap", [0, 1])
@pytest.mark.parametrize("T,N,K", [(1025, 64, 4096), (16173, 48, 1024)])
def test_stream_k_wgrad_orientations(monkeypatch, swap, T, N, K):
    force(monkeypatch, swap=swap)
    p = stream_k_plan("wgrad", T, N, K)
    if p is None:
        pytest.skip("no stream-K plan in this orientation")
    assert p["swap_ab"] == swap
    c = inputs.thin_wgrad(T, N, K, seed=swap + 3)
    ref = oracle.wgrad_bf16(c["dY"], c["X"])
    d = {k: v.to(DEV) for k, v in c.items()}
    got16 = dp.dp_gemm_wgrad(d["dY"], d["X"])
    got32 = dp.dp_gemm_wgrad(d["dY"], d["X"], out_dtype=torch.float32)
    assert_budget(as_f64(got16), ref, "bf16", f"stream-K wgrad T={T} swap={swap}")
    assert_budget(as_f64(got32), ref, "f32", f"stream-K wgrad T={T} swap={swap}")
    no_device_fault()


def test_stream_k_repeats_and_replays(monkeypatch):
    T, N, K = 4100, 128, 1024
    force(monkeypatch)
    assert stream_k_plan("wgrad", T, N, K, True) is not None
    c = {k: v.to(DEV) for k, v in inputs.thin_wgrad(T, N, K, seed=6).items()}
    out = torch.empty(N, K, dtype=torch.float32, device=DEV)
    dp.dp_gemm_wgrad(c["dY"], c["X"], out=out, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = out.clone()
    for _ in range(5):
        dp.dp_gemm_wgrad(c["dY"], c["X"], out=out, out_dtype=torch.float32)
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dp.dp_gemm_wgrad(c["dY"], c["X"], out=out, out_dtype=torch.float32)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dp.dp_gemm_wgrad(c["dY"], c["X"], out=out, out_dtype=torch.float32)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K", [("router_fwd", 1000, 256, 1024), ("router_fwd", 129, 136, 4096),
                                      ("router_wgrad", 4100, 256, 512), ("router_wgrad", 300, 136, 2048)])
@pytest.mark.parametrize("bn", [64, 128, 256])
def test_stream_k_router_integer_exact(monkeypatch, op, T, N, K, bn):
    # BF16x3 pieces: the in-kernel split of the streamed FP32 operand walks the slot's
    # pieces like the MMA issuer and the epilogue; integer operands are bf16-exact
    force(monkeypatch, bn=bn)
    monkeypatch.setenv("DP_FORCE_FFMA", "0")
    p = stream_k_plan(op, T, N, K, True)
    if p is None:
        pytest.skip("no stream-K plan of this tile width for the shape")
    c = inputs.integer_case(T, N, K, seed=T + N + bn, dtype=torch.float32)
    a, b = operands(op, c)
    got = gpu(op, a.to(DEV), b.to(DEV))
    assert np.array_equal(as_f64(got), full_ref(op, a, b)), (op, T, N, K, bn, p)
    no_device_fault()


@pytest.mark.parametrize("op", ["router_fwd", "router_wgrad"])
@pytest.mark.parametrize("T", [1024, 16384])
def test_stream_k_router_budget_and_repeats(monkeypatch, op, T):
    force(monkeypatch)
    monkeypatch.setenv("DP_FORCE_FFMA", "0")
    p = stream_k_plan(op, T, 256, 4096, True)
    assert p is not None and p["program"] == 0
    c = inputs.router(T, 4096, seed=T % 7, experts=256)
    a, b = operands(op, c)
    d = {k: v.to(DEV) for k, v in c.items()}
    got = gpu(op, *operands(op, d))
    if T == 1024:
        assert_budget(as_f64(got), full_ref(op, a, b), "f32", f"stream-K {op} T={T}")
    else:  # sampled: eight elements in every 128 x 128 block, plus the last row and column
        from gpu_common import sampled_ref, stratified_points
        shape = tuple(got.shape)
        rows, cols = stratified_points(shape, np.random.default_rng(T))
        rows = np.concatenate([rows, np.full(shape[1], shape[0] - 1), np.arange(shape[0])])
        cols = np.concatenate([cols, np.arange(shape[1]), np.full(shape[0], shape[1] - 1)])
        ref = sampled_ref(op, a, b, rows, cols)
        g = got[torch.from_numpy(rows).to(DEV), torch.from_numpy(cols).to(DEV)].double().cpu().numpy()
        assert_budget(g, ref, "f32", f"stream-K {op} T={T}")
    for _ in range(3):
        again = gpu(op, *operands(op, d))
        assert torch.equal(again.view(torch.int32), got.view(torch.int32))
    no_device_fault()
