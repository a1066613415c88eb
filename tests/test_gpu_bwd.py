"""The backward pass of one layer, dp_gemm_bwd (input gradient dX = dY W and weight
gradient dW = dY^T X from the same dY), against the FP64 oracle in both of its
forms: two single-op calls, and one co-scheduled launch over both problems'
whole-K tiles (every tile shape, either problem's tiles first).  The co-scheduled
launch gives the same bits as whole-K single-op calls of the same tile shape,
repeats bitwise, and replays bitwise from a CUDA graph.

The pages' benchmark rows include the op bwd = dgrad + wgrad (FlashInfer page
"cache the router entry points' calls ...", benchmark description)."""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
import oracle
from fp32_dense_projection_gb300 import inputs
from gpu_common import DEV, as_f64, assert_budget, no_device_fault

pytestmark = pytest.mark.gpu

TILINGS = [(0, 128), (0, 256), (1, 128), (1, 256)]


def on_device(c):
    return {k: v.to(DEV) for k, v in c.items()}


def force(monkeypatch, fuse, pair=None, bn=None):
    monkeypatch.setenv("DP_FORCE_FUSE", str(fuse))
    if pair is not None:
        monkeypatch.setenv("DP_FORCE_PAIR", str(pair))
    if bn is not None:
        monkeypatch.setenv("DP_FORCE_BN", str(bn))


@pytest.mark.parametrize("pair,bn", TILINGS)
@pytest.mark.parametrize("fuse", [2, 3])
@pytest.mark.parametrize("T,N,K", [(1000, 384, 640), (333, 136, 520), (1, 136, 264), (65, 272, 200)])
def test_co_scheduled_integer_exact(monkeypatch, pair, bn, fuse, T, N, K):
    # small-integer operands: every product and partial sum is exact in FP32, so both
    # gradients equal the oracle exactly, whatever the tile shape and tile order
    force(monkeypatch, fuse, pair, bn)
    try:
        b = dp.plan_bwd(T, N, K, True, True)
    except dp.DPError:  # (a pair needs two row tiles of work in both problems)
        b = {"fused": 0}
    if not b["fused"]:
        assert pair == 1
        pytest.skip("no co-scheduled plan of this tile shape for the shape")
    assert b["wgrad_first"] == (fuse == 2)
    assert (b["dgrad"]["cta_pair"], b["dgrad"]["block_n"]) == (pair, bn)
    c = inputs.integer_case(T, N, K, seed=T + bn + fuse)
    d = on_device(c)
    dX, dW = dp.dp_gemm_bwd(d["dY"], d["X"], d["W"], dx_dtype=torch.float32, dw_dtype=torch.float32)
    assert np.array_equal(as_f64(dX), oracle.dgrad_bf16(c["dY"], c["W"]))
    assert np.array_equal(as_f64(dW), oracle.wgrad_bf16(c["dY"], c["X"]))
    no_device_fault()


@pytest.mark.parametrize("dx32,dw32", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("T,N,K", [(1024, 512, 2048), (1000, 384, 640), (4031, 512, 1024)])
def test_bwd_budget(dx32, dw32, T, N, K):
    # the planner's own choice of form, against the pages' budgets
    c = inputs.dense_projection(T, N, K, seed=T + N)
    d = on_device(c)
    dX, dW = dp.dp_gemm_bwd(d["dY"], d["X"], d["W"], dx_dtype=torch.float32 if dx32 else torch.bfloat16,
                            dw_dtype=torch.float32 if dw32 else torch.bfloat16)
    what = f"bwd T={T} {K}->{N} fused={dp.plan_bwd(T, N, K, dx32, dw32)['fused']}"
    assert_budget(as_f64(dX), oracle.dgrad_bf16(c["dY"], c["W"]), "f32" if dx32 else "bf16", what + " dX")
    assert_budget(as_f64(dW), oracle.wgrad_bf16(c["dY"], c["X"]), "f32" if dw32 else "bf16", what + " dW")
    no_device_fault()


@pytest.mark.parametrize("pair,bn", TILINGS)
def test_co_scheduled_matches_whole_k_single_calls(monkeypatch, pair, bn):
    # the co-scheduled launch computes each tile exactly as a whole-K single-op plan of
    # the same tile shape and weight-gradient orientation: the same bits
    T, N, K = 1000, 384, 640
    d = on_device(inputs.dense_projection(T, N, K, seed=5))
    force(monkeypatch, 1, pair, bn)
    b = dp.plan_bwd(T, N, K)
    assert b["fused"]
    dX, dW = dp.dp_gemm_bwd(d["dY"], d["X"], d["W"])
    monkeypatch.setenv("DP_FORCE_SPLITS", "1")
    monkeypatch.setenv("DP_FORCE_SWAP", str(b["wgrad"]["swap_ab"]))
    assert dp.plan("dgrad", T, N, K) == b["dgrad"] and dp.plan("wgrad", T, N, K) == b["wgrad"]
    dX1 = dp.dp_gemm_dgrad(d["dY"], d["W"])
    dW1 = dp.dp_gemm_wgrad(d["dY"], d["X"])
    assert torch.equal(dX.view(torch.int16), dX1.view(torch.int16))
    assert torch.equal(dW.view(torch.int16), dW1.view(torch.int16))
    no_device_fault()


def test_two_call_form_matches_single_op_calls(monkeypatch):
    # the two-call form is the single-op calls, split plans included
    T, N, K = 16173, 128, 4096
    force(monkeypatch, 0)
    assert not dp.plan_bwd(T, N, K)["fused"]
    d = on_device(inputs.dense_projection(T, N, K, seed=6))
    dX, dW = dp.dp_gemm_bwd(d["dY"], d["X"], d["W"], dw_dtype=torch.float32)
    assert torch.equal(dX.view(torch.int16), dp.dp_gemm_dgrad(d["dY"], d["W"]).view(torch.int16))
    assert torch.equal(dW.view(torch.int32),
                       dp.dp_gemm_wgrad(d["dY"], d["X"], out_dtype=torch.float32).view(torch.int32))
    no_device_fault()


def test_co_scheduled_repeats_and_replays(monkeypatch):
    T, N, K = 1024, 1024, 2048
    force(monkeypatch, 1)
    d = on_device(inputs.dense_projection(T, N, K, seed=9))
    dX = torch.empty(T, K, dtype=torch.bfloat16, device=DEV)
    dW = torch.empty(N, K, dtype=torch.float32, device=DEV)
    dp.dp_gemm_bwd(d["dY"], d["X"], d["W"], dX=dX, dW=dW)
    torch.cuda.synchronize()
    ref = (dX.clone(), dW.clone())
    for _ in range(5):
        dp.dp_gemm_bwd(d["dY"], d["X"], d["W"], dX=dX, dW=dW)
        assert torch.equal(dX.view(torch.int16), ref[0].view(torch.int16))
        assert torch.equal(dW.view(torch.int32), ref[1].view(torch.int32))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dp.dp_gemm_bwd(d["dY"], d["X"], d["W"], dX=dX, dW=dW)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dp.dp_gemm_bwd(d["dY"], d["X"], d["W"], dX=dX, dW=dW)
    dX.zero_()
    dW.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(dX.view(torch.int16), ref[0].view(torch.int16))
    assert torch.equal(dW.view(torch.int32), ref[1].view(torch.int32))
    no_device_fault()


def test_co_scheduled_padded_outputs(monkeypatch):
    # outputs as column slices of wider buffers: only the first K columns are written
    T, N, K = 777, 264, 392
    force(monkeypatch, 1)
    c = inputs.integer_case(T, N, K, seed=11)
    d = on_device(c)
    bx = torch.full((T, K + 24), 7.0, dtype=torch.float32, device=DEV)
    bw = torch.full((N, K + 8), 7.0, dtype=torch.bfloat16, device=DEV)
    dp.dp_gemm_bwd(d["dY"], d["X"], d["W"], dX=bx[:, :K], dW=bw[:, :K])
    assert np.array_equal(as_f64(bx[:, :K]), oracle.dgrad_bf16(c["dY"], c["W"]))
    # (the FP32 sums are exact integers; the bf16 output is their one nearest-even rounding)
    want_w = torch.from_numpy(oracle.wgrad_bf16(c["dY"], c["X"])).float().bfloat16()
    assert torch.equal(bw[:, :K].cpu().view(torch.int16), want_w.view(torch.int16))
    assert bool((bx[:, K:] == 7).all()) and bool((bw[:, K:] == 7).all())
    no_device_fault()


def test_empty_tokens():
    N, K = 64, 128
    dY = torch.empty(0, N, dtype=torch.bfloat16, device=DEV)
    X = torch.empty(0, K, dtype=torch.bfloat16, device=DEV)
    W = torch.ones(N, K, dtype=torch.bfloat16, device=DEV)
    dW = torch.full((N, K), 3.0, dtype=torch.bfloat16, device=DEV)
    dX, dW = dp.dp_gemm_bwd(dY, X, W, dW=dW)
    assert dX.shape == (0, K) and bool((dW == 0).all())
    no_device_fault()
