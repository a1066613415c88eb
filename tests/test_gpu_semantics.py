"""GPU behaviour beyond the numbers: bitwise determinism (repeats, CUDA graph
replay versus eager launch), padded output rows with NaN canaries, operand views
with padded strides, fresh tensors of the same shape, empty token sets, and the
status codes of bad calls.

The canary and fresh-tensor cases follow the test practice the FlashInfer pages
describe for the deterministic package ("plan the 4096 -> 12288 input gradient
...": write into a column slice of a wider NaN-filled buffer and check that the
padding stays NaN; "cache the router entry points' calls ...": repeat a call with
new tensors of the same shape and compare with a fresh reference).
"""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
from fp32_dense_projection_gb300 import inputs
from gpu_common import DEV, as_f64, assert_budget, full_ref, gpu, no_device_fault, operands

pytestmark = pytest.mark.gpu

CASES = [  # (op, T, N, K): whole-K tiles, split reductions, router
    ("fwd", 300, 512, 1024),
    ("dgrad", 300, 512, 1024),
    ("wgrad", 300, 512, 1024),
    ("wgrad", 16173, 64, 4096),   # split over tokens
    ("fwd", 64, 1024, 4096),      # split over K
    ("router_fwd", 256, 256, 4096),
    ("router_dgrad", 256, 256, 4096),
    ("router_wgrad", 1024, 256, 4096),
]


def case_tensors(op, T, N, K, seed=0):
    if op.startswith("router"):
        return inputs.router(T, K, seed=seed, experts=N)
    return inputs.dense_projection(T, N, K, seed=seed)


@pytest.mark.parametrize("op,T,N,K", CASES)
def test_bitwise_repeatable(op, T, N, K):
    c = {k: v.to(DEV) for k, v in case_tensors(op, T, N, K).items()}
    a, b = operands(op, c)
    first = gpu(op, a, b, out_dtype=torch.float32)
    for _ in range(9):
        again = gpu(op, a, b, out_dtype=torch.float32)
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K", CASES)
def test_graph_replay_matches_eager(op, T, N, K):
    c = {k: v.to(DEV) for k, v in case_tensors(op, T, N, K).items()}
    a, b = operands(op, c)
    kw = {} if op.startswith("router") else {"out_dtype": torch.bfloat16}
    eager = gpu(op, a, b, **kw)
    ws = torch.zeros(max(1, dp.workspace_size(op, T, N, K,
                                              out_f32=op.startswith("router"))), dtype=torch.uint8, device=DEV)
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gpu(op, a, b, out=out, workspace=ws, **kw)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gpu(op, a, b, out=out, workspace=ws, **kw)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        bits = torch.int16 if out.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(out.view(bits), eager.view(bits))
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K", CASES)
def test_workspace_needs_no_initial_value(op, T, N, K):
    # the workspace is scratch: a workspace full of NaN bit patterns gives the same
    # bits as a zeroed one
    c = {k: v.to(DEV) for k, v in case_tensors(op, T, N, K).items()}
    a, b = operands(op, c)
    need = max(1, dp.workspace_size(op, T, N, K, out_f32=True))
    clean = torch.zeros(need, dtype=torch.uint8, device=DEV)
    dirty = torch.full((need,), 0xFF, dtype=torch.uint8, device=DEV)
    kw = {} if op.startswith("router") else {"out_dtype": torch.float32}
    want = gpu(op, a, b, workspace=clean, **kw)
    got = gpu(op, a, b, workspace=dirty, **kw)
    assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K", [("fwd", 200, 256, 512), ("dgrad", 200, 256, 512), ("wgrad", 200, 256, 512),
                                      ("wgrad", 4100, 64, 1024), ("router_fwd", 100, 256, 512),
                                      ("router_dgrad", 100, 256, 512), ("router_wgrad", 100, 256, 512)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_padded_output_keeps_nan_canary(op, T, N, K, out_dtype):
    if op.startswith("router"):
        if out_dtype == torch.bfloat16:
            pytest.skip("router output is FP32")
    c = case_tensors(op, T, N, K, seed=3)
    a, b = operands(op, c)
    ref = full_ref(op, a, b)
    R, C = ref.shape
    pad = 24
    wide = torch.full((R, C + pad), float("nan"), dtype=out_dtype, device=DEV)
    view = wide[:, 8:8 + C]  # 8 elements in: keeps 16-byte alignment for both dtypes
    d = {k: v.to(DEV) for k, v in c.items()}
    kw = {} if op.startswith("router") else {"out_dtype": out_dtype}
    gpu(op, *operands(op, d), out=view, **kw)
    torch.cuda.synchronize()
    got = as_f64(view)
    assert_budget(got, ref, "bf16" if out_dtype == torch.bfloat16 else "f32", op)
    assert torch.isnan(wide[:, :8].float()).all() and torch.isnan(wide[:, 8 + C:].float()).all()


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
def test_padded_operand_strides(op):
    T, N, K = 150, 128, 320
    c = inputs.dense_projection(T, N, K, seed=4)
    ref = full_ref(op, *operands(op, c))
    # every operand becomes a column slice of a wider buffer
    d = {}
    for k, v in c.items():
        big = torch.zeros(v.shape[0], v.shape[1] + 40, dtype=v.dtype, device=DEV)
        big[:, 16:16 + v.shape[1]] = v.to(DEV)
        d[k] = big[:, 16:16 + v.shape[1]]
    got = as_f64(gpu(op, *operands(op, d), out_dtype=torch.float32))
    assert_budget(got, ref, "f32", op)


def test_fresh_tensors_same_shape():
    T, N, K = 257, 256, 512
    for seed in range(3):
        c = inputs.dense_projection(T, N, K, seed=10 + seed)
        d = {k: v.to(DEV) for k, v in c.items()}
        for op in ("fwd", "dgrad", "wgrad"):
            ref = full_ref(op, *operands(op, c))
            assert_budget(as_f64(gpu(op, *operands(op, d), out_dtype=torch.float32)), ref, "f32", op)


def test_empty_token_set():
    N, K = 64, 128
    X = torch.zeros(0, K, dtype=torch.bfloat16, device=DEV)
    dY = torch.zeros(0, N, dtype=torch.bfloat16, device=DEV)
    W = torch.randn(N, K, device=DEV).to(torch.bfloat16)
    assert dp.dp_gemm_fwd(X, W).shape == (0, N)
    assert dp.dp_gemm_dgrad(dY, W).shape == (0, K)
    dW = torch.full((N, K), float("nan"), device=DEV)
    dp.dp_gemm_wgrad(dY, X, out=dW, out_dtype=torch.float32)
    assert torch.equal(dW, torch.zeros_like(dW))
    Xr = torch.zeros(0, K, device=DEV)
    dYr = torch.zeros(0, N, device=DEV)
    dWr = torch.full((N, K), float("nan"), device=DEV)
    dp.router_wgrad(dYr, Xr, out=dWr)
    assert torch.equal(dWr, torch.zeros_like(dWr))


def test_status_codes():
    X = torch.randn(64, 128, device=DEV).to(torch.bfloat16)
    W = torch.randn(64, 128, device=DEV).to(torch.bfloat16)
    # misaligned: a view starting one element in
    flat = torch.zeros(64 * 128 + 8, dtype=torch.bfloat16, device=DEV)
    Xm = flat[1:1 + 64 * 128].view(64, 128)
    with pytest.raises(dp.DPError) as e:
        dp.dp_gemm_fwd(Xm, W)
    assert e.value.status == 2
    # K not a multiple of 8
    with pytest.raises(dp.DPError) as e:
        dp.dp_gemm_fwd(X[:, :100], W[:, :100])
    assert e.value.status in (2, 3)
    # workspace too small for a split plan
    need = dp.workspace_size("fwd", 64, 1024, 4096)
    assert need > 0
    Xs = torch.randn(64, 4096, device=DEV).to(torch.bfloat16)
    Ws = torch.randn(1024, 4096, device=DEV).to(torch.bfloat16)
    small = torch.zeros(need // 2, dtype=torch.uint8, device=DEV)
    with pytest.raises(dp.DPError) as e:
        dp.dp_gemm_fwd(Xs, Ws, workspace=small)
    assert e.value.status == 4
    no_device_fault()


def test_one_workspace_serves_every_op_in_turn():
    # Router calls write bf16 operand copies into the workspace and split calls write
    # FP32 partials.  A sequence mixing them on one workspace must give the same bits
    # as each call on a fresh one: nothing a call reads is left over from another.
    seq = [("router_dgrad", 1024, 256, 4096), ("router_wgrad", 1024, 256, 4096), ("fwd", 64, 1024, 4096),
           ("router_fwd", 256, 256, 4096), ("wgrad", 16173, 64, 4096), ("router_wgrad", 1024, 256, 4096),
           ("fwd", 64, 1024, 4096)]
    need = max(dp.workspace_size(op, T, N, K, out_f32=True) for op, T, N, K in seq)
    shared = torch.zeros(need, dtype=torch.uint8, device=DEV)
    for i, (op, T, N, K) in enumerate(seq):
        c = {k: v.to(DEV) for k, v in case_tensors(op, T, N, K, seed=i).items()}
        a, b = operands(op, c)
        kw = {} if op.startswith("router") else {"out_dtype": torch.float32}
        got = gpu(op, a, b, workspace=shared, **kw)
        fresh = torch.zeros(max(1, need), dtype=torch.uint8, device=DEV)
        want = gpu(op, a, b, workspace=fresh, **kw)
        assert torch.equal(got.view(torch.int32), want.view(torch.int32)), (i, op)
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K", [("wgrad", 16173, 64, 4096), ("wgrad", 16173, 48, 5120), ("fwd", 64, 1024, 4096),
                                      ("router_fwd", 1024, 256, 4096), ("wgrad", 4100, 64, 1024)])
def test_cluster_sum_matches_reduction_kernel(monkeypatch, op, T, N, K):
    # plans with one split unit per CTA sum their partials inside the GEMM's clusters;
    # the reduction kernel adds the same partials in the same order: same bits
    c = {k: v.to(DEV) for k, v in case_tensors(op, T, N, K).items()}
    a, b = operands(op, c)
    kw = {} if op.startswith("router") else {"out_dtype": torch.bfloat16}
    p = dp.plan(op, T, N, K, out_f32=op.startswith("router"))
    if not (p["splits"] > 1 and p["full_units"] == 0 and not p["cta_pair"]):
        pytest.skip(f"not a split-everything single-CTA plan: {p}")
    in_cluster = gpu(op, a, b, **kw)
    monkeypatch.setenv("DP_FORCE_CLUSTER_SUM", "0")
    by_kernel = gpu(op, a, b, **kw)
    bits = torch.int16 if in_cluster.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(in_cluster.view(bits), by_kernel.view(bits))
    ref = full_ref(op, *operands(op, case_tensors(op, T, N, K)))
    assert_budget(as_f64(in_cluster), ref, "bf16" if bits == torch.int16 else "f32", f"{op} T={T} in-cluster sum")
    no_device_fault()


# (op, T, N, K, forced split count or None for the planner's): clusters of 2 to 8 CTAs,
# transposed output (the swapped weight gradient) and row-major output, a ragged
# N = 48 (padding columns), the forward split over K, and the router's BF16x3 tiles
CLUSTER_CASES = [("wgrad", 16173, 64, 4096, 2), ("wgrad", 16173, 64, 4096, 3), ("wgrad", 16173, 64, 4096, None),
                 ("wgrad", 4100, 64, 512, 5), ("wgrad", 4100, 64, 512, 6), ("wgrad", 4100, 64, 512, 7),
                 ("wgrad", 4100, 64, 512, 8), ("wgrad", 4100, 64, 1024, None), ("wgrad", 16173, 128, 4096, None),
                 ("wgrad", 16173, 48, 5120, None), ("fwd", 64, 1024, 4096, None), ("router_wgrad", 1024, 256, 4096, None)]


@pytest.mark.parametrize("out_f32", [False, True])
@pytest.mark.parametrize("op,T,N,K,S", CLUSTER_CASES)
def test_cluster_sum_every_cluster_size(monkeypatch, op, T, N, K, S, out_f32):
    """A plan with one split unit per CTA adds its partials inside the GEMM's clusters
    (the plan reports the cluster size): CTA r of the cluster sums its share of the
    tile's rows over all partials in ascending split order, which gives the reduction
    kernel's bits, whatever the cluster size, output type or orientation."""
    router = op.startswith("router")
    if router and not out_f32:
        pytest.skip("the router's output is FP32")
    if S:
        monkeypatch.setenv("DP_FORCE_SPLITS", str(S))
    p = dp.plan(op, T, N, K, out_f32=out_f32)
    assert (p["splits"] == S if S else p["splits"] > 1), p
    assert p["full_units"] == 0 and not p["cta_pair"] and p["units"] == p["grid"] and p["splits"] <= 8, p
    if p["cluster_sum"] == 0 and p["splits"] > 4 and p["grid"] > 64:
        # (clusters live inside one GPC: how many of 5 to 8 CTAs run at once depends on
        # the device's GPCs; the reduction kernel sums such plans)
        pytest.skip(f"the device co-schedules too few clusters of {p['splits']} CTAs for {p['grid']} CTAs")
    assert p["cluster_sum"] == p["splits"], p
    c = {k: v.to(DEV) for k, v in case_tensors(op, T, N, K).items()}
    a, b = operands(op, c)
    kw = {} if router else {"out_dtype": torch.float32 if out_f32 else torch.bfloat16}
    in_cluster = gpu(op, a, b, **kw)
    monkeypatch.setenv("DP_FORCE_CLUSTER_SUM", "0")
    assert dp.plan(op, T, N, K, out_f32=out_f32)["cluster_sum"] == 0
    by_kernel = gpu(op, a, b, **kw)
    bits = torch.int32 if out_f32 else torch.int16
    assert torch.equal(in_cluster.view(bits), by_kernel.view(bits))
    if T * N * K <= (1 << 31):
        ref = full_ref(op, *operands(op, case_tensors(op, T, N, K)))
        assert_budget(as_f64(in_cluster), ref, "f32" if out_f32 else "bf16", f"{op} T={T} S={p['splits']}")
    no_device_fault()



def test_dependent_calls_keep_their_order():
    # Consecutive GEMMs overlap only their setup with the previous kernel: a call that
    # reads the previous call's output, and a call that overwrites a buffer the
    # previous call reads, give the same bits as the same calls with a full
    # device synchronisation between them.
    T, N, K = 4100, 1024, 2048
    c = {k: v.to(DEV) for k, v in case_tensors("fwd", T, N, K, seed=4).items()}
    X, W, dY = c["X"], c["W"], c["dY"]

    def chain(sync):
        x = X.clone()
        y = dp.dp_gemm_fwd(x, W)                        # reads x
        if sync:
            torch.cuda.synchronize()
        dx = dp.dp_gemm_dgrad(y, W, out=x)              # reads y (written just before), overwrites x
        if sync:
            torch.cuda.synchronize()
        dw = dp.dp_gemm_wgrad(y, dx, out_dtype=torch.float32)  # reads both
        torch.cuda.synchronize()
        return y, dx, dw

    a, b = chain(False), chain(True)
    for u, v in zip(a, b):
        bits = torch.int16 if u.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(u.view(bits), v.view(bits))
    no_device_fault()


@pytest.mark.parametrize("op,T,N,K", [("fwd", 300, 520, 1000), ("dgrad", 300, 520, 1000), ("wgrad", 300, 520, 1000),
                                      ("fwd", 16384, 1024, 512), ("wgrad", 64, 1024, 4096), ("fwd", 64, 40, 256),
                                      ("router_dgrad", 1000, 256, 4096), ("router_fwd", 300, 256, 4096)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_tma_store_matches_direct_store(monkeypatch, op, T, N, K, out_dtype):
    # Whole tiles leave through TMA stores of the staged 32-row blocks, or through the
    # epilogue warps' own stores: the same values, so the same bits, ragged edges
    # clipped either way (the output sits in a NaN-padded wider buffer)
    if op.startswith("router") and out_dtype == torch.bfloat16:
        pytest.skip("router output is FP32")
    c = {k: v.to(DEV) for k, v in case_tensors(op, T, N, K, seed=5).items()}
    a, b = operands(op, c)
    kw = {} if op.startswith("router") else {"out_dtype": out_dtype}
    if not op.startswith("router"):
        monkeypatch.setenv("DP_FORCE_SPLITS", "1")  # whole-K tiles: the results the stores carry
    outs = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("DP_FORCE_TMA_STORE", mode)
        probe = gpu(op, a, b, **kw)
        R, C = probe.shape
        wide = torch.full((R, C + 16), float("nan"), dtype=probe.dtype, device=DEV)
        view = wide[:, 8:8 + C]
        gpu(op, a, b, out=view, **kw)
        torch.cuda.synchronize()
        assert torch.isnan(wide[:, :8].float()).all() and torch.isnan(wide[:, 8 + C:].float()).all(), mode
        outs[mode] = view.clone()
    bits = torch.int16 if outs["1"].dtype == torch.bfloat16 else torch.int32
    assert torch.equal(outs["1"].view(bits), outs["0"].view(bits))
    no_device_fault()


@pytest.mark.parametrize("weight_layout", ["nk", "kn"])
def test_tma_store_matches_direct_store_batched_and_bwd(monkeypatch, weight_layout):
    H, T, N, K = 6, 300, 192, 136
    g = torch.Generator().manual_seed(11)
    X = torch.randn(T, H, K, generator=g).bfloat16().to(DEV).permute(1, 0, 2)
    dY = torch.randn(T, H, N, generator=g).bfloat16().to(DEV).permute(1, 0, 2)
    W = (torch.randn(H, N, K, generator=g) / 16).bfloat16().to(DEV)
    if weight_layout == "kn":
        W = W.transpose(1, 2).contiguous()
    # (the backward pass, co-scheduled where a tiling admits it: T = 300, N = 520, K = 1000)
    X2 = torch.randn(300, 1000, generator=g).bfloat16().to(DEV)
    W2 = (torch.randn(520, 1000, generator=g) / 32).bfloat16().to(DEV)
    dY2 = torch.randn(300, 520, generator=g).bfloat16().to(DEV)
    res = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("DP_FORCE_TMA_STORE", mode)
        r = []
        for od in (torch.bfloat16, torch.float32):
            r.append(dp.dp_gemm_fwd_batched(X, W, out_dtype=od, weight_layout=weight_layout))
            r.append(dp.dp_gemm_dgrad_batched(dY, W, out_dtype=od, weight_layout=weight_layout))
            r.append(dp.dp_gemm_wgrad_batched(dY, X, out_dtype=od, weight_layout=weight_layout))
            monkeypatch.setenv("DP_FORCE_FUSE", "1")
            r.extend(dp.dp_gemm_bwd(dY2, X2, W2, dx_dtype=od, dw_dtype=od))
            monkeypatch.delenv("DP_FORCE_FUSE")
        torch.cuda.synchronize()
        res[mode] = r
    for i, (x, y) in enumerate(zip(res["1"], res["0"])):
        bits = torch.int16 if x.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(x.contiguous().view(bits), y.contiguous().view(bits)), i
    no_device_fault()
