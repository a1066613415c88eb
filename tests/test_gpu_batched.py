"""Batched projection GEMMs (B independent problems in one launch) against the
FP64 oracle, problem by problem: packed and strided (per-head slice) views, both
weight layouts ([N][K] and [K][N]), BF16 and FP32 output, ragged token counts.

The pages' integration runs its per-head projections as "one batched BF16 GEMM
over strided views, forward and both gradients" with a weight layout option
(FlashInfer page "cache the router entry points' calls ...", the downstream
integration text)."""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
import oracle
from fp32_dense_projection_gb300 import inputs
from gpu_common import DEV, as_f64, assert_budget, no_device_fault

pytestmark = pytest.mark.gpu


def heads(B, T, D, seed, role, scale=1.0, integer=False):
    """[B, T, D] per-head views of one [T, B, D] tensor (batch stride D, row stride B*D)."""
    if integer:
        g = torch.Generator().manual_seed(seed * 16 + role)
        full = torch.randint(-2, 3, (T, B, D), generator=g).to(torch.bfloat16)
    else:
        full = inputs.normal((T, B, D), seed, role, scale)
    return full.permute(1, 0, 2)


def refs(op, a, b, kn):
    """Per-problem FP64 oracle results, as [B, rows, cols] float64."""
    out = []
    for i in range(a.shape[0]):
        ai, bi = a[i].contiguous(), b[i].contiguous()
        if op == "fwd":
            r = oracle.fwd_bf16(ai, bi.t().contiguous() if kn else bi)
        elif op == "dgrad":
            r = oracle.dgrad_bf16(ai, bi.t().contiguous() if kn else bi)
        else:
            r = oracle.wgrad_bf16(ai, bi)
            r = r.T if kn else r
        out.append(np.ascontiguousarray(r))
    return np.stack(out)


FN = {"fwd": dp.dp_gemm_fwd_batched, "dgrad": dp.dp_gemm_dgrad_batched, "wgrad": dp.dp_gemm_wgrad_batched}


def make(op, B, T, N, K, kn, seed, integer=False, strided=True):
    sc = 1.0 if integer else 1.0 / 16
    X = heads(B, T, K, seed, inputs.ROLE_X, integer=integer)
    dY = heads(B, T, N, seed, inputs.ROLE_DY, integer=integer)
    g = torch.Generator().manual_seed(seed * 16 + inputs.ROLE_W)
    W = (torch.randint(-2, 3, (B, N, K), generator=g).to(torch.bfloat16) if integer
         else (torch.randn(B, N, K, generator=g) * sc).to(torch.bfloat16))
    if kn:
        W = W.transpose(1, 2).contiguous()
    if not strided:
        X, dY = X.contiguous(), dY.contiguous()
    a, b = {"fwd": (X, W), "dgrad": (dY, W), "wgrad": (dY, X)}[op]
    return a, b


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("kn", [False, True])
@pytest.mark.parametrize("B,T,N,K", [(3, 77, 24, 136), (5, 130, 64, 64), (2, 257, 136, 520)])
def test_batched_integer_exact(op, kn, B, T, N, K):
    a, b = make(op, B, T, N, K, kn, seed=B + T, integer=True)
    ref = refs(op, a, b, kn)
    got = FN[op](a.to(DEV), b.to(DEV), out_dtype=torch.float32, weight_layout="kn" if kn else "nk")
    assert np.array_equal(as_f64(got), ref), (op, kn, B, T, N, K)
    no_device_fault()


@pytest.mark.parametrize("op", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("kn", [False, True])
@pytest.mark.parametrize("strided", [True, False])
def test_batched_budget(op, kn, strided):
    B, T, N, K = 8, 1000, 128, 512   # per-head projections: 8 heads, 512 -> 128
    a, b = make(op, B, T, N, K, kn, seed=7, strided=strided)
    ref = refs(op, a, b, kn)
    # keep the per-head layout ([T, B, D] storage, batch stride D) on the device too
    da = a.permute(1, 0, 2).contiguous().to(DEV).permute(1, 0, 2) if strided else a.contiguous().to(DEV)
    db = b.permute(1, 0, 2).contiguous().to(DEV).permute(1, 0, 2) if strided and op == "wgrad" else b.to(DEV)
    for od, name in ((torch.bfloat16, "bf16"), (torch.float32, "f32")):
        got = FN[op](da, db, out_dtype=od, weight_layout="kn" if kn else "nk")
        assert_budget(as_f64(got).ravel(), ref.ravel(), name, f"batched {op} kn={kn} {name}")
        again = FN[op](da, db, out_dtype=od, weight_layout="kn" if kn else "nk")
        bits = torch.int16 if od == torch.bfloat16 else torch.int32
        assert torch.equal(got.view(bits), again.view(bits))
    no_device_fault()


def test_batched_split_plans(monkeypatch):
    # many tokens per problem: split contractions (ordered sums) inside a batched launch
    B, T, N, K = 4, 8192, 64, 256
    monkeypatch.setenv("DP_FORCE_SPLITS", "3")
    for kn in (False, True):
        p = dp.plan_batched("wgrad", B, T, N, K, weight_kn=kn)
        assert p["splits"] == 3 and p["batch"] == B and p["tiles"] == B * p["tiles_m"] * p["tiles_n"]
        a, b = make("wgrad", B, T, N, K, kn, seed=3)
        ref = refs("wgrad", a, b, kn)
        got = dp.dp_gemm_wgrad_batched(a.to(DEV), b.to(DEV), out_dtype=torch.float32,
                                       weight_layout="kn" if kn else "nk")
        assert_budget(as_f64(got).ravel(), ref.ravel(), "f32", f"batched split wgrad kn={kn}")
    no_device_fault()


def test_batched_empty_tokens_zero_the_weight_gradient():
    B, N, K = 3, 64, 128
    dY = torch.empty(B, 0, N, dtype=torch.bfloat16, device=DEV)
    X = torch.empty(B, 0, K, dtype=torch.bfloat16, device=DEV)
    out = torch.full((B, N, K), float("nan"), dtype=torch.float32, device=DEV)
    dp.dp_gemm_wgrad_batched(dY, X, out=out, out_dtype=torch.float32)
    assert torch.count_nonzero(out) == 0
