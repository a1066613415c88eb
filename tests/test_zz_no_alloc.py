"""The weight-gradient entry point that allocates nothing.

It serves callers that cannot allocate device memory (a runtime that reserves all
memory at start-up, a host that forbids cudaMalloc on its hot path): its split
scratch is a 64 MiB array inside the library.  Called through the C ABI, twice in a row on the same shapes (the second
call finds the first call's leftovers in the shared array), its output must match
the workspace-taking entry point's: within the FP32 budget the parity tests use,
and in fact bit for bit, since both run the same plan and kernel.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
from fp32_dense_projection_gb300 import inputs
from budgets import check

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.mark.parametrize("T,N,K,out_dtype", [(16173, 64, 4096, torch.float32), (16173, 64, 4096, torch.bfloat16),
                                             (65537, 48, 5120, torch.float32), (1025, 128, 4096, torch.float32)])
def test_noalloc_matches_workspace_entry_point(T, N, K, out_dtype):
    c = inputs.thin_wgrad(T, N, K, seed=6)
    dY, X = c["dY"].to(DEV), c["X"].to(DEV)
    assert dp.workspace_size("wgrad", T, N, K, out_f32=out_dtype == torch.float32) > 0 or T == 1025
    want = dp.dp_gemm_wgrad(dY, X, out_dtype=out_dtype)
    for call in range(2):
        got = torch.full((N, K), float("nan"), dtype=out_dtype, device=DEV)
        dp.dp_gemm_wgrad_noalloc(dY, X, out=got)
        torch.cuda.synchronize()
        ok, msg = check(got.double().cpu().numpy(), want.double().cpu().numpy(),
                        "f32" if out_dtype == torch.float32 else "bf16")
        assert ok, f"call {call}: {msg}"
        bits = torch.int32 if out_dtype == torch.float32 else torch.int16
        assert torch.equal(got.view(bits), want.view(bits)), f"call {call}"
    assert dp.device_error() == 0


def test_noalloc_non_deterministic_fp32():
    # deterministic = 0 admits atomic split sums where the planner finds them faster:
    # the result is then checked against the workspace entry point within the FP32 budget
    T, N, K = 16173, 64, 4096
    c = inputs.thin_wgrad(T, N, K, seed=7)
    dY, X = c["dY"].to(DEV), c["X"].to(DEV)
    want = dp.dp_gemm_wgrad(dY, X, out_dtype=torch.float32, deterministic=False)
    for call in range(2):
        got = torch.full((N, K), float("nan"), dtype=torch.float32, device=DEV)
        dp.dp_gemm_wgrad_noalloc(dY, X, out=got, deterministic=False)
        torch.cuda.synchronize()
        ok, msg = check(got.double().cpu().numpy(), want.double().cpu().numpy(), "f32")
        assert ok, f"call {call}: {msg}"
    assert dp.device_error() == 0


def test_noalloc_back_to_back_calls_on_one_stream():
    # two calls queued without a synchronisation between them share the scratch array:
    # the stream orders them, so each output is the workspace entry point's, bit for bit
    T, N, K = 16173, 64, 4096
    cases = [inputs.thin_wgrad(T, N, K, seed=s) for s in (8, 9)]
    dev = [{k: v.to(DEV) for k, v in c.items()} for c in cases]
    want = [dp.dp_gemm_wgrad(d["dY"], d["X"], out_dtype=torch.float32) for d in dev]
    torch.cuda.synchronize()
    got = [torch.full((N, K), float("nan"), dtype=torch.float32, device=DEV) for _ in dev]
    for d, o in zip(dev, got):
        dp.dp_gemm_wgrad_noalloc(d["dY"], d["X"], out=o)
    torch.cuda.synchronize()
    for i in range(2):
        assert torch.equal(got[i].view(torch.int32), want[i].view(torch.int32)), f"call {i}"
    assert dp.device_error() == 0


def test_noalloc_rejects_plans_beyond_its_scratch():
    # 4096 -> 512 at T = 65537 splits 7 ways: 64 tiles x 7 x 128 KB of partials, under 64 MiB;
    # 8192 -> 1024 at T = 65537 needs far more than the built-in array and is refused.
    T, N, K = 65537, 1024, 8192
    need = dp.workspace_size("wgrad", T, N, K)
    assert need > (64 << 20)
    dY = torch.zeros(T, N, dtype=torch.bfloat16, device=DEV)
    X = torch.zeros(T, K, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(N, K, dtype=torch.float32, device=DEV)
    with pytest.raises(dp.DPError) as e:
        dp.dp_gemm_wgrad_noalloc(dY, X, out=out)
    assert e.value.status == 4
