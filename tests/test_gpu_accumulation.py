"""Characterises how the tensor core adds into its FP32 accumulator, the fact the
planner's bound on accumulation length rests on: a sum is rounded toward zero
(2^24 + 3 gives 2^24 + 2, where round-to-nearest-even would give 2^24 + 4), both
across MMA instructions and inside one.  Exact small-integer inputs, one tile."""
import pytest
import torch

import fp32_dense_projection_gb300 as dp

pytestmark = pytest.mark.gpu


def test_fp32_accumulate_rounds_toward_zero():
    M, N, K = 128, 64, 64
    X = torch.zeros(M, K, dtype=torch.bfloat16)
    W = torch.ones(N, K, dtype=torch.bfloat16)
    X[0, 0], X[0, 16] = 2.0**24, 3.0        # second K=16 instruction adds 3
    X[1, 0], X[1, 1] = 2.0**24, 3.0         # same instruction
    X[2, 0], X[2, 16] = -(2.0**24), -3.0    # negative side
    X[3, 0], X[3, 16] = 2.0**24, 1.0        # a tie
    Y = dp.dp_gemm_fwd(X.cuda(), W.cuda(), out_dtype=torch.float32).cpu().double()
    base = 2.0**24
    assert Y[0, 0].item() - base == 2.0
    assert Y[1, 0].item() - base == 2.0
    assert Y[2, 0].item() + base == -2.0
    assert Y[3, 0].item() - base == 0.0
    assert torch.equal(Y[:4, :], Y[:4, :1].expand(4, N))
