"""Failure detection on the GPU without a fault: the kernels' bounded barrier wait.

Every wait in the library's kernels gives up after a limit that is a launch
argument, records the timeout in the device status word (DP_ERR_TIMEOUT from
dp_device_error) and returns.  The wait probe runs that same wait in one CTA on a
barrier nothing arrives on, with a 1 ms limit: the kernel must return, report the
timeout, and leave the stream and context usable.  Nothing here traps, faults or
spins without a bound.
"""
import numpy as np
import pytest
import torch

import fp32_dense_projection_gb300 as dp
from fp32_dense_projection_gb300 import inputs
from gpu_common import DEV, as_f64, full_ref

pytestmark = pytest.mark.gpu

DP_ERR_TIMEOUT = 7


def test_wait_that_completes_records_nothing():
    dp.device_error(clear=True)
    dp.wait_probe(1_000_000, arrive=True)
    assert dp.device_error(clear=True) == 0


def test_wait_that_runs_out_returns_and_reports_timeout():
    dp.device_error(clear=True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    dp.wait_probe(1_000_000, arrive=False)  # 1 ms limit on a barrier nothing arrives on
    b.record()
    torch.cuda.synchronize()
    waited_ms = a.elapsed_time(b)
    assert dp.device_error(clear=True) == DP_ERR_TIMEOUT
    assert dp.device_error(clear=True) == 0  # cleared
    # the limit is the launch's: the kernel gave up after about 1 ms, not the 2 s default
    assert 0.9 <= waited_ms < 100.0, waited_ms
    # the stream and the context still work: a GEMM right after it on the same stream
    c = inputs.integer_case(129, 64, 136, seed=5)
    d = {k: v.to(DEV) for k, v in c.items()}
    dp.wait_probe(1_000_000, arrive=False)
    got = as_f64(dp.dp_gemm_fwd(d["X"], d["W"], out_dtype=torch.float32))
    assert np.array_equal(got, full_ref("fwd", c["X"], c["W"]))
    assert dp.device_error(clear=True) == DP_ERR_TIMEOUT
    assert dp.device_error(clear=True) == 0


def test_wait_probe_rejects_limits_out_of_range():
    for bad in (0, 999, 2_000_000_001):
        with pytest.raises(dp.DPError) as e:
            dp.wait_probe(bad)
        assert e.value.status == 1
