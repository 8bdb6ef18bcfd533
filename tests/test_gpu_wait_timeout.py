"""Failure detection on the GPU without a GPU fault: a bounded device wait
that runs out on purpose.

fp8_selftest_wait_timeout launches one small kernel that goes through the
GEMM kernels' give-up sequence: a wait on a barrier that nothing arrives on
gives up after a short limit and raises the CTA's abort flag, a second role
waiting with the kernels' own long limit returns on that flag, the issuer
drains its tensor-core work and TMEM is freed.  The host then sees
FP8_ERR_TIMEOUT from fp8_device_status(), clears it, and the context still
runs a layer correctly.  Nothing faults, traps or waits without a bound.
"""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from fp8_w8a8_quantized_gb300 import workloads
from parity import bits, check_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
FP8_ERR_TIMEOUT = 5


@pytest.mark.parametrize("limit_ns", [1_000_000, 20_000_000])
def test_bounded_wait_runs_out_and_reports(oracle_mod, limit_ns):
    L = pkg.lib()
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0, "status word not clear before the test"
    report = torch.zeros(4, dtype=torch.int64, device=DEV)
    try:
        st = L.fp8_selftest_wait_timeout(limit_ns, report.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
        assert st == 0
        torch.cuda.synchronize()
        gave_up, returned_on_abort, t_give_up, t_second = report.cpu().tolist()
        assert gave_up == 1, "the short wait did not give up"
        assert returned_on_abort == 1, "the second role did not return on the abort flag"
        assert t_give_up >= limit_ns
        # the loop checks the clock every 64 polls: it gives up soon after
        assert t_give_up < limit_ns + 50_000_000, t_give_up
        # the other role returned on the flag, not after its own 2 s limit
        assert t_give_up <= t_second < t_give_up + 50_000_000, (t_give_up, t_second)
        assert pkg.fp8_device_status() == FP8_ERR_TIMEOUT
        assert pkg.fp8_device_status(clear=True) == FP8_ERR_TIMEOUT
        assert pkg.fp8_device_status() == 0
    finally:
        pkg.fp8_device_status(clear=True)

    # the context is still usable: a layer afterwards matches the oracle
    x = workloads.gaussian_outliers(8, 1024, 51, DEV)
    w = workloads.weights(384, 1024, 51, DEV)
    wq, s_w = pkg.fp8_quant_per_channel_weights(w)
    y = pkg.fp8_linear(x, wq, s_w)
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    qw_ref, sw_ref = oracle_mod.quant_rows_bf16(bits(w))
    y_ref, _, _ = oracle_mod.linear(bits(x), qw_ref, sw_ref)
    check_rows(y.double().cpu().numpy(), y_ref, "layer after the self-test")
