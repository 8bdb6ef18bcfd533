"""fp8_linear_static_scratch: the layer for callers that cannot allocate.

Some callers may not create device allocations of their own (a plugin inside
a host application that owns all device memory, a latency-critical loop that
must not call cudaMalloc / cudaFree).  This entry point takes no workspace:
its scratch is a fixed array inside the library.  The test calls it through
the C ABI twice in a row, with different shapes (the second call must not see
the first call's leftovers), and checks each output against fp8_linear with
a caller-provided workspace, within the parity tolerance of the other tests.
This file is collected last, and also passes when run on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from fp8_w8a8_quantized_gb300 import workloads
from parity import check_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_BYTES = 8 << 20
FP8_ERR_WORKSPACE = 3


def entry():
    f = pkg.lib().fp8_linear_static_scratch
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    return f


def call(f, x, wq, s_w, y, M, N, K):
    return f(x.data_ptr(), wq.data_ptr(), s_w.data_ptr(), y.data_ptr(), M, N, K,
             torch.cuda.current_stream().cuda_stream)


def test_matches_fp8_linear_on_two_calls_in_a_row():
    f = entry()
    # a decode-sized layer, then a smaller layer that takes the other GEMM
    # kernel; both fit in the static scratch
    for (M, K, N, seed) in [(32, 4096, 6144, 1), (80, 1024, 520, 2)]:
        assert pkg.fp8_linear_workspace_size(M, N, K) <= SCRATCH_BYTES
        x = workloads.gaussian_outliers(M, K, seed, DEV)
        w = workloads.weights(N, K, seed, DEV)
        wq, s_w = pkg.fp8_quant_per_channel_weights(w)
        y_ref = pkg.fp8_linear(x, wq, s_w)
        y = torch.full((M, N), -1.0, dtype=torch.bfloat16, device=DEV)
        assert call(f, x, wq, s_w, y, M, N, K) == 0
        torch.cuda.synchronize()
        assert pkg.fp8_device_status() == 0
        check_rows(y.double().cpu().numpy(), y_ref.double().cpu().numpy(),
                   f"static-scratch layer {M}x{N}x{K}")


def test_rejects_layers_larger_than_the_scratch():
    f = entry()
    M, K, N = 2048, 4096, 128          # M*K alone is the whole array
    assert pkg.fp8_linear_workspace_size(M, N, K) > SCRATCH_BYTES
    x = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    wq = torch.zeros(N, K, dtype=torch.uint8, device=DEV)
    s_w = torch.ones(N, dtype=torch.float32, device=DEV)
    y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    assert call(f, x, wq, s_w, y, M, N, K) == FP8_ERR_WORKSPACE
    assert call(f, x, wq, s_w, y, 0, N, K) == 0
    torch.cuda.synchronize()
    assert torch.all(y == 7.0), "a rejected call wrote its output"
