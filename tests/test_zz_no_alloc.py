"""fp8_linear_static_scratch: the layer for callers that cannot allocate.

Some callers may not create device allocations of their own (a plugin inside
a host application that owns all device memory, a latency-critical loop that
must not call cudaMalloc / cudaFree).  This entry point takes no workspace:
its scratch is a fixed array inside the library.  The tests call it through
the C ABI:
  * twice in a row, with shapes that take different GEMM kernels (the second
    call must not see the first call's leftovers): the output must equal
    fp8_linear's with a caller-provided workspace bit for bit (same kernels,
    same inputs), and lie within the parity tolerance of the oracle;
  * on a one-hot weight matrix (W = I), whose output is each quantized code
    of the scratch times its token's scale, rounded once to bf16: compared
    bit for bit with the oracle's codes and scales, on two calls in a row;
  * on a layer whose scratch need is exactly the array's size (accepted) and
    one 16-element step longer (rejected, output untouched).
This file is collected last, and also passes when run on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from fp8_w8a8_quantized_gb300 import workloads
from parity import bits, check_rows

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


def run(f, x, wq, s_w, N):
    M, K = x.shape
    y = torch.full((M, N), -1.0, dtype=torch.bfloat16, device=DEV)
    assert call(f, x, wq, s_w, y, M, N, K) == 0
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    return y


def test_matches_fp8_linear_on_two_calls_in_a_row(oracle_mod):
    f = entry()
    # a decode-sized layer, then a smaller layer that takes the other GEMM
    # kernel; both fit in the static scratch
    for (M, K, N, seed) in [(32, 4096, 6144, 1), (80, 1024, 520, 2)]:
        assert pkg.fp8_linear_workspace_size(M, N, K) <= SCRATCH_BYTES
        x = workloads.gaussian_outliers(M, K, seed, DEV)
        w = workloads.weights(N, K, seed, DEV)
        wq, s_w = pkg.fp8_quant_per_channel_weights(w)
        y_ref = pkg.fp8_linear(x, wq, s_w)
        y = run(f, x, wq, s_w, N)
        assert torch.equal(y, y_ref), f"static-scratch layer {M}x{N}x{K} differs from fp8_linear"
        qw_ref, sw_ref = oracle_mod.quant_rows_bf16(bits(w))
        y_orc, _, _ = oracle_mod.linear(bits(x), qw_ref, sw_ref)
        check_rows(y.double().cpu().numpy(), y_orc, f"static-scratch layer {M}x{N}x{K}")


def test_scratch_codes_and_scales_through_a_one_hot_layer(oracle_mod):
    # W = I (code 0x38 = 1.0 on the diagonal, weight scales 1): the GEMM sum
    # has one nonzero term, so y[m, n] = bf16(fl32(e4m3(xq[m, n]) * s_tok[m]))
    # exactly; neighbouring E4M3 values differ by at least 1/16 relatively,
    # more than a bf16 rounding, so every code in the scratch shows in y.
    f = entry()
    K = N = 1024
    wq = torch.zeros(N, K, dtype=torch.uint8, device=DEV)
    wq[torch.arange(N), torch.arange(N)] = 0x38
    s_w = torch.ones(N, dtype=torch.float32, device=DEV)
    for M, seed in [(24, 7), (80, 8)]:          # decode kernel, then paired-SM kernel
        x = workloads.gaussian_outliers(M, K, seed, DEV)
        y = run(f, x, wq, s_w, N)
        qx, s_tok = oracle_mod.quant_rows_bf16(bits(x))
        dec = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
        prod = dec[qx].astype(np.float32) * s_tok[:, None].astype(np.float32)
        expect = torch.from_numpy(prod).to(torch.bfloat16)
        assert torch.equal(y.cpu(), expect), f"scratch codes or scales differ at M={M}"


def test_layer_of_exactly_the_scratch_size(oracle_mod):
    f = entry()
    M, N, K = 16, 128, 524272            # 16*524272 = 8 MiB - 256, scales 256 B
    assert pkg.fp8_linear_workspace_size(M, N, K) == SCRATCH_BYTES
    x = workloads.gaussian_outliers(M, K, 9, DEV)
    w = workloads.weights(N, K, 9, DEV)
    wq, s_w = pkg.fp8_quant_per_channel_weights(w)
    y = run(f, x, wq, s_w, N)
    assert torch.equal(y, pkg.fp8_linear(x, wq, s_w))
    qw_ref, sw_ref = oracle_mod.quant_rows_bf16(bits(w))
    y_orc, _, _ = oracle_mod.linear(bits(x), qw_ref, sw_ref)
    check_rows(y.double().cpu().numpy(), y_orc, "layer of exactly the scratch size")
    # one 16-element step longer does not fit
    K2 = K + 16
    assert pkg.fp8_linear_workspace_size(M, N, K2) > SCRATCH_BYTES
    x2 = torch.zeros(M, K2, dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros(N, K2, dtype=torch.uint8, device=DEV)
    y2 = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=DEV)
    assert call(f, x2, w2, s_w, y2, M, N, K2) == FP8_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(y2 == 7.0), "a rejected call wrote its output"


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
