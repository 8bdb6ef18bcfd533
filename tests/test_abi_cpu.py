"""The C-ABI library loads and exports every entry point include/*.h
declares; host-side argument checks answer without touching a GPU (CPU only:
no call here reaches a kernel launch)."""
import glob
import os
import re
import subprocess

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def L():
    from fp8_w8a8_quantized_gb300 import build
    build.build()
    import fp8_w8a8_quantized_gb300 as pkg
    return pkg.lib()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names.update(re.findall(r"FP8_API\s+[\w\s\*]+?\b(fp8_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n


def test_exported_symbols_are_only_the_abi(L):
    from fp8_w8a8_quantized_gb300 import LIBRARY_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIBRARY_PATH],
                         capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    fp8 = {s for s in exported if s.startswith("fp8_")}
    assert fp8 == set(declared_symbols())


def test_status_strings(L):
    import fp8_w8a8_quantized_gb300 as pkg
    for code, name in pkg._binding.STATUS_NAMES.items():
        assert pkg.fp8_status_string(code) == name
    assert pkg.fp8_status_string(77) == "FP8_ERR_UNKNOWN"


def test_workspace_size(L):
    import fp8_w8a8_quantized_gb300 as pkg
    assert pkg.fp8_linear_workspace_size(1, 4096, 4096) == 4096 + 256
    assert pkg.fp8_linear_workspace_size(3, 10, 48) == 256 + 256
    assert pkg.fp8_linear_workspace_size(0, 10, 48) == 0
    assert pkg.fp8_linear_workspace_size(-1, 10, 48) == 0
    assert L.fp8_scaled_gemm_workspace_size(32, 4096, 4096) == 0


def test_host_checks_reject_before_any_launch(L):
    # null pointers, negative sizes, bad leading dimensions, K not a multiple
    # of 16, misaligned pointers: all answered on the host
    INVALID, UNSUP, WS = 1, 2, 3
    fake = 1 << 20  # never dereferenced: every call below is rejected first
    assert L.fp8_quant_per_token(None, 4, 32, 32, fake, 32, fake, None) == INVALID
    assert L.fp8_quant_per_token(fake, -1, 32, 32, fake, 32, fake, None) == INVALID
    assert L.fp8_quant_per_token(fake, 4, 32, 16, fake, 32, fake, None) == INVALID
    assert L.fp8_quant_per_token(fake, 4, 24, 24, fake, 32, fake, None) == UNSUP
    assert L.fp8_quant_per_token(fake + 8, 4, 32, 32, fake, 32, fake, None) == UNSUP
    assert L.fp8_quant_per_token(fake, 4, 32, 36, fake, 32, fake, None) == UNSUP
    assert L.fp8_quant_per_token(fake, 0, 32, 32, fake, 32, fake, None) == 0
    assert L.fp8_quant_per_channel_weights(fake, 4, 32, 32, None, 32, fake, None) == INVALID
    assert L.fp8_scaled_gemm(None, fake, fake, fake, fake, 4, 4, 32, None, 0, None) == INVALID
    assert L.fp8_scaled_gemm(fake, fake, fake, fake, fake, 4, 4, 40, None, 0, None) == UNSUP
    assert L.fp8_scaled_gemm(fake, fake, fake, fake, fake + 4, 4, 4, 32, None, 0, None) == UNSUP
    assert L.fp8_scaled_gemm(fake, fake, fake, fake, fake, 0, 4, 32, None, 0, None) == 0
    assert L.fp8_scaled_gemm(fake, fake, fake, fake, fake, 4, 0, 32, None, 0, None) == 0
    assert L.fp8_scaled_gemm(fake, fake, fake, fake, fake, 4, 4, -16, None, 0, None) == INVALID
    assert L.fp8_linear(fake, fake, fake, fake, 4, 4, 32, None, 0, None) == WS
    assert L.fp8_linear(fake, fake, fake, fake, 4, 4, 32, fake, 10, None) == WS
    assert L.fp8_linear(fake, fake, fake, fake, 4, 4, 32, fake + 16, 4096, None) == WS
    assert L.fp8_linear(fake, fake, fake, fake, 4, 4, 20, fake, 4096, None) == UNSUP
    assert L.fp8_linear(fake, fake, fake, fake, 0, 4, 32, None, 0, None) == 0
    assert L.fp8_linear(fake, None, fake, fake, 4, 4, 32, fake, 4096, None) == INVALID
    assert L.fp8_linear(fake, fake, fake, fake, 1 << 40, 4, 32, fake, 4096, None) == INVALID


def test_product_path_does_not_import_the_oracle():
    pkg_dir = os.path.join(ROOT, "fp8_w8a8_quantized_gb300")
    for path in glob.glob(os.path.join(pkg_dir, "**", "*"), recursive=True):
        if os.path.isfile(path) and path.endswith((".py", ".cu", ".cuh", ".h")):
            text = open(path).read()
            assert "import oracle" not in text and "from oracle" not in text, path
            assert "fp8_oracle" not in text and "orc_" not in text, path


def test_host_checks_of_the_scale_variants(L):
    INVALID, UNSUP, WS = 1, 2, 3
    fake = 1 << 20
    # static scale: x, M, K, ldx, s, xq, ldq, s_rows, stream
    assert L.fp8_quant_static(fake, 4, 32, 32, None, fake, 32, None, None) == INVALID
    assert L.fp8_quant_static(fake, 4, 24, 24, fake, fake, 32, None, None) == UNSUP
    assert L.fp8_quant_static(fake, 4, 32, 32, fake, fake, 32, fake + 2, None) == UNSUP
    assert L.fp8_quant_static(fake, 4, 32, 32, fake + 1, fake, 32, None, None) == UNSUP
    assert L.fp8_quant_static(fake, 0, 32, 32, fake, fake, 32, None, None) == 0
    # dynamic per-tensor: ..., s_out, s_rows, workspace, ws_bytes, stream
    assert L.fp8_quant_per_tensor_workspace_size(4096, 4096) == 8192
    assert L.fp8_quant_per_tensor(fake, 4, 32, 32, fake, 32, None, None, fake, 8192, None) == INVALID
    assert L.fp8_quant_per_tensor(fake, 4, 32, 32, fake, 32, fake, None, None, 0, None) == WS
    assert L.fp8_quant_per_tensor(fake, 4, 32, 32, fake, 32, fake, None, fake, 100, None) == WS
    assert L.fp8_quant_per_tensor(fake, 4, 32, 32, fake, 32, fake, None, fake + 4, 8192, None) == WS
    assert L.fp8_quant_per_tensor(fake, 4, 40, 40, fake, 48, fake, None, fake, 8192, None) == UNSUP
    assert L.fp8_quant_per_tensor(fake, 0, 32, 32, fake, 32, fake, None, None, 0, None) == 0
    # KV cache: kv, T, H, D, scale, scale_stride, slot, cache, n_slots, stream
    assert L.fp8_kv_cache_quant(fake, 4, 8, 24, fake, 1, None, fake, 16, None) == UNSUP
    assert L.fp8_kv_cache_quant(None, 4, 8, 128, fake, 1, None, fake, 16, None) == INVALID
    assert L.fp8_kv_cache_quant(fake, 4, 8, 128, None, 1, None, fake, 16, None) == INVALID
    assert L.fp8_kv_cache_quant(fake, -1, 8, 128, fake, 1, None, fake, 16, None) == INVALID
    assert L.fp8_kv_cache_quant(fake, 4, 8, 128, fake, -1, None, fake, 16, None) == INVALID
    assert L.fp8_kv_cache_quant(fake, 4, 8, 128, fake, 1, fake + 4, fake, 16, None) == UNSUP
    assert L.fp8_kv_cache_quant(fake, 4, 8, 128, fake, 1, None, fake + 8, 16, None) == UNSUP
    assert L.fp8_kv_cache_quant(fake, 4, 8, 128, fake + 2, 1, None, fake, 16, None) == UNSUP
    assert L.fp8_kv_cache_quant(fake, 0, 8, 128, fake, 1, None, fake, 16, None) == 0
    assert L.fp8_kv_cache_quant(fake, 4, 8, 128, fake, 1, None, fake, 0, None) == 0
    # keys and values: k, v, T, H, D, k_scale, v_scale, stride, slot, k_cache, v_cache, n, stream
    kv2 = L.fp8_kv_cache_quant_kv
    assert kv2(fake, None, 4, 8, 128, fake, fake, 1, None, fake, fake, 16, None) == INVALID
    assert kv2(fake, fake, 4, 8, 128, fake, None, 1, None, fake, fake, 16, None) == INVALID
    assert kv2(fake, fake, 4, 8, 128, fake, fake, 1, None, fake, None, 16, None) == INVALID
    assert kv2(fake, fake, 4, 8, 24, fake, fake, 1, None, fake, fake, 16, None) == UNSUP
    assert kv2(fake, fake + 8, 4, 8, 128, fake, fake, 1, None, fake, fake, 16, None) == UNSUP
    assert kv2(fake, fake, 4, 8, 128, fake, fake + 2, 1, None, fake, fake, 16, None) == UNSUP
    assert kv2(fake, fake, 4, 8, 128, fake, fake, 1, None, fake, fake + 8, 16, None) == UNSUP
    assert kv2(fake, fake, -1, 8, 128, fake, fake, 1, None, fake, fake, 16, None) == INVALID
    assert kv2(fake, fake, 0, 8, 128, fake, fake, 1, None, fake, fake, 16, None) == 0


def test_host_checks_of_the_blockwise_calls(L):
    INVALID, UNSUP, WS = 1, 2, 3
    fake = 1 << 20
    assert L.fp8_linear_blockwise_workspace_size(3, 7, 300) == 1024 + 256
    assert L.fp8_linear_blockwise_workspace_size(1, 4096, 4096) == 4096 + 256
    assert L.fp8_linear_blockwise_workspace_size(-1, 4, 32) == 0
    assert L.fp8_quant_per_token_group(fake, 4, 24, 24, fake, 32, fake, None) == UNSUP
    assert L.fp8_quant_per_token_group(fake, 4, 32, 32, fake, 32, None, None) == INVALID
    assert L.fp8_quant_per_token_group(fake, 0, 32, 32, fake, 32, fake, None) == 0
    assert L.fp8_quant_weight_blocks(fake, 65535 * 128 + 1, 32, 32, fake, 32, fake, None) == UNSUP
    assert L.fp8_quant_weight_blocks(fake, 4, 32, 16, fake, 32, fake, None) == INVALID
    assert L.fp8_scaled_gemm_blockwise(None, fake, fake, fake, fake, 4, 4, 32, None, 0, None) == INVALID
    assert L.fp8_scaled_gemm_blockwise(fake, fake, fake, fake, fake, 4, 4, 40, None, 0, None) == UNSUP
    assert L.fp8_scaled_gemm_blockwise(fake, fake, fake, fake, fake, 0, 4, 32, None, 0, None) == 0
    assert L.fp8_linear_blockwise(fake, fake, fake, fake, 4, 4, 32, None, 0, None) == WS
    assert L.fp8_linear_blockwise(fake, fake, fake, fake, 4, 4, 32, fake, 300, None) == WS
    assert L.fp8_linear_blockwise(fake, fake, fake, fake, 4, 4, 20, fake, 4096, None) == UNSUP
    assert L.fp8_linear_blockwise(fake, None, fake, fake, 4, 4, 32, fake, 4096, None) == INVALID


def test_host_checks_of_the_rmsnorm_calls(L):
    INVALID, UNSUP, WS = 1, 2, 3
    fake = 1 << 20
    # x, gamma, eps, M, K, ldx, xq, ldq, s_tok, y, stream
    assert L.fp8_rmsnorm_quant(fake, None, 1e-6, 4, 32, 32, fake, 32, fake, None, None) == INVALID
    assert L.fp8_rmsnorm_quant(fake, fake, -1.0, 4, 32, 32, fake, 32, fake, None, None) == INVALID
    assert L.fp8_rmsnorm_quant(fake, fake, float("nan"), 4, 32, 32, fake, 32, fake, None, None) == INVALID
    assert L.fp8_rmsnorm_quant(fake, fake + 8, 1e-6, 4, 32, 32, fake, 32, fake, None, None) == UNSUP
    assert L.fp8_rmsnorm_quant(fake, fake, 1e-6, 4, 65552, 65552, fake, 65552, fake, None, None) == UNSUP
    assert L.fp8_rmsnorm_quant(fake, fake, 1e-6, 4, 32, 32, fake, 32, fake, fake + 4, None) == UNSUP
    assert L.fp8_rmsnorm_quant(fake, fake, 1e-6, 0, 32, 32, fake, 32, fake, None, None) == 0
    # x, gamma, eps, wq, s_w, y, M, N, K, ws, ws_bytes, stream
    assert L.fp8_linear_rmsnorm(fake, fake, 1e-6, fake, fake, fake, 4, 4, 32, None, 0, None) == WS
    assert L.fp8_linear_rmsnorm(fake, None, 1e-6, fake, fake, fake, 4, 4, 32, fake, 4096, None) == INVALID
    assert L.fp8_linear_rmsnorm(fake, fake, 1e-6, fake, fake, fake, 4, 4, 24, fake, 4096, None) == UNSUP
    assert L.fp8_linear_rmsnorm(fake, fake, 1e-6, fake, fake, fake, 0, 4, 32, None, 0, None) == 0


def test_host_checks_of_the_selftest_and_static_scratch_calls(L):
    import ctypes
    INVALID, UNSUP = 1, 2
    fake = 1 << 20
    # wait self-test: limit_ns outside 1 us .. 100 ms, null or misaligned report
    assert L.fp8_selftest_wait_timeout(999, fake, None) == INVALID
    assert L.fp8_selftest_wait_timeout(100_000_001, fake, None) == INVALID
    assert L.fp8_selftest_wait_timeout(1_000_000, None, None) == INVALID
    assert L.fp8_selftest_wait_timeout(1_000_000, fake + 4, None) == UNSUP
    # static-scratch layer: the same argument checks as fp8_linear, answered
    # before the library looks at its array or at the device
    f = L.fp8_linear_static_scratch
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    assert f(None, fake, fake, fake, 4, 4, 32, None) == INVALID
    assert f(fake, fake, fake, fake, -1, 4, 32, None) == INVALID
    assert f(fake, fake, fake, fake, 4, 4, 24, None) == UNSUP
    assert f(fake + 8, fake, fake, fake, 4, 4, 32, None) == UNSUP
    assert f(fake, fake, fake + 2, fake, 4, 4, 32, None) == UNSUP
    assert f(fake, fake, fake, fake, 0, 4, 32, None) == 0
    assert f(fake, fake, fake, fake, 4, 0, 32, None) == 0


def test_calls_that_pass_the_checks_report_a_cuda_error_without_a_device(L):
    """With no usable GPU the first CUDA call fails, and a call that passed
    every host check answers FP8_ERR_CUDA (nothing is launched).  Skipped
    where a GPU is present: there these fake pointers would reach a kernel."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case needs a machine without one")
    CUDA = 4
    fake = 1 << 20
    assert L.fp8_quant_per_token(fake, 4, 32, 32, fake, 32, fake, None) == CUDA
    assert L.fp8_scaled_gemm(fake, fake, fake, fake, fake, 4, 4, 32, None, 0, None) == CUDA
    assert L.fp8_linear(fake, fake, fake, fake, 4, 4, 32, fake, 4096, None) == CUDA
    assert L.fp8_device_status(0) == CUDA
    assert L.fp8_selftest_wait_timeout(1_000_000, fake, None) == CUDA


def test_binding_rejects_tensors_the_kernels_cannot_take():
    """The Python binding checks shape, dtype, device and layout of every
    tensor before the C call, since the kernels index raw memory by the
    sizes they are given (CPU tensors are rejected too: no call is made)."""
    import torch
    import fp8_w8a8_quantized_gb300 as pkg

    M, K, N = 4, 64, 8
    x = torch.zeros(M, K, dtype=torch.bfloat16)
    wq = torch.zeros(N, K, dtype=torch.uint8)
    s_w = torch.ones(N, dtype=torch.float32)
    with pytest.raises(ValueError, match="x must be a CUDA"):
        pkg.fp8_linear(x, wq, s_w)                         # host memory
    with pytest.raises(ValueError, match="x must be a CUDA"):
        pkg.fp8_quant_per_token(x)
    with pytest.raises(ValueError, match="w must be a CUDA"):
        pkg.fp8_quant_per_channel_weights(x)
    with pytest.raises(ValueError, match="xq must be a CUDA"):
        pkg.fp8_scaled_gemm(wq[:M], s_w[:M], wq, s_w)
    with pytest.raises(ValueError, match="xq must be a CUDA"):
        pkg.fp8_scaled_gemm_blockwise(wq[:M], s_w[:M], wq, s_w)
    with pytest.raises(ValueError, match="x must be a CUDA"):
        pkg.fp8_linear_blockwise(x, wq, s_w)
    with pytest.raises(ValueError, match="x must be a CUDA"):
        pkg.fp8_linear_rmsnorm(x, x[0], 1e-6, wq, s_w)
    # the messages name what was wrong
    with pytest.raises(ValueError, match=r"shape \(8,\), contiguous; got torch.float32 \(7,\)"):
        pkg._binding._expect(s_w[:7], "s_w", (N,), torch.float32)
    with pytest.raises(ValueError, match="not contiguous"):
        pkg._binding._expect(x.t(), "y", (K, M), torch.bfloat16)
    with pytest.raises(ValueError, match="uint8"):
        pkg._binding._workspace(torch.zeros(4, dtype=torch.float32))
