"""GPU parity of RMSNorm with the per-token quantizer fused into it.

The normalised bf16 row must lie, element by element, inside the oracle's
bracket for a sum of squares within 2^-17 of the exact one (the kernel's
fp32 reduction is proven within that bound, and every later step is a
monotone IEEE operation, so the bracket is exact: most elements have a single
admissible value).  The codes and scales must then be bit-exactly the
per-token rule applied to the kernel's own normalised row, and the fused
layer must agree with the oracle GEMM on those codes."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from fp8_w8a8_quantized_gb300 import workloads
from parity import bits, check_rows, host

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL_ERR = 2.0 ** -17   # relative error bound of the kernel's sum of squares


def to_f(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).float().numpy()


def gamma(K, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (1.0 + 0.3 * torch.randn(K, generator=g)).to(torch.bfloat16).to(DEV)


def check(oracle_mod, x, g, eps):
    q, s, y = pkg.fp8_rmsnorm_quant(x, g, eps, y=True)
    torch.cuda.synchronize()
    y_lo, y_hi, _ = oracle_mod.rmsnorm_bracket_bf16(bits(x), bits(g), eps, REL_ERR)
    yg = to_f(bits(y))
    lo, hi = to_f(y_lo), to_f(y_hi)
    inside = (np.abs(yg) >= np.abs(lo)) & (np.abs(yg) <= np.abs(hi)) & \
        ((np.sign(yg) == np.sign(hi)) | (yg == 0))
    bad = np.argwhere(~inside)
    assert bad.size == 0, f"{len(bad)} normalised values outside the bracket, first at " \
        f"{tuple(bad[0])}: gpu={yg[tuple(bad[0])]!r} bracket=[{lo[tuple(bad[0])]!r}, {hi[tuple(bad[0])]!r}]"
    q_ref, s_ref = oracle_mod.quant_rows_bf16(bits(y))
    assert np.array_equal(host(s).view(np.uint32), s_ref.view(np.uint32)), "scales differ"
    assert np.array_equal(host(q), q_ref), "codes differ"
    return float(np.mean(lo != hi))


@pytest.mark.parametrize("M,K", [(1, 4096), (8, 4096), (32, 14336), (2048, 4096), (8192, 4096),
                                 (3, 16), (5, 272), (33, 1040), (130, 4112), (3, 65536),
                                 (2, 28672), (1000, 4112), (1300, 2064)])
def test_rmsnorm_quant(oracle_mod, M, K):
    x = workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, DEV)
    amb = check(oracle_mod, x, gamma(K, K), 1e-6)
    assert amb < 0.01


def test_rmsnorm_quant_stress_rows_and_eps(oracle_mod):
    x, _ = workloads.stress(DEV, M=512, K=4096)      # log-uniform, zero, ties, outliers
    g = gamma(4096, 7)
    for eps in (1e-5, 1.0):
        check(oracle_mod, x, g, eps)
    # an all-zero row with eps > 0: y = 0, scale 1
    z = torch.zeros(4, 256, dtype=torch.bfloat16, device=DEV)
    q, s, y = pkg.fp8_rmsnorm_quant(z, gamma(256, 8), 1e-6, y=True)
    torch.cuda.synchronize()
    assert torch.all(y == 0) and torch.all(s == 1.0) and torch.all(q == 0)


def test_rmsnorm_quant_strided_rows(oracle_mod):
    M, K, ldx = 37, 512, 520
    base = workloads.gaussian_outliers(M, ldx, 9, DEV)
    check(oracle_mod, base[:, :K], gamma(K, 9), 1e-6)


@pytest.mark.parametrize("M,K,N", [(1, 4096, 6144), (32, 4096, 4096), (18, 256, 256),
                                   (300, 4096, 1024), (2048, 4096, 512)])
def test_linear_rmsnorm(oracle_mod, M, K, N):
    x = workloads.student_t_outliers(M, K, 11, DEV)
    g = gamma(K, 12)
    w = workloads.weights(N, K, 13, DEV)
    wq, s_w = pkg.fp8_quant_per_channel_weights(w)
    ws = torch.empty(pkg.fp8_linear_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    y = pkg.fp8_linear_rmsnorm(x, g, 1e-6, wq, s_w, workspace=ws)
    q, s, _ = pkg.fp8_rmsnorm_quant(x, g, 1e-6)   # same kernel, same bytes
    torch.cuda.synchronize()
    off = -(-(M * K) // 256) * 256
    assert torch.equal(ws[:M * K].view(M, K), q)
    assert torch.equal(ws[off:off + 4 * M].view(torch.float32), s)
    y_ref = oracle_mod.scaled_gemm(host(q), host(s), host(wq), host(s_w))
    check_rows(host(y.float()), y_ref, f"linear rmsnorm {M}x{K}x{N}")
    assert pkg.fp8_device_status() == pkg.FP8_OK
