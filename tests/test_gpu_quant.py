"""GPU parity of the per-token / per-channel quantizer: codes and scales must
equal the CPU oracle's bit for bit, on every configuration's shapes, ragged
and strided rows, and the numerics stress rows."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from fp8_w8a8_quantized_gb300 import workloads
from parity import bits, host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def check_quant(oracle_mod, x_gpu, which="token"):
    fn = pkg.fp8_quant_per_token if which == "token" else pkg.fp8_quant_per_channel_weights
    q, s = fn(x_gpu)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_rows_bf16(bits(x_gpu))
    qg, sg = host(q), host(s)
    assert np.array_equal(sg.view(np.uint32), s_ref.view(np.uint32)), "scales differ"
    diff = np.argwhere(qg != q_ref)
    assert diff.size == 0, f"{len(diff)} codes differ, first at {tuple(diff[0])}: " \
        f"gpu={qg[tuple(diff[0])]:#x} ref={q_ref[tuple(diff[0])]:#x}"
    return q, s


def test_tiny(oracle_mod):
    x, w = workloads.tiny(DEV)
    check_quant(oracle_mod, x)
    check_quant(oracle_mod, w, "channel")


@pytest.mark.parametrize("M", workloads.DECODE_M)
@pytest.mark.parametrize("K", [4096, 14336, 8192, 28672])
def test_decode_shapes(oracle_mod, M, K):
    check_quant(oracle_mod, workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, DEV))


@pytest.mark.parametrize("M,K", [(2048, 4096), (2048, 14336), (8192, 4096)])
def test_prefill_shapes(oracle_mod, M, K):
    check_quant(oracle_mod, workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, DEV))


def test_stress_rows(oracle_mod):
    x, kinds = workloads.stress(DEV)
    q, s = check_quant(oracle_mod, x)
    sg = host(s)
    assert all(sg[r] == 1.0 for r, k in enumerate(kinds) if k == "zero")


@pytest.mark.parametrize("N,K", [(4096, 4096), (6144, 4096), (4096, 14336)])
def test_weight_channels(oracle_mod, N, K):
    check_quant(oracle_mod, workloads.weights(N, K, workloads.SEED_DECODE, DEV), "channel")


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (5, 272), (33, 1040), (7, 2064),
                                 (130, 4112), (2, 65536), (3, 65552), (1, 131072),
                                 # ragged rows in the many-rows layout (two chunks a thread)
                                 (1000, 4112), (1300, 2064)])
def test_ragged_and_long_rows(oracle_mod, M, K):
    g = torch.Generator(device=DEV)
    g.manual_seed(M * 7 + K)
    x = (torch.randn(M, K, generator=g, device=DEV) * 3).to(torch.bfloat16)
    check_quant(oracle_mod, x)


def test_strided_rows_and_output_ld(oracle_mod):
    M, K, ldx, ldq = 37, 512, 520, 544
    base = workloads.gaussian_outliers(M, ldx, 9, DEV)
    x = base[:, :K]
    xq = torch.full((M, ldq), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.empty(M, dtype=torch.float32, device=DEV)
    st = pkg.lib().fp8_quant_per_token(x.data_ptr(), M, K, ldx, xq.data_ptr(), ldq, s.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_rows_bf16(bits(x))
    assert np.array_equal(host(xq)[:, :K], q_ref)
    assert np.all(host(xq)[:, K:] == 0xAB), "wrote past K"
    assert np.array_equal(host(s), s_ref)


def test_zero_K_gives_unit_scales():
    s = torch.zeros(5, dtype=torch.float32, device=DEV)
    x = torch.zeros(5, 16, dtype=torch.bfloat16, device=DEV)
    st = pkg.lib().fp8_quant_per_token(x.data_ptr(), 5, 0, 16, x.data_ptr(), 16, s.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.all(s == 1.0)


def test_repeatable_bits():
    x = workloads.gaussian_outliers(64, 4096, 3, DEV)
    q1, s1 = pkg.fp8_quant_per_token(x)
    q2, s2 = pkg.fp8_quant_per_token(x)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2)
