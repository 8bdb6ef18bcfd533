"""Pins for the oracle's scaled FP8 GEMM and epilogue (CPU only).

Witnesses: PyTorch's float64 matmul of the decoded values (a library
routine), brute force with Python integers on the tiny layer, closed forms
with constant codes, and the factored-scale identity y = s_a s_w (q_a . q_w)
("FP8 Inference Explained, in depth", "Inside a quantized linear layer").
"""
import numpy as np
import pytest
import torch

from fp8_w8a8_quantized_gb300 import workloads

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def torch_dec(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)


@pytest.mark.parametrize("M,N,K", [(3, 5, 16), (17, 33, 48), (40, 70, 1024)])
def test_exact_gemm_vs_torch_fp64(oracle_mod, M, N, K):
    rng = np.random.default_rng(M * N + K)
    qx = rng.choice(FINITE, size=(M, K))
    qw = rng.choice(FINITE, size=(N, K))
    acc = oracle_mod.gemm_exact(qx, qw)
    ref = torch_dec(qx) @ torch_dec(qw).T          # exact: all terms on 2^-18 grid
    assert np.array_equal(acc.astype(np.float64) * 2.0 ** -18, ref.numpy())


def test_closed_forms(oracle_mod):
    K = 4096
    one, m_one, big = 0x38, 0xB8, 0x7E             # 1.0, -1.0, 448
    qx = np.full((2, K), one, dtype=np.uint8)
    qx[1] = m_one
    qw = np.full((3, K), one, dtype=np.uint8)
    qw[2] = big
    s_tok = np.array([0.5, 2.0], dtype=np.float32)
    s_w = np.array([1.0, 0.25, 3.0], dtype=np.float32)
    y = oracle_mod.scaled_gemm(qx, s_tok, qw, s_w)
    expect = np.array([[K * 0.5, K * 0.5 * 0.25, K * 448 * 0.5 * 3.0],
                       [-K * 2.0, -K * 2.0 * 0.25, -K * 448 * 2.0 * 3.0]])
    assert np.array_equal(y, expect)
    # the largest magnitude sum at the largest K the configs use stays exact
    K = 28672
    qx = np.full((1, K), big, dtype=np.uint8)
    acc = oracle_mod.gemm_exact(qx, qx)
    assert acc[0, 0] == K * (448 * 512) ** 2


def test_tiny_layer_bruteforce_python_ints(oracle_mod):
    x, w = workloads.tiny()
    qw, s_w = oracle_mod.quant_rows_bf16(bits(w))
    y, qx, s_tok = oracle_mod.linear(bits(x), qw, s_w)
    assert y.shape == (18, 256)
    ints = {int(c): int(round(v * 512)) for c, v in
            zip(FINITE, oracle_mod.e4m3_decode(FINITE))}
    X = [[ints[int(c)] for c in row] for row in qx]
    W = [[ints[int(c)] for c in row] for row in qw]
    for m in range(18):
        xm = X[m]
        for n in range(256):
            acc = sum(a * b for a, b in zip(xm, W[n]))
            ref = acc * 2.0 ** -18 * float(s_tok[m]) * float(s_w[n])
            assert abs(y[m, n] - ref) <= 1e-15 * max(1.0, abs(ref))


def test_factored_scales_identity(oracle_mod):
    x = workloads.gaussian_outliers(24, 512, seed=5)
    w = workloads.weights(40, 512, seed=5)
    qw, s_w = oracle_mod.quant_rows_bf16(bits(w))
    y, qx, s_tok = oracle_mod.linear(bits(x), qw, s_w)
    a = torch_dec(qx) * torch.from_numpy(s_tok.astype(np.float64))[:, None]
    b = torch_dec(qw) * torch.from_numpy(s_w.astype(np.float64))[:, None]
    ref = (a @ b.T).numpy()
    err = np.abs(y - ref).max() / np.abs(ref).max()
    assert err < 1e-12


def test_points_match_full(oracle_mod):
    x = workloads.gaussian_outliers(9, 256, seed=6)
    w = workloads.weights(33, 256, seed=6)
    qw, s_w = oracle_mod.quant_rows_bf16(bits(w))
    y, qx, s_tok = oracle_mod.linear(bits(x), qw, s_w)
    rows = np.repeat(np.arange(9), 33)
    cols = np.tile(np.arange(33), 9)
    yp = oracle_mod.linear_points(qx, s_tok, qw, s_w, rows, cols)
    assert np.array_equal(yp, y.ravel())


def test_fp8_layer_close_to_bf16_layer(oracle_mod):
    # FP8 W8A8 is meant to approximate the unquantized layer: relative
    # Frobenius error of a few percent at most (E4M3 steps are 12.5 %)
    x = workloads.gaussian_outliers(32, 1024, seed=8)
    w = workloads.weights(64, 1024, seed=8)
    qw, s_w = oracle_mod.quant_rows_bf16(bits(w))
    y, _, _ = oracle_mod.linear(bits(x), qw, s_w)
    ref = (x.double() @ w.double().T).numpy()
    rel = np.linalg.norm(y - ref) / np.linalg.norm(ref)
    assert rel < 0.05
