"""Pins for the oracle's block-wise scales (CPU only): 1 x 128 activation
groups, 128 x 128 weight blocks and the block-scaled GEMM, checked against
the already pinned per-row / per-tensor rules, PyTorch's E4M3 cast, exact
rational brute force and a float64 dequantize-then-matmul."""
from fractions import Fraction

import numpy as np
import torch

from fp8_w8a8_quantized_gb300 import workloads


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def randn_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def test_one_group_is_the_per_token_rule(oracle_mod):
    x = workloads.gaussian_outliers(9, 128, seed=31)
    qg, sg = oracle_mod.quant_groups_bf16(bits(x))
    qt, st = oracle_mod.quant_rows_bf16(bits(x))
    assert sg.shape == (9, 1)
    assert np.array_equal(sg[:, 0], st) and np.array_equal(qg, qt)


def test_groups_are_per_token_rule_on_each_slice(oracle_mod):
    x = workloads.student_t_outliers(7, 3 * 128 + 48, seed=32)   # last group partial
    q, s = oracle_mod.quant_groups_bf16(bits(x))
    assert s.shape == (7, 4)
    for g in range(4):
        sl = slice(128 * g, min(128 * (g + 1), x.shape[1]))
        qt, st = oracle_mod.quant_rows_bf16(bits(x[:, sl]))
        assert np.array_equal(s[:, g], st), g
        assert np.array_equal(q[:, sl], qt), g


def test_weight_blocks_are_per_tensor_rule_on_each_block(oracle_mod):
    N, K = 200, 272                    # partial blocks along both dimensions
    w = randn_bf16((N, K), 33, 0.05)
    w[130:140, 200:210] = 0            # part of a block zero, not all of it
    w[128:200, 256:272] = 0            # a whole (partial) block zero
    q, s = oracle_mod.quant_weight_blocks_bf16(bits(w))
    assert s.shape == (2, 3)
    for nb in range(2):
        for kb in range(3):
            rs = slice(128 * nb, min(N, 128 * (nb + 1)))
            ks = slice(128 * kb, min(K, 128 * (kb + 1)))
            qt, st = oracle_mod.quant_tensor_bf16(bits(w[rs, ks]))
            assert s[nb, kb] == st, (nb, kb)
            assert np.array_equal(q[rs, ks], qt), (nb, kb)
    assert s[1, 2] == 1.0 and np.all(q[128:200, 256:272] == 0)


def test_block_maximum_lands_on_448_and_torch_witness(oracle_mod):
    w = workloads.weights(256, 384, seed=34)
    q, s = oracle_mod.quant_weight_blocks_bf16(bits(w))
    wf = w.float().numpy()
    for nb in range(2):
        for kb in range(3):
            blk = wf[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)]
            qb = q[128 * nb:128 * (nb + 1), 128 * kb:128 * (kb + 1)]
            i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert qb[i] in (0x7E, 0xFE)
            quot = (blk / s[nb, kb]).astype(np.float32)
            witness = torch.tensor(quot).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(qb, witness)


def exact_blockwise(qx, s_x, qw, s_w, m, n, dec):
    """y[m, n] from the definition with every scale inside the sum, in
    rationals: sum_k dec(qx) dec(qw) s_x[m, k // 128] s_w[n // 128, k // 128]."""
    tot = Fraction(0)
    for k in range(qx.shape[1]):
        tot += (Fraction(float(dec[qx[m, k]])) * Fraction(float(dec[qw[n, k]]))
                * Fraction(float(s_x[m, k // 128])) * Fraction(float(s_w[n // 128, k // 128])))
    return tot


def test_blockwise_gemm_brute_force(oracle_mod):
    M, N, K = 3, 130, 272
    x = workloads.student_t_outliers(M, K, seed=35)
    w = randn_bf16((N, K), 36, 0.1)
    w[:, 128:256] *= 40                 # scales vary strongly along k
    qx, sx = oracle_mod.quant_groups_bf16(bits(x))
    qw, sw = oracle_mod.quant_weight_blocks_bf16(bits(w))
    dec = oracle_mod.e4m3_decode(np.arange(256, dtype=np.uint8))
    y = oracle_mod.gemm_blockwise(qx, sx, qw, sw)
    for m in range(M):
        for n in (0, 1, 64, 127, 128, 129):
            ref = exact_blockwise(qx, sx, qw, sw, m, n, dec)
            assert abs(Fraction(y[m, n]) - ref) <= abs(ref) * Fraction(1, 10**12) + \
                Fraction(1, 10**30), (m, n)
    pts = oracle_mod.gemm_blockwise(qx, sx, qw, sw, rows=[2, 0, 1], cols=[129, 5, 64])
    assert np.array_equal(pts, y[[2, 0, 1], [129, 5, 64]])


def test_blockwise_gemm_equals_dequantize_then_matmul(oracle_mod):
    M, N, K = 17, 300, 640
    x = workloads.gaussian_outliers(M, K, seed=37)
    w = workloads.weights(N, K, seed=38)
    qx, sx = oracle_mod.quant_groups_bf16(bits(x))
    qw, sw = oracle_mod.quant_weight_blocks_bf16(bits(w))
    xd = oracle_mod.e4m3_decode(qx) * np.repeat(sx.astype(np.float64), 128, axis=1)[:, :K]
    s_full = np.repeat(np.repeat(sw.astype(np.float64), 128, axis=0), 128, axis=1)[:N, :K]
    wd = oracle_mod.e4m3_decode(qw) * s_full
    ref = (torch.tensor(xd) @ torch.tensor(wd).T).numpy()
    y = oracle_mod.gemm_blockwise(qx, sx, qw, sw)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_constant_scales_reduce_to_the_per_channel_gemm(oracle_mod):
    # scales constant along k (one weight row per "block", bn = 1) are the
    # per-token x per-channel layer the scales move out of
    M, N, K = 5, 40, 384
    x = workloads.gaussian_outliers(M, K, seed=39)
    w = workloads.weights(N, K, seed=40)
    qx, st = oracle_mod.quant_rows_bf16(bits(x))
    qw, sc = oracle_mod.quant_rows_bf16(bits(w))
    y1 = oracle_mod.scaled_gemm(qx, st, qw, sc)
    y2 = oracle_mod.gemm_blockwise(qx, np.repeat(st[:, None], 3, axis=1), qw,
                                   np.repeat(sc[:, None], 3, axis=1), bn=1)
    assert np.allclose(y1, y2, rtol=1e-13, atol=0)
