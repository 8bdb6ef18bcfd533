"""Exhaustive quantizer parity: every bf16 bit pattern under many static
scales (tiny, huge and subnormal ones included) and as rows with their own
dynamic scale, and quotients placed within a few fp32 ulps of E4M3 rounding
boundaries, must give the bytes of the fp32-division definition."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from parity import bits, host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def all_bf16():
    """Every bf16 bit pattern once, as a [256, 256] tensor (row = high byte)."""
    return torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16) \
        .reshape(256, 256).to(DEV)


def nan_mask(x_bits):
    return ((x_bits & 0x7F80) == 0x7F80) & ((x_bits & 0x007F) != 0)


def assert_codes_except_nan(q_gpu, q_ref, x_bits, what):
    """Bytes equal, except that where the input or the quotient is NaN (an inf
    row scale makes inf / inf) any E4M3 NaN code (0x7F or 0xFF) is accepted:
    NaN and inf inputs are outside the layer's contract."""
    g = host(q_gpu)
    nan = nan_mask(x_bits) | (q_ref == 0x7F)
    diff = np.argwhere((g != q_ref) & ~nan)
    assert diff.size == 0, f"{what}: {len(diff)} codes differ, first at {tuple(diff[0])}: " \
        f"x={x_bits[tuple(diff[0])]:#06x} gpu={g[tuple(diff[0])]:#x} ref={q_ref[tuple(diff[0])]:#x}"
    assert np.all((g[nan] & 0x7F) == 0x7F), f"{what}: NaN input must give an E4M3 NaN code"


SCALES = [1.0, 1.0 / 3.0, 0.0123, 120.0 / 448.0, 7.5, 2.0 ** -10, 1e-3, 0.75, 1.0 / 448.0,
          3.0e-39, 1.0e-45, 2.0 ** -126, 2.0 ** 126, 3.0e38, 2.0 ** 127]


@pytest.mark.parametrize("s_val", SCALES)
def test_every_bf16_pattern_static_scale(oracle_mod, s_val):
    x = all_bf16()
    s32 = np.float32(s_val)
    s = torch.tensor([s32], dtype=torch.float32, device=DEV)
    q = pkg.fp8_quant_static(x, s)
    torch.cuda.synchronize()
    xb = bits(x)
    assert_codes_except_nan(q, oracle_mod.quant_rows_scaled_bf16(xb, s32), xb, f"s={s_val}")


def test_every_bf16_pattern_dynamic_rows(oracle_mod):
    # each row of the pattern table has its own scale (some rows hold inf,
    # whose scale is inf; NaN never counts towards the maximum)
    x = all_bf16()
    q, s = pkg.fp8_quant_per_token(x)
    torch.cuda.synchronize()
    xb = bits(x)
    q_ref, s_ref = oracle_mod.quant_rows_bf16(xb)
    assert np.array_equal(host(s).view(np.uint32), s_ref.view(np.uint32))
    assert_codes_except_nan(q, q_ref, xb, "per-token rows")
    # and every pattern again inside rows of ordinary data (finite scales)
    g = torch.Generator(device="cpu").manual_seed(5)
    base = (torch.randn(256, 256, generator=g) * 3).to(torch.bfloat16).to(DEV)
    mixed = torch.cat([base, x], dim=1)
    fin = ~torch.isfinite(mixed.float())
    mixed[fin] = 0
    q, s = pkg.fp8_quant_per_token(mixed)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_rows_bf16(bits(mixed))
    assert np.array_equal(host(s).view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(host(q), q_ref)


def test_quotients_at_rounding_boundaries(oracle_mod):
    # per-head scales of the KV-cache write put fl32(x / s) within a few fp32
    # ulps of E4M3 rounding midpoints (normal and subnormal range) and of
    # exact grid values, on both sides
    grid = oracle_mod.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    mids = (grid[:-1] + grid[1:]) / 2
    targets = np.concatenate([mids, grid[1:]])
    rng = np.random.default_rng(11)
    H, D = 1024, 16
    xs = (rng.standard_normal((H, D)) * 4).astype(np.float32)
    xs = torch.tensor(xs).to(torch.bfloat16).float().numpy()
    xs[xs == 0] = 1.0
    scale = np.empty(H, dtype=np.float32)
    for h in range(H):
        tgt = targets[rng.integers(len(targets))] * (1 + rng.integers(-4, 5) * 2.0 ** -23)
        scale[h] = np.float32(abs(xs[h, 0]) / tgt)
    kv = torch.tensor(xs).to(torch.bfloat16).reshape(1, H, D).to(DEV)
    sc = torch.tensor(scale, device=DEV)
    cache = torch.zeros((1, H, D), dtype=torch.uint8, device=DEV)
    pkg.fp8_kv_cache_quant(kv, sc, cache)
    torch.cuda.synchronize()
    ref = oracle_mod.kv_cache_quant_bf16(bits(kv), scale, None, 1)
    assert np.array_equal(host(cache), ref)
    # the constructed quotients really sit at the boundaries
    quot = np.abs((xs[:, 0] / scale).astype(np.float32))
    near = np.min(np.abs(quot[:, None].astype(np.float64) - targets[None, :]) /
                  targets[None, :], axis=1)
    assert np.mean(near < 2.0 ** -20) > 0.9


@pytest.mark.parametrize("s_val", [1.0, 0.0123, 3.0e-5, 700.0])
def test_keys_and_values_every_bf16_pattern(oracle_mod, s_val):
    # the one-launch keys-and-values write over all 65536 bf16 patterns (the
    # values are the patterns in reverse order, with their own scale)
    pat = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    H, D = 8, 128
    T = 65536 // (H * D)
    k_bits = pat.reshape(T, H, D)
    v_bits = pat[::-1].copy().reshape(T, H, D)
    k = torch.from_numpy(k_bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    v = torch.from_numpy(v_bits.view(np.int16)).view(torch.bfloat16).to(DEV)
    ks = np.float32(s_val)
    vs = np.float32(s_val * 0.75)
    kc = torch.zeros((T, H, D), dtype=torch.uint8, device=DEV)
    vc = torch.zeros((T, H, D), dtype=torch.uint8, device=DEV)
    pkg.fp8_kv_cache_quant_kv(k, v, torch.tensor([ks], device=DEV), torch.tensor([vs], device=DEV),
                              kc, vc)
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    assert np.array_equal(host(kc), oracle_mod.kv_cache_quant_bf16(k_bits, ks, None, T))
    assert np.array_equal(host(vc), oracle_mod.kv_cache_quant_bf16(v_bits, vs, None, T))
