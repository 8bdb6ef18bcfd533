"""Pins for the oracle's dynamic per-row quantization (CPU only).

The worked examples the pages print (tests/golden/*.txt), invariants of the
method (the row maximum lands on +-448, all-zero rows get scale 1), and
independent witnesses (numpy's IEEE fp32 division, PyTorch's E4M3 cast).
"""
import numpy as np
import torch

from conftest import read_golden
from fp8_w8a8_quantized_gb300 import workloads


def floats(s):
    return [float(t) for t in s.split()]


def bf16_bits(x_f32):
    t = torch.tensor(np.asarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def dequant(oracle_mod, q, s):
    return oracle_mod.e4m3_decode(q) * np.float64(s)


def test_worked_row_fp32(oracle_mod):
    g = read_golden("worked_row_fake_quant.txt")
    row = np.array([floats(g["input"])], dtype=np.float32)
    q, s = oracle_mod.quant_rows_f32(row)
    assert s[0] == np.float32(400.0) / np.float32(448.0)
    got = np.round(dequant(oracle_mod, q[0], s[0]), 4)
    assert list(got) == floats(g["dequantized_4dp"])


def test_worked_row_as_bf16_token(oracle_mod):
    # the same row entered as a bf16 token still prints the same 4 digits
    g = read_golden("worked_row_fake_quant.txt")
    row = np.zeros((1, 256), dtype=np.float32)
    vals = floats(g["input"])
    row[0, : len(vals)] = vals
    q, s = oracle_mod.quant_rows_bf16(bf16_bits(row))
    got = np.round(dequant(oracle_mod, q[0, : len(vals)], s[0]), 4)
    assert list(got) == floats(g["dequantized_4dp"])
    assert np.all(q[0, len(vals):] == 0)


def test_dynamic_tokens_A_B(oracle_mod):
    g = read_golden("dynamic_static_tokens.txt")
    a = np.array([floats(g["token_A"])], dtype=np.float32)
    b = np.array([floats(g["token_B"])], dtype=np.float32)
    qa, sa = oracle_mod.quant_rows_f32(a)
    qb, sb = oracle_mod.quant_rows_f32(b)
    assert round(float(sa[0]), 5) == float(g["scale_A_approx_5dp"])
    assert round(float(sb[0]), 3) == float(g["scale_B_approx_3dp"])
    assert sa[0] == np.float32(3.2) / np.float32(448)
    # each token's maximum lands exactly on 448
    assert qa[0, 2] == 0x7E and qb[0, 2] == 0x7E
    assert dequant(oracle_mod, qa[0, 2], sa[0]) == np.float64(sa[0]) * 448.0
    assert round(float(dequant(oracle_mod, qa[0, 0], sa[0])), 4) == float(
        g["A_0.01_dynamic_readback_4dp"])


def test_static_scale_saturation(oracle_mod):
    # a fixed calibrated scale s = 120/448: small values keep relative
    # precision, values beyond 448 s clamp to 448 (saturating mode)
    g = read_golden("dynamic_static_tokens.txt")
    s = np.float32(float(g["static_scale_num"])) / np.float32(448)
    assert round(float(s), 3) == float(g["static_scale_approx_3dp"])
    q001 = oracle_mod.e4m3_encode([float(np.float32(0.01) / s)])[0]
    r001 = float(oracle_mod.e4m3_decode([q001])[0] * np.float64(s))
    assert round(r001, 4) == float(g["A_0.01_static_readback_4dp"])
    assert round(abs(r001 - 0.01) / 0.01 * 100, 1) == float(
        g["A_0.01_static_relerr_pct_1dp"])
    quot = np.float32(180.0) / s
    assert round(float(quot)) == int(g["B_180_static_quotient"])
    q180 = oracle_mod.e4m3_encode([float(quot)])[0]
    assert q180 == 0x7E
    assert round(float(oracle_mod.e4m3_decode([q180])[0] * np.float64(s)), 3) == float(
        g["B_180_static_readback"])


def test_row_max_lands_on_448_and_zero_rows(oracle_mod):
    x, kinds = workloads.stress(M=64, K=512)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle_mod.quant_rows_bf16(bits)
    xf = x.float().numpy()
    for r in range(x.shape[0]):
        amax = np.max(np.abs(xf[r]))
        if amax == 0:
            assert s[r] == 1.0
            signs = np.signbit(xf[r])
            assert np.all(q[r] == np.where(signs, 0x80, 0x00))
        else:
            assert s[r] == np.float32(amax) / np.float32(448)
            k = int(np.argmax(np.abs(xf[r])))
            assert q[r, k] == (0xFE if xf[r, k] < 0 else 0x7E)
            # no code exceeds the maximum magnitude
            assert np.all((q[r] & 0x7F) <= 0x7E)


def test_tie_rows_round_half_to_even(oracle_mod):
    x, kinds = workloads.stress(M=48, K=256)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle_mod.quant_rows_bf16(bits)
    xf = x.float().numpy()
    n_ties = 0
    for r, kind in enumerate(kinds):
        if kind != "ties":
            continue
        n_ties += 1
        # the scale is an exact power of two, so x / s is the exact midpoint
        assert float(s[r]) == 2.0 ** round(np.log2(float(s[r])))
        quot = (xf[r] / s[r]).astype(np.float32)
        witness = torch.tensor(quot).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q[r], witness)
        # every quotient is a midpoint (or 448 itself): all codes are even
        assert np.all((q[r] & 1) == 0)
    assert n_ties > 0


def test_division_not_reciprocal(oracle_mod):
    """The reading: divide each value by s = amax/448 in IEEE fp32.  Rows
    exist where multiplying by fl32(448/amax) instead gives another code; on
    those the oracle must follow the division."""
    rng = np.random.default_rng(99)
    grid = oracle_mod.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2
    found = 0
    for _ in range(4000):
        t = float(mids[rng.integers(8, len(mids) - 1)])
        s = np.float32(rng.integers(1 << 18, 1 << 19) * 2.0 ** -19)  # 19-bit
        amax = np.float32(448.0) * s
        x = np.float32(t) * s
        if float(x) != t * float(s) or amax / np.float32(448) != s:
            continue
        recip = np.float32(448.0) / amax
        q_div = np.float32(x) / s
        q_mul = np.float32(x) * recip
        c_div = torch.tensor([q_div]).to(torch.float8_e4m3fn).view(torch.uint8).item()
        c_mul = torch.tensor([q_mul]).to(torch.float8_e4m3fn).view(torch.uint8).item()
        if c_div == c_mul:
            continue
        row = np.array([[x, amax]], dtype=np.float32)
        q, srow = oracle_mod.quant_rows_f32(row)
        assert srow[0] == s
        assert q[0, 0] == c_div and q[0, 0] != c_mul
        found += 1
        if found >= 5:
            break
    assert found >= 1


def test_quant_matches_torch_witness_on_random_rows(oracle_mod):
    x = workloads.gaussian_outliers(32, 1024, seed=11)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = oracle_mod.quant_rows_bf16(bits)
    xf = x.float().numpy()
    amax = np.max(np.abs(xf), axis=1).astype(np.float32)
    s_ref = np.where(amax > 0, amax / np.float32(448), np.float32(1)).astype(np.float32)
    assert np.array_equal(s, s_ref)
    quot = (xf / s_ref[:, None]).astype(np.float32)      # numpy IEEE division
    witness = torch.tensor(quot).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, witness)
