"""Pins for the oracle's per-tensor, static-scale and KV-cache quantization
(CPU only): the pages' static-scale and KV examples, reduction to the
already pinned per-row rule, and PyTorch's E4M3 cast as a witness."""
import numpy as np
import torch

from conftest import read_golden
from fp8_w8a8_quantized_gb300 import workloads


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16(vals):
    return torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)


def torch_codes(f32):
    return torch.tensor(np.asarray(f32, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_static_scale_tokens_a_b(oracle_mod):
    # "Dynamic scales or static scales": a calibrated s = 120/448 for both
    # tokens; A's 0.01 reads back as 0.0105, B's 180 clamps to 448 -> 120
    g = read_golden("dynamic_static_tokens.txt")
    s = np.float32(float(g["static_scale_num"])) / np.float32(448)
    row = bf16([[0.01, -0.8, 3.2, 2.0, -45.0, 180.0]])
    q = oracle_mod.quant_rows_scaled_bf16(bits(row), s)
    back = oracle_mod.e4m3_decode(q[0]) * np.float64(s)
    assert round(float(back[0]), 4) == float(g["A_0.01_static_readback_4dp"])
    assert q[0, 5] == 0x7E
    assert round(float(back[5]), 3) == float(g["B_180_static_readback"])
    # with its own dynamic scale, B's maximum reads back as 180 (to fp32 rounding of s)
    qd, sd = oracle_mod.quant_rows_bf16(bits(bf16([[2.0, -45.0, 180.0]])))
    assert qd[0, 2] == 0x7E
    assert round(float(oracle_mod.e4m3_decode([0x7E])[0] * sd[0]), 4) == 180.0


def test_scaled_rows_match_torch_witness(oracle_mod):
    x = workloads.gaussian_outliers(16, 512, seed=13)
    s = np.exp2(np.linspace(-6, 3, 16)).astype(np.float32)
    q = oracle_mod.quant_rows_scaled_bf16(bits(x), s)
    quot = (x.float().numpy() / s[:, None]).astype(np.float32)
    witness = torch_codes(np.clip(quot, -448, 448))
    assert np.array_equal(q, witness)


def test_per_tensor_equals_per_row_of_the_flattened_tensor(oracle_mod):
    x = workloads.gaussian_outliers(12, 256, seed=14)
    q, s = oracle_mod.quant_tensor_bf16(bits(x))
    q1, s1 = oracle_mod.quant_rows_bf16(bits(x).reshape(1, -1))
    assert s == s1[0]
    assert np.array_equal(q.reshape(1, -1), q1)
    amax = np.abs(x.float().numpy()).max()
    assert s == np.float32(amax) / np.float32(448)
    z = np.zeros((3, 32), dtype=np.uint16)
    qz, sz = oracle_mod.quant_tensor_bf16(z)
    assert sz == 1.0 and np.all(qz == 0)


def test_kv_cache_scale_one_and_clipping(oracle_mod):
    # "Turning it on in an engine": with scale 1.0, 0.001 rounds up to the
    # smallest subnormal 2^-9 and values beyond 448 are clipped
    g = read_golden("e4m3_format_facts.txt")
    x = bf16([[[0.001, -0.001, 500.0, -1000.0, 1.0, 0.0, 96.0, 95.0]]])
    cache = oracle_mod.kv_cache_quant_bf16(bits(x), 1.0, None, 1)
    c = cache[0, 0]
    assert oracle_mod.e4m3_decode([c[0]])[0] == 2.0 ** int(g["kv_scale1_0.001_rounds_to_log2"])
    assert c[1] == 0x81
    assert c[2] == 0x7E and c[3] == 0xFE
    assert c[4] == 0x38 and c[5] == 0x00
    assert c[6] == int(g["bits_96"], 2) and c[7] == int(g["bits_96"], 2)


def test_kv_cache_per_head_scales_and_slots(oracle_mod):
    T, H, D = 6, 4, 64
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(T, H, D, generator=g) * 4).to(torch.bfloat16)
    scale = np.array([0.5, 1.0, 2.0, 0.125], dtype=np.float32)
    slots = np.array([7, -1, 0, 3, 9, 10], dtype=np.int64)  # 10 is past the cache
    cache = oracle_mod.kv_cache_quant_bf16(bits(x), scale, slots, 10)
    for t in range(T):
        if slots[t] < 0 or slots[t] >= 10:
            continue
        for h in range(H):
            ref = oracle_mod.quant_rows_scaled_bf16(bits(x[t, h][None]), scale[h])[0]
            assert np.array_equal(cache[slots[t], h], ref)
    untouched = [r for r in range(10) if r not in set(slots.tolist())]
    assert np.all(cache[untouched] == 0)
