"""Pins for the oracle's RMSNorm feeding the per-token quantizer (CPU only):
torch's float64 rms_norm as an independent witness of the formula, closed
forms, the fp32 step sequence against the real values, and the bracket's
soundness (monotone in the sum of squares, narrow)."""
import numpy as np
import torch

from fp8_w8a8_quantized_gb300 import workloads


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def to_f(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).float().numpy()


def gamma(K, seed):
    g = torch.Generator().manual_seed(seed)
    return (1.0 + 0.2 * torch.randn(K, generator=g)).to(torch.bfloat16)


def test_formula_against_torch_rms_norm(oracle_mod):
    x = workloads.student_t_outliers(9, 384, seed=41)
    g = gamma(384, 42)
    for eps in (1e-6, 1e-5, 0.5):
        y = oracle_mod.rmsnorm_f64(bits(x), bits(g), eps)
        ref = torch.nn.functional.rms_norm(x.double(), (384,), g.double(), eps).numpy()
        assert np.allclose(y, ref, rtol=1e-12, atol=0), eps


def test_closed_forms(oracle_mod):
    K = 256
    ones = torch.ones(K, dtype=torch.bfloat16)
    for c in (0.25, 2.0, -8.0):
        x = torch.full((1, K), c, dtype=torch.bfloat16)
        y_lo, y_hi, ss = oracle_mod.rmsnorm_bracket_bf16(bits(x), bits(ones), 0.0, 2.0 ** -17)
        assert ss[0] == K * c * c
        assert np.all(to_f(y_lo) == np.sign(c)) and np.all(to_f(y_hi) == np.sign(c))
    # with eps: y = c / sqrt(c^2 + eps) (a bf16 of it), gamma scales it
    x = torch.full((1, K), 3.0, dtype=torch.bfloat16)
    g = torch.full((K,), 0.5, dtype=torch.bfloat16)
    y = oracle_mod.rmsnorm_f64(bits(x), bits(g), 7.0)
    assert np.allclose(y, 0.5 * 3.0 / 4.0, rtol=1e-15)


def test_fp32_steps_match_the_real_values(oracle_mod):
    x = workloads.gaussian_outliers(64, 4096, seed=43)
    g = gamma(4096, 44)
    # with no error budget the bracket is the two fp32 neighbours of the
    # exact sum of squares: almost every element is determined
    y_lo, y_hi, _ = oracle_mod.rmsnorm_bracket_bf16(bits(x), bits(g), 1e-5, 0.0)
    assert np.mean(y_lo != y_hi) < 1e-3
    real = oracle_mod.rmsnorm_f64(bits(x), bits(g), 1e-5)
    rounded = to_f(bits(torch.tensor(real, dtype=torch.float32).to(torch.bfloat16)))
    got = to_f(y_lo)
    # away from bf16 rounding boundaries the fp32 steps give the real value's bf16
    mant, _ = np.frexp(np.abs(real))              # |real| = mant 2^e, mant in [0.5, 1)
    frac = (mant * 256.0) % 1.0                   # position between bf16 neighbours
    far = (np.abs(frac - 0.5) > 2.0 ** -10) & (real != 0) & (y_lo == y_hi)
    assert np.array_equal(got[far], rounded[far])
    assert np.mean(got == rounded) > 0.999


def test_bracket_is_ordered_and_narrow(oracle_mod):
    x = workloads.student_t_outliers(128, 4096, seed=45)
    g = gamma(4096, 46)
    y_lo, y_hi, _ = oracle_mod.rmsnorm_bracket_bf16(bits(x), bits(g), 1e-6, 2.0 ** -17)
    lo, hi = to_f(y_lo), to_f(y_hi)
    assert np.all(np.abs(lo) <= np.abs(hi))
    assert np.all(np.sign(lo) * np.sign(hi) >= 0)
    assert np.mean(lo != hi) < 0.01
    # a wider uncertainty widens the bracket
    w_lo, w_hi, _ = oracle_mod.rmsnorm_bracket_bf16(bits(x), bits(g), 1e-6, 2.0 ** -10)
    assert np.mean(to_f(w_lo) != to_f(w_hi)) > np.mean(lo != hi)
    assert np.all(np.abs(to_f(w_lo)) <= np.abs(lo)) and np.all(np.abs(hi) <= np.abs(to_f(w_hi)))
