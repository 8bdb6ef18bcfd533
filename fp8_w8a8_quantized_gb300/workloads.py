"""Seeded synthetic inputs for the W8A8 linear layer.

This module only draws random bf16 activations X [M, K] and bf16 weights
W [N, K]; it holds none of the layer's arithmetic (no scales, no E4M3
rounding, no GEMM).  Both the CUDA path and the CPU oracle are fed from the
tensors it returns.  Every generator takes an explicit seed and device;
draws use ``torch.Generator`` on that device, so the same call on the same
machine always returns the same bits.

Workload recipes (layer shapes follow Llama-3.1-8B / 70B projections):

* ``tiny``: X [16, 256] ~ N(0, 1) with columns 3 and 77 scaled x50, plus two
  extra tokens -- the worked row [0.02, -0.5, 1.3, 7.9, -0.004, 3.1, 400]
  ("FP8 Inference Explained, in depth", "The numbers in one byte") and token
  A [0.01, -0.8, 3.2] ("Quantization: FP8 inference and KV-cache
  quantization", "Dynamic scales or static scales"), each zero-padded to
  K = 256 -- and W [256, 256] ~ N(0, 0.02^2).
* ``gaussian_outliers``: X ~ N(0, 1) with round(0.001 K) seeded channels x30
  (decode and 70B shapes).
* ``student_t_outliers``: X = t(nu=4) / sqrt(2) (unit rms) with 8 seeded
  channels x100 (prefill shapes).  t(4) is drawn as Z / sqrt(chi2_4 / 4).
* ``weights``: W ~ N(0, 1/K) (standard deviation 1/sqrt(K)).
* ``stress``: M = K = 4096 rows mixing log-uniform magnitudes over
  [2^-14, 2^12] with random signs, all-zero rows (with signed zeros), rows
  whose x / scale lands exactly on E4M3 midpoints, rows with one 1e4 outlier
  among N(0, 1), and sign-mixed rows packed near their maximum.
"""
from __future__ import annotations

import math

import torch

SHAPES_8B = (  # (name, K, N)
    ("qkv", 4096, 6144),
    ("o_proj", 4096, 4096),
    ("gate_up", 4096, 28672),
    ("down", 14336, 4096),
)
SHAPES_70B = (
    ("qkv", 8192, 10240),
    ("o_proj", 8192, 8192),
    ("gate_up", 8192, 57344),
    ("down", 28672, 8192),
)
DECODE_M = (1, 8, 32)
PREFILL_M = (2048, 8192)
M_70B = (32, 4096)

SEED_TINY, SEED_DECODE, SEED_PREFILL, SEED_70B, SEED_STRESS = 0, 1, 2, 3, 4

WORKED_ROW = (0.02, -0.5, 1.3, 7.9, -0.004, 3.1, 400.0)
TOKEN_A = (0.01, -0.8, 3.2)
TOKEN_B = (2.0, -45.0, 180.0)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def tiny(device="cpu"):
    """The 18 x 256 x 256 layer (seed 0).  Returns (X bf16 [18,256],
    W bf16 [256,256])."""
    g = _gen(SEED_TINY, device)
    x = torch.randn(16, 256, generator=g, device=device, dtype=torch.float32)
    x[:, 3] *= 50.0
    x[:, 77] *= 50.0
    extra = torch.zeros(2, 256, dtype=torch.float32)
    extra[0, : len(WORKED_ROW)] = torch.tensor(WORKED_ROW)
    extra[1, : len(TOKEN_A)] = torch.tensor(TOKEN_A)
    x = torch.cat([x, extra.to(device)], dim=0).to(torch.bfloat16)
    w = (torch.randn(256, 256, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return x, w


def outlier_channels(K: int, count: int, seed: int, device="cpu") -> torch.Tensor:
    """`count` distinct seeded column indices in [0, K)."""
    g = _gen(seed * 1000003 + K, "cpu")
    return torch.randperm(K, generator=g)[:count].to(device)


def gaussian_outliers(M: int, K: int, seed: int, device="cpu", frac=0.001, mult=30.0):
    """X ~ N(0,1) with round(frac*K) channels multiplied by `mult`."""
    g = _gen(seed * 7919 + M * 31 + K, device)
    x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    cols = outlier_channels(K, max(1, round(frac * K)), seed, device)
    x[:, cols] *= mult
    return x.to(torch.bfloat16)


def student_t_outliers(M: int, K: int, seed: int, device="cpu", n_out=8, mult=100.0):
    """X = t(4)/sqrt(2) (unit variance) with `n_out` channels x `mult`."""
    g = _gen(seed * 7919 + M * 31 + K, device)
    z = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros_like(z)
    for _ in range(4):
        e = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
        chi2.addcmul_(e, e)
    x = z / torch.sqrt(chi2 / 4.0) / math.sqrt(2.0)
    del chi2, z
    cols = outlier_channels(K, n_out, seed, device)
    x[:, cols] *= mult
    return x.to(torch.bfloat16)


def weights(N: int, K: int, seed: int, device="cpu"):
    """W ~ N(0, 1/K) in bf16, [N, K] (nn.Linear layout)."""
    g = _gen(seed * 104729 + N * 17 + K, device)
    w = torch.randn(N, K, generator=g, device=device, dtype=torch.float32)
    w.mul_(1.0 / math.sqrt(K))
    return w.to(torch.bfloat16)


def _e4m3_positive_grid() -> list:
    """The positive finite E4M3 values from the format's field layout
    (exponent bias 7, 3 mantissa bits, no infinities), used only to place
    inputs exactly on rounding midpoints."""
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append(m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return sorted(set(vals))


def stress(device="cpu", M=4096, K=4096):
    """Numerics stress activations (seed 4), [M, K] bf16, plus a per-row
    kind label (list of str)."""
    g = _gen(SEED_STRESS, "cpu")
    x = torch.empty(M, K, dtype=torch.float32)
    kinds = []
    grid = _e4m3_positive_grid()
    mids = torch.tensor([(a + b) / 2 for a, b in zip(grid[:-1], grid[1:])],
                        dtype=torch.float32)
    for r in range(M):
        sel = r % 8
        if sel < 4:                                   # 1/2 log-uniform
            u = torch.rand(K, generator=g) * 26.0 - 14.0
            sign = torch.where(torch.rand(K, generator=g) < 0.5, -1.0, 1.0)
            x[r] = sign * torch.exp2(u)
            kinds.append("loguniform")
        elif sel == 4:                                # all-zero, signed zeros
            sign = torch.where(torch.rand(K, generator=g) < 0.5, -1.0, 1.0)
            x[r] = sign * 0.0
            kinds.append("zero")
        elif sel == 5:                                # exact E4M3 midpoints
            j = int(torch.randint(-10, 11, (1,), generator=g))
            idx = torch.randint(0, len(mids), (K,), generator=g)
            sign = torch.where(torch.rand(K, generator=g) < 0.5, -1.0, 1.0)
            row = sign * mids[idx] * (2.0 ** j)
            pos = int(torch.randint(0, K, (1,), generator=g))
            row[pos] = 448.0 * (2.0 ** j)             # fixes the scale at 2^j
            x[r] = row
            kinds.append("ties")
        elif sel == 6:                                # one 1e4 outlier
            row = torch.randn(K, generator=g)
            row[int(torch.randint(0, K, (1,), generator=g))] = 1.0e4
            x[r] = row
            kinds.append("outlier")
        else:                                         # sign-mixed near max
            amax = float(torch.exp2(torch.rand(1, generator=g) * 16.0 - 8.0))
            mag = amax * (0.9 + 0.1 * torch.rand(K, generator=g))
            sign = torch.where(torch.rand(K, generator=g) < 0.5, -1.0, 1.0)
            row = sign * mag
            row[0], row[1] = amax, -amax
            x[r] = row
            kinds.append("saturation")
    return x.to(torch.bfloat16).to(device), kinds
