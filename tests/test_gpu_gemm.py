"""GPU parity of the scaled FP8 GEMM (both kernels: the weight-streaming
split-K kernel for M <= 256, token tiles of 16 to 256, and the paired-SM
256 x 256 tile kernel above, partial row and column tiles included), fed
with the oracle's own codes and scales, against the oracle's fp64 result."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from parity import check_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_gemm(qx, s_tok, qw, s_w):
    y = pkg.fp8_scaled_gemm(dev(qx), dev(s_tok), dev(qw), dev(s_w))
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    return y.double().cpu().numpy()


def random_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    qx = rng.choice(FINITE, size=(M, K))
    qw = rng.choice(FINITE, size=(N, K))
    s_tok = np.exp2(rng.uniform(-12, 4, M)).astype(np.float32)
    s_w = np.exp2(rng.uniform(-12, 0, N)).astype(np.float32)
    return qx, s_tok, qw, s_w


SHAPES = [  # (M, N, K): ragged edges, single k-block, many k-blocks, both kernels
    (1, 8, 16), (1, 128, 128), (3, 24, 48), (16, 256, 256), (17, 100, 272), (32, 264, 1024),
    (33, 1000, 4096), (64, 384, 2048), (65, 256, 256), (128, 256, 128), (129, 520, 1040),
    (200, 300, 4112), (256, 512, 4096), (300, 1000, 1024), (513, 777, 2064),
    (256, 256, 128), (257, 264, 256), (1000, 4100, 512), (2048, 520, 272), (384, 128, 8192),
    # degenerate edges: one output column, the smallest K, one partial k-block
    (5, 1, 32), (200, 3, 128), (300, 1, 64), (300, 520, 16), (512, 768, 48), (200, 300, 16),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_random_codes(oracle_mod, M, N, K):
    qx, s_tok, qw, s_w = random_operands(M, N, K, M * 1000 + N + K)
    y = run_gemm(qx, s_tok, qw, s_w)
    ref = oracle_mod.scaled_gemm(qx, s_tok, qw, s_w)
    check_rows(y, ref, f"gemm {M}x{N}x{K}")


# The persistent paired-SM kernel walking more than one output tile per CTA
# pair (at most 76 pairs of 256 x 256 tiles): the second TMEM accumulator
# buffer, its phase flips and the tile walk; rows of a tile past M are
# zero-filled by TMA and never stored, nor are columns past N.  And the weight-streaming kernel with
# wide token tiles over many weight slabs.  Full outputs against the oracle.
MULTI_TILE = [
    (200, 28672, 1024),   # 256-token tiles, 224 slabs
    (255, 49152, 256),    # 256-token tiles, 384 slabs, two k-blocks (no K split)
    (80, 24576, 512),     # 128-token tiles, 48 of 128 token columns empty
    (8, 57344, 1024),     # 448 slabs, unsplit, 16-token tiles (pushed to themselves)
    (1024, 8192, 1024),   # paired: 4 x 32 = 128 tiles, up to 2 per pair
    (1536, 8192, 256),    # paired: 6 x 32 = 192 tiles, up to 3 per pair
    (2304, 4864, 272),    # paired: 9 x 19 = 171 tiles, ragged K
    (2048, 16384, 272),   # paired: 8 x 64 = 512 tiles, up to 7 per pair, ragged K
    (1800, 12296, 144),   # paired: 8 rows in the last row tile, 8 columns in the last
    (1032, 20812, 256),   # paired: 5 x 82 tiles, last column tile 76 wide (not 8-aligned)
]


@pytest.mark.parametrize("M,N,K", MULTI_TILE)
def test_multi_tile_persistent(oracle_mod, M, N, K):
    qx, s_tok, qw, s_w = random_operands(M, N, K, M + 7 * N + K)
    y = run_gemm(qx, s_tok, qw, s_w)
    ref = oracle_mod.scaled_gemm(qx, s_tok, qw, s_w)
    check_rows(y, ref, f"multi-tile gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 8, 32, 64, 128, 1024])
def test_all_positive_long_k_accumulation(oracle_mod, M):
    # all products positive and large: exposes any loss of accumulator bits
    # at the longest K the layers use (fp32 accumulation keeps 24 bits)
    K, N = 28672, 256
    rng = np.random.default_rng(M)
    qx = rng.integers(0x70, 0x7F, size=(M, K), dtype=np.uint8)
    qw = rng.integers(0x30, 0x40, size=(N, K), dtype=np.uint8)
    s_tok = np.full(M, 1e-3, dtype=np.float32)
    s_w = np.full(N, 1e-4, dtype=np.float32)
    y = run_gemm(qx, s_tok, qw, s_w)
    ref = oracle_mod.scaled_gemm(qx, s_tok, qw, s_w)
    rel = np.max(np.abs(y - ref) / np.abs(ref))
    assert rel < 4e-3, rel


def test_identity_like_columns(oracle_mod):
    # W rows are one-hot (code 1.0 at column n % K): y picks one x value per n,
    # so any row/column/k mix-up in tiling shows as a wrong exact value
    M, N, K = 130, 300, 512
    rng = np.random.default_rng(5)
    qx = rng.choice(FINITE, size=(M, K))
    qw = np.zeros((N, K), dtype=np.uint8)
    qw[np.arange(N), np.arange(N) % K] = 0x38
    s_tok = np.ones(M, dtype=np.float32)
    s_w = np.ones(N, dtype=np.float32)
    for m_sub in (M, 7):
        y = run_gemm(qx[:m_sub], s_tok[:m_sub], qw, s_w)
        ref = oracle_mod.scaled_gemm(qx[:m_sub], s_tok[:m_sub], qw, s_w)
        # every output is a single e4m3 value: exact in bf16
        assert np.array_equal(y, ref), m_sub


def test_deterministic_bits():
    qx, s_tok, qw, s_w = random_operands(32, 4096, 4096, 1)
    assert np.array_equal(run_gemm(qx, s_tok, qw, s_w), run_gemm(qx, s_tok, qw, s_w))
    qx, s_tok, qw, s_w = random_operands(300, 1024, 4096, 2)
    assert np.array_equal(run_gemm(qx, s_tok, qw, s_w), run_gemm(qx, s_tok, qw, s_w))


@pytest.mark.parametrize("M", [5, 200])
def test_output_guard_bands(oracle_mod, M):
    N, K = 136, 256
    qx, s_tok, qw, s_w = random_operands(M, N, K, 77)
    pad = 64
    buf = torch.full((pad + M * N + pad,), -12288.0, dtype=torch.bfloat16, device=DEV)
    y = buf[pad:pad + M * N]
    a, b, c, d = dev(qx), dev(s_tok), dev(qw), dev(s_w)
    st = pkg.lib().fp8_scaled_gemm(a.data_ptr(), b.data_ptr(), c.data_ptr(), d.data_ptr(),
                                   y.data_ptr(), M, N, K, None, 0,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    bb = buf.float().cpu().numpy()
    assert np.all(bb[:pad] == -12288.0) and np.all(bb[pad + M * N:] == -12288.0)
    check_rows(y.view(M, N).double().cpu().numpy(),
               oracle_mod.scaled_gemm(qx, s_tok, qw, s_w), "guarded")


def test_empty_and_rejected_calls():
    L = pkg.lib()
    x = torch.zeros(64, 64, dtype=torch.uint8, device=DEV)
    f = torch.ones(64, dtype=torch.float32, device=DEV)
    y = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.current_stream().cuda_stream
    assert L.fp8_scaled_gemm(x.data_ptr(), f.data_ptr(), x.data_ptr(), f.data_ptr(),
                             y.data_ptr(), 0, 64, 64, None, 0, s) == 0
    assert L.fp8_scaled_gemm(x.data_ptr(), f.data_ptr(), x.data_ptr(), f.data_ptr(),
                             y.data_ptr() + 2, 4, 4, 64, None, 0, s) == 2
    torch.cuda.synchronize()
    assert torch.all(y == 0)


# Codes whose values lie in [1, 2) (E4M3 exponent field 7, either sign):
# every product is a multiple of 2^-6 below 4, so for K <= 2048 every partial
# sum is exactly representable in fp32, whatever order and split the kernel
# adds in.  The GPU's fp32 accumulator then equals the oracle's exact sum, and
# the output must equal bf16_rn(fl32(fl32(acc * s_tok[m]) * s_w[n])) bit for
# bit: this pins the epilogue (its multiplication order and the round to
# nearest even into bf16) on all three GEMM kernels, beyond the tolerance.
# Codes whose values make every fp32 partial sum exact, in any order and any
# split of K: +-1 alone (integer sums, at most K), and all codes with values
# in [1, 2) (products are multiples of 2^-6 below 4, so sums of up to 2048 of
# them need at most 19 significant bits).  With the accumulator fixed, the
# epilogue's fp32 products and bf16 rounding are compared bit for bit.
EXACT_CODE_SETS = {
    "unit": np.array([0x38, 0xB8], dtype=np.uint8),
    "one_to_two": np.array([c | s for c in range(0x38, 0x40) for s in (0x00, 0x80)],
                           dtype=np.uint8),
}


@pytest.mark.parametrize("codes", sorted(EXACT_CODE_SETS))
@pytest.mark.parametrize("M,N,K", [(1, 256, 1024), (8, 520, 512), (32, 384, 2048),
                                   (64, 1000, 1040), (100, 300, 1024), (200, 28672, 256),
                                   (300, 520, 1024), (1024, 8192, 512)])
def test_epilogue_bits_with_exact_sums(oracle_mod, codes, M, N, K):
    rng = np.random.default_rng(M * 7 + N + K)
    qx = rng.choice(EXACT_CODE_SETS[codes], size=(M, K))
    qw = rng.choice(EXACT_CODE_SETS[codes], size=(N, K))
    s_tok = np.exp2(rng.uniform(-12, 4, M)).astype(np.float32)
    s_w = np.exp2(rng.uniform(-12, 0, N)).astype(np.float32)
    y = pkg.fp8_scaled_gemm(dev(qx), dev(s_tok), dev(qw), dev(s_w))
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    acc = oracle_mod.gemm_exact(qx, qw)                       # exact, scaled by 2^18
    acc32 = (acc.astype(np.float64) * 2.0 ** -18).astype(np.float32)
    assert np.array_equal(acc32.astype(np.float64) * 2.0 ** 18, acc.astype(np.float64))
    t = (acc32 * s_tok[:, None]) * s_w[None, :]              # fp32 products, in order
    expect = torch.from_numpy(t.astype(np.float32)).to(torch.bfloat16).float()
    got = y.cpu().float()                                     # exact widening
    # value equality: bitwise except that +0 and -0 of a zero sum are equal
    diff = (got != expect).nonzero()
    assert diff.numel() == 0, (
        f"{codes} {M}x{N}x{K}: {diff.shape[0]} outputs differ, first at {diff[0].tolist()}: "
        f"got {got[tuple(diff[0])].item()!r}, expected {expect[tuple(diff[0])].item()!r}")
