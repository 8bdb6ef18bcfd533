"""GPU parity of the whole W8A8 layer (fp8_linear) on every configuration:
quantized activation bytes and scales bit-exact (read back from the
workspace), weight codes and scales bit-exact, outputs within tolerance.
Small shapes, every decode batch and the mid-size batches of the smaller
layers are compared in full; the prefill shapes on full output rows of one
token from every 128-row block (so every row tile of the persistent kernel
is checked), with the same launch configuration the benchmark times."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from fp8_w8a8_quantized_gb300 import workloads
from parity import bits, check_rows, host, sample_rows, tile_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def layer(oracle_mod, x, w, rows=None, check_weight_rows=None):
    """Run the layer on the GPU; compare with the oracle on `rows` tokens."""
    M, K = x.shape
    N = w.shape[0]
    wq, s_w = pkg.fp8_quant_per_channel_weights(w)
    ws = torch.empty(pkg.fp8_linear_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    y = pkg.fp8_linear(x, wq, s_w, workspace=ws)
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    rows = np.arange(M) if rows is None else rows
    wrows = np.arange(N) if check_weight_rows is None else check_weight_rows
    qw_ref, sw_ref = oracle_mod.quant_rows_bf16(bits(w))
    qw_g, sw_g = host(wq), host(s_w)
    assert np.array_equal(sw_g, sw_ref), "weight scales"
    assert np.array_equal(qw_g[wrows], qw_ref[wrows]), "weight codes"
    # activations: the workspace holds xq [M, K] then s_tok [M]
    off = (M * K + 255) // 256 * 256
    xq_g = host(ws[: M * K].view(M, K))
    st_g = host(ws[off: off + 4 * M].view(torch.float32))
    qx_ref, st_ref = oracle_mod.quant_rows_bf16(bits(x))
    assert np.array_equal(st_g, st_ref), "token scales"
    assert np.array_equal(xq_g, qx_ref), "activation codes"
    y_ref = oracle_mod.scaled_gemm(qx_ref[rows], st_ref[rows], qw_ref, sw_ref)
    check_rows(y[torch.from_numpy(rows).to(DEV)].double().cpu().numpy(), y_ref,
               f"linear {M}x{N}x{K}")
    return y


def test_tiny_config(oracle_mod):
    x, w = workloads.tiny(DEV)
    layer(oracle_mod, x, w)


@pytest.mark.parametrize("M", workloads.DECODE_M)
@pytest.mark.parametrize("name,K,N", workloads.SHAPES_8B)
def test_decode_8b(oracle_mod, M, name, K, N):
    x = workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, DEV)
    w = workloads.weights(N, K, workloads.SEED_DECODE, DEV)
    layer(oracle_mod, x, w)


# Batches between the decode and prefill configurations (serving batches of
# 64-256 sequences, chunked prefill): the weight-streaming kernel with 128-
# and 256-token tiles (two CTAs, or one, per SM).  Every output row where
# the oracle's exact sums stay within a few seconds, else one token from
# every 16 (and the first and last); activation and weight codes in full.
@pytest.mark.parametrize("M", [65, 128, 129, 256])
@pytest.mark.parametrize("name,K,N", workloads.SHAPES_8B)
def test_mid_batch_8b(oracle_mod, M, name, K, N):
    x = workloads.gaussian_outliers(M, K, workloads.SEED_DECODE + M, DEV)
    w = workloads.weights(N, K, workloads.SEED_DECODE, DEV)
    rows = None if M * N * K <= 16 * 10 ** 9 else tile_rows(M, M + N, block=16)
    layer(oracle_mod, x, w, rows=rows)


@pytest.mark.parametrize("M", workloads.PREFILL_M)
@pytest.mark.parametrize("name,K,N", workloads.SHAPES_8B)
def test_prefill_8b(oracle_mod, M, name, K, N):
    x = workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, DEV)
    w = workloads.weights(N, K, workloads.SEED_DECODE, DEV)
    layer(oracle_mod, x, w, rows=tile_rows(M, M + N))


@pytest.mark.parametrize("M", workloads.M_70B)
@pytest.mark.parametrize("name,K,N", workloads.SHAPES_70B)
def test_llama70b(oracle_mod, M, name, K, N):
    x = workloads.gaussian_outliers(M, K, workloads.SEED_70B, DEV)
    w = workloads.weights(N, K, workloads.SEED_70B, DEV)
    # every token of the decode batch; one token of every 128-row block of
    # the prefill batch (both halves of every 256-row tile); all weight rows
    rows = None if M <= 64 else tile_rows(M, M + N)
    layer(oracle_mod, x, w, rows=rows)


def test_stress_config(oracle_mod):
    x, kinds = workloads.stress(DEV)
    w = workloads.weights(4096, 4096, workloads.SEED_STRESS, DEV)
    # every row kind is represented among the checked output rows
    rows = np.unique(np.concatenate([np.arange(64), sample_rows(4096, 64, 4)]))
    layer(oracle_mod, x, w, rows=rows)


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (7, 40, 48), (65, 264, 272), (300, 100, 1040)])
def test_ragged_layers(oracle_mod, M, N, K):
    x = workloads.gaussian_outliers(M, K, 21, DEV)
    w = workloads.weights(N, K, 21, DEV)
    layer(oracle_mod, x, w)


# Decode batches (M <= 32): one token, token counts around the tile
# boundaries (16/17, 32), K that is not a multiple of the 128-deep k-block,
# ragged N, and shapes from one to eight K-splits.
@pytest.mark.parametrize("M", [1, 2, 3, 5, 15, 16, 17, 24, 31, 32])
@pytest.mark.parametrize("N,K", [(392, 1040), (256, 4096), (1000, 2064), (6144, 144)])
def test_decode_batch_shapes(oracle_mod, M, N, K):
    x = workloads.gaussian_outliers(M, K, 41 + M, DEV)
    w = workloads.weights(N, K, 41, DEV)
    layer(oracle_mod, x, w)


# One token with long rows: 32 to 64 k-blocks per CTA at eight K-splits,
# with and without a ragged last k-block.
@pytest.mark.parametrize("K", [4096, 28672, 32768, 32784, 65536])
def test_single_token_long_rows(oracle_mod, K):
    x = workloads.gaussian_outliers(1, K, 43, DEV)
    w = workloads.weights(256, K, 43, DEV)
    layer(oracle_mod, x, w)


# The stress rows (log-uniform magnitudes, all-zero rows with signed zeros,
# exact E4M3 ties, a single 1e4 outlier, sign-mixed rows near their maximum)
# at decode batch sizes, where the per-token scales are found inside the GEMM.
@pytest.mark.parametrize("M", [1, 8, 16, 32])
def test_decode_stress_rows(oracle_mod, M):
    x, kinds = workloads.stress(DEV, M=64, K=4096)
    # round robin over the row kinds, an all-zero row first
    by_kind = {}
    for r, k in enumerate(kinds):
        by_kind.setdefault(k, []).append(r)
    names = ["zero"] + sorted(k for k in by_kind if k != "zero")
    order = [by_kind[k][i] for i in range(64) for k in names if i < len(by_kind[k])]
    xs = x[torch.tensor(order[:M], device=DEV)].contiguous()
    w = workloads.weights(1024, 4096, workloads.SEED_STRESS, DEV)
    layer(oracle_mod, xs, w)


def test_decode_repeatable(oracle_mod):
    """Two calls on the same inputs give the same bits (fixed reduction order)."""
    for M in (4, 24):
        x = workloads.gaussian_outliers(M, 4096, 5, DEV)
        w = workloads.weights(2048, 4096, 5, DEV)
        wq, s_w = pkg.fp8_quant_per_channel_weights(w)
        ws = torch.empty(pkg.fp8_linear_workspace_size(M, 2048, 4096), dtype=torch.uint8,
                         device=DEV)
        y1 = pkg.fp8_linear(x, wq, s_w, workspace=ws)
        y2 = pkg.fp8_linear(x, wq, s_w, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2)


def test_quantized_linear_module(oracle_mod):
    x = workloads.gaussian_outliers(8, 1024, 31, DEV)
    w = workloads.weights(512, 1024, 31, DEV)
    lin = pkg.QuantizedLinear(w)
    y1 = lin(x)
    y2 = lin(x)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    qw_ref, sw_ref = oracle_mod.quant_rows_bf16(bits(w))
    y_ref, _, _ = oracle_mod.linear(bits(x), qw_ref, sw_ref)
    check_rows(y1.double().cpu().numpy(), y_ref, "module")


def test_workspace_too_small_is_rejected():
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device=DEV)
    w = torch.zeros(8, 64, dtype=torch.uint8, device=DEV)
    s = torch.ones(8, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(pkg.Fp8Error) as e:
        pkg.fp8_linear(x, w, s, workspace=ws)
    assert e.value.status == 3
