"""GPU parity of the block-wise scales: 1 x 128 activation groups and
128 x 128 weight blocks must equal the CPU oracle's codes and scales bit for
bit; the block-scaled GEMM (decode and prefill kernels) and the whole
block-scaled layer must stay within the output tolerance of the fp64 oracle."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from fp8_w8a8_quantized_gb300 import workloads
from parity import bits, check_rows, host, sample_rows, tile_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def assert_bytes(gpu, ref, what):
    g = host(gpu)
    diff = np.argwhere(g != ref)
    assert diff.size == 0, f"{what}: {len(diff)} bytes differ, first at {tuple(diff[0])}: " \
        f"gpu={g[tuple(diff[0])]:#x} ref={ref[tuple(diff[0])]:#x}"


def assert_scales(gpu, ref, what):
    g = host(gpu)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    bad = np.argwhere(g.view(np.uint32) != ref.view(np.uint32))
    assert bad.size == 0, f"{what}: {len(bad)} scales differ, first at {tuple(bad[0])}"


def blocky(x: torch.Tensor, seed: int, rows: bool) -> torch.Tensor:
    """Scale 128-wide column blocks (and, for weights, 128-row blocks) of x by
    factors spread over 2^-6 .. 2^6, so every block gets a different scale."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    R, K = x.shape
    kb = -(-K // 128)
    f = torch.exp2(torch.randint(-6, 7, (kb,), generator=g).float())
    fk = f.repeat_interleave(128)[:K].to(x.device)
    out = x.float() * fk
    if rows:
        nb = -(-R // 128)
        fr = torch.exp2(torch.randint(-3, 4, (nb,), generator=g).float())
        out = out * fr.repeat_interleave(128)[:R].to(x.device)[:, None]
    return out.to(torch.bfloat16)


# ------------------------------------------------------------ quantizers

@pytest.mark.parametrize("M,K", [(1, 4096), (8, 4096), (32, 14336), (2048, 4096),
                                 (3, 16), (5, 272), (33, 1040), (130, 4112)])
def test_groups(oracle_mod, M, K):
    x = blocky(workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, DEV), M + K, False)
    q, s = pkg.fp8_quant_per_token_group(x)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_groups_bf16(bits(x))
    assert_scales(s, s_ref, "group scales")
    assert_bytes(q, q_ref, "group codes")


def test_groups_stress_and_strided(oracle_mod):
    x, _ = workloads.stress(DEV, M=512, K=4096)
    q, s = pkg.fp8_quant_per_token_group(x)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_groups_bf16(bits(x))
    assert_scales(s, s_ref, "stress scales")
    assert_bytes(q, q_ref, "stress codes")
    M, K, ldx, ldq = 37, 400, 520, 432
    base = workloads.gaussian_outliers(M, ldx, 9, DEV)
    xs = base[:, :K]
    xq = torch.full((M, ldq), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.empty((M, 4), dtype=torch.float32, device=DEV)
    st = pkg.lib().fp8_quant_per_token_group(xs.data_ptr(), M, K, ldx, xq.data_ptr(), ldq,
                                             s.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_groups_bf16(bits(xs))
    assert_bytes(xq[:, :K], q_ref, "strided codes")
    assert np.all(host(xq)[:, K:] == 0xAB), "wrote past K"
    assert_scales(s, s_ref, "strided scales")


@pytest.mark.parametrize("N,K", [(4096, 4096), (6144, 4096), (4096, 14336), (200, 272),
                                 (130, 16), (1, 1040)])
def test_weight_blocks(oracle_mod, N, K):
    w = blocky(workloads.weights(N, K, workloads.SEED_DECODE, DEV), N * 3 + K, True)
    if N >= 200:
        w[128:256, 128:256] = 0          # one all-zero block
    q, s = pkg.fp8_quant_weight_blocks(w)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_weight_blocks_bf16(bits(w))
    assert_scales(s, s_ref, "block scales")
    assert_bytes(q, q_ref, "block codes")
    if N >= 200:
        assert host(s)[1, 1] == 1.0


# ------------------------------------------------------------ GEMM

def make_layer(M, N, K, seed, prefill=False):
    gen = workloads.student_t_outliers if prefill else workloads.gaussian_outliers
    x = blocky(gen(M, K, seed, DEV), seed + 1, False)
    w = blocky(workloads.weights(N, K, seed, DEV), seed + 2, True)
    wq, s_w = pkg.fp8_quant_weight_blocks(w)
    xq, s_x = pkg.fp8_quant_per_token_group(x)
    return x, xq, s_x, wq, s_w


@pytest.mark.parametrize("M", [1, 8, 16, 17, 32, 48, 64])
@pytest.mark.parametrize("N,K", [(1024, 4096), (4096, 1024), (300, 1040), (640, 14336),
                                 (1, 32), (3, 16)])
def test_gemm_decode_sizes(oracle_mod, M, N, K):
    _, xq, s_x, wq, s_w = make_layer(M, N, K, 50 + M)
    y = pkg.fp8_scaled_gemm_blockwise(xq, s_x, wq, s_w)
    torch.cuda.synchronize()
    y_ref = oracle_mod.gemm_blockwise(host(xq), host(s_x), host(wq), host(s_w))
    check_rows(host(y.float()), y_ref, f"blockwise decode M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K", [(65, 512, 1024), (130, 300, 1040), (256, 1024, 4096),
                                   (1000, 768, 2048), (129, 4096, 512),
                                   # 240 and 336 tiles on 152 persistent CTAs
                                   (640, 12288, 512), (200, 43008, 256),
                                   # one output column, K = 16, a partial k-block
                                   (130, 1, 16), (300, 3, 144)])
def test_gemm_prefill_sizes(oracle_mod, M, N, K):
    _, xq, s_x, wq, s_w = make_layer(M, N, K, 70 + M, prefill=True)
    y = pkg.fp8_scaled_gemm_blockwise(xq, s_x, wq, s_w)
    torch.cuda.synchronize()
    y_ref = oracle_mod.gemm_blockwise(host(xq), host(s_x), host(wq), host(s_w))
    check_rows(host(y.float()), y_ref, f"blockwise prefill M={M} N={N} K={K}")


@pytest.mark.parametrize("M,K,N", [(2048, 4096, 6144), (8192, 4096, 4096), (4096, 8192, 10240)])
def test_gemm_prefill_full_size_sampled(oracle_mod, M, K, N):
    _, xq, s_x, wq, s_w = make_layer(M, N, K, 90, prefill=True)
    y = pkg.fp8_scaled_gemm_blockwise(xq, s_x, wq, s_w)
    torch.cuda.synchronize()
    rows = tile_rows(M, seed=M + N)
    yr = oracle_mod.gemm_blockwise(host(xq[rows]), host(s_x[rows]), host(wq), host(s_w))
    check_rows(host(y[rows].float()), yr, f"blockwise prefill {M}x{K}x{N} sampled rows")


def test_gemm_deterministic():
    _, xq, s_x, wq, s_w = make_layer(32, 4096, 4096, 91)
    a = pkg.fp8_scaled_gemm_blockwise(xq, s_x, wq, s_w)
    b = pkg.fp8_scaled_gemm_blockwise(xq, s_x, wq, s_w)
    _, xq2, s_x2, wq2, s_w2 = make_layer(512, 1024, 4096, 92)
    c = pkg.fp8_scaled_gemm_blockwise(xq2, s_x2, wq2, s_w2)
    d = pkg.fp8_scaled_gemm_blockwise(xq2, s_x2, wq2, s_w2)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(c, d)


# ------------------------------------------------------------ whole layer

@pytest.mark.parametrize("M,K,N", [(1, 4096, 6144), (32, 14336, 4096), (18, 256, 256),
                                   (300, 4096, 1024)])
def test_linear_blockwise(oracle_mod, M, K, N):
    x, _, _, wq, s_w = make_layer(M, N, K, 100 + M)
    ws = torch.empty(pkg.fp8_linear_blockwise_workspace_size(M, N, K), dtype=torch.uint8,
                     device=DEV)
    y = pkg.fp8_linear_blockwise(x, wq, s_w, workspace=ws)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_groups_bf16(bits(x))
    KB = -(-K // 128)
    off = -(-(M * K) // 256) * 256
    assert_bytes(ws[:M * K].view(M, K), q_ref, "workspace codes")
    assert_scales(ws[off:off + 4 * M * KB].view(torch.float32).view(M, KB), s_ref,
                  "workspace scales")
    y_ref = oracle_mod.gemm_blockwise(q_ref, s_ref, host(wq), host(s_w))
    check_rows(host(y.float()), y_ref, f"linear blockwise {M}x{K}x{N}")
    assert pkg.fp8_device_status() == pkg.FP8_OK
