"""GPU parity of the other scale granularities: quantization with a given
(static) per-tensor scale, with one dynamic scale for the whole tensor, and
the FP8 KV-cache write with per-tensor or per-head scales.  Codes and scales
must equal the CPU oracle's bit for bit; the codes then feed the scaled GEMM
unchanged (a per-tensor scale is a per-token scale that is the same on every
row)."""
import numpy as np
import pytest
import torch

import fp8_w8a8_quantized_gb300 as pkg
from fp8_w8a8_quantized_gb300 import workloads
from parity import bits, check_rows, host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def assert_codes(q_gpu, q_ref, what):
    qg = host(q_gpu)
    diff = np.argwhere(qg != q_ref)
    assert diff.size == 0, f"{what}: {len(diff)} codes differ, first at {tuple(diff[0])}: " \
        f"gpu={qg[tuple(diff[0])]:#x} ref={q_ref[tuple(diff[0])]:#x}"


def randn(shape, seed, scale=3.0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g, device=DEV) * scale).to(torch.bfloat16)


# ---------------------------------------------------------------- static scale

@pytest.mark.parametrize("M,K", [(1, 4096), (16, 4096), (32, 14336), (2048, 4096),
                                 (3, 48), (7, 2064), (130, 4112), (1, 16), (1000, 4112)])
@pytest.mark.parametrize("s_val", [1.0, 0.0123, 120.0 / 448.0])
def test_static_scale(oracle_mod, M, K, s_val):
    x = workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, DEV)
    s = torch.tensor([s_val], dtype=torch.float32, device=DEV)
    s_rows = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    q = pkg.fp8_quant_static(x, s, s_rows=s_rows)
    torch.cuda.synchronize()
    s32 = np.float32(s_val)
    assert_codes(q, oracle_mod.quant_rows_scaled_bf16(bits(x), s32), "static")
    assert np.all(host(s_rows) == s32)


@pytest.mark.parametrize("M,K", [(3, 65536), (2, 65552), (2, 131072)])
def test_static_scale_long_rows(oracle_mod, M, K):
    # the longest rows the register layout holds (4096 chunks), and rows
    # beyond it (the grid-stride loop)
    x = workloads.gaussian_outliers(M, K, 17, DEV)
    s = torch.tensor([0.0123], dtype=torch.float32, device=DEV)
    s_rows = torch.full((M,), -1.0, dtype=torch.float32, device=DEV)
    q = pkg.fp8_quant_static(x, s, s_rows=s_rows)
    torch.cuda.synchronize()
    assert_codes(q, oracle_mod.quant_rows_scaled_bf16(bits(x), np.float32(0.0123)), "static long")
    assert np.all(host(s_rows) == np.float32(0.0123))


def test_static_scale_saturates_and_strides(oracle_mod):
    # a scale far too small for the data: most codes clip to +-448
    M, K, ldx, ldq = 37, 512, 520, 544
    base = workloads.gaussian_outliers(M, ldx, 9, DEV)
    x = base[:, :K]
    s = torch.tensor([1e-3], dtype=torch.float32, device=DEV)
    xq = torch.full((M, ldq), 0xAB, dtype=torch.uint8, device=DEV)
    st = pkg.lib().fp8_quant_static(x.data_ptr(), M, K, ldx, s.data_ptr(), xq.data_ptr(), ldq,
                                    None, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    q_ref = oracle_mod.quant_rows_scaled_bf16(bits(x), np.float32(1e-3))
    assert_codes(xq[:, :K], q_ref, "static strided")
    assert np.all(host(xq)[:, K:] == 0xAB), "wrote past K"
    assert np.mean(np.isin(q_ref, [0x7E, 0xFE])) > 0.5


def test_static_scale_stress_rows(oracle_mod):
    x, _ = workloads.stress(DEV)
    s = torch.tensor([0.5], dtype=torch.float32, device=DEV)
    q = pkg.fp8_quant_static(x, s)
    torch.cuda.synchronize()
    assert_codes(q, oracle_mod.quant_rows_scaled_bf16(bits(x), np.float32(0.5)), "static stress")


# ---------------------------------------------------------- dynamic per-tensor

@pytest.mark.parametrize("M,K", [(1, 16), (1, 4096), (32, 4096), (2048, 4096), (8192, 4096),
                                 (5, 272), (33, 1040), (3, 65552)])
def test_per_tensor(oracle_mod, M, K):
    x = workloads.student_t_outliers(M, K, workloads.SEED_PREFILL, DEV)
    s_rows = torch.empty(M, dtype=torch.float32, device=DEV)
    q, s = pkg.fp8_quant_per_tensor(x, s_rows=s_rows)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_tensor_bf16(bits(x))
    assert host(s)[0].view(np.uint32) == np.float32(s_ref).view(np.uint32)
    assert np.all(host(s_rows) == np.float32(s_ref))
    assert_codes(q, q_ref, "per-tensor")


def test_per_tensor_max_in_last_element_and_zero_tensor(oracle_mod):
    M, K = 300, 4096
    x = randn((M, K), 21, 0.5)
    x[M - 1, K - 1] = -1000.0  # the maximum sits in the very last chunk
    q, s = pkg.fp8_quant_per_tensor(x)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_tensor_bf16(bits(x))
    assert host(s)[0] == np.float32(s_ref) == np.float32(1000.0) / np.float32(448.0)
    assert_codes(q, q_ref, "per-tensor max last")
    z = torch.zeros(64, 128, dtype=torch.bfloat16, device=DEV)
    qz, sz = pkg.fp8_quant_per_tensor(z)
    torch.cuda.synchronize()
    assert host(sz)[0] == 1.0 and np.all(host(qz) == 0)


def test_per_tensor_is_deterministic():
    x = workloads.student_t_outliers(4096, 4096, 5, DEV)
    q1, s1 = pkg.fp8_quant_per_tensor(x)
    q2, s2 = pkg.fp8_quant_per_tensor(x)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


def test_per_tensor_strided_rows(oracle_mod):
    # rows with a stride (the row-wise loops of both passes)
    M, K, ldx, ldq = 301, 1024, 1040, 1056
    base = workloads.gaussian_outliers(M, ldx, 13, DEV)
    x = base[:, :K]
    xq = torch.full((M, ldq), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    ws = torch.empty(int(pkg.lib().fp8_quant_per_tensor_workspace_size(M, K)), dtype=torch.uint8,
                     device=DEV)
    st = pkg.lib().fp8_quant_per_tensor(x.data_ptr(), M, K, ldx, xq.data_ptr(), ldq, s.data_ptr(),
                                        None, ws.data_ptr(), ws.numel(),
                                        torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    q_ref, s_ref = oracle_mod.quant_tensor_bf16(bits(x))
    assert host(s)[0].view(np.uint32) == np.float32(s_ref).view(np.uint32)
    assert_codes(xq[:, :K], q_ref, "per-tensor strided")
    assert np.all(host(xq)[:, K:] == 0xAB), "wrote past K"


@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_per_tensor_maximum_anywhere_in_a_large_tensor(oracle_mod, where):
    # 64 MB of activations (the grid-stride passes wrap many times); the
    # maximum is planted at the first value (the first chunk of the first
    # CTA), in the middle, or at the very last value (the last chunk, read
    # first by the second pass)
    M, K = 8192, 4096
    x = randn((M, K), 31, 1.0)
    r, c = {"first": (0, 0), "middle": (M // 2 + 5, K // 3 + 1), "last": (M - 1, K - 1)}[where]
    x[r, c] = -3072.0
    s_rows = torch.empty(M, dtype=torch.float32, device=DEV)
    q, s = pkg.fp8_quant_per_tensor(x, s_rows=s_rows)
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    assert host(s)[0] == np.float32(3072.0) / np.float32(448.0)
    assert np.all(host(s_rows) == host(s)[0])
    q_ref, s_ref = oracle_mod.quant_tensor_bf16(bits(x))
    assert np.float32(s_ref) == host(s)[0]
    assert_codes(q, q_ref, f"per-tensor, maximum {where}")


def test_per_tensor_in_a_cuda_graph(oracle_mod):
    # both launches of the per-tensor quantizer captured in a CUDA graph:
    # replays with new contents give new, exact results (nothing is kept
    # from one call to the next in the workspace)
    M, K = 2048, 4096
    x = torch.empty((M, K), dtype=torch.bfloat16, device=DEV)
    q = torch.empty((M, K), dtype=torch.uint8, device=DEV)
    s = torch.empty(1, dtype=torch.float32, device=DEV)
    x.copy_(randn((M, K), 40, 1.0))
    pkg.fp8_quant_per_tensor(x, xq=q, s=s)  # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            pkg.fp8_quant_per_tensor(x, xq=q, s=s)
    for seed, scale in [(41, 0.25), (42, 7.0), (43, 0.001)]:
        x.copy_(randn((M, K), seed, scale))
        g.replay()
        torch.cuda.synchronize()
        assert pkg.fp8_device_status() == 0
        q_ref, s_ref = oracle_mod.quant_tensor_bf16(bits(x))
        assert host(s)[0].view(np.uint32) == np.float32(s_ref).view(np.uint32)
        assert_codes(q, q_ref, f"per-tensor graph replay {seed}")


@pytest.mark.parametrize("M", [4, 32, 300])
def test_per_tensor_codes_feed_the_scaled_gemm(oracle_mod, M):
    N, K = 512, 4096
    x = workloads.gaussian_outliers(M, K, workloads.SEED_DECODE, DEV)
    w = workloads.weights(N, K, workloads.SEED_DECODE, DEV)
    wq, s_w = pkg.fp8_quant_per_channel_weights(w)
    s_rows = torch.empty(M, dtype=torch.float32, device=DEV)
    xq, _ = pkg.fp8_quant_per_tensor(x, s_rows=s_rows)
    y = pkg.fp8_scaled_gemm(xq, s_rows, wq, s_w)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_tensor_bf16(bits(x))
    y_ref = oracle_mod.scaled_gemm(q_ref, np.full(M, s_ref, np.float32), host(wq), host(s_w))
    check_rows(host(y.float()), y_ref, "per-tensor GEMM")


def test_static_codes_feed_the_scaled_gemm(oracle_mod):
    M, N, K = 48, 1024, 2048
    x = workloads.gaussian_outliers(M, K, 3, DEV)
    w = workloads.weights(N, K, 3, DEV)
    wq, s_w = pkg.fp8_quant_per_channel_weights(w)
    s = torch.tensor([0.05], dtype=torch.float32, device=DEV)
    s_rows = torch.empty(M, dtype=torch.float32, device=DEV)
    xq = pkg.fp8_quant_static(x, s, s_rows=s_rows)
    y = pkg.fp8_scaled_gemm(xq, s_rows, wq, s_w)
    torch.cuda.synchronize()
    q_ref = oracle_mod.quant_rows_scaled_bf16(bits(x), np.float32(0.05))
    y_ref = oracle_mod.scaled_gemm(q_ref, np.full(M, 0.05, np.float32), host(wq), host(s_w))
    check_rows(host(y.float()), y_ref, "static GEMM")


# ------------------------------------------------------------------- KV cache

def kv_case(oracle_mod, T, H, D, scale, slots, n_slots, seed):
    kv = randn((T, H, D), seed, 4.0)
    sc = torch.tensor(np.atleast_1d(np.asarray(scale, np.float32)), device=DEV)
    sl = None if slots is None else torch.tensor(slots, dtype=torch.int64, device=DEV)
    cache = torch.full((n_slots, H, D), 0xAB, dtype=torch.uint8, device=DEV)
    pkg.fp8_kv_cache_quant(kv, sc, cache, sl)
    torch.cuda.synchronize()
    ref = oracle_mod.kv_cache_quant_bf16(bits(kv), scale, slots, n_slots)
    rows = np.arange(min(T, n_slots)) if slots is None else np.asarray(slots)
    written = sorted({int(r) for r in rows if 0 <= r < n_slots})
    untouched = [r for r in range(n_slots) if r not in set(written)]
    cg = host(cache)
    assert_codes(cache[written], ref[written], "kv cache")
    assert np.all(cg[untouched] == 0xAB), "wrote a row no token maps to"


@pytest.mark.parametrize("T", [1, 32, 4096])
def test_kv_cache_per_head_scales_paged_slots(oracle_mod, T):
    # 8 KV heads of dimension 128 (the 8B and 70B models' attention)
    H, D, n_slots = 8, 128, 2 * T + 16
    rng = np.random.default_rng(T)
    slots = rng.permutation(n_slots)[:T].astype(np.int64)
    slots[:: 7] = -1                   # padding tokens
    scale = np.exp2(rng.uniform(-3, 2, H)).astype(np.float32)
    kv_case(oracle_mod, T, H, D, scale, slots, n_slots, T + 1)


def test_kv_cache_keys_and_values_identity_slots(oracle_mod):
    # no slot mapping (token t -> row t), one head of 16, a cache with spare rows
    T, H, D, n_slots = 5, 1, 16, 8
    k, v = randn((T, H, D), 71, 3.0), randn((T, H, D), 72, 0.5)
    kc = torch.full((n_slots, H, D), 0xAB, dtype=torch.uint8, device=DEV)
    vc = torch.full((n_slots, H, D), 0xCD, dtype=torch.uint8, device=DEV)
    ks = torch.tensor([0.02], device=DEV)
    vs = torch.tensor([1.0], device=DEV)
    pkg.fp8_kv_cache_quant_kv(k, v, ks, vs, kc, vc)
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    k_ref = oracle_mod.kv_cache_quant_bf16(bits(k), np.float32(0.02), None, n_slots)
    v_ref = oracle_mod.kv_cache_quant_bf16(bits(v), np.float32(1.0), None, n_slots)
    assert_codes(kc[:T], k_ref[:T], "keys")
    assert_codes(vc[:T], v_ref[:T], "values")
    assert np.all(host(kc)[T:] == 0xAB) and np.all(host(vc)[T:] == 0xCD)


@pytest.mark.parametrize("T,H,D,per_head", [(1, 8, 128, True), (33, 8, 128, True),
                                             (4096, 8, 128, True), (17, 3, 64, False),
                                             (9, 40, 80, True)])
def test_kv_cache_keys_and_values_in_one_launch(oracle_mod, T, H, D, per_head):
    # both caches must equal two separate writes with the same slots
    n_slots = 2 * T + 16
    rng = np.random.default_rng(T * 3 + H)
    slots = rng.permutation(n_slots)[:T].astype(np.int64)
    slots[:: 5] = -1
    slots[1:: 11] = n_slots + 3        # beyond the cache: skipped
    if per_head:
        ks = np.exp2(rng.uniform(-3, 2, H)).astype(np.float32)
        vs = np.exp2(rng.uniform(-3, 2, H)).astype(np.float32)
    else:
        ks, vs = np.float32(0.75), np.float32(1.0)
    k, v = randn((T, H, D), T + 5, 4.0), randn((T, H, D), T + 6, 2.0)
    kc = torch.full((n_slots, H, D), 0xAB, dtype=torch.uint8, device=DEV)
    vc = torch.full((n_slots, H, D), 0xCD, dtype=torch.uint8, device=DEV)
    dev_sc = lambda a: torch.tensor(np.atleast_1d(np.asarray(a, np.float32)), device=DEV)
    pkg.fp8_kv_cache_quant_kv(k, v, dev_sc(ks), dev_sc(vs), kc, vc,
                              torch.tensor(slots, device=DEV))
    torch.cuda.synchronize()
    assert pkg.fp8_device_status() == 0
    written = sorted({int(r) for r in slots if 0 <= r < n_slots})
    untouched = [r for r in range(n_slots) if r not in set(written)]
    k_ref = oracle_mod.kv_cache_quant_bf16(bits(k), ks, slots, n_slots)
    v_ref = oracle_mod.kv_cache_quant_bf16(bits(v), vs, slots, n_slots)
    assert_codes(kc[written], k_ref[written], "keys")
    assert_codes(vc[written], v_ref[written], "values")
    assert np.all(host(kc)[untouched] == 0xAB) and np.all(host(vc)[untouched] == 0xCD)


@pytest.mark.parametrize("T,H,D", [(64, 8, 128), (5, 1, 16), (17, 3, 64), (9, 40, 80)])
def test_kv_cache_per_tensor_scale_identity_slots(oracle_mod, T, H, D):
    kv_case(oracle_mod, T, H, D, 1.0, None, T + 3, T * H + D)


def test_kv_cache_out_of_range_slots_and_tiny_scale(oracle_mod):
    T, H, D = 12, 8, 128
    slots = np.array([0, 5, -3, 11, 12, 40, 3, 7, -1, 2, 9, 100], dtype=np.int64)
    kv_case(oracle_mod, T, H, D, 1e-3, slots, 12, 77)
