"""ctypes binding of the C ABI in include/fp8w8a8.h.

Argument marshalling only: every step of the layer runs in the CUDA library
(``_build/libfp8w8a8.so``).  If the library is missing the calls raise; there
is no CPU or PyTorch fallback.  Since the C ABI takes raw pointers and sizes,
each call first checks that its tensors are CUDA tensors of the shapes and
dtypes the sizes imply (ValueError otherwise); the library checks the rest
(alignment, K % 16, workspace size) and its status becomes Fp8Error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_HERE, "_build", "libfp8w8a8.so")

FP8_OK = 0
STATUS_NAMES = {
    0: "FP8_OK",
    1: "FP8_ERR_INVALID_ARG",
    2: "FP8_ERR_UNSUPPORTED",
    3: "FP8_ERR_WORKSPACE",
    4: "FP8_ERR_CUDA",
    5: "FP8_ERR_TIMEOUT",
}

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_st = ctypes.c_int


class Fp8Error(RuntimeError):
    """A call of the library returned a status other than FP8_OK."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


def lib() -> ctypes.CDLL:
    """The loaded CUDA library, with argument types declared."""
    global _lib
    L = _lib
    if L is not None:  # loaded: no lock on the per-call path
        return L
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIBRARY_PATH):
            raise RuntimeError(
                f"CUDA library not built ({LIBRARY_PATH}); run "
                "`python -m fp8_w8a8_quantized_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIBRARY_PATH)
        L.fp8_quant_per_token.restype = _st
        L.fp8_quant_per_token.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]
        L.fp8_quant_per_channel_weights.restype = _st
        L.fp8_quant_per_channel_weights.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]
        L.fp8_scaled_gemm.restype = _st
        L.fp8_scaled_gemm.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp,
                                      ctypes.c_size_t, _vp]
        L.fp8_linear.restype = _st
        L.fp8_linear.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, ctypes.c_size_t, _vp]
        L.fp8_linear_workspace_size.restype = ctypes.c_size_t
        L.fp8_linear_workspace_size.argtypes = [_i64, _i64, _i64]
        L.fp8_scaled_gemm_workspace_size.restype = ctypes.c_size_t
        L.fp8_scaled_gemm_workspace_size.argtypes = [_i64, _i64, _i64]
        L.fp8_quant_static.restype = _st
        L.fp8_quant_static.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _vp]
        L.fp8_quant_per_tensor.restype = _st
        L.fp8_quant_per_tensor.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp,
                                           ctypes.c_size_t, _vp]
        L.fp8_quant_per_tensor_workspace_size.restype = ctypes.c_size_t
        L.fp8_quant_per_tensor_workspace_size.argtypes = [_i64, _i64]
        L.fp8_kv_cache_quant.restype = _st
        L.fp8_kv_cache_quant.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64, _vp]
        L.fp8_kv_cache_quant_kv.restype = _st
        L.fp8_kv_cache_quant_kv.argtypes = [_vp, _vp, _i64, _i64, _i64, _vp, _vp, _i64, _vp, _vp,
                                            _vp, _i64, _vp]
        L.fp8_quant_per_token_group.restype = _st
        L.fp8_quant_per_token_group.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]
        L.fp8_quant_weight_blocks.restype = _st
        L.fp8_quant_weight_blocks.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp]
        L.fp8_scaled_gemm_blockwise.restype = _st
        L.fp8_scaled_gemm_blockwise.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp,
                                                ctypes.c_size_t, _vp]
        L.fp8_linear_blockwise.restype = _st
        L.fp8_linear_blockwise.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp,
                                           ctypes.c_size_t, _vp]
        L.fp8_linear_blockwise_workspace_size.restype = ctypes.c_size_t
        L.fp8_linear_blockwise_workspace_size.argtypes = [_i64, _i64, _i64]
        L.fp8_rmsnorm_quant.restype = _st
        L.fp8_rmsnorm_quant.argtypes = [_vp, _vp, ctypes.c_float, _i64, _i64, _i64, _vp, _i64,
                                        _vp, _vp, _vp]
        L.fp8_linear_rmsnorm.restype = _st
        L.fp8_linear_rmsnorm.argtypes = [_vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i64, _i64,
                                         _i64, _vp, ctypes.c_size_t, _vp]
        L.fp8_status_string.restype = ctypes.c_char_p
        L.fp8_status_string.argtypes = [_st]
        L.fp8_device_status.restype = _st
        L.fp8_device_status.argtypes = [ctypes.c_int]
        L.fp8_selftest_wait_timeout.restype = _st
        L.fp8_selftest_wait_timeout.argtypes = [_i64, _vp, _vp]
        _lib = L
        return L


def _check(status: int, what: str):
    if status != FP8_OK:
        raise Fp8Error(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _expect(t, name: str, shape: tuple, dtype, contiguous: bool = True):
    """The kernels index raw device memory by the sizes they are given: every
    tensor must be a CUDA tensor of exactly the expected shape and dtype (and
    contiguous, or with unit stride along its last dimension)."""
    if (not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda
            or tuple(t.shape) != tuple(shape)
            or (not t.is_contiguous() if contiguous else (t.dim() == 2 and t.shape[1] > 1
                                                          and t.stride(1) != 1))):
        got = (f"{t.dtype} {tuple(t.shape)} on {t.device}"
               f"{'' if t.is_contiguous() else ', not contiguous'}"
               if isinstance(t, torch.Tensor) else type(t).__name__)
        raise ValueError(f"{name} must be a CUDA {dtype} tensor of shape {tuple(shape)}"
                         f"{', contiguous' if contiguous else ''}; got {got}")


def _workspace(t, name: str = "workspace"):
    if not isinstance(t, torch.Tensor) or t.dtype != torch.uint8 or not t.is_cuda \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA uint8 tensor")


def _rows(t: torch.Tensor, name: str):
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be 2-D with unit stride along K")
    return t.shape[0], t.shape[1], t.stride(0)


def fp8_status_string(status: int) -> str:
    return lib().fp8_status_string(status).decode()


def fp8_device_status(clear: bool = False) -> int:
    """FP8_OK, or FP8_ERR_TIMEOUT if a kernel gave up a bounded wait."""
    return lib().fp8_device_status(1 if clear else 0)


def fp8_linear_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().fp8_linear_workspace_size(M, N, K))


def fp8_quant_per_token(x: torch.Tensor, xq: torch.Tensor | None = None,
                        s_tok: torch.Tensor | None = None, stream=None):
    """bf16 [M, K] -> (E4M3 codes uint8 [M, K], fp32 scales [M])."""
    M, K, ldx = _rows(x, "x")
    _expect(x, "x", (M, K), torch.bfloat16, contiguous=False)
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if s_tok is None:
        s_tok = torch.empty((M,), dtype=torch.float32, device=x.device)
    _expect(xq, "xq", (M, K), torch.uint8, contiguous=False)
    _expect(s_tok, "s_tok", (M,), torch.float32)
    _check(lib().fp8_quant_per_token(_ptr(x), M, K, ldx, _ptr(xq), xq.stride(0) if M else K,
                                     _ptr(s_tok), _stream(stream)), "fp8_quant_per_token")
    return xq, s_tok


def fp8_quant_per_channel_weights(w: torch.Tensor, wq: torch.Tensor | None = None,
                                  s_w: torch.Tensor | None = None, stream=None):
    """bf16 [N, K] -> (E4M3 codes uint8 [N, K], fp32 per-row scales [N])."""
    N, K, ldw = _rows(w, "w")
    _expect(w, "w", (N, K), torch.bfloat16, contiguous=False)
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if s_w is None:
        s_w = torch.empty((N,), dtype=torch.float32, device=w.device)
    _expect(wq, "wq", (N, K), torch.uint8, contiguous=False)
    _expect(s_w, "s_w", (N,), torch.float32)
    _check(lib().fp8_quant_per_channel_weights(_ptr(w), N, K, ldw, _ptr(wq),
                                               wq.stride(0) if N else K, _ptr(s_w),
                                               _stream(stream)),
           "fp8_quant_per_channel_weights")
    return wq, s_w


def fp8_scaled_gemm(xq: torch.Tensor, s_tok: torch.Tensor, wq: torch.Tensor,
                    s_w: torch.Tensor, y: torch.Tensor | None = None, stream=None):
    """(codes [M, K], scales [M]) x (codes [N, K], scales [N]) -> bf16 [M, N]."""
    M, K = xq.shape
    N = wq.shape[0]
    _expect(xq, "xq", (M, K), torch.uint8)
    _expect(s_tok, "s_tok", (M,), torch.float32)
    _expect(wq, "wq", (N, K), torch.uint8)
    _expect(s_w, "s_w", (N,), torch.float32)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    _expect(y, "y", (M, N), torch.bfloat16)
    _check(lib().fp8_scaled_gemm(_ptr(xq), _ptr(s_tok), _ptr(wq), _ptr(s_w), _ptr(y),
                                 M, N, K, None, 0, _stream(stream)), "fp8_scaled_gemm")
    return y


def fp8_linear(x: torch.Tensor, wq: torch.Tensor, s_w: torch.Tensor,
               y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
               stream=None):
    """The whole W8A8 layer: bf16 X [M, K] and offline-quantized W -> bf16 [M, N]."""
    M, K = x.shape
    N = wq.shape[0]
    _expect(x, "x", (M, K), torch.bfloat16)
    _expect(wq, "wq", (N, K), torch.uint8)
    _expect(s_w, "s_w", (N,), torch.float32)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _expect(y, "y", (M, N), torch.bfloat16)
    if workspace is None:  # (a given workspace is size-checked by the library)
        workspace = torch.empty((max(fp8_linear_workspace_size(M, N, K), 1),), dtype=torch.uint8, device=x.device)
    _workspace(workspace)
    _check(lib().fp8_linear(_ptr(x), _ptr(wq), _ptr(s_w), _ptr(y), M, N, K,
                            _ptr(workspace), workspace.numel(), _stream(stream)), "fp8_linear")
    return y


def fp8_quant_static(x: torch.Tensor, s: torch.Tensor, xq: torch.Tensor | None = None,
                     s_rows: torch.Tensor | None = None, stream=None):
    """bf16 [M, K] with a given fp32 scale s [1] -> E4M3 codes uint8 [M, K].
    If s_rows (fp32 [M]) is given, s is written to every entry."""
    M, K, ldx = _rows(x, "x")
    _expect(x, "x", (M, K), torch.bfloat16, contiguous=False)
    _expect(s, "s", tuple(s.shape), torch.float32)
    if s.numel() != 1:
        raise ValueError("s must hold one scale")
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    _expect(xq, "xq", (M, K), torch.uint8, contiguous=False)
    if s_rows is not None:
        _expect(s_rows, "s_rows", (M,), torch.float32)
    _check(lib().fp8_quant_static(_ptr(x), M, K, ldx, _ptr(s), _ptr(xq),
                                  xq.stride(0) if M else K, _ptr(s_rows), _stream(stream)),
           "fp8_quant_static")
    return xq


def fp8_quant_per_tensor(x: torch.Tensor, xq: torch.Tensor | None = None,
                         s: torch.Tensor | None = None, s_rows: torch.Tensor | None = None,
                         workspace: torch.Tensor | None = None, stream=None):
    """bf16 [M, K] -> (E4M3 codes uint8 [M, K], fp32 scale [1]) with one
    dynamic scale amax / 448 for the whole tensor."""
    M, K, ldx = _rows(x, "x")
    _expect(x, "x", (M, K), torch.bfloat16, contiguous=False)
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if s is None:
        s = torch.empty((1,), dtype=torch.float32, device=x.device)
    _expect(xq, "xq", (M, K), torch.uint8, contiguous=False)
    _expect(s, "s", tuple(s.shape), torch.float32)
    if s.numel() != 1:
        raise ValueError("s must hold one scale")
    if s_rows is not None:
        _expect(s_rows, "s_rows", (M,), torch.float32)
    need = int(lib().fp8_quant_per_tensor_workspace_size(M, K))
    if workspace is None:
        workspace = torch.empty((need,), dtype=torch.uint8, device=x.device)
    _workspace(workspace)
    _check(lib().fp8_quant_per_tensor(_ptr(x), M, K, ldx, _ptr(xq), xq.stride(0) if M else K,
                                      _ptr(s), _ptr(s_rows), _ptr(workspace), workspace.numel(),
                                      _stream(stream)), "fp8_quant_per_tensor")
    return xq, s


def fp8_kv_cache_quant(kv: torch.Tensor, scale: torch.Tensor, cache: torch.Tensor,
                       slot_mapping: torch.Tensor | None = None, stream=None):
    """Write bf16 keys or values [T, H, D] into the E4M3 cache [n_slots, H, D]
    (uint8) at rows slot_mapping [T] (int64; negative skips), each head h
    divided by scale[h] (per-head, [H]) or scale[0] (per-tensor, [1])."""
    if kv.dim() != 3 or not kv.is_contiguous() or cache.dim() != 3 or not cache.is_contiguous():
        raise ValueError("kv and cache must be contiguous [T, H, D] / [n_slots, H, D]")
    T, H, D = kv.shape
    if cache.shape[1:] != (H, D):
        raise ValueError("cache must be [n_slots, H, D]")
    _expect(kv, "kv", (T, H, D), torch.bfloat16)
    _expect(cache, "cache", tuple(cache.shape), torch.uint8)
    _expect(scale, "scale", tuple(scale.shape), torch.float32)
    if slot_mapping is not None:
        _expect(slot_mapping, "slot_mapping", (T,), torch.int64)
    stride = 1 if scale.numel() == H and H > 1 else 0
    if stride == 0 and scale.numel() != 1:
        raise ValueError("scale must have 1 or H entries")
    _check(lib().fp8_kv_cache_quant(_ptr(kv), T, H, D, _ptr(scale), stride, _ptr(slot_mapping),
                                    _ptr(cache), cache.shape[0], _stream(stream)),
           "fp8_kv_cache_quant")
    return cache


def fp8_kv_cache_quant_kv(k: torch.Tensor, v: torch.Tensor, k_scale: torch.Tensor,
                          v_scale: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          slot_mapping: torch.Tensor | None = None, stream=None):
    """Keys and values of one layer in one launch: fp8_kv_cache_quant on
    (k, k_scale, k_cache) and on (v, v_scale, v_cache) with the same slots."""
    for t in (k, v, k_cache, v_cache):
        if t.dim() != 3 or not t.is_contiguous():
            raise ValueError("k, v and the caches must be contiguous [T, H, D] / [n_slots, H, D]")
    T, H, D = k.shape
    if v.shape != k.shape or k_cache.shape != v_cache.shape or k_cache.shape[1:] != (H, D):
        raise ValueError("k and v must be [T, H, D], both caches [n_slots, H, D]")
    for t, name in ((k, "k"), (v, "v")):
        _expect(t, name, (T, H, D), torch.bfloat16)
    for t, name in ((k_cache, "k_cache"), (v_cache, "v_cache")):
        _expect(t, name, tuple(k_cache.shape), torch.uint8)
    for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _expect(t, name, tuple(t.shape), torch.float32)
    if slot_mapping is not None:
        _expect(slot_mapping, "slot_mapping", (T,), torch.int64)
    if k_scale.numel() != v_scale.numel():
        raise ValueError("k_scale and v_scale must have the same number of entries")
    stride = 1 if k_scale.numel() == H and H > 1 else 0
    if stride == 0 and k_scale.numel() != 1:
        raise ValueError("scales must have 1 or H entries")
    _check(lib().fp8_kv_cache_quant_kv(_ptr(k), _ptr(v), T, H, D, _ptr(k_scale), _ptr(v_scale),
                                       stride, _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                       k_cache.shape[0], _stream(stream)),
           "fp8_kv_cache_quant_kv")
    return k_cache, v_cache


def fp8_rmsnorm_quant(x: torch.Tensor, gamma: torch.Tensor, eps: float,
                      xq: torch.Tensor | None = None, s_tok: torch.Tensor | None = None,
                      y: torch.Tensor | bool | None = None, stream=None):
    """RMSNorm of bf16 x [M, K] with weights gamma [K], quantized per token.
    Returns (codes uint8 [M, K], fp32 scales [M], normalised bf16 rows or
    None); pass y=True (or a bf16 [M, K] tensor) to get the rows."""
    M, K, ldx = _rows(x, "x")
    _expect(x, "x", (M, K), torch.bfloat16, contiguous=False)
    _expect(gamma, "gamma", (K,), torch.bfloat16)
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if s_tok is None:
        s_tok = torch.empty((M,), dtype=torch.float32, device=x.device)
    if y is True:
        y = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    elif y is False:
        y = None
    _expect(xq, "xq", (M, K), torch.uint8, contiguous=False)
    _expect(s_tok, "s_tok", (M,), torch.float32)
    if y is not None:
        _expect(y, "y", (M, K), torch.bfloat16)
    _check(lib().fp8_rmsnorm_quant(_ptr(x), _ptr(gamma), float(eps), M, K, ldx, _ptr(xq),
                                   xq.stride(0) if M else K, _ptr(s_tok), _ptr(y),
                                   _stream(stream)), "fp8_rmsnorm_quant")
    return xq, s_tok, y


def fp8_linear_rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float, wq: torch.Tensor,
                       s_w: torch.Tensor, y: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None):
    """The layer fed by RMSNorm: y = fp8_linear(rms_norm(x) * gamma) with the
    per-token quantization fused into the normalisation kernel."""
    M, K = x.shape
    N = wq.shape[0]
    _expect(x, "x", (M, K), torch.bfloat16)
    _expect(gamma, "gamma", (K,), torch.bfloat16)
    _expect(wq, "wq", (N, K), torch.uint8)
    _expect(s_w, "s_w", (N,), torch.float32)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _expect(y, "y", (M, N), torch.bfloat16)
    if workspace is None:  # (a given workspace is size-checked by the library)
        workspace = torch.empty((max(fp8_linear_workspace_size(M, N, K), 1),), dtype=torch.uint8, device=x.device)
    _workspace(workspace)
    _check(lib().fp8_linear_rmsnorm(_ptr(x), _ptr(gamma), float(eps), _ptr(wq), _ptr(s_w),
                                    _ptr(y), M, N, K, _ptr(workspace), workspace.numel(),
                                    _stream(stream)), "fp8_linear_rmsnorm")
    return y


BLOCK = 128  # edge of the block-wise scales


def _blocks(n: int) -> int:
    return (n + BLOCK - 1) // BLOCK


def fp8_quant_per_token_group(x: torch.Tensor, xq: torch.Tensor | None = None,
                              s_x: torch.Tensor | None = None, stream=None):
    """bf16 [M, K] -> (codes uint8 [M, K], fp32 scales [M, ceil(K/128)]),
    one scale per token per 128 inputs."""
    M, K, ldx = _rows(x, "x")
    _expect(x, "x", (M, K), torch.bfloat16, contiguous=False)
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if s_x is None:
        s_x = torch.empty((M, _blocks(K)), dtype=torch.float32, device=x.device)
    _expect(xq, "xq", (M, K), torch.uint8, contiguous=False)
    _expect(s_x, "s_x", (M, _blocks(K)), torch.float32)
    _check(lib().fp8_quant_per_token_group(_ptr(x), M, K, ldx, _ptr(xq), xq.stride(0) if M else K,
                                           _ptr(s_x), _stream(stream)),
           "fp8_quant_per_token_group")
    return xq, s_x


def fp8_quant_weight_blocks(w: torch.Tensor, wq: torch.Tensor | None = None,
                            s_w: torch.Tensor | None = None, stream=None):
    """bf16 [N, K] -> (codes uint8 [N, K], fp32 scales [ceil(N/128), ceil(K/128)]),
    one scale per 128 x 128 block."""
    N, K, ldw = _rows(w, "w")
    _expect(w, "w", (N, K), torch.bfloat16, contiguous=False)
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if s_w is None:
        s_w = torch.empty((_blocks(N), _blocks(K)), dtype=torch.float32, device=w.device)
    _expect(wq, "wq", (N, K), torch.uint8, contiguous=False)
    _expect(s_w, "s_w", (_blocks(N), _blocks(K)), torch.float32)
    _check(lib().fp8_quant_weight_blocks(_ptr(w), N, K, ldw, _ptr(wq), wq.stride(0) if N else K,
                                         _ptr(s_w), _stream(stream)), "fp8_quant_weight_blocks")
    return wq, s_w


def fp8_scaled_gemm_blockwise(xq: torch.Tensor, s_x: torch.Tensor, wq: torch.Tensor,
                              s_w: torch.Tensor, y: torch.Tensor | None = None, stream=None):
    """Block-scaled GEMM: (codes [M, K], s_x [M, KB]) x (codes [N, K], s_w [NB, KB]) -> bf16."""
    M, K = xq.shape
    N = wq.shape[0]
    _expect(xq, "xq", (M, K), torch.uint8)
    _expect(s_x, "s_x", (M, _blocks(K)), torch.float32)
    _expect(wq, "wq", (N, K), torch.uint8)
    _expect(s_w, "s_w", (_blocks(N), _blocks(K)), torch.float32)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    _expect(y, "y", (M, N), torch.bfloat16)
    _check(lib().fp8_scaled_gemm_blockwise(_ptr(xq), _ptr(s_x), _ptr(wq), _ptr(s_w), _ptr(y),
                                           M, N, K, None, 0, _stream(stream)),
           "fp8_scaled_gemm_blockwise")
    return y


def fp8_linear_blockwise_workspace_size(M: int, N: int, K: int) -> int:
    return int(lib().fp8_linear_blockwise_workspace_size(M, N, K))


def fp8_linear_blockwise(x: torch.Tensor, wq: torch.Tensor, s_w: torch.Tensor,
                         y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         stream=None):
    """The block-scaled layer: bf16 X [M, K] and block-quantized W -> bf16 [M, N]."""
    M, K = x.shape
    N = wq.shape[0]
    _expect(x, "x", (M, K), torch.bfloat16)
    _expect(wq, "wq", (N, K), torch.uint8)
    _expect(s_w, "s_w", (_blocks(N), _blocks(K)), torch.float32)
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _expect(y, "y", (M, N), torch.bfloat16)
    if workspace is None:  # (a given workspace is size-checked by the library)
        workspace = torch.empty((max(fp8_linear_blockwise_workspace_size(M, N, K), 1),), dtype=torch.uint8, device=x.device)
    _workspace(workspace)
    _check(lib().fp8_linear_blockwise(_ptr(x), _ptr(wq), _ptr(s_w), _ptr(y), M, N, K,
                                      _ptr(workspace), workspace.numel(), _stream(stream)),
           "fp8_linear_blockwise")
    return y


class QuantizedLinear:
    """A bias-free linear layer whose weight was quantized once (per output
    channel) by the library, and whose forward is fp8_linear.  The
    workspace is kept and grown as needed; one instance must not be called
    from two streams at once."""

    def __init__(self, weight_bf16: torch.Tensor, stream=None):
        self.out_features, self.in_features = weight_bf16.shape
        self.wq, self.s_w = fp8_quant_per_channel_weights(weight_bf16, stream=stream)
        self._ws = None

    def __call__(self, x: torch.Tensor, y: torch.Tensor | None = None, stream=None):
        need = fp8_linear_workspace_size(x.shape[0], self.out_features, self.in_features)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty((max(need, 1),), dtype=torch.uint8, device=x.device)
        return fp8_linear(x, self.wq, self.s_w, y=y, workspace=self._ws, stream=stream)
