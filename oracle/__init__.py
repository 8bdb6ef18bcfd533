"""CPU oracle for the FP8_DYNAMIC W8A8 linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import this package.  The
product path (``fp8_w8a8_quantized_gb300``) never imports it, and the two
share no code: the arithmetic lives in ``fp8_oracle.c`` (plain C, compiled
with gcc, no fast-math), and this module only marshals numpy arrays.

What it computes (page title, section):

* E4M3 codec -- "FP8 Inference Explained, in depth", "The numbers in one
  byte"; bit layout from "FP8 Quantization", "FP8 Representation".  A value
  is encoded as the nearest entry of the decoded code table (ties to the even
  code, saturating at +-448); a test checks that this equals the pages'
  step-by-step rounding (binade, grid spacing, half to even, clip).
* Per-token dynamic quantization, s = amax/448, q = E4M3(fl32(x / s)) --
  "FP8 Inference Explained", "Scales and their granularity"; "Quantization:
  FP8 inference and KV-cache quantization", "Dynamic scales or static scales".
* Per-output-channel weight quantization: the same rule over the rows of W
  ("FP8 Quantization", "Granularity", per-channel).
* The scaled GEMM y = s_tok[m] s_w[n] sum_k q_x[m,k] q_w[n,k], with the dot
  product of codes computed exactly in int64 and the scales applied in fp64
  -- "FP8 Inference Explained", "Inside a quantized linear layer".

Parity status of each function is recorded in the test files that pin it;
the BF16 rounding of the GPU output has no bitwise oracle (its parity is
"unpinned" bitwise and is covered by the stated tolerance instead).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


# Compiler command for the oracle source (also used by the mutation test,
# which compiles copies of it with one planted mistake each).
CC_FLAGS = ["-O2", "-std=c11", "-fopenmp", "-pthread", "-ffp-contract=off",
            "-fno-fast-math", "-fPIC", "-shared"]


def compile_source(src: str, out: str) -> None:
    subprocess.run(["gcc"] + CC_FLAGS + ["-o", out, src, "-lm"], check=True)


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP, IEEE fp32 division, no FMA
    contraction).  Returns the path of the shared library.  The environment
    variable FP8_ORACLE_LIB names another compiled copy to load instead (the
    mutation test's planted-mistake builds)."""
    alt = os.environ.get("FP8_ORACLE_LIB")
    if alt:
        return alt
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    compile_source(_SRC, tmp)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_round_e4m3.restype = ctypes.c_double
        lib.orc_round_e4m3.argtypes = [ctypes.c_double]
        lib.orc_e4m3_pack.restype = ctypes.c_uint8
        lib.orc_e4m3_pack.argtypes = [ctypes.c_double]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
        lib.orc_bf16_to_f32.restype = ctypes.c_float
        lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.orc_quant_rows_bf16.restype = None
        lib.orc_quant_rows_bf16.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp]
        lib.orc_quant_rows_f32.restype = None
        lib.orc_quant_rows_f32.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp]
        lib.orc_gemm_exact.restype = None
        lib.orc_gemm_exact.argtypes = [_vp, _i64, _vp, _i64, _i64, _i64, _i64, _vp]
        lib.orc_epilogue.restype = None
        lib.orc_epilogue.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp]
        lib.orc_linear_points.restype = None
        lib.orc_linear_points.argtypes = [_vp, _i64, _vp, _vp, _i64, _vp, _i64,
                                          _i64, _vp, _vp, _vp]
        lib.orc_quant_rows_scaled_bf16.restype = None
        lib.orc_quant_rows_scaled_bf16.argtypes = [_vp, _i64, _i64, _i64, _vp, _vp, _i64]
        lib.orc_quant_tensor_bf16.restype = None
        lib.orc_quant_tensor_bf16.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp]
        lib.orc_kv_cache_quant_bf16.restype = None
        lib.orc_kv_cache_quant_bf16.argtypes = [_vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp]
        lib.orc_quant_blocks_bf16.restype = None
        lib.orc_quant_blocks_bf16.argtypes = [_vp, _i64, _i64, _i64, _i64, _i64, _vp, _i64, _vp]
        lib.orc_gemm_blockwise.restype = None
        lib.orc_gemm_blockwise.argtypes = [_vp, _i64, _vp, _vp, _i64, _vp, _i64, _i64, _i64,
                                           _i64, _i64, _i64, _vp, _vp, _vp]
        lib.orc_rmsnorm_bracket_bf16.restype = None
        lib.orc_rmsnorm_bracket_bf16.argtypes = [_vp, _i64, _i64, _i64, _vp, ctypes.c_float,
                                                 ctypes.c_double, _vp, _vp, _vp]
        lib.orc_rmsnorm_f64.restype = None
        lib.orc_rmsnorm_f64.argtypes = [_vp, _i64, _i64, _i64, _vp, ctypes.c_double, _vp]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_num_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().orc_num_threads())


# --------------------------------------------------------------------------
# codec
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Real value (fp64) of each E4M3 code; NaN for 0x7F / 0xFF."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e4m3_decode(int(v)) for v in c.ravel()],
                    dtype=np.float64).reshape(c.shape)


def round_e4m3(values) -> np.ndarray:
    """Nearest E4M3 value (fp64), ties to even, saturating at +-448, zero
    and NaN unchanged (the decoded code of e4m3_encode)."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.array([lib.orc_round_e4m3(float(x)) for x in v.ravel()],
                    dtype=np.float64).reshape(v.shape)


def e4m3_encode(values) -> np.ndarray:
    """Saturating round-to-nearest-even E4M3 code of each value."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.array([lib.orc_e4m3_encode(float(x)) for x in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


def e4m3_pack(values) -> np.ndarray:
    """Bit pattern of values that already lie on the E4M3 grid."""
    lib = _load()
    v = np.asarray(values, dtype=np.float64)
    return np.array([lib.orc_e4m3_pack(float(x)) for x in v.ravel()],
                    dtype=np.uint8).reshape(v.shape)


# --------------------------------------------------------------------------
# quantization
# --------------------------------------------------------------------------

def quant_rows_bf16(x_bits: np.ndarray):
    """Dynamic per-row quantization of bf16 rows (given as uint16 bit
    patterns, shape [R, K]).  Returns (codes uint8 [R, K], scales fp32 [R]).
    Used for per-token activations and per-output-channel weights alike."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, K = x.shape
    q = np.empty((R, K), dtype=np.uint8)
    s = np.empty((R,), dtype=np.float32)
    if R and K:
        lib.orc_quant_rows_bf16(_ptr(x), R, K, K, _ptr(q), K, _ptr(s))
    elif R:
        s[:] = 1.0
    return q, s


def quant_rows_f32(x: np.ndarray):
    """Same rule for rows given in fp32 (the pages' fp32 worked examples)."""
    lib = _load()
    xf = np.ascontiguousarray(x, dtype=np.float32)
    R, K = xf.shape
    q = np.empty((R, K), dtype=np.uint8)
    s = np.empty((R,), dtype=np.float32)
    if R:
        lib.orc_quant_rows_f32(_ptr(xf), R, K, K, _ptr(q), K, _ptr(s))
    return q, s


def quant_rows_scaled_bf16(x_bits: np.ndarray, scales) -> np.ndarray:
    """Each row r quantized with the given scale s[r] (a static scale is the
    same value for every row): q = E4M3(fl32(x / s))."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, K = x.shape
    s = np.ascontiguousarray(np.broadcast_to(np.asarray(scales, dtype=np.float32), (R,)))
    q = np.empty((R, K), dtype=np.uint8)
    if R and K:
        lib.orc_quant_rows_scaled_bf16(_ptr(x), R, K, K, _ptr(s), _ptr(q), K)
    return q


def quant_tensor_bf16(x_bits: np.ndarray):
    """Dynamic per-tensor quantization: one scale amax(all)/448 (1 if all
    zero).  Returns (codes, scale as fp32 scalar)."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, K = x.shape
    q = np.empty((R, K), dtype=np.uint8)
    s = np.ones((1,), dtype=np.float32)
    if R and K:
        lib.orc_quant_tensor_bf16(_ptr(x), R, K, K, _ptr(q), K, _ptr(s))
    return q, s[0]


def kv_cache_quant_bf16(x_bits: np.ndarray, scale, slots, n_slots: int) -> np.ndarray:
    """KV-cache write: x [T, H, D] bf16 bits, scale [H] (per head) or a
    scalar (per tensor), slots [T] or None (identity); a token whose slot is
    negative or >= n_slots is skipped.
    Returns the cache [n_slots, H, D] of E4M3 codes (untouched rows 0)."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H, D = x.shape
    sc = np.atleast_1d(np.asarray(scale, dtype=np.float32))
    stride = 1 if sc.size == H and H > 1 else 0
    sl = None if slots is None else np.ascontiguousarray(slots, dtype=np.int64)
    cache = np.zeros((n_slots, H, D), dtype=np.uint8)
    if T and H and D:
        lib.orc_kv_cache_quant_bf16(_ptr(x), T, H, D, _ptr(sc), stride,
                                    None if sl is None else _ptr(sl), n_slots, _ptr(cache))
    return cache


# --------------------------------------------------------------------------
# GEMM + epilogue
# --------------------------------------------------------------------------

def gemm_exact(qx: np.ndarray, qw: np.ndarray) -> np.ndarray:
    """acc[m, n] = sum_k (512 q_x[m,k]) (512 q_w[n,k]) exactly, int64.
    The true dot product of the decoded values is acc * 2^-18."""
    lib = _load()
    a = np.ascontiguousarray(qx, dtype=np.uint8)
    b = np.ascontiguousarray(qw, dtype=np.uint8)
    M, K = a.shape
    N, K2 = b.shape
    assert K == K2
    acc = np.zeros((M, N), dtype=np.int64)
    if M and N:
        lib.orc_gemm_exact(_ptr(a), K, _ptr(b), K, M, N, K, _ptr(acc))
    return acc


def epilogue(acc: np.ndarray, s_tok: np.ndarray, s_w: np.ndarray) -> np.ndarray:
    """y = acc * 2^-18 * s_tok[m] * s_w[n] in fp64."""
    lib = _load()
    a = np.ascontiguousarray(acc, dtype=np.int64)
    st = np.ascontiguousarray(s_tok, dtype=np.float32)
    sw = np.ascontiguousarray(s_w, dtype=np.float32)
    M, N = a.shape
    y = np.empty((M, N), dtype=np.float64)
    if M and N:
        lib.orc_epilogue(_ptr(a), M, N, _ptr(st), _ptr(sw), _ptr(y))
    return y


def scaled_gemm(qx, s_tok, qw, s_w) -> np.ndarray:
    """Full fp64 output of the scaled FP8 GEMM."""
    return epilogue(gemm_exact(qx, qw), s_tok, s_w)


def linear(x_bits: np.ndarray, qw: np.ndarray, s_w: np.ndarray):
    """The whole layer: per-token quantization of x, then the scaled GEMM.
    Returns (y fp64 [M, N], q_x, s_tok)."""
    qx, st = quant_rows_bf16(x_bits)
    return scaled_gemm(qx, st, qw, s_w), qx, st


def linear_points(qx, s_tok, qw, s_w, rows, cols) -> np.ndarray:
    """y at the given (row, col) points only (fp64)."""
    lib = _load()
    a = np.ascontiguousarray(qx, dtype=np.uint8)
    b = np.ascontiguousarray(qw, dtype=np.uint8)
    st = np.ascontiguousarray(s_tok, dtype=np.float32)
    sw = np.ascontiguousarray(s_w, dtype=np.float32)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    assert r.shape == c.shape
    K = a.shape[1]
    assert b.shape[1] == K
    y = np.empty(r.shape, dtype=np.float64)
    if r.size:
        lib.orc_linear_points(_ptr(a), K, _ptr(st), _ptr(b), K, _ptr(sw), K,
                              r.size, _ptr(r), _ptr(c), _ptr(y))
    return y


# --------------------------------------------------------------------------
# Block-wise scales
# --------------------------------------------------------------------------

GROUP = 128   # activation group length along K and weight block edge


def quant_blocks_bf16(x_bits: np.ndarray, br: int, bk: int):
    """Block-wise quantization of bf16 bits [R, K]: one scale per br x bk
    block (partial at the edges).  Returns (codes [R, K], scales
    [ceil(R/br), ceil(K/bk)])."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    R, K = x.shape
    RB, KB = -(-R // br), -(-K // bk)
    q = np.empty((R, K), dtype=np.uint8)
    s = np.empty((RB, KB), dtype=np.float32)
    if R and K:
        lib.orc_quant_blocks_bf16(_ptr(x), R, K, K, br, bk, _ptr(q), K, _ptr(s))
    return q, s


def quant_groups_bf16(x_bits: np.ndarray, group: int = GROUP):
    """Activations: one scale per token per `group` inputs, s [M, ceil(K/group)]."""
    return quant_blocks_bf16(x_bits, 1, group)


def quant_weight_blocks_bf16(w_bits: np.ndarray, block: int = GROUP):
    """Weights: one scale per block x block tile, s [ceil(N/block), ceil(K/block)]."""
    return quant_blocks_bf16(w_bits, block, block)


def gemm_blockwise(qx, s_x, qw, s_w, bn: int = GROUP, bk: int = GROUP,
                   rows=None, cols=None) -> np.ndarray:
    """y = sum_kb s_x[m,kb] s_w[n//bn,kb] (exact block dot product), fp64.
    Full [M, N] output, or the values at the (rows[i], cols[i]) points."""
    lib = _load()
    a = np.ascontiguousarray(qx, dtype=np.uint8)
    b = np.ascontiguousarray(qw, dtype=np.uint8)
    sx = np.ascontiguousarray(s_x, dtype=np.float32)
    sw = np.ascontiguousarray(s_w, dtype=np.float32)
    M, K = a.shape
    N, K2 = b.shape
    assert K == K2
    KB = -(-K // bk)
    assert sx.shape == (M, KB) and sw.shape == (-(-N // bn), KB)
    if rows is None:
        y = np.zeros((M, N), dtype=np.float64)
        if M and N:
            lib.orc_gemm_blockwise(_ptr(a), K, _ptr(sx), _ptr(b), K, _ptr(sw), M, N, K, bn, bk,
                                   0, None, None, _ptr(y))
        return y
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    y = np.zeros(r.shape, dtype=np.float64)
    if r.size:
        lib.orc_gemm_blockwise(_ptr(a), K, _ptr(sx), _ptr(b), K, _ptr(sw), M, N, K, bn, bk,
                               r.size, _ptr(r), _ptr(c), _ptr(y))
    return y


# --------------------------------------------------------------------------
# RMSNorm -> per-token quantization
# --------------------------------------------------------------------------

def rmsnorm_bracket_bf16(x_bits: np.ndarray, g_bits: np.ndarray, eps: float, rel_err: float):
    """bf16 RMSNorm of every row under the fp32 reading, bracketed for a sum
    of squares known to relative rel_err: returns (y_lo, y_hi, ss) where y_lo
    / y_hi are bf16 bits [R, K] (equal wherever the sum's error cannot change
    the rounding) and ss the exact sums of squares (fp64)."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    g = np.ascontiguousarray(g_bits, dtype=np.uint16)
    R, K = x.shape
    assert g.shape == (K,)
    y_lo = np.zeros((R, K), dtype=np.uint16)
    y_hi = np.zeros((R, K), dtype=np.uint16)
    ss = np.zeros(R, dtype=np.float64)
    if R and K:
        lib.orc_rmsnorm_bracket_bf16(_ptr(x), R, K, K, _ptr(g), float(eps), float(rel_err),
                                     _ptr(y_lo), _ptr(y_hi), _ptr(ss))
    return y_lo, y_hi, ss


def rmsnorm_f64(x_bits: np.ndarray, g_bits: np.ndarray, eps: float) -> np.ndarray:
    """The real normalised values (fp64, no intermediate rounding)."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    g = np.ascontiguousarray(g_bits, dtype=np.uint16)
    R, K = x.shape
    y = np.zeros((R, K), dtype=np.float64)
    if R and K:
        lib.orc_rmsnorm_f64(_ptr(x), R, K, K, _ptr(g), float(eps), _ptr(y))
    return y
