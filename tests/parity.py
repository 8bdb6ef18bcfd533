"""Helpers shared by the GPU parity tests: move tensors between the CUDA path
and the CPU oracle, and apply the output tolerance.

Output tolerance (per element, against the fp64 oracle):
    |y_gpu - y_ref| <= 8e-3 * |y_ref| + 1e-3 * rms(y_ref[m, :])
where rms is over the oracle's whole output row m.  bf16 rounding alone is at
most 2^-9 = 1.95e-3 relative, fp32 accumulation and scaling add a few ulps;
the row-rms term absorbs cancellation in outputs near zero.
"""
import numpy as np
import torch

REL_TOL = 8e-3
ROW_TOL = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 bit patterns on the host."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def check_rows(y_gpu: np.ndarray, y_ref: np.ndarray, what: str):
    """y_gpu, y_ref: [rows, N] with full output rows."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    if y_ref.size == 0:
        return
    rms = np.sqrt(np.mean(y_ref * y_ref, axis=1, keepdims=True))
    bound = REL_TOL * np.abs(y_ref) + ROW_TOL * rms
    excess = np.abs(y_gpu - y_ref) - bound
    bad = np.argwhere(excess > 0)
    assert bad.size == 0, (
        f"{what}: {len(bad)} outputs outside tolerance, first at {tuple(bad[0])}: "
        f"gpu={y_gpu[tuple(bad[0])]!r} ref={y_ref[tuple(bad[0])]!r} "
        f"bound={bound[tuple(bad[0])]!r}")


def sample_rows(M: int, count: int, seed: int) -> np.ndarray:
    """Sorted distinct token indices, always including the first and last."""
    if M <= count:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(1, M - 1), size=count - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], mid]))


def tile_rows(M: int, seed: int, block: int = 128) -> np.ndarray:
    """One seeded token from every `block`-row block of M (so both 128-row
    halves of every 256-row tile are checked), plus the first and last."""
    rng = np.random.default_rng(seed)
    starts = np.arange(0, M, block)
    picks = [s + int(rng.integers(0, min(block, M - s))) for s in starts]
    return np.unique(np.concatenate([[0, M - 1], picks]))
