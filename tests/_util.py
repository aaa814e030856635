"""Shared helpers for the parity tests (comparison rules, conversions)."""
from __future__ import annotations

import numpy as np
import torch

# D tolerance of the block-scaled GEMM (per element, relative to the oracle
# and to the oracle's RMS over the compared elements) and of the global
# cosine-style difference 1 - 2<x,y>/(|x|^2+|y|^2).
RTOL = 1e-2
ATOL_RMS = 1e-2
GLOBAL_DIFF = 1e-4


def u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).cpu().numpy()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def assert_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = "") -> float:
    """Per-element |g - o| <= RTOL*|o| + ATOL_RMS*rms(o) and global diff < GLOBAL_DIFF."""
    g = bits_to_f64(got_bits).ravel()
    o = bits_to_f64(ref_bits).ravel()
    assert g.shape == o.shape
    assert np.isfinite(o).all(), f"{what}: oracle produced non-finite values"
    assert np.isfinite(g).all(), f"{what}: GPU produced non-finite values"
    rms = float(np.sqrt(np.mean(o * o))) if o.size else 0.0
    err = np.abs(g - o)
    bound = RTOL * np.abs(o) + ATOL_RMS * rms
    bad = err > bound
    if bad.any():
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: {int(bad.sum())} of {g.size} elements out of tolerance; "
                             f"worst at flat {i}: gpu {g[i]!r} oracle {o[i]!r} rms {rms:.4g}")
    denom = float((g * g).sum() + (o * o).sum())
    diff = 0.0 if denom == 0 else 1.0 - 2.0 * float((g * o).sum()) / denom
    assert diff < GLOBAL_DIFF, f"{what}: global diff {diff:.3e}"
    return diff


def sb_rows(sfb: torch.Tensor, n: int) -> np.ndarray:
    """128x128 block scales [.., ceil(N/128), sf_k] -> one row per N index (fp64)."""
    s = sfb.double().numpy()
    return s[..., np.arange(n) // 128, :]
