"""Helpers shared by the GPU parity tests (test side only)."""
from __future__ import annotations

import numpy as np
import torch

FMT = {"e4m3": 0, "e5m2": 1}


def lib():
    import fp8_quantized_gemm_gb300 as F
    return F


def to_np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(np.uint8)


def f32_bits(v) -> int:
    return int(np.asarray(v, dtype=np.float32).view(np.uint32))


def mx_pack(local_bytes: np.ndarray) -> np.ndarray:
    """Oracle's logical local factors [R, K/32] -> the documented word layout
    int32 [K/128, R_pad]: word (r, g) at g*R_pad + (r & ~127) + 4*(r % 32) +
    (r % 128) // 32 holds in byte j the factor of block 4g + j; padding rows
    hold 127 in every byte."""
    r, nb = local_bytes.shape
    g = nb // 4
    rpad = (r + 127) // 128 * 128
    words = np.full((g, rpad), 0x7F7F7F7F, dtype=np.uint32)
    lb = local_bytes.astype(np.uint32).reshape(r, g, 4)
    packed = lb[:, :, 0] | (lb[:, :, 1] << 8) | (lb[:, :, 2] << 16) | (lb[:, :, 3] << 24)
    rows = np.arange(r)
    pos = (rows & ~127) + 4 * (rows % 32) + (rows % 128) // 32
    words[:, pos] = packed.T
    return words.view(np.int32)


def mx_unpack(words: np.ndarray, r: int, k: int) -> np.ndarray:
    """Inverse of mx_pack for the first r rows: -> uint8 [r, K/32]."""
    w = np.asarray(words).view(np.uint32)
    rows = np.arange(r)
    pos = (rows & ~127) + 4 * (rows % 32) + (rows % 128) // 32
    sel = w[:, pos].T  # [r, G]
    out = np.stack([(sel >> (8 * j)) & 0xFF for j in range(4)], axis=2)
    return out.reshape(r, k // 32).astype(np.uint8)


def sample_positions(m: int, n: int, count: int, seed: int):
    """Output positions to check at full size: random ones plus the corners of
    every edge tile (first/last rows and columns)."""
    rng = np.random.default_rng(seed)
    rows = list(rng.integers(0, m, count))
    cols = list(rng.integers(0, n, count))
    for r in (0, m - 1, min(127, m - 1), min(128, m - 1)):
        for c in (0, n - 1, min(255, n - 1), min(256, n - 1)):
            rows.append(r)
            cols.append(c)
    return np.asarray(rows), np.asarray(cols)
