"""Seeded synthetic inputs shared by the tests, the bench and the oracle runs.

This module only draws random numbers and converts them to the storage types
the attention path consumes (bf16, or e4m3 codes with a per-tensor scale).  It
holds none of the attention arithmetic: no window rule, no softmax, no layout
change.  Both the CUDA path and the CPU oracle read the tensors it returns, so
the two sides see identical bytes.

Raster layout of every token tensor: ``[B, T, H, W, heads, d]`` (token-major,
heads innermost before the feature dim), the layout a video/image transformer's
QKV projection produces.  A 2-D image grid is ``T = 1``.
"""
from __future__ import annotations

import numpy as np
import torch

#: Base of the per-workload seeds; workload ``n`` uses ``SEED_BASE + n`` and
#: the three tensors Q, K, V use that seed + 0, + 1, + 2.
SEED_BASE = 20261202

#: Largest finite magnitude of float8 e4m3 (OCP "fn" variant).
E4M3_MAX = 448.0


def normal_raster(seed: int, B: int, dims, heads: int, head_dim: int) -> np.ndarray:
    """iid N(0, 1) float32 array of shape ``[B, T, H, W, heads, head_dim]``."""
    T, H, W = (int(x) for x in dims)
    rng = np.random.default_rng(int(seed))
    return rng.standard_normal((B, T, H, W, heads, head_dim), dtype=np.float32)


def qkv_normal(workload_index: int, B: int, dims, heads: int, head_dim: int):
    """Q, K, V float32 rasters for one workload, seeds (s, s+1, s+2)."""
    s = SEED_BASE + int(workload_index)
    return tuple(normal_raster(s + i, B, dims, heads, head_dim) for i in range(3))


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """Round float32 values to bf16 (round-to-nearest-even, torch's CPU cast)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def quantize_e4m3(x: np.ndarray):
    """Per-tensor amax scaling to float8 e4m3.

    Returns ``(codes, scale)`` with ``codes`` a ``torch.float8_e4m3fn`` tensor
    and ``scale = amax / 448`` so that ``codes.float() * scale`` approximates
    ``x``.  The cast is torch's CPU conversion (round-to-nearest-even); the
    scaled values never exceed 448 in magnitude, so no saturation occurs.
    """
    t = torch.from_numpy(np.ascontiguousarray(x))
    amax = float(t.abs().max())
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    codes = (t / scale).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return codes, scale


def exact_f32(t: torch.Tensor) -> np.ndarray:
    """The exact values a bf16 tensor (or the codes of an e4m3 tensor) holds, as float32.

    Every bf16 and e4m3 value is exactly representable in float32.  For e4m3
    the per-tensor scale is applied separately, in float64, by the consumer.
    """
    return t.to(torch.float32).numpy()
