"""Plain definition of the tile-major token layout the attention path consumes.

TEST INFRASTRUCTURE ONLY (see the package docstring).

GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践"), §1.1: the input
feature map is divided into fixed-size multi-dimensional Q and KV tiles; §2.2:
tokens are permuted before the model and permuted back after it.  The layout
chosen here makes each multi-dimensional tile a contiguous run of rows:

    raster : [B, T, H, W, heads, d]
    tiled  : [B, heads, nT, nH, nW, tT * tH * tW, d],   n_ = ceil(L_ / t_)

Inside a tile the element index is ``(it * tH + iy) * tW + ix``.  Grid
positions past the end of a dimension (the padding of the last tile) hold
zeros.  The per-token ``lse`` uses the same mapping with ``d = 1``.  The value
layout stores every tile of the tiled layout transposed, ``[.., d, 128]``.
"""
from __future__ import annotations

import numpy as np


def tile_counts(dims, tile):
    return tuple(-(-int(L) // int(t)) for L, t in zip(dims, tile))


def permute_reference(x: np.ndarray, tile) -> np.ndarray:
    """Raster ``[B, T, H, W, heads, d]`` -> tiled ``[B, heads, nT, nH, nW, tT*tH*tW, d]``."""
    B, T, H, W, heads, d = x.shape
    tT, tH, tW = tile
    nT, nH, nW = tile_counts((T, H, W), tile)
    padded = np.zeros((B, nT * tT, nH * tH, nW * tW, heads, d), dtype=x.dtype)
    padded[:, :T, :H, :W] = x
    y = padded.reshape(B, nT, tT, nH, tH, nW, tW, heads, d)
    # axes: 0 B, 1 nT, 2 tT, 3 nH, 4 tH, 5 nW, 6 tW, 7 heads, 8 d
    y = y.transpose(0, 7, 1, 3, 5, 2, 4, 6, 8)
    return np.ascontiguousarray(y).reshape(B, heads, nT, nH, nW, tT * tH * tW, d)


def unpermute_reference(y: np.ndarray, dims, tile) -> np.ndarray:
    """Inverse of :func:`permute_reference`: drops the padding."""
    B, heads, nT, nH, nW, e, d = y.shape
    tT, tH, tW = tile
    T, H, W = dims
    z = y.reshape(B, heads, nT, nH, nW, tT, tH, tW, d)
    # back to 0 B, 1 nT, 2 tT, 3 nH, 4 tH, 5 nW, 6 tW, 7 heads, 8 d
    z = z.transpose(0, 2, 5, 3, 6, 4, 7, 1, 8)
    z = np.ascontiguousarray(z).reshape(B, nT * tT, nH * tH, nW * tW, heads, d)
    return np.ascontiguousarray(z[:, :T, :H, :W])


def permute_v_reference(x: np.ndarray, tile) -> np.ndarray:
    """Raster -> value layout ``[B, heads, nT, nH, nW, d, tT*tH*tW]``: every tile of
    :func:`permute_reference` transposed to feature-major."""
    return np.ascontiguousarray(np.swapaxes(permute_reference(x, tile), -1, -2))


def tiled_row(b, h, t, y, x, heads, dims, tile) -> int:
    """Row index of raster token ``(b, t, y, x)``, head ``h``, in the tiled layout."""
    nT, nH, nW = tile_counts(dims, tile)
    tT, tH, tW = tile
    tile_id = ((t // tT) * nH + y // tH) * nW + x // tW
    elem = ((t % tT) * tH + y % tH) * tW + x % tW
    return ((b * heads + h) * (nT * nH * nW) + tile_id) * (tT * tH * tW) + elem
