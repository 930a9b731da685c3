"""Plain, slow CPU definition of the Generalized Neighborhood Attention forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library.

Everything here is written for a reader checking it against the sources by eye;
it is float64 throughout and makes no attempt to be fast.  Citations name the
web page by its title and the section on it:

* GNA page -- "GNA稀疏注意力机制：视觉Transformer计算优化实践":
  §1.1 (core design): a per-dimension stride moves each query's window of keys
  between the sliding-window mode (stride 1, neighborhood attention, which is
  translation equivariant) and the blocked mode (stride > 1: the window moves in
  jumps, giving block / checkerboard patterns); queries attend only to keys in
  their window.  §1.2 (complexity): each query processes k keys, O(n k).
* Video tutorial page -- "视频生成推理提速:稀疏注意力组合配置教程", §3.3:
  memory-efficient attention accumulates the softmax block by block and never
  materialises the n x n matrix; its result is that of plain softmax attention.
* Sparse-attention page -- "稀疏注意力机制：提升AI模型效率的关键技术", §2.1:
  sliding-window local attention, each token attends to a fixed range of
  neighbours, O(n w).

Readings taken where the pages are silent (each is a named constant or a
parameter so the alternative can be run):

* Stride groups.  Queries are split, per dimension, into consecutive groups of
  ``s`` positions; all queries of a group share the window of the group's
  leader.  The leader is the group's centre, offset ``floor(s/2)`` from the
  group's first position (``LEADER_CENTER``), clipped to the last position.
  With this offset, stride = window on a grid divisible by the window gives
  exactly independent attention inside each block (the blocked mode of §1.1).
  The alternative offset ``floor((s-1)/2)`` (``LEADER_LITERAL``) agrees for
  odd strides and is kept for comparison.
* Window placement.  The window of ``w`` positions puts ``floor(w/2)`` positions
  before the leader, and is shifted to stay inside ``[0, L)``.
* Scale ``1/sqrt(head_dim)``; no causal mask, no dilation.
* ``lse`` is the natural-log sum of exponentials of the scaled scores.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch

LEADER_CENTER = "center"
LEADER_LITERAL = "literal"


def leader(i: int, L: int, s: int, rule: str = LEADER_CENTER) -> int:
    """Position of the stride-group leader of position ``i`` in one dimension."""
    off = s // 2 if rule == LEADER_CENTER else (s - 1) // 2
    return min((i // s) * s + off, L - 1)


def window_start(i: int, L: int, w: int, s: int, rule: str = LEADER_CENTER) -> int:
    """First key position of the window of query position ``i`` (one dimension)."""
    c = leader(i, L, s, rule)
    return min(max(c - w // 2, 0), L - w)


def check_geometry(dims, window, stride):
    for L, w, s in zip(dims, window, stride):
        if not (1 <= s <= w <= L):
            raise ValueError(f"need 1 <= stride <= window <= length, got s={s} w={w} L={L}")


def neighborhood(idx, dims, window, stride, rule: str = LEADER_CENTER):
    """All key multi-indices ``(t, y, x)`` in the window of query ``idx``."""
    ranges = []
    for i, L, w, s in zip(idx, dims, window, stride):
        a = window_start(i, L, w, s, rule)
        ranges.append(range(a, a + w))
    return list(itertools.product(*ranges))


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def gna_forward_loops(q, k, v, dims, window, stride, scale=None, rule=LEADER_CENTER,
                      tensor_scales=(1.0, 1.0, 1.0)):
    """GNA forward by its definition, one query at a time.

    ``q, k, v``: arrays ``[B, T, H, W, heads, d]`` (any real dtype).  The values
    used are ``q * tensor_scales[0]`` etc. (per-tensor dequantisation scales; 1
    for bf16 inputs).  Returns ``out [B, T, H, W, heads, d]`` and
    ``lse [B, T, H, W, heads]`` in float64.

    For each query i with neighbourhood N(i):
        s_ij  = scale * <q_i, k_j>
        lse_i = log sum_{j in N(i)} exp(s_ij)
        out_i = sum_{j in N(i)} exp(s_ij - lse_i) v_j
    computed with the max subtracted before exponentiating (two passes).
    Pure-Python loop over queries: small grids only.
    """
    check_geometry(dims, window, stride)
    q = np.asarray(q, dtype=np.float64) * tensor_scales[0]
    k = np.asarray(k, dtype=np.float64) * tensor_scales[1]
    v = np.asarray(v, dtype=np.float64) * tensor_scales[2]
    B, T, H, W, heads, d = q.shape
    assert (T, H, W) == tuple(dims)
    if scale is None:
        scale = default_scale(d)
    out = np.zeros_like(q)
    lse = np.zeros((B, T, H, W, heads))
    for b in range(B):
        for idx in itertools.product(range(T), range(H), range(W)):
            keys = neighborhood(idx, dims, window, stride, rule)
            kt, ky, kx = (np.array(c) for c in zip(*keys))
            for h in range(heads):
                kk = k[b, kt, ky, kx, h]          # [|N|, d]
                vv = v[b, kt, ky, kx, h]
                s = scale * (kk @ q[(b,) + idx + (h,)])
                m = s.max()
                e = np.exp(s - m)
                z = e.sum()
                lse[(b,) + idx + (h,)] = m + math.log(z)
                out[(b,) + idx + (h,)] = (e / z) @ vv
    return out, lse


def softmax_backward(p: np.ndarray, dp: np.ndarray) -> np.ndarray:
    """Gradient of the scores from the gradient of the probabilities.

    For p = softmax(s), the Jacobian dp_j/ds_l = p_j (delta_jl - p_l), so
    ds_l = p_l (dp_l - sum_j p_j dp_j).
    """
    return p * (dp - (p * dp).sum())


def gna_backward_loops(q, k, v, dout, dims, window, stride, scale=None, rule=LEADER_CENTER):
    """Gradients of the GNA forward, one query at a time (float64).

    The GNA page asks for training with GNA in the loop (§4.2, problem 1: add
    GNA during training, not only at inference; §5: fold GNA into training) but
    writes no backward pass.  The reading taken here: the backward is the
    derivative of the forward definition above.  For the loss
    ``L = sum_i <dout_i, out_i>`` it returns ``dL/dq, dL/dk, dL/dv``, arrays
    ``[B, T, H, W, heads, d]``.  With p_ij = exp(s_ij - lse_i) for j in N(i):

        dv_j  += p_ij dout_i                        (out_i is linear in v_j)
        dp_ij  = <dout_i, v_j>
        ds_ij  = p_ij (dp_ij - sum_l p_il dp_il)    (softmax Jacobian)
        dq_i   = scale sum_j ds_ij k_j
        dk_j  += scale ds_ij q_i

    A key collects from every query whose window holds it.  Pure-Python loop
    over queries: small grids only.
    """
    check_geometry(dims, window, stride)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    B, T, H, W, heads, d = q.shape
    assert (T, H, W) == tuple(dims) and k.shape == q.shape and v.shape == q.shape and dout.shape == q.shape
    if scale is None:
        scale = default_scale(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for idx in itertools.product(range(T), range(H), range(W)):
            keys = neighborhood(idx, dims, window, stride, rule)
            kt, ky, kx = (np.array(c) for c in zip(*keys))
            for h in range(heads):
                qi = q[(b,) + idx + (h,)]
                doi = dout[(b,) + idx + (h,)]
                kk = k[b, kt, ky, kx, h]          # [|N|, d]
                vv = v[b, kt, ky, kx, h]
                s = scale * (kk @ qi)
                e = np.exp(s - s.max())
                p = e / e.sum()
                dp = vv @ doi
                ds = softmax_backward(p, dp)
                dq[(b,) + idx + (h,)] = scale * (ds @ kk)
                # keys of one window are distinct, so these scatters never collide
                dk[b, kt, ky, kx, h] += scale * ds[:, None] * qi[None, :]
                dv[b, kt, ky, kx, h] += p[:, None] * doi[None, :]
    return dq, dk, dv


def window_mask(dims, window, stride, rule=LEADER_CENTER) -> np.ndarray:
    """Boolean ``[N, N]`` matrix, ``mask[i, j]`` true iff key j is in the window of query i.

    Tokens are numbered in raster order ``(t * H + y) * W + x``.  Built from the
    per-dimension window starts: key j is in the window iff, in every dimension,
    ``start(i) <= j_d < start(i) + w``.
    """
    check_geometry(dims, window, stride)
    T, H, W = dims
    per_dim = []
    for L, w, s in zip(dims, window, stride):
        st = np.array([window_start(i, L, w, s, rule) for i in range(L)])
        j = np.arange(L)
        per_dim.append((j[None, :] >= st[:, None]) & (j[None, :] < st[:, None] + w))
    mt, my, mx = per_dim
    m = (mt[:, None, None, :, None, None] & my[None, :, None, None, :, None]
         & mx[None, None, :, None, None, :])
    n = T * H * W
    return m.reshape(n, n)


def gna_forward_masked_dense(q, k, v, dims, window, stride, scale=None, rule=LEADER_CENTER,
                             tensor_scales=(1.0, 1.0, 1.0)):
    """The same quantity as dense softmax attention with a boolean window mask (torch, float64).

    A second, independent formulation for small grids: scores for all pairs,
    ``-inf`` outside the window, then ``logsumexp`` / ``softmax`` and a matrix
    product.  Same argument and return conventions as :func:`gna_forward_loops`.
    """
    q = torch.as_tensor(np.asarray(q), dtype=torch.float64) * tensor_scales[0]
    k = torch.as_tensor(np.asarray(k), dtype=torch.float64) * tensor_scales[1]
    v = torch.as_tensor(np.asarray(v), dtype=torch.float64) * tensor_scales[2]
    B, T, H, W, heads, d = q.shape
    if scale is None:
        scale = default_scale(d)
    n = T * H * W
    mask = torch.from_numpy(window_mask(dims, window, stride, rule))
    qf = q.reshape(B, n, heads, d).permute(0, 2, 1, 3)   # [B, heads, n, d]
    kf = k.reshape(B, n, heads, d).permute(0, 2, 1, 3)
    vf = v.reshape(B, n, heads, d).permute(0, 2, 1, 3)
    s = scale * (qf @ kf.transpose(-1, -2))
    s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)                     # [B, heads, n]
    p = torch.exp(s - lse[..., None])
    out = p @ vf                                         # [B, heads, n, d]
    out = out.permute(0, 2, 1, 3).reshape(B, T, H, W, heads, d)
    lse = lse.permute(0, 2, 1).reshape(B, T, H, W, heads)
    return out.numpy(), lse.numpy()


def useful_flops(B, heads, dims, window, head_dim) -> int:
    """Work of the window only: 2 flops per multiply-add in QK^T and in PV.

    GNA page §1.2: every query processes |window| keys, so the work is
    ``4 * B * heads * N * |window| * d``.
    """
    n = int(np.prod(dims))
    return 4 * B * heads * n * int(np.prod(window)) * head_dim
