"""GNA as a differentiable PyTorch operation on raster tensors.

:func:`gna_attention` takes q, k, v in the raster layout ``[B, T, H, W, heads,
head_dim]`` (T = 1 for 2-D grids), returns out in the same layout, and
back-propagates through the library's backward kernels.  It only chains calls
of the C ABI (permutes, the fused forward, the three backward calls) and lets
PyTorch allocate the tiled buffers between them; every value is computed by the
library's CUDA kernels.

GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践") §4.2 (problem 1) and
§5 recommend training with GNA rather than switching it on at inference only;
the backward is the derivative of the forward definition.
"""
from __future__ import annotations

import torch

from . import gna as G


class _GNAFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, window, stride, leader_rule, scale):
        B, T, H, W, heads, d = q.shape
        dims = (T, H, W)
        shp = G.tiled_shape(B, heads, dims, d)
        vshp = G.value_shape(B, heads, dims, d)
        bf = torch.bfloat16
        # the backward also needs v tiled and k in the value layout
        train = any(ctx.needs_input_grad[:3])
        qt, kt = (torch.empty(shp, dtype=bf, device=q.device) for _ in range(2))
        v_value = torch.empty(vshp, dtype=bf, device=q.device)
        for src, dst in ((q, qt), (k, kt)):
            G.gna_permute(src, dst, B, heads, dims, d)
        G.gna_permute_v(v, v_value, B, heads, dims, d)
        vt = k_value = None
        if train:
            vt = torch.empty(shp, dtype=bf, device=q.device)
            k_value = torch.empty(vshp, dtype=bf, device=q.device)
            G.gna_permute(v, vt, B, heads, dims, d)
            G.gna_permute_v(k, k_value, B, heads, dims, d)
        out_t = torch.empty(shp, dtype=bf, device=q.device)
        lse_t = torch.empty(shp[:-1], dtype=torch.float32, device=q.device)
        G.gna_forward(qt, kt, v_value, out_t, lse_t, B, heads, dims, window, stride, d, leader_rule=leader_rule,
                      scale=scale)
        out = torch.empty_like(q)
        G.gna_unpermute(out_t, out, B, heads, dims, d)
        if train:
            ctx.save_for_backward(qt, kt, k_value, vt, out_t, lse_t)
        ctx.geom = (B, heads, dims, d, tuple(window), tuple(stride), leader_rule, scale)
        return out

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(ctx, dout):
        qt, kt, k_value, vt, out_t, lse_t = ctx.saved_tensors
        B, heads, dims, d, window, stride, rule, scale = ctx.geom
        dout = dout.to(torch.bfloat16).contiguous()
        shp = qt.shape
        dout_t = torch.empty(shp, dtype=torch.bfloat16, device=qt.device)
        G.gna_permute(dout, dout_t, B, heads, dims, d)
        delta = torch.empty(shp[:-1], dtype=torch.float32, device=qt.device)
        G.gna_backward_delta(out_t, dout_t, delta, B, heads, dims, d)
        dq_t, dk_t, dv_t = (torch.empty(shp, dtype=torch.bfloat16, device=qt.device) for _ in range(3))
        G.gna_backward_dq(qt, kt, k_value, vt, dout_t, lse_t, delta, dq_t, B, heads, dims, window, stride, d,
                          leader_rule=rule, scale=scale)
        G.gna_backward_dkdv(qt, kt, vt, dout_t, lse_t, delta, dk_t, dv_t, B, heads, dims, window, stride, d,
                            leader_rule=rule, scale=scale)
        grads = []
        for g_t in (dq_t, dk_t, dv_t):
            g = torch.empty(dout.shape, dtype=torch.bfloat16, device=qt.device)
            G.gna_unpermute(g_t, g, B, heads, dims, d)
            grads.append(g)
        return grads[0], grads[1], grads[2], None, None, None, None


def gna_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window, stride=(1, 1, 1), *,
                  leader_rule: int = G.GNA_LEADER_CENTER, scale: float = 0.0) -> torch.Tensor:
    """GNA over raster bf16 tensors ``[B, T, H, W, heads, head_dim]`` (head_dim 32,
    64 or 128), differentiable in q, k and v.  ``window`` and ``stride`` are per
    (T, H, W) dimension; ``scale`` 0 means 1/sqrt(head_dim).  Both passes run
    asynchronously on the current stream; call :func:`gna_get_status` (which
    synchronises) to learn whether a kernel gave up a bounded wait."""
    if q.dim() != 6 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k and v must share one shape [B, T, H, W, heads, head_dim]")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
    return _GNAFunction.apply(q.contiguous(), k.contiguous(), v.contiguous(), tuple(window), tuple(stride),
                              leader_rule, scale)
