"""The forward on raster Q, K, O and lse (``gna_forward_raster``), and on raster
Q, K, V, O and lse (``gna_forward_raster_all``), against the CPU oracle.

The raster entry point gathers each Q and K tile straight from the token grid,
so its arithmetic is that of the tiled path on the same tiles: every test checks
it against the oracle, and the small ones also check that it is bit-identical to
the tiled path.  Output buffers start as NaN, so a query the kernel skips shows
up, and a guard region past the end of each buffer must stay untouched (padded
tile slots have no raster row and are never written).
"""
import numpy as np
import pytest
import torch

import oracle
from dimensional_sparse_attention_gna_b300 import gna as G
from synthetic_inputs import exact_f32, normal_raster, quantize_e4m3
from tests.gpu_helpers import (REL_RMS_BF16, REL_RMS_FP8, TOL_BF16_LSE, TOL_BF16_OUT, TOL_FP8, bf16_inputs, compare, gpu_gna, oracle_threads,
                               sample_queries)

pytestmark = pytest.mark.gpu

GUARD = 4096          # elements past each output, checked to stay NaN


def gpu_gna_raster(q, k, v, dims, window, stride, *, tile=None, leader_rule=G.GNA_LEADER_CENTER, descale=None,
                   with_lse=True, raster_v=False):
    """Raster CPU tensors -> (out float32 raster [.., heads, d], lse [.., heads] or None), through the raster
    call (V permuted to the value layout), or with ``raster_v`` through the all-raster call (V as it is)."""
    B, T, H, W, heads, d = q.shape
    dev = torch.device("cuda")
    qd, kd = q.to(dev).contiguous(), k.to(dev).contiguous()
    n_rows = B * T * H * W * heads
    out_buf = torch.full((n_rows * d + GUARD,), float("nan"), dtype=torch.bfloat16, device=dev)
    lse_buf = torch.full((n_rows + GUARD,), float("nan"), dtype=torch.float32, device=dev)
    if raster_v:
        assert descale is None
        G.gna_forward_raster_all(qd, kd, v.to(dev).contiguous(), out_buf, lse_buf if with_lse else None, B, heads,
                                 dims, window, stride, d, tile=tile, leader_rule=leader_rule)
    else:
        vt = torch.empty(G.value_shape(B, heads, dims, d, tile), dtype=v.dtype, device=dev)
        G.gna_permute_v(v.to(dev).contiguous(), vt, B, heads, dims, d, tile=tile)
        ds = None if descale is None else torch.tensor(descale, dtype=torch.float32, device=dev)
        G.gna_forward_raster(qd, kd, vt, out_buf, lse_buf if with_lse else None, B, heads, dims, window, stride, d,
                             tile=tile, leader_rule=leader_rule, descale=ds)
    G.gna_get_status()
    torch.cuda.synchronize()
    assert torch.isnan(out_buf[n_rows * d:].float()).all(), "write past the end of out"
    assert torch.isnan(lse_buf[n_rows:]).all(), "write past the end of lse"
    out = out_buf[:n_rows * d].float().cpu().numpy().reshape(B, T, H, W, heads, d)
    lse = lse_buf[:n_rows].cpu().numpy().reshape(B, T, H, W, heads) if with_lse else None
    if not with_lse:
        assert torch.isnan(lse_buf).all()
    return out, lse


@pytest.mark.parametrize("d,dims,window,stride,tile", [
    (128, (5, 19, 23), (3, 9, 11), (1, 1, 1), None),          # every dimension ragged
    (128, (6, 20, 24), (4, 8, 8), (2, 4, 4), None),
    (64, (3, 17, 40), (3, 7, 13), (1, 2, 5), (1, 8, 16)),     # explicit tile, ragged H and W
    (32, (1, 45, 37), (1, 12, 9), (1, 1, 1), None),           # 2-D, the 64-byte swizzle
    (64, (9, 9, 9), (9, 9, 9), (9, 9, 9), (4, 4, 8)),          # window = grid, cubic tile
])
def test_raster_small_grids_all_queries(d, dims, window, stride, tile):
    B, heads = 2, 3
    q, k, v = bf16_inputs(7000 + d + sum(dims), B, dims, heads, d)
    out, lse = gpu_gna_raster(q, k, v, dims, window, stride, tile=tile)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    threads=oracle_threads())
    rel, info = compare(out, lse, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE)
    assert rel < REL_RMS_BF16, info
    out_t, lse_t = gpu_gna(q, k, v, dims, window, stride, tile=tile)
    np.testing.assert_array_equal(out, out_t)
    np.testing.assert_array_equal(lse, lse_t)


def test_raster_literal_rule_and_no_lse():
    dims, window, stride, d = (6, 20, 24), (4, 8, 8), (2, 4, 4), 64
    q, k, v = bf16_inputs(7100, 1, dims, 2, d)
    out, _ = gpu_gna_raster(q, k, v, dims, window, stride, leader_rule=G.GNA_LEADER_LITERAL, with_lse=False)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    rule=oracle.LEADER_LITERAL, threads=oracle_threads())
    compare(out, l_ref.astype(np.float32), o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE)


def test_raster_e4m3_ragged():
    dims, d, heads = (6, 20, 24), 128, 2
    (q, sq), (k, sk), (v, sv) = (quantize_e4m3(normal_raster(7200 + i, 1, dims, heads, d)) for i in range(3))
    out, lse = gpu_gna_raster(q, k, v, dims, (4, 9, 8), (2, 3, 8), descale=(sq, sk, sv))
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, (4, 9, 8), (2, 3, 8),
                                    tensor_scales=(sq, sk, sv), threads=oracle_threads())
    rel, info = compare(out, lse, o_ref, l_ref, TOL_FP8, TOL_FP8)
    assert rel < REL_RMS_FP8, info


@pytest.mark.parametrize("stride", [(1, 1, 1), (16, 8, 8)])
def test_raster_video_720p_latent_sampled(stride):
    """Full-size 3-D video workload (30x48x80 tokens, 24 heads, d=128, window
    16x32x48) through the raster call; sampled queries against the oracle."""
    B, heads, dims, d, window = 1, 24, (30, 48, 80), 128, (16, 32, 48)
    seed = 7300
    q, k, v = bf16_inputs(seed, B, dims, heads, d)
    out, lse = gpu_gna_raster(q, k, v, dims, window, stride)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    rng = np.random.default_rng(seed)
    sel = sample_queries(rng, B, heads, dims, G.gna_tile_shape(dims), 256)
    ids = oracle.query_ids(sel[:, 0], sel[:, 1], sel[:, 2], sel[:, 3], sel[:, 4], heads, dims)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride, sel=ids,
                                    threads=oracle_threads())
    o_gpu = out[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]]
    l_gpu = lse[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]]
    rel, info = compare(o_gpu, l_gpu, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE)
    assert rel < REL_RMS_BF16, info


# ------------------------------------------------------------------ all-raster (V raster too)

@pytest.mark.parametrize("dims,window,stride,tile,rule", [
    ((5, 19, 23), (3, 9, 11), (1, 1, 1), None, G.GNA_LEADER_CENTER),        # every dimension ragged
    ((6, 20, 24), (4, 8, 8), (2, 4, 4), None, G.GNA_LEADER_LITERAL),
    ((3, 17, 40), (3, 7, 13), (1, 2, 5), (1, 8, 16), G.GNA_LEADER_CENTER),  # explicit tile
    ((1, 45, 37), (1, 12, 9), (1, 1, 1), None, G.GNA_LEADER_CENTER),        # 2-D
    ((9, 9, 9), (9, 9, 9), (9, 9, 9), (4, 4, 8), G.GNA_LEADER_CENTER),      # window = grid, runtime tile
])
def test_raster_all_small_grids_all_queries(dims, window, stride, tile, rule):
    """V read token-major straight from the raster layout: every query against
    the oracle (the products differ from the value-layout path only in the order
    the tensor core reads V, so no bit equality is asked)."""
    B, heads, d = 2, 3, 128
    q, k, v = bf16_inputs(7500 + sum(dims), B, dims, heads, d)
    out, lse = gpu_gna_raster(q, k, v, dims, window, stride, tile=tile, leader_rule=rule, raster_v=True)
    orule = oracle.LEADER_CENTER if rule == G.GNA_LEADER_CENTER else oracle.LEADER_LITERAL
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride, rule=orule,
                                    threads=oracle_threads())
    rel, info = compare(out, lse, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE, seed=7500 + sum(dims), dims=list(dims),
                        window=list(window), stride=list(stride), dtype="bf16", heads=heads, B=B, head_dim=d)
    assert rel < REL_RMS_BF16, info


def test_raster_all_coordinate_probe():
    """Q = 0 and V = each key's coordinates: out = the window centre of every query,
    exact, on a grid whose tiles are all padded."""
    from tests.gpu_helpers import coordinate_probe_expected, coordinate_probe_inputs
    dims, window, stride = (6, 20, 24), (4, 9, 8), (2, 3, 8)
    q, k, v = coordinate_probe_inputs(1, dims, 2, 128)
    out, lse = gpu_gna_raster(q, k, v, dims, window, stride, raster_v=True)
    want = [torch.from_numpy(w).to(torch.bfloat16).double().numpy() for w in coordinate_probe_expected(dims, window, stride)]
    np.testing.assert_array_equal(out[..., 0], np.broadcast_to(want[0][None, :, None, None, None], out.shape[:-1]))
    np.testing.assert_array_equal(out[..., 1], np.broadcast_to(want[1][None, None, :, None, None], out.shape[:-1]))
    np.testing.assert_array_equal(out[..., 2], np.broadcast_to(want[2][None, None, None, :, None], out.shape[:-1]))
    assert (out[..., 3:] == 0).all()


@pytest.mark.parametrize("stride", [(1, 1, 1), (16, 8, 8)])
def test_raster_all_video_720p_latent_sampled(stride):
    """Full-size 3-D video workload through the all-raster call; sampled queries."""
    B, heads, dims, d, window = 1, 24, (30, 48, 80), 128, (16, 32, 48)
    seed = 7600
    q, k, v = bf16_inputs(seed, B, dims, heads, d)
    out, lse = gpu_gna_raster(q, k, v, dims, window, stride, raster_v=True)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    rng = np.random.default_rng(seed)
    sel = sample_queries(rng, B, heads, dims, G.gna_tile_shape(dims), 256)
    ids = oracle.query_ids(sel[:, 0], sel[:, 1], sel[:, 2], sel[:, 3], sel[:, 4], heads, dims)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride, sel=ids,
                                    threads=oracle_threads())
    o_gpu = out[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]]
    l_gpu = lse[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]]
    rel, info = compare(o_gpu, l_gpu, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE, seed=seed, dims=list(dims),
                        window=list(window), stride=list(stride), dtype="bf16", heads=heads, B=B, head_dim=d,
                        sampled=True)
    assert rel < REL_RMS_BF16, info
