"""The forward with query tiles and key/value tiles of different shapes
(``gna_options.tile_kv``; GNA page §1.2: Q and KV tiles sized independently),
against the CPU oracle.

q, out and lse are tiled with the query tile, k and v with the key/value tile;
each CTA walks the box of KV tiles (in units of the KV tile) that its queries'
windows reach.  Small grids compare every query, including grids where every
tile of both tilings is padded; the 720p-video latent compares sampled queries
under the planner's pair and pins every query's window with the coordinate
probe.  The raster entry points take the same pair.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from dimensional_sparse_attention_gna_b300 import gna as G
from synthetic_inputs import exact_f32, normal_raster, quantize_e4m3
from tests.gpu_helpers import (REL_RMS_BF16, REL_RMS_FP8, TOL_BF16_LSE, TOL_BF16_OUT, TOL_FP8, bf16_inputs, compare,
                               coordinate_probe_expected, coordinate_probe_inputs, gpu_gna, oracle_threads,
                               sample_queries)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,dims,window,stride,tile,tile_kv", [
    (128, (6, 20, 24), (4, 9, 8), (2, 3, 8), (2, 8, 8), (4, 4, 8)),
    (64, (5, 24, 40), (3, 7, 9), (1, 2, 3), (1, 8, 16), (2, 4, 16)),
    (32, (3, 5, 7), (2, 3, 4), (2, 2, 3), (2, 8, 8), (1, 4, 32)),       # every tile of both tilings padded
    (128, (8, 16, 16), (4, 8, 8), (4, 8, 8), (4, 4, 8), (2, 8, 8)),     # blocked
    (64, (1, 37, 45), (1, 11, 13), (1, 1, 1), (1, 8, 16), (1, 16, 8)),  # 2-D sliding window
    (128, (4, 16, 32), (4, 16, 32), (1, 1, 1), (2, 8, 8), (1, 4, 32)),  # window = grid
])
def test_decoupled_small_grids_all_queries(d, dims, window, stride, tile, tile_kv):
    B, heads = 2, 3
    q, k, v = bf16_inputs(9300 + d + sum(dims), B, dims, heads, d)
    out, lse = gpu_gna(q, k, v, dims, window, stride, tile=tile, tile_kv=tile_kv)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    threads=oracle_threads())
    rel, info = compare(out, lse, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE, dims=list(dims), window=list(window),
                        stride=list(stride), heads=heads, B=B, head_dim=d)
    assert rel < REL_RMS_BF16, info


def test_decoupled_literal_leader_rule_and_scale():
    """The pair with the literal leader offset (GNA_LEADER_LITERAL) and a custom
    softmax scale, every query against the oracle."""
    dims, window, stride, d, B, heads = (6, 20, 24), (4, 8, 8), (2, 4, 4), 64, 1, 2
    q, k, v = bf16_inputs(9350, B, dims, heads, d)
    out, lse = gpu_gna(q, k, v, dims, window, stride, tile=(2, 8, 8), tile_kv=(2, 4, 16),
                       leader_rule=G.GNA_LEADER_LITERAL, scale=0.2)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    rule=oracle.LEADER_LITERAL, scale=0.2, threads=oracle_threads())
    rel, info = compare(out, lse, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE, dims=list(dims), window=list(window),
                        stride=list(stride), heads=heads, B=B, head_dim=d)
    assert rel < REL_RMS_BF16, info


def test_decoupled_equal_tiles_match_the_single_tile_call():
    """tile_kv equal to the tile is the single-tile call: bit-identical output."""
    dims, window, stride, d = (6, 20, 24), (4, 9, 8), (2, 3, 8), 64
    q, k, v = bf16_inputs(9400, 1, dims, 2, d)
    a = gpu_gna(q, k, v, dims, window, stride, tile=(2, 8, 8))
    b = gpu_gna(q, k, v, dims, window, stride, tile=(2, 8, 8), tile_kv=(2, 8, 8))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_decoupled_e4m3_ragged():
    dims, window, stride, d, B, heads = (6, 20, 24), (4, 9, 8), (2, 3, 8), 128, 2, 2
    (q, sq), (k, sk), (v, sv) = (quantize_e4m3(normal_raster(9500 + i, B, dims, heads, d)) for i in range(3))
    out, lse = gpu_gna(q, k, v, dims, window, stride, tile=(2, 8, 8), tile_kv=(4, 4, 8), descale=(sq, sk, sv))
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    tensor_scales=(sq, sk, sv), threads=oracle_threads())
    rel, info = compare(out, lse, o_ref, l_ref, TOL_FP8, TOL_FP8, dims=list(dims), window=list(window),
                        stride=list(stride), dtype="fp8", heads=heads, B=B, head_dim=d)
    assert rel < REL_RMS_FP8, info


@pytest.mark.parametrize("raster_v", [False, True])
def test_decoupled_raster_matches_tiled(raster_v):
    """gna_forward_raster (v in the value layout of the KV tile) and
    gna_forward_raster_all with a decoupled pair: the same arithmetic as the
    tiled call, so bit-identical to it, and within the bars of the oracle."""
    dims, window, stride, d, B, heads = (5, 19, 23), (3, 9, 11), (1, 2, 3), 128, 1, 2
    tile, tile_kv = (1, 8, 16), (2, 4, 16)
    q, k, v = bf16_inputs(9600, B, dims, heads, d)
    dev = torch.device("cuda")
    n_rows = B * math.prod(dims) * heads
    out = torch.empty(n_rows * d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(n_rows, dtype=torch.float32, device=dev)
    qd, kd, vd = (x.to(dev).contiguous() for x in (q, k, v))
    if raster_v:
        G.gna_forward_raster_all(qd, kd, vd, out, lse, B, heads, dims, window, stride, d, tile=tile, tile_kv=tile_kv)
    else:
        vt = torch.empty(G.value_shape(B, heads, dims, d, tile_kv), dtype=v.dtype, device=dev)
        G.gna_permute_v(vd, vt, B, heads, dims, d, tile=tile_kv)
        G.gna_forward_raster(qd, kd, vt, out, lse, B, heads, dims, window, stride, d, tile=tile, tile_kv=tile_kv)
    G.gna_get_status()
    torch.cuda.synchronize()
    out_r = out.float().cpu().numpy().reshape(B, *dims, heads, d)
    lse_r = lse.cpu().numpy().reshape(B, *dims, heads)
    out_t, lse_t = gpu_gna(q, k, v, dims, window, stride, tile=tile, tile_kv=tile_kv)
    if not raster_v:
        np.testing.assert_array_equal(out_r, out_t)
        np.testing.assert_array_equal(lse_r, lse_t)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    threads=oracle_threads())
    rel, info = compare(out_r, lse_r, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE, dims=list(dims),
                        window=list(window), stride=list(stride), heads=heads, B=B, head_dim=d)
    assert rel < REL_RMS_BF16, info


@pytest.mark.parametrize("stride", [(8, 8, 8), (16, 8, 8)])
def test_decoupled_video_720p_planned_pair(stride):
    """The 720p-video latent (30x48x80, window 16x32x48) with the pair
    gna_plan_tiles picks (it visits fewer tile pairs than any single tile at
    these strides): sampled queries against the oracle, 2 heads."""
    dims, window, d, B, heads, seed = (30, 48, 80), (16, 32, 48), 128, 1, 2, 9700
    tile, tile_kv, overhead, _ = G.gna_plan_tiles(dims, window, stride)
    assert tile != tile_kv and overhead < G.gna_plan_tile(dims, window, stride)[1]
    q, k, v = bf16_inputs(seed, B, dims, heads, d)
    out, lse = gpu_gna(q, k, v, dims, window, stride, tile=tile, tile_kv=tile_kv)
    sel = sample_queries(np.random.default_rng(seed), B, heads, dims, tile, 256)
    ids = oracle.query_ids(sel[:, 0], sel[:, 1], sel[:, 2], sel[:, 3], sel[:, 4], heads, dims)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride, sel=ids,
                                    threads=oracle_threads())
    o_gpu = out[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]]
    l_gpu = lse[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]]
    rel, info = compare(o_gpu, l_gpu, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE, seed=seed, dims=list(dims),
                        window=list(window), stride=list(stride), heads=heads, B=B, head_dim=d, sampled=True,
                        tile=list(tile), tile_kv=list(tile_kv))
    assert rel < REL_RMS_BF16, info


@pytest.mark.parametrize("stride,tile,tile_kv", [
    ((16, 8, 8), (2, 8, 8), (2, 4, 16)),
    ((1, 1, 1), (2, 8, 8), (4, 4, 8)),
    ((8, 8, 8), (1, 8, 16), (4, 4, 8)),
])
def test_decoupled_video_720p_coordinate_probe(stride, tile, tile_kv):
    """Every query of the 720p-video latent lands on exactly its window under a
    decoupled pair (Q = 0: out = the window's mean key coordinate, exact in bf16)."""
    dims, window, d = (30, 48, 80), (16, 32, 48), 128
    q, k, v = coordinate_probe_inputs(1, dims, 2, d)
    out, lse = gpu_gna(q, k, v, dims, window, stride, tile=tile, tile_kv=tile_kv)
    want = [torch.from_numpy(w).to(torch.bfloat16).double().numpy()
            for w in coordinate_probe_expected(dims, window, stride)]
    np.testing.assert_array_equal(out[..., 0], np.broadcast_to(want[0][None, :, None, None, None], out.shape[:-1]))
    np.testing.assert_array_equal(out[..., 1], np.broadcast_to(want[1][None, None, :, None, None], out.shape[:-1]))
    np.testing.assert_array_equal(out[..., 2], np.broadcast_to(want[2][None, None, None, :, None], out.shape[:-1]))
    assert (out[..., 3:] == 0).all()
    np.testing.assert_allclose(lse, math.log(np.prod(window)), rtol=0, atol=2e-5)
