"""Parity of the CUDA GNA forward (through the C ABI) with the CPU oracle.

Small grids compare every query; the full-size workloads (4K-image latent
256x256, 720p-video latent 30x48x80) compare sampled queries the oracle computes
one by one, plus a structured probe that checks every query exactly: with
Q = 0 every score is 0, so out_i is the mean of V over i's window; with V
holding each key's (t, y, x) coordinates that mean is start_d(i) + (w_d-1)/2,
exact in bf16, which pins the window of every single query.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from dimensional_sparse_attention_gna_b300 import gna as G
from synthetic_inputs import exact_f32, normal_raster, quantize_e4m3, to_bf16
from tests.gpu_helpers import (REL_RMS_BF16, REL_RMS_FP8, TOL_BF16_LSE, TOL_BF16_OUT, TOL_FP8, bf16_inputs, compare,
                               coordinate_probe_expected, coordinate_probe_inputs, gpu_gna, oracle_threads,
                               sample_queries)

pytestmark = pytest.mark.gpu


def _full_parity(B, heads, dims, d, window, stride, seed, tile=None, rule=oracle.LEADER_CENTER):
    q, k, v = bf16_inputs(seed, B, dims, heads, d)
    out, lse = gpu_gna(q, k, v, dims, window, stride, tile=tile,
                       leader_rule=G.GNA_LEADER_CENTER if rule == oracle.LEADER_CENTER else G.GNA_LEADER_LITERAL)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride, rule=rule,
                                    threads=oracle_threads())
    rel, info = compare(out, lse, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE, seed=seed, dims=list(dims),
                        window=list(window), stride=list(stride), dtype="bf16", heads=heads, B=B, head_dim=d)
    assert rel < REL_RMS_BF16, info


def test_tiny_2d_config():
    """2-D tiny: B=1, 2 heads, 16x16, d=32, window 5x5, stride 1 (fp32 inputs rounded to bf16)."""
    _full_parity(1, 2, (1, 16, 16), 32, (1, 5, 5), (1, 1, 1), seed=20261202)


@pytest.mark.parametrize("d", [32, 64, 128])
@pytest.mark.parametrize("dims,window,stride", [
    ((3, 5, 7), (2, 3, 4), (2, 2, 3)),          # ragged: every tile padded
    ((6, 20, 24), (4, 9, 8), (2, 3, 8)),        # several tiles, ragged tail
    ((1, 37, 45), (1, 11, 13), (1, 1, 1)),      # 2-D sliding window
])
def test_small_grids_all_queries(d, dims, window, stride):
    _full_parity(2, 3, dims, d, window, stride, seed=1000 + d)


@pytest.mark.parametrize("dims,window,stride,tile", [
    ((4, 16, 32), (4, 16, 32), (1, 1, 1), None),        # window = grid: dense attention
    ((4, 16, 32), (2, 8, 8), (2, 8, 8), None),          # blocked, tile-aligned: no masks
    ((8, 16, 16), (4, 8, 8), (4, 8, 8), (4, 4, 8)),     # blocked, another tile
    ((5, 24, 40), (3, 7, 9), (1, 2, 3), (1, 8, 16)),
    ((5, 24, 40), (3, 7, 9), (1, 2, 3), (2, 4, 16)),
    ((2, 40, 40), (1, 40, 3), (1, 1, 1), (1, 1, 128)),  # tile wider than 32 columns
    ((1, 64, 64), (1, 17, 33), (1, 4, 8), (1, 4, 32)),
])
def test_window_modes_and_tiles(dims, window, stride, tile):
    _full_parity(1, 2, dims, 64, window, stride, seed=2000, tile=tile)


def test_literal_leader_rule():
    _full_parity(1, 2, (6, 20, 24), 64, (4, 8, 8), (2, 4, 4), seed=3000, rule=oracle.LEADER_LITERAL)


def test_custom_scale():
    dims, window, stride = (2, 16, 16), (2, 5, 5), (1, 1, 1)
    q, k, v = bf16_inputs(3100, 1, dims, 2, 64)
    out, lse = gpu_gna(q, k, v, dims, window, stride, scale=0.3)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride, scale=0.3)
    compare(out, lse, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE)


def _coordinate_probe(B, heads, dims, d, window, stride, dtype=torch.bfloat16, descale=None):
    q, k, v = coordinate_probe_inputs(B, dims, heads, d, dtype)
    out, lse = gpu_gna(q, k, v, dims, window, stride, descale=descale)
    # the kernel forms the mean exactly in fp32 and rounds once to bf16
    # (round-to-nearest-even), so the expectation is rounded the same way
    want = [torch.from_numpy(w).to(torch.bfloat16).double().numpy()
            for w in coordinate_probe_expected(dims, window, stride)]
    T, H, W = dims
    np.testing.assert_array_equal(out[..., 0], np.broadcast_to(want[0][None, :, None, None, None], out.shape[:-1]))
    np.testing.assert_array_equal(out[..., 1], np.broadcast_to(want[1][None, None, :, None, None], out.shape[:-1]))
    np.testing.assert_array_equal(out[..., 2], np.broadcast_to(want[2][None, None, None, :, None], out.shape[:-1]))
    assert (out[..., 3:] == 0).all()
    np.testing.assert_allclose(lse, math.log(np.prod(window)), rtol=0, atol=2e-5)


@pytest.mark.parametrize("dims,window,stride", [
    ((1, 16, 16), (1, 5, 5), (1, 1, 1)),
    ((3, 5, 7), (2, 3, 4), (2, 2, 3)),
    ((6, 20, 24), (4, 9, 8), (2, 3, 8)),
])
def test_coordinate_probe_small(dims, window, stride):
    _coordinate_probe(1, 2, dims, 128, window, stride)


# ------------------------------------------------------------------ full-size workloads

def _sampled_parity(B, heads, dims, d, window, stride, seed, n_random, dtype="bf16"):
    tile = G.gna_tile_shape(dims)
    if dtype == "bf16":
        q, k, v = bf16_inputs(seed, B, dims, heads, d)
        scales = (1.0, 1.0, 1.0)
        descale = None
        tol_out, tol_lse = TOL_BF16_OUT, TOL_BF16_LSE
    else:
        qs = [quantize_e4m3(normal_raster(seed + i, B, dims, heads, d)) for i in range(3)]
        (q, sq), (k, sk), (v, sv) = qs
        scales = (sq, sk, sv)
        descale = scales
        tol_out = tol_lse = TOL_FP8
    out, lse = gpu_gna(q, k, v, dims, window, stride, descale=descale)
    rng = np.random.default_rng(seed)
    sel = sample_queries(rng, B, heads, dims, tile, n_random)
    ids = oracle.query_ids(sel[:, 0], sel[:, 1], sel[:, 2], sel[:, 3], sel[:, 4], heads, dims)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    tensor_scales=scales, sel=ids, threads=oracle_threads())
    o_gpu = out[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]]
    l_gpu = lse[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]]
    rel, info = compare(o_gpu, l_gpu, o_ref, l_ref, tol_out, tol_lse, seed=seed, dims=list(dims),
                        window=list(window), stride=list(stride), dtype=dtype, heads=heads, B=B, head_dim=d,
                        sampled=True)
    print(f"{dims} w={window} s={stride} {dtype}: {info}")
    assert rel < (REL_RMS_BF16 if dtype == "bf16" else REL_RMS_FP8), info


@pytest.mark.parametrize("stride", [(1, 1, 1), (1, 16, 16)])
def test_image_4k_latent(stride):
    """2-D image GNA: 256x256 tokens, 24 heads, d=128, window 64x64."""
    _sampled_parity(1, 24, (1, 256, 256), 128, (1, 64, 64), stride, seed=20261203, n_random=1024)


@pytest.mark.parametrize("stride", [(1, 1, 1), (16, 8, 8)])
def test_video_720p_latent(stride):
    """3-D video GNA: 30x48x80 tokens, 24 heads, d=128, window 16x32x48."""
    _sampled_parity(1, 24, (30, 48, 80), 128, (16, 32, 48), stride, seed=20261204, n_random=512)


@pytest.mark.parametrize("stride", [(1, 1, 1), (16, 8, 8)])
def test_video_720p_latent_fp8(stride):
    """FP8 3-D video GNA, B=2: e4m3 Q/K/V with per-tensor amax scales, bf16 out."""
    _sampled_parity(2, 24, (30, 48, 80), 128, (16, 32, 48), stride, seed=20261206, n_random=256, dtype="fp8")


@pytest.mark.parametrize("stride,window", [
    ((2, 4, 4), (16, 32, 48)), ((4, 8, 8), (16, 32, 48)), ((8, 8, 8), (16, 32, 48)), ((16, 32, 48), (16, 32, 48)),
    ((1, 1, 1), (30, 48, 80)),
])
def test_video_stride_sweep_random_inputs(stride, window):
    """The 3-D stride sweep on the full 30x48x80 grid with random N(0,1) inputs
    (2 heads; strides 1x1x1 and 16x8x8 run at 24 heads above): sampled queries
    against the oracle, so that the running maximum, the lazy rescale and the
    partial-tile masks meet real scores at every sweep geometry, window = grid
    (dense attention) included."""
    _sampled_parity(1, 2, (30, 48, 80), 128, window, stride, seed=20261205, n_random=256)


@pytest.mark.parametrize("stride,window", [
    ((1, 1, 1), (16, 32, 48)), ((2, 4, 4), (16, 32, 48)), ((4, 8, 8), (16, 32, 48)), ((8, 8, 8), (16, 32, 48)),
    ((16, 8, 8), (16, 32, 48)), ((16, 32, 48), (16, 32, 48)), ((1, 1, 1), (30, 48, 80)),
])
def test_video_stride_sweep_coordinate_probe(stride, window):
    """Every query of the 3-D stride sweep lands on exactly its window (exact check)."""
    _coordinate_probe(1, 2, (30, 48, 80), 128, window, stride)


@pytest.mark.parametrize("stride", [(1, 1, 1), (1, 16, 16)])
def test_image_coordinate_probe(stride):
    _coordinate_probe(1, 2, (1, 256, 256), 128, (1, 64, 64), stride)


# ------------------------------------------------------------------ failure detection

def test_abandoned_wait_reports_timeout_and_context_survives():
    """A producer that skips one KV load leaves the consumers waiting; their bounded
    waits give up, the kernel exits, and the host reads GNA_ERR_TIMEOUT.  The next
    call on the same context works."""
    dims, window, stride = (1, 16, 16), (1, 5, 5), (1, 1, 1)
    q, k, v = bf16_inputs(4000, 1, dims, 1, 32)
    G.gna_test_skip_kv_load(0, 1)
    try:
        with pytest.raises(G.GNAError) as ei:
            gpu_gna(q, k, v, dims, window, stride)
        assert ei.value.status == G.GNA_ERR_TIMEOUT
    finally:
        G.gna_test_skip_kv_load(0, -1)
    G.gna_get_status()   # cleared
    out, lse = gpu_gna(q, k, v, dims, window, stride)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride)
    compare(out, lse, o_ref, l_ref, TOL_BF16_OUT, TOL_BF16_LSE)
