"""Edge cases of the CUDA GNA forward against the CPU oracle, every query compared.

Degenerate windows and grids, grids where every tile is padded, a head count far
above the workloads', e4m3 on a ragged grid, and scores large enough that the
running maximum jumps by many powers of two between KV tiles (the lazy rescale
and its overflow guard).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic_inputs import exact_f32, normal_raster, quantize_e4m3, to_bf16
from tests.gpu_helpers import (REL_RMS_BF16, REL_RMS_FP8, TOL_BF16_LSE, TOL_BF16_OUT, TOL_FP8, bf16_inputs, compare,
                               gpu_gna, oracle_threads)

pytestmark = pytest.mark.gpu


def _parity(q, k, v, dims, window, stride, scales=(1.0, 1.0, 1.0), tol_out=TOL_BF16_OUT, tol_lse=TOL_BF16_LSE,
            descale=None):
    out, lse = gpu_gna(q, k, v, dims, window, stride, descale=descale)
    o_ref, l_ref = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    tensor_scales=scales, threads=oracle_threads())
    rel, info = compare(out, lse, o_ref, l_ref, tol_out, tol_lse)
    return out, lse, rel, info


def test_unit_window_returns_own_value_exactly():
    """w = 1 in every dimension: each query sees only its own key, so out = v
    (exact: one weight of 1, one bf16 rounding of an exact bf16 value) and
    lse = scale * <q, k> of that key."""
    dims, d = (3, 9, 11), 64
    q, k, v = bf16_inputs(5000, 2, dims, 3, d)
    out, lse, _, info = _parity(q, k, v, dims, (1, 1, 1), (1, 1, 1))
    np.testing.assert_array_equal(out, v.float().numpy())
    qk = (q.double() * k.double()).sum(-1).numpy() / math.sqrt(d)
    np.testing.assert_allclose(lse, qk, rtol=0, atol=2e-4)


def test_single_token_grid():
    dims = (1, 1, 1)
    q, k, v = bf16_inputs(5001, 3, dims, 2, 128)
    out, lse, _, _ = _parity(q, k, v, dims, (1, 1, 1), (1, 1, 1))
    np.testing.assert_array_equal(out, v.float().numpy())


@pytest.mark.parametrize("dims,window,stride", [
    ((1, 1, 300), (1, 1, 37), (1, 1, 5)),        # a 1-D sequence as a degenerate grid
    ((1, 300, 1), (1, 64, 1), (1, 8, 1)),
    ((5, 19, 23), (2, 4, 6), (2, 4, 6)),          # blocked, grid not divisible by the window
    ((4, 16, 20), (4, 5, 20), (1, 2, 1)),         # window = grid in two dimensions only
    ((7, 3, 2), (7, 3, 2), (7, 3, 2)),            # one block covering a tiny grid
])
def test_degenerate_geometries(dims, window, stride):
    q, k, v = bf16_inputs(5100 + sum(dims), 1, dims, 2, 64)
    _, _, rel, info = _parity(q, k, v, dims, window, stride)
    assert rel < REL_RMS_BF16, info


def test_every_tile_padded_many_batches():
    dims = (3, 5, 7)                               # default tile pads every dimension
    q, k, v = bf16_inputs(5200, 3, dims, 1, 128)
    _, _, rel, info = _parity(q, k, v, dims, (3, 3, 5), (1, 2, 2))
    assert rel < REL_RMS_BF16, info


def test_many_heads():
    dims = (1, 8, 24)
    q, k, v = bf16_inputs(5300, 1, dims, 64, 64)
    _, _, rel, info = _parity(q, k, v, dims, (1, 5, 9), (1, 1, 3))
    assert rel < REL_RMS_BF16, info


def test_e4m3_ragged_grid_all_queries():
    dims, d, heads = (6, 20, 24), 128, 2
    qs = [quantize_e4m3(normal_raster(5400 + i, 1, dims, heads, d)) for i in range(3)]
    (q, sq), (k, sk), (v, sv) = qs
    _, _, rel, info = _parity(q, k, v, dims, (4, 9, 8), (2, 3, 8), scales=(sq, sk, sv), tol_out=TOL_FP8,
                              tol_lse=TOL_FP8, descale=(sq, sk, sv))
    assert rel < REL_RMS_FP8, info


@pytest.mark.parametrize("amp", [6.0, 24.0])
def test_large_scores_lazy_rescale(amp):
    """Q scaled up so that the scores' spread is dozens of natural units: the
    row maximum keeps jumping between KV tiles, forcing O rescales; with amp 24
    a jump can exceed 2^64 and the reference must never overflow."""
    dims, d = (4, 16, 32), 128
    q32 = normal_raster(5500, 1, dims, 2, d) * amp
    q = to_bf16(q32)
    k = to_bf16(normal_raster(5501, 1, dims, 2, d))
    v = to_bf16(normal_raster(5502, 1, dims, 2, d))
    out, lse, rel, info = _parity(q, k, v, dims, (3, 9, 17), (1, 1, 1), tol_lse=1e-2 * amp)
    assert rel < REL_RMS_BF16, info


def test_without_lse_and_on_a_side_stream():
    """lse = NULL writes the same out; the call runs on the stream it is given."""
    from dimensional_sparse_attention_gna_b300 import gna as G
    dims, window, stride, d = (4, 16, 24), (3, 9, 11), (1, 2, 3), 64
    q, k, v = bf16_inputs(5600, 1, dims, 2, d)
    out_ref, lse_ref = gpu_gna(q, k, v, dims, window, stride)
    dev = torch.device("cuda")
    B, heads = 1, 2
    shp = G.tiled_shape(B, heads, dims, d)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        qt, kt = (torch.empty(shp, dtype=torch.bfloat16, device=dev) for _ in range(2))
        vt = torch.empty(G.value_shape(B, heads, dims, d), dtype=torch.bfloat16, device=dev)
        G.gna_permute(q.to(dev), qt, B, heads, dims, d, stream=side)
        G.gna_permute(k.to(dev), kt, B, heads, dims, d, stream=side)
        G.gna_permute_v(v.to(dev), vt, B, heads, dims, d, stream=side)
        out_t = torch.empty(shp, dtype=torch.bfloat16, device=dev)
        G.gna_forward(qt, kt, vt, out_t, None, B, heads, dims, window, stride, d, stream=side)
        out = torch.empty((B,) + dims + (heads, d), dtype=torch.bfloat16, device=dev)
        G.gna_unpermute(out_t, out, B, heads, dims, d, stream=side)
    side.synchronize()
    G.gna_get_status(side)
    np.testing.assert_array_equal(out.float().cpu().numpy(), out_ref)


@pytest.mark.parametrize("B,dt,stride", [(2, torch.float8_e4m3fn, (1, 1, 1)), (1, torch.bfloat16, (1, 1, 1)),
                                         (2, torch.float8_e4m3fn, (16, 8, 8))])
def test_repeat_runs_are_bit_identical(B, dt, stride):
    """The forward has one result per input: repeated launches of the full-size
    3-D video workload (30x48x80 tokens, 24 heads, window 16x32x48) write the
    same bytes.  A wait that lets the epilogue read O before the last P V
    products land shows up here as rows that change from run to run."""
    from dimensional_sparse_attention_gna_b300 import gna as G
    dims, window, heads, d = (30, 48, 80), (16, 32, 48), 24, 128
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(5700)
    shp = G.tiled_shape(B, heads, dims, d)
    qt, kt = (torch.randn(shp, device=dev, generator=gen).to(dt) for _ in range(2))
    vt = torch.randn(G.value_shape(B, heads, dims, d), device=dev, generator=gen).to(dt)
    ds = torch.ones(3, device=dev) if dt != torch.bfloat16 else None
    ref = torch.empty(shp, dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(ref)
    lse_ref = torch.empty(shp[:-1], dtype=torch.float32, device=dev)
    lse = torch.empty_like(lse_ref)
    G.gna_forward(qt, kt, vt, ref, lse_ref, B, heads, dims, window, stride, d, descale=ds)
    for _ in range(4):
        G.gna_forward(qt, kt, vt, out, lse, B, heads, dims, window, stride, d, descale=ds)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))
    G.gna_get_status()
