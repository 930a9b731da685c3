"""The CUDA backward (``gna_backward_delta``, ``gna_backward_dq``,
``gna_backward_dkdv``) against the pinned backward oracle, every element of dq,
dk and dv compared.

The GPU path reads the bf16 out and lse of its own forward; the oracle
recomputes everything in float64 from the same bf16 inputs.  The differences
come from bf16 dS, bf16 out in delta and the bf16 result, so the bar is a
relative one: relative RMS < 5e-3 and max |error| <= 1 % of max |gradient|
(measured: relative RMS <= 2.5e-3, max |error| <= 0.53 %, the size of bf16
rounding).
"""
import numpy as np
import pytest
import torch

import oracle
from dimensional_sparse_attention_gna_b300 import gna as G
from synthetic_inputs import exact_f32, normal_raster, to_bf16
from tests.gpu_helpers import MAX_ERR_GRAD, REL_RMS_GRAD, record_parity, sample_queries

pytestmark = pytest.mark.gpu


def gpu_backward(q, k, v, dout, dims, window, stride, tile=None, rule=G.GNA_LEADER_CENTER, scale=0.0):
    """(dq, dk, dv) raster float32 and the tiled bf16 results, through the C ABI."""
    B, T, H, W, heads, d = q.shape
    dev = torch.device("cuda")
    shp = G.tiled_shape(B, heads, dims, d, tile)
    tiled = {}
    for name, x in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        t = torch.empty(shp, dtype=torch.bfloat16, device=dev)
        G.gna_permute(x.to(dev).contiguous(), t, B, heads, dims, d, tile=tile)
        tiled[name] = t
    vshape = G.value_shape(B, heads, dims, d, tile)
    k_val, v_val = (torch.empty(vshape, dtype=torch.bfloat16, device=dev) for _ in range(2))
    G.gna_permute_v(k.to(dev).contiguous(), k_val, B, heads, dims, d, tile=tile)
    G.gna_permute_v(v.to(dev).contiguous(), v_val, B, heads, dims, d, tile=tile)
    out_t = torch.empty(shp, dtype=torch.bfloat16, device=dev)
    lse_t = torch.empty(shp[:-1], dtype=torch.float32, device=dev)
    G.gna_forward(tiled["q"], tiled["k"], v_val, out_t, lse_t, B, heads, dims, window, stride, d, tile=tile,
                  leader_rule=rule, scale=scale)
    delta = torch.empty(shp[:-1], dtype=torch.float32, device=dev)
    G.gna_backward_delta(out_t, tiled["dout"], delta, B, heads, dims, d, tile=tile)
    dq_t = torch.empty(shp, dtype=torch.bfloat16, device=dev)
    G.gna_backward_dq(tiled["q"], tiled["k"], k_val, tiled["v"], tiled["dout"], lse_t, delta, dq_t, B, heads, dims,
                      window, stride, d, tile=tile, leader_rule=rule, scale=scale)
    dk_t, dv_t = (torch.empty(shp, dtype=torch.bfloat16, device=dev) for _ in range(2))
    G.gna_backward_dkdv(tiled["q"], tiled["k"], tiled["v"], tiled["dout"], lse_t, delta, dk_t, dv_t, B, heads, dims,
                        window, stride, d, tile=tile, leader_rule=rule, scale=scale)
    res = []
    for t in (dq_t, dk_t, dv_t):
        r = torch.empty((B,) + tuple(dims) + (heads, d), dtype=torch.bfloat16, device=dev)
        G.gna_unpermute(t, r, B, heads, dims, d, tile=tile)
        res.append(r)
    G.gna_get_status()
    torch.cuda.synchronize()
    return [r.float().cpu().numpy() for r in res], (dq_t, dk_t, dv_t)


def _check_grads(seed, B, heads, dims, window, stride, tile=None, rule=G.GNA_LEADER_CENTER, d=128, scale=None):
    q, k, v, dout = (to_bf16(normal_raster(seed + i, B, dims, heads, d)) for i in range(4))
    got, _ = gpu_backward(q, k, v, dout, dims, window, stride, tile=tile, rule=rule, scale=scale or 0.0)
    orule = oracle.LEADER_CENTER if rule == G.GNA_LEADER_CENTER else oracle.LEADER_LITERAL
    refs = oracle.backward_c(exact_f32(q), exact_f32(k), exact_f32(v), exact_f32(dout), dims, window, stride,
                             scale=scale, rule=orule)
    for name, g, r in zip(("dq", "dk", "dv"), got, refs):
        err = np.abs(g.astype(np.float64) - r)
        rel = float(np.sqrt((err ** 2).mean() / (r ** 2).mean()))
        info = f"{name}: max|err|={err.max():.3e} max|ref|={np.abs(r).max():.3e} relRMS={rel:.3e}"
        print(info)
        record_parity(kind="backward", grad=name, seed=seed, dims=list(dims), window=list(window),
                      stride=list(stride), heads=heads, B=B, head_dim=d, max_abs_err=float(err.max()),
                      max_abs_ref=float(np.abs(r).max()), rel_rms=rel)
        assert np.isfinite(g).all(), info
        assert rel < REL_RMS_GRAD, info
        assert err.max() <= MAX_ERR_GRAD * np.abs(r).max(), info


@pytest.mark.parametrize("B,heads,dims,window,stride,tile,rule", [
    (1, 2, (4, 16, 20), (3, 7, 9), (1, 1, 1), None, G.GNA_LEADER_CENTER),
    (2, 2, (5, 19, 23), (3, 9, 11), (1, 2, 3), None, G.GNA_LEADER_CENTER),     # ragged: every tile padded
    (1, 2, (6, 20, 24), (4, 8, 8), (2, 4, 4), None, G.GNA_LEADER_LITERAL),
    (1, 2, (3, 17, 40), (3, 7, 13), (1, 2, 5), (1, 8, 16), G.GNA_LEADER_CENTER),
    (1, 3, (1, 45, 37), (1, 12, 9), (1, 1, 1), None, G.GNA_LEADER_CENTER),     # 2-D
    (1, 2, (2, 8, 16), (2, 8, 16), (1, 1, 1), None, G.GNA_LEADER_CENTER),      # window = grid
    (1, 2, (4, 16, 16), (2, 8, 8), (2, 8, 8), None, G.GNA_LEADER_CENTER),      # blocked
])
def test_gradients_small_grids_all_elements(B, heads, dims, window, stride, tile, rule):
    _check_grads(8000 + sum(dims), B, heads, dims, window, stride, tile=tile, rule=rule)


@pytest.mark.parametrize("B,heads,dims,window,stride,tile,rule", [
    (1, 2, (4, 16, 20), (3, 7, 9), (1, 1, 1), None, G.GNA_LEADER_CENTER),
    (2, 2, (5, 19, 23), (3, 9, 11), (1, 2, 3), None, G.GNA_LEADER_CENTER),     # ragged: every tile padded
    (1, 2, (6, 20, 24), (4, 8, 8), (2, 4, 4), None, G.GNA_LEADER_LITERAL),
    (1, 2, (3, 17, 40), (3, 7, 13), (1, 2, 5), (1, 8, 16), G.GNA_LEADER_CENTER),
    (1, 3, (1, 45, 37), (1, 12, 9), (1, 1, 1), None, G.GNA_LEADER_CENTER),     # 2-D
    (1, 2, (2, 8, 16), (2, 8, 16), (1, 1, 1), None, G.GNA_LEADER_CENTER),      # window = grid
])
def test_gradients_head_dim_64_small_grids_all_elements(B, heads, dims, window, stride, tile, rule):
    """head_dim 64: one 128-byte swizzle span per token row, dQ / dK / dV accumulators of 64 columns."""
    _check_grads(8300 + sum(dims), B, heads, dims, window, stride, tile=tile, rule=rule, d=64)


def test_gradients_mid_size_video_grid():
    """Several KV tiles per dimension and full interior tiles (8x24x40 tokens, 4 heads)."""
    _check_grads(8100, 1, 4, (8, 24, 40), (4, 12, 16), (1, 1, 1))


@pytest.mark.parametrize("d", [64, 128])
def test_gradients_with_a_custom_softmax_scale(d):
    """gna_options.scale in place of 1/sqrt(head_dim), in the forward and both
    backward kernels (0.2 sharpens the softmax at head_dim 64 and flattens it at 128)."""
    _check_grads(8700 + d, 1, 2, (5, 19, 23), (3, 9, 11), (1, 2, 3), d=d, scale=0.2)


def test_gradients_head_dim_64_mid_size_video_grid():
    _check_grads(8400, 1, 4, (8, 24, 40), (4, 12, 16), (1, 1, 1), d=64)


@pytest.mark.parametrize("B,heads,dims,window,stride,tile,rule", [
    (1, 2, (1, 16, 16), (1, 5, 5), (1, 1, 1), None, G.GNA_LEADER_CENTER),     # the tiny 2-D case at head_dim 32
    (2, 2, (5, 19, 23), (3, 9, 11), (1, 2, 3), None, G.GNA_LEADER_CENTER),     # ragged
    (1, 2, (6, 20, 24), (4, 8, 8), (2, 4, 4), None, G.GNA_LEADER_LITERAL),
    (1, 3, (3, 17, 40), (3, 7, 13), (1, 2, 5), (1, 8, 16), G.GNA_LEADER_CENTER),
])
def test_gradients_head_dim_32_small_grids_all_elements(B, heads, dims, window, stride, tile, rule):
    """head_dim 32: 64-byte token rows (64-byte swizzle), dQ / dK / dV accumulators of 32 columns."""
    _check_grads(8500 + sum(dims), B, heads, dims, window, stride, tile=tile, rule=rule, d=32)


def test_gradients_head_dim_32_mid_size_video_grid():
    _check_grads(8600, 1, 4, (8, 24, 40), (4, 12, 16), (1, 1, 1), d=32)


def test_gradients_repeat_runs_bit_identical():
    dims, window, stride, d = (4, 16, 24), (3, 9, 11), (1, 2, 3), 128
    q, k, v, dout = (to_bf16(normal_raster(8200 + i, 1, dims, 2, d)) for i in range(4))
    _, a = gpu_backward(q, k, v, dout, dims, window, stride)
    _, b = gpu_backward(q, k, v, dout, dims, window, stride)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_backward_abandoned_wait_reports_timeout_and_context_survives():
    """The dQ producer skips one KV load (test hook): the MMA warp's bounded wait
    gives up, the kernel exits, and the host reads GNA_ERR_TIMEOUT.  The next
    backward on the same context is correct again."""
    dims, window, stride, d = (1, 16, 16), (1, 5, 5), (1, 1, 1), 128
    q, k, v, dout = (to_bf16(normal_raster(8300 + i, 1, dims, 1, d)) for i in range(4))
    G.gna_test_skip_kv_load(1, 1)
    try:
        with pytest.raises(G.GNAError) as ei:
            gpu_backward(q, k, v, dout, dims, window, stride)
        assert ei.value.status == G.GNA_ERR_TIMEOUT
    finally:
        G.gna_test_skip_kv_load(1, -1)
    G.gna_get_status()   # cleared
    _check_grads(8300, 1, 1, dims, window, stride)


def _compare_sampled(name, got, ref, **rec):
    err = np.abs(got.astype(np.float64) - ref)
    rel = float(np.sqrt((err ** 2).mean() / (ref ** 2).mean()))
    info = f"{name}: max|err|={err.max():.3e} max|ref|={np.abs(ref).max():.3e} relRMS={rel:.3e}"
    print(info)
    record_parity(kind="backward", grad=name, max_abs_err=float(err.max()), max_abs_ref=float(np.abs(ref).max()),
                  rel_rms=rel, sampled=True, **rec)
    assert np.isfinite(got).all(), info
    assert rel < REL_RMS_GRAD and err.max() <= MAX_ERR_GRAD * np.abs(ref).max(), info


def test_gradients_video_720p_sampled_and_identities():
    """Full-size 3-D video workload (30x48x80 tokens, 24 heads, d=128, window
    16x32x48, stride 1), every gradient compared with the oracle at samples:
    dq at sampled queries (corner Q tiles of the first and last head plus
    random queries of any head), dk and dv at sampled keys (every key of the
    corner KV tiles of the first and last head plus random keys of those two
    heads: the key-side oracle recomputes lse and delta for every query of each
    plane it touches, so the keys stay in two planes).  dv also meets an
    identity of the derivative that holds at any size: sum_j dv_j = sum_i
    dout_i per head and feature (each query's probabilities sum to 1)."""
    B, heads, dims, window, stride, d = 1, 24, (30, 48, 80), (16, 32, 48), (1, 1, 1), 128
    q, k, v, dout = (to_bf16(normal_raster(8400 + i, B, dims, heads, d)) for i in range(4))
    (dq, dk, dv), _ = gpu_backward(q, k, v, dout, dims, window, stride)
    qf, kf, vf, gf = (exact_f32(x) for x in (q, k, v, dout))
    geo = dict(seed=8400, dims=list(dims), window=list(window), stride=list(stride), heads=heads, B=B)
    tile = G.gna_tile_shape(dims)
    rng = np.random.default_rng(8400)
    sel = sample_queries(rng, B, heads, dims, tile, 128)
    ids = oracle.query_ids(sel[:, 0], sel[:, 1], sel[:, 2], sel[:, 3], sel[:, 4], heads, dims)
    ref = oracle.backward_dq_c(qf, kf, vf, gf, dims, window, stride, ids)
    _compare_sampled("dq", dq[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]], ref, **geo)

    ksel = sample_queries(rng, B, heads, dims, tile, 256)
    ksel[len(ksel) - 256:, 1] = rng.choice([0, heads - 1], 256)       # random keys in the corner heads' planes
    kids = oracle.query_ids(ksel[:, 0], ksel[:, 1], ksel[:, 2], ksel[:, 3], ksel[:, 4], heads, dims)
    dk_ref, dv_ref = oracle.backward_kv_c(qf, kf, vf, gf, dims, window, stride, kids)
    at = (ksel[:, 0], ksel[:, 2], ksel[:, 3], ksel[:, 4], ksel[:, 1])
    _compare_sampled("dk", dk[at], dk_ref, **geo)
    _compare_sampled("dv", dv[at], dv_ref, **geo)

    axes = (0, 1, 2, 3)
    dsum = gf.astype(np.float64).sum(axis=axes)          # [heads, d]
    gap = np.abs(dv.astype(np.float64).sum(axis=axes) - dsum)
    assert gap.max() <= 1e-3 * np.abs(dsum).max(), (gap.max(), np.abs(dsum).max())
