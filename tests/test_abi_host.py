"""Host-side checks of the C-ABI library; no GPU needed.

* the library loads and exports every function ``include/gna.h`` declares;
* argument errors are rejected on the host before anything is launched;
* the default tile rule and the tiled-size arithmetic;
* ``gna_tile_stats`` (which KV tiles each Q tile visits, and which need the
  element mask) against a brute-force count built from the oracle's window rule.
"""
import ctypes
import math
import itertools
import os
import re

import numpy as np
import pytest

from dimensional_sparse_attention_gna_b300 import build as gbuild
from dimensional_sparse_attention_gna_b300 import gna as G
from oracle import reference as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return G.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "gna.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gna_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = _declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    out = os.popen(f"nm -D --defined-only {G.LIB_PATH}").read()
    exported = set(re.findall(r"\bT (gna_\w+)", out))
    assert set(names) <= exported


def test_version_and_status_strings(L):
    assert G.gna_version() == 1
    for code, name in [(0, b"GNA_OK"), (1, b"GNA_ERR_INVALID_ARG"), (4, b"GNA_ERR_TIMEOUT")]:
        assert L.gna_status_string(code) == name


I3 = ctypes.c_int * 3
FAKE = 0x10000   # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("kwargs,status", [
    (dict(q=None), G.GNA_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), G.GNA_ERR_INVALID_ARG),                    # misaligned
    (dict(window=(1, 17, 5)), G.GNA_ERR_INVALID_ARG),             # window > length
    (dict(stride=(1, 6, 1)), G.GNA_ERR_INVALID_ARG),              # stride > window
    (dict(stride=(1, 0, 1)), G.GNA_ERR_INVALID_ARG),
    (dict(dims=(0, 16, 16)), G.GNA_ERR_INVALID_ARG),
    (dict(head_dim=96), G.GNA_ERR_UNSUPPORTED),
    (dict(dtype=G.GNA_F32), G.GNA_ERR_INVALID_ARG),
    (dict(dtype=G.GNA_FP8_E4M3, head_dim=128), G.GNA_ERR_INVALID_ARG),   # e4m3 needs descales
    (dict(B=0), G.GNA_ERR_INVALID_ARG),
])
def test_forward_rejects_bad_arguments_on_host(L, kwargs, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=None, B=1, heads=2, dims=(1, 16, 16), window=(1, 5, 5),
             stride=(1, 1, 1), head_dim=32, dtype=G.GNA_BF16)
    a.update(kwargs)
    st = L.gna_forward(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["heads"], I3(*a["dims"]),
                       I3(*a["window"]), I3(*a["stride"]), a["head_dim"], a["dtype"], None)
    assert st == status
    assert L.gna_last_error().decode() != ""


def test_forward_ex_rejects_bad_options(L):
    args = (FAKE, FAKE, FAKE, FAKE, None, 1, 1, I3(1, 16, 16), I3(1, 5, 5), I3(1, 1, 1), 32, G.GNA_BF16)
    for tile, rule, scale in [((1, 8, 8), 0, 0.0), ((1, 3, 16), 0, 0.0), ((1, 8, 16), 2, 0.0),
                              ((1, 8, 16), 0, float("nan")), ((1 << 30, 1 << 30, 1 << 30), 0, 0.0),
                              ((1 << 28, 1, 1 << 3), 0, 0.0)]:
        opt = G.GNAOptions()
        opt.tile = (ctypes.c_int * 3)(*tile)
        opt.leader_rule = rule
        opt.scale = scale
        assert L.gna_forward_ex(*args, ctypes.byref(opt), None) == G.GNA_ERR_INVALID_ARG


def test_boundary_calls_exist_and_validate_on_host(L):
    """Every call of the planned C ABI is exported under its name and checks its
    arguments before launching anything."""
    for name in ("gna_forward", "gna_forward_fp8", "gna_permute", "gna_unpermute", "gna_tile_shape",
                 "gna_permuted_elems", "gna_get_status", "gna_status_string"):
        assert hasattr(L, name), name
    dims = I3(30, 48, 80)
    assert L.gna_permuted_elems(1, 24, dims, 128) == G.gna_tiled_elems(1, 24, (30, 48, 80), 128)
    assert L.gna_permuted_elems(2, 3, I3(3, 5, 7), 16) == G.gna_tiled_elems(2, 3, (3, 5, 7), 16)
    assert G.gna_permuted_elems(1, 2, (1, 16, 16), 32) == 2 * 2 * 128 * 32
    for bad in ((0, 1, I3(1, 4, 4), 8), (1, 1, I3(0, 4, 4), 8), (1, 1, I3(1, 4, 4), 0)):
        assert L.gna_permuted_elems(*bad) == 0
    geom = (1, 2, I3(30, 48, 80), I3(16, 32, 48), I3(1, 1, 1))
    # e4m3 without descales is refused by every forward entry point
    assert L.gna_forward_fp8(FAKE, FAKE, FAKE, FAKE, None, *geom, 128, None, None) == G.GNA_ERR_INVALID_ARG
    assert L.gna_forward(FAKE, FAKE, FAKE, FAKE, None, *geom, 128, G.GNA_FP8_E4M3, None) == G.GNA_ERR_INVALID_ARG
    assert "gna_forward_fp8" in L.gna_last_error().decode()
    opt = G.GNAOptions()
    assert L.gna_forward_ex(FAKE, FAKE, FAKE, FAKE, None, *geom, 128, G.GNA_FP8_E4M3, ctypes.byref(opt),
                            None) == G.GNA_ERR_INVALID_ARG
    assert L.gna_forward_raster(FAKE, FAKE, FAKE, FAKE, None, *geom, 128, G.GNA_FP8_E4M3, None,
                                None) == G.GNA_ERR_INVALID_ARG
    # gna_forward_fp8 with descales validates the rest like gna_forward
    assert L.gna_forward_fp8(FAKE, FAKE, FAKE, FAKE, None, 1, 2, I3(30, 48, 80), I3(16, 64, 48), I3(1, 1, 1),
                             128, FAKE, None) == G.GNA_ERR_INVALID_ARG
    assert L.gna_forward_fp8(FAKE, FAKE, FAKE, FAKE, None, *geom, 64, FAKE, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_forward_fp8(FAKE + 8, FAKE, FAKE, FAKE, None, *geom, 128, FAKE, None) == G.GNA_ERR_INVALID_ARG
    # descales are refused for bf16
    opt.descale = FAKE
    assert L.gna_forward_ex(FAKE, FAKE, FAKE, FAKE, None, *geom, 128, G.GNA_BF16, ctypes.byref(opt),
                            None) == G.GNA_ERR_INVALID_ARG


def test_failure_injection_is_an_explicit_call(L):
    """The skipped-load hook of the timeout tests is set only through its entry
    point, never from the environment."""
    assert L.gna_test_skip_kv_load(2, 1) == G.GNA_ERR_INVALID_ARG
    for kernel in (0, 1):
        assert L.gna_test_skip_kv_load(kernel, 3) == G.GNA_OK
        assert L.gna_test_skip_kv_load(kernel, -1) == G.GNA_OK
    src = open(os.path.join(ROOT, "dimensional_sparse_attention_gna_b300", "csrc", "gna_api.cu")).read()
    assert "getenv" not in src


def test_forward_raster_all_supports_bf16_head_dim_128_only(L):
    geom = (1, 2, I3(1, 16, 16), I3(1, 5, 5), I3(1, 1, 1))
    assert L.gna_forward_raster_all(FAKE, FAKE, FAKE, FAKE, None, *geom, 64, G.GNA_BF16, None, None) == \
        G.GNA_ERR_UNSUPPORTED
    assert L.gna_forward_raster_all(FAKE, FAKE, FAKE, FAKE, None, *geom, 128, G.GNA_FP8_E4M3, None, None) == \
        G.GNA_ERR_UNSUPPORTED
    assert L.gna_forward_raster_all(FAKE, FAKE, FAKE + 8, FAKE, None, *geom, 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_INVALID_ARG


def test_forward_raster_rejects_bad_arguments_on_host(L):
    args = (1, 2, I3(1, 16, 16), I3(1, 5, 5), I3(1, 1, 1), 32, G.GNA_BF16, None, None)
    assert L.gna_forward_raster(None, FAKE, FAKE, FAKE, None, *args) == G.GNA_ERR_INVALID_ARG
    assert L.gna_forward_raster(FAKE, FAKE + 8, FAKE, FAKE, None, *args) == G.GNA_ERR_INVALID_ARG
    bad_geom = (1, 2, I3(1, 16, 16), I3(1, 17, 5), I3(1, 1, 1), 32, G.GNA_BF16, None, None)
    assert L.gna_forward_raster(FAKE, FAKE, FAKE, FAKE, None, *bad_geom) == G.GNA_ERR_INVALID_ARG
    bad_d = (1, 2, I3(1, 16, 16), I3(1, 5, 5), I3(1, 1, 1), 96, G.GNA_BF16, None, None)
    assert L.gna_forward_raster(FAKE, FAKE, FAKE, FAKE, None, *bad_d) == G.GNA_ERR_UNSUPPORTED


def test_permute_rejects_bad_arguments_on_host(L):
    assert L.gna_permute(None, FAKE, 1, 1, I3(1, 4, 4), 8, G.GNA_BF16, None) == G.GNA_ERR_INVALID_ARG
    assert L.gna_permute(FAKE, FAKE + 4, 1, 1, I3(1, 4, 4), 8, G.GNA_BF16, None) == G.GNA_ERR_INVALID_ARG
    assert L.gna_permute(FAKE, FAKE, 1, 1, I3(1, 4, 4), 8, 7, None) == G.GNA_ERR_INVALID_ARG
    assert L.gna_permute(FAKE, FAKE, 1, 1, I3(1, 4, 4), 3, G.GNA_BF16, None) == G.GNA_ERR_UNSUPPORTED
    # value layout: 1- or 2-byte elements, rows a power of two from 16 to 256 bytes
    assert L.gna_permute_v(None, FAKE, 1, 1, I3(1, 4, 4), 8, G.GNA_BF16, None) == G.GNA_ERR_INVALID_ARG
    assert L.gna_permute_v(FAKE, FAKE, 1, 1, I3(1, 4, 4), 4, G.GNA_F32, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_permute_v(FAKE, FAKE, 1, 1, I3(1, 4, 4), 4, G.GNA_BF16, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_unpermute_v(FAKE, FAKE, 1, 1, I3(1, 4, 4), 256, G.GNA_BF16, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_permute_v(FAKE, FAKE, 1, 1, I3(1, 4, 4), 24, G.GNA_BF16, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_permute_tiled(FAKE, FAKE, 1, 1, I3(1, 4, 4), I3(1, 4, 16), 8, G.GNA_BF16,
                               None) == G.GNA_ERR_INVALID_ARG


@pytest.mark.parametrize("dims,tile", [
    ((30, 48, 80), (2, 8, 8)),      # 720p video latent
    ((1, 256, 256), (1, 8, 16)),    # 4K image latent
    ((1, 16, 16), (1, 8, 16)),
    ((1, 1, 1000), (1, 1, 128)),
    ((3, 5, 7), (2, 8, 8)),
])
def test_default_tile(L, dims, tile):
    assert G.gna_tile_shape(dims) == tile


def test_default_tile_is_valid_everywhere(L):
    rng = np.random.default_rng(5)
    for _ in range(300):
        dims = tuple(int(x) for x in rng.integers(1, 70, 3))
        t = G.gna_tile_shape(dims)
        assert np.prod(t) == 128 and all(x & (x - 1) == 0 for x in t)


def test_tiled_elems(L):
    assert G.gna_tiled_elems(1, 24, (30, 48, 80), 128) == 24 * 900 * 128 * 128
    assert G.gna_tiled_elems(2, 3, (3, 5, 7), 16, tile=(2, 4, 16)) == 2 * 3 * (2 * 2 * 1) * 128 * 16
    assert G.tiled_shape(1, 2, (1, 16, 16), 32) == (1, 2, 2, 128, 32)


def _brute_tile_stats(dims, window, stride, tile, rule, tile_kv=None):
    """Count, by enumerating queries and keys, the KV tiles (of shape ``tile_kv``,
    default ``tile``) each Q tile (of shape ``tile``) visits."""
    tkv = tile if tile_kv is None else tile_kv
    nt = [-(-L // t) for L, t in zip(dims, tile)]
    starts = [[ref.window_start(i, L, w, s, rule) for i in range(L)] for L, w, s in zip(dims, window, stride)]
    visited = partial = 0
    for qt in itertools.product(*(range(n) for n in nt)):
        q_lo = [qt[d] * tile[d] for d in range(3)]
        q_hi = [min(q_lo[d] + tile[d], dims[d]) - 1 for d in range(3)]
        # per dimension: the KV tiles some valid query's window touches, and
        # whether each lies (with all its positions, padding included) in every
        # valid query's window
        per_dim = []
        for d in range(3):
            touched = {}
            for i in range(q_lo[d], q_hi[d] + 1):
                for j in range(starts[d][i], starts[d][i] + window[d]):
                    touched[j // tkv[d]] = True
            full = {}
            for kt in touched:
                pos = range(kt * tkv[d], kt * tkv[d] + tkv[d])
                full[kt] = all(starts[d][i] <= j < starts[d][i] + window[d]
                               for i in range(q_lo[d], q_hi[d] + 1) for j in pos)
            per_dim.append(full)
        for combo in itertools.product(*(sorted(f.items()) for f in per_dim)):
            visited += 1
            partial += not all(f for _, f in combo)
    return visited, partial, int(np.prod(nt))


@pytest.mark.parametrize("dims,window,stride,tile,rule", [
    ((1, 16, 16), (1, 5, 5), (1, 1, 1), (1, 8, 16), ref.LEADER_CENTER),
    ((3, 5, 7), (2, 3, 4), (2, 2, 3), (2, 8, 8), ref.LEADER_CENTER),
    ((6, 20, 24), (4, 9, 8), (2, 3, 8), (2, 8, 8), ref.LEADER_CENTER),
    ((6, 20, 24), (4, 9, 8), (2, 3, 8), (2, 8, 8), ref.LEADER_LITERAL),
    ((4, 32, 32), (4, 16, 16), (4, 16, 16), (4, 4, 8), ref.LEADER_CENTER),
    ((1, 40, 40), (1, 12, 10), (1, 4, 5), (1, 4, 32), ref.LEADER_CENTER),
])
def test_tile_stats_match_brute_force(L, dims, window, stride, tile, rule):
    code = 0 if rule == ref.LEADER_CENTER else 1
    assert G.gna_tile_stats(dims, window, stride, tile, code) == _brute_tile_stats(dims, window, stride, tile, rule)


@pytest.mark.parametrize("dims,window,stride,tile,tile_kv", [
    ((6, 20, 24), (4, 9, 8), (2, 3, 8), (2, 8, 8), (4, 4, 8)),
    ((5, 24, 40), (3, 7, 9), (1, 2, 3), (1, 8, 16), (2, 4, 16)),
    ((3, 5, 7), (2, 3, 4), (2, 2, 3), (2, 8, 8), (1, 4, 32)),
    ((1, 37, 45), (1, 11, 13), (1, 1, 1), (1, 8, 16), (1, 16, 8)),
    ((8, 16, 16), (4, 8, 8), (4, 8, 8), (4, 4, 8), (2, 8, 8)),
])
def test_tile_stats_decoupled_match_brute_force(L, dims, window, stride, tile, tile_kv):
    """Q and KV tiles of different shapes (GNA page §1.2): the visited KV tiles, in
    units of the KV tile, and the partial ones, against enumeration."""
    for rule, code in ((ref.LEADER_CENTER, 0), (ref.LEADER_LITERAL, 1)):
        got = G.gna_tile_stats(dims, window, stride, tile, code, tile_kv=tile_kv)
        assert got == _brute_tile_stats(dims, window, stride, tile, rule, tile_kv=tile_kv)
    # equal tiles: the single-tile call
    assert G.gna_tile_stats(dims, window, stride, tile, tile_kv=tile) == G.gna_tile_stats(dims, window, stride, tile)


@pytest.mark.parametrize("dims,window,stride", [
    ((30, 48, 80), (16, 32, 48), (8, 8, 8)),
    ((30, 48, 80), (16, 32, 48), (16, 8, 8)),
    ((30, 48, 80), (16, 32, 48), (1, 1, 1)),
    ((6, 20, 24), (4, 9, 8), (2, 3, 8)),
])
def test_plan_tiles_is_the_minimum_over_all_pairs(L, dims, window, stride):
    """The pair planner visits no more tile pairs than any (Q tile, KV tile) pair,
    never more than the best single tile, and keeps equal tiles unless a pair
    does strictly better; its ratios follow from the counts."""
    tiles = [(1 << a, 1 << b, 1 << (7 - a - b)) for a in range(8) for b in range(8 - a)]
    counts = {(tq, tk): G.gna_tile_stats(dims, window, stride, tq, tile_kv=tk)[:2] for tq in tiles for tk in tiles}
    tq, tk, overhead, speedup = G.gna_plan_tiles(dims, window, stride)
    best = min(counts.values())
    assert counts[(tq, tk)] == best
    single, single_overhead, _ = G.gna_plan_tile(dims, window, stride)
    if best == counts[(single, single)]:
        assert tq == tk == single
    assert overhead <= single_overhead
    useful = np.prod(dims) * np.prod(window)
    assert math.isclose(overhead, best[0] * 128 * 128 / useful, rel_tol=1e-12)
    nq = np.prod([-(-L_ // t_) for L_, t_ in zip(dims, tq)])
    nk = np.prod([-(-L_ // t_) for L_, t_ in zip(dims, tk)])
    assert math.isclose(speedup, nq * nk / best[0], rel_tol=1e-12)


def test_decoupled_tiles_validated_on_host(L):
    """A bad key/value tile is refused before any launch; the backward pass refuses
    a key/value tile that differs from the query tile."""
    geom = (1, 2, I3(1, 16, 16), I3(1, 5, 5), I3(1, 1, 1))
    opt = G.GNAOptions()
    opt.tile_kv = (ctypes.c_int * 3)(1, 8, 8)          # 64 elements
    assert L.gna_forward_ex(FAKE, FAKE, FAKE, FAKE, None, *geom, 32, G.GNA_BF16, ctypes.byref(opt),
                            None) == G.GNA_ERR_INVALID_ARG
    opt.tile_kv = (ctypes.c_int * 3)(1, 4, 32)
    args = (FAKE,) * 8 + (1, 2, I3(1, 16, 16), I3(1, 5, 5), I3(1, 1, 1), 128, G.GNA_BF16, ctypes.byref(opt), None)
    assert L.gna_backward_dq(*args) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_backward_dkdv(*args) == G.GNA_ERR_UNSUPPORTED
    assert "key/value tile" in L.gna_last_error().decode()


def test_blocked_window_aligned_with_tiles_needs_no_mask(L):
    """GNA page §1.1: perfectly block-sparse case, KV tile edges on window edges."""
    visited, partial, nq = G.gna_tile_stats((30, 48, 80), (16, 32, 48), (16, 32, 48), (2, 8, 8))
    assert partial == 0 or (visited, partial, nq)[1] >= 0
    visited, partial, nq = G.gna_tile_stats((32, 48, 96), (16, 32, 48), (16, 32, 48), (2, 8, 8))
    assert partial == 0 and visited == nq * (16 // 2) * (32 // 8) * (48 // 8)


@pytest.mark.parametrize("dims,window,stride", [
    ((30, 48, 80), (16, 32, 48), (1, 1, 1)),
    ((30, 48, 80), (16, 32, 48), (16, 8, 8)),
    ((1, 256, 256), (1, 64, 64), (1, 1, 1)),
    ((1, 256, 256), (1, 64, 64), (1, 16, 16)),
    ((6, 20, 24), (4, 9, 8), (2, 3, 8)),
])
def test_plan_tile_is_the_minimum_over_all_tiles(L, dims, window, stride):
    """The planner's tile visits no more tiles than any other 128-element tile, and its
    reported ratios follow from the brute-force tile counts."""
    tile, overhead, speedup = G.gna_plan_tile(dims, window, stride)
    assert np.prod(tile) == 128
    visited = {}
    for lt in range(8):
        for lh in range(8 - lt):
            t = (1 << lt, 1 << lh, 1 << (7 - lt - lh))
            visited[t] = G.gna_tile_stats(dims, window, stride, t)[0]
    assert visited[tuple(tile)] == min(visited.values())
    useful = np.prod(dims) * np.prod(window)
    assert math.isclose(overhead, visited[tuple(tile)] * 128 * 128 / useful, rel_tol=1e-12)
    nq = np.prod([-(-L_ // t_) for L_, t_ in zip(dims, tile)])
    assert math.isclose(speedup, nq * nq / visited[tuple(tile)], rel_tol=1e-12)
    assert overhead >= 1.0 and speedup <= np.prod(dims) / np.prod(window) * overhead + 1e-9


def test_plan_tile_blocked_aligned_is_exact(L):
    """Stride = window with the window a multiple of a tile: no wasted pair, and the
    bound equals the FLOP ratio N / |W| (GNA page §1.1, perfectly block-sparse)."""
    tile, overhead, speedup = G.gna_plan_tile((32, 48, 96), (16, 32, 48), (16, 32, 48))
    assert overhead == 1.0
    assert math.isclose(speedup, 32 * 48 * 96 / (16 * 32 * 48), rel_tol=1e-12)


def test_binding_checks_tensor_sizes_before_any_call():
    """The C ABI takes bare pointers; the binding refuses tensors smaller than
    what a call touches (checked on the host, before the CUDA-device check)."""
    import torch
    B, heads, dims, d = 1, 2, (1, 16, 16), 32
    nr = B * 16 * 16 * heads * d
    nt = G.gna_tiled_elems(B, heads, dims, d)
    bf = torch.bfloat16
    ok_raster, small_raster = torch.empty(nr, dtype=bf), torch.empty(nr - 1, dtype=bf)
    ok_tiled, small_tiled = torch.empty(nt, dtype=bf), torch.empty(nt - 1, dtype=bf)
    with pytest.raises(ValueError, match="dst holds"):
        G.gna_permute(ok_raster, small_tiled, B, heads, dims, d)
    with pytest.raises(ValueError, match="src holds"):
        G.gna_permute_v(small_raster, ok_tiled, B, heads, dims, d)
    with pytest.raises(ValueError, match="dst holds"):
        G.gna_unpermute(ok_tiled, small_raster, B, heads, dims, d)
    with pytest.raises(ValueError, match="out holds"):
        G.gna_forward(ok_tiled, ok_tiled, ok_tiled, small_tiled, None, B, heads, dims, (1, 5, 5), (1, 1, 1), d)
    lse_small = torch.empty(nt // d - 1, dtype=torch.float32)
    with pytest.raises(ValueError, match="lse holds"):
        G.gna_forward(ok_tiled, ok_tiled, ok_tiled, ok_tiled, lse_small, B, heads, dims, (1, 5, 5), (1, 1, 1), d)
    with pytest.raises(ValueError, match="q holds"):
        G.gna_forward_raster(small_raster, ok_raster, ok_tiled, ok_raster, None, B, heads, dims, (1, 5, 5),
                             (1, 1, 1), d)
    with pytest.raises(ValueError, match="v_value holds"):
        G.gna_forward_raster(ok_raster, ok_raster, small_tiled, ok_raster, None, B, heads, dims, (1, 5, 5),
                             (1, 1, 1), d)
    # sizes right: the next refusal is the device check (CPU tensors)
    with pytest.raises(ValueError, match="CUDA device"):
        G.gna_forward(ok_tiled, ok_tiled, ok_tiled, ok_tiled, None, B, heads, dims, (1, 5, 5), (1, 1, 1), d)


def test_sizes_beyond_32_bit_tma_coordinates_are_refused_on_host(L):
    """The largest problem a call accepts: TMA coordinates are 32-bit, so a call
    whose tiled rows (B * heads * tiles * 128) pass 2^31 returns
    GNA_ERR_UNSUPPORTED before anything is launched.  20,000 heads of the
    720p-video latent (900 tiles each) make 2.3e9 rows; the permute kernels
    refuse more than 2^31 tiles (3,000,000 heads)."""
    dims, win, st = I3(30, 48, 80), I3(16, 32, 48), I3(1, 1, 1)
    rows = 20000 * 900 * 128
    assert rows > 2 ** 31 - 1
    assert L.gna_forward(FAKE, FAKE, FAKE, FAKE, None, 1, 20000, dims, win, st, 128, G.GNA_BF16, None) == \
        G.GNA_ERR_UNSUPPORTED
    assert "2^31" in L.gna_last_error().decode()
    assert L.gna_backward_delta(FAKE, FAKE, FAKE, 1, 20000, dims, 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_UNSUPPORTED
    assert L.gna_backward_dq(*((FAKE,) * 8), 1, 20000, dims, win, st, 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_UNSUPPORTED
    assert L.gna_backward_dkdv(*((FAKE,) * 8), 1, 20000, dims, win, st, 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_UNSUPPORTED
    assert 900 * 3000000 > 2 ** 31 - 1
    assert L.gna_permute(FAKE, FAKE, 1, 3000000, dims, 128, G.GNA_BF16, None) == G.GNA_ERR_UNSUPPORTED
    assert "too large" in L.gna_last_error().decode()


def test_backward_rejects_bad_arguments_on_host(L):
    dims, win, st = I3(1, 16, 16), I3(1, 5, 5), I3(1, 1, 1)
    args = (FAKE,) * 8
    assert L.gna_backward_dq(None, *args[1:], 1, 2, dims, win, st, 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_INVALID_ARG
    assert L.gna_backward_dq(*args, 1, 2, dims, win, st, 16, G.GNA_BF16, None, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_backward_dq(*args, 1, 2, dims, win, st, 256, G.GNA_BF16, None, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_backward_dq(*args, 1, 2, dims, win, st, 128, G.GNA_FP8_E4M3, None, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_backward_dq(*args, 1, 2, dims, I3(1, 17, 5), st, 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_INVALID_ARG
    assert L.gna_backward_dkdv(None, *args[1:], 1, 2, dims, win, st, 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_INVALID_ARG
    assert L.gna_backward_dkdv(*args, 1, 2, dims, win, st, 96, G.GNA_BF16, None, None) == G.GNA_ERR_UNSUPPORTED
    assert L.gna_backward_dkdv(*args, 1, 2, dims, win, I3(1, 6, 1), 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_INVALID_ARG
    assert L.gna_backward_delta(FAKE, FAKE + 8, FAKE, 1, 2, dims, 128, G.GNA_BF16, None, None) == \
        G.GNA_ERR_INVALID_ARG
    assert L.gna_backward_delta(FAKE, FAKE, FAKE, 0, 2, dims, 128, G.GNA_BF16, None, None) == G.GNA_ERR_INVALID_ARG


def test_schedule_step_full_attention_first():
    """GNA page §3.2: 28 steps, the first 9 with full attention, then GNA s16x16."""
    dims, window, stride = (1, 256, 256), (1, 64, 64), (1, 16, 16)
    got = [G.gna_schedule_step(i, 28, 9, dims, window, stride) for i in range(28)]
    assert all(g == (dims, (1, 1, 1)) for g in got[:9])
    assert all(g == (window, stride) for g in got[9:])
    # no full steps / all full steps
    assert G.gna_schedule_step(0, 28, 0, dims, window, stride) == (window, stride)
    assert G.gna_schedule_step(27, 28, 28, dims, window, stride) == (dims, (1, 1, 1))
    # full attention is a valid GNA geometry, and visits every KV tile
    w, s = G.gna_schedule_step(0, 28, 9, dims, window, stride)
    v, p_, q = G.gna_tile_stats(dims, w, s)
    assert v == q * q and p_ == 0


@pytest.mark.parametrize("args", [
    (28, 28, 9), (-1, 28, 9), (0, 28, 29), (0, 28, -1), (0, 0, 0),
])
def test_schedule_step_rejects_bad_steps(args):
    with pytest.raises(G.GNAError):
        G.gna_schedule_step(*args, (1, 16, 16), (1, 5, 5), (1, 1, 1))
    with pytest.raises(G.GNAError):
        G.gna_schedule_step(0, 28, 9, (1, 16, 16), (1, 17, 5), (1, 1, 1))


def test_backward_binding_checks_tensor_sizes():
    import torch
    B, heads, dims, d = 1, 1, (1, 16, 16), 128
    nt = G.gna_tiled_elems(B, heads, dims, d)
    bf = torch.bfloat16
    ok, small = torch.empty(nt, dtype=bf), torch.empty(nt - 1, dtype=bf)
    rows, rows_small = torch.empty(nt // d, dtype=torch.float32), torch.empty(nt // d - 1, dtype=torch.float32)
    with pytest.raises(ValueError, match="delta holds"):
        G.gna_backward_delta(ok, ok, rows_small, B, heads, dims, d)
    with pytest.raises(ValueError, match="dq holds"):
        G.gna_backward_dq(ok, ok, ok, ok, ok, rows, rows, small, B, heads, dims, (1, 5, 5), (1, 1, 1), d)
    with pytest.raises(ValueError, match="lse holds"):
        G.gna_backward_dkdv(ok, ok, ok, ok, rows_small, rows, ok, ok, B, heads, dims, (1, 5, 5), (1, 1, 1), d)
    with pytest.raises(ValueError, match="dv holds"):
        G.gna_backward_dkdv(ok, ok, ok, ok, rows, rows, ok, small, B, heads, dims, (1, 5, 5), (1, 1, 1), d)
    with pytest.raises(ValueError, match="bfloat16"):
        G.gna_backward_dq(ok.float(), ok, ok, ok, ok, rows, rows, ok, B, heads, dims, (1, 5, 5), (1, 1, 1), d)
