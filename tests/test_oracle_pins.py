"""Pins of the CPU oracle against facts fixed by the sources and by mathematics.

None of these tests needs a GPU.  They check the oracle (``oracle/``) against
things other than itself: hand-derived window tables, a brute-force statement
of the window rule, special cases that reduce to torch's dense attention
routine, closed forms and invariants.  ``test_planted_mistakes_are_caught``
plants plausible mistakes in the oracle's window rule and checks that a pin
fails for each.

Sources: GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践") §1.1
(stride semantics: sliding window at stride 1, translation equivariant; blocked
when the window jumps) and §1.2 (each query processes k keys).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import layout, reference as ref
from synthetic_inputs import normal_raster, qkv_normal, to_bf16, exact_f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_window_rows():
    rows = []
    with open(os.path.join(GOLDEN, "window_starts_1d.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, tail = line.split(":")
            L, w, s, rule = head.split()
            rows.append((int(L), int(w), int(s), rule, [int(x) for x in tail.split()]))
    return rows


# ---------------------------------------------------------------- window rule

@pytest.mark.parametrize("L,w,s,rule,expected", _golden_window_rows())
def test_window_starts_match_hand_table(L, w, s, rule, expected):
    assert len(expected) == L
    got = [ref.window_start(i, L, w, s, rule) for i in range(L)]
    assert got == expected
    assert list(oracle.window_starts_c(L, w, s, rule)) == expected


def _brute_force_start(i, L, w, s, off):
    """The window as a search, not a formula.

    The stride group of i is the set of positions sharing floor(i/s); its leader
    is the group member ``off`` places after the group's first position (the
    group's last in-range member if that runs past the end).  Among all
    in-range windows [a, a+w), pick the one whose centre a + floor(w/2) is
    nearest the leader.
    """
    group = [j for j in range(L) if j // s == i // s]
    lead = min(group[0] + off, L - 1)
    best = min(range(0, L - w + 1), key=lambda a: abs(a + w // 2 - lead))
    return best


@pytest.mark.parametrize("rule", [ref.LEADER_CENTER, ref.LEADER_LITERAL])
def test_window_start_equals_brute_force(rule):
    for L in range(1, 14):
        for w in range(1, L + 1):
            for s in range(1, w + 1):
                off = s // 2 if rule == ref.LEADER_CENTER else (s - 1) // 2
                want = [_brute_force_start(i, L, w, s, off) for i in range(L)]
                got = [ref.window_start(i, L, w, s, rule) for i in range(L)]
                assert got == want, (L, w, s)
                assert list(oracle.window_starts_c(L, w, s, rule)) == want, (L, w, s)


def test_sliding_window_interior_is_centred():
    """Stride 1, away from the borders: the window is [i - floor(w/2), i - floor(w/2) + w)."""
    for L, w in [(20, 5), (20, 4), (33, 7), (48, 32)]:
        for i in range(w // 2, L - (w - w // 2) + 1):
            assert ref.window_start(i, L, w, 1) == i - w // 2


def test_blocked_mode_is_the_block():
    """Stride = window on a length divisible by it: the window of i is i's own block."""
    for w in range(1, 9):
        for nblocks in range(1, 5):
            L = w * nblocks
            for i in range(L):
                assert ref.window_start(i, L, w, w) == (i // w) * w


def test_every_query_sees_exactly_window_volume_keys():
    """GNA page §1.2: every query processes the same number of keys, prod(window)."""
    dims, window = (3, 5, 7), (2, 3, 4)
    for stride in [(1, 1, 1), (2, 3, 2), (2, 1, 4)]:
        for idx in itertools.product(*(range(L) for L in dims)):
            nb = ref.neighborhood(idx, dims, window, stride)
            assert len(nb) == len(set(nb)) == int(np.prod(window))
            for j in nb:
                assert all(0 <= j[d] < dims[d] for d in range(3))
        m = ref.window_mask(dims, window, stride)
        assert (m.sum(axis=1) == int(np.prod(window))).all()


# ---------------------------------------------------------------- attention math

def _sdpa_f64(q, k, v):
    """torch's dense attention routine in float64 on [B, heads, n, d] tensors."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v)).numpy()


def _as_bhnd(x):
    B, T, H, W, heads, d = x.shape
    return np.ascontiguousarray(x.reshape(B, T * H * W, heads, d).transpose(0, 2, 1, 3)).astype(np.float64)


def test_full_window_equals_dense_attention():
    """Stride 1 and window = grid: every query sees every key, i.e. full attention."""
    dims = (2, 3, 4)
    q, k, v = (normal_raster(s, 2, dims, 3, 8) for s in (1, 2, 3))
    want = _sdpa_f64(_as_bhnd(q), _as_bhnd(k), _as_bhnd(v))
    for fn in (ref.gna_forward_loops, ref.gna_forward_masked_dense):
        out, _ = fn(q, k, v, dims, dims, (1, 1, 1))
        np.testing.assert_allclose(_as_bhnd(out), want, rtol=0, atol=1e-12)
    out, _ = oracle.forward_c(q, k, v, dims, dims, (1, 1, 1))
    np.testing.assert_allclose(_as_bhnd(out), want, rtol=0, atol=1e-12)


def test_blocked_equals_blockwise_dense_attention():
    """Stride = window, grid divisible by window: independent full attention per block."""
    dims, window = (4, 6, 4), (2, 3, 2)
    B, heads, d = 1, 2, 8
    q, k, v = (normal_raster(s, B, dims, heads, d) for s in (4, 5, 6))
    out, _ = oracle.forward_c(q, k, v, dims, window, window)
    out_np, _ = ref.gna_forward_loops(q, k, v, dims, window, window)
    np.testing.assert_allclose(out, out_np, rtol=0, atol=1e-12)
    for bt, by, bx in itertools.product(*(range(L // w) for L, w in zip(dims, window))):
        sl = (slice(None), slice(bt * 2, bt * 2 + 2), slice(by * 3, by * 3 + 3), slice(bx * 2, bx * 2 + 2))
        blk = [_as_bhnd(np.ascontiguousarray(x[sl])) for x in (q, k, v)]
        want = _sdpa_f64(*blk)
        np.testing.assert_allclose(_as_bhnd(np.ascontiguousarray(out[sl])), want, rtol=0, atol=1e-12)


def test_unit_window_returns_own_value():
    """Window 1: the only key is the query's own position: out = v_i, lse = scale <q_i, k_i>."""
    dims = (2, 3, 5)
    q, k, v = (normal_raster(s, 1, dims, 2, 16) for s in (7, 8, 9))
    out, lse = oracle.forward_c(q, k, v, dims, (1, 1, 1), (1, 1, 1))
    np.testing.assert_array_equal(out, v.astype(np.float64))
    expect = (q.astype(np.float64) * k.astype(np.float64)).sum(-1) / 4.0
    np.testing.assert_allclose(lse, expect, rtol=0, atol=1e-12)


@pytest.mark.parametrize("stride", [(1, 1, 1), (2, 2, 3), (3, 1, 2)])
def test_zero_queries_give_window_mean_and_log_volume(stride):
    """Q = 0: all scores 0, so lse = ln prod(w) and out = mean of V over the window.

    With V = the key's coordinates, the mean is start + (w - 1)/2 in every
    dimension: a closed form for the window's position.
    """
    dims, window = (4, 6, 7), (3, 4, 3)
    B, heads, d = 1, 1, 3
    q = np.zeros((B,) + dims + (heads, d), np.float32)
    k = normal_raster(11, B, dims, heads, d)
    v = np.zeros_like(q)
    grid = np.stack(np.meshgrid(*(np.arange(L) for L in dims), indexing="ij"), axis=-1)
    v[0, :, :, :, 0, :] = grid
    out, lse = oracle.forward_c(q, k, v, dims, window, stride)
    np.testing.assert_allclose(lse, math.log(np.prod(window)), rtol=0, atol=1e-13)
    for idx in itertools.product(*(range(L) for L in dims)):
        for dd in range(3):
            a = ref.window_start(idx[dd], dims[dd], window[dd], stride[dd])
            assert abs(out[(0,) + idx + (0, dd)] - (a + (window[dd] - 1) / 2)) < 1e-12


def test_constant_keys_give_closed_form_lse():
    """k_j = k for all j: every score equals scale <q_i, k>, so lse = that + ln prod(w)."""
    dims, window, stride = (3, 4, 5), (2, 3, 3), (1, 2, 3)
    q = normal_raster(12, 1, dims, 2, 8)
    k = np.broadcast_to(normal_raster(13, 1, (1, 1, 1), 2, 8), q.shape).copy()
    v = normal_raster(14, 1, dims, 2, 8)
    _, lse = oracle.forward_c(q, k, v, dims, window, stride)
    s = (q.astype(np.float64) * k.astype(np.float64)).sum(-1) / math.sqrt(8)
    np.testing.assert_allclose(lse, s + math.log(np.prod(window)), rtol=0, atol=1e-12)


def test_indicator_value_probe():
    """V = indicator of one key j0 and Q = 0: out_i = 1/prod(w) iff j0 is in i's window."""
    dims, window, stride = (3, 5, 6), (2, 3, 4), (2, 1, 2)
    q = np.zeros((1,) + dims + (1, 1), np.float32)
    k = np.zeros_like(q)
    j0 = (1, 2, 3)
    v = np.zeros_like(q)
    v[(0,) + j0 + (0, 0)] = 1.0
    out, _ = oracle.forward_c(q, k, v, dims, window, stride)
    for idx in itertools.product(*(range(L) for L in dims)):
        inside = all(ref.window_start(idx[d], dims[d], window[d], stride[d]) <= j0[d]
                     < ref.window_start(idx[d], dims[d], window[d], stride[d]) + window[d] for d in range(3))
        want = 1.0 / np.prod(window) if inside else 0.0
        assert abs(out[(0,) + idx + (0, 0)] - want) < 1e-15


def test_translation_equivariance_of_sliding_window():
    """GNA page §1.1: stride 1 keeps translation equivariance.

    Shift the inputs by one position along W; an interior query's output moves
    with it.
    """
    dims, window = (1, 9, 16), (1, 3, 5)
    q, k, v = (normal_raster(s, 1, dims, 2, 8) for s in (21, 22, 23))
    out, lse = oracle.forward_c(q, k, v, dims, window, (1, 1, 1))
    sh = [np.roll(x, 1, axis=3) for x in (q, k, v)]
    out2, lse2 = oracle.forward_c(*sh, dims, window, (1, 1, 1))
    for y in range(1, 8):
        for x in range(3, 12):   # neither window touches a border or the wrapped column
            np.testing.assert_allclose(out2[0, 0, y, x + 1], out[0, 0, y, x], atol=1e-12)
            np.testing.assert_allclose(lse2[0, 0, y, x + 1], lse[0, 0, y, x], atol=1e-12)


@pytest.mark.parametrize("dims,window,stride,rule", [
    ((1, 16, 16), (1, 5, 5), (1, 1, 1), ref.LEADER_CENTER),
    ((3, 5, 7), (2, 3, 4), (2, 2, 3), ref.LEADER_CENTER),
    ((3, 5, 7), (2, 3, 4), (2, 2, 3), ref.LEADER_LITERAL),
    ((4, 6, 8), (4, 2, 8), (4, 2, 4), ref.LEADER_CENTER),
])
def test_three_formulations_agree(dims, window, stride, rule):
    """C loops, NumPy loops and torch masked dense attention agree to 1e-12."""
    q, k, v = (normal_raster(s, 2, dims, 2, 16) for s in (31, 32, 33))
    o1, l1 = oracle.forward_c(q, k, v, dims, window, stride, rule=rule)
    o2, l2 = ref.gna_forward_loops(q, k, v, dims, window, stride, rule=rule)
    o3, l3 = ref.gna_forward_masked_dense(q, k, v, dims, window, stride, rule=rule)
    for o, l in ((o2, l2), (o3, l3)):
        np.testing.assert_allclose(o1, o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l1, l, rtol=0, atol=1e-12)


def test_selected_queries_match_full_run():
    dims, window, stride = (3, 5, 7), (2, 3, 4), (1, 2, 2)
    q, k, v = (normal_raster(s, 2, dims, 3, 8) for s in (41, 42, 43))
    out, lse = oracle.forward_c(q, k, v, dims, window, stride)
    rng = np.random.default_rng(0)
    b, h, t, y, x = (rng.integers(0, n, 50) for n in (2, 3) + dims)
    sel = oracle.query_ids(b, h, t, y, x, 3, dims)
    o_s, l_s = oracle.forward_c(q, k, v, dims, window, stride, sel=sel)
    np.testing.assert_array_equal(o_s, out[b, t, y, x, h])
    np.testing.assert_array_equal(l_s, lse[b, t, y, x, h])


def test_tensor_scales_are_applied():
    """Per-tensor scales (e4m3 dequantisation): sq, sk scale the scores, sv the output.

    Powers of two keep the pre-scaled float32 inputs exact.
    """
    dims, window, stride = (2, 4, 4), (2, 3, 3), (1, 1, 1)
    q, k, v = (normal_raster(s, 1, dims, 1, 8) for s in (51, 52, 53))
    o1, l1 = oracle.forward_c(q, k, v, dims, window, stride, tensor_scales=(0.5, 4.0, 0.25))
    o2, l2 = oracle.forward_c(q * 0.5, k * 4.0, v * 0.25, dims, window, stride)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_oracle_rejects_bad_geometry():
    q = np.zeros((1, 1, 4, 4, 1, 4), np.float32)
    for window, stride in [((1, 5, 1), (1, 1, 1)), ((1, 2, 2), (1, 3, 1)), ((1, 0, 1), (1, 1, 1))]:
        with pytest.raises(ValueError):
            oracle.forward_c(q, q, q, (1, 4, 4), window, stride)


def test_bf16_rounding_is_exact_in_f32():
    x = normal_raster(61, 1, (1, 2, 3), 1, 64)
    xb = to_bf16(x)
    f = exact_f32(xb)
    assert f.dtype == np.float32
    np.testing.assert_array_equal(torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy(),
                                  xb.view(torch.int16).numpy())


def test_workload_seeds_are_distinct():
    q, k, v = qkv_normal(0, 1, (1, 2, 2), 1, 4)
    assert not np.array_equal(q, k) and not np.array_equal(k, v)


# ---------------------------------------------------------------- tiled layout

def test_layout_hand_example():
    """dims (1, 2, 4), tile (1, 2, 2): tiles are the 2x2 squares, row-major inside.

    Tokens numbered 0..7 in raster order (y*4 + x):
        0 1 | 2 3
        4 5 | 6 7
    tile 0 = [0 1 4 5], tile 1 = [2 3 6 7].
    """
    x = np.arange(8, dtype=np.float32).reshape(1, 1, 2, 4, 1, 1)
    y = layout.permute_reference(x, (1, 2, 2))
    assert y.shape == (1, 1, 1, 1, 2, 4, 1)
    assert y[0, 0, 0, 0, :, :, 0].tolist() == [[0, 1, 4, 5], [2, 3, 6, 7]]


def test_value_layout_is_the_tile_transposed():
    """Value layout: feature f of token e of a tile sits at [.., f, e]; hand example
    on a 1 x 2 x 4 grid with tile (1, 2, 2), one head, d = 3."""
    x = np.arange(1 * 1 * 2 * 4 * 1 * 3).reshape(1, 1, 2, 4, 1, 3)
    y = layout.permute_v_reference(x, (1, 2, 2))
    assert y.shape == (1, 1, 1, 1, 2, 3, 4)
    # tile 0 holds x = 0, 1 of both rows: tokens (y, x) = (0,0), (0,1), (1,0), (1,1)
    tok = [(0, 0), (0, 1), (1, 0), (1, 1)]
    for e, (yy, xx) in enumerate(tok):
        for f in range(3):
            assert y[0, 0, 0, 0, 0, f, e] == x[0, 0, yy, xx, 0, f]
            assert y[0, 0, 0, 0, 1, f, e] == x[0, 0, yy, xx + 2, 0, f]
    np.testing.assert_array_equal(np.swapaxes(y, -1, -2), layout.permute_reference(x, (1, 2, 2)))


def test_layout_padding_and_round_trip():
    """Ragged dims: padding positions are zero; unpermute inverts permute exactly."""
    dims, tile = (3, 5, 7), (2, 4, 4)
    x = normal_raster(71, 2, dims, 3, 5)
    y = layout.permute_reference(x, tile)
    assert y.shape == (2, 3, 2, 2, 2, 32, 5)
    np.testing.assert_array_equal(layout.unpermute_reference(y, dims, tile), x)
    # zero count = padded positions x heads x d x B
    padded = (4 * 8 * 8 - 3 * 5 * 7)
    assert int((y == 0).sum()) == 2 * 3 * 5 * padded
    for (b, h, t, yy, xx) in [(0, 0, 0, 0, 0), (1, 2, 2, 4, 6), (0, 1, 1, 3, 5)]:
        r = layout.tiled_row(b, h, t, yy, xx, 3, dims, tile)
        np.testing.assert_array_equal(y.reshape(-1, 5)[r], x[b, t, yy, xx, h])


# ---------------------------------------------------------------- planted mistakes

def _window_off_by_one(i, L, w, s, rule=ref.LEADER_CENTER):
    c = ref.leader(i, L, s, rule)
    return min(max(c - w // 2 + 1, 0), L - w)


def _window_no_low_clamp(i, L, w, s, rule=ref.LEADER_CENTER):
    c = ref.leader(i, L, s, rule)
    return max(min(c - w // 2, L - w), -(w // 2))


def _window_literal_leader(i, L, w, s, rule=ref.LEADER_CENTER):
    c = min((i // s) * s + (s - 1) // 2, L - 1)
    return min(max(c - w // 2, 0), L - w)


def _window_ceil_half(i, L, w, s, rule=ref.LEADER_CENTER):
    c = ref.leader(i, L, s, rule)
    return min(max(c - (w - 1) // 2, 0), L - w)


@pytest.mark.parametrize("mutant", [_window_off_by_one, _window_no_low_clamp,
                                    _window_literal_leader, _window_ceil_half])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    """Each plausible slip in the window rule makes at least one pin fail."""
    monkeypatch.setattr(ref, "window_start", mutant)
    failures = 0
    for L, w, s, rule, expected in _golden_window_rows():
        if rule != ref.LEADER_CENTER:
            continue
        try:
            got = [ref.window_start(i, L, w, s) for i in range(L)]
        except Exception:
            failures += 1
            continue
        failures += got != expected
    try:
        test_blocked_mode_is_the_block()
    except AssertionError:
        failures += 1
    assert failures > 0
