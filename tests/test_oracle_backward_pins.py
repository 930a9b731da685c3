"""Pins of the backward oracle (``oracle.reference.gna_backward_loops`` and the C
``oracle.backward_c``), none of which retypes its formulas:

* central finite differences of the forward oracle, in float64, at random
  coordinates of q, k and v, on strided, clipped and literal-leader geometries;
* window = grid: torch's CPU scaled-dot-product attention differentiated by
  autograd in float64 (a library routine);
* stride = window on a divisible grid: the same, block by block;
* window 1: out = v exactly, so dv = dout and dq = dk = 0;
* the C and the loop versions agree on random cases, and the selected-query dq
  and selected-key dk, dv of the C oracle equal its whole-plane results;
* three identities of the derivative that hold at any size (sums of dv and dk,
  and sum <dq, q> = sum <dk, k>);
* planted mistakes in the softmax Jacobian are caught by the finite differences.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle import reference as ref


def _inputs(seed, B, dims, heads, d):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal((B,) + tuple(dims) + (heads, d)) for _ in range(4)]


def _fd_errors(dims, window, stride, rule, seed, n_coords=12, eps=1e-6):
    """Largest |finite difference - oracle gradient| over random coordinates."""
    q, k, v, dout = _inputs(seed, 1, dims, 2, 6)
    grads = dict(zip("qkv", ref.gna_backward_loops(q, k, v, dout, dims, window, stride, rule=rule)))
    rng = np.random.default_rng(seed + 1)
    worst = 0.0
    for name in "qkv":
        for _ in range(n_coords):
            ix = tuple(int(rng.integers(0, n)) for n in q.shape)
            vals = []
            for sgn in (1.0, -1.0):
                args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
                args[name][ix] += sgn * eps
                out, _ = ref.gna_forward_loops(args["q"], args["k"], args["v"], dims, window, stride, rule=rule)
                vals.append(float((out * dout).sum()))
            fd = (vals[0] - vals[1]) / (2 * eps)
            worst = max(worst, abs(fd - grads[name][ix]))
    return worst


@pytest.mark.parametrize("dims,window,stride,rule", [
    ((2, 5, 6), (2, 3, 3), (1, 1, 1), ref.LEADER_CENTER),
    ((3, 6, 7), (2, 3, 5), (1, 2, 3), ref.LEADER_CENTER),      # strided, clipped at both borders
    ((1, 8, 8), (1, 4, 6), (1, 4, 2), ref.LEADER_LITERAL),
])
def test_backward_matches_central_differences(dims, window, stride, rule):
    assert _fd_errors(dims, window, stride, rule, seed=11) < 1e-7


def _to_bhnd(x):
    B, T, H, W, heads, d = x.shape
    return torch.tensor(x.reshape(B, T * H * W, heads, d).transpose(0, 2, 1, 3), dtype=torch.float64,
                        requires_grad=True)


def _from_bhnd(g, shape):
    B, T, H, W, heads, d = shape
    return g.detach().numpy().transpose(0, 2, 1, 3).reshape(shape)


def _sdpa_grads(q, k, v, dout):
    qt, kt, vt = (_to_bhnd(x) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)
    (out * _to_bhnd(dout).detach()).sum().backward()
    return [_from_bhnd(t.grad, q.shape) for t in (qt, kt, vt)]


def test_full_window_backward_equals_dense_autograd():
    dims = (2, 3, 4)
    # float32-exact values, so the C oracle (which reads float32) sees the same inputs
    q, k, v, dout = (x.astype(np.float32).astype(np.float64) for x in _inputs(21, 2, dims, 3, 8))
    want = _sdpa_grads(q, k, v, dout)
    for got in (ref.gna_backward_loops(q, k, v, dout, dims, dims, (1, 1, 1)),
                oracle.backward_c(q, k, v, dout, dims, dims, (1, 1, 1), threads=3)):
        for g, w in zip(got, want):
            np.testing.assert_allclose(g, w, rtol=0, atol=1e-12)


def test_blocked_backward_equals_blockwise_autograd():
    dims, window = (4, 6, 4), (2, 3, 2)
    q, k, v, dout = _inputs(23, 1, dims, 2, 8)
    got = ref.gna_backward_loops(q, k, v, dout, dims, window, window)
    for bt, by, bx in itertools.product(*(range(L // w) for L, w in zip(dims, window))):
        sl = (slice(None), slice(bt * 2, bt * 2 + 2), slice(by * 3, by * 3 + 3), slice(bx * 2, bx * 2 + 2))
        want = _sdpa_grads(*(np.ascontiguousarray(x[sl]) for x in (q, k, v, dout)))
        for g, w in zip(got, want):
            np.testing.assert_allclose(g[sl], w, rtol=0, atol=1e-12)


def test_unit_window_gradients():
    """Window 1: out_i = v_i whatever q and k are."""
    dims = (2, 3, 5)
    q, k, v, dout = _inputs(24, 1, dims, 2, 16)
    dq, dk, dv = oracle.backward_c(q, k, v, dout, dims, (1, 1, 1), (1, 1, 1))
    np.testing.assert_array_equal(dv, dout.astype(np.float32).astype(np.float64))
    np.testing.assert_array_equal(dq, 0.0)
    np.testing.assert_array_equal(dk, 0.0)


@pytest.mark.parametrize("dims,window,stride,rule", [
    ((3, 6, 7), (2, 3, 5), (1, 2, 3), ref.LEADER_CENTER),
    ((2, 8, 9), (2, 4, 4), (2, 4, 4), ref.LEADER_LITERAL),
    ((1, 7, 11), (1, 7, 3), (1, 1, 2), ref.LEADER_CENTER),
])
def test_c_backward_equals_loops(dims, window, stride, rule):
    q, k, v, dout = (x.astype(np.float32) for x in _inputs(25, 2, dims, 3, 8))
    want = ref.gna_backward_loops(q, k, v, dout, dims, window, stride, rule=rule)
    got = oracle.backward_c(q, k, v, dout, dims, window, stride, rule=rule, threads=4)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dims,window,stride,rule", [
    ((3, 6, 7), (2, 3, 5), (1, 2, 3), ref.LEADER_CENTER),
    ((2, 8, 9), (2, 4, 4), (2, 4, 4), ref.LEADER_LITERAL),
])
def test_backward_identities(dims, window, stride, rule):
    """Identities of the derivative, true at any size:
    sum_j dv_j = sum_i dout_i (each query's probabilities sum to 1);
    sum_j dk_j = 0 (each query's row of dS sums to 0);
    sum_i <dq_i, q_i> = sum_j <dk_j, k_j> (both are sum_ij ds_ij s_ij)."""
    q, k, v, dout = _inputs(26, 2, dims, 3, 8)
    dq, dk, dv = ref.gna_backward_loops(q, k, v, dout, dims, window, stride, rule=rule)
    axes = (1, 2, 3)                                   # the grid; per batch, head and feature
    np.testing.assert_allclose(dv.sum(axis=axes), dout.sum(axis=axes), rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk.sum(axis=axes), 0.0, rtol=0, atol=1e-10)
    lhs = (dq * q).sum(axis=(1, 2, 3, 5))
    rhs = (dk * k).sum(axis=(1, 2, 3, 5))
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-10)


def test_selected_query_dq_matches_whole_planes():
    dims, window, stride = (3, 6, 7), (2, 3, 5), (1, 2, 3)
    q, k, v, dout = (x.astype(np.float32) for x in _inputs(27, 2, dims, 3, 8))
    dq, _, _ = oracle.backward_c(q, k, v, dout, dims, window, stride, threads=2)
    rng = np.random.default_rng(27)
    sel = np.array([tuple(int(rng.integers(0, n)) for n in (2, 3) + dims) for _ in range(40)])
    ids = oracle.query_ids(sel[:, 0], sel[:, 1], sel[:, 2], sel[:, 3], sel[:, 4], 3, dims)
    got = oracle.backward_dq_c(q, k, v, dout, dims, window, stride, ids, threads=3)
    np.testing.assert_allclose(got, dq[sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1]], rtol=0, atol=1e-12)


@pytest.mark.parametrize("dims,window,stride,rule", [
    ((3, 6, 7), (2, 3, 5), (1, 2, 3), ref.LEADER_CENTER),
    ((2, 8, 9), (2, 4, 4), (2, 4, 4), ref.LEADER_LITERAL),
])
def test_selected_key_dk_dv_match_whole_planes(dims, window, stride, rule):
    q, k, v, dout = (x.astype(np.float32) for x in _inputs(28, 2, dims, 3, 8))
    _, dk, dv = oracle.backward_c(q, k, v, dout, dims, window, stride, rule=rule, threads=2)
    rng = np.random.default_rng(28)
    sel = np.array([tuple(int(rng.integers(0, n)) for n in (2, 3) + dims) for _ in range(40)])
    ids = oracle.query_ids(sel[:, 0], sel[:, 1], sel[:, 2], sel[:, 3], sel[:, 4], 3, dims)
    gk, gv = oracle.backward_kv_c(q, k, v, dout, dims, window, stride, ids, rule=rule, threads=3)
    at = (sel[:, 0], sel[:, 2], sel[:, 3], sel[:, 4], sel[:, 1])
    np.testing.assert_allclose(gk, dk[at], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gv, dv[at], rtol=0, atol=1e-12)


def _jac_no_centering(p, dp):
    return p * dp


def _jac_no_p_factor(p, dp):
    return dp - (p * dp).sum()


def _jac_mean_centering(p, dp):
    return p * (dp - dp.mean())


@pytest.mark.parametrize("mutant", [_jac_no_centering, _jac_no_p_factor, _jac_mean_centering])
def test_planted_jacobian_mistakes_are_caught(monkeypatch, mutant):
    """Each slip fails the finite differences, and the identities as well."""
    monkeypatch.setattr(ref, "softmax_backward", mutant)
    assert _fd_errors((2, 5, 6), (2, 3, 3), (1, 1, 1), ref.LEADER_CENTER, seed=11) > 1e-4
    with pytest.raises(AssertionError):
        test_backward_identities((3, 6, 7), (2, 3, 5), (1, 2, 3), ref.LEADER_CENTER)
