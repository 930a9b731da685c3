"""gna_backward_noalloc: the backward pass for callers that cannot allocate
device memory (a framework's own memory pool or arena that owns every
allocation, a fixed allocation budget, host code that must not call
cudaMalloc).  It keeps the delta workspace in a fixed array of the library's
device memory instead of a caller-owned buffer.

The GPU test calls it through the C ABI twice in a row, on two different
problems, and compares each result with the regular entry points
(gna_backward_delta, gna_backward_dq, gna_backward_dkdv with a caller-owned
delta) on the same inputs: within the backward tests' tolerance, and in fact
byte for byte, since the same kernels run on the same values.  The second call
is smaller than the first, so it runs over whatever the first left in the
shared array.

This file is named to be collected last, so that a run stopping at its first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from dimensional_sparse_attention_gna_b300 import gna as G
from synthetic_inputs import normal_raster, to_bf16
from tests.gpu_helpers import MAX_ERR_GRAD, REL_RMS_GRAD

I3 = ctypes.c_int * 3
FAKE = 0x10000   # never dereferenced: the call below fails validation first


def test_no_alloc_backward_rejects_sizes_beyond_its_workspace():
    """Host only: a problem with more tiled rows than the static workspace holds
    (64 heads of the 30x48x80 grid: 7,372,800 > 2^22) is refused before any
    launch, with a message naming the limit."""
    L = G.lib()
    st = L.gna_backward_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, I3(30, 48, 80),
                                I3(16, 32, 48), I3(1, 1, 1), 128, G.GNA_BF16, None, None)
    assert st == G.GNA_ERR_INVALID_ARG
    msg = L.gna_last_error().decode()
    assert "4194304" in msg and "static workspace" in msg, msg
    # the 720p-video latent at 24 heads fits (argument checks pass up to the
    # size check; a NULL pointer is then the first error)
    st = L.gna_backward_noalloc(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 24, I3(30, 48, 80),
                                I3(16, 32, 48), I3(1, 1, 1), 128, G.GNA_BF16, None, None)
    assert st == G.GNA_ERR_INVALID_ARG and "NULL" in L.gna_last_error().decode()


def _problem(seed, B, heads, dims, window, stride, d):
    """Tiled bf16 inputs on the GPU and the forward's out and lse."""
    dev = torch.device("cuda")
    shp = G.tiled_shape(B, heads, dims, d)
    x = {}
    for i, name in enumerate(("q", "k", "v", "dout")):
        r = to_bf16(normal_raster(seed + i, B, dims, heads, d)).to(dev)
        t = torch.empty(shp, dtype=torch.bfloat16, device=dev)
        G.gna_permute(r, t, B, heads, dims, d)
        x[name] = t
        if name in ("k", "v"):
            tv = torch.empty(G.value_shape(B, heads, dims, d), dtype=torch.bfloat16, device=dev)
            G.gna_permute_v(r, tv, B, heads, dims, d)
            x[name + "_value"] = tv
    x["out"] = torch.empty(shp, dtype=torch.bfloat16, device=dev)
    x["lse"] = torch.empty(shp[:-1], dtype=torch.float32, device=dev)
    G.gna_forward(x["q"], x["k"], x["v_value"], x["out"], x["lse"], B, heads, dims, window, stride, d)
    return x


def _regular_backward(x, B, heads, dims, window, stride, d):
    delta = torch.empty(x["lse"].shape, dtype=torch.float32, device=x["q"].device)
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    G.gna_backward_delta(x["out"], x["dout"], delta, B, heads, dims, d)
    G.gna_backward_dq(x["q"], x["k"], x["k_value"], x["v"], x["dout"], x["lse"], delta, dq, B, heads, dims, window,
                      stride, d)
    G.gna_backward_dkdv(x["q"], x["k"], x["v"], x["dout"], x["lse"], delta, dk, dv, B, heads, dims, window,
                        stride, d)
    return dq, dk, dv


def _no_alloc_backward(x, B, heads, dims, window, stride, d):
    dq, dk, dv = (torch.empty_like(x["q"]) for _ in range(3))
    G.gna_backward_noalloc(x["q"], x["k"], x["k_value"], x["v"], x["out"], x["dout"], x["lse"], dq, dk, dv, B,
                           heads, dims, window, stride, d)
    return dq, dk, dv


@pytest.mark.gpu
def test_no_alloc_backward_matches_regular_entry_points_twice_in_a_row():
    problems = [
        (9100, 2, 3, (6, 20, 24), (4, 9, 8), (2, 3, 8), 128),   # larger: fills more of the shared array
        (9200, 1, 2, (3, 17, 19), (3, 7, 5), (1, 2, 1), 128),   # smaller, ragged: runs over the first's leftovers
        (9250, 1, 2, (5, 19, 23), (3, 9, 11), (1, 2, 3), 64),   # head_dim 64
        (9260, 2, 2, (3, 17, 19), (3, 7, 5), (1, 2, 1), 32),    # head_dim 32
    ]
    for seed, B, heads, dims, window, stride, d in problems:
        x = _problem(seed, B, heads, dims, window, stride, d)
        got = _no_alloc_backward(x, B, heads, dims, window, stride, d)
        want = _regular_backward(x, B, heads, dims, window, stride, d)
        G.gna_get_status()
        torch.cuda.synchronize()
        for name, g, w in zip(("dq", "dk", "dv"), got, want):
            gf, wf = g.double().cpu().numpy(), w.double().cpu().numpy()
            err = np.abs(gf - wf)
            rel = float(np.sqrt((err ** 2).mean() / max((wf ** 2).mean(), 1e-30)))
            info = f"{dims} {name}: max|diff|={err.max():.3e} relRMS={rel:.3e}"
            # the backward tests' tolerance ...
            assert np.isfinite(gf).all(), info
            assert rel < REL_RMS_GRAD and err.max() <= MAX_ERR_GRAD * np.abs(wf).max(), info
            # ... and, the kernels being the same, identical bytes
            assert torch.equal(g.view(torch.int16), w.view(torch.int16)), info
