"""The C ABI under CUDA graph capture: every entry point of the forward step
(permutes, forward, unpermutes) and of the backward pass enqueues kernels only,
with no allocation and no synchronisation, so a whole step can be captured once
and replayed.  A replay on new input values (written into the captured buffers)
must give the same bytes as running the calls eagerly on those values.
"""
import pytest
import torch

from dimensional_sparse_attention_gna_b300 import gna as G
from synthetic_inputs import normal_raster, to_bf16

pytestmark = pytest.mark.gpu


def _raster(seed, B, dims, heads, d, dev):
    return to_bf16(normal_raster(seed, B, dims, heads, d)).to(dev)


def test_forward_step_replays_from_a_cuda_graph():
    dims, window, stride, B, heads, d = (6, 20, 24), (4, 9, 8), (2, 3, 8), 1, 3, 128
    dev = torch.device("cuda")
    q, k, v = (_raster(9800 + i, B, dims, heads, d, dev) for i in range(3))
    shp = G.tiled_shape(B, heads, dims, d)
    qt, kt = torch.empty(shp, dtype=torch.bfloat16, device=dev), torch.empty(shp, dtype=torch.bfloat16, device=dev)
    vt = torch.empty(G.value_shape(B, heads, dims, d), dtype=torch.bfloat16, device=dev)
    out_t = torch.empty(shp, dtype=torch.bfloat16, device=dev)
    lse_t = torch.empty(shp[:-1], dtype=torch.float32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1] + (1,), dtype=torch.float32, device=dev)

    def step():
        G.gna_permute(q, qt, B, heads, dims, d)
        G.gna_permute(k, kt, B, heads, dims, d)
        G.gna_permute_v(v, vt, B, heads, dims, d)
        G.gna_forward(qt, kt, vt, out_t, lse_t, B, heads, dims, window, stride, d)
        G.gna_unpermute(out_t, out, B, heads, dims, d)
        G.gna_unpermute(lse_t.unsqueeze(-1), lse, B, heads, dims, 1)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):           # first calls (one-time set-up) outside the capture
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (9900, 9910):
        for i, x in enumerate((q, k, v)):
            x.copy_(_raster(seed + i, B, dims, heads, d, dev))
        graph.replay()
        torch.cuda.synchronize()
        got_out, got_lse = out.clone(), lse.clone()
        step()                               # the same calls, eagerly
        G.gna_get_status()
        torch.cuda.synchronize()
        assert torch.equal(got_out.view(torch.int16), out.view(torch.int16))
        assert torch.equal(got_lse, lse)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_backward_replays_from_a_cuda_graph(d):
    dims, window, stride, B, heads = (6, 20, 24), (4, 9, 8), (2, 3, 8), 1, 2
    dev = torch.device("cuda")
    shp = G.tiled_shape(B, heads, dims, d)
    t = {}
    for i, name in enumerate(("q", "k", "v", "dout")):
        t[name] = torch.empty(shp, dtype=torch.bfloat16, device=dev)
        G.gna_permute(_raster(9950 + i, B, dims, heads, d, dev), t[name], B, heads, dims, d)
    k_value = torch.empty(G.value_shape(B, heads, dims, d), dtype=torch.bfloat16, device=dev)
    v_value = torch.empty_like(k_value)
    out = torch.empty(shp, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(shp[:-1], dtype=torch.float32, device=dev)
    delta = torch.empty_like(lse)
    dq, dk, dv = (torch.empty(shp, dtype=torch.bfloat16, device=dev) for _ in range(3))

    def step():
        # the forward's value layouts straight from the tiled tensors: each tile transposed
        k_value.copy_(t["k"].view(-1, 128, d).transpose(1, 2).reshape(k_value.shape))
        v_value.copy_(t["v"].view(-1, 128, d).transpose(1, 2).reshape(v_value.shape))
        G.gna_forward(t["q"], t["k"], v_value, out, lse, B, heads, dims, window, stride, d)
        G.gna_backward_delta(out, t["dout"], delta, B, heads, dims, d)
        G.gna_backward_dq(t["q"], t["k"], k_value, t["v"], t["dout"], lse, delta, dq, B, heads, dims, window,
                          stride, d)
        G.gna_backward_dkdv(t["q"], t["k"], t["v"], t["dout"], lse, delta, dk, dv, B, heads, dims, window, stride, d)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for i, name in enumerate(("q", "k", "v", "dout")):
        G.gna_permute(_raster(9960 + i, B, dims, heads, d, dev), t[name], B, heads, dims, d)
    graph.replay()
    torch.cuda.synchronize()
    got = [x.clone() for x in (out, dq, dk, dv)]
    step()
    G.gna_get_status()
    torch.cuda.synchronize()
    for g, w in zip(got, (out, dq, dk, dv)):
        assert torch.equal(g.view(torch.int16), w.view(torch.int16))
