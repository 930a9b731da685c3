"""gna_attention: the differentiable operation on raster tensors (permutes, the
fused forward and the backward calls chained through the C ABI), against the
oracle's forward and gradients, and bit-identical to calling the entry points
directly."""
import numpy as np
import pytest
import torch

import oracle
from dimensional_sparse_attention_gna_b300 import gna_attention
from dimensional_sparse_attention_gna_b300 import gna as G
from synthetic_inputs import exact_f32, normal_raster, to_bf16
from tests.gpu_helpers import MAX_ERR_GRAD, REL_RMS_BF16, REL_RMS_GRAD, TOL_BF16_OUT, oracle_threads
from tests.test_gpu_backward import gpu_backward

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,dims,window,stride", [
    (64, (4, 16, 20), (3, 7, 9), (1, 2, 3)),
    (128, (1, 24, 40), (1, 9, 13), (1, 1, 1)),          # 2-D
    (32, (5, 19, 23), (3, 9, 11), (1, 1, 1)),            # ragged
])
def test_gna_attention_forward_and_gradients_match_the_oracle(d, dims, window, stride):
    B, heads, seed = 1, 2, 9900 + d
    q, k, v, g = (to_bf16(normal_raster(seed + i, B, dims, heads, d)) for i in range(4))
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev).requires_grad_() for x in (q, k, v))
    out = gna_attention(qd, kd, vd, window, stride)
    out.backward(g.to(dev))
    G.gna_get_status()
    torch.cuda.synchronize()
    o_ref, _ = oracle.forward_c(exact_f32(q), exact_f32(k), exact_f32(v), dims, window, stride,
                                    threads=oracle_threads())
    d_out = np.abs(out.detach().float().cpu().numpy().astype(np.float64) - o_ref)
    rel = float(np.sqrt((d_out ** 2).mean() / (o_ref ** 2).mean()))
    assert d_out.max() <= TOL_BF16_OUT and rel < REL_RMS_BF16, (d_out.max(), rel)
    refs = oracle.backward_c(exact_f32(q), exact_f32(k), exact_f32(v), exact_f32(g), dims, window, stride)
    for name, t, r in zip(("dq", "dk", "dv"), (qd, kd, vd), refs):
        got = t.grad.float().cpu().numpy()
        err = np.abs(got.astype(np.float64) - r)
        rel = float(np.sqrt((err ** 2).mean() / (r ** 2).mean()))
        info = f"{name}: max|err|={err.max():.3e} max|ref|={np.abs(r).max():.3e} relRMS={rel:.3e}"
        assert np.isfinite(got).all(), info
        assert rel < REL_RMS_GRAD and err.max() <= MAX_ERR_GRAD * np.abs(r).max(), info
    # the same kernels as the direct calls: identical gradients
    direct, _ = gpu_backward(q, k, v, g, dims, window, stride)
    for t, w in zip((qd, kd, vd), direct):
        np.testing.assert_array_equal(t.grad.float().cpu().numpy(), w)


def test_gna_attention_without_gradients_gives_the_same_output():
    """Inputs that need no gradient skip the backward's extra layouts; the
    forward's output is the same bytes."""
    B, heads, dims, d, window, stride = 1, 2, (4, 16, 20), 64, (3, 7, 9), (1, 2, 3)
    dev = torch.device("cuda")
    q, k, v = (to_bf16(normal_raster(9950 + i, B, dims, heads, d)).to(dev) for i in range(3))
    with torch.no_grad():
        a = gna_attention(q, k, v, window, stride)
    b = gna_attention(q.clone().requires_grad_(), k, v, window, stride)
    G.gna_get_status()
    assert not a.requires_grad and b.requires_grad
    assert torch.equal(a.view(torch.int16), b.detach().view(torch.int16))
