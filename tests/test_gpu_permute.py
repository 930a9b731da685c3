"""gna_permute / gna_unpermute and gna_permute_v / gna_unpermute_v against the
layout definitions: bit-exact."""
import numpy as np
import pytest
import torch

from dimensional_sparse_attention_gna_b300 import gna as G
from oracle import layout
from synthetic_inputs import normal_raster

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    itemsize = t.element_size()
    view = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[itemsize]
    return t.view(view).cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float8_e4m3fn, torch.float32])
@pytest.mark.parametrize("B,heads,dims,d,tile", [
    (1, 2, (1, 16, 16), 32, None),
    (2, 3, (3, 5, 7), 8, None),
    (1, 4, (5, 24, 40), 128, (1, 8, 16)),
    (2, 1, (6, 20, 24), 64, (2, 4, 16)),
    (1, 2, (2, 40, 40), 16, (1, 1, 128)),
    (1, 3, (4, 9, 9), 1, (4, 4, 8)),        # d = 1: the lse path for float32 (4-byte rows)
])
def test_permute_matches_layout_definition(dtype, B, heads, dims, d, tile):
    if d * torch.tensor([], dtype=dtype).element_size() % 4:
        pytest.skip("row must be a multiple of 4 bytes")
    x = torch.from_numpy(normal_raster(7, B, dims, heads, d)).to(dtype)
    t = tile or G.gna_tile_shape(dims)
    want = layout.permute_reference(_bits(x), t)
    xd = x.cuda()
    shape = G.tiled_shape(B, heads, dims, d, tile)
    nbytes = int(np.prod(shape)) * x.element_size()
    y = torch.full((nbytes,), 0x55, dtype=torch.uint8, device="cuda").view(dtype).reshape(shape)   # poison
    G.gna_permute(xd, y, B, heads, dims, d, tile=tile)
    got = _bits(y).reshape(want.shape)
    np.testing.assert_array_equal(got, want)
    back = torch.zeros_like(xd)
    G.gna_unpermute(y, back, B, heads, dims, d, tile=tile)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(back), _bits(x))


@pytest.mark.parametrize("B,heads,dims,dtype", [
    (1, 24, (30, 48, 80), torch.bfloat16),
    (1, 24, (1, 256, 256), torch.bfloat16),
    (2, 24, (30, 48, 80), torch.float8_e4m3fn),
])
def test_permute_full_size_round_trip_and_samples(B, heads, dims, dtype):
    d = 128
    gen = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn((B,) + dims + (heads, d), device="cuda", generator=gen).to(dtype)
    y = torch.empty(G.tiled_shape(B, heads, dims, d), dtype=dtype, device="cuda")
    G.gna_permute(x, y, B, heads, dims, d)
    back = torch.empty_like(x)
    G.gna_unpermute(y, back, B, heads, dims, d)
    torch.cuda.synchronize()
    assert torch.equal(_bits_gpu(back), _bits_gpu(x))
    # sampled rows against the layout definition's index map
    tile = G.gna_tile_shape(dims)
    rng = np.random.default_rng(3)
    yr = y.reshape(-1, d)
    for _ in range(256):
        b, h = int(rng.integers(B)), int(rng.integers(heads))
        t, yy, xx = (int(rng.integers(L)) for L in dims)
        r = layout.tiled_row(b, h, t, yy, xx, heads, dims, tile)
        assert torch.equal(_bits_gpu(yr[r]), _bits_gpu(x[b, t, yy, xx, h]))


def _bits_gpu(t):
    view = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[t.element_size()]
    return t.view(view)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float8_e4m3fn])
@pytest.mark.parametrize("B,heads,dims,d,tile", [
    (1, 2, (1, 16, 16), 32, None),
    (2, 3, (3, 5, 7), 64, None),             # every tile padded
    (1, 4, (5, 24, 40), 128, (1, 8, 16)),
    (2, 1, (6, 20, 24), 128, (2, 4, 16)),
    (1, 2, (2, 40, 40), 16, (1, 1, 128)),
    (1, 1, (2, 16, 16), 256, None),          # 256-byte feature rows at 1 byte
])
def test_value_permute_matches_layout_definition(dtype, B, heads, dims, d, tile):
    esz = torch.tensor([], dtype=dtype).element_size()
    rb = d * esz
    if rb < 16 or rb > 256 or rb & (rb - 1):
        pytest.skip("value layout rows are a power of two from 16 to 256 bytes")
    x = torch.from_numpy(normal_raster(8, B, dims, heads, d)).to(dtype)
    t = tile or G.gna_tile_shape(dims)
    want = layout.permute_v_reference(_bits(x), t)
    xd = x.cuda()
    shape = G.value_shape(B, heads, dims, d, tile)
    nbytes = int(np.prod(shape)) * x.element_size()
    y = torch.full((nbytes,), 0x55, dtype=torch.uint8, device="cuda").view(dtype).reshape(shape)   # poison
    G.gna_permute_v(xd, y, B, heads, dims, d, tile=tile)
    got = _bits(y).reshape(want.shape)
    np.testing.assert_array_equal(got, want)
    back = torch.zeros_like(xd)
    G.gna_unpermute_v(y, back, B, heads, dims, d, tile=tile)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(back), _bits(x))


@pytest.mark.parametrize("B,heads,dims,dtype", [
    (1, 24, (30, 48, 80), torch.bfloat16),
    (2, 24, (30, 48, 80), torch.float8_e4m3fn),
])
def test_value_permute_full_size_round_trip_and_samples(B, heads, dims, dtype):
    d = 128
    gen = torch.Generator(device="cuda").manual_seed(12)
    x = torch.randn((B,) + dims + (heads, d), device="cuda", generator=gen).to(dtype)
    y = torch.empty(G.value_shape(B, heads, dims, d), dtype=dtype, device="cuda")
    G.gna_permute_v(x, y, B, heads, dims, d)
    back = torch.empty_like(x)
    G.gna_unpermute_v(y, back, B, heads, dims, d)
    torch.cuda.synchronize()
    assert torch.equal(_bits_gpu(back), _bits_gpu(x))
    # sampled tokens: feature column of the token's tile equals the raster row
    tile = G.gna_tile_shape(dims)
    rng = np.random.default_rng(4)
    yt = y.reshape(-1, d, 128)
    for _ in range(256):
        b, h = int(rng.integers(B)), int(rng.integers(heads))
        t, yy, xx = (int(rng.integers(L)) for L in dims)
        r = layout.tiled_row(b, h, t, yy, xx, heads, dims, tile)
        assert torch.equal(_bits_gpu(yt[r // 128, :, r % 128].contiguous()), _bits_gpu(x[b, t, yy, xx, h]))
