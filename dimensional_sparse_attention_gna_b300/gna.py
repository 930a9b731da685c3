"""Thin ctypes binding of ``libgna_b300.so`` (C ABI in ``include/gna.h``).

Argument marshalling only: every function forwards device pointers, sizes and
the current CUDA stream to the C entry point of the same name and turns a
non-zero status into :class:`GNAError`.  All computation happens in the
library's CUDA kernels; there is no fallback.  PyTorch only provides device
memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

GNA_OK = 0
GNA_ERR_INVALID_ARG = 1
GNA_ERR_UNSUPPORTED = 2
GNA_ERR_CUDA = 3
GNA_ERR_TIMEOUT = 4

GNA_BF16 = 0
GNA_FP8_E4M3 = 1
GNA_F32 = 2

GNA_LEADER_CENTER = 0
GNA_LEADER_LITERAL = 1

TILE_ELEMS = 128

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgna_b300.so")

_DTYPE_CODES = {torch.bfloat16: GNA_BF16, torch.float8_e4m3fn: GNA_FP8_E4M3, torch.float32: GNA_F32}

_I3 = ctypes.c_int * 3
_P = ctypes.c_void_p
_INT = ctypes.c_int


class GNAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_status_name(status)}: {message}")
        self.status = status


def _status_name(s: int) -> str:
    return {0: "GNA_OK", 1: "GNA_ERR_INVALID_ARG", 2: "GNA_ERR_UNSUPPORTED", 3: "GNA_ERR_CUDA",
            4: "GNA_ERR_TIMEOUT"}.get(s, f"status {s}")


class GNAOptions(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int * 3), ("leader_rule", ctypes.c_int), ("scale", ctypes.c_float),
                ("descale", ctypes.c_void_p), ("tile_kv", ctypes.c_int * 3)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no other path."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m dimensional_sparse_attention_gna_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        st = ctypes.c_int
        i64 = ctypes.c_int64
        L.gna_version.restype = ctypes.c_int
        L.gna_status_string.restype = ctypes.c_char_p
        L.gna_status_string.argtypes = [st]
        L.gna_last_error.restype = ctypes.c_char_p
        L.gna_tile_shape.restype = st
        L.gna_tile_shape.argtypes = [_I3, _I3]
        L.gna_tiled_elems.restype = i64
        L.gna_tiled_elems.argtypes = [_INT, _INT, _I3, _P, _INT]
        for name in ("gna_permute", "gna_unpermute"):
            f = getattr(L, name)
            f.restype = st
            f.argtypes = [_P, _P, _INT, _INT, _I3, _INT, _INT, _P]
        for name in ("gna_permute_v", "gna_unpermute_v"):
            f = getattr(L, name)
            f.restype = st
            f.argtypes = [_P, _P, _INT, _INT, _I3, _INT, _INT, _P]
        for name in ("gna_permute_tiled", "gna_unpermute_tiled", "gna_permute_v_tiled", "gna_unpermute_v_tiled"):
            f = getattr(L, name)
            f.restype = st
            f.argtypes = [_P, _P, _INT, _INT, _I3, _I3, _INT, _INT, _P]
        L.gna_forward.restype = st
        L.gna_forward.argtypes = [_P, _P, _P, _P, _P, _INT, _INT, _I3, _I3, _I3, _INT, _INT, _P]
        L.gna_forward_ex.restype = st
        L.gna_forward_ex.argtypes = [_P, _P, _P, _P, _P, _INT, _INT, _I3, _I3, _I3, _INT, _INT,
                                     ctypes.POINTER(GNAOptions), _P]
        L.gna_forward_raster.restype = st
        L.gna_forward_raster.argtypes = L.gna_forward_ex.argtypes
        L.gna_forward_raster_all.restype = st
        L.gna_forward_raster_all.argtypes = L.gna_forward_ex.argtypes
        L.gna_forward_fp8.restype = st
        L.gna_forward_fp8.argtypes = [_P, _P, _P, _P, _P, _INT, _INT, _I3, _I3, _I3, _INT, _P, _P]
        L.gna_permuted_elems.restype = ctypes.c_size_t
        L.gna_permuted_elems.argtypes = [_INT, _INT, _I3, _INT]
        L.gna_test_skip_kv_load.restype = st
        L.gna_test_skip_kv_load.argtypes = [_INT, _INT]
        L.gna_backward_delta.restype = st
        L.gna_backward_delta.argtypes = [_P, _P, _P, _INT, _INT, _I3, _INT, _INT, ctypes.POINTER(GNAOptions), _P]
        L.gna_backward_dq.restype = st
        L.gna_backward_dq.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _INT, _INT, _I3, _I3, _I3, _INT, _INT,
                                      ctypes.POINTER(GNAOptions), _P]
        L.gna_backward_dkdv.restype = st
        L.gna_backward_dkdv.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _INT, _INT, _I3, _I3, _I3, _INT, _INT,
                                        ctypes.POINTER(GNAOptions), _P]
        L.gna_backward_noalloc.restype = st
        L.gna_backward_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _INT, _INT, _I3, _I3, _I3, _INT,
                                           _INT, ctypes.POINTER(GNAOptions), _P]
        L.gna_tile_stats.restype = st
        L.gna_tile_stats.argtypes = [_I3, _I3, _I3, _P, _INT, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                     ctypes.POINTER(i64)]
        L.gna_plan_tile.restype = st
        L.gna_plan_tile.argtypes = [_I3, _I3, _I3, _INT, _I3, ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double)]
        L.gna_tile_stats_qkv.restype = st
        L.gna_tile_stats_qkv.argtypes = [_I3, _I3, _I3, _P, _P, _INT, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                         ctypes.POINTER(i64)]
        L.gna_plan_tiles.restype = st
        L.gna_plan_tiles.argtypes = [_I3, _I3, _I3, _INT, _I3, _I3, ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_double)]
        L.gna_schedule_step.restype = st
        L.gna_schedule_step.argtypes = [_INT, _INT, _INT, _I3, _I3, _I3, _I3, _I3]
        L.gna_get_status.restype = st
        L.gna_get_status.argtypes = [_P]
        _lib = L
    return _lib


def _check(status: int):
    if status != GNA_OK:
        raise GNAError(status, lib().gna_last_error().decode())


def _stream_ptr(stream, device: torch.device | None = None) -> int | None:
    """The stream handle a call enqueues on.  ``device`` is the device of the
    call's tensors: the C ABI works on the current CUDA device (its TMA
    descriptors and launches assume it), so tensors elsewhere are refused."""
    if device is not None and device.type != "cuda":
        raise ValueError("tensors must live on a CUDA device")
    if device is not None:
        cur = torch.cuda.current_device()
        if device.index is not None and device.index != cur:
            raise ValueError(f"tensors live on {device}, but the current CUDA device is cuda:{cur}; "
                             "call under torch.cuda.device(...)")
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        if device is not None and stream.device != device:
            raise ValueError(f"stream of {stream.device} for tensors on {device}")
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _raster_elems(B: int, heads: int, dims, head_dim: int) -> int:
    return B * dims[0] * dims[1] * dims[2] * heads * head_dim


def _need(**tensors_and_sizes) -> torch.device | None:
    """Every tensor must hold at least the elements the call touches (the C ABI
    takes bare pointers and cannot check), and all must share one device, which
    is returned."""
    devices = set()
    for name, (t, n) in tensors_and_sizes.items():
        if t is None:
            continue
        if t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements, the call touches {n}")
        devices.add(t.device)
    if len(devices) > 1:
        raise ValueError(f"tensors on different devices: {sorted(map(str, devices))}")
    return next(iter(devices)) if devices else None


def dtype_code(dtype: torch.dtype) -> int:
    try:
        return _DTYPE_CODES[dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {dtype}") from None


def gna_version() -> int:
    return lib().gna_version()


def gna_tile_shape(dims) -> tuple[int, int, int]:
    out = _I3()
    _check(lib().gna_tile_shape(_I3(*dims), out))
    return tuple(out)


def gna_tiled_elems(B: int, heads: int, dims, head_dim: int, tile=None) -> int:
    t = None if tile is None else ctypes.cast(_I3(*tile), _P)
    n = lib().gna_tiled_elems(B, heads, _I3(*dims), t, head_dim)
    if n < 0:
        raise GNAError(GNA_ERR_INVALID_ARG, "invalid layout arguments")
    return n


def tiled_shape(B: int, heads: int, dims, head_dim: int, tile=None) -> tuple[int, ...]:
    """Shape ``[B, heads, tiles, 128, head_dim]`` of a tiled tensor."""
    n = gna_tiled_elems(B, heads, dims, head_dim, tile)
    return (B, heads, n // (B * heads * TILE_ELEMS * head_dim), TILE_ELEMS, head_dim)


def gna_permute(src: torch.Tensor, dst: torch.Tensor, B: int, heads: int, dims, head_dim: int,
                tile=None, stream=None):
    """Raster ``[B, T, H, W, heads, d]`` -> tiled ``[B, heads, tiles, 128, d]`` (zero padding)."""
    code = dtype_code(src.dtype)
    if dst.dtype != src.dtype:
        raise ValueError("src and dst dtypes differ")
    dev = _need(src=(src, _raster_elems(B, heads, dims, head_dim)),
                dst=(dst, gna_tiled_elems(B, heads, dims, head_dim, tile)))
    stream = _stream_ptr(stream, dev)
    if tile is None:
        st = lib().gna_permute(_ptr(src), _ptr(dst), B, heads, _I3(*dims), head_dim, code, stream)
    else:
        st = lib().gna_permute_tiled(_ptr(src), _ptr(dst), B, heads, _I3(*dims), _I3(*tile), head_dim, code,
                                     stream)
    _check(st)


def gna_unpermute(src: torch.Tensor, dst: torch.Tensor, B: int, heads: int, dims, head_dim: int,
                  tile=None, stream=None):
    """Tiled ``[B, heads, tiles, 128, d]`` -> raster ``[B, T, H, W, heads, d]``."""
    code = dtype_code(src.dtype)
    if dst.dtype != src.dtype:
        raise ValueError("src and dst dtypes differ")
    dev = _need(src=(src, gna_tiled_elems(B, heads, dims, head_dim, tile)),
                dst=(dst, _raster_elems(B, heads, dims, head_dim)))
    stream = _stream_ptr(stream, dev)
    if tile is None:
        st = lib().gna_unpermute(_ptr(src), _ptr(dst), B, heads, _I3(*dims), head_dim, code, stream)
    else:
        st = lib().gna_unpermute_tiled(_ptr(src), _ptr(dst), B, heads, _I3(*dims), _I3(*tile), head_dim, code,
                                       stream)
    _check(st)


def value_shape(B: int, heads: int, dims, head_dim: int, tile=None) -> tuple[int, ...]:
    """Shape ``[B, heads, tiles, head_dim, 128]`` of a tensor in the value layout."""
    s = tiled_shape(B, heads, dims, head_dim, tile)
    return (B, heads, s[2], head_dim, TILE_ELEMS)


def gna_permute_v(src: torch.Tensor, dst: torch.Tensor, B: int, heads: int, dims, head_dim: int,
                  tile=None, stream=None):
    """Raster ``[B, T, H, W, heads, d]`` -> value layout ``[B, heads, tiles, d, 128]`` (zero padding)."""
    code = dtype_code(src.dtype)
    if dst.dtype != src.dtype:
        raise ValueError("src and dst dtypes differ")
    dev = _need(src=(src, _raster_elems(B, heads, dims, head_dim)),
                dst=(dst, gna_tiled_elems(B, heads, dims, head_dim, tile)))
    stream = _stream_ptr(stream, dev)
    if tile is None:
        st = lib().gna_permute_v(_ptr(src), _ptr(dst), B, heads, _I3(*dims), head_dim, code, stream)
    else:
        st = lib().gna_permute_v_tiled(_ptr(src), _ptr(dst), B, heads, _I3(*dims), _I3(*tile), head_dim, code,
                                       stream)
    _check(st)


def gna_unpermute_v(src: torch.Tensor, dst: torch.Tensor, B: int, heads: int, dims, head_dim: int,
                    tile=None, stream=None):
    """Value layout ``[B, heads, tiles, d, 128]`` -> raster ``[B, T, H, W, heads, d]``."""
    code = dtype_code(src.dtype)
    if dst.dtype != src.dtype:
        raise ValueError("src and dst dtypes differ")
    dev = _need(src=(src, gna_tiled_elems(B, heads, dims, head_dim, tile)),
                dst=(dst, _raster_elems(B, heads, dims, head_dim)))
    stream = _stream_ptr(stream, dev)
    if tile is None:
        st = lib().gna_unpermute_v(_ptr(src), _ptr(dst), B, heads, _I3(*dims), head_dim, code, stream)
    else:
        st = lib().gna_unpermute_v_tiled(_ptr(src), _ptr(dst), B, heads, _I3(*dims), _I3(*tile), head_dim, code,
                                         stream)
    _check(st)


def _options(tile, leader_rule: int, scale: float, descale: torch.Tensor | None, tile_kv=None) -> GNAOptions:
    opt = GNAOptions()
    opt.tile = (ctypes.c_int * 3)(*(tile or (0, 0, 0)))
    opt.leader_rule = leader_rule
    opt.scale = scale
    opt.descale = _ptr(descale)
    opt.tile_kv = (ctypes.c_int * 3)(*(tile_kv or (0, 0, 0)))
    return opt


def _descale_arg(descale: torch.Tensor | None) -> torch.Tensor | None:
    if descale is not None and (descale.dtype != torch.float32 or descale.numel() != 3):
        raise ValueError("descale must be 3 float32 values")
    return descale


def gna_forward(q: torch.Tensor, k: torch.Tensor, v_value: torch.Tensor, out: torch.Tensor,
                lse: torch.Tensor | None, B: int, heads: int, dims, window, stride, head_dim: int, *, tile=None,
                leader_rule: int = GNA_LEADER_CENTER, scale: float = 0.0, descale: torch.Tensor | None = None,
                tile_kv=None, stream=None):
    """GNA forward on tiled tensors (see ``include/gna.h``).

    ``q, k``: bf16 or float8_e4m3fn, tiled; ``v_value``: same dtype, V in the
    VALUE layout (:func:`gna_permute_v`, not :func:`gna_permute`); ``out``:
    bf16 tiled; ``lse``: float32 ``[B, heads, tiles, 128]`` or None;
    ``descale``: float32 device tensor of 3 values, required for e4m3 and
    refused for bf16; ``tile_kv``: the tile of ``k`` and ``v_value`` when it
    differs from ``tile`` (the tile of ``q``, ``out``, ``lse``).  The plain bf16
    call goes to ``gna_forward``, an e4m3 call with default options to
    ``gna_forward_fp8``, anything else to ``gna_forward_ex``.
    """
    code = dtype_code(q.dtype)
    if k.dtype != q.dtype or v_value.dtype != q.dtype:
        raise ValueError("q, k, v_value must share a dtype")
    if out.dtype != torch.bfloat16:
        raise ValueError("out must be bfloat16")
    if lse is not None and lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    descale = _descale_arg(descale)
    nt = gna_tiled_elems(B, heads, dims, head_dim, tile)
    nkv = gna_tiled_elems(B, heads, dims, head_dim, tile_kv if tile_kv is not None else tile)
    dev = _need(q=(q, nt), k=(k, nkv), v_value=(v_value, nkv), out=(out, nt), lse=(lse, nt // head_dim),
                descale=(descale, 3))
    st_ptr = _stream_ptr(stream, dev)
    defaults = tile is None and tile_kv is None and leader_rule == GNA_LEADER_CENTER and scale == 0.0
    if defaults and code == GNA_BF16 and descale is None:
        st = lib().gna_forward(_ptr(q), _ptr(k), _ptr(v_value), _ptr(out), _ptr(lse), B, heads, _I3(*dims),
                               _I3(*window), _I3(*stride), head_dim, code, st_ptr)
    elif defaults and code == GNA_FP8_E4M3 and descale is not None:
        st = lib().gna_forward_fp8(_ptr(q), _ptr(k), _ptr(v_value), _ptr(out), _ptr(lse), B, heads, _I3(*dims),
                                   _I3(*window), _I3(*stride), head_dim, _ptr(descale), st_ptr)
    else:
        opt = _options(tile, leader_rule, scale, descale, tile_kv)
        st = lib().gna_forward_ex(_ptr(q), _ptr(k), _ptr(v_value), _ptr(out), _ptr(lse), B, heads, _I3(*dims),
                                  _I3(*window), _I3(*stride), head_dim, code, ctypes.byref(opt), st_ptr)
    _check(st)


def gna_forward_fp8(q: torch.Tensor, k: torch.Tensor, v_value: torch.Tensor, out: torch.Tensor,
                    lse: torch.Tensor | None, B: int, heads: int, dims, window, stride, head_dim: int,
                    descale: torch.Tensor, *, stream=None):
    """``gna_forward_fp8`` (see ``include/gna.h``): e4m3 codes, the 3 per-tensor
    descales of q, k, v on the device, bf16 ``out``."""
    if q.dtype != torch.float8_e4m3fn:
        raise ValueError("gna_forward_fp8 takes float8_e4m3fn q, k, v_value")
    if descale is None:
        raise ValueError("descale is required")
    gna_forward(q, k, v_value, out, lse, B, heads, dims, window, stride, head_dim, descale=descale, stream=stream)


def gna_forward_raster(q: torch.Tensor, k: torch.Tensor, v_value: torch.Tensor, out: torch.Tensor,
                       lse: torch.Tensor | None, B: int, heads: int, dims, window, stride, head_dim: int, *,
                       tile=None, leader_rule: int = GNA_LEADER_CENTER, scale: float = 0.0,
                       descale: torch.Tensor | None = None, tile_kv=None, stream=None):
    """GNA forward with q, k, out and lse in the raster layout (see ``include/gna.h``).

    ``q, k``: bf16 or float8_e4m3fn ``[B, T, H, W, heads, head_dim]``;
    ``v_value``: same dtype, value layout (:func:`gna_permute_v` with
    ``tile_kv``, else ``tile``); ``out``: bf16 raster; ``lse``: float32
    ``[B, T, H, W, heads]`` or None; ``descale`` as for :func:`gna_forward`.
    """
    code = dtype_code(q.dtype)
    if k.dtype != q.dtype or v_value.dtype != q.dtype:
        raise ValueError("q, k, v_value must share a dtype")
    if out.dtype != torch.bfloat16:
        raise ValueError("out must be bfloat16")
    if lse is not None and lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    descale = _descale_arg(descale)
    nr = _raster_elems(B, heads, dims, head_dim)
    nkv = gna_tiled_elems(B, heads, dims, head_dim, tile_kv if tile_kv is not None else tile)
    dev = _need(q=(q, nr), k=(k, nr), v_value=(v_value, nkv), out=(out, nr), lse=(lse, nr // head_dim),
                descale=(descale, 3))
    opt = _options(tile, leader_rule, scale, descale, tile_kv)
    _check(lib().gna_forward_raster(_ptr(q), _ptr(k), _ptr(v_value), _ptr(out), _ptr(lse), B, heads, _I3(*dims),
                                    _I3(*window), _I3(*stride), head_dim, code, ctypes.byref(opt),
                                    _stream_ptr(stream, dev)))


def gna_forward_raster_all(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                           lse: torch.Tensor | None, B: int, heads: int, dims, window, stride, head_dim: int, *,
                           tile=None, leader_rule: int = GNA_LEADER_CENTER, scale: float = 0.0, tile_kv=None,
                           stream=None):
    """GNA forward with every tensor in the raster layout (see ``include/gna.h``):
    q, k, v bf16 ``[B, T, H, W, heads, 128]``, ``out`` bf16 raster, ``lse`` float32
    ``[B, T, H, W, heads]`` or None.  No permute; slower P V than
    :func:`gna_forward_raster` with v in the value layout."""
    code = dtype_code(q.dtype)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share a dtype")
    if out.dtype != torch.bfloat16:
        raise ValueError("out must be bfloat16")
    if lse is not None and lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    nr = _raster_elems(B, heads, dims, head_dim)
    dev = _need(q=(q, nr), k=(k, nr), v=(v, nr), out=(out, nr), lse=(lse, nr // head_dim))
    opt = _options(tile, leader_rule, scale, None, tile_kv)
    _check(lib().gna_forward_raster_all(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, heads, _I3(*dims),
                                        _I3(*window), _I3(*stride), head_dim, code, ctypes.byref(opt),
                                        _stream_ptr(stream, dev)))


def gna_backward_delta(out: torch.Tensor, dout: torch.Tensor, delta: torch.Tensor, B: int, heads: int, dims,
                       head_dim: int, *, tile=None, stream=None):
    """delta = <dout, out> per tiled row (see ``include/gna.h``); bf16 in, float32 out."""
    if out.dtype != torch.bfloat16 or dout.dtype != torch.bfloat16 or delta.dtype != torch.float32:
        raise ValueError("out, dout must be bfloat16 and delta float32")
    nt = gna_tiled_elems(B, heads, dims, head_dim, tile)
    dev = _need(out=(out, nt), dout=(dout, nt), delta=(delta, nt // head_dim))
    opt = GNAOptions()
    opt.tile = (ctypes.c_int * 3)(*(tile or (0, 0, 0)))
    _check(lib().gna_backward_delta(_ptr(out), _ptr(dout), _ptr(delta), B, heads, _I3(*dims), head_dim, GNA_BF16,
                                    ctypes.byref(opt), _stream_ptr(stream, dev)))


def gna_backward_dq(q: torch.Tensor, k: torch.Tensor, k_value: torch.Tensor, v: torch.Tensor, dout: torch.Tensor,
                    lse: torch.Tensor, delta: torch.Tensor, dq: torch.Tensor, B: int, heads: int, dims, window,
                    stride, head_dim: int, *, tile=None, leader_rule: int = GNA_LEADER_CENTER, scale: float = 0.0,
                    stream=None):
    """dq of the GNA forward (see ``include/gna.h``): tiled bf16 tensors, ``k_value``
    in the value layout, the forward's tiled ``lse`` and ``delta`` from
    :func:`gna_backward_delta`."""
    for name, t in (("q", q), ("k", k), ("k_value", k_value), ("v", v), ("dout", dout), ("dq", dq)):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
    if lse.dtype != torch.float32 or delta.dtype != torch.float32:
        raise ValueError("lse and delta must be float32")
    nt = gna_tiled_elems(B, heads, dims, head_dim, tile)
    dev = _need(q=(q, nt), k=(k, nt), k_value=(k_value, nt), v=(v, nt), dout=(dout, nt), dq=(dq, nt),
                lse=(lse, nt // head_dim), delta=(delta, nt // head_dim))
    opt = GNAOptions()
    opt.tile = (ctypes.c_int * 3)(*(tile or (0, 0, 0)))
    opt.leader_rule = leader_rule
    opt.scale = scale
    _check(lib().gna_backward_dq(_ptr(q), _ptr(k), _ptr(k_value), _ptr(v), _ptr(dout), _ptr(lse), _ptr(delta),
                                 _ptr(dq), B, heads, _I3(*dims), _I3(*window), _I3(*stride), head_dim, GNA_BF16,
                                 ctypes.byref(opt), _stream_ptr(stream, dev)))


def gna_backward_dkdv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor, lse: torch.Tensor,
                      delta: torch.Tensor, dk: torch.Tensor, dv: torch.Tensor, B: int, heads: int, dims, window,
                      stride, head_dim: int, *, tile=None, leader_rule: int = GNA_LEADER_CENTER, scale: float = 0.0,
                      stream=None):
    """dk and dv of the GNA forward (see ``include/gna.h``): tiled bf16 tensors,
    the forward's tiled ``lse`` and ``delta`` from :func:`gna_backward_delta`."""
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout), ("dk", dk), ("dv", dv)):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
    if lse.dtype != torch.float32 or delta.dtype != torch.float32:
        raise ValueError("lse and delta must be float32")
    nt = gna_tiled_elems(B, heads, dims, head_dim, tile)
    dev = _need(q=(q, nt), k=(k, nt), v=(v, nt), dout=(dout, nt), dk=(dk, nt), dv=(dv, nt),
                lse=(lse, nt // head_dim), delta=(delta, nt // head_dim))
    opt = GNAOptions()
    opt.tile = (ctypes.c_int * 3)(*(tile or (0, 0, 0)))
    opt.leader_rule = leader_rule
    opt.scale = scale
    _check(lib().gna_backward_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(delta), _ptr(dk),
                                   _ptr(dv), B, heads, _I3(*dims), _I3(*window), _I3(*stride), head_dim, GNA_BF16,
                                   ctypes.byref(opt), _stream_ptr(stream, dev)))


def gna_backward_noalloc(q: torch.Tensor, k: torch.Tensor, k_value: torch.Tensor, v: torch.Tensor,
                         out: torch.Tensor, dout: torch.Tensor, lse: torch.Tensor, dq: torch.Tensor, dk: torch.Tensor,
                         dv: torch.Tensor, B: int, heads: int, dims, window, stride, head_dim: int, *, tile=None,
                         leader_rule: int = GNA_LEADER_CENTER, scale: float = 0.0, stream=None):
    """dq, dk and dv in one call that allocates nothing (see ``include/gna.h``):
    for callers that cannot allocate the delta workspace themselves.  The
    library keeps delta in a fixed device array (at most 2^22 tiled rows) that
    all calls share: calls must not overlap on the GPU."""
    for name, t in (("q", q), ("k", k), ("k_value", k_value), ("v", v), ("out", out), ("dout", dout), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    nt = gna_tiled_elems(B, heads, dims, head_dim, tile)
    dev = _need(q=(q, nt), k=(k, nt), k_value=(k_value, nt), v=(v, nt), out=(out, nt), dout=(dout, nt),
                lse=(lse, nt // head_dim), dq=(dq, nt), dk=(dk, nt), dv=(dv, nt))
    opt = GNAOptions()
    opt.tile = (ctypes.c_int * 3)(*(tile or (0, 0, 0)))
    opt.leader_rule = leader_rule
    opt.scale = scale
    _check(lib().gna_backward_noalloc(_ptr(q), _ptr(k), _ptr(k_value), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse),
                                      _ptr(dq), _ptr(dk), _ptr(dv), B, heads, _I3(*dims), _I3(*window),
                                      _I3(*stride), head_dim, GNA_BF16, ctypes.byref(opt), _stream_ptr(stream, dev)))


def gna_schedule_step(step: int, num_steps: int, full_steps: int, dims, window, stride):
    """(window, stride) for diffusion step ``step``: the whole grid with stride 1
    (full attention) for the first ``full_steps`` steps, then ``window``/``stride``."""
    w, s_ = _I3(), _I3()
    _check(lib().gna_schedule_step(step, num_steps, full_steps, _I3(*dims), _I3(*window), _I3(*stride), w, s_))
    return tuple(w), tuple(s_)


def gna_tile_stats(dims, window, stride, tile=None, leader_rule: int = GNA_LEADER_CENTER, *, tile_kv=None):
    """(visited KV tiles, KV tiles needing the element mask, Q tiles) of one (b, head) plane;
    with ``tile_kv`` (``gna_tile_stats_qkv``) the KV tiles have their own shape."""
    v, p_, q = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    t = None if tile is None else ctypes.cast(_I3(*tile), _P)
    if tile_kv is None:
        _check(lib().gna_tile_stats(_I3(*dims), _I3(*window), _I3(*stride), t, leader_rule,
                                    ctypes.byref(v), ctypes.byref(p_), ctypes.byref(q)))
    else:
        _check(lib().gna_tile_stats_qkv(_I3(*dims), _I3(*window), _I3(*stride), t, ctypes.cast(_I3(*tile_kv), _P),
                                        leader_rule, ctypes.byref(v), ctypes.byref(p_), ctypes.byref(q)))
    return v.value, p_.value, q.value


def gna_plan_tile(dims, window, stride, leader_rule: int = GNA_LEADER_CENTER):
    """(tile, tile_overhead, speedup_bound): the tile with the fewest visited 128 x 128
    tiles, its visited-over-useful work ratio and its speedup bound over dense attention."""
    t = _I3()
    ov, sp = ctypes.c_double(), ctypes.c_double()
    _check(lib().gna_plan_tile(_I3(*dims), _I3(*window), _I3(*stride), leader_rule, t, ctypes.byref(ov),
                               ctypes.byref(sp)))
    return tuple(t), ov.value, sp.value


def gna_plan_tiles(dims, window, stride, leader_rule: int = GNA_LEADER_CENTER):
    """(tile_q, tile_kv, tile_overhead, speedup_bound): the query and key/value tiles,
    chosen independently, with the fewest visited 128 x 128 tile pairs."""
    tq, tk = _I3(), _I3()
    ov, sp = ctypes.c_double(), ctypes.c_double()
    _check(lib().gna_plan_tiles(_I3(*dims), _I3(*window), _I3(*stride), leader_rule, tq, tk, ctypes.byref(ov),
                                ctypes.byref(sp)))
    return tuple(tq), tuple(tk), ov.value, sp.value


def gna_permuted_elems(B: int, heads: int, dims, head_dim: int) -> int:
    """Elements of one tensor written by :func:`gna_permute` under the default tile."""
    n = lib().gna_permuted_elems(B, heads, _I3(*dims), head_dim)
    if n == 0:
        raise GNAError(GNA_ERR_INVALID_ARG, "invalid layout arguments")
    return n


def gna_test_skip_kv_load(kernel: int, kv_index: int):
    """TEST ONLY (``gna_test_skip_kv_load``): kernel 0 = forward, 1 = dQ backward;
    kv_index < 0 turns the injected skipped load off."""
    _check(lib().gna_test_skip_kv_load(kernel, kv_index))


def gna_get_status(stream=None):
    """Synchronise the stream and raise if a kernel abandoned a pipeline wait."""
    _check(lib().gna_get_status(_stream_ptr(stream)))
