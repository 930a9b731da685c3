"""CPU oracle of the GNA forward pass and its gradients -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
library never does, and the oracle shares no code, header, table or helper with
the CUDA sources under ``dimensional_sparse_attention_gna_b300/csrc``.

Contents
--------
* :mod:`oracle.reference` -- the definition in NumPy / torch-CPU float64 (one
  query at a time, and the same quantity as masked dense attention).
* :mod:`oracle.layout`    -- the tile-major layout definition (reshape/transpose).
* ``gna_oracle.c``        -- the same definition in plain C, threaded over
  queries, float64 accumulation; wrapped here by :func:`forward_c`; and its
  derivative (the backward pass), threaded over (b, head) planes, wrapped by
  :func:`backward_c`, its dq at selected queries (:func:`backward_dq_c`) and its
  dk, dv at selected keys (:func:`backward_kv_c`), cheap enough for samples of
  the full-size workloads.

Every function is pinned by ``tests/test_oracle_pins.py`` (the backward by
``tests/test_oracle_backward_pins.py``) against hand-derived
tables, closed forms, special cases that reduce to library routines, brute
force and invariants.  Parity of the large workloads is checked on sampled
queries, which this C oracle computes one by one.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .reference import LEADER_CENTER, LEADER_LITERAL, default_scale  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gna_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libgna_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gna_oracle.c`` with gcc into ``oracle/_build/libgna_oracle.so``."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.gna_oracle_forward.restype = ctypes.c_int
            lib.gna_oracle_forward.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.gna_oracle_backward.restype = ctypes.c_int
            lib.gna_oracle_backward.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.gna_oracle_backward_dq_sel.restype = ctypes.c_int
            lib.gna_oracle_backward_dq_sel.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
            lib.gna_oracle_backward_kv_sel.restype = ctypes.c_int
            lib.gna_oracle_backward_kv_sel.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
            lib.gna_oracle_window_starts.restype = None
            lib.gna_oracle_window_starts.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_void_p]
            _lib = lib
    return _lib


def _rule_code(rule: str) -> int:
    if rule == LEADER_CENTER:
        return 0
    if rule == LEADER_LITERAL:
        return 1
    raise ValueError(rule)


def window_starts_c(L: int, w: int, s: int, rule: str = LEADER_CENTER) -> np.ndarray:
    out = np.zeros(L, dtype=np.int32)
    _load().gna_oracle_window_starts(L, w, s, _rule_code(rule), out.ctypes.data)
    return out


def query_ids(b, h, t, y, x, heads, dims) -> np.ndarray:
    """Flat query ids ``((b*heads + h)*N + (t*H + y)*W + x)`` used by :func:`forward_c`."""
    T, H, W = dims
    n = T * H * W
    return ((np.asarray(b, np.int64) * heads + np.asarray(h, np.int64)) * n
            + (np.asarray(t, np.int64) * H + np.asarray(y, np.int64)) * W + np.asarray(x, np.int64))


def forward_c(q, k, v, dims, window, stride, scale=None, rule=LEADER_CENTER,
              tensor_scales=(1.0, 1.0, 1.0), sel=None, threads=None):
    """Run the C oracle.

    ``q, k, v``: float32 rasters ``[B, T, H, W, heads, d]`` holding the exact
    input values (bf16 values or e4m3 codes); ``tensor_scales`` multiplies each
    tensor (e4m3 dequantisation).  ``sel``: flat query ids (see
    :func:`query_ids`) or None for every query.  Returns ``(out, lse)`` float64:
    ``out [nsel, d]`` and ``lse [nsel]`` for a selection, or raster-shaped
    ``[B, T, H, W, heads, d]`` / ``[B, T, H, W, heads]`` when ``sel`` is None.
    """
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    B, T, H, W, heads, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and (T, H, W) == tuple(dims)
    if scale is None:
        scale = default_scale(d)
    if threads is None:
        threads = os.cpu_count() or 1
    n_all = B * heads * T * H * W
    if sel is None:
        nsel, selp = n_all, None
    else:
        sel = np.ascontiguousarray(sel, dtype=np.int64)
        nsel, selp = sel.size, sel.ctypes.data
    out = np.empty((nsel, d), dtype=np.float64)
    lse = np.empty((nsel,), dtype=np.float64)
    arr3 = ctypes.c_int * 3
    rc = _load().gna_oracle_forward(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, B, heads,
        arr3(*dims), arr3(*window), arr3(*stride), d, _rule_code(rule),
        float(scale), float(tensor_scales[0]), float(tensor_scales[1]), float(tensor_scales[2]),
        selp, nsel, out.ctypes.data, lse.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"gna_oracle_forward failed with {rc}")
    if sel is None:
        # flat order is (b, h, token): move heads after the grid
        out = out.reshape(B, heads, T, H, W, d).transpose(0, 2, 3, 4, 1, 5)
        lse = lse.reshape(B, heads, T, H, W).transpose(0, 2, 3, 4, 1)
        return np.ascontiguousarray(out), np.ascontiguousarray(lse)
    return out, lse


def backward_c(q, k, v, dout, dims, window, stride, scale=None, rule=LEADER_CENTER, threads=None):
    """Run the C backward oracle: ``(dq, dk, dv)`` float64 rasters for the loss
    ``sum(dout * out)``.  ``q, k, v, dout``: float32 rasters
    ``[B, T, H, W, heads, d]`` holding the exact input values."""
    q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
    B, T, H, W, heads, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and dout.shape == q.shape and (T, H, W) == tuple(dims)
    if scale is None:
        scale = default_scale(d)
    if threads is None:
        threads = os.cpu_count() or 1
    dq, dk, dv = (np.empty(q.shape, dtype=np.float64) for _ in range(3))
    arr3 = ctypes.c_int * 3
    rc = _load().gna_oracle_backward(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, heads,
        arr3(*dims), arr3(*window), arr3(*stride), d, _rule_code(rule), float(scale),
        dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"gna_oracle_backward failed with {rc}")
    return dq, dk, dv


def backward_dq_c(q, k, v, dout, dims, window, stride, sel, scale=None, rule=LEADER_CENTER, threads=None):
    """dq of the selected queries (flat ids, see :func:`query_ids`): float64 ``[nsel, d]``."""
    q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
    B, T, H, W, heads, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and dout.shape == q.shape and (T, H, W) == tuple(dims)
    if scale is None:
        scale = default_scale(d)
    if threads is None:
        threads = os.cpu_count() or 1
    sel = np.ascontiguousarray(sel, dtype=np.int64)
    dq = np.empty((sel.size, d), dtype=np.float64)
    arr3 = ctypes.c_int * 3
    rc = _load().gna_oracle_backward_dq_sel(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, heads,
        arr3(*dims), arr3(*window), arr3(*stride), d, _rule_code(rule), float(scale),
        sel.ctypes.data, sel.size, dq.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"gna_oracle_backward_dq_sel failed with {rc}")
    return dq


def backward_kv_c(q, k, v, dout, dims, window, stride, sel, scale=None, rule=LEADER_CENTER, threads=None):
    """dk and dv of the selected keys (flat ids, see :func:`query_ids`): two
    float64 arrays ``[nsel, d]``.  Computes lse and delta for every query of the
    planes that hold a selected key first (O(N |W| d) per plane)."""
    q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
    B, T, H, W, heads, d = q.shape
    assert k.shape == q.shape and v.shape == q.shape and dout.shape == q.shape and (T, H, W) == tuple(dims)
    if scale is None:
        scale = default_scale(d)
    if threads is None:
        threads = os.cpu_count() or 1
    sel = np.ascontiguousarray(sel, dtype=np.int64)
    dk = np.empty((sel.size, d), dtype=np.float64)
    dv = np.empty((sel.size, d), dtype=np.float64)
    arr3 = ctypes.c_int * 3
    rc = _load().gna_oracle_backward_kv_sel(
        q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, B, heads,
        arr3(*dims), arr3(*window), arr3(*stride), d, _rule_code(rule), float(scale),
        sel.ctypes.data, sel.size, dk.ctypes.data, dv.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError(f"gna_oracle_backward_kv_sel failed with {rc}")
    return dk, dv
