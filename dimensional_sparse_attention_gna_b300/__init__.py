"""B300 (sm_103a) Generalized Neighborhood Attention forward.

The compute lives in ``libgna_b300.so`` (CUDA kernels behind the C ABI in
``include/gna.h``); :mod:`.gna` is its thin ctypes binding, and
:func:`gna_attention` (:mod:`.attention`) the differentiable operation on raster
tensors built from those calls.
"""
from .gna import (  # noqa: F401
    GNA_BF16, GNA_F32, GNA_FP8_E4M3, GNA_LEADER_CENTER, GNA_LEADER_LITERAL, GNAError, TILE_ELEMS,
    gna_forward, gna_get_status, gna_permute, gna_tile_shape, gna_tile_stats, gna_tiled_elems, gna_unpermute,
    gna_version, lib, tiled_shape,
)
from .attention import gna_attention  # noqa: F401
