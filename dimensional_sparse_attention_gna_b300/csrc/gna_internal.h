// Internal interface between the C-ABI shim (gna_api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gna.h"

namespace gna {

// Records a printf-style message as the calling thread's gna_last_error() and
// returns `s` (defined with the C ABI in gna_api.cu).
gna_status api_fail(gna_status s, const char* fmt, ...);

// Geometry of one permute / unpermute launch.
struct PermuteGeom {
    int64_t B;
    int heads;
    int dims[3];          // T, H, W
    int nt[3];            // tiles per dimension
    int tlog[3];          // log2 of the tile extent per dimension
    int ntiles_total;     // nt[0] * nt[1] * nt[2]
    int row_bytes;        // head_dim * element size (multiple of 4)
};

cudaError_t launch_permute(const void* src, void* dst, const PermuteGeom& g, bool to_tiled, cudaStream_t stream);

// Raster <-> value layout (each tile stored feature-major, d x 128).  Element
// size 1 or 2 bytes, row_bytes a power of two from 16 to kMaxValueRowBytes;
// returns cudaErrorNotSupported otherwise.
constexpr int kMaxValueRowBytes = 256;
cudaError_t launch_permute_v(const void* src, void* dst, const PermuteGeom& g, int elem_size, bool to_tiled,
                             cudaStream_t stream);

// Parameters of one attention launch (passed by value as a __grid_constant__).
struct FwdParams {
    CUtensorMap tmK;             // 2-D TMA view [rows, head_dim] of the tiled k, or (raster) the
                                 // 5-D view [B, T, H, W, heads * head_dim] of the raster k
    CUtensorMap tmV;             // 2-D TMA view [rows * head_dim / 128, 128] of v in the value layout, or
                                 // (raster == 2) the 5-D view of the raster v, like tmK
    const void* q;               // tiled q [rows, head_dim], or raster q (read row by row into TMEM)
    int raster;                  // 1: q, k, out and lse use the raster layout (v in the value layout);
                                 // 2: v too (bf16, head_dim 128)
    void* out;                   // tiled bf16 [rows, head_dim]
    float* lse;                  // tiled float [rows] or nullptr
    const float* descale;        // e4m3 only: 3 device floats (q, k, v) or nullptr
    int dims[3], win[3], str[3], off[3];
    int tile[3], tlog[3], nt[3];  // key / value tiles (layout of k and v, the KV tile box)
    int tile_q[3], tlog_q[3], nt_q[3];   // query tiles (layout of q, out and lse; one per CTA)
    int heads;
    int tiles_per_head;          // KV tiles per (b, head) plane: nt[0] * nt[1] * nt[2]
    int tiles_per_head_q;        // query tiles per plane: nt_q[0] * nt_q[1] * nt_q[2]
    float scale;                 // softmax scale
    int fault_skip_kv;           // test hook: >= 0 makes the producer skip that KV load
};

// Launches the fused forward kernel for (head_dim, element size) on `stream`
// over `num_q_tiles` CTAs.  Returns cudaErrorNotSupported for a head_dim /
// dtype pair without a kernel.
cudaError_t launch_forward(const FwdParams& p, int head_dim, int elem_size, int64_t num_q_tiles,
                           cudaStream_t stream);

// Device status word: read-and-clear.
cudaError_t read_and_clear_status(int* status, cudaStream_t stream);

// Parameters of one dQ launch of the backward pass (bf16, head_dim 32, 64 or 128;
// all tensors tiled except kv, which is k in the value layout).
struct BwdParams {
    CUtensorMap tmK;             // 2-D TMA view [rows, head_dim] of the tiled k
    CUtensorMap tmV;             // 2-D TMA view [rows, head_dim] of the tiled v
    CUtensorMap tmKv;            // 2-D TMA view [tiles * head_dim, 128] of k in the value layout
    CUtensorMap tmDO;            // 2-D TMA view [rows, head_dim] of the tiled dout
    const void* q;               // tiled q [rows, head_dim]
    const void* dout;            // tiled dout [rows, head_dim]
    const float* lse;            // tiled lse [rows] of the forward (natural log)
    const float* delta;          // tiled <dout, out> [rows]
    void* dq;                    // tiled bf16 dq [rows, head_dim]
    int dims[3], win[3], str[3], off[3];
    int tile[3], tlog[3], nt[3];
    int tiles_per_head;
    float scale;
    int fault_skip_kv;           // test hook: >= 0 makes the producer skip that KV load
};

// Parameters of one dK / dV launch of the backward pass (bf16, head_dim 64 or
// 128, all tensors tiled).
struct BwdKVParams {
    CUtensorMap tmQ;             // 2-D TMA views [rows, head_dim] of the tiled q, dout, k and v
    CUtensorMap tmDO;
    CUtensorMap tmK;
    CUtensorMap tmV;
    const float* lse;            // tiled lse [rows] of the forward (natural log)
    const float* delta;          // tiled <dout, out> [rows]
    void* dk;                    // tiled bf16 dk [rows, head_dim]
    void* dv;                    // tiled bf16 dv [rows, head_dim]
    int dims[3], win[3], str[3], off[3];
    int tile[3], tlog[3], nt[3];
    int tiles_per_head;
    float scale;
};

// dK / dV over num_kv_tiles CTAs, dQ over num_q_tiles CTAs, and delta =
// <dout, out> over `rows` tiled rows; head_dim 32, 64 or 128 (else
// cudaErrorNotSupported).
cudaError_t launch_backward_dkdv(const BwdKVParams& p, int head_dim, int64_t num_kv_tiles, cudaStream_t stream);
cudaError_t launch_backward_dq(const BwdParams& p, int head_dim, int64_t num_q_tiles, cudaStream_t stream);
cudaError_t launch_backward_delta(const void* out, const void* dout, float* delta, int64_t rows, int head_dim,
                                  cudaStream_t stream);
// Status word of the backward kernels: read-and-clear.
cudaError_t read_and_clear_bwd_status(int* status, cudaStream_t stream);

}  // namespace gna
