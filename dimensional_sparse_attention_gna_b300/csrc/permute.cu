// Token permutation between the raster layout [B, T, H, W, heads, d] and the
// tile-major layout [B, heads, nT, nH, nW, tT*tH*tW, d] the attention kernel
// reads with TMA.
//
// GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践"), §2.2: tokens
// are permuted before attention and back after it; a generic
// permute().contiguous() reaches a small fraction of memory bandwidth, and a
// dedicated copy kernel that fuses the permutation with the padding is the
// planned fix.  This is that kernel: a pure HBM copy, every byte read once and
// written once.
//
// One CTA moves one tile (128 token rows of one head).  Row r of the tile is a
// contiguous run of d * elem_size bytes on both sides (on the raster side it
// sits at stride heads * d * elem_size from its neighbours), so the copy is a
// stream of 16-byte vectors: consecutive threads take consecutive vectors of
// the tile, which makes the tile side fully coalesced and the raster side a
// sequence of whole rows.  The raster offset of each row is computed once per
// CTA into shared memory (-1 for padding rows, which read as zero and are
// skipped on the way back).
#include <cstdint>
#include <cuda_runtime.h>

#include "gna_geometry.cuh"
#include "gna_internal.h"

namespace gna {

namespace {

constexpr int kPermThreads = 256;

template <int VEC>
struct VecT;
template <> struct VecT<16> { using type = uint4; };
template <> struct VecT<8> { using type = uint2; };
template <> struct VecT<4> { using type = uint32_t; };

template <int VEC, bool TO_TILED>
__global__ void __launch_bounds__(kPermThreads)
permute_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, PermuteGeom g)
{
    using V = typename VecT<VEC>::type;
    __shared__ int64_t row_off[kTileElems];

    const int64_t tile_global = blockIdx.x;                   // (b*heads + h)*ntiles + tile
    const int tile_id = static_cast<int>(tile_global % g.ntiles_total);
    const int64_t bh = tile_global / g.ntiles_total;
    const int h = static_cast<int>(bh % g.heads);
    const int64_t b = bh / g.heads;
    const int tx = tile_id % g.nt[2];
    const int ty = (tile_id / g.nt[2]) % g.nt[1];
    const int tt = tile_id / (g.nt[2] * g.nt[1]);

    for (int e = threadIdx.x; e < kTileElems; e += kPermThreads) {
        const int ix = e & ((1 << g.tlog[2]) - 1);
        const int iy = (e >> g.tlog[2]) & ((1 << g.tlog[1]) - 1);
        const int it = e >> (g.tlog[1] + g.tlog[2]);
        const int t = tt * (1 << g.tlog[0]) + it;
        const int y = ty * (1 << g.tlog[1]) + iy;
        const int x = tx * (1 << g.tlog[2]) + ix;
        int64_t off = -1;
        if (t < g.dims[0] && y < g.dims[1] && x < g.dims[2])
            off = ((((b * g.dims[0] + t) * g.dims[1] + y) * g.dims[2] + x) * g.heads + h) * g.row_bytes;
        row_off[e] = off;
    }
    __syncthreads();

    const int vpr = g.row_bytes / VEC;                        // vectors per row
    const int nvec = kTileElems * vpr;
    const int64_t tile_base = tile_global * kTileElems * static_cast<int64_t>(g.row_bytes);
    constexpr int U = 4;
    for (int base = threadIdx.x; base < nvec; base += kPermThreads * U) {
        V val[U];
        int64_t raster[U];
        int idx[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            idx[u] = base + u * kPermThreads;
            raster[u] = -1;
            if (idx[u] < nvec) {
                const int r = idx[u] / vpr;
                const int v = idx[u] - r * vpr;
                const int64_t o = row_off[r];
                raster[u] = o < 0 ? -1 : o + static_cast<int64_t>(v) * VEC;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (idx[u] >= nvec) continue;
            if (TO_TILED) {
                if (raster[u] >= 0) val[u] = *reinterpret_cast<const V*>(src + raster[u]);
                else val[u] = V{};
            } else {
                val[u] = *reinterpret_cast<const V*>(src + tile_base + static_cast<int64_t>(idx[u]) * VEC);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (idx[u] >= nvec) continue;
            if (TO_TILED) {
                *reinterpret_cast<V*>(dst + tile_base + static_cast<int64_t>(idx[u]) * VEC) = val[u];
            } else if (raster[u] >= 0) {
                *reinterpret_cast<V*>(dst + raster[u]) = val[u];
            }
        }
    }
}

template <bool TO_TILED>
cudaError_t launch(const void* src, void* dst, const PermuteGeom& g, cudaStream_t stream)
{
    const int64_t nblocks = g.B * static_cast<int64_t>(g.heads) * g.ntiles_total;
    if (nblocks <= 0) return cudaSuccess;
    dim3 grid(static_cast<unsigned>(nblocks));
    const auto* s = static_cast<const uint8_t*>(src);
    auto* d = static_cast<uint8_t*>(dst);
    if (g.row_bytes % 16 == 0)
        permute_kernel<16, TO_TILED><<<grid, kPermThreads, 0, stream>>>(s, d, g);
    else if (g.row_bytes % 8 == 0)
        permute_kernel<8, TO_TILED><<<grid, kPermThreads, 0, stream>>>(s, d, g);
    else
        permute_kernel<4, TO_TILED><<<grid, kPermThreads, 0, stream>>>(s, d, g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_permute(const void* src, void* dst, const PermuteGeom& g, bool to_tiled, cudaStream_t stream)
{
    return to_tiled ? launch<true>(src, dst, g, stream) : launch<false>(src, dst, g, stream);
}

}  // namespace gna
