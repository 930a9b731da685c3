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
//
// The value layout [B, heads, nT, nH, nW, d, tT*tH*tW] stores each tile
// feature-major (its d x 128 transpose), so that the attention kernel's P V
// product reads V with the token index contiguous, the operand order the
// tensor core consumes fastest.  permute_v_kernel stages one tile in shared
// memory and transposes it in registers with byte permutes.
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

// Raster byte offset of every element of tile `tile_global` ((b*heads + h)*ntiles
// + tile), or -1 for padding, into row_off[0..127].  Ends with __syncthreads().
__device__ __forceinline__ void tile_row_offsets(const PermuteGeom& g, int64_t tile_global, int64_t* row_off)
{
    const int tile_id = static_cast<int>(tile_global % g.ntiles_total);
    const int64_t bh = tile_global / g.ntiles_total;
    const int h = static_cast<int>(bh % g.heads);
    const int64_t b = bh / g.heads;
    const int tx = tile_id % g.nt[2];
    const int ty = (tile_id / g.nt[2]) % g.nt[1];
    const int tt = tile_id / (g.nt[2] * g.nt[1]);

    for (int e = threadIdx.x; e < kTileElems; e += blockDim.x) {
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
}

template <int VEC, bool TO_TILED>
__global__ void __launch_bounds__(kPermThreads)
permute_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, PermuteGeom g)
{
    using V = typename VecT<VEC>::type;
    __shared__ int64_t row_off[kTileElems];

    const int64_t tile_global = blockIdx.x;                   // (b*heads + h)*ntiles + tile
    tile_row_offsets(g, tile_global, row_off);

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

// Raster <-> value layout for elements of E bytes (E = 1 or 2; rows of a
// power of two from 16 to 256 bytes).  A block moves one half tile (64 tokens):
// shared memory holds it token-major, [64 tokens][W words] (W = d*E/4), with
// the 16-byte groups XOR-swizzled by token group (vsm_word).  On the
// transposed side a thread owns word column c (features 4/E*c ..) of a group
// of 16 tokens: 16*E contiguous bytes of each of its 4/E feature rows.  Four
// consecutive lanes take the four token groups of one column, so a warp writes
// (or reads) 64*E contiguous bytes of each feature row it touches, and the
// swizzle keeps its shared-memory accesses on distinct banks.
template <int E>
__device__ __forceinline__ void words_to_feature_rows(const uint32_t (&w)[16], uint4 (&rows)[4 / E][E])
{
    if constexpr (E == 2) {
        uint32_t lo[8], hi[8];                       // feature 2c / 2c+1 of tokens 2i, 2i+1
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            lo[i] = __byte_perm(w[2 * i], w[2 * i + 1], 0x5410);
            hi[i] = __byte_perm(w[2 * i], w[2 * i + 1], 0x7632);
        }
        rows[0][0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        rows[0][1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        rows[1][0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        rows[1][1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    } else {
        uint32_t r[4][4];                            // [feature byte][group of 4 tokens]
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            // 4 x 4 byte transpose of words w[4q..4q+3]
            const uint32_t a = __byte_perm(w[4 * q], w[4 * q + 1], 0x5140);
            const uint32_t b = __byte_perm(w[4 * q + 2], w[4 * q + 3], 0x5140);
            const uint32_t c = __byte_perm(w[4 * q], w[4 * q + 1], 0x7362);
            const uint32_t d = __byte_perm(w[4 * q + 2], w[4 * q + 3], 0x7362);
            r[0][q] = __byte_perm(a, b, 0x5410);
            r[1][q] = __byte_perm(a, b, 0x7632);
            r[2][q] = __byte_perm(c, d, 0x5410);
            r[3][q] = __byte_perm(c, d, 0x7632);
        }
#pragma unroll
        for (int f = 0; f < 4; ++f) rows[f][0] = make_uint4(r[f][0], r[f][1], r[f][2], r[f][3]);
    }
}

// Inverse of words_to_feature_rows (both byte networks are involutions up to
// the grouping of their inputs).
template <int E>
__device__ __forceinline__ void feature_rows_to_words(const uint4 (&rows)[4 / E][E], uint32_t (&w)[16])
{
    if constexpr (E == 2) {
        const uint32_t lo[8] = {rows[0][0].x, rows[0][0].y, rows[0][0].z, rows[0][0].w,
                                rows[0][1].x, rows[0][1].y, rows[0][1].z, rows[0][1].w};
        const uint32_t hi[8] = {rows[1][0].x, rows[1][0].y, rows[1][0].z, rows[1][0].w,
                                rows[1][1].x, rows[1][1].y, rows[1][1].z, rows[1][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w[2 * i] = __byte_perm(lo[i], hi[i], 0x5410);
            w[2 * i + 1] = __byte_perm(lo[i], hi[i], 0x7632);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t r0 = (&rows[0][0].x)[q], r1 = (&rows[1][0].x)[q];
            const uint32_t r2 = (&rows[2][0].x)[q], r3 = (&rows[3][0].x)[q];
            const uint32_t a = __byte_perm(r0, r1, 0x5140);
            const uint32_t b = __byte_perm(r2, r3, 0x5140);
            const uint32_t c = __byte_perm(r0, r1, 0x7362);
            const uint32_t d = __byte_perm(r2, r3, 0x7362);
            w[4 * q] = __byte_perm(a, b, 0x5410);
            w[4 * q + 1] = __byte_perm(a, b, 0x7632);
            w[4 * q + 2] = __byte_perm(c, d, 0x5410);
            w[4 * q + 3] = __byte_perm(c, d, 0x7632);
        }
    }
}

// Word (token r of the half tile, column c) in shared memory: rows of W words;
// 16-byte group g of token r sits at group g ^ 2 * (r / 16) (mod W / 4).
__device__ __forceinline__ int vsm_word(int r, int c, int W)
{
    const int groups = W >> 2;
    return r * W + ((((c >> 2) ^ ((r >> 4) << 1)) & (groups - 1)) << 2) + (c & 3);
}

constexpr int kVThreads = 128;          // one block moves half a tile: 64 tokens
constexpr int kVTokens = kTileElems / 2;

template <int E, bool TO_TILED>
__global__ void __launch_bounds__(kVThreads)
permute_v_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, PermuteGeom g)
{
    constexpr int F = 4 / E;                                  // features per 32-bit word
    extern __shared__ __align__(16) uint32_t vsm[];
    __shared__ int64_t row_off[kTileElems];

    const int64_t tile_global = blockIdx.x >> 1;
    const int hh = blockIdx.x & 1;                            // which 64 tokens of the tile
    tile_row_offsets(g, tile_global, row_off);

    const int W = g.row_bytes / 4;                            // words per token row (a power of two, >= 4)
    const int vpr = g.row_bytes / 16;                         // 16-byte vectors per token row
    const int64_t tile_base = tile_global * kTileElems * static_cast<int64_t>(g.row_bytes);
    const int frow = kTileElems * E;                          // bytes of one feature row
    // work item i of the transposed side: (column group, token group, column in group);
    // four token groups of 16 per half tile
    auto item = [&](int i, int& c, int& grp) {
        grp = (i >> 2) & 3;
        c = ((i >> 4) << 2) + (i & 3);
    };
    const int nvec = kVTokens * vpr;
    const int nitem = W * 4;

    // at most 64 rows x 16 vectors = 8 vectors per thread; all loads of a
    // thread are issued before the first shared-memory store
    constexpr int kVecPerThread = kVTokens * (kMaxValueRowBytes / 16) / kVThreads;
    if (TO_TILED) {
        uint4 val[kVecPerThread];
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int i = threadIdx.x + u * kVThreads;
            val[u] = make_uint4(0, 0, 0, 0);
            if (i < nvec) {
                const int r = i / vpr, v = i - r * vpr;
                const int64_t o = row_off[hh * kVTokens + r];
                if (o >= 0) val[u] = __ldcs(reinterpret_cast<const uint4*>(src + o + v * 16));
            }
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int i = threadIdx.x + u * kVThreads;
            if (i < nvec) {
                const int r = i / vpr, v = i - r * vpr;
                *reinterpret_cast<uint4*>(vsm + vsm_word(r, 4 * v, W)) = val[u];
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nitem; i += kVThreads) {
            int c, grp;
            item(i, c, grp);
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = vsm[vsm_word(grp * 16 + k, c, W)];
            uint4 rows[F][E];
            words_to_feature_rows<E>(w, rows);
            const int tok0 = hh * kVTokens + grp * 16;
#pragma unroll
            for (int f = 0; f < F; ++f) {
                uint4* o = reinterpret_cast<uint4*>(dst + tile_base + static_cast<int64_t>(c * F + f) * frow + tok0 * E);
#pragma unroll
                for (int e = 0; e < E; ++e) __stcs(o + e, rows[f][e]);
            }
        }
    } else {
        for (int i = threadIdx.x; i < nitem; i += kVThreads) {
            int c, grp;
            item(i, c, grp);
            uint4 rows[F][E];
            const int tok0 = hh * kVTokens + grp * 16;
#pragma unroll
            for (int f = 0; f < F; ++f) {
                const uint4* o =
                    reinterpret_cast<const uint4*>(src + tile_base + static_cast<int64_t>(c * F + f) * frow + tok0 * E);
#pragma unroll
                for (int e = 0; e < E; ++e) rows[f][e] = o[e];
            }
            uint32_t w[16];
            feature_rows_to_words<E>(rows, w);
#pragma unroll
            for (int k = 0; k < 16; ++k) vsm[vsm_word(grp * 16 + k, c, W)] = w[k];
        }
        __syncthreads();
        uint4 val[kVecPerThread];
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int i = threadIdx.x + u * kVThreads;
            if (i < nvec) {
                const int r = i / vpr, v = i - r * vpr;
                val[u] = *reinterpret_cast<const uint4*>(vsm + vsm_word(r, 4 * v, W));
            }
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
            const int i = threadIdx.x + u * kVThreads;
            if (i < nvec) {
                const int r = i / vpr, v = i - r * vpr;
                const int64_t o = row_off[hh * kVTokens + r];
                if (o >= 0) *reinterpret_cast<uint4*>(dst + o + v * 16) = val[u];
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

cudaError_t launch_permute_v(const void* src, void* dst, const PermuteGeom& g, int elem_size, bool to_tiled,
                             cudaStream_t stream)
{
    const int64_t nblocks = g.B * static_cast<int64_t>(g.heads) * g.ntiles_total;
    if (nblocks <= 0) return cudaSuccess;
    if (g.row_bytes < 16 || g.row_bytes > kMaxValueRowBytes || (g.row_bytes & (g.row_bytes - 1)) != 0 ||
        (elem_size != 1 && elem_size != 2))
        return cudaErrorNotSupported;
    const size_t smem = static_cast<size_t>(kVTokens) * (g.row_bytes / 4) * sizeof(uint32_t);
    if (2 * nblocks > INT32_MAX) return cudaErrorNotSupported;
    dim3 grid(static_cast<unsigned>(2 * nblocks));
    const auto* s = static_cast<const uint8_t*>(src);
    auto* d = static_cast<uint8_t*>(dst);
    if (elem_size == 2) {
        if (to_tiled) permute_v_kernel<2, true><<<grid, kVThreads, smem, stream>>>(s, d, g);
        else permute_v_kernel<2, false><<<grid, kVThreads, smem, stream>>>(s, d, g);
    } else {
        if (to_tiled) permute_v_kernel<1, true><<<grid, kVThreads, smem, stream>>>(s, d, g);
        else permute_v_kernel<1, false><<<grid, kVThreads, smem, stream>>>(s, d, g);
    }
    return cudaGetLastError();
}

}  // namespace gna
