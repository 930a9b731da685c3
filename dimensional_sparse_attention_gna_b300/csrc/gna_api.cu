// C ABI of libgna_b300.so (declared in include/gna.h): argument validation,
// tile planning, TMA descriptor encoding and kernel launches.  Nothing here
// allocates device memory; every call enqueues on the caller's stream.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/gna.h"
#include "gna_geometry.cuh"
#include "gna_internal.h"

namespace {

thread_local std::string t_last_error;

// Failure injection of the bounded-wait tests (gna_test_skip_kv_load): the KV
// load iteration the producer of the forward / dQ kernel skips, -1 = none.
std::atomic<int> g_skip_kv_forward{-1};
std::atomic<int> g_skip_kv_backward_dq{-1};

gna_status fail(gna_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

gna_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(GNA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int ilog2_exact(int v)
{
    if (v <= 0 || (v & (v - 1)) != 0) return -1;
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

int elem_size(gna_dtype dt)
{
    switch (dt) {
        case GNA_BF16: return 2;
        case GNA_FP8_E4M3: return 1;
        case GNA_F32: return 4;
        default: return 0;
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_ok(const int dims[3])
{
    return dims != nullptr && dims[0] >= 1 && dims[1] >= 1 && dims[2] >= 1;
}

int64_t padded_volume(const int dims[3], const int tile[3])
{
    int64_t v = 1;
    for (int d = 0; d < 3; ++d) v *= static_cast<int64_t>((dims[d] + tile[d] - 1) / tile[d]) * tile[d];
    return v;
}

void default_tile(const int dims[3], int tile[3])
{
    // least padding first; among equals the shape nearest (1, 8, 16) for
    // images (T = 1) and (2, 8, 8) for videos, in log2 distance
    const int target[3] = {dims[0] == 1 ? 0 : 1, 3, dims[0] == 1 ? 4 : 3};
    int64_t best_pad = -1;
    int best_dist = 0, best_w = 0;
    for (int lt = 0; lt <= 7; ++lt)
        for (int lh = 0; lt + lh <= 7; ++lh) {
            const int lw = 7 - lt - lh;
            const int t[3] = {1 << lt, 1 << lh, 1 << lw};
            const int64_t pad = padded_volume(dims, t);
            const int dist = std::abs(lt - target[0]) + std::abs(lh - target[1]) + std::abs(lw - target[2]);
            const bool better = best_pad < 0 || pad < best_pad ||
                                (pad == best_pad && (dist < best_dist || (dist == best_dist && t[2] > best_w)));
            if (better) {
                best_pad = pad;
                best_dist = dist;
                best_w = t[2];
                tile[0] = t[0];
                tile[1] = t[1];
                tile[2] = t[2];
            }
        }
}

gna_status check_tile(const int tile[3], int tlog[3])
{
    int log_sum = 0;          // log2 of the volume (summed, so no product can overflow)
    for (int d = 0; d < 3; ++d) {
        tlog[d] = ilog2_exact(tile[d]);
        if (tlog[d] < 0) return fail(GNA_ERR_INVALID_ARG, "tile[%d] = %d is not a positive power of two", d, tile[d]);
        log_sum += tlog[d];
    }
    static_assert(gna::kTileElems == 1 << 7, "tile volume is 2^7");
    if (log_sum != 7)
        return fail(GNA_ERR_INVALID_ARG, "tile %d x %d x %d does not hold %d elements", tile[0], tile[1], tile[2],
                    gna::kTileElems);
    return GNA_OK;
}

gna_status resolve_tile(const int dims[3], const int* tile_in, int tile[3], int tlog[3])
{
    if (tile_in == nullptr || (tile_in[0] == 0 && tile_in[1] == 0 && tile_in[2] == 0))
        default_tile(dims, tile);
    else
        for (int d = 0; d < 3; ++d) tile[d] = tile_in[d];
    return check_tile(tile, tlog);
}

gna_status check_geometry(const int dims[3], const int window[3], const int stride[3])
{
    if (!dims_ok(dims)) return fail(GNA_ERR_INVALID_ARG, "dims must be >= 1");
    if (window == nullptr || stride == nullptr) return fail(GNA_ERR_INVALID_ARG, "window / stride is NULL");
    for (int d = 0; d < 3; ++d) {
        if (!(1 <= stride[d] && stride[d] <= window[d] && window[d] <= dims[d]))
            return fail(GNA_ERR_INVALID_ARG,
                        "dimension %d: need 1 <= stride (%d) <= window (%d) <= length (%d)", d, stride[d],
                        window[d], dims[d]);
    }
    return GNA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D TMA view [rows, head_dim] of a tiled tensor, box = 128 rows x one
// swizzle span (128 B, or the whole row when it is shorter).
gna_status make_tile_map(CUtensorMap* map, const void* ptr, int64_t rows, int head_dim, int esize)
{
    auto enc = encode_fn();
    if (enc == nullptr) return fail(GNA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    const int row_bytes = head_dim * esize;
    const int span = row_bytes >= 128 ? 128 : row_bytes;
    const CUtensorMapSwizzle sw =
        span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(span / esize), static_cast<cuuint32_t>(gna::kTileElems)};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(map, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                     const_cast<void*>(ptr), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GNA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return GNA_OK;
}

// 5-D TMA view of a raster tensor [B, T, H, W, heads * head_dim] (innermost
// last), box = one swizzle span of features x (tW, tH, tT) tokens x 1 batch:
// the box lands in shared memory in tile element order (t, y, x).
gna_status make_raster_map(CUtensorMap* map, const void* ptr, int B, const int dims[3], int heads, int head_dim,
                           int esize, const int tile[3])
{
    auto enc = encode_fn();
    if (enc == nullptr) return fail(GNA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    const int row_bytes = head_dim * esize;
    const int span = row_bytes >= 128 ? 128 : row_bytes;
    const CUtensorMapSwizzle sw =
        span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    const cuuint64_t token = static_cast<cuuint64_t>(heads) * row_bytes;     // bytes per (t, y, x) position
    cuuint64_t gdim[5] = {static_cast<cuuint64_t>(heads) * head_dim, static_cast<cuuint64_t>(dims[2]),
                          static_cast<cuuint64_t>(dims[1]), static_cast<cuuint64_t>(dims[0]),
                          static_cast<cuuint64_t>(B)};
    cuuint64_t gstride[4] = {token, token * dims[2], token * dims[2] * dims[1],
                             token * dims[2] * dims[1] * dims[0]};
    cuuint32_t box[5] = {static_cast<cuuint32_t>(span / esize), static_cast<cuuint32_t>(tile[2]),
                         static_cast<cuuint32_t>(tile[1]), static_cast<cuuint32_t>(tile[0]), 1};
    cuuint32_t estride[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
                     const_cast<void*>(ptr), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GNA_ERR_CUDA, "cuTensorMapEncodeTiled (raster) failed (%d)", static_cast<int>(r));
    return GNA_OK;
}

// 2-D TMA view of a tensor in the value layout: [tiles * head_dim rows, 128
// tokens], box = head_dim rows x 128 bytes of tokens.
gna_status make_value_map(CUtensorMap* map, const void* ptr, int64_t tiles, int head_dim, int esize)
{
    auto enc = encode_fn();
    if (enc == nullptr) return fail(GNA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    cuuint64_t gdim[2] = {static_cast<cuuint64_t>(gna::kTileElems), static_cast<cuuint64_t>(tiles * head_dim)};
    cuuint64_t gstride[1] = {static_cast<cuuint64_t>(gna::kTileElems * esize)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), static_cast<cuuint32_t>(head_dim)};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = enc(map, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                     const_cast<void*>(ptr), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(GNA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return GNA_OK;
}

gna_status permute_common(const void* src, void* dst, int B, int heads, const int dims[3], const int* tile_in,
                          int head_dim, gna_dtype dtype, void* stream, bool to_tiled, bool value_layout = false)
{
    if (src == nullptr || dst == nullptr) return fail(GNA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(src) || !aligned16(dst)) return fail(GNA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (B < 1 || heads < 1 || head_dim < 1) return fail(GNA_ERR_INVALID_ARG, "B, heads and head_dim must be >= 1");
    if (!dims_ok(dims)) return fail(GNA_ERR_INVALID_ARG, "dims must be >= 1");
    const int es = elem_size(dtype);
    if (es == 0) return fail(GNA_ERR_INVALID_ARG, "unknown dtype %d", static_cast<int>(dtype));
    if ((static_cast<int64_t>(head_dim) * es) % 4 != 0)
        return fail(GNA_ERR_UNSUPPORTED, "head_dim * element size must be a multiple of 4 bytes");
    int tile[3], tlog[3];
    gna_status st = resolve_tile(dims, tile_in, tile, tlog);
    if (st != GNA_OK) return st;
    gna::PermuteGeom g{};
    g.B = B;
    g.heads = heads;
    int64_t ntiles = 1;
    for (int d = 0; d < 3; ++d) {
        g.dims[d] = dims[d];
        g.nt[d] = (dims[d] + tile[d] - 1) / tile[d];
        g.tlog[d] = tlog[d];
        ntiles *= g.nt[d];
    }
    const int64_t blocks = ntiles * B * heads;
    if (blocks > INT32_MAX || static_cast<int64_t>(head_dim) * es > (1 << 20))
        return fail(GNA_ERR_UNSUPPORTED, "tensor too large");
    g.ntiles_total = static_cast<int>(ntiles);
    g.row_bytes = head_dim * es;
    if (value_layout) {
        if (es != 1 && es != 2) return fail(GNA_ERR_UNSUPPORTED, "the value layout holds 1- or 2-byte elements");
        if (g.row_bytes < 16 || g.row_bytes > gna::kMaxValueRowBytes || (g.row_bytes & (g.row_bytes - 1)) != 0)
            return fail(GNA_ERR_UNSUPPORTED, "value layout: head_dim * element size must be a power of two "
                                             "from 16 to %d bytes", gna::kMaxValueRowBytes);
        cudaError_t e = gna::launch_permute_v(src, dst, g, es, to_tiled, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, to_tiled ? "value permute launch" : "value unpermute launch");
        t_last_error.clear();
        return GNA_OK;
    }
    cudaError_t e = gna::launch_permute(src, dst, g, to_tiled, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, to_tiled ? "permute launch" : "unpermute launch");
    t_last_error.clear();
    return GNA_OK;
}

}  // namespace

namespace gna {

gna_status api_fail(gna_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

}  // namespace gna

extern "C" {

int gna_version(void) { return GNA_VERSION; }

const char* gna_status_string(gna_status s)
{
    switch (s) {
        case GNA_OK: return "GNA_OK";
        case GNA_ERR_INVALID_ARG: return "GNA_ERR_INVALID_ARG";
        case GNA_ERR_UNSUPPORTED: return "GNA_ERR_UNSUPPORTED";
        case GNA_ERR_CUDA: return "GNA_ERR_CUDA";
        case GNA_ERR_TIMEOUT: return "GNA_ERR_TIMEOUT";
        default: return "GNA_ERR_UNKNOWN";
    }
}

const char* gna_last_error(void) { return t_last_error.c_str(); }

gna_status gna_tile_shape(const int dims[3], int tile[3])
{
    if (!dims_ok(dims) || tile == nullptr) return fail(GNA_ERR_INVALID_ARG, "dims must be >= 1");
    default_tile(dims, tile);
    return GNA_OK;
}

int64_t gna_tiled_elems(int B, int heads, const int dims[3], const int tile_in[3], int head_dim)
{
    if (B < 1 || heads < 1 || head_dim < 1 || !dims_ok(dims)) return -1;
    int tile[3], tlog[3];
    if (resolve_tile(dims, tile_in, tile, tlog) != GNA_OK) return -1;
    int64_t n = static_cast<int64_t>(B) * heads * head_dim * gna::kTileElems;
    for (int d = 0; d < 3; ++d) n *= (dims[d] + tile[d] - 1) / tile[d];
    return n;
}

size_t gna_permuted_elems(int B, int heads, const int dims[3], int head_dim)
{
    const int64_t n = gna_tiled_elems(B, heads, dims, nullptr, head_dim);
    return n < 0 ? 0 : static_cast<size_t>(n);
}

gna_status gna_permute(const void* src, void* dst, int B, int heads, const int dims[3], int head_dim,
                       gna_dtype dtype, void* stream)
{
    return permute_common(src, dst, B, heads, dims, nullptr, head_dim, dtype, stream, true);
}

gna_status gna_unpermute(const void* src, void* dst, int B, int heads, const int dims[3], int head_dim,
                         gna_dtype dtype, void* stream)
{
    return permute_common(src, dst, B, heads, dims, nullptr, head_dim, dtype, stream, false);
}

gna_status gna_permute_tiled(const void* src, void* dst, int B, int heads, const int dims[3], const int tile[3],
                             int head_dim, gna_dtype dtype, void* stream)
{
    if (tile == nullptr) return fail(GNA_ERR_INVALID_ARG, "tile is NULL");
    return permute_common(src, dst, B, heads, dims, tile, head_dim, dtype, stream, true);
}

gna_status gna_unpermute_tiled(const void* src, void* dst, int B, int heads, const int dims[3], const int tile[3],
                               int head_dim, gna_dtype dtype, void* stream)
{
    if (tile == nullptr) return fail(GNA_ERR_INVALID_ARG, "tile is NULL");
    return permute_common(src, dst, B, heads, dims, tile, head_dim, dtype, stream, false);
}

gna_status gna_permute_v(const void* src, void* dst, int B, int heads, const int dims[3], int head_dim,
                         gna_dtype dtype, void* stream)
{
    return permute_common(src, dst, B, heads, dims, nullptr, head_dim, dtype, stream, true, true);
}

gna_status gna_unpermute_v(const void* src, void* dst, int B, int heads, const int dims[3], int head_dim,
                           gna_dtype dtype, void* stream)
{
    return permute_common(src, dst, B, heads, dims, nullptr, head_dim, dtype, stream, false, true);
}

gna_status gna_permute_v_tiled(const void* src, void* dst, int B, int heads, const int dims[3], const int tile[3],
                               int head_dim, gna_dtype dtype, void* stream)
{
    if (tile == nullptr) return fail(GNA_ERR_INVALID_ARG, "tile is NULL");
    return permute_common(src, dst, B, heads, dims, tile, head_dim, dtype, stream, true, true);
}

gna_status gna_unpermute_v_tiled(const void* src, void* dst, int B, int heads, const int dims[3],
                                 const int tile[3], int head_dim, gna_dtype dtype, void* stream)
{
    if (tile == nullptr) return fail(GNA_ERR_INVALID_ARG, "tile is NULL");
    return permute_common(src, dst, B, heads, dims, tile, head_dim, dtype, stream, false, true);
}

gna_status gna_tile_stats_qkv(const int dims[3], const int window[3], const int stride[3], const int tile_q_in[3],
                              const int tile_kv_in[3], int leader_rule, int64_t* visited_kv_tiles,
                              int64_t* partial_kv_tiles, int64_t* q_tiles)
{
    gna_status st = check_geometry(dims, window, stride);
    if (st != GNA_OK) return st;
    if (leader_rule != GNA_LEADER_CENTER && leader_rule != GNA_LEADER_LITERAL)
        return fail(GNA_ERR_INVALID_ARG, "unknown leader rule %d", leader_rule);
    int tq[3], tkv[3], tlog[3];
    if ((st = resolve_tile(dims, tile_q_in, tq, tlog)) != GNA_OK) return st;
    if ((st = resolve_tile(dims, tile_kv_in, tkv, tlog)) != GNA_OK) return st;
    // The visited box of a Q tile is a product of per-dimension ranges, so
    // the totals over all Q tiles factor into per-dimension sums.
    int64_t visited = 1, full = 1, nq = 1;
    for (int d = 0; d < 3; ++d) {
        const int nt = (dims[d] + tq[d] - 1) / tq[d];
        const int off = gna::leader_offset(stride[d], leader_rule);
        int64_t sum_cnt = 0, sum_full = 0;
        for (int qt = 0; qt < nt; ++qt) {
            const gna::DimRange r = gna::dim_range(qt, tq[d], tkv[d], dims[d], window[d], stride[d], off);
            sum_cnt += r.k1 - r.k0 + 1;
            // the kernel's full-tile test: the interval form of dim_tile_full
            int flo, fhi;
            gna::dim_full_range(tkv[d], dims[d], window[d], r, flo, fhi);
            for (int kt = r.k0; kt <= r.k1; ++kt) sum_full += (kt >= flo && kt <= fhi);
        }
        visited *= sum_cnt;
        full *= sum_full;
        nq *= nt;
    }
    if (visited_kv_tiles) *visited_kv_tiles = visited;
    if (partial_kv_tiles) *partial_kv_tiles = visited - full;
    if (q_tiles) *q_tiles = nq;
    return GNA_OK;
}

gna_status gna_tile_stats(const int dims[3], const int window[3], const int stride[3], const int tile_in[3],
                          int leader_rule, int64_t* visited_kv_tiles, int64_t* partial_kv_tiles, int64_t* q_tiles)
{
    return gna_tile_stats_qkv(dims, window, stride, tile_in, tile_in, leader_rule, visited_kv_tiles,
                              partial_kv_tiles, q_tiles);
}

gna_status gna_plan_tile(const int dims[3], const int window[3], const int stride[3], int leader_rule, int tile[3],
                         double* tile_overhead, double* speedup_bound)
{
    gna_status st = check_geometry(dims, window, stride);
    if (st != GNA_OK) return st;
    if (tile == nullptr) return fail(GNA_ERR_INVALID_ARG, "tile is NULL");
    if (leader_rule != GNA_LEADER_CENTER && leader_rule != GNA_LEADER_LITERAL)
        return fail(GNA_ERR_INVALID_ARG, "unknown leader rule %d", leader_rule);
    // every 128-element power-of-two tile; fewest visited 128 x 128 tiles
    // wins, then fewest partial tiles, then the default tile of the grid
    int def[3];
    default_tile(dims, def);
    int64_t best_v = -1, best_p = 0;
    int best[3] = {def[0], def[1], def[2]};
    for (int lt = 0; lt <= 7; ++lt)
        for (int lh = 0; lt + lh <= 7; ++lh) {
            const int t[3] = {1 << lt, 1 << lh, 1 << (7 - lt - lh)};
            int64_t v = 0, pa = 0, nq = 0;
            if (gna_tile_stats(dims, window, stride, t, leader_rule, &v, &pa, &nq) != GNA_OK) continue;
            const bool is_def = t[0] == def[0] && t[1] == def[1] && t[2] == def[2];
            if (best_v < 0 || v < best_v || (v == best_v && (pa < best_p || (pa == best_p && is_def)))) {
                best_v = v;
                best_p = pa;
                best[0] = t[0];
                best[1] = t[1];
                best[2] = t[2];
            }
        }
    tile[0] = best[0];
    tile[1] = best[1];
    tile[2] = best[2];
    double useful = 1.0, tiles_q = 1.0;
    for (int d = 0; d < 3; ++d) {
        useful *= static_cast<double>(dims[d]) * window[d];
        tiles_q *= (dims[d] + best[d] - 1) / best[d];
    }
    const double tile_pairs = static_cast<double>(gna::kTileElems) * gna::kTileElems;
    if (tile_overhead) *tile_overhead = static_cast<double>(best_v) * tile_pairs / useful;
    // dense attention on the same tiling visits every KV tile from every Q tile
    if (speedup_bound) *speedup_bound = tiles_q * tiles_q / static_cast<double>(best_v);
    t_last_error.clear();
    return GNA_OK;
}

gna_status gna_plan_tiles(const int dims[3], const int window[3], const int stride[3], int leader_rule,
                          int tile_q[3], int tile_kv[3], double* tile_overhead, double* speedup_bound)
{
    gna_status st = check_geometry(dims, window, stride);
    if (st != GNA_OK) return st;
    if (tile_q == nullptr || tile_kv == nullptr) return fail(GNA_ERR_INVALID_ARG, "tile is NULL");
    if (leader_rule != GNA_LEADER_CENTER && leader_rule != GNA_LEADER_LITERAL)
        return fail(GNA_ERR_INVALID_ARG, "unknown leader rule %d", leader_rule);
    // start from the best equal pair, so that a decoupled pair is chosen only
    // when it visits strictly fewer tile pairs, or as many with fewer partial ones
    int eq[3];
    if ((st = gna_plan_tile(dims, window, stride, leader_rule, eq, nullptr, nullptr)) != GNA_OK) return st;
    int64_t best_v = 0, best_p = 0;
    if ((st = gna_tile_stats(dims, window, stride, eq, leader_rule, &best_v, &best_p, nullptr)) != GNA_OK) return st;
    int bq[3] = {eq[0], eq[1], eq[2]}, bk[3] = {eq[0], eq[1], eq[2]};
    for (int qt = 0; qt <= 7; ++qt)
        for (int qh = 0; qt + qh <= 7; ++qh)
            for (int kt = 0; kt <= 7; ++kt)
                for (int kh = 0; kt + kh <= 7; ++kh) {
                    const int tq[3] = {1 << qt, 1 << qh, 1 << (7 - qt - qh)};
                    const int tk[3] = {1 << kt, 1 << kh, 1 << (7 - kt - kh)};
                    int64_t v = 0, pa = 0;
                    if (gna_tile_stats_qkv(dims, window, stride, tq, tk, leader_rule, &v, &pa, nullptr) != GNA_OK)
                        continue;
                    if (v < best_v || (v == best_v && pa < best_p)) {
                        best_v = v;
                        best_p = pa;
                        for (int d = 0; d < 3; ++d) {
                            bq[d] = tq[d];
                            bk[d] = tk[d];
                        }
                    }
                }
    double useful = 1.0, tiles_q = 1.0, tiles_kv = 1.0;
    for (int d = 0; d < 3; ++d) {
        tile_q[d] = bq[d];
        tile_kv[d] = bk[d];
        useful *= static_cast<double>(dims[d]) * window[d];
        tiles_q *= (dims[d] + bq[d] - 1) / bq[d];
        tiles_kv *= (dims[d] + bk[d] - 1) / bk[d];
    }
    const double tile_pairs = static_cast<double>(gna::kTileElems) * gna::kTileElems;
    if (tile_overhead) *tile_overhead = static_cast<double>(best_v) * tile_pairs / useful;
    if (speedup_bound) *speedup_bound = tiles_q * tiles_kv / static_cast<double>(best_v);
    t_last_error.clear();
    return GNA_OK;
}

namespace {

// raster: 0 = tiled q, k, out, lse; 1 = raster q, k, out, lse; 2 = raster v as well
gna_status forward_impl(const void* q, const void* k, const void* v, void* out, float* lse, int B, int heads,
                        const int dims[3], const int window[3], const int stride[3], int head_dim, gna_dtype dtype,
                        const gna_options* opt, void* stream, int raster)
{
    if (q == nullptr || k == nullptr || v == nullptr || out == nullptr)
        return fail(GNA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return fail(GNA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (B < 1 || heads < 1) return fail(GNA_ERR_INVALID_ARG, "B and heads must be >= 1");
    gna_status st = check_geometry(dims, window, stride);
    if (st != GNA_OK) return st;
    const int es = (dtype == GNA_BF16) ? 2 : (dtype == GNA_FP8_E4M3) ? 1 : 0;
    if (es == 0) return fail(GNA_ERR_INVALID_ARG, "forward dtype must be GNA_BF16 or GNA_FP8_E4M3");
    if (!((es == 2 && (head_dim == 32 || head_dim == 64 || head_dim == 128)) || (es == 1 && head_dim == 128)))
        return fail(GNA_ERR_UNSUPPORTED, "head_dim %d is not supported for this dtype", head_dim);
    if (raster == 2 && !(es == 2 && head_dim == 128))
        return fail(GNA_ERR_UNSUPPORTED, "raster v: bf16 with head_dim 128 only (use gna_forward_raster with v in the "
                                         "value layout)");
    const int rule = opt ? opt->leader_rule : GNA_LEADER_CENTER;
    if (rule != GNA_LEADER_CENTER && rule != GNA_LEADER_LITERAL)
        return fail(GNA_ERR_INVALID_ARG, "unknown leader rule %d", rule);
    if (opt && !(opt->scale >= 0.0f && std::isfinite(opt->scale)))
        return fail(GNA_ERR_INVALID_ARG, "scale must be finite and >= 0");
    if (opt && opt->descale && es != 1) return fail(GNA_ERR_INVALID_ARG, "descale is only used with GNA_FP8_E4M3");
    if (es == 1 && (opt == nullptr || opt->descale == nullptr))
        return fail(GNA_ERR_INVALID_ARG, "GNA_FP8_E4M3 needs the per-tensor descales of q, k, v "
                                         "(gna_forward_fp8, or gna_options.descale)");
    if (opt && opt->descale && (reinterpret_cast<uintptr_t>(opt->descale) & 3u))
        return fail(GNA_ERR_INVALID_ARG, "descale must be 4-byte aligned");

    gna::FwdParams p{};
    int tlog[3], tlog_q[3];
    st = resolve_tile(dims, opt ? opt->tile : nullptr, p.tile_q, tlog_q);
    if (st != GNA_OK) return st;
    // key / value tile: opt->tile_kv when set, else the query tile
    const bool kv_own = opt && (opt->tile_kv[0] != 0 || opt->tile_kv[1] != 0 || opt->tile_kv[2] != 0);
    st = resolve_tile(dims, kv_own ? opt->tile_kv : p.tile_q, p.tile, tlog);
    if (st != GNA_OK) return st;
    int64_t tiles_per_head = 1, tiles_per_head_q = 1;
    for (int d = 0; d < 3; ++d) {
        p.dims[d] = dims[d];
        p.win[d] = window[d];
        p.str[d] = stride[d];
        p.off[d] = gna::leader_offset(stride[d], rule);
        p.tlog[d] = tlog[d];
        p.nt[d] = (dims[d] + p.tile[d] - 1) / p.tile[d];
        tiles_per_head *= p.nt[d];
        p.tlog_q[d] = tlog_q[d];
        p.nt_q[d] = (dims[d] + p.tile_q[d] - 1) / p.tile_q[d];
        tiles_per_head_q *= p.nt_q[d];
    }
    const int64_t num_q_tiles = tiles_per_head_q * B * heads;
    const int64_t num_kv_tiles = tiles_per_head * B * heads;
    const int64_t rows = num_q_tiles * gna::kTileElems;
    const int64_t rows_kv = num_kv_tiles * gna::kTileElems;
    if (rows > INT32_MAX || rows_kv > INT32_MAX) return fail(GNA_ERR_UNSUPPORTED, "more than 2^31 tiled rows");
    p.heads = heads;
    p.tiles_per_head = static_cast<int>(tiles_per_head);
    p.tiles_per_head_q = static_cast<int>(tiles_per_head_q);
    p.out = out;
    p.lse = lse;
    p.descale = (opt && es == 1) ? opt->descale : nullptr;
    p.scale = (opt && opt->scale > 0.0f) ? opt->scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    p.fault_skip_kv = g_skip_kv_forward.load(std::memory_order_relaxed);

    p.q = q;
    p.raster = raster;
    if (raster) {
        if (static_cast<int64_t>(B) * dims[0] > INT32_MAX || static_cast<int64_t>(heads) * head_dim > INT32_MAX)
            return fail(GNA_ERR_UNSUPPORTED, "raster tensor too large for TMA coordinates");
        if ((st = make_raster_map(&p.tmK, k, B, dims, heads, head_dim, es, p.tile)) != GNA_OK) return st;
    } else if ((st = make_tile_map(&p.tmK, k, rows_kv, head_dim, es)) != GNA_OK) {
        return st;
    }
    if (raster == 2) {
        if ((st = make_raster_map(&p.tmV, v, B, dims, heads, head_dim, es, p.tile)) != GNA_OK) return st;
    } else if ((st = make_value_map(&p.tmV, v, num_kv_tiles, head_dim, es)) != GNA_OK) {
        return st;
    }

    cudaError_t e = gna::launch_forward(p, head_dim, es, num_q_tiles, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return fail(GNA_ERR_UNSUPPORTED, "no kernel for head_dim %d", head_dim);
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    t_last_error.clear();
    return GNA_OK;
}

}  // namespace

gna_status gna_forward_ex(const void* q, const void* k, const void* v, void* out, float* lse, int B, int heads,
                          const int dims[3], const int window[3], const int stride[3], int head_dim, gna_dtype dtype,
                          const gna_options* opt, void* stream)
{
    return forward_impl(q, k, v, out, lse, B, heads, dims, window, stride, head_dim, dtype, opt, stream, 0);
}

gna_status gna_forward(const void* q, const void* k, const void* v, void* out, float* lse, int B, int heads,
                       const int dims[3], const int window[3], const int stride[3], int head_dim, gna_dtype dtype,
                       void* stream)
{
    if (dtype == GNA_FP8_E4M3)
        return fail(GNA_ERR_INVALID_ARG, "gna_forward takes GNA_BF16; e4m3 codes need their descales: "
                                         "call gna_forward_fp8");
    return forward_impl(q, k, v, out, lse, B, heads, dims, window, stride, head_dim, dtype, nullptr, stream, 0);
}

gna_status gna_forward_fp8(const void* q, const void* k, const void* v, void* out, float* lse, int B, int heads,
                           const int dims[3], const int window[3], const int stride[3], int head_dim,
                           const float* descale_qkv, void* stream)
{
    if (descale_qkv == nullptr) return fail(GNA_ERR_INVALID_ARG, "descale_qkv is NULL");
    gna_options opt{};
    opt.descale = descale_qkv;
    return forward_impl(q, k, v, out, lse, B, heads, dims, window, stride, head_dim, GNA_FP8_E4M3, &opt, stream,
                        0);
}

gna_status gna_forward_raster(const void* q, const void* k, const void* v, void* out, float* lse, int B, int heads,
                              const int dims[3], const int window[3], const int stride[3], int head_dim,
                              gna_dtype dtype, const gna_options* opt, void* stream)
{
    return forward_impl(q, k, v, out, lse, B, heads, dims, window, stride, head_dim, dtype, opt, stream, 1);
}

gna_status gna_forward_raster_all(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                                  int heads, const int dims[3], const int window[3], const int stride[3],
                                  int head_dim, gna_dtype dtype, const gna_options* opt, void* stream)
{
    return forward_impl(q, k, v, out, lse, B, heads, dims, window, stride, head_dim, dtype, opt, stream, 2);
}

gna_status gna_schedule_step(int step, int num_steps, int full_steps, const int dims[3], const int window[3],
                             const int stride[3], int out_window[3], int out_stride[3])
{
    if (out_window == nullptr || out_stride == nullptr) return fail(GNA_ERR_INVALID_ARG, "output is NULL");
    if (!(0 <= step && step < num_steps)) return fail(GNA_ERR_INVALID_ARG, "need 0 <= step < num_steps");
    if (!(0 <= full_steps && full_steps <= num_steps))
        return fail(GNA_ERR_INVALID_ARG, "need 0 <= full_steps <= num_steps");
    gna_status st = check_geometry(dims, window, stride);
    if (st != GNA_OK) return st;
    const bool full = step < full_steps;
    for (int d = 0; d < 3; ++d) {
        out_window[d] = full ? dims[d] : window[d];
        out_stride[d] = full ? 1 : stride[d];
    }
    t_last_error.clear();
    return GNA_OK;
}

gna_status gna_test_skip_kv_load(int kernel, int kv_index)
{
    const int v = kv_index < 0 ? -1 : kv_index;
    if (kernel == 0) g_skip_kv_forward.store(v, std::memory_order_relaxed);
    else if (kernel == 1) g_skip_kv_backward_dq.store(v, std::memory_order_relaxed);
    else return fail(GNA_ERR_INVALID_ARG, "unknown kernel %d (0 = forward, 1 = dQ backward)", kernel);
    t_last_error.clear();
    return GNA_OK;
}

gna_status gna_get_status(void* stream)
{
    int status = 0, bwd_status = 0;
    cudaError_t e = gna::read_and_clear_status(&status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    e = gna::read_and_clear_bwd_status(&bwd_status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (status == 0) status = bwd_status;
    if (status != 0) return fail(static_cast<gna_status>(status), "a kernel abandoned a pipeline wait");
    return GNA_OK;
}

namespace {

// Shared checks of the backward entry points: geometry, dtype, head_dim,
// options; fills the tile and the tiled row count.
gna_status backward_common(int B, int heads, const int dims[3], const int window[3], const int stride[3],
                           int head_dim, gna_dtype dtype, const gna_options* opt, int tile[3], int tlog[3],
                           int64_t* num_q_tiles)
{
    if (B < 1 || heads < 1) return fail(GNA_ERR_INVALID_ARG, "B and heads must be >= 1");
    gna_status st = check_geometry(dims, window, stride);
    if (st != GNA_OK) return st;
    if (dtype != GNA_BF16 || (head_dim != 32 && head_dim != 64 && head_dim != 128))
        return fail(GNA_ERR_UNSUPPORTED, "the backward pass supports bf16 with head_dim 32, 64 or 128");
    const int rule = opt ? opt->leader_rule : GNA_LEADER_CENTER;
    if (rule != GNA_LEADER_CENTER && rule != GNA_LEADER_LITERAL)
        return fail(GNA_ERR_INVALID_ARG, "unknown leader rule %d", rule);
    if (opt && !(opt->scale >= 0.0f && std::isfinite(opt->scale)))
        return fail(GNA_ERR_INVALID_ARG, "scale must be finite and >= 0");
    if (opt && opt->descale) return fail(GNA_ERR_INVALID_ARG, "descale is only used with GNA_FP8_E4M3");
    st = resolve_tile(dims, opt ? opt->tile : nullptr, tile, tlog);
    if (st != GNA_OK) return st;
    if (opt && (opt->tile_kv[0] != 0 || opt->tile_kv[1] != 0 || opt->tile_kv[2] != 0) &&
        (opt->tile_kv[0] != tile[0] || opt->tile_kv[1] != tile[1] || opt->tile_kv[2] != tile[2]))
        return fail(GNA_ERR_UNSUPPORTED, "the backward pass needs the key/value tile equal to the query tile");
    int64_t n = static_cast<int64_t>(B) * heads;
    for (int d = 0; d < 3; ++d) n *= (dims[d] + tile[d] - 1) / tile[d];
    if (n * gna::kTileElems > INT32_MAX) return fail(GNA_ERR_UNSUPPORTED, "more than 2^31 tiled rows");
    *num_q_tiles = n;
    return GNA_OK;
}

}  // namespace

gna_status gna_backward_delta(const void* out, const void* dout, float* delta, int B, int heads, const int dims[3],
                              int head_dim, gna_dtype dtype, const gna_options* opt, void* stream)
{
    if (out == nullptr || dout == nullptr || delta == nullptr) return fail(GNA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(out) || !aligned16(dout) || !aligned16(delta))
        return fail(GNA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (!dims_ok(dims)) return fail(GNA_ERR_INVALID_ARG, "dims must be >= 1");
    int tile[3], tlog[3];
    int64_t nq = 0;
    gna_status st = backward_common(B, heads, dims, dims, dims, head_dim, dtype, opt, tile, tlog, &nq);
    if (st != GNA_OK) return st;
    cudaError_t e = gna::launch_backward_delta(out, dout, delta, nq * gna::kTileElems, head_dim,
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "backward delta launch");
    t_last_error.clear();
    return GNA_OK;
}

gna_status gna_backward_dkdv(const void* q, const void* k, const void* v, const void* dout, const float* lse,
                             const float* delta, void* dk, void* dv, int B, int heads, const int dims[3],
                             const int window[3], const int stride[3], int head_dim, gna_dtype dtype,
                             const gna_options* opt, void* stream)
{
    if (!q || !k || !v || !dout || !lse || !delta || !dk || !dv) return fail(GNA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(lse) || !aligned16(delta) ||
        !aligned16(dk) || !aligned16(dv))
        return fail(GNA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    int tile[3], tlog[3];
    int64_t nt_all = 0;
    gna_status st = backward_common(B, heads, dims, window, stride, head_dim, dtype, opt, tile, tlog, &nt_all);
    if (st != GNA_OK) return st;
    const int rule = opt ? opt->leader_rule : GNA_LEADER_CENTER;
    gna::BwdKVParams p{};
    int64_t tiles_per_head = 1;
    for (int d = 0; d < 3; ++d) {
        p.dims[d] = dims[d];
        p.win[d] = window[d];
        p.str[d] = stride[d];
        p.off[d] = gna::leader_offset(stride[d], rule);
        p.tile[d] = tile[d];
        p.tlog[d] = tlog[d];
        p.nt[d] = (dims[d] + tile[d] - 1) / tile[d];
        tiles_per_head *= p.nt[d];
    }
    p.tiles_per_head = static_cast<int>(tiles_per_head);
    p.scale = (opt && opt->scale > 0.0f) ? opt->scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    p.lse = lse;
    p.delta = delta;
    p.dk = dk;
    p.dv = dv;
    const int64_t rows = nt_all * gna::kTileElems;
    if ((st = make_tile_map(&p.tmQ, q, rows, head_dim, 2)) != GNA_OK) return st;
    if ((st = make_tile_map(&p.tmDO, dout, rows, head_dim, 2)) != GNA_OK) return st;
    if ((st = make_tile_map(&p.tmK, k, rows, head_dim, 2)) != GNA_OK) return st;
    if ((st = make_tile_map(&p.tmV, v, rows, head_dim, 2)) != GNA_OK) return st;
    cudaError_t e = gna::launch_backward_dkdv(p, head_dim, nt_all, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "backward dk/dv launch");
    t_last_error.clear();
    return GNA_OK;
}

gna_status gna_backward_dq(const void* q, const void* k, const void* k_value, const void* v, const void* dout,
                           const float* lse, const float* delta, void* dq, int B, int heads, const int dims[3],
                           const int window[3], const int stride[3], int head_dim, gna_dtype dtype,
                           const gna_options* opt, void* stream)
{
    if (!q || !k || !k_value || !v || !dout || !lse || !delta || !dq)
        return fail(GNA_ERR_INVALID_ARG, "NULL tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(k_value) || !aligned16(v) || !aligned16(dout) ||
        !aligned16(lse) || !aligned16(delta) || !aligned16(dq))
        return fail(GNA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    int tile[3], tlog[3];
    int64_t nq = 0;
    gna_status st = backward_common(B, heads, dims, window, stride, head_dim, dtype, opt, tile, tlog, &nq);
    if (st != GNA_OK) return st;
    const int rule = opt ? opt->leader_rule : GNA_LEADER_CENTER;
    gna::BwdParams p{};
    int64_t tiles_per_head = 1;
    for (int d = 0; d < 3; ++d) {
        p.dims[d] = dims[d];
        p.win[d] = window[d];
        p.str[d] = stride[d];
        p.off[d] = gna::leader_offset(stride[d], rule);
        p.tile[d] = tile[d];
        p.tlog[d] = tlog[d];
        p.nt[d] = (dims[d] + tile[d] - 1) / tile[d];
        tiles_per_head *= p.nt[d];
    }
    p.tiles_per_head = static_cast<int>(tiles_per_head);
    p.scale = (opt && opt->scale > 0.0f) ? opt->scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    p.q = q;
    p.dout = dout;
    p.lse = lse;
    p.delta = delta;
    p.dq = dq;
    p.fault_skip_kv = g_skip_kv_backward_dq.load(std::memory_order_relaxed);
    const int64_t rows = nq * gna::kTileElems;
    if ((st = make_tile_map(&p.tmK, k, rows, head_dim, 2)) != GNA_OK) return st;
    if ((st = make_tile_map(&p.tmV, v, rows, head_dim, 2)) != GNA_OK) return st;
    if ((st = make_value_map(&p.tmKv, k_value, nq, head_dim, 2)) != GNA_OK) return st;
    if ((st = make_tile_map(&p.tmDO, dout, rows, head_dim, 2)) != GNA_OK) return st;
    cudaError_t e = gna::launch_backward_dq(p, head_dim, nq, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "backward dq launch");
    t_last_error.clear();
    return GNA_OK;
}

}  // extern "C"
