// Window geometry of Generalized Neighborhood Attention, shared by the host
// launcher and the device kernels of this library.
//
// GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践"), §1.1: a stride
// moves each query's window from the sliding window (stride 1) to blocked
// attention (stride = window); queries of one stride group share the window of
// the group's leader.  Per dimension of length L, window w, stride s and leader
// offset off:
//     leader(i) = min(floor(i / s) * s + off, L - 1)
//     start(i)  = clamp(leader(i) - floor(w / 2), 0, L - w)
// Query i sees keys [start(i), start(i) + w) in every dimension.
//
// Because start() is non-decreasing in i, a box of queries [lo, hi] sees the
// key range [start(lo), start(hi) + w - 1]; a KV tile lies inside every one of
// those windows iff it starts at or after start(hi) and ends at or before
// start(lo) + w - 1.  These two facts give the per-Q-tile KV-tile range (§1.1)
// and the "mask only partial tiles" test (§2.1).
#pragma once

#include <cstdint>

namespace gna {

constexpr int kTileElems = 128;   // tokens per layout tile (one MMA M / N extent)

__host__ __device__ __forceinline__ int window_start(int i, int L, int w, int s, int off)
{
    int c = (i / s) * s + off;
    c = c < L - 1 ? c : L - 1;
    int a = c - w / 2;
    a = a > 0 ? a : 0;
    return a < L - w ? a : L - w;
}

__host__ __device__ __forceinline__ int leader_offset(int s, int rule)
{
    return rule == 0 ? s / 2 : (s - 1) / 2;
}

// Range of KV tiles (inclusive) and the window-start extremes of the query
// tile `qt` along one dimension.  Query tiles have extent tq, KV tiles extent
// tkv (equal unless the two tilings are chosen separately, GNA page §1.2).
struct DimRange {
    int k0, k1;        // first / last KV tile index visited
    int smin, smax;    // window start of the first / last valid query
};

__host__ __device__ __forceinline__ DimRange dim_range(int qt, int tq, int tkv, int L, int w, int s, int off)
{
    int lo = qt * tq;
    int hi = lo + tq - 1;
    hi = hi < L - 1 ? hi : L - 1;
    DimRange r;
    r.smin = window_start(lo, L, w, s, off);
    r.smax = window_start(hi, L, w, s, off);
    r.k0 = r.smin / tkv;
    r.k1 = (r.smax + w - 1) / tkv;
    return r;
}

// True iff KV tile `kt` along this dimension needs no element mask for any
// valid query of the Q tile: it lies inside every query's window and holds no
// padding.
__host__ __device__ __forceinline__ bool dim_tile_full(int kt, int t, int L, int w, const DimRange& r)
{
    int lo = kt * t;
    int hi = lo + t - 1;
    return lo >= r.smax && hi <= r.smin + w - 1 && hi < L;
}

// The KV tiles along this dimension for which dim_tile_full holds form one
// interval [lo, hi] (empty when hi < lo): tile kt is full iff
// kt * t >= r.smax and kt * t + t <= min(r.smin + w, L).
__host__ __device__ __forceinline__ void dim_full_range(int t, int L, int w, const DimRange& r, int& lo, int& hi)
{
    lo = (r.smax + t - 1) / t;
    const int end = (r.smin + w < L ? r.smin + w : L) - t;     // last allowed tile start
    hi = end >= 0 ? end / t : -1;
}

// Bit c of the result is set iff element 32 * wi + c of a tile lies inside a
// box: the tile has 2^tl[d] elements per dimension, stored in (t, y, x) order,
// and the box holds the element coordinates with 0 <= c_d - lo_d < len_d in
// every dimension (len_d <= 0: empty).  One word covers 32 consecutive
// elements, i.e. one or more whole x rows of the tile, or part of one.
__host__ __device__ __forceinline__ uint32_t box_mask_word(int wi, int tl_t, int tl_y, int tl_x, int lo_t, int lo_y,
                                                           int lo_x, int len_t, int len_y, int len_x)
{
    auto in = [](int c, int lo, int len) { return static_cast<unsigned>(c - lo) < static_cast<unsigned>(len); };
    auto bits = [](int a, int b) -> uint32_t {   // bits [a, b) clipped to [0, 32)
        a = a < 0 ? 0 : a;
        b = b > 32 ? 32 : b;
        if (b <= a) return 0u;
        return ((b - a) >= 32 ? 0xffffffffu : ((1u << (b - a)) - 1u)) << a;
    };
    if (len_t <= 0 || len_y <= 0 || len_x <= 0) return 0u;
    const int tw = 1 << tl_x;
    if (tl_x >= 5) {
        // the word is part of one x row: group (t, y) of element 32 wi
        const int e0 = wi * 32;
        const int g = e0 >> tl_x;
        const int cy = g & ((1 << tl_y) - 1), ct = g >> tl_y;
        if (!in(ct, lo_t, len_t) || !in(cy, lo_y, len_y)) return 0u;
        const int bx = e0 & (tw - 1);
        return bits(lo_x - bx, lo_x - bx + len_x);
    }
    const uint32_t xrow = bits(lo_x, lo_x + len_x) & ((1u << tw) - 1u);
    uint32_t w = 0u;
    for (int gi = 0; gi < (32 >> tl_x); ++gi) {
        const int g = ((wi * 32) >> tl_x) + gi;
        const int cy = g & ((1 << tl_y) - 1), ct = g >> tl_y;
        if (in(ct, lo_t, len_t) && in(cy, lo_y, len_y)) w |= xrow << (gi * tw);
    }
    return w;
}

}  // namespace gna
