// Fused Generalized Neighborhood Attention forward kernel for sm_103a.
//
// GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践"):
//  §1.1  Q and KV are cut into fixed-size multi-dimensional tiles; the stride
//        decides which KV tiles each Q tile must visit; a producer warp maps
//        the loop index to multi-dimensional KV tile coordinates and loads the
//        tiles with TMA.
//  §2.1  the element mask is applied only to KV tiles that are not entirely
//        inside the attention window; loads overlap compute.
// Video tutorial page ("视频生成推理提速:稀疏注意力组合配置教程"), §3.3: the
// softmax is accumulated block by block and the n x n matrix never exists.
//
// One CTA owns one 128-query tile of one (batch, head) and walks the box of
// KV tiles its windows touch.  Query tiles (q, out, lse) and key/value tiles
// (k, v) are both 128-token boxes of the grid, of the same shape or, as the GNA
// page's §1.2 allows, of two different shapes; the KV box, the element mask and
// the K / V loads use the KV tile, the query rows the query tile.  Warp roles
// (320 threads):
//   warp 0      TMA producer: K and V tiles through NS-stage mbarrier rings
//   warp 1      TMEM allocator and tcgen05.mma issuer (lane 0)
//   warps 2..9  softmax / correction / epilogue.  Thread = (query row, half):
//               warps 2..5 own score columns [0, 64) of their 32 rows, warps
//               6..9 columns [64, 128) (TMEM lane quarter = warp % 4).  The two
//               halves of a row swap their partial maxima through shared
//               memory once per tile; row sums stay partial until the end.
// TMEM (512 columns): O [0, 128), S double buffer [128, 256) and [256, 384),
// Q [384, 384 + head_dim * elem / 4), and for e4m3 a P double buffer [448,
// 512).  Q sits in TMEM so S = Q K^T reads only K from shared memory; P feeds
// O += P V straight from TMEM.  bf16 P (64 columns) has no room of its own
// and overwrites the front of its S buffer, so QK(j + 2) writes columns that
// PV(j), an MMA on another accumulator issued just before it, reads: the
// kernel relies on the tensor core executing MMAs in issue order.  e4m3 P
// (32 columns) sits in buffers of its own and needs no such ordering: P(j)
// is written after S(j) arrived, so PV(j - 2), the last reader of its buffer,
// is complete.  V comes in the value layout (each tile feature-major), so both
// MMAs read their shared-memory operand K-major.
// MMA issue order  QK(0) QK(1) PV(0) QK(2) PV(1) ...  keeps the tensor core on
// the next S while the softmax warps work on the current one.
//
// The running row maximum is updated lazily: O is rescaled only when the
// maximum grows by more than `tau` (log2 units); in between P may exceed 1 by
// up to 2^tau, which the final O / l cancels exactly.  For e4m3 P the exponent
// is shifted by `p_shift` so that P uses the normal range of e4m3 (at most
// 2^(p_shift + tau) <= 448).
//
// Every mbarrier wait is bounded (see ptx.cuh); a role that gives up raises
// the CTA abort flag and the device status word, the other roles drop out of
// their loops, in-flight TMA loads and MMAs are drained (again bounded), TMEM
// is freed and the CTA exits.  The waits of every other CTA of the launch also
// give up as soon as they see the status word set, so a stuck launch ends after
// one wait bound instead of one bound per wave of CTAs.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "gna_geometry.cuh"
#include "gna_internal.h"
#include "ptx.cuh"

namespace gna {

__device__ int g_device_status = 0;     // GNA_ERR_TIMEOUT once any CTA gave up a wait

namespace {

constexpr int kThreads = 320;
constexpr int kSoftmaxWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS0 = 128;
constexpr uint32_t kColQ = 384;
constexpr uint32_t kColP8 = 448;       // e4m3: P double buffer [448, 480) and [480, 512)

// TMEM column of P(j) in buffer b = j & 1: bf16 P (64 columns) overwrites the
// front of S buffer b; e4m3 P (32 columns) has two buffers of its own.
template <int ESZ>
__device__ __forceinline__ uint32_t p_col(int b)
{
    return ESZ == 1 ? kColP8 + static_cast<uint32_t>(b) * 32 : kColS0 + static_cast<uint32_t>(b) * 128;
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int ESZ>
struct Precision;
template <>
struct Precision<2> {                       // bf16 inputs, bf16 P
    static constexpr uint32_t fmt = kFmtBF16;
    static constexpr float tau = 8.0f;
    static constexpr float p_shift = 0.0f;
};
template <>
struct Precision<1> {                       // e4m3 inputs, e4m3 P
    static constexpr uint32_t fmt = kFmtE4M3;
    static constexpr float tau = 2.0f;
    static constexpr float p_shift = 6.0f;
};

template <int D, int ESZ, int NS>
struct Cfg {
    static constexpr int kRowBytesAll = D * ESZ;                             // bytes of one token row
    static constexpr int kRowBytes = kRowBytesAll >= 128 ? 128 : kRowBytesAll;   // swizzle span
    static constexpr int kChunks = kRowBytesAll / kRowBytes;                 // TMA boxes per tile
    static constexpr int kChunkElems = kRowBytes / ESZ;
    static constexpr uint32_t kSwizzle = kRowBytes == 128 ? kSwizzle128B : kRowBytes == 64 ? kSwizzle64B : kSwizzle32B;
    static constexpr int kTileBytes = kTileElems * kRowBytesAll;
    static constexpr int kSmemK = 0;
    static constexpr int kSmemV = kTileBytes * NS;
    static constexpr int kSmemData = kTileBytes * 2 * NS;
    // at least ~116 KB so that only one CTA (which owns all 512 TMEM columns)
    // is resident per SM
    static constexpr int kSmemAlloc = (kSmemData + 1024) > 118784 ? (kSmemData + 1024) : 118784;
    static constexpr int kKPerInstr = 32 / ESZ;                              // MMA K extent (elements)
    static constexpr int kQKSteps = kRowBytesAll / 32;
    static constexpr int kPVSteps = kTileElems / kKPerInstr;
    static constexpr uint32_t kIdescQK = make_idesc(128, 128, Precision<ESZ>::fmt, false);
    static constexpr uint32_t kIdescPV = make_idesc(128, D, Precision<ESZ>::fmt, false);
    // raster V (RASTER_V): the tile lands token-major like K, the MN-major B of P V
    static constexpr uint32_t kIdescPVmn = make_idesc(128, D, Precision<ESZ>::fmt, true);
    // V arrives in the value layout: a d x 128 (feature-major) tile, loaded as
    // ESZ boxes of d rows x 128 bytes, which is the K-major B operand of P V
    static constexpr int kVChunks = ESZ;
    static constexpr int kVChunkBytes = D * 128;
    static constexpr int kVChunkElems = 128 / ESZ;
    static constexpr int kQHalfWords = kRowBytesAll / 8;                     // TMEM columns of half a Q row
    static constexpr int kPHalfWords = 64 * ESZ / 4;                         // TMEM columns of half a P row
    static constexpr int kOHalf = D / 2;                                     // O columns per half
};

struct Barriers {
    uint64_t q_full;
    uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
    uint64_t s_full[2], p_full[2];
    uint64_t o_done;             // one phase per P V product (rescale waits)
    uint64_t o_final;            // one phase: the last P V product (epilogue wait)
    uint64_t drain;
};

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (a.x * b.x + c.x, a.y * b.y + c.y) in one packed instruction
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    uint64_t ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.ftz.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ void raise_status(volatile int* abort_flag)
{
    *abort_flag = 1;
    atomicExch(&g_device_status, 4 /* GNA_ERR_TIMEOUT */);
}

// Box of KV tiles a Q tile visits (row-major), and per dimension the interval
// of KV tiles that lie inside every window of the Q tile.
struct KvBox {
    int k0[3], cnt[3];
    int full_lo[3], full_hi[3];
};

__device__ __forceinline__ void advance_odometer(int (&kc)[3], const KvBox& box)
{
    if (++kc[2] < box.k0[2] + box.cnt[2]) return;
    kc[2] = box.k0[2];
    if (++kc[1] < box.k0[1] + box.cnt[1]) return;
    kc[1] = box.k0[1];
    ++kc[0];
}

__device__ __forceinline__ uint32_t range_bits32(int lo, int hi)
{
    // bits [lo, hi) clipped to [0, 32)
    lo = lo < 0 ? 0 : lo;
    hi = hi > 32 ? 32 : hi;
    if (hi <= lo) return 0u;
    const uint32_t width_mask = (hi - lo) >= 32 ? 0xffffffffu : ((1u << (hi - lo)) - 1u);
    return width_mask << lo;
}

// Word `wi` (tile elements 32*wi .. 32*wi+31) of the column mask of one query
// row against one KV tile: bit set iff that key lies in the row's window in
// every dimension.  lo_* = the row's window start relative to the tile origin.
__device__ __forceinline__ uint32_t row_mask_word(const FwdParams& p, int wi, int lo_t, int lo_y, int lo_x)
{
    const int tw = p.tile[2];
    const int lw = p.tlog[2];
    const int lh = p.tlog[1];
    if (tw >= 32) {
        const int c0 = wi * 32;
        const int g = c0 >> lw;
        const int cy = g & ((1 << lh) - 1);
        const int ct = g >> lh;
        const int bx = c0 & (tw - 1);
        const bool ok = static_cast<unsigned>(ct - lo_t) < static_cast<unsigned>(p.win[0]) &&
                        static_cast<unsigned>(cy - lo_y) < static_cast<unsigned>(p.win[1]);
        return ok ? range_bits32(lo_x - bx, lo_x - bx + p.win[2]) : 0u;
    }
    const uint32_t mx = range_bits32(lo_x, lo_x + p.win[2]) & ((1u << tw) - 1u);
    const int groups = 32 >> lw;
    uint32_t bits = 0;
    for (int gi = 0; gi < groups; ++gi) {
        const int g = ((wi * 32) >> lw) + gi;
        const int cy = g & ((1 << lh) - 1);
        const int ct = g >> lh;
        const bool ok = static_cast<unsigned>(ct - lo_t) < static_cast<unsigned>(p.win[0]) &&
                        static_cast<unsigned>(cy - lo_y) < static_cast<unsigned>(p.win[1]);
        if (ok) bits |= mx << (gi * tw);
    }
    return bits;
}

template <int ESZ>
__device__ __forceinline__ void pack_p(const float (&x)[64], uint32_t (&out)[64 * ESZ / 4]);

template <>
__device__ __forceinline__ void pack_p<2>(const float (&x)[64], uint32_t (&out)[32])
{
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        out[i] = *reinterpret_cast<uint32_t*>(&h);
    }
}

template <>
__device__ __forceinline__ void pack_p<1>(const float (&x)[64], uint32_t (&out)[16])
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * i], x[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * i + 2], x[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
        out[i] = (lo & 0xffffu) | (hi << 16);
    }
}

// Orders later uses of registers filled by tcgen05.ld after the preceding
// tcgen05.wait::ld (the compiler sees the registers redefined here).
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 8)
        asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]),
                     "+r"(r[i + 6]), "+r"(r[i + 7]));
}

// Store N (8, 16 or 32) consecutive 32-bit TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_store_n(uint32_t taddr, const uint32_t* r)
{
    if constexpr (N == 32) {
        uint32_t a[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) a[i] = r[i];
        tmem_st32(taddr, a);
    } else if constexpr (N == 16) {
        uint32_t a[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = r[i];
        tmem_st16(taddr, a);
    } else {
        static_assert(N == 8, "8, 16 or 32 columns");
        uint32_t a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = r[i];
        tmem_st8(taddr, a);
    }
}

// Load N (16, 32 or 64) consecutive 32-bit TMEM columns of this thread's lane.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N])
{
    if constexpr (N == 64) {
        tmem_ld64(taddr, r);
    } else if constexpr (N == 32) {
        tmem_ld32(taddr, r);
    } else {
        static_assert(N == 16, "16, 32 or 64 columns");
        tmem_ld16(taddr, r);
    }
}

// Multiply O columns [0, N) at taddr of this thread's row by alpha (N multiple of 16).
template <int N>
__device__ __forceinline__ void rescale_o(uint32_t taddr, float alpha)
{
#pragma unroll
    for (int c = 0; c < N; c += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + c, r);
        tmem_wait_ld();
        reg_fence(r);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st16(taddr + c, r);
    }
    tmem_wait_st();
}

// TT, TH, TW: the layout tile when known at compile time (the default tiles),
// or 0, 0, 0 for any tile (runtime shape, slower mask construction).  RASTER:
// q, k, out and lse in the raster layout; RASTER_V: v too (bf16, head_dim 128),
// loaded like k and read by P V as an MN-major operand.
template <int D, int ESZ, int NS, int TT, int TH, int TW, bool RASTER, bool RASTER_V>
__global__ void __launch_bounds__(kThreads, 1) gna_fwd_kernel(const __grid_constant__ FwdParams p)
{
    static_assert(!RASTER_V || (RASTER && ESZ == 2 && D == 128), "raster V: bf16, head_dim 128, raster q and k");
    using C = Cfg<D, ESZ, NS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Barriers bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;
    __shared__ float xchg[2][2][kTileElems];        // [tile parity][half][row]: partial row maxima / sums

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // ---------------------------------------------------------------- tile geometry (all threads)
    const int64_t q_tile_global = blockIdx.x;                 // (b*heads + h)*tiles_per_head_q + qt
    const int qt_id = static_cast<int>(q_tile_global % p.tiles_per_head_q);
    const int64_t bh = q_tile_global / p.tiles_per_head_q;
    int qc[3];
    qc[2] = qt_id % p.nt_q[2];
    qc[1] = (qt_id / p.nt_q[2]) % p.nt_q[1];
    qc[0] = qt_id / (p.nt_q[2] * p.nt_q[1]);
    KvBox box;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        const DimRange r = dim_range(qc[d], p.tile_q[d], p.tile[d], p.dims[d], p.win[d], p.str[d], p.off[d]);
        box.k0[d] = r.k0;
        box.cnt[d] = r.k1 - r.k0 + 1;
        dim_full_range(p.tile[d], p.dims[d], p.win[d], r, box.full_lo[d], box.full_hi[d]);
    }
    const int n_kv = box.cnt[0] * box.cnt[1] * box.cnt[2];
    const int64_t kv_row_base = bh * p.tiles_per_head * kTileElems;
    const int b_idx = static_cast<int>(bh / p.heads);          // batch and head of this CTA
    const int h_idx = static_cast<int>(bh % p.heads);

    const uint32_t sK = smem_u32(smem + C::kSmemK);
    const uint32_t sV = smem_u32(smem + C::kSmemV);
    auto bar = [](uint64_t& b) { return smem_u32(&b); };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(bars.q_full), kSoftmaxWarps);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(bars.k_full[s]), 1);
            mbar_init(bar(bars.k_empty[s]), 1);
            mbar_init(bar(bars.v_full[s]), 1);
            mbar_init(bar(bars.v_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(bars.s_full[s]), 1);
            mbar_init(bar(bars.p_full[s]), kSoftmaxWarps);
        }
        mbar_init(bar(bars.o_done), 1);
        mbar_init(bar(bars.o_final), 1);
        mbar_init(bar(bars.drain), 1);
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    // The producer and MMA warps run converged: every lane polls the
    // barriers, one elected lane issues the TMA copies / MMAs / commits, so
    // the addresses and descriptors stay warp-uniform.
    if (warp == 0) {
        // ============================================================ TMA producer
        if (elect_one_sync()) {
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmV);
        }
        int k_issued = 0, v_issued = 0;              // KV tiles whose K / V loads were issued
        bool early = false;
        int kc[3] = {box.k0[0], box.k0[1], box.k0[2]};
        for (int j = 0; j < n_kv; ++j, advance_odometer(kc, box)) {
            const int s = j % NS;
            const uint32_t ph = ((j / NS) & 1) ^ 1;
            const int tile_id = (kc[0] * p.nt[1] + kc[1]) * p.nt[2] + kc[2];
            const int32_t row = static_cast<int32_t>(kv_row_base + static_cast<int64_t>(tile_id) * kTileElems);
            if (j >= NS && !__all_sync(0xffffffffu, mbar_wait(bar(bars.k_empty[s]), ph, &abort_flag, &g_device_status))) {
                early = true;
                break;
            }
            if (j == p.fault_skip_kv) { early = true; break; }   // test hook: consumers wait in vain
            if (elect_one_sync()) {
                mbar_arrive_expect_tx(bar(bars.k_full[s]), C::kTileBytes);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    const uint32_t dst = sK + s * C::kTileBytes + c * kTileElems * C::kRowBytes;
                    if constexpr (RASTER) {
                        // the tile's 128 tokens of this head straight from the raster
                        // layout: the box (t, y, x) lands in tile element order,
                        // positions past the grid read as zero
                        tma_load_5d(dst, &p.tmK, bar(bars.k_full[s]), h_idx * D + c * C::kChunkElems,
                                    kc[2] * p.tile[2], kc[1] * p.tile[1], kc[0] * p.tile[0], b_idx);
                    } else {
                        tma_load_2d(dst, &p.tmK, bar(bars.k_full[s]), c * C::kChunkElems, row);
                    }
                }
            }
            __syncwarp();
            ++k_issued;
            if (j >= NS && !__all_sync(0xffffffffu, mbar_wait(bar(bars.v_empty[s]), ph, &abort_flag, &g_device_status))) {
                early = true;
                break;
            }
            if (elect_one_sync()) {
                mbar_arrive_expect_tx(bar(bars.v_full[s]), C::kTileBytes);
                if constexpr (RASTER_V) {
                    // token-major, exactly as the K tile (positions past the grid read as zero)
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c)
                        tma_load_5d(sV + s * C::kTileBytes + c * kTileElems * C::kRowBytes, &p.tmV, bar(bars.v_full[s]),
                                    h_idx * D + c * C::kChunkElems, kc[2] * p.tile[2], kc[1] * p.tile[1],
                                    kc[0] * p.tile[0], b_idx);
                } else {
                    const int32_t vrow = static_cast<int32_t>((kv_row_base / kTileElems + tile_id) * D);
#pragma unroll
                    for (int c = 0; c < C::kVChunks; ++c)
                        tma_load_2d(sV + s * C::kTileBytes + c * C::kVChunkBytes, &p.tmV, bar(bars.v_full[s]),
                                    c * C::kVChunkElems, vrow);
                }
            }
            __syncwarp();
            ++v_issued;
        }
        if (early) {
            if (p.fault_skip_kv < 0 && lane == 0) raise_status(&abort_flag);
            // Drain: wait (bounded, ignoring the abort flag) for the loads
            // still in flight so that no TMA write lands after the CTA exits.
            const volatile int never = 0;
            for (int j = (k_issued > NS ? k_issued - NS : 0); j < k_issued; ++j)
                mbar_wait(bar(bars.k_full[j % NS]), (j / NS) & 1, &never);
            for (int j = (v_issued > NS ? v_issued - NS : 0); j < v_issued; ++j)
                mbar_wait(bar(bars.v_full[j % NS]), (j / NS) & 1, &never);
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        const uint32_t tO = tmem + kColO;
        const uint32_t tQ = tmem + kColQ;
        // descriptors of stage 0, chunk 0; stage / k-step offsets are added
        // to the start-address field (addresses >> 4 stay below 2^14)
        const uint64_t dK0 = make_smem_desc(sK, 16, 8 * C::kRowBytes, C::kSwizzle);
        // value layout: K-major (feature rows of 128 tokens); raster V: MN-major (token
        // rows, the next 64 features 16 KB on, 8-token groups 1 KB apart)
        const uint64_t dV0 = RASTER_V ? make_smem_desc(sV, kTileElems * C::kRowBytes, 8 * C::kRowBytes, kSwizzle128B)
                                      : make_smem_desc(sV, 16, 1024, kSwizzle128B);
        auto issue_pv = [&](int i) -> bool {
            const int s = i % NS;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.v_full[s]), (i / NS) & 1, &abort_flag, &g_device_status))) return false;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.p_full[i & 1]), (i >> 1) & 1, &abort_flag, &g_device_status))) return false;
            tc_fence_after();
            if (elect_one_sync()) {
                const uint64_t dv = dV0 + static_cast<uint64_t>((s * C::kTileBytes) >> 4);
                const uint32_t tP = tmem + p_col<ESZ>(i & 1);
#pragma unroll
                for (int kk = 0; kk < C::kPVSteps; ++kk) {
                    // k-step kk covers tokens [kk * K, kk * K + K): 32 bytes of every feature
                    // row (value layout), or K token rows (raster V)
                    const int off = RASTER_V ? kk * C::kKPerInstr * C::kRowBytes
                                             : ((kk * 32) / 128) * C::kVChunkBytes + ((kk * 32) % 128);
                    const uint64_t d = dv + static_cast<uint64_t>(off >> 4);
                    const uint32_t idesc = RASTER_V ? C::kIdescPVmn : C::kIdescPV;
                    if (ESZ == 2) mma_f16_ts(tO, tP + kk * 8, d, idesc, (i > 0 || kk > 0) ? 1u : 0u);
                    else mma_f8_ts(tO, tP + kk * 8, d, idesc, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(bars.o_done));
                if (i == n_kv - 1) mma_commit(bar(bars.o_final));
                if (i + NS < n_kv) mma_commit(bar(bars.v_empty[s]));
            }
            __syncwarp();
            return true;
        };
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.q_full), 0, &abort_flag, &g_device_status));
        for (int j = 0; ok && j < n_kv; ++j) {
            const int s = j % NS;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.k_full[s]), (j / NS) & 1, &abort_flag, &g_device_status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (elect_one_sync()) {
                const uint64_t dk = dK0 + static_cast<uint64_t>((s * C::kTileBytes) >> 4);
                const uint32_t tS = tmem + kColS0 + (j & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < C::kQKSteps; ++kk) {
                    constexpr int kChunkStride = kTileElems * C::kRowBytes;
                    const int off = ((kk * 32) / C::kRowBytes) * kChunkStride + ((kk * 32) % C::kRowBytes);
                    const uint64_t d = dk + static_cast<uint64_t>(off >> 4);
                    if (ESZ == 2) mma_f16_ts(tS, tQ + kk * 8, d, C::kIdescQK, kk > 0 ? 1u : 0u);
                    else mma_f8_ts(tS, tQ + kk * 8, d, C::kIdescQK, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(bars.s_full[j & 1]));
                if (j + NS < n_kv) mma_commit(bar(bars.k_empty[s]));
            }
            __syncwarp();
            if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
        }
        if (ok) ok = issue_pv(n_kv - 1);
        if (!ok) {
            // wait for every MMA issued so far before TMEM is released
            if (elect_one_sync()) {
                raise_status(&abort_flag);
                mma_commit(bar(bars.drain));
            }
            __syncwarp();
            const volatile int never = 0;
            mbar_wait(bar(bars.drain), 0, &never);
        }
    } else {
        // ============================================================ softmax / correction / epilogue
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t pair_bar = 1 + quarter;            // named barrier of the two warps sharing these rows

        // query coordinates of this row
        int qpos[3], st[3];
        {
            const int ix = row & (p.tile_q[2] - 1);
            const int iy = (row >> p.tlog_q[2]) & (p.tile_q[1] - 1);
            const int it = row >> (p.tlog_q[1] + p.tlog_q[2]);
            qpos[0] = qc[0] * p.tile_q[0] + it;
            qpos[1] = qc[1] * p.tile_q[1] + iy;
            qpos[2] = qc[2] * p.tile_q[2] + ix;
        }
        const bool row_valid = qpos[0] < p.dims[0] && qpos[1] < p.dims[1] && qpos[2] < p.dims[2];
        // row of this query in the tensor q / out / lse are stored in
        const int64_t io_row = RASTER
            ? (((static_cast<int64_t>(b_idx) * p.dims[0] + qpos[0]) * p.dims[1] + qpos[1]) * p.dims[2] + qpos[2]) *
                      p.heads + h_idx
            : q_tile_global * kTileElems + row;

        // Q row -> TMEM (A operand of S = Q K^T); padding rows of the raster
        // layout do not exist and are zero
        {
            constexpr int W = C::kQHalfWords;
            const uint4* src = reinterpret_cast<const uint4*>(
                static_cast<const uint8_t*>(p.q) + io_row * C::kRowBytesAll + half * (C::kRowBytesAll / 2));
            const bool load = row_valid || !RASTER;
            uint32_t qw[W];
#pragma unroll
            for (int i = 0; i < W / 4; ++i) {
                const uint4 v = load ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
                qw[4 * i] = v.x;
                qw[4 * i + 1] = v.y;
                qw[4 * i + 2] = v.z;
                qw[4 * i + 3] = v.w;
            }
            tmem_store_n<W>(tmem + kColQ + lane_addr + half * W, qw);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.q_full));
        }

        // window starts of this query
#pragma unroll
        for (int d = 0; d < 3; ++d) st[d] = window_start(qpos[d], p.dims[d], p.win[d], p.str[d], p.off[d]);

        float scale_log2 = p.scale * kLog2e;
        float out_scale = 1.0f;
        if (ESZ == 1 && p.descale != nullptr) {
            scale_log2 *= p.descale[0] * p.descale[1];
            out_scale = p.descale[2];
        }
        constexpr float kTau = Precision<ESZ>::tau;
        constexpr float kShift = Precision<ESZ>::p_shift;

        float m_run = -INFINITY;   // running reference maximum, log2 units (scaled scores)
        float l_run = 0.0f;        // this half's running sum of P (same shifted units as P)
        bool ok = true;
        const uint32_t t_ohalf = tmem + kColO + lane_addr + half * C::kOHalf;

        // A failed wait never leaves the loop early: the two warps sharing
        // these rows meet at a named barrier every tile, so a warp that gives
        // up raises the abort flag and keeps iterating without doing work
        // until both have passed the same number of barriers.
        int kc[3] = {box.k0[0], box.k0[1], box.k0[2]};   // KV tile of iteration j (row-major odometer)
        for (int j = 0; j < n_kv; ++j, advance_odometer(kc, box)) {
            const int sb = j & 1;
            if (ok) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.s_full[sb]), (j >> 1) & 1, &abort_flag, &g_device_status));
                if (!ok) raise_status(&abort_flag);
            }
            const uint32_t t_s = tmem + kColS0 + sb * 128 + lane_addr;
            float s[64];
            float mx = -INFINITY;
            if (ok) {
                tc_fence_after();
                uint32_t rs[64];
                tmem_ld64(t_s + half * 64, rs);
                // while the scores travel from TMEM: is this KV tile partial?
                // per dimension: does this KV tile lie inside every window of the Q tile?
                bool fd[3];
#pragma unroll
                for (int d = 0; d < 3; ++d) fd[d] = kc[d] >= box.full_lo[d] && kc[d] <= box.full_hi[d];
                const bool full = fd[0] && fd[1] && fd[2];
                const int lo_t = st[0] - kc[0] * p.tile[0];
                const int lo_y = st[1] - kc[1] * p.tile[1];
                const int lo_x = st[2] - kc[2] * p.tile[2];
                if constexpr (TW > 0) {
                    tmem_wait_ld();
                    reg_fence(rs);
#pragma unroll
                    for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(rs[i]);
                    // element (ct, cy, cx) of the tile is masked iff one of its
                    // coordinates leaves the row's window: -inf biases per x
                    // position (only if x is partial) and per (t, y) group of
                    // TW columns (only if t or y is partial)
                    if (!fd[2]) {
                        float bx[TW];
#pragma unroll
                        for (int cx = 0; cx < TW; ++cx)
                            bx[cx] = static_cast<unsigned>(cx - lo_x) < static_cast<unsigned>(p.win[2]) ? 0.0f : -INFINITY;
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            const float2 v = fadd2(make_float2(s[c], s[c + 1]), make_float2(bx[c % TW], bx[(c + 1) % TW]));
                            s[c] = v.x;
                            s[c + 1] = v.y;
                        }
                    }
                    if (!(fd[0] && fd[1])) {
                        constexpr int GPH = 64 / TW;      // (t, y) groups per half row
                        float bg[GPH];
#pragma unroll
                        for (int gi = 0; gi < GPH; ++gi) {
                            const int g = half * GPH + gi;
                            const int cy = g % TH, ct = g / TH;
                            bg[gi] = (static_cast<unsigned>(ct - lo_t) < static_cast<unsigned>(p.win[0]) &&
                                      static_cast<unsigned>(cy - lo_y) < static_cast<unsigned>(p.win[1]))
                                         ? 0.0f : -INFINITY;
                        }
#pragma unroll
                        for (int c = 0; c < 64; c += 2) {
                            const float2 v = fadd2(make_float2(s[c], s[c + 1]), make_float2(bg[c / TW], bg[c / TW]));
                            s[c] = v.x;
                            s[c + 1] = v.y;
                        }
                    }
                } else {
                    uint32_t m0 = 0xffffffffu, m1 = 0xffffffffu;
                    if (!full) {
                        m0 = row_mask_word(p, 2 * half, lo_t, lo_y, lo_x);
                        m1 = row_mask_word(p, 2 * half + 1, lo_t, lo_y, lo_x);
                    }
                    tmem_wait_ld();
                    reg_fence(rs);
#pragma unroll
                    for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(rs[i]);
                    if (!full) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            s[c] = (m0 >> c) & 1u ? s[c] : -INFINITY;
                            s[32 + c] = (m1 >> c) & 1u ? s[32 + c] : -INFINITY;
                        }
                    }
                }
                // maximum of this half row (four independent 3-input chains)
                float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; c += 8) {
                    a0 = max3(a0, s[c], s[c + 1]);
                    a1 = max3(a1, s[c + 2], s[c + 3]);
                    a2 = max3(a2, s[c + 4], s[c + 5]);
                    a3 = max3(a3, s[c + 6], s[c + 7]);
                }
                mx = fmaxf(max3(a0, a1, a2), a3);
            }
            // combine with the other half of the row (always executed)
            xchg[sb][half][row] = mx;
            named_bar_sync(pair_bar, 64);
            mx = fmaxf(mx, xchg[sb][half ^ 1][row]);
            if (!ok) continue;
            const float m_tile = mx * scale_log2;   // -inf if the row is fully masked

            const bool need = m_tile > m_run + kTau;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? m_tile : m_run;
                const float alpha = need ? fast_exp2(m_run - m_new) : 1.0f;   // 0 when m_run = -inf
                m_run = m_new;
                l_run *= alpha;
                if (j > 0) {
                    // O holds PV(0..j-1): wait for PV(j-1), then rescale this half's
                    // columns.  S(j) has arrived, so every MMA issued before QK(j),
                    // PV(j-2) included, is complete: o_done is at most one phase
                    // behind and the parity wait is exact.
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.o_done), (j - 1) & 1, &abort_flag, &g_device_status));
                    if (!ok) {
                        raise_status(&abort_flag);
                        continue;
                    }
                    tc_fence_after();
                    rescale_o<C::kOHalf>(t_ohalf, alpha);
                }
            }
            const float m_eff = (m_run == -INFINITY) ? 0.0f : m_run - kShift;
            const float2 sc2 = make_float2(scale_log2, scale_log2);
            const float2 nm2 = make_float2(-m_eff, -m_eff);
            float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
#pragma unroll
            for (int c = 0; c < 64; c += 8) {
                float2 t0 = ffma2(make_float2(s[c], s[c + 1]), sc2, nm2);
                float2 t1 = ffma2(make_float2(s[c + 2], s[c + 3]), sc2, nm2);
                float2 t2 = ffma2(make_float2(s[c + 4], s[c + 5]), sc2, nm2);
                float2 t3 = ffma2(make_float2(s[c + 6], s[c + 7]), sc2, nm2);
                t0 = make_float2(fast_exp2(t0.x), fast_exp2(t0.y));
                t1 = make_float2(fast_exp2(t1.x), fast_exp2(t1.y));
                t2 = make_float2(fast_exp2(t2.x), fast_exp2(t2.y));
                t3 = make_float2(fast_exp2(t3.x), fast_exp2(t3.y));
                s[c] = t0.x; s[c + 1] = t0.y; s[c + 2] = t1.x; s[c + 3] = t1.y;
                s[c + 4] = t2.x; s[c + 5] = t2.y; s[c + 6] = t3.x; s[c + 7] = t3.y;
                acc0 = fadd2(acc0, t0);
                acc1 = fadd2(acc1, t1);
                acc2 = fadd2(acc2, t2);
                acc3 = fadd2(acc3, t3);
            }
            acc0 = fadd2(fadd2(acc0, acc1), fadd2(acc2, acc3));
            l_run += acc0.x + acc0.y;
            {
                uint32_t pk[C::kPHalfWords];
                pack_p<ESZ>(s, pk);
                tmem_store_n<C::kPHalfWords>(tmem + p_col<ESZ>(sb) + lane_addr + half * C::kPHalfWords, pk);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.p_full[sb]));
        }

        // ------------------------------------------------------------ epilogue
        if (ok) {
            // A parity wait on o_done could pass here while the barrier is
            // still two phases behind (P V of the second-to-last tile not yet
            // done): the last product has a barrier of its own.
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.o_final), 0, &abort_flag, &g_device_status));
            if (!ok) raise_status(&abort_flag);
        }
        // every thread of the pair reaches this exchange (even on failure)
        xchg[n_kv & 1][half][row] = l_run;
        named_bar_sync(pair_bar, 64);
        const float l_tot = l_run + xchg[n_kv & 1][half ^ 1][row];
        if (ok) {
            tc_fence_after();
            const bool has = row_valid && l_tot > 0.0f;
            const float inv_l = has ? out_scale / l_tot : 0.0f;
            uint8_t* out_row = static_cast<uint8_t*>(p.out) + io_row * (D * 2) + half * D;
            const bool store = row_valid || !RASTER;
            // this half of the O row in one TMEM load (16, 32 or 64 columns)
            uint32_t r[C::kOHalf];
            tmem_ld_n<C::kOHalf>(t_ohalf, r);
            tmem_wait_ld();
            reg_fence(r);
#pragma unroll
            for (int c = 0; c < C::kOHalf; c += 16) {
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[c + 2 * i]) * inv_l,
                                                             __uint_as_float(r[c + 2 * i + 1]) * inv_l);
                    pk[i] = *reinterpret_cast<uint32_t*>(&h);
                }
                if (store) {
                    uint4* dst = reinterpret_cast<uint4*>(out_row + c * 2);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
            if (p.lse != nullptr && half == 0 && store) {
                const float lse = has ? (m_run - kShift + __log2f(l_tot)) * kLn2 : -INFINITY;
                p.lse[io_row] = lse;
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int ESZ, int NS, int TT, int TH, int TW, bool RASTER, bool RASTER_V>
cudaError_t launch_tile(const FwdParams& p, int64_t num_q_tiles, cudaStream_t stream)
{
    using C = Cfg<D, ESZ, NS>;
    static_assert(NS <= 4, "barrier arrays hold 4 stages");
    static_assert(C::kSmemAlloc <= 232448 - 4096, "shared memory budget");
    static_assert(C::kQHalfWords == 8 || C::kQHalfWords == 16 || C::kQHalfWords == 32, "Q half-row width");
    static_assert(ESZ == 2 || (kColQ + 2 * C::kQHalfWords <= kColP8 && kColP8 + 4 * C::kPHalfWords <= kTmemCols),
                  "TMEM columns of the e4m3 P buffers");
    auto kern = gna_fwd_kernel<D, ESZ, NS, TT, TH, TW, RASTER, RASTER_V>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    kern<<<dim3(static_cast<unsigned>(num_q_tiles)), kThreads, C::kSmemAlloc, stream>>>(p);
    return cudaGetLastError();
}

// The default tiles, and (head_dim 128) the key/value tiles the pair planner
// picks for the video latent, get a kernel with the KV tile shape compiled into
// the mask code; any other tile runs the generic mask.
template <int D, int ESZ, int NS, bool RASTER, bool RASTER_V = false>
cudaError_t launch_layout(const FwdParams& p, int64_t num_q_tiles, cudaStream_t stream)
{
    if (p.tile[0] == 2 && p.tile[1] == 8 && p.tile[2] == 8)
        return launch_tile<D, ESZ, NS, 2, 8, 8, RASTER, RASTER_V>(p, num_q_tiles, stream);
    if (p.tile[0] == 1 && p.tile[1] == 8 && p.tile[2] == 16)
        return launch_tile<D, ESZ, NS, 1, 8, 16, RASTER, RASTER_V>(p, num_q_tiles, stream);
    if constexpr (D == 128) {
        if (p.tile[0] == 2 && p.tile[1] == 4 && p.tile[2] == 16)
            return launch_tile<D, ESZ, NS, 2, 4, 16, RASTER, RASTER_V>(p, num_q_tiles, stream);
        if (p.tile[0] == 4 && p.tile[1] == 4 && p.tile[2] == 8)
            return launch_tile<D, ESZ, NS, 4, 4, 8, RASTER, RASTER_V>(p, num_q_tiles, stream);
    }
    return launch_tile<D, ESZ, NS, 0, 0, 0, RASTER, RASTER_V>(p, num_q_tiles, stream);
}

// The raster layout of q, k, out and lse is a separate kernel, so the tiled
// path carries none of its addressing.
template <int D, int ESZ, int NS>
cudaError_t launch_impl(const FwdParams& p, int64_t num_q_tiles, cudaStream_t stream)
{
    if constexpr (ESZ == 2 && D == 128) {
        if (p.raster == 2) return launch_layout<D, ESZ, NS, true, true>(p, num_q_tiles, stream);
    }
    if (p.raster == 2) return cudaErrorNotSupported;
    return p.raster ? launch_layout<D, ESZ, NS, true>(p, num_q_tiles, stream)
                    : launch_layout<D, ESZ, NS, false>(p, num_q_tiles, stream);
}

}  // namespace

cudaError_t launch_forward(const FwdParams& p, int head_dim, int elem_size, int64_t num_q_tiles, cudaStream_t stream)
{
    if (num_q_tiles <= 0) return cudaSuccess;
    if (elem_size == 2) {
        switch (head_dim) {
            case 32: return launch_impl<32, 2, 4>(p, num_q_tiles, stream);
            case 64: return launch_impl<64, 2, 4>(p, num_q_tiles, stream);
            case 128: return launch_impl<128, 2, 3>(p, num_q_tiles, stream);
            default: return cudaErrorNotSupported;
        }
    }
    if (elem_size == 1 && head_dim == 128) return launch_impl<128, 1, 4>(p, num_q_tiles, stream);
    return cudaErrorNotSupported;
}

cudaError_t read_and_clear_status(int* status, cudaStream_t stream)
{
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_device_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*status != 0) {
        e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return e;
        e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace gna
