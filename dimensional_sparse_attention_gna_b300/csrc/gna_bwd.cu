// Backward pass of the GNA forward for sm_103a: the per-query delta, dQ (one CTA
// per Q tile, below) and dK / dV (one CTA per KV tile, further down).
//
// GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践") §4.2, problem 1
// and §5 ask for GNA in training; the page gives no backward, so this is the
// derivative of the forward (for L = sum_i <dout_i, out_i>):
//
//   p_ij  = exp(s_ij - lse_i)   for j in the window of query i
//   dp_ij = <dout_i, v_j>
//   ds_ij = p_ij (dp_ij - delta_i),   delta_i = <dout_i, out_i> = sum_j p_ij dp_ij
//   dq_i  = scale sum_j ds_ij k_j
//
// dq_i needs only query i's own window, so the dQ kernel walks a Q tile's box
// of KV tiles exactly as the forward does (GNA page §1.1: the stride decides
// which KV tiles a Q tile visits; §2.1: the element mask only on partial KV
// tiles).  One CTA per 128-query tile, 320 threads:
//   warp 0      TMA producer: dO once; per KV tile K, V (tiled) and K in the
//               value layout (feature-major), each through a 2-slot ring of
//               its own, so a slot is refilled as soon as its one product is done
//   warp 1      TMEM allocator and tcgen05.mma issuer
//   warps 2..9  dS: thread = (query row, half of the 128 key columns)
// TMEM (512 columns): dQ [0, d), S [128, 256), dP [256, 384), dS [384, 448),
// Q [448, 448 + d / 2) for head_dim d.  Per KV tile: S = Q K^T (A from TMEM),
// dP = dO V^T (both operands from shared memory), then dQ += dS K with dS
// (bf16) in TMEM as the A operand and K in the value layout as the K-major B
// operand (as V is for P V in the forward).  S, dP and dS each have columns of
// their own: the dS warps hand S back as soon as they hold it in registers and
// form p (bf16) from it while dP is computed, then hand dP back once read, so
// S and dP of the next KV tile are computed while they form dS; only the store
// of dS waits for the previous dQ product.  No TMEM reuse depends on the order
// in which the tensor core executes products: every reuse waits on a barrier.
// The element mask of a partial tile is one 32-bit word per 32 key columns
// (box_mask_word).
//
// Every mbarrier wait is bounded; a role that gives up raises the abort flag
// and the device status word, and the CTA drains and exits.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gna_geometry.cuh"
#include "gna_internal.h"
#include "ptx.cuh"

namespace gna {

__device__ int g_bwd_status = 0;     // GNA_ERR_TIMEOUT once any CTA gave up a wait (every wait also stops then)

namespace {

constexpr int kBThreads = 320;
constexpr int kBSoftmaxWarps = 8;
constexpr uint32_t kBTmemCols = 512;
constexpr uint32_t kColDQ = 0;
constexpr uint32_t kColS = 128;
constexpr uint32_t kColDP = 256;
constexpr uint32_t kColDS = 384;
constexpr uint32_t kColQ = 448;
constexpr int kBStages = 2;
constexpr float kBLog2e = 1.4426950408889634f;

constexpr int kDQSteps = kTileElems / 16;        // K = 16 bf16 per MMA over 128 keys / queries
constexpr uint32_t kIdesc = make_idesc(128, 128, kFmtBF16, false);

// bf16 tiles of head_dim D (32, 64 or 128): a token row is 2 D bytes, one 64-byte
// or one or two 128-byte swizzle spans
template <int D>
struct BwdCfg {
    static constexpr int kRowBytes = D * 2;                    // bytes per token row
    static constexpr int kSpan = kRowBytes < 128 ? kRowBytes : 128;     // swizzle span of a tiled tile
    static constexpr uint32_t kSwizzle = kSpan == 128 ? kSwizzle128B : kSwizzle64B;
    static constexpr int kChunks = kRowBytes / kSpan;          // spans per row (TMA boxes per tile)
    static constexpr int kTileBytes = kTileElems * kRowBytes;  // one 128-token tile (either layout)
    // at least ~116 KB, so that one CTA (which takes all 512 TMEM columns) is
    // resident per SM and a second one never waits in the TMEM allocation
    static constexpr int kMinSmem = 118784;
    // dQ kernel: dO, then two slots each of K, V and K (value layout)
    static constexpr int kDQSmemAlloc = (7 * kTileBytes + 1024) > kMinSmem ? (7 * kTileBytes + 1024) : kMinSmem;
    static constexpr int kQKSteps = kRowBytes / 32;            // MMA k-steps over the head dimension
    static constexpr int kHalfWords = kRowBytes / 8;           // TMEM columns of half a Q / dO row
    static constexpr int kHalfCols = D / 2;                    // TMEM columns of half a dQ / dK / dV row
    static constexpr uint32_t kIdescDQ = make_idesc(128, D, kFmtBF16, false);    // dQ += dS K: N = D
    static constexpr int kKVStageBytes = 2 * kTileBytes + 1024;                  // Q_i, dO_i, lse_i, delta_i
    static constexpr int kKVSmemAlloc = (2 * kTileBytes + kBStages * kKVStageBytes + 1024) > kMinSmem
                                            ? (2 * kTileBytes + kBStages * kKVStageBytes + 1024) : kMinSmem;
    static constexpr uint32_t kIdescMN = make_idesc(128, D, kFmtBF16, true);     // dV, dK: N = D, B MN-major
    static_assert(D == 32 || D == 64 || D == 128, "head_dim 32, 64 or 128");
};

// the dQ kernel's three shared-memory rings (one per operand of a KV tile)
enum { kRingK = 0, kRingV = 1, kRingKv = 2, kRings = 3 };

struct BwdBars {
    uint64_t q_full;              // Q rows stored in TMEM (8 warps)
    uint64_t do_full;             // the dO tile landed in shared memory
    uint64_t full[kRings][2];     // K / V / K (value layout) of a KV tile landed in its slot
    uint64_t empty[kRings][2];    // the one product that reads the slot is done
    uint64_t s_full;              // S of KV tile j is in TMEM (one phase per tile)
    uint64_t s_free;              // the dS warps hold S(j) in registers: S may take S(j + 1) (8 warps)
    uint64_t dp_full;             // dP of KV tile j is in TMEM
    uint64_t dp_free;             // the dS warps hold dP(j) in registers (8 warps)
    uint64_t ds_full;             // dS of KV tile j is in TMEM (8 warps)
    uint64_t ds_free;             // dQ(j) is done: dS may take dS(j + 1)
    uint64_t dq_final;            // the last dQ product is done
    uint64_t drain;
};

struct BwdBox {
    int k0[3], cnt[3];
    int full_lo[3], full_hi[3];
};

__device__ __forceinline__ void bwd_odometer(int (&kc)[3], const BwdBox& box)
{
    if (++kc[2] < box.k0[2] + box.cnt[2]) return;
    kc[2] = box.k0[2];
    if (++kc[1] < box.k0[1] + box.cnt[1]) return;
    kc[1] = box.k0[1];
    ++kc[0];
}

__device__ __forceinline__ void bwd_raise(volatile int* abort_flag)
{
    *abort_flag = 1;
    atomicExch(&g_bwd_status, 4 /* GNA_ERR_TIMEOUT */);
}

__device__ __forceinline__ float bwd_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs: (a.x * b.x + c.x, a.y * b.y + c.y), a + b and a * b in one
// instruction each.
__device__ __forceinline__ float2 bwd_ffma2(float2 a, float2 b, float2 c)
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

__device__ __forceinline__ float2 bwd_fadd2(float2 a, float2 b)
{
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("add.rn.ftz.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ float2 bwd_fmul2(float2 a, float2 b)
{
    uint64_t ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mul.rn.ftz.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

// N = 8, 16 or 32 consecutive TMEM columns of this warp's lane quarter
template <int N>
__device__ __forceinline__ void bwd_tmem_st(uint32_t taddr, const uint32_t (&r)[N])
{
    if constexpr (N == 32) {
        tmem_st32(taddr, r);
    } else if constexpr (N == 16) {
        tmem_st16(taddr, r);
    } else {
        static_assert(N == 8, "8, 16 or 32 columns");
        tmem_st8(taddr, r);
    }
}

template <int N>
__device__ __forceinline__ void bwd_reg_fence(uint32_t (&r)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 8)
        asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]),
                     "+r"(r[i + 6]), "+r"(r[i + 7]));
}

// N (16 or 32) fp32 TMEM columns of this thread's lane, times mul, to N bf16 at
// dst (16-byte aligned); zeros when !load
template <int N>
__device__ __forceinline__ void bwd_store_cols(uint32_t taddr, bool load, float mul, uint8_t* dst)
{
    uint32_t r[N];
    if (load) {
        if constexpr (N == 32) {
            tmem_ld32(taddr, r);
        } else {
            static_assert(N == 16, "16 or 32 columns");
            tmem_ld16(taddr, r);
        }
        tmem_wait_ld();
        bwd_reg_fence(r);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) r[i] = 0u;
    }
    uint32_t pk[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
        pk[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < N / 8; ++i) d[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

template <int D>
__global__ void __launch_bounds__(kBThreads, 1) gna_bwd_dq_kernel(const __grid_constant__ BwdParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ BwdBars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // ---------------------------------------------------------------- tile geometry
    const int64_t q_tile_global = blockIdx.x;                 // (b*heads + h)*tiles_per_head + qt
    const int qt_id = static_cast<int>(q_tile_global % p.tiles_per_head);
    const int64_t bh = q_tile_global / p.tiles_per_head;
    int qc[3];
    qc[2] = qt_id % p.nt[2];
    qc[1] = (qt_id / p.nt[2]) % p.nt[1];
    qc[0] = qt_id / (p.nt[2] * p.nt[1]);
    BwdBox box;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        const DimRange r = dim_range(qc[d], p.tile[d], p.tile[d], p.dims[d], p.win[d], p.str[d], p.off[d]);
        box.k0[d] = r.k0;
        box.cnt[d] = r.k1 - r.k0 + 1;
        dim_full_range(p.tile[d], p.dims[d], p.win[d], r, box.full_lo[d], box.full_hi[d]);
    }
    const int n_kv = box.cnt[0] * box.cnt[1] * box.cnt[2];
    const int64_t kv_tile_base = bh * p.tiles_per_head;       // first tile of this (b, head) plane

    auto bar = [](uint64_t& b) { return smem_u32(&b); };
    // shared memory: dO, then slots K0 K1 V0 V1 Kv0 Kv1 (one tile each)
    const uint32_t sDO = smem_u32(smem);
    auto slot_addr = [&](int ring, int slot) {
        return sDO + static_cast<uint32_t>((1 + 2 * ring + slot) * C::kTileBytes);
    };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(bars.q_full), kBSoftmaxWarps);
        mbar_init(bar(bars.do_full), 1);
        for (int r = 0; r < kRings; ++r) {
            for (int s = 0; s < 2; ++s) {
                mbar_init(bar(bars.full[r][s]), 1);
                mbar_init(bar(bars.empty[r][s]), 1);
            }
        }
        mbar_init(bar(bars.s_full), 1);
        mbar_init(bar(bars.s_free), kBSoftmaxWarps);
        mbar_init(bar(bars.dp_full), 1);
        mbar_init(bar(bars.dp_free), kBSoftmaxWarps);
        mbar_init(bar(bars.ds_full), kBSoftmaxWarps);
        mbar_init(bar(bars.ds_free), 1);
        mbar_init(bar(bars.dq_final), 1);
        mbar_init(bar(bars.drain), 1);
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base_sh), kBTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0) {
        // ============================================================ TMA producer
        if (elect_one_sync()) {
            prefetch_tensormap(&p.tmDO);
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmV);
            prefetch_tensormap(&p.tmKv);
            // this Q tile's dO rows: 128 rows x 64 elements per box (128-byte swizzle)
            mbar_arrive_expect_tx(bar(bars.do_full), C::kTileBytes);
            const int32_t row = static_cast<int32_t>(q_tile_global * kTileElems);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d(sDO + c * kTileElems * C::kSpan, &p.tmDO, bar(bars.do_full), c * (C::kSpan / 2), row);
        }
        __syncwarp();
        int issued[kRings] = {0, 0, 0};
        bool early = false;
        int kc[3] = {box.k0[0], box.k0[1], box.k0[2]};
        for (int j = 0; j < n_kv && !early; ++j, bwd_odometer(kc, box)) {
            if (j == p.fault_skip_kv) { early = true; break; }   // test hook: consumers wait in vain
            const int slot = j & 1;
            const int64_t tile = kv_tile_base + (kc[0] * p.nt[1] + kc[1]) * p.nt[2] + kc[2];
            for (int r = 0; r < kRings; ++r) {
                // the slot's previous tile (j - 2) is done with it
                if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar(bars.empty[r][slot]), ((j >> 1) & 1) ^ 1,
                                                                 &abort_flag, &g_bwd_status))) {
                    early = true;
                    break;
                }
                if (elect_one_sync()) {
                    const uint32_t dst = slot_addr(r, slot);
                    const uint32_t fb = bar(bars.full[r][slot]);
                    mbar_arrive_expect_tx(fb, C::kTileBytes);
                    if (r == kRingKv) {
                        // K in the value layout: D rows x 64 tokens per box
                        const int32_t vrow = static_cast<int32_t>(tile * D);
#pragma unroll
                        for (int c = 0; c < 2; ++c) tma_load_2d(dst + c * D * 128, &p.tmKv, fb, c * 64, vrow);
                    } else {
                        // K or V tile: 128 rows x 64 elements per box
                        const int32_t row = static_cast<int32_t>(tile * kTileElems);
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_2d(dst + c * kTileElems * C::kSpan, r == kRingK ? &p.tmK : &p.tmV, fb, c * (C::kSpan / 2),
                                        row);
                    }
                }
                __syncwarp();
                ++issued[r];
            }
        }
        // a skipped load (test hook) is left for the consumers' waits to find
        if (early && p.fault_skip_kv < 0 && lane == 0) bwd_raise(&abort_flag);
        // every load this warp issued lands before the CTA may exit (the last
        // load of each slot is the slot's latest phase)
        const volatile int never = 0;
        for (int r = 0; r < kRings; ++r)
            for (int j = (issued[r] > 2 ? issued[r] - 2 : 0); j < issued[r]; ++j)
                mbar_wait(bar(bars.full[r][j & 1]), (j >> 1) & 1, &never);
        mbar_wait(bar(bars.do_full), 0, &never);
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        const uint32_t tDQ = tmem + kColDQ, tS = tmem + kColS, tDP = tmem + kColDP;
        const uint32_t tDS = tmem + kColDS, tQ = tmem + kColQ;
        const uint64_t dDO = make_smem_desc(sDO, 16, 8 * C::kSpan, C::kSwizzle);
        auto wait_slot = [&](int r, int j) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar(bars.full[r][j & 1]), (j >> 1) & 1, &abort_flag,
                                                     &g_bwd_status));
        };
        // S(j) = Q K(j)^T: A (Q) from TMEM
        auto issue_s = [&](int j) -> bool {
            if (!wait_slot(kRingK, j)) return false;
            tc_fence_after();
            const uint64_t dK = make_smem_desc(slot_addr(kRingK, j & 1), 16, 8 * C::kSpan, C::kSwizzle);
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < C::kQKSteps; ++kk) {
                    // k-step kk: features [16 kk, 16 kk + 16) = 32 bytes of every token row
                    const int off = ((kk * 32) / C::kSpan) * (kTileElems * C::kSpan) + ((kk * 32) % C::kSpan);
                    mma_f16_ts(tS, tQ + kk * 8, dK + static_cast<uint64_t>(off >> 4), kIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(bars.s_full));
                mma_commit(bar(bars.empty[kRingK][j & 1]));
            }
            __syncwarp();
            return true;
        };
        // dP(j) = dO V(j)^T: both operands from shared memory
        auto issue_dp = [&](int j) -> bool {
            if (!wait_slot(kRingV, j)) return false;
            tc_fence_after();
            const uint64_t dV = make_smem_desc(slot_addr(kRingV, j & 1), 16, 8 * C::kSpan, C::kSwizzle);
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < C::kQKSteps; ++kk) {
                    const int off = ((kk * 32) / C::kSpan) * (kTileElems * C::kSpan) + ((kk * 32) % C::kSpan);
                    mma_f16_ss(tDP, dDO + static_cast<uint64_t>(off >> 4), dV + static_cast<uint64_t>(off >> 4),
                               kIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(bars.dp_full));
                mma_commit(bar(bars.empty[kRingV][j & 1]));
            }
            __syncwarp();
            return true;
        };
        // dQ += dS(j) K(j): A (dS) from TMEM, B = K in the value layout (K-major)
        auto issue_dq = [&](int j) -> bool {
            if (!wait_slot(kRingKv, j) ||
                !__all_sync(0xffffffffu, mbar_wait(bar(bars.ds_full), j & 1, &abort_flag, &g_bwd_status)))
                return false;
            tc_fence_after();
            const uint64_t dKv = make_smem_desc(slot_addr(kRingKv, j & 1), 16, 8 * 128, kSwizzle128B);
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < kDQSteps; ++kk) {
                    // k-step kk: key columns [16 kk, 16 kk + 16) = dS columns [8 kk, 8 kk + 8)
                    const int off = ((kk * 32) / 128) * (D * 128) + ((kk * 32) % 128);
                    mma_f16_ts(tDQ, tDS + kk * 8, dKv + static_cast<uint64_t>(off >> 4), C::kIdescDQ,
                               (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(bars.empty[kRingKv][j & 1]));
                mma_commit(bar(bars.ds_free));
                if (j == n_kv - 1) mma_commit(bar(bars.dq_final));
            }
            __syncwarp();
            return true;
        };
        // Issue order  S(0) dP(0) | S(1) dP(1) dQ(0) | S(2) dP(2) dQ(1) | ...:
        // S(j + 1) and dP(j + 1) wait only until the dS warps hold S(j) and
        // dP(j) in registers, so they run while dS(j) is formed and stored.
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.q_full), 0, &abort_flag, &g_bwd_status)) &&
                  __all_sync(0xffffffffu, mbar_wait(bar(bars.do_full), 0, &abort_flag, &g_bwd_status));
        if (ok && n_kv > 0) ok = issue_s(0) && issue_dp(0);
        for (int j = 0; ok && j < n_kv; ++j) {
            if (j + 1 < n_kv) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.s_free), j & 1, &abort_flag, &g_bwd_status)) &&
                     issue_s(j + 1) &&
                     __all_sync(0xffffffffu, mbar_wait(bar(bars.dp_free), j & 1, &abort_flag, &g_bwd_status)) &&
                     issue_dp(j + 1);
                if (!ok) break;
            }
            ok = issue_dq(j);
        }
        if (!ok) {
            if (elect_one_sync()) {
                bwd_raise(&abort_flag);
                mma_commit(bar(bars.drain));
            }
            __syncwarp();
            const volatile int never = 0;
            mbar_wait(bar(bars.drain), 0, &never);
        }
    } else {
        // ============================================================ dS / epilogue
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int64_t grow = q_tile_global * kTileElems + row;   // tiled row of this query

        int qpos[3], st[3];
        {
            const int ix = row & (p.tile[2] - 1);
            const int iy = (row >> p.tlog[2]) & (p.tile[1] - 1);
            const int it = row >> (p.tlog[1] + p.tlog[2]);
            qpos[0] = qc[0] * p.tile[0] + it;
            qpos[1] = qc[1] * p.tile[1] + iy;
            qpos[2] = qc[2] * p.tile[2] + ix;
        }
        const bool row_valid = qpos[0] < p.dims[0] && qpos[1] < p.dims[1] && qpos[2] < p.dims[2];
#pragma unroll
        for (int d = 0; d < 3; ++d) st[d] = window_start(qpos[d], p.dims[d], p.win[d], p.str[d], p.off[d]);

        // this half of the Q row -> TMEM (the A operand of S)
        {
            constexpr int W = C::kHalfWords;
            const uint4* qs = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.q) + grow * C::kRowBytes +
                                                             half * (C::kRowBytes / 2));
            uint32_t w[W];
#pragma unroll
            for (int i = 0; i < W / 4; ++i) {
                const uint4 v = __ldg(qs + i);
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
            }
            bwd_tmem_st<W>(tmem + kColQ + lane_addr + half * W, w);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.q_full));
        }
        // lse (natural log) and delta of this query; padding rows contribute nothing
        const float lse2 = row_valid ? p.lse[grow] * kBLog2e : 0.0f;
        const float delta = row_valid ? p.delta[grow] : 0.0f;
        const float scale_log2 = p.scale * kBLog2e;

        bool ok = true;
        int kc[3] = {box.k0[0], box.k0[1], box.k0[2]};
        for (int j = 0; j < n_kv && ok; ++j, bwd_odometer(kc, box)) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.s_full), j & 1, &abort_flag, &g_bwd_status));
            if (!ok) {
                bwd_raise(&abort_flag);
                break;
            }
            tc_fence_after();
            // this half row of S(j), then its columns go back to the MMA warp for S(j + 1)
            uint32_t rs[64];
            tmem_ld32(tmem + kColS + lane_addr + half * 64, *reinterpret_cast<uint32_t(*)[32]>(rs));
            tmem_ld32(tmem + kColS + lane_addr + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(rs + 32));
            bool full = true;
#pragma unroll
            for (int d = 0; d < 3; ++d) full = full && kc[d] >= box.full_lo[d] && kc[d] <= box.full_hi[d];
            // this row's window relative to the KV tile's origin, per dimension
            const int lo_t = st[0] - kc[0] * p.tile[0];
            const int lo_y = st[1] - kc[1] * p.tile[1];
            const int lo_x = st[2] - kc[2] * p.tile[2];
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.s_free));
            bwd_reg_fence(rs);
            // p = exp2(s scale log2(e) - lse log2(e)), 0 outside the window, as
            // bf16 pairs, while dP(j) is being computed.  Key column c of a
            // 32-column piece is inside the window iff bit c of the piece's mask
            // word is set (all set on a tile that lies in every window of the Q tile).
            const float2 sc2 = make_float2(scale_log2, scale_log2);
            const float2 nl2 = make_float2(-lse2, -lse2);
            uint32_t pp[32];
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                const uint32_t m = !row_valid ? 0u
                                   : full     ? 0xffffffffu
                                              : box_mask_word(half * 2 + pc, p.tlog[0], p.tlog[1], p.tlog[2], lo_t,
                                                              lo_y, lo_x, p.win[0], p.win[1], p.win[2]);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = 2 * i;
                    const float s0 = (m >> c) & 1u ? __uint_as_float(rs[pc * 32 + c]) : -INFINITY;
                    const float s1 = (m >> (c + 1)) & 1u ? __uint_as_float(rs[pc * 32 + c + 1]) : -INFINITY;
                    const float2 x = bwd_ffma2(make_float2(s0, s1), sc2, nl2);
                    __nv_bfloat162 h = __floats2bfloat162_rn(bwd_exp2(x.x), bwd_exp2(x.y));
                    pp[pc * 16 + i] = *reinterpret_cast<uint32_t*>(&h);
                }
            }
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.dp_full), j & 1, &abort_flag, &g_bwd_status));
            if (!ok) {
                bwd_raise(&abort_flag);
                break;
            }
            tc_fence_after();
            // this half row of dP(j) (both pieces in flight together); then its
            // columns go back to the MMA warp for dP(j + 1)
            uint32_t rp[64];
            tmem_ld32(tmem + kColDP + lane_addr + half * 64, *reinterpret_cast<uint32_t(*)[32]>(rp));
            tmem_ld32(tmem + kColDP + lane_addr + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(rp + 32));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.dp_free));
            bwd_reg_fence(rp);
            // dS goes to its own columns once dQ(j - 1) has read dS(j - 1)
            if (j > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.ds_free), (j - 1) & 1, &abort_flag, &g_bwd_status));
                if (!ok) {
                    bwd_raise(&abort_flag);
                    break;
                }
                tc_fence_after();
            }
            // dS = p (dP - delta) (bf16), two pieces of 32 key columns (16 TMEM columns each)
            const float2 nd2 = make_float2(-delta, -delta);
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = 2 * i;
                    const uint32_t hp = pp[pc * 16 + i];
                    const float2 pr = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hp));
                    const float2 dd = bwd_fadd2(make_float2(__uint_as_float(rp[pc * 32 + c]),
                                                            __uint_as_float(rp[pc * 32 + c + 1])), nd2);
                    const float2 ds2 = bwd_fmul2(pr, dd);
                    __nv_bfloat162 h = __floats2bfloat162_rn(ds2.x, ds2.y);
                    pk[i] = *reinterpret_cast<uint32_t*>(&h);
                }
                tmem_st16(tmem + kColDS + lane_addr + half * 32 + pc * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.ds_full));
        }

        // ------------------------------------------------------------ epilogue
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.dq_final), 0, &abort_flag, &g_bwd_status));
            if (!ok) bwd_raise(&abort_flag);
        }
        if (ok) {
            tc_fence_after();
            uint8_t* dst_row = static_cast<uint8_t*>(p.dq) + grow * C::kRowBytes + half * (C::kRowBytes / 2);
            // this half of the dQ row, in pieces of up to 32 columns
            constexpr int P = C::kHalfCols < 32 ? C::kHalfCols : 32;
#pragma unroll
            for (int pc = 0; pc < C::kHalfCols / P; ++pc)
                bwd_store_cols<P>(tmem + kColDQ + lane_addr + half * C::kHalfCols + pc * P, true, p.scale,
                                  dst_row + pc * P * 2);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kBTmemCols);
    }
}

// ---------------------------------------------------------------------------- dK, dV
//
// One CTA per 128-key tile j of one (batch, head).  It visits the Q tiles
// whose windows reach tile j: per dimension the KV box [k0(qt), k1(qt)] of a Q
// tile moves monotonically with qt, so those Q tiles form an interval per
// dimension (the inverse box).  Per Q tile i:
//   S^T  = K_j Q_i^T,  dP^T = V_j dO_i^T            (A, B from shared memory)
//   P^T  = exp(S^T - lse_i),  dS^T = P^T (dP^T - delta_i)   (per key row)
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i               (A from TMEM, B MN-major)
// TMEM: dV [0, d), dK [128, 128 + d), S^T [256, 384), dP^T [384, 512) for
// head_dim d; P^T and dS^T of each 32-query piece go over that piece's own
// dP^T columns (16 + 16), so S^T is free once it is in registers and S^T of
// the next Q tile is computed while the key-row warps work; they form P^T
// from S^T while dP^T is computed.  Q_i and dO_i are read as tiled tiles
// in both roles: K-major for S^T and dP^T, MN-major (token rows, 16 per
// k-step) for dV and dK.  The element mask comes from, per dimension, the
// interval of query positions whose window holds this thread's key (one
// 32-bit word per 32 query columns, box_mask_word); a key row whose interval
// covers the whole Q tile needs no mask.

constexpr uint32_t kColDV = 0;
constexpr uint32_t kColDK = 128;
constexpr uint32_t kColST = 256;
constexpr uint32_t kColDPT = 384;

struct KVBars {
    uint64_t kv_full;             // K_j and V_j landed
    uint64_t full[kBStages];      // Q_i, dO_i, lse_i, delta_i landed
    uint64_t empty[kBStages];     // the four MMAs of step i are done
    uint64_t s_full;              // S^T of step i is in TMEM (one phase per step)
    uint64_t s_free;              // the key-row warps hold S^T(i) in registers (8 warps)
    uint64_t dp_full;             // dP^T of step i is in TMEM
    uint64_t p_full;              // P^T and dS^T of step i are in TMEM, over dP^T (8 warps)
    uint64_t final_;              // the last dV / dK products are done
    uint64_t drain;
};

template <int D>
__global__ void __launch_bounds__(kBThreads, 1) gna_bwd_dkdv_kernel(const __grid_constant__ BwdKVParams p)
{
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ KVBars bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // ---------------------------------------------------------------- geometry
    const int64_t kv_tile_global = blockIdx.x;                // (b*heads + h)*tiles_per_head + kt
    const int kt_id = static_cast<int>(kv_tile_global % p.tiles_per_head);
    const int64_t plane_base = kv_tile_global - kt_id;        // first tile of this (b, head) plane
    int kc[3];
    kc[2] = kt_id % p.nt[2];
    kc[1] = (kt_id / p.nt[2]) % p.nt[1];
    kc[0] = kt_id / (p.nt[2] * p.nt[1]);
    BwdBox qbox;                                              // inverse box: Q tiles reaching tile kc
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        int lo = -1, hi = -2;
        for (int qt = 0; qt < p.nt[d]; ++qt) {
            const DimRange r = dim_range(qt, p.tile[d], p.tile[d], p.dims[d], p.win[d], p.str[d], p.off[d]);
            if (r.k0 <= kc[d] && kc[d] <= r.k1) {
                if (lo < 0) lo = qt;
                hi = qt;
            }
        }
        qbox.k0[d] = lo < 0 ? 0 : lo;
        qbox.cnt[d] = lo < 0 ? 0 : hi - lo + 1;
    }
    const int n_q = qbox.cnt[0] * qbox.cnt[1] * qbox.cnt[2];

    auto bar = [](uint64_t& b) { return smem_u32(&b); };
    const uint32_t sK = smem_u32(smem);
    const uint32_t sV = sK + C::kTileBytes;
    const uint32_t sStage = sK + 2 * C::kTileBytes;
    const float* stage_f = reinterpret_cast<const float*>(smem + 2 * C::kTileBytes);   // float view of the stages

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(bars.kv_full), 1);
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(bar(bars.full[s]), 1);
            mbar_init(bar(bars.empty[s]), 1);
        }
        mbar_init(bar(bars.s_full), 1);
        mbar_init(bar(bars.s_free), kBSoftmaxWarps);
        mbar_init(bar(bars.dp_full), 1);
        mbar_init(bar(bars.p_full), kBSoftmaxWarps);
        mbar_init(bar(bars.final_), 1);
        mbar_init(bar(bars.drain), 1);
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base_sh), kBTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0) {
        // ============================================================ TMA producer
        if (elect_one_sync()) {
            prefetch_tensormap(&p.tmQ);
            prefetch_tensormap(&p.tmDO);
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmV);
        }
        if (n_q > 0 && elect_one_sync()) {
            const int32_t row = static_cast<int32_t>(kv_tile_global * kTileElems);
            mbar_arrive_expect_tx(bar(bars.kv_full), 2 * C::kTileBytes);
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
                tma_load_2d(sK + c * kTileElems * C::kSpan, &p.tmK, bar(bars.kv_full), c * (C::kSpan / 2), row);
                tma_load_2d(sV + c * kTileElems * C::kSpan, &p.tmV, bar(bars.kv_full), c * (C::kSpan / 2), row);
            }
        }
        __syncwarp();
        int issued = 0;
        bool early = false;
        int qc[3] = {qbox.k0[0], qbox.k0[1], qbox.k0[2]};
        for (int i = 0; i < n_q; ++i, bwd_odometer(qc, qbox)) {
            const int s = i % kBStages;
            const int64_t qtile = plane_base + (qc[0] * p.nt[1] + qc[1]) * p.nt[2] + qc[2];
            if (i >= kBStages &&
                !__all_sync(0xffffffffu, mbar_wait(bar(bars.empty[s]), ((i / kBStages) & 1) ^ 1, &abort_flag, &g_bwd_status))) {
                early = true;
                break;
            }
            if (elect_one_sync()) {
                const uint32_t st = sStage + s * C::kKVStageBytes;
                const int32_t row = static_cast<int32_t>(qtile * kTileElems);
                mbar_arrive_expect_tx(bar(bars.full[s]), 2 * C::kTileBytes + 2 * kTileElems * 4);
#pragma unroll
                for (int c = 0; c < C::kChunks; ++c) {
                    tma_load_2d(st + c * kTileElems * C::kSpan, &p.tmQ, bar(bars.full[s]), c * (C::kSpan / 2), row);
                    tma_load_2d(st + C::kTileBytes + c * kTileElems * C::kSpan, &p.tmDO, bar(bars.full[s]),
                                c * (C::kSpan / 2), row);
                }
                bulk_load_g2s(st + 2 * C::kTileBytes, p.lse + qtile * kTileElems, kTileElems * 4, bar(bars.full[s]));
                bulk_load_g2s(st + 2 * C::kTileBytes + kTileElems * 4, p.delta + qtile * kTileElems, kTileElems * 4,
                              bar(bars.full[s]));
            }
            __syncwarp();
            ++issued;
        }
        if (early) {
            if (lane == 0) bwd_raise(&abort_flag);
            const volatile int never = 0;
            for (int i = (issued > kBStages ? issued - kBStages : 0); i < issued; ++i)
                mbar_wait(bar(bars.full[i % kBStages]), (i / kBStages) & 1, &never);
            mbar_wait(bar(bars.kv_full), 0, &never);
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        const uint32_t tDV = tmem + kColDV, tDK = tmem + kColDK, tST = tmem + kColST, tDPT = tmem + kColDPT;
        const uint64_t dKj = make_smem_desc(sK, 16, 8 * C::kSpan, C::kSwizzle);
        const uint64_t dVj = make_smem_desc(sV, 16, 8 * C::kSpan, C::kSwizzle);
        auto stage_of = [&](int i) { return sStage + (i % kBStages) * C::kKVStageBytes; };
        // S^T(i) = K_j Q_i^T (both operands from shared memory)
        auto issue_s = [&](int i) -> bool {
            const int s = i % kBStages;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.full[s]), (i / kBStages) & 1, &abort_flag, &g_bwd_status)))
                return false;
            tc_fence_after();
            const uint64_t dQk = make_smem_desc(stage_of(i), 16, 8 * C::kSpan, C::kSwizzle);   // K-major
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < C::kQKSteps; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(
                        (((kk * 32) / C::kSpan) * (kTileElems * C::kSpan) + ((kk * 32) % C::kSpan)) >> 4);
                    mma_f16_ss(tST, dKj + off, dQk + off, kIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(bars.s_full));
            }
            __syncwarp();
            return true;
        };
        // dP^T(i) = V_j dO_i^T (step i's stage has landed: issue_s(i) waited for it)
        auto issue_dp = [&](int i) {
            const uint64_t dDOk = make_smem_desc(stage_of(i) + C::kTileBytes, 16, 8 * C::kSpan, C::kSwizzle);
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < C::kQKSteps; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(
                        (((kk * 32) / C::kSpan) * (kTileElems * C::kSpan) + ((kk * 32) % C::kSpan)) >> 4);
                    mma_f16_ss(tDPT, dVj + off, dDOk + off, kIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(bars.dp_full));
            }
            __syncwarp();
        };
        // Issue order  S^T(0) dP^T(0) | S^T(1) dV(0) dK(0) dP^T(1) | ...: S^T(i + 1)
        // runs while the key-row warps work on step i (they release the S^T
        // columns once S^T(i) is in their registers); P^T(i) and dS^T(i) go over
        // dP^T(i)'s columns, which dP^T(i + 1) overwrites after dV(i) and dK(i)
        // have read them: the tensor core executes one thread's MMAs in issue
        // order.
        bool ok = n_q == 0 || __all_sync(0xffffffffu, mbar_wait(bar(bars.kv_full), 0, &abort_flag, &g_bwd_status));
        if (ok && n_q > 0) {
            ok = issue_s(0);
            if (ok) issue_dp(0);
        }
        for (int i = 0; ok && i < n_q; ++i) {
            const int s = i % kBStages;
            if (i + 1 < n_q) {
                if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.s_free), i & 1, &abort_flag, &g_bwd_status)) ||
                    !issue_s(i + 1)) {
                    ok = false;
                    break;
                }
            }
            if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.p_full), i & 1, &abort_flag, &g_bwd_status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t st = stage_of(i);
            // MN-major: feature spans kTileElems rows apart, 8-token groups 8 spans apart
            const uint64_t dQm = make_smem_desc(st, kTileElems * C::kSpan, 8 * C::kSpan, C::kSwizzle);
            const uint64_t dDOm = make_smem_desc(st + C::kTileBytes, kTileElems * C::kSpan, 8 * C::kSpan, C::kSwizzle);
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < kDQSteps; ++kk) {
                    // k-step kk: query columns [16 kk, 16 kk + 16) = token rows of Q_i / dO_i.
                    // Query piece c (32 columns) keeps P^T at dP^T columns [32 c, 32 c + 16)
                    // and dS^T at [32 c + 16, 32 c + 32)
                    const uint32_t a = (kk >> 1) * 32 + (kk & 1) * 8;
                    const uint64_t off = static_cast<uint64_t>((kk * 16 * C::kSpan) >> 4);
                    const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                    mma_f16_ts(tDV, tDPT + a, dDOm + off, C::kIdescMN, acc);
                    mma_f16_ts(tDK, tDPT + a + 16, dQm + off, C::kIdescMN, acc);
                }
                mma_commit(bar(bars.empty[s]));
                if (i == n_q - 1) mma_commit(bar(bars.final_));
            }
            __syncwarp();
            if (i + 1 < n_q) issue_dp(i + 1);
        }
        if (!ok) {
            if (elect_one_sync()) {
                bwd_raise(&abort_flag);
                mma_commit(bar(bars.drain));
            }
            __syncwarp();
            const volatile int never = 0;
            mbar_wait(bar(bars.drain), 0, &never);
        }
    } else {
        // ============================================================ P^T, dS^T / epilogue
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;                   // key row of this thread
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const int64_t grow = kv_tile_global * kTileElems + row;

        // this key's position and, per dimension, the query positions whose
        // window holds it (an interval: window starts grow with the position)
        int kpos[3];
        kpos[2] = kc[2] * p.tile[2] + (row & (p.tile[2] - 1));
        kpos[1] = kc[1] * p.tile[1] + ((row >> p.tlog[2]) & (p.tile[1] - 1));
        kpos[0] = kc[0] * p.tile[0] + (row >> (p.tlog[1] + p.tlog[2]));
        int qlo[3], qhi[3];
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            qlo[d] = 1;
            qhi[d] = 0;                                        // empty unless found
            if (kpos[d] < p.dims[d]) {
                for (int q = 0; q < p.dims[d]; ++q) {
                    const int a = window_start(q, p.dims[d], p.win[d], p.str[d], p.off[d]);
                    if (a <= kpos[d] && kpos[d] < a + p.win[d]) {
                        if (qlo[d] > qhi[d]) qlo[d] = q;
                        qhi[d] = q;
                    }
                }
            }
        }
        const float scale_log2 = p.scale * kBLog2e;

        bool ok = true;
        int qc[3] = {qbox.k0[0], qbox.k0[1], qbox.k0[2]};
        for (int i = 0; i < n_q && ok; ++i, bwd_odometer(qc, qbox)) {
            const int s = i % kBStages;
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.full[s]), (i / kBStages) & 1, &abort_flag, &g_bwd_status)) &&
                 __all_sync(0xffffffffu, mbar_wait(bar(bars.s_full), i & 1, &abort_flag, &g_bwd_status));
            if (!ok) {
                bwd_raise(&abort_flag);
                break;
            }
            tc_fence_after();
            // this half row of S^T(i); then its columns go back for S^T(i + 1)
            uint32_t rs[64];
            tmem_ld32(tmem + kColST + lane_addr + half * 64, *reinterpret_cast<uint32_t(*)[32]>(rs));
            tmem_ld32(tmem + kColST + lane_addr + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(rs + 32));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.s_free));
            bwd_reg_fence(rs);
            // the queries whose window holds this key, in the Q tile's own
            // coordinates: [lo_d, lo_d + len_d) per dimension
            int lo[3], len[3];
            bool full = true;
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                lo[d] = qlo[d] - qc[d] * p.tile[d];
                len[d] = qhi[d] - qlo[d] + 1;                      // <= 0: empty
                full = full && len[d] > 0 && lo[d] <= 0 && lo[d] + len[d] >= p.tile[d];
            }
            const float* lse_s = stage_f + s * (C::kKVStageBytes / 4) + 2 * (C::kTileBytes / 4);
            const float* delta_s = lse_s + kTileElems;
            const float2 sc2 = make_float2(scale_log2, scale_log2);
            const float2 nlog2e = make_float2(-kBLog2e, -kBLog2e);
            // P^T of this half row (bf16 pairs) while dP^T(i) is being computed:
            // p = exp2(s scale log2(e) - lse log2(e)), 0 where the query does not
            // reach the key (selected after the exponential: a padding query's
            // lse is -inf, so its exponent may be anything there)
            uint32_t pkp[32];
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                // query column c of the piece reaches this key iff bit c is set
                const uint32_t m = full ? 0xffffffffu
                                        : box_mask_word(half * 2 + pc, p.tlog[0], p.tlog[1], p.tlog[2], lo[0], lo[1],
                                                        lo[2], len[0], len[1], len[2]);
                const int col0 = half * 64 + pc * 32;
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                    const float4 L4 = *reinterpret_cast<const float4*>(lse_s + col0 + 4 * g4);
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int k = 4 * g4 + e;                      // column of the piece
                        const float2 lse2 = e == 0 ? make_float2(L4.x, L4.y) : make_float2(L4.z, L4.w);
                        const float2 x = bwd_ffma2(make_float2(__uint_as_float(rs[pc * 32 + k]),
                                                               __uint_as_float(rs[pc * 32 + k + 1])),
                                                   sc2, bwd_fmul2(lse2, nlog2e));
                        const float2 pr = make_float2((m >> k) & 1u ? bwd_exp2(x.x) : 0.0f,
                                                      (m >> (k + 1)) & 1u ? bwd_exp2(x.y) : 0.0f);
                        __nv_bfloat162 hp = __floats2bfloat162_rn(pr.x, pr.y);
                        pkp[pc * 16 + k / 2] = *reinterpret_cast<uint32_t*>(&hp);
                    }
                }
            }
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.dp_full), i & 1, &abort_flag, &g_bwd_status));
            if (!ok) {
                bwd_raise(&abort_flag);
                break;
            }
            tc_fence_after();
            // dP^T(i) in two pieces of 32 query columns; P^T and dS^T of a piece
            // (16 columns each) go over the piece's own dP^T columns once read.
            // dS = p (dP - delta) with p as the bf16 value that dV's product reads.
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                const int col0 = half * 64 + pc * 32;
                uint32_t rp[32];
                tmem_ld32(tmem + kColDPT + lane_addr + col0, rp);
                tmem_wait_ld();
                bwd_reg_fence(rp);
                uint32_t pkd[16];
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {
                    const float4 D4 = *reinterpret_cast<const float4*>(delta_s + col0 + 4 * g4);
#pragma unroll
                    for (int e = 0; e < 4; e += 2) {
                        const int k = 4 * g4 + e;
                        const float2 dl2 = e == 0 ? make_float2(D4.x, D4.y) : make_float2(D4.z, D4.w);
                        const uint32_t hp = pkp[pc * 16 + k / 2];
                        const float2 pr = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hp));
                        const float2 dd = bwd_fadd2(make_float2(__uint_as_float(rp[k]), __uint_as_float(rp[k + 1])),
                                                    make_float2(-dl2.x, -dl2.y));
                        const float2 ds2 = bwd_fmul2(pr, dd);
                        __nv_bfloat162 hd = __floats2bfloat162_rn(ds2.x, ds2.y);
                        pkd[k / 2] = *reinterpret_cast<uint32_t*>(&hd);
                    }
                }
                tmem_st16(tmem + kColDPT + lane_addr + col0, *reinterpret_cast<const uint32_t(*)[16]>(pkp + pc * 16));
                tmem_st16(tmem + kColDPT + lane_addr + col0 + 16, pkd);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.p_full));
        }

        // ------------------------------------------------------------ epilogue
        if (ok && n_q > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.final_), 0, &abort_flag, &g_bwd_status));
            if (!ok) bwd_raise(&abort_flag);
        }
        if (ok) {
            tc_fence_after();
#pragma unroll
            for (int which = 0; which < 2; ++which) {              // 0: dv, 1: dk (times scale)
                uint8_t* dst_row = static_cast<uint8_t*>(which == 0 ? p.dv : p.dk) + grow * C::kRowBytes +
                                   half * (C::kRowBytes / 2);
                const float mul = which == 0 ? 1.0f : p.scale;
                // no query reaches this key tile when n_q == 0: zeros
                constexpr int P = C::kHalfCols < 32 ? C::kHalfCols : 32;
#pragma unroll
                for (int pc = 0; pc < C::kHalfCols / P; ++pc)
                    bwd_store_cols<P>(tmem + (which == 0 ? kColDV : kColDK) + lane_addr + half * C::kHalfCols + pc * P,
                                      n_q > 0, mul, dst_row + pc * P * 2);
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kBTmemCols);
    }
}

// delta_i = <dout_i, out_i> (fp32 accumulation of the bf16 rows), one warp per
// tiled row: 128 elements, 4 per lane.
template <int D>
__global__ void gna_bwd_delta_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                                     float* __restrict__ delta, int64_t rows)
{
    const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
    if (r >= rows) return;
    const int lane = threadIdx.x % 32;
    float acc;
    if constexpr (D == 128) {
        const uint2 o = *reinterpret_cast<const uint2*>(out + r * D + lane * 4);
        const uint2 g = *reinterpret_cast<const uint2*>(dout + r * D + lane * 4);
        const float2 o0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.x));
        const float2 o1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.y));
        const float2 g0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g.x));
        const float2 g1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g.y));
        acc = o0.x * g0.x + o0.y * g0.y + o1.x * g1.x + o1.y * g1.y;
    } else if constexpr (D == 64) {
        const float2 o0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(out + r * D + lane * 2));
        const float2 g0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(dout + r * D + lane * 2));
        acc = o0.x * g0.x + o0.y * g0.y;
    } else {
        static_assert(D == 32, "head_dim 32, 64 or 128");
        acc = __bfloat162float(out[r * D + lane]) * __bfloat162float(dout[r * D + lane]);
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) delta[r] = acc;
}

}  // namespace

namespace {

template <int D>
cudaError_t launch_dq(const BwdParams& p, int64_t num_q_tiles, cudaStream_t stream)
{
    using C = BwdCfg<D>;
    // the opt-in limit of 227 KB per block holds dynamic and static shared memory
    static_assert(C::kDQSmemAlloc <= 232448 - 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(gna_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kDQSmemAlloc);
    if (e != cudaSuccess) return e;
    gna_bwd_dq_kernel<D><<<dim3(static_cast<unsigned>(num_q_tiles)), kBThreads, C::kDQSmemAlloc, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_dkdv(const BwdKVParams& p, int64_t num_kv_tiles, cudaStream_t stream)
{
    using C = BwdCfg<D>;
    static_assert(C::kKVSmemAlloc <= 232448 - 4096, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(gna_bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kKVSmemAlloc);
    if (e != cudaSuccess) return e;
    gna_bwd_dkdv_kernel<D><<<dim3(static_cast<unsigned>(num_kv_tiles)), kBThreads, C::kKVSmemAlloc, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_dq(const BwdParams& p, int head_dim, int64_t num_q_tiles, cudaStream_t stream)
{
    if (num_q_tiles <= 0) return cudaSuccess;
    if (head_dim == 128) return launch_dq<128>(p, num_q_tiles, stream);
    if (head_dim == 64) return launch_dq<64>(p, num_q_tiles, stream);
    if (head_dim == 32) return launch_dq<32>(p, num_q_tiles, stream);
    return cudaErrorNotSupported;
}

cudaError_t launch_backward_dkdv(const BwdKVParams& p, int head_dim, int64_t num_kv_tiles, cudaStream_t stream)
{
    if (num_kv_tiles <= 0) return cudaSuccess;
    if (head_dim == 128) return launch_dkdv<128>(p, num_kv_tiles, stream);
    if (head_dim == 64) return launch_dkdv<64>(p, num_kv_tiles, stream);
    if (head_dim == 32) return launch_dkdv<32>(p, num_kv_tiles, stream);
    return cudaErrorNotSupported;
}

cudaError_t launch_backward_delta(const void* out, const void* dout, float* delta, int64_t rows, int head_dim,
                                  cudaStream_t stream)
{
    if (rows <= 0) return cudaSuccess;
    const int warps = 8;
    const int64_t blocks = (rows + warps - 1) / warps;
    const auto* o = static_cast<const __nv_bfloat16*>(out);
    const auto* g = static_cast<const __nv_bfloat16*>(dout);
    if (head_dim == 128)
        gna_bwd_delta_kernel<128><<<dim3(static_cast<unsigned>(blocks)), warps * 32, 0, stream>>>(o, g, delta, rows);
    else if (head_dim == 64)
        gna_bwd_delta_kernel<64><<<dim3(static_cast<unsigned>(blocks)), warps * 32, 0, stream>>>(o, g, delta, rows);
    else if (head_dim == 32)
        gna_bwd_delta_kernel<32><<<dim3(static_cast<unsigned>(blocks)), warps * 32, 0, stream>>>(o, g, delta, rows);
    else
        return cudaErrorNotSupported;
    return cudaGetLastError();
}

cudaError_t read_and_clear_bwd_status(int* status, cudaStream_t stream)
{
    int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_bwd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    if (*status != 0) {
        e = cudaMemcpyToSymbolAsync(g_bwd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return e;
        e = cudaStreamSynchronize(stream);
    }
    return e;
}

}  // namespace gna
