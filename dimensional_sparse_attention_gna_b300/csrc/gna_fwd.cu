// Fused Generalized Neighborhood Attention forward kernel for sm_103a.
//
// GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践"):
//  §1.1  Q and KV are cut into fixed-size multi-dimensional tiles; the stride
//        decides which KV tiles each Q tile must visit; a producer warp maps
//        the loop index to multi-dimensional KV tile coordinates and loads the
//        tiles with TMA.
//  §2.1  the element mask is applied only to KV tiles that are not entirely
//        inside the attention window; loads overlap compute.
//  §1.2  Q-tile and KV-tile sizes are decoupled.
// Video tutorial page ("视频生成推理提速:稀疏注意力组合配置教程"), §3.3: the
// softmax is accumulated block by block and the n x n matrix never exists.
//
// One CTA owns one 128-query tile of one (batch, head) and walks the box of
// KV tiles its windows touch.  Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then K and V through NS-stage rings
//   warp 1      TMEM allocator and tcgen05.mma issuer (one elected lane)
//   warps 2..5  softmax + correction + epilogue; thread = one query row,
//               TMEM lane quarter = warp % 4
// TMEM (512 columns): O at [0, 128), S double buffer at [128, 256) and
// [256, 384).  P overwrites the front of its S buffer (bf16: 64 columns,
// e4m3: 32 columns) and feeds the P*V MMA straight from TMEM.
// MMA issue order  QK(0) QK(1) PV(0) QK(2) PV(1) ...  keeps the tensor core on
// the next S while the softmax warps work on the current one.
//
// The running row maximum is updated lazily: the output accumulator is only
// rescaled when the maximum grows by more than kTau (log2 units); between
// rescales P may exceed 1 by up to 2^kTau, which the final O / l cancels
// exactly.  For e4m3 P the exponent is shifted by kP8Shift so that P uses the
// normal range of e4m3 (values up to 2^(kP8Shift + kTau) <= 448).
//
// Every mbarrier wait is bounded (see ptx.cuh); a role that gives up raises
// the CTA abort flag and the device status word, the other roles drop out of
// their loops, in-flight TMA loads and MMAs are drained (again bounded), TMEM
// is freed and the CTA exits.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "gna_geometry.cuh"
#include "gna_internal.h"
#include "ptx.cuh"

namespace gna {

__device__ int g_device_status = 0;

namespace {

constexpr int kThreads = 192;
constexpr int kSoftmaxWarp0 = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS0 = 128;
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
    static constexpr int kRowBytes = (D * ESZ) >= 128 ? 128 : D * ESZ;      // swizzle span
    static constexpr int kChunks = (D * ESZ) / kRowBytes;                    // TMA boxes per tile
    static constexpr int kChunkElems = kRowBytes / ESZ;
    static constexpr uint32_t kSwizzle = kRowBytes == 128 ? kSwizzle128B : kRowBytes == 64 ? kSwizzle64B : kSwizzle32B;
    static constexpr int kTileBytes = kTileElems * D * ESZ;
    static constexpr int kSmemQ = 0;
    static constexpr int kSmemK = kTileBytes;
    static constexpr int kSmemV = kTileBytes * (1 + NS);
    static constexpr int kSmemData = kTileBytes * (1 + 2 * NS);
    // at least ~116 KB so that only one CTA (which owns all 512 TMEM columns)
    // is resident per SM
    static constexpr int kSmemAlloc = (kSmemData + 1024) > 118784 ? (kSmemData + 1024) : 118784;
    static constexpr int kKPerInstr = 32 / ESZ;                              // MMA K extent (elements)
    static constexpr int kQKSteps = D / kKPerInstr;
    static constexpr int kPVSteps = kTileElems / kKPerInstr;
    static constexpr uint32_t kIdescQK = make_idesc(128, 128, Precision<ESZ>::fmt, false);
    static constexpr uint32_t kIdescPV = make_idesc(128, D, Precision<ESZ>::fmt, true);
    static constexpr int kPCols = kTileElems * ESZ / 4;                      // TMEM columns of P
};

struct Barriers {
    uint64_t q_full;
    uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
    uint64_t s_full[2], p_full[2];
    uint64_t o_done;
    uint64_t drain;
};

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void raise_status(volatile int* abort_flag)
{
    *abort_flag = 1;
    atomicExch(&g_device_status, 4 /* GNA_ERR_TIMEOUT */);
}

// KV tile visited at loop index j (row-major over the box).
struct KvBox {
    int k0[3], cnt[3];
    DimRange r[3];
    __device__ __forceinline__ void coords(int j, int (&kc)[3]) const
    {
        kc[2] = k0[2] + j % cnt[2];
        kc[1] = k0[1] + (j / cnt[2]) % cnt[1];
        kc[0] = k0[0] + j / (cnt[2] * cnt[1]);
    }
};

__device__ __forceinline__ uint32_t range_bits32(int lo, int hi)
{
    // bits [lo, hi) clipped to [0, 32)
    lo = lo < 0 ? 0 : lo;
    hi = hi > 32 ? 32 : hi;
    if (hi <= lo) return 0u;
    const uint32_t width_mask = (hi - lo) >= 32 ? 0xffffffffu : ((1u << (hi - lo)) - 1u);
    return width_mask << lo;
}

// 128-bit column mask of one query row against KV tile kc: bit c set iff the
// key at tile element c lies in the row's window in every dimension.
__device__ __forceinline__ void build_row_mask(const FwdParams& p, const int (&kc)[3], const int (&st)[3],
                                               uint32_t (&m)[4])
{
    const int lo_t = st[0] - kc[0] * p.tile[0];
    const int lo_y = st[1] - kc[1] * p.tile[1];
    const int lo_x = st[2] - kc[2] * p.tile[2];
    const int tw = p.tile[2];
    const int lw = p.tlog[2];
    const int lh = p.tlog[1];
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        uint32_t bits = 0;
        if (tw >= 32) {
            const int c0 = wi * 32;
            const int g = c0 >> lw;
            const int cy = g & ((1 << lh) - 1);
            const int ct = g >> lh;
            const int bx = c0 & (tw - 1);
            const bool ok = static_cast<unsigned>(ct - lo_t) < static_cast<unsigned>(p.win[0]) &&
                            static_cast<unsigned>(cy - lo_y) < static_cast<unsigned>(p.win[1]);
            bits = ok ? range_bits32(lo_x - bx, lo_x - bx + p.win[2]) : 0u;
        } else {
            const uint32_t mx = range_bits32(lo_x, lo_x + p.win[2]) & ((1u << tw) - 1u);
            const int groups = 32 >> lw;
            for (int gi = 0; gi < groups; ++gi) {
                const int g = (wi * 32 >> lw) + gi;
                const int cy = g & ((1 << lh) - 1);
                const int ct = g >> lh;
                const bool ok = static_cast<unsigned>(ct - lo_t) < static_cast<unsigned>(p.win[0]) &&
                                static_cast<unsigned>(cy - lo_y) < static_cast<unsigned>(p.win[1]);
                if (ok) bits |= mx << (gi * tw);
            }
        }
        m[wi] = bits;
    }
}

template <int ESZ>
__device__ __forceinline__ void pack_p(const float (&x)[32], uint32_t* out);

template <>
__device__ __forceinline__ void pack_p<2>(const float (&x)[32], uint32_t* out)
{
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        out[i] = *reinterpret_cast<uint32_t*>(&h);
    }
}

template <>
__device__ __forceinline__ void pack_p<1>(const float (&x)[32], uint32_t* out)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * i], x[4 * i + 1]), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(x[4 * i + 2], x[4 * i + 3]), __NV_SATFINITE, __NV_E4M3);
        out[i] = (lo & 0xffffu) | (hi << 16);
    }
}

template <int D, int ESZ, int NS>
__global__ void __launch_bounds__(kThreads, 1) gna_fwd_kernel(const __grid_constant__ FwdParams p)
{
    using C = Cfg<D, ESZ, NS>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ Barriers bars;
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    // ---------------------------------------------------------------- tile geometry (all threads)
    const int64_t q_tile_global = blockIdx.x;                 // (b*heads + h)*tiles_per_head + qt
    const int qt_id = static_cast<int>(q_tile_global % p.tiles_per_head);
    const int64_t bh = q_tile_global / p.tiles_per_head;
    int qc[3];
    qc[2] = qt_id % p.nt[2];
    qc[1] = (qt_id / p.nt[2]) % p.nt[1];
    qc[0] = qt_id / (p.nt[2] * p.nt[1]);
    KvBox box;
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        box.r[d] = dim_range(qc[d], p.tile[d], p.dims[d], p.win[d], p.str[d], p.off[d]);
        box.k0[d] = box.r[d].k0;
        box.cnt[d] = box.r[d].k1 - box.r[d].k0 + 1;
    }
    const int n_kv = box.cnt[0] * box.cnt[1] * box.cnt[2];
    const int64_t kv_row_base = bh * p.tiles_per_head * kTileElems;

    const uint32_t sQ = smem_u32(smem + C::kSmemQ);
    const uint32_t sK = smem_u32(smem + C::kSmemK);
    const uint32_t sV = smem_u32(smem + C::kSmemV);
    auto bar = [](uint64_t& b) { return smem_u32(&b); };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(bars.q_full), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(bars.k_full[s]), 1);
            mbar_init(bar(bars.k_empty[s]), 1);
            mbar_init(bar(bars.v_full[s]), 1);
            mbar_init(bar(bars.v_empty[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(bars.s_full[s]), 1);
            mbar_init(bar(bars.p_full[s]), 4);
        }
        mbar_init(bar(bars.o_done), 1);
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

    if (warp == 0) {
        // ============================================================ TMA producer
        if (lane == 0) {
            prefetch_tensormap(&p.tmQ);
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmV);
            const int32_t q_row = static_cast<int32_t>(q_tile_global * kTileElems);
            mbar_arrive_expect_tx(bar(bars.q_full), C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d(sQ + c * kTileElems * C::kRowBytes, &p.tmQ, bar(bars.q_full), c * C::kChunkElems, q_row);
            int k_issued = 0, v_issued = 0;          // KV tiles whose K / V loads were issued
            bool early = false;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % NS;
                const uint32_t ph = ((j / NS) & 1) ^ 1;
                int kc[3];
                box.coords(j, kc);
                const int tile_id = (kc[0] * p.nt[1] + kc[1]) * p.nt[2] + kc[2];
                const int32_t row = static_cast<int32_t>(kv_row_base + static_cast<int64_t>(tile_id) * kTileElems);
                if (j >= NS && !mbar_wait(bar(bars.k_empty[s]), ph, &abort_flag)) { early = true; break; }
                if (j == p.fault_skip_kv) { early = true; break; }   // test hook: consumers wait in vain
                mbar_arrive_expect_tx(bar(bars.k_full[s]), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sK + s * C::kTileBytes + c * kTileElems * C::kRowBytes, &p.tmK, bar(bars.k_full[s]),
                                c * C::kChunkElems, row);
                ++k_issued;
                if (j >= NS && !mbar_wait(bar(bars.v_empty[s]), ph, &abort_flag)) { early = true; break; }
                mbar_arrive_expect_tx(bar(bars.v_full[s]), C::kTileBytes);
                for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sV + s * C::kTileBytes + c * kTileElems * C::kRowBytes, &p.tmV, bar(bars.v_full[s]),
                                c * C::kChunkElems, row);
                ++v_issued;
            }
            if (early) {
                if (p.fault_skip_kv < 0) raise_status(&abort_flag);
                // Drain: wait (bounded, ignoring the abort flag) for the loads
                // still in flight so that no TMA write lands after the CTA exits.
                const volatile int never = 0;
                for (int j = (k_issued > NS ? k_issued - NS : 0); j < k_issued; ++j)
                    mbar_wait(bar(bars.k_full[j % NS]), (j / NS) & 1, &never);
                for (int j = (v_issued > NS ? v_issued - NS : 0); j < v_issued; ++j)
                    mbar_wait(bar(bars.v_full[j % NS]), (j / NS) & 1, &never);
                mbar_wait(bar(bars.q_full), 0, &never);
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            const uint32_t tS[2] = {tmem + kColS0, tmem + kColS0 + 128};
            const uint32_t tO = tmem + kColO;
            auto issue_pv = [&](int i) -> bool {
                const int s = i % NS;
                if (!mbar_wait(bar(bars.v_full[s]), (i / NS) & 1, &abort_flag)) return false;
                if (!mbar_wait(bar(bars.p_full[i & 1]), (i >> 1) & 1, &abort_flag)) return false;
                tc_fence_after();
                const uint32_t vbase = sV + s * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < C::kPVSteps; ++kk) {
                    const uint64_t dv = make_smem_desc(vbase + kk * C::kKPerInstr * C::kRowBytes,
                                                       kTileElems * C::kRowBytes, 8 * C::kRowBytes, C::kSwizzle);
                    if (ESZ == 2) mma_f16_ts(tO, tS[i & 1] + kk * 8, dv, C::kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                    else mma_f8_ts(tO, tS[i & 1] + kk * 8, dv, C::kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(bars.o_done));
                if (i + NS < n_kv) mma_commit(bar(bars.v_empty[s]));
                return true;
            };
            bool ok = mbar_wait(bar(bars.q_full), 0, &abort_flag);
            for (int j = 0; ok && j < n_kv; ++j) {
                const int s = j % NS;
                if (!mbar_wait(bar(bars.k_full[s]), (j / NS) & 1, &abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t kbase = sK + s * C::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < C::kQKSteps; ++kk) {
                    const int byte = kk * 32;
                    const uint32_t off = (byte / C::kRowBytes) * kTileElems * C::kRowBytes + (byte % C::kRowBytes);
                    const uint64_t da = make_smem_desc(sQ + off, 16, 8 * C::kRowBytes, C::kSwizzle);
                    const uint64_t db = make_smem_desc(kbase + off, 16, 8 * C::kRowBytes, C::kSwizzle);
                    if (ESZ == 2) mma_f16_ss(tS[j & 1], da, db, C::kIdescQK, kk > 0 ? 1u : 0u);
                    else mma_f8_ss(tS[j & 1], da, db, C::kIdescQK, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(bars.s_full[j & 1]));
                if (j + NS < n_kv) mma_commit(bar(bars.k_empty[s]));
                if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok) ok = issue_pv(n_kv - 1);
            if (!ok) {
                raise_status(&abort_flag);
                // wait for every MMA issued so far before TMEM is released
                const volatile int never = 0;
                mma_commit(bar(bars.drain));
                mbar_wait(bar(bars.drain), 0, &never);
            }
        }
    } else {
        // ============================================================ softmax / correction / epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;

        // query coordinates of this row and its window starts
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

        float scale_log2 = p.scale * kLog2e;
        float out_scale = 1.0f;
        if (ESZ == 1 && p.descale != nullptr) {
            scale_log2 *= p.descale[0] * p.descale[1];
            out_scale = p.descale[2];
        }
        constexpr float kTau = Precision<ESZ>::tau;
        constexpr float kShift = Precision<ESZ>::p_shift;

        float m_run = -INFINITY;   // running reference maximum, log2 units (scaled scores)
        float l_run = 0.0f;        // running sum of P (in the same shifted units as P)
        bool ok = true;

        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            ok = mbar_wait(bar(bars.s_full[sb]), (j >> 1) & 1, &abort_flag);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();

            int kc[3];
            box.coords(j, kc);
            bool full = true;
#pragma unroll
            for (int d = 0; d < 3; ++d)
                full = full && dim_tile_full(kc[d], p.tile[d], p.dims[d], p.win[d], box.r[d]);

            float s[128];
            {
                uint32_t r0[32], r1[32], r2[32], r3[32];
                const uint32_t ts = tmem + kColS0 + sb * 128 + lane_addr;
                tmem_ld32(ts, r0);
                tmem_ld32(ts + 32, r1);
                tmem_ld32(ts + 64, r2);
                tmem_ld32(ts + 96, r3);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    s[i] = __uint_as_float(r0[i]);
                    s[32 + i] = __uint_as_float(r1[i]);
                    s[64 + i] = __uint_as_float(r2[i]);
                    s[96 + i] = __uint_as_float(r3[i]);
                }
            }
            if (!full) {
                uint32_t m[4];
                build_row_mask(p, kc, st, m);
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    s[c] = (m[c >> 5] >> (c & 31)) & 1u ? s[c] : -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
            const float m_tile = mx * scale_log2;   // -inf if the row is fully masked

            const bool need = m_tile > m_run + kTau;
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? m_tile : m_run;
                const float alpha = need ? fast_exp2(m_run - m_new) : 1.0f;   // 0 when m_run = -inf
                m_run = m_new;
                l_run *= alpha;
                if (j > 0) {
                    // O holds PV(0..j-1): wait for PV(j-1), then rescale
                    ok = mbar_wait(bar(bars.o_done), (j - 1) & 1, &abort_flag);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        uint32_t r[32];
                        tmem_ld32(tmem + kColO + lane_addr + c, r);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        tmem_st32(tmem + kColO + lane_addr + c, r);
                    }
                    tmem_wait_st();
                }
            }
            const float m_eff = (m_run == -INFINITY) ? 0.0f : m_run - kShift;
            float rowsum = 0.0f;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
                s[c] = fast_exp2(fmaf(s[c], scale_log2, -m_eff));
                rowsum += s[c];
            }
            l_run += rowsum;
            {
                uint32_t pk[C::kPCols];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float x[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = s[c * 32 + i];
                    pack_p<ESZ>(x, pk + c * (32 * ESZ / 4));
                }
                if constexpr (C::kPCols == 64) {
                    uint32_t a[32], b[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) { a[i] = pk[i]; b[i] = pk[32 + i]; }
                    tmem_st32(tmem + kColS0 + sb * 128 + lane_addr, a);
                    tmem_st32(tmem + kColS0 + sb * 128 + lane_addr + 32, b);
                } else {
                    uint32_t a[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = pk[i];
                    tmem_st32(tmem + kColS0 + sb * 128 + lane_addr, a);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.p_full[sb]));
        }

        // ------------------------------------------------------------ epilogue
        if (ok) {
            ok = mbar_wait(bar(bars.o_done), (n_kv - 1) & 1, &abort_flag);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (!ok) {
            raise_status(&abort_flag);
        } else {
            tc_fence_after();
            const bool has = row_valid && l_run > 0.0f;
            const float inv_l = has ? out_scale / l_run : 0.0f;
            auto* out_row = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) +
                                                     (q_tile_global * kTileElems + row) * static_cast<int64_t>(D) * 2);
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + kColO + lane_addr + c, r);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * i]) * inv_l,
                                                             __uint_as_float(r[2 * i + 1]) * inv_l);
                    pk[i] = *reinterpret_cast<uint32_t*>(&h);
                }
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    out_row[c / 8 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
            if (p.lse != nullptr) {
                const float lse = has ? (m_run - kShift + __log2f(l_run)) * kLn2 : -INFINITY;
                p.lse[q_tile_global * kTileElems + row] = lse;
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

template <int D, int ESZ, int NS>
cudaError_t launch_impl(const FwdParams& p, int64_t num_q_tiles, cudaStream_t stream)
{
    using C = Cfg<D, ESZ, NS>;
    static_assert(NS <= 4, "barrier arrays hold 4 stages");
    static_assert(C::kSmemAlloc <= 232448, "shared memory budget");
    auto kern = gna_fwd_kernel<D, ESZ, NS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    kern<<<dim3(static_cast<unsigned>(num_q_tiles)), kThreads, C::kSmemAlloc, stream>>>(p);
    return cudaGetLastError();
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
