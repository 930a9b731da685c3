// Backward pass of the GNA forward for sm_103a: dQ and the per-query delta.
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
//   warp 0      TMA producer: per KV tile, K (tiled), V (tiled) and K in the
//               value layout (feature-major) through a 2-stage ring
//   warp 1      TMEM allocator and tcgen05.mma issuer
//   warps 2..9  dS: thread = (query row, half of the 128 key columns)
// TMEM (512 columns): dQ [0, 128), S [128, 256), dP [256, 384), Q [384, 448),
// dO [448, 512).  Per KV tile: S = Q K^T and dP = dO V^T (A from TMEM), then
// dQ += dS K with dS (bf16) in TMEM as the A operand: each half writes its 32
// columns of dS over the front of its own 64 S columns, so the halves never
// touch each other's scores.  K in the value layout is the K-major B operand
// of dS K, as V is for P V in the forward.
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

__device__ int g_bwd_status = 0;

namespace {

constexpr int kBThreads = 320;
constexpr int kBSoftmaxWarps = 8;
constexpr uint32_t kBTmemCols = 512;
constexpr uint32_t kColDQ = 0;
constexpr uint32_t kColS = 128;
constexpr uint32_t kColDP = 256;
constexpr uint32_t kColQ = 384;
constexpr uint32_t kColDO = 448;
constexpr int kBStages = 2;
constexpr float kBLog2e = 1.4426950408889634f;

// bf16, head_dim 128
constexpr int kD = 128;
constexpr int kRowBytes = kD * 2;                  // 256 B per token row
constexpr int kTileBytes = kTileElems * kRowBytes; // 32 KB per 128-token tile
constexpr int kStageBytes = 3 * kTileBytes;        // K, V, K (value layout)
constexpr int kSmemAlloc = kStageBytes * kBStages + 1024;
constexpr int kQKSteps = kRowBytes / 32;           // K = 16 bf16 per MMA
constexpr int kDQSteps = kTileElems / 16;
constexpr uint32_t kIdesc = make_idesc(128, 128, kFmtBF16, false);

struct BwdBars {
    uint64_t qdo_full;            // Q and dO rows stored in TMEM (8 warps)
    uint64_t full[kBStages];      // K, V, K (value layout) of a KV tile landed
    uint64_t empty[kBStages];     // the KV tile's three MMAs are done
    uint64_t sdp_full;            // S and dP of the current KV tile are in TMEM
    uint64_t ds_full;             // dS of the current KV tile is in TMEM (8 warps)
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

template <int N>
__device__ __forceinline__ void bwd_reg_fence(uint32_t (&r)[N])
{
#pragma unroll
    for (int i = 0; i < N; i += 8)
        asm volatile("" : "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), "+r"(r[i + 5]),
                     "+r"(r[i + 6]), "+r"(r[i + 7]));
}

__global__ void __launch_bounds__(kBThreads, 1) gna_bwd_dq_kernel(const __grid_constant__ BwdParams p)
{
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
        const DimRange r = dim_range(qc[d], p.tile[d], p.dims[d], p.win[d], p.str[d], p.off[d]);
        box.k0[d] = r.k0;
        box.cnt[d] = r.k1 - r.k0 + 1;
        dim_full_range(p.tile[d], p.dims[d], p.win[d], r, box.full_lo[d], box.full_hi[d]);
    }
    const int n_kv = box.cnt[0] * box.cnt[1] * box.cnt[2];
    const int64_t kv_tile_base = bh * p.tiles_per_head;       // first tile of this (b, head) plane

    auto bar = [](uint64_t& b) { return smem_u32(&b); };
    const uint32_t s_base = smem_u32(smem);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(bar(bars.qdo_full), kBSoftmaxWarps);
        for (int s = 0; s < kBStages; ++s) {
            mbar_init(bar(bars.full[s]), 1);
            mbar_init(bar(bars.empty[s]), 1);
        }
        mbar_init(bar(bars.sdp_full), 1);
        mbar_init(bar(bars.ds_full), kBSoftmaxWarps);
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
            prefetch_tensormap(&p.tmK);
            prefetch_tensormap(&p.tmV);
            prefetch_tensormap(&p.tmKv);
        }
        int issued = 0;
        bool early = false;
        int kc[3] = {box.k0[0], box.k0[1], box.k0[2]};
        for (int j = 0; j < n_kv; ++j, bwd_odometer(kc, box)) {
            const int s = j % kBStages;
            const int64_t tile = kv_tile_base + (kc[0] * p.nt[1] + kc[1]) * p.nt[2] + kc[2];
            if (j >= kBStages &&
                !__all_sync(0xffffffffu, mbar_wait(bar(bars.empty[s]), ((j / kBStages) & 1) ^ 1, &abort_flag))) {
                early = true;
                break;
            }
            if (elect_one_sync()) {
                const uint32_t st = s_base + s * kStageBytes;
                mbar_arrive_expect_tx(bar(bars.full[s]), kStageBytes);
                const int32_t row = static_cast<int32_t>(tile * kTileElems);
                const int32_t vrow = static_cast<int32_t>(tile * kD);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    // K and V tiles: 128 rows x 64 elements per box (128-byte swizzle)
                    tma_load_2d(st + c * kTileElems * 128, &p.tmK, bar(bars.full[s]), c * 64, row);
                    tma_load_2d(st + kTileBytes + c * kTileElems * 128, &p.tmV, bar(bars.full[s]), c * 64, row);
                    // K in the value layout: d rows x 64 tokens per box
                    tma_load_2d(st + 2 * kTileBytes + c * kD * 128, &p.tmKv, bar(bars.full[s]), c * 64, vrow);
                }
            }
            __syncwarp();
            ++issued;
        }
        if (early) {
            if (lane == 0) bwd_raise(&abort_flag);
            const volatile int never = 0;
            for (int j = (issued > kBStages ? issued - kBStages : 0); j < issued; ++j)
                mbar_wait(bar(bars.full[j % kBStages]), (j / kBStages) & 1, &never);
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        const uint32_t tDQ = tmem + kColDQ, tS = tmem + kColS, tDP = tmem + kColDP;
        const uint32_t tQ = tmem + kColQ, tDO = tmem + kColDO;
        const uint64_t d0 = make_smem_desc(s_base, 16, 8 * 128, kSwizzle128B);
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.qdo_full), 0, &abort_flag));
        for (int j = 0; ok && j < n_kv; ++j) {
            const int s = j % kBStages;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.full[s]), (j / kBStages) & 1, &abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint64_t dK = d0 + static_cast<uint64_t>((s * kStageBytes) >> 4);
            const uint64_t dV = d0 + static_cast<uint64_t>((s * kStageBytes + kTileBytes) >> 4);
            const uint64_t dKv = d0 + static_cast<uint64_t>((s * kStageBytes + 2 * kTileBytes) >> 4);
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < kQKSteps; ++kk) {
                    // k-step kk: features [16 kk, 16 kk + 16) = 32 bytes of every token row
                    const int off = ((kk * 32) / 128) * (kTileElems * 128) + ((kk * 32) % 128);
                    mma_f16_ts(tS, tQ + kk * 8, dK + static_cast<uint64_t>(off >> 4), kIdesc, kk > 0 ? 1u : 0u);
                    mma_f16_ts(tDP, tDO + kk * 8, dV + static_cast<uint64_t>(off >> 4), kIdesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(bars.sdp_full));
            }
            __syncwarp();
            if (!__all_sync(0xffffffffu, mbar_wait(bar(bars.ds_full), j & 1, &abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (elect_one_sync()) {
#pragma unroll
                for (int kk = 0; kk < kDQSteps; ++kk) {
                    // k-step kk: key columns [16 kk, 16 kk + 16); dS of key column
                    // half h sits at the front of S columns [64 h, 64 h + 64)
                    const uint32_t a = tS + (kk >> 2) * 64 + (kk & 3) * 8;
                    const int off = ((kk * 32) / 128) * (kD * 128) + ((kk * 32) % 128);
                    mma_f16_ts(tDQ, a, dKv + static_cast<uint64_t>(off >> 4), kIdesc, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(bars.empty[s]));
                if (j == n_kv - 1) mma_commit(bar(bars.dq_final));
            }
            __syncwarp();
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

        // this half of the Q and dO rows -> TMEM (A operands of S and dP)
        {
            const uint4* qs = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.q) + grow * kRowBytes +
                                                             half * (kRowBytes / 2));
            const uint4* ds = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.dout) +
                                                             grow * kRowBytes + half * (kRowBytes / 2));
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 v = __ldg(qs + i);
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
            }
            tmem_st32(tmem + kColQ + lane_addr + half * 32, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 v = __ldg(ds + i);
                w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
            }
            tmem_st32(tmem + kColDO + lane_addr + half * 32, w);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.qdo_full));
        }
        // lse (natural log) and delta of this query; padding rows contribute nothing
        const float lse2 = row_valid ? p.lse[grow] * kBLog2e : 0.0f;
        const float delta = row_valid ? p.delta[grow] : 0.0f;
        const float scale_log2 = p.scale * kBLog2e;

        bool ok = true;
        int kc[3] = {box.k0[0], box.k0[1], box.k0[2]};
        for (int j = 0; j < n_kv && ok; ++j, bwd_odometer(kc, box)) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.sdp_full), j & 1, &abort_flag));
            if (!ok) {
                bwd_raise(&abort_flag);
                break;
            }
            tc_fence_after();
            bool full = true;
#pragma unroll
            for (int d = 0; d < 3; ++d) full = full && kc[d] >= box.full_lo[d] && kc[d] <= box.full_hi[d];
            // two pieces of 32 key columns: S, dP -> dS (bf16) over the front of this half's S columns
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                uint32_t rs[32], rp[32];
                const uint32_t col = half * 64 + pc * 32;
                tmem_ld32(tmem + kColS + lane_addr + col, rs);
                tmem_ld32(tmem + kColDP + lane_addr + col, rp);
                tmem_wait_ld();
                bwd_reg_fence(rs);
                bwd_reg_fence(rp);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float ds2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int c = 2 * i + e;
                        bool valid = row_valid;
                        if (!full) {
                            // key (t, y, x) of column col + c inside this KV tile
                            const int kcol = static_cast<int>(col) + c;
                            const int cx = kcol & (p.tile[2] - 1);
                            const int cy = (kcol >> p.tlog[2]) & (p.tile[1] - 1);
                            const int ct = kcol >> (p.tlog[1] + p.tlog[2]);
                            valid = valid &&
                                    static_cast<unsigned>(kc[0] * p.tile[0] + ct - st[0]) < static_cast<unsigned>(p.win[0]) &&
                                    static_cast<unsigned>(kc[1] * p.tile[1] + cy - st[1]) < static_cast<unsigned>(p.win[1]) &&
                                    static_cast<unsigned>(kc[2] * p.tile[2] + cx - st[2]) < static_cast<unsigned>(p.win[2]);
                        }
                        const float pr = valid ? bwd_exp2(__uint_as_float(rs[c]) * scale_log2 - lse2) : 0.0f;
                        ds2[e] = pr * (__uint_as_float(rp[c]) - delta);
                    }
                    __nv_bfloat162 h = __floats2bfloat162_rn(ds2[0], ds2[1]);
                    pk[i] = *reinterpret_cast<uint32_t*>(&h);
                }
                tmem_st16(tmem + kColS + lane_addr + half * 64 + pc * 16, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bars.ds_full));
        }

        // ------------------------------------------------------------ epilogue
        if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(bars.dq_final), 0, &abort_flag));
            if (!ok) bwd_raise(&abort_flag);
        }
        if (ok) {
            tc_fence_after();
            uint8_t* dst_row = static_cast<uint8_t*>(p.dq) + grow * kRowBytes + half * (kRowBytes / 2);
#pragma unroll
            for (int pc = 0; pc < 2; ++pc) {
                uint32_t r[32];
                tmem_ld32(tmem + kColDQ + lane_addr + half * 64 + pc * 32, r);
                tmem_wait_ld();
                bwd_reg_fence(r);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[2 * i]) * p.scale,
                                                             __uint_as_float(r[2 * i + 1]) * p.scale);
                    pk[i] = *reinterpret_cast<uint32_t*>(&h);
                }
                uint4* dst = reinterpret_cast<uint4*>(dst_row + pc * 64);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
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
__global__ void gna_bwd_delta_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                                     float* __restrict__ delta, int64_t rows)
{
    const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
    if (r >= rows) return;
    const int lane = threadIdx.x % 32;
    const uint2 o = *reinterpret_cast<const uint2*>(out + r * kD + lane * 4);
    const uint2 g = *reinterpret_cast<const uint2*>(dout + r * kD + lane * 4);
    const float2 o0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.x));
    const float2 o1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.y));
    const float2 g0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g.x));
    const float2 g1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g.y));
    float acc = o0.x * g0.x + o0.y * g0.y + o1.x * g1.x + o1.y * g1.y;
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (lane == 0) delta[r] = acc;
}

}  // namespace

cudaError_t launch_backward_dq(const BwdParams& p, int64_t num_q_tiles, cudaStream_t stream)
{
    if (num_q_tiles <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gna_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    gna_bwd_dq_kernel<<<dim3(static_cast<unsigned>(num_q_tiles)), kBThreads, kSmemAlloc, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_backward_delta(const void* out, const void* dout, float* delta, int64_t rows, cudaStream_t stream)
{
    if (rows <= 0) return cudaSuccess;
    const int warps = 8;
    const int64_t blocks = (rows + warps - 1) / warps;
    gna_bwd_delta_kernel<<<dim3(static_cast<unsigned>(blocks)), warps * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), delta, rows);
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
