// gna_backward_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// The regular backward (gna_backward_delta, gna_backward_dq, gna_backward_dkdv)
// needs one caller-owned float workspace, delta = <dout, out> per tiled row,
// between its first call and the other two.  Some callers have no way to get
// that memory: code running inside a framework's fixed memory pool or arena
// that owns every device allocation, a process under a hard allocation budget,
// or host code that must not call cudaMalloc at all (it synchronises the
// device and can fail at an arbitrary moment).  For them this file keeps the
// delta workspace in a fixed array in the library's own device memory and
// runs the three kernels with it.  The caller still passes every input and
// output tensor.
//
// The array lives in global memory of every GPU that loads the library, from
// module load until the process exits: kStaticDeltaRows floats (16 MiB).
#include <cstdint>
#include <cmath>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/gna.h"
#include "gna_internal.h"

namespace gna {
namespace {

// delta of at most 2^22 tiled rows (B * heads * tiles * 128): 16 MiB.  The
// 720p-video latent (30 x 48 x 80 tokens, 24 heads, B = 1) needs 2,764,800.
constexpr int64_t kStaticDeltaRows = int64_t(1) << 22;

__device__ __align__(256) float g_static_delta[kStaticDeltaRows];

// The array's device address, looked up once per device.  In host code the
// name g_static_delta is only a host-side stand-in for the symbol, never a
// device address, so the kernels get this pointer instead.
constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
float* g_addr[kMaxDevices] = {};

gna_status static_delta_address(float** ptr)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return api_fail(GNA_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return api_fail(GNA_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_addr_mutex);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_delta);
        if (e != cudaSuccess || p == nullptr)
            return api_fail(GNA_ERR_CUDA, "cudaGetSymbolAddress of the static delta array failed");
        g_addr[dev] = static_cast<float*>(p);
    }
    *ptr = g_addr[dev];
    return GNA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gna

extern "C" gna_status gna_backward_noalloc(const void* q, const void* k, const void* k_value, const void* v,
                                           const void* out, const void* dout, const float* lse, void* dq, void* dk,
                                           void* dv, int B, int heads, const int dims[3], const int window[3],
                                           const int stride[3], int head_dim, gna_dtype dtype,
                                           const gna_options* opt, void* stream)
{
    // Every check of the three calls below runs first, so that an argument
    // error launches nothing at all.
    const void* ptrs[] = {q, k, k_value, v, out, dout, lse, dq, dk, dv};
    for (const void* p : ptrs) {
        if (p == nullptr) return gna::api_fail(GNA_ERR_INVALID_ARG, "NULL tensor pointer");
        if (!gna::aligned16(p)) return gna::api_fail(GNA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    }
    if (B < 1 || heads < 1) return gna::api_fail(GNA_ERR_INVALID_ARG, "B and heads must be >= 1");
    const int rule = opt ? opt->leader_rule : GNA_LEADER_CENTER;
    gna_status st = gna_tile_stats(dims, window, stride, opt ? opt->tile : nullptr, rule, nullptr, nullptr, nullptr);
    if (st != GNA_OK) return st;
    if (dtype != GNA_BF16 || (head_dim != 32 && head_dim != 64 && head_dim != 128))
        return gna::api_fail(GNA_ERR_UNSUPPORTED, "the backward pass supports bf16 with head_dim 32, 64 or 128");
    if (opt && !(opt->scale >= 0.0f && std::isfinite(opt->scale)))
        return gna::api_fail(GNA_ERR_INVALID_ARG, "scale must be finite and >= 0");
    if (opt && opt->descale) return gna::api_fail(GNA_ERR_INVALID_ARG, "descale is only used with GNA_FP8_E4M3");
    const int64_t elems = gna_tiled_elems(B, heads, dims, opt ? opt->tile : nullptr, head_dim);
    if (elems < 0) return gna::api_fail(GNA_ERR_INVALID_ARG, "invalid layout arguments");
    const int64_t rows = elems / head_dim;
    if (rows > gna::kStaticDeltaRows)
        return gna::api_fail(GNA_ERR_INVALID_ARG,
                             "gna_backward_noalloc: %lld tiled rows (B * heads * tiles * 128) exceed the %lld rows "
                             "of its static workspace; use gna_backward_delta / _dq / _dkdv with a caller-owned "
                             "delta",
                             static_cast<long long>(rows), static_cast<long long>(gna::kStaticDeltaRows));

    float* delta = nullptr;
    if ((st = gna::static_delta_address(&delta)) != GNA_OK) return st;
    // The delta kernel writes every one of the `rows` entries (padding rows
    // included) before the other two kernels read them, on the same stream:
    // nothing left in the array by an earlier call is read.
    if ((st = gna_backward_delta(out, dout, delta, B, heads, dims, head_dim, dtype, opt, stream)) != GNA_OK)
        return st;
    if ((st = gna_backward_dq(q, k, k_value, v, dout, lse, delta, dq, B, heads, dims, window, stride, head_dim, dtype,
                              opt, stream)) != GNA_OK)
        return st;
    return gna_backward_dkdv(q, k, v, dout, lse, delta, dk, dv, B, heads, dims, window, stride, head_dim, dtype, opt,
                             stream);
}
