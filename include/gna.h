/*
 * gna.h -- C ABI of the B300 (sm_103a) Generalized Neighborhood Attention
 * library (libgna_b300.so): the forward pass with its layout permutes, a
 * backward pass (bf16, head_dim 32, 64 or 128) and host-side planning.
 *
 * What the library computes
 * -------------------------
 * GNA page ("GNA稀疏注意力机制：视觉Transformer计算优化实践"), §1.1: every
 * query attends only to a window of keys around it on the 2-D / 3-D token
 * grid; a per-dimension stride moves that window in jumps, from the sliding
 * window of neighborhood attention (stride 1) to blocked attention (stride =
 * window).  Written out, for a grid (T, H, W), window (wT, wH, wW) and stride
 * (sT, sH, sW), per dimension of length L with window w and stride s:
 *
 *     leader(i) = min(floor(i / s) * s + off(s), L - 1)
 *     start(i)  = clamp(leader(i) - floor(w / 2), 0, L - w)
 *
 * with off(s) = floor(s / 2) (GNA_LEADER_CENTER, the default: queries of a
 * stride group share the window of the group's centre, so stride = window on a
 * divisible grid is exactly blocked attention) or floor((s - 1) / 2)
 * (GNA_LEADER_LITERAL; identical for odd strides).  Query i attends to the
 * keys j with start_d(i) <= j_d < start_d(i) + w_d in every dimension, i.e.
 * exactly wT*wH*wW keys (§1.2: O(n k) work), with
 *
 *     lse_i = ln sum_j exp(scale * <q_i, k_j>),
 *     out_i = sum_j exp(scale * <q_i, k_j> - lse_i) v_j,   scale = 1/sqrt(d).
 *
 * Layouts
 * -------
 * raster : [B, T, H, W, heads, d]   (a 2-D image grid is T = 1)
 * tiled  : [B, heads, nT, nH, nW, tT*tH*tW, d],  n_ = ceil(L_ / t_)
 *          Inside a tile the element index is (it*tH + iy)*tW + ix.  Grid
 *          positions past the end of a dimension (padding of the last tile)
 *          are zero.  The tile (tT, tH, tW) has 128 elements, each a power of
 *          two (GNA page §1.1: Q and KV are split into fixed-size
 *          multi-dimensional tiles; §2.2: tokens are permuted into this order
 *          before attention and back after it).
 * value  : [B, heads, nT, nH, nW, d, tT*tH*tW]
 *          the tiled layout with every tile stored transposed (feature-major:
 *          row f of a tile holds feature f of its 128 tokens).  gna_forward
 *          reads v in this layout: P V then streams V with the token index
 *          contiguous, the operand order the tensor core reads fastest.
 * gna_forward reads q and k in the tiled layout, v in the value layout, and
 * writes out tiled; gna_permute / gna_unpermute and gna_permute_v /
 * gna_unpermute_v convert.  lse is tiled like a d = 1 float tensor:
 * [B, heads, tiles, 128], and gna_unpermute(head_dim = 1, GNA_F32) turns it
 * into raster [B, T, H, W, heads].
 *
 * Conventions
 * -----------
 * * Every pointer is CUDA device memory owned by the caller (global memory on
 *   the current device) and must be 16-byte aligned.  The library allocates
 *   nothing per call.
 * * `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Calls enqueue work and return GNA_OK without synchronising.
 *   Apart from gna_get_status (which synchronises), every call may be
 *   captured into a CUDA graph once it has been made on the device outside a
 *   capture (the first call sets kernel attributes and, for
 *   gna_backward_noalloc, looks up its workspace); a replay reads the
 *   captured buffers' current contents.
 * * Argument errors are detected on the host before anything is enqueued and
 *   return GNA_ERR_INVALID_ARG / GNA_ERR_UNSUPPORTED; nothing is launched.
 *   Launch failures return GNA_ERR_CUDA.  gna_last_error() gives a message.
 * * A kernel that gives up waiting on an internal pipeline barrier (a bound of
 *   about two seconds) records GNA_ERR_TIMEOUT in a device status word and
 *   exits cleanly; its outputs are then incomplete although the call itself
 *   returned GNA_OK.  Read gna_get_status() after the calls whose results
 *   you use: it is the only report of such a failure.
 * * No C++ exception crosses this boundary.  Functions are thread-safe.
 */
#ifndef GNA_B300_H
#define GNA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GNA_VERSION 1

typedef enum {
    GNA_OK = 0,
    GNA_ERR_INVALID_ARG = 1,  /* bad size, geometry, pointer or alignment */
    GNA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head_dim 96) */
    GNA_ERR_CUDA = 3,         /* a CUDA runtime / driver call failed */
    GNA_ERR_TIMEOUT = 4       /* a kernel abandoned a pipeline wait (device status) */
} gna_status;

typedef enum {
    GNA_BF16 = 0,      /* bfloat16 */
    GNA_FP8_E4M3 = 1,  /* float8 e4m3 ("fn": finite, max 448) */
    GNA_F32 = 2        /* float32: permute / unpermute only (lse) */
} gna_dtype;

typedef enum {
    GNA_LEADER_CENTER = 0,   /* off(s) = floor(s/2)      (default) */
    GNA_LEADER_LITERAL = 1   /* off(s) = floor((s-1)/2) */
} gna_leader_rule;

/* Options of gna_forward_ex.  Zero-initialise for the defaults. */
typedef struct {
    int tile[3];          /* layout tile; {0,0,0} = gna_tile_shape(dims)               */
    int leader_rule;      /* gna_leader_rule                                            */
    float scale;          /* softmax scale; 0 = 1/sqrt(head_dim)                        */
    const float* descale; /* GNA_FP8_E4M3: device pointer to 3 floats, the
                             per-tensor dequantisation scales of q, k, v (value =
                             code * descale); required (pass 1, 1, 1 explicitly for
                             unscaled codes).  Must be NULL for GNA_BF16.           */
    int tile_kv[3];       /* forward only: tile of k and v when it differs from the
                             tile of q, out and lse (GNA page §1.2: query and
                             key/value tiles sized independently); {0,0,0} = the
                             same tile as q.  Both are 128-element power-of-two
                             tiles; k and v are then permuted with tile_kv (the
                             *_tiled permutes), q, out and lse with `tile`.
                             gna_plan_tiles picks a pair.  The backward pass
                             needs the two equal (GNA_ERR_UNSUPPORTED).          */
} gna_options;

/* ------------------------------------------------------------ layout ---- */

/* Default tile of the tiled layout for a grid: 128 elements, powers of two,
 * least zero padding first, then the preferred shapes (2,8,8) for 3-D grids
 * and (1,8,16) for 2-D grids.  dims[0] = T (1 for images).
 * Returns GNA_ERR_INVALID_ARG for non-positive dims. */
gna_status gna_tile_shape(const int dims[3], int tile[3]);

/* Number of elements of one tiled tensor: B*heads*nT*nH*nW*128*head_dim
 * (returns -1 on invalid arguments; tile NULL = default tile). */
int64_t gna_tiled_elems(int B, int heads, const int dims[3], const int tile[3], int head_dim);

/* Elements of one tensor that gna_permute / gna_permute_v write for these
 * sizes under the default tile: gna_tiled_elems(B, heads, dims, NULL,
 * head_dim), the size to allocate for q, k, v_value and out of gna_forward.
 * Returns 0 on invalid arguments.  GNA page §2.2 (the tokens are permuted
 * into tile order before attention) and §1.1 (fixed-size tiles: the grid is
 * padded up to whole tiles). */
size_t gna_permuted_elems(int B, int heads, const int dims[3], int head_dim);

/* Raster -> tiled (zero padding) and tiled -> raster (padding dropped).
 * src and dst must not overlap.  Any head_dim >= 1 with head_dim * element
 * size a multiple of 4 bytes; dtype GNA_BF16, GNA_FP8_E4M3 or GNA_F32.
 * The *_tiled variants take an explicit tile (128 elements, powers of two).
 * GNA page §2.2 (memory operations: token permutation before and after the
 * model, as a dedicated copy kernel). */
gna_status gna_permute(const void* src, void* dst, int B, int heads, const int dims[3],
                       int head_dim, gna_dtype dtype, void* stream);
gna_status gna_unpermute(const void* src, void* dst, int B, int heads, const int dims[3],
                         int head_dim, gna_dtype dtype, void* stream);
gna_status gna_permute_tiled(const void* src, void* dst, int B, int heads, const int dims[3],
                             const int tile[3], int head_dim, gna_dtype dtype, void* stream);
gna_status gna_unpermute_tiled(const void* src, void* dst, int B, int heads, const int dims[3],
                               const int tile[3], int head_dim, gna_dtype dtype, void* stream);

/* Raster -> value layout (zero padding) and back (padding dropped): the
 * tiled layout with each tile transposed to d x 128.  Same element count as
 * the tiled layout (gna_tiled_elems).  dtype GNA_BF16 or GNA_FP8_E4M3 with
 * head_dim * element size a power of two from 16 to 256 bytes (otherwise
 * GNA_ERR_UNSUPPORTED); src and dst must not overlap.  GNA page
 * §2.2 (the permutation is a dedicated copy kernel; here it also produces the
 * operand order of the P V product). */
gna_status gna_permute_v(const void* src, void* dst, int B, int heads, const int dims[3],
                         int head_dim, gna_dtype dtype, void* stream);
gna_status gna_unpermute_v(const void* src, void* dst, int B, int heads, const int dims[3],
                           int head_dim, gna_dtype dtype, void* stream);
gna_status gna_permute_v_tiled(const void* src, void* dst, int B, int heads, const int dims[3],
                               const int tile[3], int head_dim, gna_dtype dtype, void* stream);
gna_status gna_unpermute_v_tiled(const void* src, void* dst, int B, int heads, const int dims[3],
                                 const int tile[3], int head_dim, gna_dtype dtype, void* stream);

/* ------------------------------------------------------------ forward ---- */

/* GNA forward pass (GNA page §1.1 window rule, §2.1 kernel structure).
 *
 * q, k    : tiled [B, heads, tiles, 128, head_dim] (gna_permute)
 * v_value : V in the VALUE layout [B, heads, tiles, head_dim, 128]
 *           (gna_permute_v), NOT the tiled layout of q and k.  The two layouts
 *           have the same size and cannot be told apart from the pointer: a
 *           tiled V gives wrong results without any error.  (The value layout
 *           lets P V read V in the operand order the tensor core streams at
 *           full rate; see the layout notes above.)
 *           q, k, v_value all GNA_BF16 (gna_forward_fp8 for GNA_FP8_E4M3)
 * out     : tiled [B, heads, tiles, 128, head_dim] bfloat16; padding rows are
 *           written as zero
 * lse     : tiled [B, heads, tiles, 128] float32, natural log; may be NULL
 * dims, window, stride : per dimension (T, H, W); 1 <= stride <= window <= dims
 * head_dim: 32, 64 or 128
 * Uses the default tile, GNA_LEADER_CENTER and scale 1/sqrt(head_dim).
 * dtype must be GNA_BF16: e4m3 codes need their per-tensor descales, so
 * GNA_FP8_E4M3 returns GNA_ERR_INVALID_ARG here (use gna_forward_fp8).
 * Asynchronous on `stream`. */
gna_status gna_forward(const void* q, const void* k, const void* v_value, void* out, float* lse,
                       int B, int heads, const int dims[3], const int window[3], const int stride[3],
                       int head_dim, gna_dtype dtype, void* stream);

/* gna_forward on float8 e4m3 codes (GNA page §1.2 and §2.1: the FP8 mode).
 * q, k, v_value hold e4m3 codes in the layouts of gna_forward; descale_qkv is
 * a device pointer to 3 floats, the per-tensor dequantisation scales of q, k
 * and v (value = code * descale, e.g. amax / 448 of each tensor).  The q and
 * k scales fold into the softmax scale and the v scale into the epilogue; P
 * is rounded to e4m3 for P V; out stays bfloat16.  head_dim 128.  NULL
 * descale_qkv is GNA_ERR_INVALID_ARG. */
gna_status gna_forward_fp8(const void* q, const void* k, const void* v_value, void* out, float* lse,
                           int B, int heads, const int dims[3], const int window[3], const int stride[3],
                           int head_dim, const float* descale_qkv, void* stream);

/* gna_forward with explicit options (tile, leader rule, scale, fp8 descales,
 * a separate key/value tile), for either dtype; GNA_FP8_E4M3 requires
 * opt->descale.  With opt->tile_kv set, q, out and lse are tiled with
 * opt->tile and k, v_value with opt->tile_kv (sizes gna_tiled_elems of each). */
gna_status gna_forward_ex(const void* q, const void* k, const void* v_value, void* out, float* lse,
                          int B, int heads, const int dims[3], const int window[3], const int stride[3],
                          int head_dim, gna_dtype dtype, const gna_options* opt, void* stream);

/* gna_forward_ex without the tiled permutes of Q, K, O and lse.  The same
 * arithmetic on the same tiles (GNA page §2.1: the multi-dimensional tiling is
 * a view of the token grid); the kernel gathers each 128-token Q and K tile
 * straight from the raster tensors, a 5-D TMA box for K and row loads for Q,
 * and writes O and lse back to raster rows.  Query rows of padded tile slots
 * are neither read nor written.  opt->tile_kv, if set, shapes the K boxes and
 * the value layout of v_value; opt->tile the query tiles.
 *
 * q, k    : raster [B, T, H, W, heads, head_dim], row stride heads*head_dim
 * v_value : value layout [B, heads, tiles, head_dim, 128] (gna_permute_v_tiled
 *           with the key/value tile; not raster)
 * out     : raster [B, T, H, W, heads, head_dim] bfloat16
 * lse     : raster [B, T, H, W, heads] float32, natural log; may be NULL
 * Everything else as gna_forward_ex; opt may be NULL.  All pointers 16-byte
 * aligned.  GNA_ERR_INVALID_ARG / GNA_ERR_UNSUPPORTED as gna_forward_ex. */
gna_status gna_forward_raster(const void* q, const void* k, const void* v_value, void* out, float* lse,
                              int B, int heads, const int dims[3], const int window[3], const int stride[3],
                              int head_dim, gna_dtype dtype, const gna_options* opt, void* stream);

/* gna_forward_raster with V in the raster layout as well: no permute at all
 * (GNA page §2.2: the permutation before and after the model is memory work
 * the page plans to remove).  v is raster [B, T, H, W, heads, head_dim]; the
 * kernel loads each V tile like K (a 5-D TMA box) and P V reads it token-major,
 * an operand order the tensor core streams more slowly than the value layout
 * of gna_forward_raster (about 930 against 600 cycles per 128-token tile on one
 * SM), so this call trades forward speed for the V permute it saves.
 * GNA_BF16 with head_dim 128 only (otherwise GNA_ERR_UNSUPPORTED); everything
 * else as gna_forward_raster. */
gna_status gna_forward_raster_all(const void* q, const void* k, const void* v, void* out, float* lse,
                                  int B, int heads, const int dims[3], const int window[3], const int stride[3],
                                  int head_dim, gna_dtype dtype, const gna_options* opt, void* stream);

/* ------------------------------------------------------------ backward ---- */

/* The GNA page asks for GNA in training (§4.2, problem 1; §5) and writes no
 * backward; the backward here is the derivative of the forward for the loss
 * L = sum_i <dout_i, out_i>.  It runs in three calls, all bf16 with head_dim
 * 32, 64 or 128, all tensors in the tiled layout of the forward (same tile):
 *
 * gna_backward_delta: delta_i = <dout_i, out_i> (fp32), the row term of the
 * softmax Jacobian, from the forward's bf16 out.
 *   out, dout : tiled [B, heads, tiles, 128, head_dim] bfloat16
 *   delta     : tiled [B, heads, tiles, 128] float32, written (caller-owned
 *               workspace of the dq call)
 *   opt       : tile (NULL or zero = default); other fields must be defaults
 *
 * gna_backward_dq: dq_i = scale sum_{j in N(i)} p_ij (<dout_i, v_j> - delta_i) k_j
 * with p_ij = exp(scale <q_i, k_j> - lse_i).
 *   q, k, v, dout : tiled bfloat16 (the forward's inputs and the gradient of out)
 *   k_value       : k in the value layout (gna_permute_v, same tile)
 *   lse           : the forward's tiled lse; delta: from gna_backward_delta
 *   dq            : tiled bfloat16, written (padding rows zero)
 *   window, stride, opt : as given to the forward
 *
 * gna_backward_dkdv: dv_j = sum_{i : j in N(i)} p_ij dout_i and
 * dk_j = scale sum_{i : j in N(i)} p_ij (<dout_i, v_j> - delta_i) q_i: one CTA
 * per KV tile walks the Q tiles whose windows reach it.
 *   q, k, v, dout : tiled bfloat16; lse, delta as for gna_backward_dq
 *   dk, dv        : tiled bfloat16, written (padding rows zero)
 *
 * Asynchronous on `stream`; a kernel that abandons a wait reports through
 * gna_get_status.  GNA_ERR_UNSUPPORTED for other dtypes or head_dims,
 * GNA_ERR_INVALID_ARG as gna_forward_ex. */
gna_status gna_backward_delta(const void* out, const void* dout, float* delta, int B, int heads,
                              const int dims[3], int head_dim, gna_dtype dtype, const gna_options* opt,
                              void* stream);
gna_status gna_backward_dkdv(const void* q, const void* k, const void* v, const void* dout, const float* lse,
                             const float* delta, void* dk, void* dv, int B, int heads, const int dims[3],
                             const int window[3], const int stride[3], int head_dim, gna_dtype dtype,
                             const gna_options* opt, void* stream);
gna_status gna_backward_dq(const void* q, const void* k, const void* k_value, const void* v,
                           const void* dout, const float* lse, const float* delta, void* dq, int B,
                           int heads, const int dims[3], const int window[3], const int stride[3],
                           int head_dim, gna_dtype dtype, const gna_options* opt, void* stream);

/* gna_backward_noalloc: the three backward calls above in one, for callers
 * that cannot allocate device memory.  The pages have no counterpart of this
 * call; it exists for a need of the callers, not of the method.
 *
 * gna_backward_dq and gna_backward_dkdv read a caller-owned float workspace
 * (delta, one value per tiled row).  Callers that cannot provide it are, for
 * example, code that runs inside a framework's memory pool or arena that owns
 * every device allocation, a process held to a fixed allocation budget, and
 * host code that must not call cudaMalloc (which can synchronise the device
 * and fail at any moment).  This call keeps delta in a fixed array of the
 * library's own device memory instead.  It allocates nothing and calls no
 * allocating routine; the caller still passes every input and output.
 *
 *   q, k, v, dout : tiled bfloat16 (as gna_backward_dq); k_value: k in the
 *                   value layout; out, lse: the forward's tiled out and lse
 *   dq, dk, dv    : tiled bfloat16, written
 *   other arguments as gna_backward_dq; bf16 with head_dim 32, 64 or 128 only
 *
 * Limit: B * heads * tiles * 128 (the tiled rows) must not exceed 2^22 =
 * 4,194,304; larger problems return GNA_ERR_INVALID_ARG before anything is
 * launched (use the three calls above with your own delta).  The array, 16
 * MiB, occupies global memory on every GPU that loads the library until the
 * process exits.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call on a device shares the one array and leaves its delta
 * values there; each call writes all the entries it reads before reading
 * them, so nothing needs clearing between calls.  Calls whose kernels overlap
 * on the GPU (on different streams, or from different threads) race on the
 * array and give wrong gradients: serialise them.  Asynchronous on `stream`;
 * errors as gna_backward_dq. */
gna_status gna_backward_noalloc(const void* q, const void* k, const void* k_value, const void* v,
                                const void* out, const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                int B, int heads, const int dims[3], const int window[3], const int stride[3],
                                int head_dim, gna_dtype dtype, const gna_options* opt, void* stream);

/* ------------------------------------------------------------ planning ---- */

/* Tile statistics of one (b, head) plane under the given tile (NULL =
 * default): total KV tiles the Q tiles visit, how many of those need the
 * element mask (not fully inside every query's window, or padded), and the
 * number of Q tiles.  Host only, no GPU needed.  GNA page §1.1 (the stride
 * decides which KV tiles each Q tile visits) and §2.1 (the mask is applied
 * only on partially covered tiles). */
gna_status gna_tile_stats(const int dims[3], const int window[3], const int stride[3],
                          const int tile[3], int leader_rule,
                          int64_t* visited_kv_tiles, int64_t* partial_kv_tiles, int64_t* q_tiles);

/* gna_tile_stats for query tiles `tile_q` and key/value tiles `tile_kv` (NULL =
 * default tile for either): the KV tiles, in units of tile_kv, that the
 * windows of each Q tile reach, and how many of them need the mask; q_tiles
 * counts tile_q tiles.  gna_tile_stats(..., tile, ...) is this call with
 * tile_q = tile_kv = tile.  Host only. */
gna_status gna_tile_stats_qkv(const int dims[3], const int window[3], const int stride[3], const int tile_q[3],
                              const int tile_kv[3], int leader_rule, int64_t* visited_kv_tiles,
                              int64_t* partial_kv_tiles, int64_t* q_tiles);

/* Tile planner: the analytic speedup bound the GNA page suggests checking before
 * deployment (§4.2, problem 2; a NATTENSim-like count).  Over every 128-element
 * power-of-two tile it counts, with gna_tile_stats, the 128 x 128 tiles the
 * forward pass visits and picks the tile with the fewest (ties: fewer partial
 * tiles, then the default tile).  Outputs:
 *   tile          the chosen tile (use it with the *_tiled permutes and
 *                 gna_forward_ex);
 *   tile_overhead visited tile pairs / useful (query, key) pairs, >= 1 (NULL ok);
 *   speedup_bound dense attention's visited tiles / these visited tiles on the
 *                 same tiling: the speedup over dense attention at equal
 *                 tile throughput (NULL ok).
 * Host only.  GNA_ERR_INVALID_ARG on bad geometry or leader rule. */
gna_status gna_plan_tile(const int dims[3], const int window[3], const int stride[3], int leader_rule,
                         int tile[3], double* tile_overhead, double* speedup_bound);

/* gna_plan_tile over pairs: query tile and key/value tile chosen independently
 * (GNA page §1.2, decoupled Q and KV tiles) among all 128-element power-of-two
 * tiles, fewest visited 128 x 128 tile pairs first, then fewest partial ones,
 * then equal tiles (the default tile preferred).  speedup_bound = the Q tiles
 * x KV tiles of dense attention on this tiling / the visited pairs.  Host
 * only; errors as gna_plan_tile.  The count is all it weighs: the forward
 * kernel has the element mask of KV tiles 2x8x8 and 1x8x16 (at head_dim 128
 * also 2x4x16 and 4x4x8) compiled in and runs any other KV tile with a
 * generic, slower mask, so a pair that saves only a few percent of the tile
 * pairs with another KV tile may run slower than the default tile. */
gna_status gna_plan_tiles(const int dims[3], const int window[3], const int stride[3], int leader_rule,
                          int tile_q[3], int tile_kv[3], double* tile_overhead, double* speedup_bound);

/* Step schedule of a diffusion sampler.  The GNA page keeps full attention for
 * the first steps and switches to GNA afterwards: §3.2 runs the first 9 of 28
 * FLUX steps with full attention, §4.2 advises full attention for the first
 * 10-20 % of the steps, §5 larger windows early.  Full attention is GNA with
 * window = grid and stride 1 (the forward then visits every KV tile).  For step
 * `step` (0-based) of `num_steps`, writes the window and stride to pass to the
 * forward: the whole grid with stride 1 while step < full_steps, else `window`
 * and `stride`.  Host only.  GNA_ERR_INVALID_ARG unless 0 <= step < num_steps,
 * 0 <= full_steps <= num_steps and the geometry is valid. */
gna_status gna_schedule_step(int step, int num_steps, int full_steps, const int dims[3], const int window[3],
                             const int stride[3], int out_window[3], int out_stride[3]);

/* ------------------------------------------------------------ status ---- */

/* Synchronises `stream`, then returns and clears the device status word
 * (GNA_OK, or GNA_ERR_TIMEOUT if a kernel abandoned a wait since the last
 * call).  Returns GNA_ERR_CUDA if synchronisation itself failed. */
gna_status gna_get_status(void* stream);

const char* gna_status_string(gna_status s);

/* TEST ONLY: failure injection for the tests of the bounded waits.  Makes the
 * TMA producer of every later launch of one kernel skip the K/V load of loop
 * iteration `kv_index`, so that the consumers' bounded waits run out and the
 * kernel reports GNA_ERR_TIMEOUT through gna_get_status (after about two
 * seconds, with that launch's outputs incomplete).  kernel 0 = the forward,
 * 1 = the dQ backward; kv_index < 0 turns the injection off (the state at
 * load).  Process-wide; nothing else sets it.  GNA_ERR_INVALID_ARG for an
 * unknown kernel. */
gna_status gna_test_skip_kv_load(int kernel, int kv_index);

/* Message of the last error returned on the calling thread ("" if none). */
const char* gna_last_error(void);

int gna_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GNA_B300_H */
