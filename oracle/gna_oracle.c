/*
 * Plain C oracle of the Generalized Neighborhood Attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY: called from tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py, never from the product library.  It shares no
 * code with the CUDA sources.
 *
 * What it computes (GNA page, "GNA稀疏注意力机制：视觉Transformer计算优化实践",
 * §1.1 and §1.2; blockwise-free plain softmax as in the video tutorial page,
 * "视频生成推理提速:稀疏注意力组合配置教程", §3.3):
 *
 *   per dimension:  leader(i) = min(floor(i/s)*s + off(s), L-1)
 *                   start(i)  = clamp(leader(i) - floor(w/2), 0, L-w)
 *   N(i) = { j : start_d(i) <= j_d < start_d(i) + w_d in every dimension d }
 *   s_ij  = scale * <q_i, k_j>
 *   lse_i = ln sum_{j in N(i)} exp(s_ij)
 *   out_i = sum_{j in N(i)} exp(s_ij - lse_i) v_j
 *
 * off(s) = floor(s/2) (rule 0, group centre) or floor((s-1)/2) (rule 1).
 * Inputs are float32 holding the exact values the GPU reads (bf16 values, or
 * e4m3 codes); per-tensor scales are applied in double.  Everything is
 * accumulated in double with the maximum subtracted first (two passes).
 * Queries are split over POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static int leader_of(int i, int L, int s, int rule)
{
    int off = (rule == 0) ? s / 2 : (s - 1) / 2;
    int c = (i / s) * s + off;
    return c < L - 1 ? c : L - 1;
}

static int start_of(int i, int L, int w, int s, int rule)
{
    int a = leader_of(i, L, s, rule) - w / 2;
    if (a < 0) a = 0;
    if (a > L - w) a = L - w;
    return a;
}

/* Window start of every position 0..L-1 of one dimension (for pinning tests). */
void gna_oracle_window_starts(int L, int w, int s, int rule, int *out)
{
    for (int i = 0; i < L; ++i) out[i] = start_of(i, L, w, s, rule);
}

typedef struct {
    const float *q, *k, *v;
    int B, heads, dims[3], win[3], str[3], d, rule;
    double scale, sq, sk, sv;
    const int64_t *sel;
    int64_t begin, end;
    double *out, *lse;
    int status;
} job_t;

static void one_query(const job_t *J, int64_t row, int64_t flat, double *sbuf)
{
    const int T = J->dims[0], H = J->dims[1], W = J->dims[2];
    const int64_t N = (int64_t)T * H * W;
    const int d = J->d, heads = J->heads;
    int64_t tok = flat % N;
    int64_t bh = flat / N;
    int h = (int)(bh % heads), b = (int)(bh / heads);
    int x = (int)(tok % W), y = (int)((tok / W) % H), t = (int)(tok / ((int64_t)W * H));

    int a0 = start_of(t, T, J->win[0], J->str[0], J->rule);
    int a1 = start_of(y, H, J->win[1], J->str[1], J->rule);
    int a2 = start_of(x, W, J->win[2], J->str[2], J->rule);

    const float *qi = J->q + ((((int64_t)b * T + t) * H + y) * W + x) * heads * d + (int64_t)h * d;
    double qs = J->scale * J->sq * J->sk;

    /* pass 1: scores and their maximum */
    int64_t n = 0;
    double m = -INFINITY;
    for (int kt = a0; kt < a0 + J->win[0]; ++kt)
        for (int ky = a1; ky < a1 + J->win[1]; ++ky)
            for (int kx = a2; kx < a2 + J->win[2]; ++kx) {
                const float *kj = J->k + ((((int64_t)b * T + kt) * H + ky) * W + kx) * heads * d + (int64_t)h * d;
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += (double)qi[c] * (double)kj[c];
                double s = qs * acc;
                sbuf[n++] = s;
                if (s > m) m = s;
            }

    /* pass 2: exponentials, their sum, and the weighted sum of values */
    double *o = J->out + row * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    double z = 0.0;
    n = 0;
    for (int kt = a0; kt < a0 + J->win[0]; ++kt)
        for (int ky = a1; ky < a1 + J->win[1]; ++ky)
            for (int kx = a2; kx < a2 + J->win[2]; ++kx) {
                const float *vj = J->v + ((((int64_t)b * T + kt) * H + ky) * W + kx) * heads * d + (int64_t)h * d;
                double e = exp(sbuf[n++] - m);
                z += e;
                for (int c = 0; c < d; ++c) o[c] += e * (double)vj[c];
            }
    for (int c = 0; c < d; ++c) o[c] = o[c] / z * J->sv;
    J->lse[row] = m + log(z);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    int64_t wsz = (int64_t)J->win[0] * J->win[1] * J->win[2];
    double *sbuf = (double *)malloc(sizeof(double) * (size_t)wsz);
    if (!sbuf) { J->status = -2; return NULL; }
    for (int64_t r = J->begin; r < J->end; ++r) {
        int64_t flat = J->sel ? J->sel[r] : r;
        one_query(J, r, flat, sbuf);
    }
    free(sbuf);
    return NULL;
}

/*
 * q, k, v : float32 rasters [B, T, H, W, heads, d]
 * sel     : flat query ids ((b*heads + h)*N + (t*H + y)*W + x), or NULL for all
 *           B*heads*N queries in that order
 * out     : double [nsel, d];  lse : double [nsel]
 * Returns 0, -1 on invalid arguments, -2 on allocation failure.
 */
int gna_oracle_forward(const float *q, const float *k, const float *v,
                       int B, int heads, const int dims[3], const int window[3],
                       const int stride[3], int head_dim, int rule,
                       double scale, double scale_q, double scale_k, double scale_v,
                       const int64_t *sel, int64_t nsel,
                       double *out, double *lse, int nthreads)
{
    if (B < 1 || heads < 1 || head_dim < 1 || (rule != 0 && rule != 1)) return -1;
    for (int i = 0; i < 3; ++i)
        if (!(1 <= stride[i] && stride[i] <= window[i] && window[i] <= dims[i])) return -1;
    int64_t N = (int64_t)dims[0] * dims[1] * dims[2];
    int64_t total = sel ? nsel : (int64_t)B * heads * N;
    if (sel)
        for (int64_t r = 0; r < nsel; ++r)
            if (sel[r] < 0 || sel[r] >= (int64_t)B * heads * N) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = total > 0 ? (int)total : 1;

    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -2; }
    for (int i = 0; i < nthreads; ++i) {
        job_t *J = &jobs[i];
        J->q = q; J->k = k; J->v = v;
        J->B = B; J->heads = heads; J->d = head_dim; J->rule = rule;
        for (int c = 0; c < 3; ++c) { J->dims[c] = dims[c]; J->win[c] = window[c]; J->str[c] = stride[c]; }
        J->scale = scale; J->sq = scale_q; J->sk = scale_k; J->sv = scale_v;
        J->sel = sel; J->out = out; J->lse = lse;
        J->begin = total * i / nthreads;
        J->end = total * (i + 1) / nthreads;
        J->status = 0;
    }
    int rc = 0;
    if (nthreads == 1) {
        worker(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &jobs[i]);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    }
    for (int i = 0; i < nthreads; ++i) if (jobs[i].status) rc = jobs[i].status;
    free(jobs);
    free(th);
    return rc;
}

/*
 * Backward pass: the derivative of the forward above (the GNA page asks for
 * training with GNA, §4.2 problem 1 and §5, and writes no backward; this is
 * the chain rule applied to the definition).  For L = sum_i <dout_i, out_i>:
 *
 *   p_ij   = exp(s_ij - lse_i)                for j in N(i)
 *   dv_j  += p_ij dout_i
 *   dp_ij  = <dout_i, v_j>
 *   ds_ij  = p_ij (dp_ij - sum_l p_il dp_il)
 *   dq_i   = scale sum_j ds_ij k_j
 *   dk_j  += scale ds_ij q_i
 *
 * A thread owns whole (b, head) planes, so the scatters into dk and dv of one
 * plane never race.
 */
typedef struct {
    const float *q, *k, *v, *dout;
    int B, heads, dims[3], win[3], str[3], d, rule;
    double scale;
    int p_begin, p_end;
    double *dq, *dk, *dv;
    int status;
} bjob_t;

static int64_t row_of(const bjob_t *J, int b, int t, int y, int x, int h)
{
    return ((((int64_t)b * J->dims[0] + t) * J->dims[1] + y) * J->dims[2] + x) * J->heads + h;
}

static void backward_plane(const bjob_t *J, int plane, double *pbuf, double *dpbuf)
{
    const int T = J->dims[0], H = J->dims[1], W = J->dims[2], d = J->d;
    const int b = plane / J->heads, h = plane % J->heads;
    for (int t = 0; t < T; ++t)
        for (int y = 0; y < H; ++y)
            for (int x = 0; x < W; ++x) {
                const int a0 = start_of(t, T, J->win[0], J->str[0], J->rule);
                const int a1 = start_of(y, H, J->win[1], J->str[1], J->rule);
                const int a2 = start_of(x, W, J->win[2], J->str[2], J->rule);
                const int64_t qi = row_of(J, b, t, y, x, h) * d;
                /* probabilities of the window (max subtracted), and dp */
                int64_t n = 0;
                double m = -INFINITY;
                for (int kt = a0; kt < a0 + J->win[0]; ++kt)
                    for (int ky = a1; ky < a1 + J->win[1]; ++ky)
                        for (int kx = a2; kx < a2 + J->win[2]; ++kx) {
                            const int64_t kj = row_of(J, b, kt, ky, kx, h) * d;
                            double acc = 0.0, dacc = 0.0;
                            for (int c = 0; c < d; ++c) {
                                acc += (double)J->q[qi + c] * (double)J->k[kj + c];
                                dacc += (double)J->dout[qi + c] * (double)J->v[kj + c];
                            }
                            pbuf[n] = J->scale * acc;
                            dpbuf[n] = dacc;
                            if (pbuf[n] > m) m = pbuf[n];
                            ++n;
                        }
                double z = 0.0;
                for (int64_t l = 0; l < n; ++l) { pbuf[l] = exp(pbuf[l] - m); z += pbuf[l]; }
                double dsum = 0.0;
                for (int64_t l = 0; l < n; ++l) { pbuf[l] /= z; dsum += pbuf[l] * dpbuf[l]; }
                /* scatter */
                n = 0;
                for (int kt = a0; kt < a0 + J->win[0]; ++kt)
                    for (int ky = a1; ky < a1 + J->win[1]; ++ky)
                        for (int kx = a2; kx < a2 + J->win[2]; ++kx) {
                            const int64_t kj = row_of(J, b, kt, ky, kx, h) * d;
                            const double p = pbuf[n];
                            const double ds = p * (dpbuf[n] - dsum);
                            ++n;
                            for (int c = 0; c < d; ++c) {
                                J->dq[qi + c] += J->scale * ds * (double)J->k[kj + c];
                                J->dk[kj + c] += J->scale * ds * (double)J->q[qi + c];
                                J->dv[kj + c] += p * (double)J->dout[qi + c];
                            }
                        }
            }
}

static void *bworker(void *arg)
{
    bjob_t *J = (bjob_t *)arg;
    int64_t wsz = (int64_t)J->win[0] * J->win[1] * J->win[2];
    double *pbuf = (double *)malloc(sizeof(double) * (size_t)wsz);
    double *dpbuf = (double *)malloc(sizeof(double) * (size_t)wsz);
    if (!pbuf || !dpbuf) { free(pbuf); free(dpbuf); J->status = -2; return NULL; }
    for (int plane = J->p_begin; plane < J->p_end; ++plane) backward_plane(J, plane, pbuf, dpbuf);
    free(pbuf);
    free(dpbuf);
    return NULL;
}

/*
 * q, k, v, dout : float32 rasters [B, T, H, W, heads, d] (exact input values)
 * dq, dk, dv    : double rasters of the same shape, overwritten
 * Returns 0, -1 on invalid arguments, -2 on allocation failure.
 */
int gna_oracle_backward(const float *q, const float *k, const float *v, const float *dout,
                        int B, int heads, const int dims[3], const int window[3],
                        const int stride[3], int head_dim, int rule, double scale,
                        double *dq, double *dk, double *dv, int nthreads)
{
    if (B < 1 || heads < 1 || head_dim < 1 || (rule != 0 && rule != 1)) return -1;
    for (int i = 0; i < 3; ++i)
        if (!(1 <= stride[i] && stride[i] <= window[i] && window[i] <= dims[i])) return -1;
    const int64_t n_el = (int64_t)B * dims[0] * dims[1] * dims[2] * heads * head_dim;
    memset(dq, 0, sizeof(double) * (size_t)n_el);
    memset(dk, 0, sizeof(double) * (size_t)n_el);
    memset(dv, 0, sizeof(double) * (size_t)n_el);
    const int planes = B * heads;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > planes) nthreads = planes;
    bjob_t *jobs = (bjob_t *)calloc((size_t)nthreads, sizeof(bjob_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -2; }
    for (int i = 0; i < nthreads; ++i) {
        bjob_t *J = &jobs[i];
        J->q = q; J->k = k; J->v = v; J->dout = dout;
        J->B = B; J->heads = heads; J->d = head_dim; J->rule = rule; J->scale = scale;
        for (int c = 0; c < 3; ++c) { J->dims[c] = dims[c]; J->win[c] = window[c]; J->str[c] = stride[c]; }
        J->dq = dq; J->dk = dk; J->dv = dv;
        J->p_begin = (int)((int64_t)planes * i / nthreads);
        J->p_end = (int)((int64_t)planes * (i + 1) / nthreads);
        J->status = 0;
    }
    int rc = 0;
    if (nthreads == 1) {
        bworker(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, bworker, &jobs[i]);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    }
    for (int i = 0; i < nthreads; ++i) if (jobs[i].status) rc = jobs[i].status;
    free(jobs);
    free(th);
    return rc;
}

/*
 * dq of selected queries (the same derivative as gna_oracle_backward; dq_i
 * depends only on query i's own window, so a sample costs O(|W| d) per query).
 * sel: flat query ids ((b*heads + h)*N + (t*H + y)*W + x); dq: double [nsel, d].
 */
typedef struct {
    const bjob_t *J;
    const int64_t *sel;
    int64_t begin, end;
    double *dq;
    int status;
} dqjob_t;

static void *dq_worker(void *arg)
{
    dqjob_t *Q = (dqjob_t *)arg;
    const bjob_t *J = Q->J;
    const int T = J->dims[0], H = J->dims[1], W = J->dims[2], d = J->d;
    const int64_t N = (int64_t)T * H * W;
    int64_t wsz = (int64_t)J->win[0] * J->win[1] * J->win[2];
    double *pbuf = (double *)malloc(sizeof(double) * (size_t)wsz);
    double *dpbuf = (double *)malloc(sizeof(double) * (size_t)wsz);
    if (!pbuf || !dpbuf) { free(pbuf); free(dpbuf); Q->status = -2; return NULL; }
    for (int64_t r = Q->begin; r < Q->end; ++r) {
        const int64_t flat = Q->sel[r];
        const int64_t tok = flat % N, bh = flat / N;
        const int h = (int)(bh % J->heads), b = (int)(bh / J->heads);
        const int x = (int)(tok % W), y = (int)((tok / W) % H), t = (int)(tok / ((int64_t)W * H));
        const int a0 = start_of(t, T, J->win[0], J->str[0], J->rule);
        const int a1 = start_of(y, H, J->win[1], J->str[1], J->rule);
        const int a2 = start_of(x, W, J->win[2], J->str[2], J->rule);
        const int64_t qi = row_of(J, b, t, y, x, h) * d;
        int64_t n = 0;
        double m = -INFINITY;
        for (int kt = a0; kt < a0 + J->win[0]; ++kt)
            for (int ky = a1; ky < a1 + J->win[1]; ++ky)
                for (int kx = a2; kx < a2 + J->win[2]; ++kx) {
                    const int64_t kj = row_of(J, b, kt, ky, kx, h) * d;
                    double acc = 0.0, dacc = 0.0;
                    for (int c = 0; c < d; ++c) {
                        acc += (double)J->q[qi + c] * (double)J->k[kj + c];
                        dacc += (double)J->dout[qi + c] * (double)J->v[kj + c];
                    }
                    pbuf[n] = J->scale * acc;
                    dpbuf[n] = dacc;
                    if (pbuf[n] > m) m = pbuf[n];
                    ++n;
                }
        double z = 0.0, dsum = 0.0;
        for (int64_t l = 0; l < n; ++l) { pbuf[l] = exp(pbuf[l] - m); z += pbuf[l]; }
        for (int64_t l = 0; l < n; ++l) { pbuf[l] /= z; dsum += pbuf[l] * dpbuf[l]; }
        double *o = Q->dq + r * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        n = 0;
        for (int kt = a0; kt < a0 + J->win[0]; ++kt)
            for (int ky = a1; ky < a1 + J->win[1]; ++ky)
                for (int kx = a2; kx < a2 + J->win[2]; ++kx) {
                    const int64_t kj = row_of(J, b, kt, ky, kx, h) * d;
                    const double ds = pbuf[n] * (dpbuf[n] - dsum);
                    ++n;
                    for (int c = 0; c < d; ++c) o[c] += J->scale * ds * (double)J->k[kj + c];
                }
    }
    free(pbuf);
    free(dpbuf);
    return NULL;
}

int gna_oracle_backward_dq_sel(const float *q, const float *k, const float *v, const float *dout,
                               int B, int heads, const int dims[3], const int window[3],
                               const int stride[3], int head_dim, int rule, double scale,
                               const int64_t *sel, int64_t nsel, double *dq, int nthreads)
{
    if (B < 1 || heads < 1 || head_dim < 1 || (rule != 0 && rule != 1) || !sel || nsel < 0) return -1;
    for (int i = 0; i < 3; ++i)
        if (!(1 <= stride[i] && stride[i] <= window[i] && window[i] <= dims[i])) return -1;
    const int64_t total = (int64_t)B * heads * dims[0] * dims[1] * dims[2];
    for (int64_t r = 0; r < nsel; ++r)
        if (sel[r] < 0 || sel[r] >= total) return -1;
    bjob_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.dout = dout;
    J.B = B; J.heads = heads; J.d = head_dim; J.rule = rule; J.scale = scale;
    for (int c = 0; c < 3; ++c) { J.dims[c] = dims[c]; J.win[c] = window[c]; J.str[c] = stride[c]; }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nsel) nthreads = nsel > 0 ? (int)nsel : 1;
    dqjob_t *jobs = (dqjob_t *)calloc((size_t)nthreads, sizeof(dqjob_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -2; }
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].J = &J; jobs[i].sel = sel; jobs[i].dq = dq;
        jobs[i].begin = nsel * i / nthreads;
        jobs[i].end = nsel * (i + 1) / nthreads;
    }
    int rc = 0;
    if (nthreads == 1) {
        dq_worker(&jobs[0]);
    } else {
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, dq_worker, &jobs[i]);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    }
    for (int i = 0; i < nthreads; ++i) if (jobs[i].status) rc = jobs[i].status;
    free(jobs);
    free(th);
    return rc;
}

/*
 * dk and dv of selected keys.  Phase 1 computes, for every query of each
 * (b, head) plane that holds a selected key, lse_i and delta_i = sum_l p_il
 * <dout_i, v_l>.  Phase 2 walks, per selected key j, the queries whose window
 * holds j (per dimension an interval of positions, found by scanning the
 * window starts) and sums their contributions:
 *   dv_j = sum_i p_ij dout_i,   dk_j = scale sum_i p_ij (<dout_i, v_j> - delta_i) q_i.
 * sel: flat key ids ((b*heads + h)*N + (t*H + y)*W + x); dk, dv: double [nsel, d].
 */
typedef struct {
    const bjob_t *J;
    const int *planes;       /* planes needing lse / delta */
    int nplanes;
    int64_t begin, end;      /* range over nplanes * N queries */
    double *lse, *delta;     /* [B*heads*N], only the listed planes filled */
    const int64_t *sel;      /* phase 2 */
    int64_t kbegin, kend;
    double *dk, *dv;
    int status;
} kvjob_t;

static void *kv_phase1(void *arg)
{
    kvjob_t *Q = (kvjob_t *)arg;
    const bjob_t *J = Q->J;
    const int T = J->dims[0], H = J->dims[1], W = J->dims[2], d = J->d;
    const int64_t N = (int64_t)T * H * W;
    int64_t wsz = (int64_t)J->win[0] * J->win[1] * J->win[2];
    double *pbuf = (double *)malloc(sizeof(double) * (size_t)wsz);
    double *dpbuf = (double *)malloc(sizeof(double) * (size_t)wsz);
    if (!pbuf || !dpbuf) { free(pbuf); free(dpbuf); Q->status = -2; return NULL; }
    for (int64_t r = Q->begin; r < Q->end; ++r) {
        const int plane = Q->planes[r / N];
        const int64_t tok = r % N;
        const int h = plane % J->heads, b = plane / J->heads;
        const int x = (int)(tok % W), y = (int)((tok / W) % H), t = (int)(tok / ((int64_t)W * H));
        const int a0 = start_of(t, T, J->win[0], J->str[0], J->rule);
        const int a1 = start_of(y, H, J->win[1], J->str[1], J->rule);
        const int a2 = start_of(x, W, J->win[2], J->str[2], J->rule);
        const int64_t qi = row_of(J, b, t, y, x, h) * d;
        int64_t n = 0;
        double m = -INFINITY;
        for (int kt = a0; kt < a0 + J->win[0]; ++kt)
            for (int ky = a1; ky < a1 + J->win[1]; ++ky)
                for (int kx = a2; kx < a2 + J->win[2]; ++kx) {
                    const int64_t kj = row_of(J, b, kt, ky, kx, h) * d;
                    double acc = 0.0, dacc = 0.0;
                    for (int c = 0; c < d; ++c) {
                        acc += (double)J->q[qi + c] * (double)J->k[kj + c];
                        dacc += (double)J->dout[qi + c] * (double)J->v[kj + c];
                    }
                    pbuf[n] = J->scale * acc;
                    dpbuf[n] = dacc;
                    if (pbuf[n] > m) m = pbuf[n];
                    ++n;
                }
        double z = 0.0, dsum = 0.0;
        for (int64_t l = 0; l < n; ++l) { pbuf[l] = exp(pbuf[l] - m); z += pbuf[l]; }
        for (int64_t l = 0; l < n; ++l) dsum += pbuf[l] / z * dpbuf[l];
        const int64_t flat = (int64_t)plane * N + tok;
        Q->lse[flat] = m + log(z);
        Q->delta[flat] = dsum;
    }
    free(pbuf);
    free(dpbuf);
    return NULL;
}

/* query positions of one dimension whose window holds key position j: [lo, hi] */
static void inverse_window(int j, int L, int w, int s, int rule, int *lo, int *hi)
{
    *lo = 1;
    *hi = 0;
    for (int i = 0; i < L; ++i) {
        const int a = start_of(i, L, w, s, rule);
        if (a <= j && j < a + w) {
            if (*lo > *hi) *lo = i;
            *hi = i;
        }
    }
}

static void *kv_phase2(void *arg)
{
    kvjob_t *Q = (kvjob_t *)arg;
    const bjob_t *J = Q->J;
    const int T = J->dims[0], H = J->dims[1], W = J->dims[2], d = J->d;
    const int64_t N = (int64_t)T * H * W;
    for (int64_t r = Q->kbegin; r < Q->kend; ++r) {
        const int64_t flat = Q->sel[r];
        const int64_t tok = flat % N, plane = flat / N;
        const int h = (int)(plane % J->heads), b = (int)(plane / J->heads);
        const int x = (int)(tok % W), y = (int)((tok / W) % H), t = (int)(tok / ((int64_t)W * H));
        const int64_t kj = row_of(J, b, t, y, x, h) * d;
        int lo[3], hi[3];
        inverse_window(t, T, J->win[0], J->str[0], J->rule, &lo[0], &hi[0]);
        inverse_window(y, H, J->win[1], J->str[1], J->rule, &lo[1], &hi[1]);
        inverse_window(x, W, J->win[2], J->str[2], J->rule, &lo[2], &hi[2]);
        double *dk = Q->dk + r * d, *dv = Q->dv + r * d;
        for (int c = 0; c < d; ++c) { dk[c] = 0.0; dv[c] = 0.0; }
        for (int qt = lo[0]; qt <= hi[0]; ++qt)
            for (int qy = lo[1]; qy <= hi[1]; ++qy)
                for (int qx = lo[2]; qx <= hi[2]; ++qx) {
                    const int64_t qi = row_of(J, b, qt, qy, qx, h) * d;
                    const int64_t qflat = plane * N + ((int64_t)qt * H + qy) * W + qx;
                    double acc = 0.0, dacc = 0.0;
                    for (int c = 0; c < d; ++c) {
                        acc += (double)J->q[qi + c] * (double)J->k[kj + c];
                        dacc += (double)J->dout[qi + c] * (double)J->v[kj + c];
                    }
                    const double p = exp(J->scale * acc - Q->lse[qflat]);
                    const double ds = p * (dacc - Q->delta[qflat]);
                    for (int c = 0; c < d; ++c) {
                        dv[c] += p * (double)J->dout[qi + c];
                        dk[c] += J->scale * ds * (double)J->q[qi + c];
                    }
                }
    }
    return NULL;
}

static int run_kv_jobs(kvjob_t *jobs, int n, void *(*fn)(void *))
{
    pthread_t *th = (pthread_t *)calloc((size_t)n, sizeof(pthread_t));
    if (!th) return -2;
    if (n == 1) {
        fn(&jobs[0]);
    } else {
        for (int i = 0; i < n; ++i) pthread_create(&th[i], NULL, fn, &jobs[i]);
        for (int i = 0; i < n; ++i) pthread_join(th[i], NULL);
    }
    free(th);
    int rc = 0;
    for (int i = 0; i < n; ++i) if (jobs[i].status) rc = jobs[i].status;
    return rc;
}

int gna_oracle_backward_kv_sel(const float *q, const float *k, const float *v, const float *dout,
                               int B, int heads, const int dims[3], const int window[3],
                               const int stride[3], int head_dim, int rule, double scale,
                               const int64_t *sel, int64_t nsel, double *dk, double *dv, int nthreads)
{
    if (B < 1 || heads < 1 || head_dim < 1 || (rule != 0 && rule != 1) || !sel || nsel < 0) return -1;
    for (int i = 0; i < 3; ++i)
        if (!(1 <= stride[i] && stride[i] <= window[i] && window[i] <= dims[i])) return -1;
    const int64_t N = (int64_t)dims[0] * dims[1] * dims[2];
    const int planes_all = B * heads;
    for (int64_t r = 0; r < nsel; ++r)
        if (sel[r] < 0 || sel[r] >= (int64_t)planes_all * N) return -1;
    bjob_t J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.dout = dout;
    J.B = B; J.heads = heads; J.d = head_dim; J.rule = rule; J.scale = scale;
    for (int c = 0; c < 3; ++c) { J.dims[c] = dims[c]; J.win[c] = window[c]; J.str[c] = stride[c]; }
    /* planes holding a selected key */
    char *need = (char *)calloc((size_t)planes_all, 1);
    int *planes = (int *)calloc((size_t)planes_all, sizeof(int));
    double *lse = (double *)calloc((size_t)(planes_all * N), sizeof(double));
    double *delta = (double *)calloc((size_t)(planes_all * N), sizeof(double));
    if (nthreads < 1) nthreads = 1;
    kvjob_t *jobs = (kvjob_t *)calloc((size_t)nthreads, sizeof(kvjob_t));
    int rc = 0;
    if (!need || !planes || !lse || !delta || !jobs) { rc = -2; goto done; }
    int nplanes = 0;
    for (int64_t r = 0; r < nsel; ++r) need[sel[r] / N] = 1;
    for (int p = 0; p < planes_all; ++p) if (need[p]) planes[nplanes++] = p;
    const int64_t nq = (int64_t)nplanes * N;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].J = &J; jobs[i].planes = planes; jobs[i].nplanes = nplanes;
        jobs[i].begin = nq * i / nthreads; jobs[i].end = nq * (i + 1) / nthreads;
        jobs[i].lse = lse; jobs[i].delta = delta;
        jobs[i].sel = sel; jobs[i].kbegin = nsel * i / nthreads; jobs[i].kend = nsel * (i + 1) / nthreads;
        jobs[i].dk = dk; jobs[i].dv = dv;
    }
    rc = run_kv_jobs(jobs, nthreads, kv_phase1);
    if (rc == 0) rc = run_kv_jobs(jobs, nthreads, kv_phase2);
done:
    free(need); free(planes); free(lse); free(delta); free(jobs);
    return rc;
}
