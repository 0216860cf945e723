/*
 * attn_oracle.c -- fp64 CPU oracle for grouped-query scaled-dot-product
 * attention (forward + per-row max/log-sum, cached decode, batched prefill).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct
 * reference that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark load it; the
 * library itself never links, calls or reads anything here, and nothing here
 * includes a header of the library.
 *
 * What it computes.  The three shader pages (meganeura 0.2.0
 * src/shaders/attention.wgsl, meganeura 0.2.0 src/shaders/cached_attention.wgsl,
 * cera src/backend/shaders/attention_prefill.wgsl) compute softmax attention
 * with an online (streaming) softmax; the prefill page's header comment states
 * the result equals a plain batched softmax up to floating-point roundoff.  So
 * the oracle is that plain definition, one (query row, head) at a time:
 *
 *   g      = h / (H / G)                          (GQA head map, all pages)
 *   s_t    = scale * sum_d q[d] * k[t][g][d]       t in [0, n)
 *   m      = max_t s_t
 *   l      = sum_t exp(s_t - m)
 *   out[d] = sum_t exp(s_t - m) * v[t][g][d] / l
 *   lse    = (m, log l)        (attention.wgsl, fn main, final store: the
 *                               pair (max_score, log(sum_exp)))
 *   n == 0 -> out = 0, lse = (-1e30, -1e30)   (attention.wgsl, fn main: the
 *                               select() guards on sum_exp == 0 with the
 *                               initial max of -1e30 left in place)
 *
 * Window length n per row (its first key is always 0):
 *   forward causal  n = pos + 1        attention.wgsl header "Variants"
 *   forward full    n = q_seq          (same)
 *   forward cross   n = kv_seq         (same)
 *   decode          n = min(kv_pos + 1, max_seq)
 *                   cached_attention.wgsl, fn main (kv_len = kv_pos + 1);
 *                   the max_seq clamp is the prefill page's defensive belt
 *                   applied to decode as well.
 *   prefill         n = min(start_pos + q_base + i + 1, max_seq)
 *                   attention_prefill.wgsl, fn attention_prefill (pos_q,
 *                   seq_len).
 * Sliding window (every entry point's last argument, 0 = none): the window
 * becomes keys [lo, n) with lo = max(0, n - window).  attention.wgsl's key
 * loop starts at a $KV_START placeholder whose body the page leaves open; the
 * plainest reading, taken here, is a per-row lower bound that keeps the last
 * `window` positions of the row's window.
 *
 * Scores, exponentials and sums are fp64; the fp32 inputs are widened
 * exactly.  scale is 1/sqrt(head_dim) in fp64 for forward and decode (both
 * meganeura pages use inverseSqrt(head_dim)); prefill takes the fp32 scale
 * argument (the cera page passes it as f32 bits) and widens it.
 *
 * Parallelism: rows are independent; with OpenMP the (row, head) loop is
 * split across threads.  Nothing else is reordered: each score row is
 * materialised in full and reduced in index order.
 *
 * Return value of every entry point: 0 on success, -1 on invalid arguments.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_EMPTY_LSE (-1e30)

/* One (row, head): q points at head_dim query values; k and v point at key
 * row 0 of this kv head, consecutive key rows kv_stride floats apart.
 * s is caller scratch with room for n doubles. */
static void attend_row(const float *q, const float *k, const float *v,
                       size_t kv_stride, size_t n, int head_dim, double scale,
                       double *s, double *out, double *m_out, double *logl_out)
{
    if (n == 0) {
        for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
        *m_out = ORACLE_EMPTY_LSE;
        *logl_out = ORACLE_EMPTY_LSE;
        return;
    }
    double m = -INFINITY;
    for (size_t t = 0; t < n; ++t) {
        const float *kt = k + t * kv_stride;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += (double)q[d] * (double)kt[d];
        s[t] = dot * scale;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (size_t t = 0; t < n; ++t) {
        s[t] = exp(s[t] - m);
        l += s[t];
    }
    for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (size_t t = 0; t < n; ++t) acc += s[t] * (double)v[t * kv_stride + d];
        out[d] = acc / l;
    }
    *m_out = m;
    *logl_out = log(l);
}

/* First key of a row whose window ends at n (exclusive), under a sliding
 * window of `window` keys (0 = no limit). */
static size_t window_start(size_t n, int window)
{
    return (window > 0 && n > (size_t)window) ? n - (size_t)window : 0;
}

static int bad_heads(int H, int G, int D)
{
    return H <= 0 || G <= 0 || D <= 0 || (H % G) != 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Forward attention (attention.wgsl, fn main).
 *   q    [q_seq, H*D]        out [q_seq, H*D] (only the listed rows written)
 *   k, v [kv_seq, G*D]       lse [q_seq, H, 2] or NULL
 *   mask 0 causal (needs kv_seq == q_seq), 1 full (kv_seq == q_seq), 2 cross
 *   rows: query positions to compute (NULL -> all q_seq of them)
 */
int oracle_forward(const float *q, const float *k, const float *v,
                   double *out, double *lse, int q_seq, int kv_seq,
                   int H, int G, int D, int mask, const int *rows, int n_rows, int window)
{
    if (bad_heads(H, G, D) || q_seq < 0 || kv_seq < 0 || mask < 0 || mask > 2 || window < 0) return -1;
    if (mask != 2 && kv_seq != q_seq) return -1;
    if (rows == NULL) n_rows = q_seq;
    for (int r = 0; r < n_rows; ++r) {
        int pos = rows ? rows[r] : r;
        if (pos < 0 || pos >= q_seq) return -1;
    }
    const int gs = H / G;
    const size_t kv_dim = (size_t)G * D;
    const double scale = 1.0 / sqrt((double)D);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(kv_seq > 0 ? kv_seq : 1));
        if (s == NULL) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (int r = 0; r < n_rows; ++r) {
                for (int h = 0; h < H; ++h) {
                    const int pos = rows ? rows[r] : r;
                    const int g = h / gs;
                    size_t n = (mask == 0) ? (size_t)pos + 1 : (size_t)kv_seq;
                    const size_t lo = window_start(n, window);
                    const size_t qo = (size_t)pos * H * D + (size_t)h * D;
                    double m, logl;
                    attend_row(q + qo, k + lo * kv_dim + (size_t)g * D, v + lo * kv_dim + (size_t)g * D, kv_dim,
                               n - lo, D, scale, s, out + qo, &m, &logl);
                    if (lse) {
                        lse[((size_t)pos * H + h) * 2] = m;
                        lse[((size_t)pos * H + h) * 2 + 1] = logl;
                    }
                }
            }
        }
        free(s);
    }
    return err;
}

/*
 * Cached single-token decode (cached_attention.wgsl, fn main).
 *   q [1, H*D]; k_cache, v_cache [max_seq, G*D]; out [1, H*D]
 *   attends to key positions 0..kv_pos inclusive, clamped to max_seq rows.
 */
int oracle_decode(const float *q, const float *k_cache, const float *v_cache,
                  unsigned kv_pos, double *out, int H, int G, int D, int max_seq, int window)
{
    if (bad_heads(H, G, D) || max_seq < 0 || window < 0) return -1;
    const int gs = H / G;
    const size_t kv_dim = (size_t)G * D;
    const double scale = 1.0 / sqrt((double)D);
    size_t n = (size_t)kv_pos + 1;
    if (n > (size_t)max_seq) n = (size_t)max_seq;
    double *s = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    if (s == NULL) return -1;
    const size_t lo = window_start(n, window);
    for (int h = 0; h < H; ++h) {
        const int g = h / gs;
        double m, logl;
        attend_row(q + (size_t)h * D, k_cache + lo * kv_dim + (size_t)g * D, v_cache + lo * kv_dim + (size_t)g * D,
                   kv_dim, n - lo, D, scale, s, out + (size_t)h * D, &m, &logl);
    }
    free(s);
    return 0;
}

/*
 * Batched causal prefill (attention_prefill.wgsl, fn attention_prefill).
 *   q_batch rows (q_base + i) * q_stride, head slice at h * D
 *   out_batch rows (q_base + i) * out_stride, head slice at h * D
 *   k_cache, v_cache [max_seq, kv_dim], kv head slice at g * D
 *   window of local query i: min(start_pos + q_base + i + 1, max_seq)
 *   rows: local query indices i to compute (NULL -> 0..n_queries-1)
 */
int oracle_prefill(const float *q_batch, const float *k_cache, const float *v_cache,
                   double *out_batch, int n_queries, int H, int G, int D, int kv_dim,
                   int max_seq, float scale, int start_pos, int q_stride, int out_stride,
                   int q_base, const int *rows, int n_rows, int window)
{
    if (bad_heads(H, G, D) || n_queries < 0 || max_seq < 0 || start_pos < 0 || q_base < 0 || window < 0)
        return -1;
    if (kv_dim < G * D || q_stride < H * D || out_stride < H * D) return -1;
    if (rows == NULL) n_rows = n_queries;
    for (int r = 0; r < n_rows; ++r) {
        int i = rows ? rows[r] : r;
        if (i < 0 || i >= n_queries) return -1;
    }
    const int gs = H / G;
    const double sc = (double)scale;
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(max_seq > 0 ? max_seq : 1));
        if (s == NULL) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (int r = 0; r < n_rows; ++r) {
                for (int h = 0; h < H; ++h) {
                    const int i = rows ? rows[r] : r;
                    const size_t q_global = (size_t)q_base + (size_t)i;
                    size_t n = (size_t)start_pos + q_global + 1;
                    if (n > (size_t)max_seq) n = (size_t)max_seq;
                    const int g = h / gs;
                    const size_t lo = window_start(n, window);
                    double m, logl;
                    attend_row(q_batch + q_global * q_stride + (size_t)h * D,
                               k_cache + lo * kv_dim + (size_t)g * D, v_cache + lo * kv_dim + (size_t)g * D,
                               (size_t)kv_dim, n - lo, D, sc, s,
                               out_batch + q_global * out_stride + (size_t)h * D, &m, &logl);
                }
            }
        }
        free(s);
    }
    return err;
}

/*
 * Backward of the forward attention (the pages emit the per-row (max,
 * log-sum) pair for a backward pass -- attention.wgsl header and final LSE
 * store -- but print no backward; this is the plain gradient of the forward
 * definition above).  For a loss L with dL/dout = dout, one (row, head) with
 * kept keys t in [lo, n):
 *
 *   p_t   = softmax_t(s_t),  s_t = scale * q . k_t
 *   dv_t += p_t * dout                       (out = sum_t p_t v_t)
 *   dp_t  = dout . v_t
 *   ds_t  = p_t * (dp_t - sum_u p_u dp_u)    (Jacobian of softmax)
 *   dq    = scale * sum_t ds_t k_t
 *   dk_t += scale * ds_t q
 *
 * dk and dv of kv head g collect every row of every query head h with
 * h / (H/G) == g.  The LSE output itself is not differentiated (its
 * gradient is taken as zero).  Empty windows contribute nothing.
 *   q, dout [q_seq, H*D]; k, v [kv_seq, G*D]
 *   dq [q_seq, H*D]; dk, dv [kv_seq, G*D]  (all written in full)
 *   mask, window: as oracle_forward.
 * Parallel over kv heads only; within a kv head rows are taken in order.
 */
int oracle_backward(const float *q, const float *k, const float *v, const float *dout,
                    double *dq, double *dk, double *dv, int q_seq, int kv_seq,
                    int H, int G, int D, int mask, int window)
{
    if (bad_heads(H, G, D) || q_seq < 0 || kv_seq < 0 || mask < 0 || mask > 2 || window < 0) return -1;
    if (mask != 2 && kv_seq != q_seq) return -1;
    const int gs = H / G;
    const size_t kv_dim = (size_t)G * D;
    const double scale = 1.0 / sqrt((double)D);
    for (size_t i = 0; i < (size_t)q_seq * H * D; ++i) dq[i] = 0.0;
    for (size_t i = 0; i < (size_t)kv_seq * kv_dim; ++i) dk[i] = dv[i] = 0.0;
    int err = 0;
#pragma omp parallel
    {
        const size_t cap = (size_t)(kv_seq > 0 ? kv_seq : 1);
        double *p = (double *)malloc(sizeof(double) * cap);
        double *dp = (double *)malloc(sizeof(double) * cap);
        if (p == NULL || dp == NULL) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int g = 0; g < G; ++g) {
                for (int hh = 0; hh < gs; ++hh) {
                    const int h = g * gs + hh;
                    for (int pos = 0; pos < q_seq; ++pos) {
                        const size_t n = (mask == 0) ? (size_t)pos + 1 : (size_t)kv_seq;
                        const size_t lo = window_start(n, window);
                        if (n == lo) continue;
                        const float *qr = q + (size_t)pos * H * D + (size_t)h * D;
                        const float *dor = dout + (size_t)pos * H * D + (size_t)h * D;
                        double *dqr = dq + (size_t)pos * H * D + (size_t)h * D;
                        /* p = softmax of the scores over the kept keys */
                        double m = -INFINITY;
                        for (size_t t = lo; t < n; ++t) {
                            const float *kt = k + t * kv_dim + (size_t)g * D;
                            double dot = 0.0;
                            for (int d = 0; d < D; ++d) dot += (double)qr[d] * (double)kt[d];
                            p[t] = dot * scale;
                            if (p[t] > m) m = p[t];
                        }
                        double l = 0.0;
                        for (size_t t = lo; t < n; ++t) {
                            p[t] = exp(p[t] - m);
                            l += p[t];
                        }
                        for (size_t t = lo; t < n; ++t) p[t] /= l;
                        /* dp_t = dout . v_t and its p-weighted mean */
                        double mean = 0.0;
                        for (size_t t = lo; t < n; ++t) {
                            const float *vt = v + t * kv_dim + (size_t)g * D;
                            double dot = 0.0;
                            for (int d = 0; d < D; ++d) dot += (double)dor[d] * (double)vt[d];
                            dp[t] = dot;
                            mean += p[t] * dot;
                        }
                        for (size_t t = lo; t < n; ++t) {
                            const double ds = p[t] * (dp[t] - mean);
                            const float *kt = k + t * kv_dim + (size_t)g * D;
                            double *dkt = dk + t * kv_dim + (size_t)g * D;
                            double *dvt = dv + t * kv_dim + (size_t)g * D;
                            for (int d = 0; d < D; ++d) {
                                dqr[d] += scale * ds * (double)kt[d];
                                dkt[d] += scale * ds * (double)qr[d];
                                dvt[d] += p[t] * (double)dor[d];
                            }
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return err;
}

/*
 * Forward with rotary position embedding (RoPE) applied to q and k.  The
 * forward page leaves its RoPE hooks ($ROPE_DECL, $ROPE_Q_APPLY on the query
 * value, $K_VAL_EXPR on each key value) to the host framework, so the
 * convention is this library's reading: pairs (d, d + D/2) for d < D/2
 * rotated by the angle pos * base^(-2d/D),
 *   x'[d]       = x[d] cos(a) - x[d + D/2] sin(a)
 *   x'[d + D/2] = x[d + D/2] cos(a) + x[d] sin(a),
 * with query row i at position i and key row t at position t.  The rotated
 * q and k (fp64) then go through the plain definition above.  D even.
 */
static void rope_rotate(const float *x, double *y, int D, size_t pos, double base)
{
    const int half = D / 2;
    for (int d = 0; d < half; ++d) {
        const double a = (double)pos * pow(base, -2.0 * (double)d / (double)D);
        const double c = cos(a), s = sin(a);
        y[d] = (double)x[d] * c - (double)x[d + half] * s;
        y[d + half] = (double)x[d + half] * c + (double)x[d] * s;
    }
}

int oracle_forward_rope(const float *q, const float *k, const float *v,
                        double *out, double *lse, int q_seq, int kv_seq,
                        int H, int G, int D, int mask, const int *rows, int n_rows, int window,
                        double rope_base)
{
    if (bad_heads(H, G, D) || (D % 2) != 0 || q_seq < 0 || kv_seq < 0 || mask < 0 || mask > 2 || window < 0 ||
        !(rope_base > 1.0))
        return -1;
    if (mask != 2 && kv_seq != q_seq) return -1;
    if (rows == NULL) n_rows = q_seq;
    for (int r = 0; r < n_rows; ++r) {
        int pos = rows ? rows[r] : r;
        if (pos < 0 || pos >= q_seq) return -1;
    }
    const int gs = H / G;
    const size_t kv_dim = (size_t)G * D;
    const double scale = 1.0 / sqrt((double)D);
    /* every key row of every kv head, rotated at its position */
    double *kr = (double *)malloc(sizeof(double) * (kv_seq > 0 ? (size_t)kv_seq * kv_dim : 1));
    if (kr == NULL) return -1;
    for (size_t t = 0; t < (size_t)kv_seq; ++t)
        for (int g = 0; g < G; ++g) rope_rotate(k + t * kv_dim + (size_t)g * D, kr + t * kv_dim + (size_t)g * D, D, t,
                                               rope_base);
    int err = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(kv_seq > 0 ? kv_seq : 1));
        double *qr = (double *)malloc(sizeof(double) * (size_t)D);
        if (s == NULL || qr == NULL) {
#pragma omp atomic write
            err = -1;
        } else {
#pragma omp for collapse(2) schedule(dynamic, 4)
            for (int r = 0; r < n_rows; ++r) {
                for (int h = 0; h < H; ++h) {
                    const int pos = rows ? rows[r] : r;
                    const int g = h / gs;
                    const size_t n = (mask == 0) ? (size_t)pos + 1 : (size_t)kv_seq;
                    const size_t lo = window_start(n, window);
                    const size_t qo = (size_t)pos * H * D + (size_t)h * D;
                    double *o = out + qo;
                    double m = ORACLE_EMPTY_LSE, logl = ORACLE_EMPTY_LSE;
                    if (n == lo) {
                        for (int d = 0; d < D; ++d) o[d] = 0.0;
                    } else {
                        rope_rotate(q + qo, qr, D, (size_t)pos, rope_base);
                        m = -INFINITY;
                        for (size_t t = lo; t < n; ++t) {
                            const double *kt = kr + t * kv_dim + (size_t)g * D;
                            double dot = 0.0;
                            for (int d = 0; d < D; ++d) dot += qr[d] * kt[d];
                            s[t - lo] = dot * scale;
                            if (s[t - lo] > m) m = s[t - lo];
                        }
                        double l = 0.0;
                        for (size_t t = lo; t < n; ++t) {
                            s[t - lo] = exp(s[t - lo] - m);
                            l += s[t - lo];
                        }
                        for (int d = 0; d < D; ++d) {
                            double acc = 0.0;
                            for (size_t t = lo; t < n; ++t) acc += s[t - lo] * (double)v[t * kv_dim + (size_t)g * D + d];
                            o[d] = acc / l;
                        }
                        logl = log(l);
                    }
                    if (lse) {
                        lse[((size_t)pos * H + h) * 2] = m;
                        lse[((size_t)pos * H + h) * 2 + 1] = logl;
                    }
                }
            }
        }
        free(s);
        free(qr);
    }
    free(kr);
    return err;
}

/*
 * Backward of the RoPE forward (oracle_forward_rope).  With q' and k' the
 * turned rows (rotations are orthogonal), the gradient is the plain one of
 * the forward at (q', k', v), turned back: dq = R_q^T dq', dk = R_k^T dk',
 * dv unchanged.  The steps below are those of oracle_backward on fp64 rows.
 */
static void rope_unrotate(double *x, int D, size_t pos, double base)
{
    const int half = D / 2;
    for (int d = 0; d < half; ++d) {
        const double a = (double)pos * pow(base, -2.0 * (double)d / (double)D);
        const double c = cos(a), s = sin(a);
        const double x0 = x[d], x1 = x[d + half];
        x[d] = x0 * c + x1 * s;
        x[d + half] = x1 * c - x0 * s;
    }
}

int oracle_backward_rope(const float *q, const float *k, const float *v, const float *dout,
                         double *dq, double *dk, double *dv, int q_seq, int kv_seq,
                         int H, int G, int D, int mask, int window, double rope_base)
{
    if (bad_heads(H, G, D) || (D % 2) != 0 || q_seq < 0 || kv_seq < 0 || mask < 0 || mask > 2 || window < 0 ||
        !(rope_base > 1.0))
        return -1;
    if (mask != 2 && kv_seq != q_seq) return -1;
    const int gs = H / G;
    const size_t kv_dim = (size_t)G * D;
    const double scale = 1.0 / sqrt((double)D);
    double *qr = (double *)malloc(sizeof(double) * ((size_t)q_seq * H * D + 1));
    double *kr = (double *)malloc(sizeof(double) * ((size_t)kv_seq * kv_dim + 1));
    double *p = (double *)malloc(sizeof(double) * (size_t)(kv_seq > 0 ? kv_seq : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(kv_seq > 0 ? kv_seq : 1));
    if (qr == NULL || kr == NULL || p == NULL || dp == NULL) {
        free(qr); free(kr); free(p); free(dp);
        return -1;
    }
    for (size_t i = 0; i < (size_t)q_seq; ++i)
        for (int h = 0; h < H; ++h) rope_rotate(q + (i * H + h) * D, qr + (i * H + h) * D, D, i, rope_base);
    for (size_t t = 0; t < (size_t)kv_seq; ++t)
        for (int g = 0; g < G; ++g) rope_rotate(k + t * kv_dim + (size_t)g * D, kr + t * kv_dim + (size_t)g * D, D, t,
                                               rope_base);
    for (size_t i = 0; i < (size_t)q_seq * H * D; ++i) dq[i] = 0.0;
    for (size_t i = 0; i < (size_t)kv_seq * kv_dim; ++i) dk[i] = dv[i] = 0.0;
    for (int g = 0; g < G; ++g) {
        for (int hh = 0; hh < gs; ++hh) {
            const int h = g * gs + hh;
            for (int pos = 0; pos < q_seq; ++pos) {
                const size_t n = (mask == 0) ? (size_t)pos + 1 : (size_t)kv_seq;
                const size_t lo = window_start(n, window);
                if (n == lo) continue;
                const double *qrow = qr + (size_t)pos * H * D + (size_t)h * D;
                const float *dor = dout + (size_t)pos * H * D + (size_t)h * D;
                double *dqr = dq + (size_t)pos * H * D + (size_t)h * D;
                double m = -INFINITY;
                for (size_t t = lo; t < n; ++t) {
                    const double *kt = kr + t * kv_dim + (size_t)g * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qrow[d] * kt[d];
                    p[t] = dot * scale;
                    if (p[t] > m) m = p[t];
                }
                double l = 0.0;
                for (size_t t = lo; t < n; ++t) {
                    p[t] = exp(p[t] - m);
                    l += p[t];
                }
                for (size_t t = lo; t < n; ++t) p[t] /= l;
                double mean = 0.0;
                for (size_t t = lo; t < n; ++t) {
                    const float *vt = v + t * kv_dim + (size_t)g * D;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += (double)dor[d] * (double)vt[d];
                    dp[t] = dot;
                    mean += p[t] * dot;
                }
                for (size_t t = lo; t < n; ++t) {
                    const double ds = p[t] * (dp[t] - mean);
                    const double *kt = kr + t * kv_dim + (size_t)g * D;
                    double *dkt = dk + t * kv_dim + (size_t)g * D;
                    double *dvt = dv + t * kv_dim + (size_t)g * D;
                    for (int d = 0; d < D; ++d) {
                        dqr[d] += scale * ds * kt[d];
                        dkt[d] += scale * ds * qrow[d];
                        dvt[d] += p[t] * (double)dor[d];
                    }
                }
            }
        }
    }
    /* back from the turned frame */
    for (size_t i = 0; i < (size_t)q_seq; ++i)
        for (int h = 0; h < H; ++h) rope_unrotate(dq + (i * H + h) * D, D, i, rope_base);
    for (size_t t = 0; t < (size_t)kv_seq; ++t)
        for (int g = 0; g < G; ++g) rope_unrotate(dk + t * kv_dim + (size_t)g * D, D, t, rope_base);
    free(qr); free(kr); free(p); free(dp);
    return 0;
}
