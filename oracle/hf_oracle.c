/*
 * hf_oracle.c -- plain, slow CPU oracle for the hybrid attention step of
 * Hybrid Forcing ("Long-Horizon Streaming Video Generation via Hybrid
 * Attention with Decoupled Distillation").
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header or table with the CUDA
 * library; it sees the same seeded inputs and nothing else.
 *
 * What it computes, step by step (every input is a bf16 value, exact in
 * float and double):
 *
 *  1. Geometry.  Window frames w = 0..n_win-1, oldest first; the query
 *     chunk is the last C of them.  Blocks tile each frame on its own from
 *     its first token: block j of a frame covers tokens
 *     [j*beta, min((j+1)*beta, N_f)), so the last block may be partial.
 *     Key block kb = w*bpf + j, query block qb = c*bpf + j (c = chunk-local
 *     frame), bpf = ceil(N_f / beta).
 *  2. Block importance scores (English technical summary, section 2.A.2,
 *     "Block-Sparse Sliding Window Attention": block importance scores are
 *     computed and only the top-K blocks are kept).  Reading taken: the
 *     score of a (query block, key block) pair is the dot product of the
 *     blocks' mean-pooled query and key vectors.  Because exact top-K
 *     indices are compared bit for bit, the arithmetic of the selection is
 *     fixed in float32: the mean is a sequential float sum in ascending
 *     token order divided (IEEE RN) by the token count, and the score is a
 *     sequential fused multiply-add chain over channels in ascending order,
 *     with -0 mapped to +0.
 *  3. Top-K per query block: order key blocks by (score desc, index asc),
 *     keep the first K, report them in ascending index order.
 *  4. Block-sparse softmax attention (same section): for each query token,
 *     softmax(scale * q.k) over the tokens of its query block's selected key
 *     blocks, times V; scale = 1/sqrt(d).  No other mask inside the window.
 *     Double precision.
 *  5. Linear temporal attention state (English technical summary, section
 *     2.A.1 "Linear Temporal Attention"; arXiv abstract: a compact key-value
 *     state incrementally absorbs evicted tokens).  Reading taken: the
 *     kernelised linear attention of Katharopoulos et al. (2020), with
 *     S = sum_t phi(k_t) v_t^T (row = key feature, column = value channel),
 *     z = sum_t phi(k_t), phi(x) = elu(x) + 1.  Double precision.
 *  6. Linear read: o_lin = phi(q)^T S / (phi(q)^T z + eps).
 *  7. Output = o_swa + o_lin (Spanish technical summary, section 2.A: the
 *     final output is the sum of the compressed history and the sparse
 *     local attention).
 *
 *  8. Relative temporal RoPE (English technical summary, section 2.C
 *     "Stability Enhancements": temporal RoPE indices are kept under a fixed
 *     upper bound in training and inference, positions taken as relative
 *     offsets).  Readings taken: the rotary embedding of Su et al.
 *     (RoFormer, 2021) on channel pairs (2i, 2i+1), i < rot_dims/2, angle
 *     p * base^(-2i/rot_dims); the temporal index p of a token is its
 *     frame's offset inside the current window, clamped to [0, max_offset];
 *     channels >= rot_dims pass unchanged.  Double precision.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -shared -fPIC.
 * -ffp-contract=off keeps every float add and multiply separately rounded;
 * fmaf() is the C library's correctly rounded fused multiply-add.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static float bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static int ceil_div(int a, int b) { return (a + b - 1) / b; }

int hfo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- step 1+2: mean pooling (float32, sequential) ---------------------- */
/* x: [n_frames][nf][d] bf16 of one head.  out: [n_frames*bpf][d] float. */
void hfo_pool(const uint16_t *x, int n_frames, int nf, int d, int beta, float *out)
{
    int bpf = ceil_div(nf, beta);
    for (int f = 0; f < n_frames; ++f)
        for (int j = 0; j < bpf; ++j) {
            int t0 = j * beta;
            int t1 = t0 + beta < nf ? t0 + beta : nf;
            float n = (float)(t1 - t0);
            for (int c = 0; c < d; ++c) {
                float acc = 0.0f;
                for (int t = t0; t < t1; ++t)
                    acc = acc + bf16_to_float(x[((size_t)f * nf + t) * d + c]);
                out[((size_t)f * bpf + j) * d + c] = acc / n;
            }
        }
}

/* ---- step 2: scores (float32 FMA chain) -------------------------------- */
void hfo_scores(const float *qp, int nqb, const float *kp, int nkb, int d, float *s)
{
    for (int qb = 0; qb < nqb; ++qb)
        for (int kb = 0; kb < nkb; ++kb) {
            float acc = 0.0f;
            for (int c = 0; c < d; ++c)
                acc = fmaf(qp[(size_t)qb * d + c], kp[(size_t)kb * d + c], acc);
            s[(size_t)qb * nkb + kb] = acc + 0.0f;   /* -0 -> +0 */
        }
}

/* ---- step 3: top-K ----------------------------------------------------- */
typedef struct { float s; int32_t i; } scored_t;

static int by_score_desc_index_asc(const void *pa, const void *pb)
{
    const scored_t *a = (const scored_t *)pa, *b = (const scored_t *)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

static int by_index(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* Returns 0, or -1 if a score is not finite or k is out of [1, nkb]. */
int hfo_topk(const float *s, int nqb, int nkb, int k, int32_t *idx)
{
    if (k < 1 || k > nkb) return -1;
    scored_t *row = (scored_t *)malloc(sizeof(scored_t) * (size_t)nkb);
    if (!row) return -1;
    for (int qb = 0; qb < nqb; ++qb) {
        for (int kb = 0; kb < nkb; ++kb) {
            float v = s[(size_t)qb * nkb + kb];
            if (!isfinite(v)) { free(row); return -1; }
            row[kb].s = v;
            row[kb].i = kb;
        }
        qsort(row, (size_t)nkb, sizeof(scored_t), by_score_desc_index_asc);
        int32_t *out = idx + (size_t)qb * k;
        for (int m = 0; m < k; ++m) out[m] = row[m].i;
        qsort(out, (size_t)k, sizeof(int32_t), by_index);
    }
    free(row);
    return 0;
}

/* Diagnostic: double-precision scores of the same pooled blocks, and for each
 * query block the gap between the K-th and (K+1)-th largest score (0 if
 * K = nkb).  Small gaps flag rows where a different rounding could change the
 * selection; the selection itself is defined by the float32 arithmetic. */
void hfo_score_margin(const float *qp, int nqb, const float *kp, int nkb, int d, int k,
                      double *margin)
{
    double *row = (double *)malloc(sizeof(double) * (size_t)nkb);
    for (int qb = 0; qb < nqb; ++qb) {
        for (int kb = 0; kb < nkb; ++kb) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += (double)qp[(size_t)qb * d + c] * (double)kp[(size_t)kb * d + c];
            row[kb] = acc;
        }
        if (k >= nkb) { margin[qb] = 0.0; continue; }
        /* k-th and (k+1)-th largest by repeated selection (nkb is small) */
        double kth = 0.0, next = 0.0;
        char *used = (char *)calloc((size_t)nkb, 1);
        for (int r = 0; r <= k; ++r) {
            int best = -1;
            for (int kb = 0; kb < nkb; ++kb)
                if (!used[kb] && (best < 0 || row[kb] > row[best])) best = kb;
            used[best] = 1;
            if (r == k - 1) kth = row[best];
            if (r == k) next = row[best];
        }
        free(used);
        margin[qb] = kth - next;
    }
    free(row);
}

/* ---- step 5/6: feature map, state, linear read (double) ---------------- */
static double phi(double x) { return x > 0.0 ? x + 1.0 : exp(x); }

/* S [d][d] += sum_t phi(k_t) v_t^T ; z [d] += sum_t phi(k_t).  k, v: [n][d]. */
void hfo_absorb(double *S, double *z, const uint16_t *k, const uint16_t *v, int n, int d)
{
    double *pk = (double *)malloc(sizeof(double) * (size_t)d);
    for (int t = 0; t < n; ++t) {
        for (int c = 0; c < d; ++c) pk[c] = phi((double)bf16_to_float(k[(size_t)t * d + c]));
        for (int c = 0; c < d; ++c) {
            z[c] += pk[c];
            for (int j = 0; j < d; ++j)
                S[(size_t)c * d + j] += pk[c] * (double)bf16_to_float(v[(size_t)t * d + j]);
        }
    }
    free(pk);
}

/* All heads: S [BH][d][d], z [BH][d] += the state of k, v [BH][n][d]. */
void hfo_absorb_heads(int BH, double *S, double *z, const uint16_t *k, const uint16_t *v,
                      int n, int d)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < BH; ++h)
        hfo_absorb(S + (size_t)h * d * d, z + (size_t)h * d, k + (size_t)h * n * d,
                   v + (size_t)h * n * d, n, d);
}

/* o [d] = phi(q)^T S / (phi(q)^T z + eps) for one query row q [d]. */
static void linear_read_row(const uint16_t *q, const double *S, const double *z, int d,
                            double eps, double *pq, double *o)
{
    double den = eps;
    for (int c = 0; c < d; ++c) {
        pq[c] = phi((double)bf16_to_float(q[c]));
        den += pq[c] * z[c];
    }
    for (int j = 0; j < d; ++j) {
        double num = 0.0;
        for (int c = 0; c < d; ++c) num += pq[c] * S[(size_t)c * d + j];
        o[j] = num / den;
    }
}

void hfo_linear_read(const uint16_t *q, int nq, const double *S, const double *z, int d,
                     double eps, double *o)
{
    double *pq = (double *)malloc(sizeof(double) * (size_t)d);
    for (int i = 0; i < nq; ++i)
        linear_read_row(q + (size_t)i * d, S, z, d, eps, pq, o + (size_t)i * d);
    free(pq);
}

/* ---- step 4: block-sparse softmax attention for one query row ---------- */
/* q row [d]; k, v: logical window [n_win*nf][d]; sel: the K selected key
 * blocks of this row's query block.  lbuf: scratch of K*beta doubles. */
static void sparse_attn_row(const uint16_t *qrow, const uint16_t *k, const uint16_t *v,
                            int nf, int d, int beta, const int32_t *sel, int kk,
                            double scale, double *lbuf, double *o)
{
    int bpf = ceil_div(nf, beta);
    int n = 0;
    double m = -INFINITY;
    for (int s = 0; s < kk; ++s) {
        int w = sel[s] / bpf, jb = sel[s] % bpf;
        int t0 = jb * beta, t1 = t0 + beta < nf ? t0 + beta : nf;
        for (int t = t0; t < t1; ++t) {
            const uint16_t *krow = k + ((size_t)w * nf + t) * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += (double)bf16_to_float(qrow[c]) * (double)bf16_to_float(krow[c]);
            lbuf[n] = scale * dot;
            if (lbuf[n] > m) m = lbuf[n];
            ++n;
        }
    }
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    double l = 0.0;
    n = 0;
    for (int s = 0; s < kk; ++s) {
        int w = sel[s] / bpf, jb = sel[s] % bpf;
        int t0 = jb * beta, t1 = t0 + beta < nf ? t0 + beta : nf;
        for (int t = t0; t < t1; ++t) {
            double p = exp(lbuf[n++] - m);
            const uint16_t *vrow = v + ((size_t)w * nf + t) * d;
            l += p;
            for (int c = 0; c < d; ++c) o[c] += p * (double)bf16_to_float(vrow[c]);
        }
    }
    for (int c = 0; c < d; ++c) o[c] /= l;
}

/* Sparse attention of the listed query rows of one head (rows == NULL: all
 * C*nf rows).  q [C*nf][d], k/v [n_win*nf][d], idx [C*bpf][kk]. */
void hfo_sparse_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, int C, int nf,
                     int d, int beta, const int32_t *idx, int kk, double scale,
                     const int32_t *rows, int n_rows, double *o)
{
    int bpf = ceil_div(nf, beta);
    int total = rows ? n_rows : C * nf;
    if (scale == 0.0) scale = 1.0 / sqrt((double)d);
#pragma omp parallel
    {
        double *lbuf = (double *)malloc(sizeof(double) * (size_t)kk * beta);
#pragma omp for schedule(dynamic, 16)
        for (int r = 0; r < total; ++r) {
            int i = rows ? rows[r] : r;
            int qb = (i / nf) * bpf + (i % nf) / beta;
            sparse_attn_row(q + (size_t)i * d, k, v, nf, d, beta, idx + (size_t)qb * kk, kk,
                            scale, lbuf, o + (size_t)r * d);
        }
        free(lbuf);
    }
}

/* ---- the whole step, all heads ----------------------------------------- */
/* Q [BH][C*nf][d]; K, V [BH][n_win*nf][d] (logical window order);
 * S [BH][d][d], z [BH][d] (double; may be NULL for an empty state).
 * rows: query rows to evaluate (NULL: all).  Outputs: idx [BH][C*bpf][kk],
 * O [BH][n_rows][d] = o_swa + o_lin, and optionally O_swa, O_lin split out
 * (same shape) and margin [BH][C*bpf].  Returns 0, or -1 on a bad argument
 * or a non-finite score. */
int hfo_hybrid_forward(int BH, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                       const double *S, const double *z, int C, int n_win, int nf, int d,
                       int beta, int kk, double scale, double eps, const int32_t *rows,
                       int n_rows, int32_t *idx, double *O, double *O_swa, double *O_lin,
                       double *margin)
{
    int bpf = ceil_div(nf, beta);
    int nqb = C * bpf, nkb = n_win * bpf;
    int total = rows ? n_rows : C * nf;
    if (C < 1 || n_win < C || kk < 1 || kk > nkb || beta < 1 || d < 1) return -1;
    if (scale == 0.0) scale = 1.0 / sqrt((double)d);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int h = 0; h < BH; ++h) {
        float *qp = (float *)malloc(sizeof(float) * (size_t)nqb * d);
        float *kp = (float *)malloc(sizeof(float) * (size_t)nkb * d);
        float *sc = (float *)malloc(sizeof(float) * (size_t)nqb * nkb);
        const uint16_t *Qh = Q + (size_t)h * C * nf * d;
        const uint16_t *Kh = K + (size_t)h * n_win * nf * d;
        hfo_pool(Qh, C, nf, d, beta, qp);
        hfo_pool(Kh, n_win, nf, d, beta, kp);
        hfo_scores(qp, nqb, kp, nkb, d, sc);
        if (hfo_topk(sc, nqb, nkb, kk, idx + (size_t)h * nqb * kk) != 0) bad |= 1;
        if (margin) hfo_score_margin(qp, nqb, kp, nkb, d, kk, margin + (size_t)h * nqb);
        free(qp); free(kp); free(sc);
    }
    if (bad) return -1;
#pragma omp parallel
    {
        double *lbuf = (double *)malloc(sizeof(double) * (size_t)kk * beta);
        double *pq = (double *)malloc(sizeof(double) * (size_t)d);
        double *ol = (double *)malloc(sizeof(double) * (size_t)d);
        double *os = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 16) collapse(2)
        for (int h = 0; h < BH; ++h)
            for (int r = 0; r < total; ++r) {
                int i = rows ? rows[r] : r;
                int qb = (i / nf) * bpf + (i % nf) / beta;
                const uint16_t *qrow = Q + ((size_t)h * C * nf + i) * d;
                sparse_attn_row(qrow, K + (size_t)h * n_win * nf * d, V + (size_t)h * n_win * nf * d,
                                nf, d, beta, idx + ((size_t)h * nqb + qb) * kk, kk, scale, lbuf, os);
                if (S && z)
                    linear_read_row(qrow, S + (size_t)h * d * d, z + (size_t)h * d, d, eps, pq, ol);
                else
                    for (int c = 0; c < d; ++c) ol[c] = 0.0;
                size_t off = ((size_t)h * total + r) * d;
                for (int c = 0; c < d; ++c) {
                    O[off + c] = os[c] + ol[c];
                    if (O_swa) O_swa[off + c] = os[c];
                    if (O_lin) O_lin[off + c] = ol[c];
                }
            }
        free(lbuf); free(pq); free(ol); free(os);
    }
    return 0;
}

/* Step 8: x [BH][F][nf][d] bf16 -> y fp64, frame f rotated by the clamped
 * offset offsets[f]. */
void hfo_rope_relative(const uint16_t *x, int BH, int F, int nf, int d, const int32_t *offsets,
                       int max_offset, int rot_dims, double base, double *y)
{
    for (int h = 0; h < BH; ++h)
        for (int f = 0; f < F; ++f) {
            int p = offsets[f];
            if (p < 0) p = 0;
            if (p > max_offset) p = max_offset;
            for (int t = 0; t < nf; ++t) {
                const size_t row = (((size_t)h * F + f) * nf + t) * d;
                for (int c = 0; c < d; ++c) y[row + c] = bf16_to_float(x[row + c]);
                for (int i = 0; i < rot_dims / 2; ++i) {
                    const double ang = (double)p * pow(base, -2.0 * i / rot_dims);
                    const double x0 = y[row + 2 * i], x1 = y[row + 2 * i + 1];
                    y[row + 2 * i] = x0 * cos(ang) - x1 * sin(ang);
                    y[row + 2 * i + 1] = x0 * sin(ang) + x1 * cos(ang);
                }
            }
        }
}
