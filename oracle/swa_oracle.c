/*
 * swa_oracle.c -- plain fp64 CPU oracle for causal sliding-window attention,
 * local+strided sparse causal attention and differential causal attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may call this code.  It shares nothing with
 * the CUDA path (no headers, no helpers, no tables) and the CUDA path never
 * calls it.
 *
 * Sources (web pages, cited by title and section):
 *   [AV]   "注意力变体——滑动窗口、稀疏、差分" (Attention variants lesson,
 *          ai-engineering.com.cn, Phase 07 lesson 15), "Build it" steps 1-4.
 *   [AVpt] "Variantes de Atenção — Janela Deslizante, Esparsa, Diferencial"
 *          (ai-engineering.academy), "Atenção Diferencial" (the A1, A2,
 *          DiffAttn formulas) and "Implemente" steps 1-4.
 *   [SWA]  "SWA：滑动窗口注意力与跨层信息传递" (lizn-zn.github.io),
 *          §3.1 (window set N_W(i), mask M^SWA, Attention_SWA), §4.1 (pair counts).
 *
 * What it computes, for every batch b, query head h (key/value head h / g with
 * g = Hq / Hkv) and query row i (0-indexed):
 *   1. the row i of the additive mask, built the way the pages build it:
 *      every entry -inf, then 0 on the allowed keys
 *        causal  : j <= i                                   ([AV] step 1)
 *        window  : max(0, i - W + 1) <= j <= i               ([AV] step 2, [SWA] §3.1)
 *        strided : window  plus  j = 0, s, 2s, ... <= i       ([AV] step 3)
 *        global  : window  plus  the global prefix j < n_g (j <= i); the `stride`
 *                  argument carries n_g for this kind ([AV] "稀疏 / 块注意力": a few
 *                  global tokens such as [CLS] attend to all and are attended by all;
 *                  under the causal mask a global row i < n_g reads every j <= i)
 *   2. z_j = scale * (q_i . k_j) + M_ij in fp64 (masked j give -inf and are not
 *      dotted: -inf + finite = -inf),
 *   3. a two-pass softmax over the row: m = max_j z_j, p_j = exp(z_j - m),
 *      a_j = p_j / sum_j p_j  (each row renormalises inside its own mask,
 *      [SWA] §3.1),
 *   4. out_i = sum_j a_j v_j.
 *   Differential ([AVpt] "Atenção Diferencial"): out_i = sum_j (a1_j - lambda a2_j) v_j
 *   with a1 from (q1, k1) and a2 from (q2, k2), both under the same window mask of width
 *   W; W >= N is the causal mask of the page's formulas, a smaller W a differential head
 *   inside an SWA layer ([AV] opening list: the variants coexist, most layers SWA and a few
 *   differential heads).
 *   Backward (oracle_attn_bwd): the gradients of step 4's output with respect to q, k and
 *   v by the chain rule through the row softmax (written out above that function).
 *   Decode against a rolling cache ([SWA] §4.2): the K, V of absolute position j sit in
 *   cache slot j mod W (the note's 1-indexed slot (i-1) mod W); a query at position t reads
 *   the positions max(0, t-W+1) .. t through their slots, steps 2-4 as above.
 *
 * Inputs are fp64 arrays in layout [B, H, N, d] (q: H = Hq, k and v: H = Hkv).
 * Output is fp64 [B, Hq, nrows, d] where nrows rows (a list, or all N) are computed.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { MASK_WINDOW = 0, MASK_STRIDED = 1, MASK_CAUSAL = 2, MASK_GLOBAL = 3 };

/* Row i of the additive mask, for keys 0..i (keys j > i are -inf in every mask
 * kind, so they are neither stored nor visited). */
static void mask_row(int kind, int64_t i, int64_t window, int64_t stride, double* M) {
    for (int64_t j = 0; j <= i; ++j) M[j] = -INFINITY;
    if (kind == MASK_CAUSAL) {
        for (int64_t j = 0; j <= i; ++j) M[j] = 0.0;
        return;
    }
    int64_t lo = i - window + 1;
    if (lo < 0) lo = 0;
    for (int64_t j = lo; j <= i; ++j) M[j] = 0.0;
    if (kind == MASK_STRIDED) {
        for (int64_t j = 0; j <= i; j += stride) M[j] = 0.0;
    }
    if (kind == MASK_GLOBAL) {
        for (int64_t j = 0; j <= i && j < stride; ++j) M[j] = 0.0;
    }
}

/* Softmax weights a_j (j = 0..i) of one row: steps 2-3 above.  z is scratch. */
static void softmax_row(const double* qi, const double* kh, int64_t d, int64_t i, double scale,
                        const double* M, double* z, double* a) {
    double m = -INFINITY;
    for (int64_t j = 0; j <= i; ++j) {
        if (M[j] == 0.0) {
            const double* kj = kh + j * d;
            double dot = 0.0;
            for (int64_t t = 0; t < d; ++t) dot += qi[t] * kj[t];
            z[j] = scale * dot + M[j];
        } else {
            z[j] = -INFINITY;
        }
        if (z[j] > m) m = z[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j <= i; ++j) {
        a[j] = (z[j] == -INFINITY) ? 0.0 : exp(z[j] - m);
        l += a[j];
    }
    for (int64_t j = 0; j <= i; ++j) a[j] /= l;
}

static int check_shape(int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return 2;
    if (Hq % Hkv != 0) return 2;
    return 0;
}

/*
 * Masked attention, one of the three mask kinds.  rows == NULL computes all N
 * rows (nrows must then equal N).  nthreads <= 0 uses the OpenMP default.
 * Returns 0, or 2 on a bad shape / row index.
 */
int oracle_attn(int kind, const double* q, const double* k, const double* v, double* out,
                int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int64_t W,
                int64_t stride, double scale, const int64_t* rows, int64_t nrows,
                int nthreads) {
    if (check_shape(B, Hq, Hkv, N, d)) return 2;
    if (kind != MASK_WINDOW && kind != MASK_STRIDED && kind != MASK_CAUSAL && kind != MASK_GLOBAL)
        return 2;
    if (kind != MASK_CAUSAL && W < 1) return 2;
    if (kind == MASK_STRIDED && stride < 1) return 2;
    if (kind == MASK_GLOBAL && stride < 0) return 2;
    if (rows == NULL && nrows != N) return 2;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return 2;
    const int64_t g = Hq / Hkv;
    const int64_t total = B * Hq * nrows;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        double* M = (double*)malloc(sizeof(double) * (size_t)N);
        double* z = (double*)malloc(sizeof(double) * (size_t)N);
        double* a = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 8)
        for (int64_t t = 0; t < total; ++t) {
            const int64_t r = t % nrows;
            const int64_t h = (t / nrows) % Hq;
            const int64_t b = t / (nrows * Hq);
            const int64_t i = rows ? rows[r] : r;
            const int64_t hk = h / g;
            const double* qi = q + ((b * Hq + h) * N + i) * d;
            const double* kh = k + (b * Hkv + hk) * N * d;
            const double* vh = v + (b * Hkv + hk) * N * d;
            mask_row(kind, i, W, stride, M);
            softmax_row(qi, kh, d, i, scale, M, z, a);
            double* o = out + ((b * Hq + h) * nrows + r) * d;
            for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
            for (int64_t j = 0; j <= i; ++j) {
                if (a[j] == 0.0) continue;
                const double* vj = vh + j * d;
                for (int64_t c = 0; c < d; ++c) o[c] += a[j] * vj[c];
            }
        }
        free(M);
        free(z);
        free(a);
    }
    return 0;
}

/*
 * Differential attention: out = (A1 - lambda A2) V, A1 = softmax(Q1 K1^T * scale + M),
 * A2 = softmax(Q2 K2^T * scale + M), M the window mask of width W (W >= N: causal).  Same
 * layouts and row selection as oracle_attn.
 */
int oracle_diff(const double* q1, const double* k1, const double* q2, const double* k2,
                const double* v, double lambda, double* out, int64_t B, int64_t Hq, int64_t Hkv,
                int64_t N, int64_t d, int64_t W, double scale, const int64_t* rows,
                int64_t nrows, int nthreads) {
    if (check_shape(B, Hq, Hkv, N, d)) return 2;
    if (W < 1) return 2;
    if (rows == NULL && nrows != N) return 2;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return 2;
    const int64_t g = Hq / Hkv;
    const int64_t total = B * Hq * nrows;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        double* M = (double*)malloc(sizeof(double) * (size_t)N);
        double* z = (double*)malloc(sizeof(double) * (size_t)N);
        double* a1 = (double*)malloc(sizeof(double) * (size_t)N);
        double* a2 = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 8)
        for (int64_t t = 0; t < total; ++t) {
            const int64_t r = t % nrows;
            const int64_t h = (t / nrows) % Hq;
            const int64_t b = t / (nrows * Hq);
            const int64_t i = rows ? rows[r] : r;
            const int64_t hk = h / g;
            const size_t qoff = (size_t)(((b * Hq + h) * N + i) * d);
            const size_t koff = (size_t)((b * Hkv + hk) * N * d);
            mask_row(MASK_WINDOW, i, W, 0, M);
            softmax_row(q1 + qoff, k1 + koff, d, i, scale, M, z, a1);
            softmax_row(q2 + qoff, k2 + koff, d, i, scale, M, z, a2);
            double* o = out + ((b * Hq + h) * nrows + r) * d;
            for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
            for (int64_t j = 0; j <= i; ++j) {
                const double w = a1[j] - lambda * a2[j];
                const double* vj = v + koff + (size_t)(j * d);
                for (int64_t c = 0; c < d; ++c) o[c] += w * vj[c];
            }
        }
        free(M);
        free(z);
        free(a1);
        free(a2);
    }
    return 0;
}

/* The softmax weights of one row (length N; keys after i are 0). */
int oracle_weights_row(int kind, const double* q, const double* k, int64_t B, int64_t Hq,
                       int64_t Hkv, int64_t N, int64_t d, int64_t W, int64_t stride,
                       double scale, int64_t b, int64_t h, int64_t i, double* w) {
    if (check_shape(B, Hq, Hkv, N, d)) return 2;
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= N) return 2;
    if (kind != MASK_CAUSAL && W < 1) return 2;
    if (kind == MASK_STRIDED && stride < 1) return 2;
    if (kind == MASK_GLOBAL && stride < 0) return 2;
    const int64_t hk = h / (Hq / Hkv);
    double* M = (double*)malloc(sizeof(double) * (size_t)N);
    double* z = (double*)malloc(sizeof(double) * (size_t)N);
    mask_row(kind, i, W, stride, M);
    for (int64_t j = 0; j < N; ++j) w[j] = 0.0;
    softmax_row(q + ((b * Hq + h) * N + i) * d, k + (b * Hkv + hk) * N * d, d, i, scale, M, z, w);
    free(M);
    free(z);
    return 0;
}

/* Number of allowed (i, j) pairs of one head: the zeros of the mask, counted row by row. */
int64_t oracle_pair_count(int kind, int64_t N, int64_t W, int64_t stride) {
    if (N < 1 || (kind != MASK_CAUSAL && W < 1) || (kind == MASK_STRIDED && stride < 1) ||
        (kind == MASK_GLOBAL && stride < 0))
        return -1;
    double* M = (double*)malloc(sizeof(double) * (size_t)N);
    int64_t count = 0;
    for (int64_t i = 0; i < N; ++i) {
        mask_row(kind, i, W, stride, M);
        for (int64_t j = 0; j <= i; ++j) count += (M[j] == 0.0);
    }
    free(M);
    return count;
}

/* Row i of the mask as 0/1 allowed flags (length N), for pattern checks. */
int oracle_mask_row(int kind, int64_t N, int64_t W, int64_t stride, int64_t i, uint8_t* allowed) {
    if (i < 0 || i >= N) return 2;
    double* M = (double*)malloc(sizeof(double) * (size_t)N);
    mask_row(kind, i, W, stride, M);
    for (int64_t j = 0; j < N; ++j) allowed[j] = (j <= i && M[j] == 0.0) ? 1 : 0;
    free(M);
    return 0;
}

/*
 * Decode against a rolling W-slot cache ([SWA] §4.2).  q: [B, Hq, d] (one query per
 * sequence and head), kc, vc: [B, Hkv, W, d], pos: [B] absolute position of each query.
 * The window of position t is j = max(0, t-W+1) .. t ([SWA] §3.1, 0-indexed); the key and
 * value of position j are read from slot j mod W, where the rolling writes put them.
 * out: [B, Hq, d].  Returns 0, or 2 on bad arguments.
 */
int oracle_decode(const double* q, const double* kc, const double* vc, const int64_t* pos,
                  double* out, int64_t B, int64_t Hq, int64_t Hkv, int64_t W, int64_t d,
                  double scale) {
    if (check_shape(B, Hq, Hkv, W, d) || W < 1) return 2;
    for (int64_t b = 0; b < B; ++b)
        if (pos[b] < 0) return 2;
    const int64_t g = Hq / Hkv;
    double* z = (double*)malloc(sizeof(double) * (size_t)W);
    for (int64_t b = 0; b < B; ++b) {
        const int64_t t = pos[b];
        const int64_t lo = t - W + 1 > 0 ? t - W + 1 : 0;
        for (int64_t h = 0; h < Hq; ++h) {
            const int64_t hk = h / g;
            const double* qi = q + (b * Hq + h) * d;
            const double* kh = kc + (b * Hkv + hk) * W * d;
            const double* vh = vc + (b * Hkv + hk) * W * d;
            double m = -INFINITY;
            for (int64_t j = lo; j <= t; ++j) {  /* absolute positions of the window */
                const double* kj = kh + (j % W) * d;
                double dot = 0.0;
                for (int64_t c = 0; c < d; ++c) dot += qi[c] * kj[c];
                z[j - lo] = scale * dot;
                if (z[j - lo] > m) m = z[j - lo];
            }
            double l = 0.0;
            for (int64_t j = lo; j <= t; ++j) {
                z[j - lo] = exp(z[j - lo] - m);
                l += z[j - lo];
            }
            double* o = out + (b * Hq + h) * d;
            for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
            for (int64_t j = lo; j <= t; ++j) {
                const double a = z[j - lo] / l;
                const double* vj = vh + (j % W) * d;
                for (int64_t c = 0; c < d; ++c) o[c] += a * vj[c];
            }
        }
    }
    free(z);
    return 0;
}

/*
 * Log-sum-exp of every row's masked scores: lse_i = log sum_j exp(scale q_i . k_j) over the
 * allowed keys of row i (the normaliser of the row softmax, steps 1-3 above), written with the
 * row maximum taken out: m + log sum_j exp(z_j - m).  lse: [B, Hq, nrows].
 */
int oracle_lse(int kind, const double* q, const double* k, double* lse, int64_t B, int64_t Hq,
               int64_t Hkv, int64_t N, int64_t d, int64_t W, int64_t stride, double scale,
               const int64_t* rows, int64_t nrows) {
    if (check_shape(B, Hq, Hkv, N, d)) return 2;
    if (kind != MASK_WINDOW && kind != MASK_STRIDED && kind != MASK_CAUSAL && kind != MASK_GLOBAL)
        return 2;
    if (kind != MASK_CAUSAL && W < 1) return 2;
    if (kind == MASK_STRIDED && stride < 1) return 2;
    if (kind == MASK_GLOBAL && stride < 0) return 2;
    if (rows == NULL && nrows != N) return 2;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return 2;
    const int64_t g = Hq / Hkv;
    double* M = (double*)malloc(sizeof(double) * (size_t)N);
    double* z = (double*)malloc(sizeof(double) * (size_t)N);
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < Hq; ++h)
            for (int64_t r = 0; r < nrows; ++r) {
                const int64_t i = rows ? rows[r] : r;
                const double* qi = q + ((b * Hq + h) * N + i) * d;
                const double* kh = k + (b * Hkv + h / g) * N * d;
                mask_row(kind, i, W, stride, M);
                double m = -INFINITY;
                for (int64_t j = 0; j <= i; ++j) {
                    z[j] = -INFINITY;
                    if (M[j] == 0.0) {
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += qi[c] * kh[j * d + c];
                        z[j] = scale * dot;
                    }
                    if (z[j] > m) m = z[j];
                }
                double sum = 0.0;
                for (int64_t j = 0; j <= i; ++j) sum += (z[j] == -INFINITY) ? 0.0 : exp(z[j] - m);
                lse[(b * Hq + h) * nrows + r] = m + log(sum);
            }
    free(M);
    free(z);
    return 0;
}

/*
 * Gradients of the masked attention forward (the backward pass that training with SWA needs,
 * [AV] exercises 2-3 train models with SWA layers).  For a loss L with dL/dout = dout, the
 * chain rule through out_i = sum_j a_ij v_j and the row softmax a_ij = softmax_j(z_ij),
 * z_ij = scale q_i.k_j + M_ij, gives, row by row:
 *   dv_j  += a_ij dout_i                               (out is linear in v)
 *   da_ij  = dout_i . v_j
 *   dz_ij  = a_ij (da_ij - sum_j' a_ij' da_ij')        (the softmax Jacobian)
 *   dq_i  += scale sum_j dz_ij k_j,   dk_j += scale dz_ij q_i
 * Masked pairs have a_ij = 0 and contribute nothing.  A KV head's dk and dv sum the
 * contributions of all g query heads that read it.  dq: [B, Hq, N, d]; dk, dv: [B, Hkv, N, d].
 */
/*
 * The same gradients restricted to the terms of a subset of query rows (the nrows entries
 * of rows, each in [0, N); rows = NULL means every row): dq holds the rows of the subset
 * (0 elsewhere) and dk, dv hold the sums over the subset's rows only.  Summing the results
 * of a partition of the rows gives the full gradients; a key's dk and dv are complete as
 * soon as the subset holds every row that reads the key.
 */
int oracle_attn_bwd_rows(int kind, const double* q, const double* k, const double* v,
                         const double* dout, double* dq, double* dk, double* dv, int64_t B,
                         int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int64_t W,
                         int64_t stride, double scale, const int64_t* rows, int64_t nrows,
                         int nthreads);

int oracle_attn_bwd(int kind, const double* q, const double* k, const double* v,
                    const double* dout, double* dq, double* dk, double* dv, int64_t B,
                    int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int64_t W, int64_t stride,
                    double scale, int nthreads) {
    return oracle_attn_bwd_rows(kind, q, k, v, dout, dq, dk, dv, B, Hq, Hkv, N, d, W, stride,
                                scale, NULL, N, nthreads);
}

int oracle_attn_bwd_rows(int kind, const double* q, const double* k, const double* v,
                         const double* dout, double* dq, double* dk, double* dv, int64_t B,
                         int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int64_t W,
                         int64_t stride, double scale, const int64_t* rows, int64_t nrows,
                         int nthreads) {
    if (check_shape(B, Hq, Hkv, N, d)) return 2;
    if (rows) {
        if (nrows < 0) return 2;
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= N) return 2;
    } else if (nrows != N) {
        return 2;
    }
    if (kind != MASK_WINDOW && kind != MASK_STRIDED && kind != MASK_CAUSAL && kind != MASK_GLOBAL)
        return 2;
    if (kind != MASK_CAUSAL && W < 1) return 2;
    if (kind == MASK_STRIDED && stride < 1) return 2;
    if (kind == MASK_GLOBAL && stride < 0) return 2;
    const int64_t g = Hq / Hkv;
    memset(dq, 0, sizeof(double) * (size_t)(B * Hq * N * d));
    memset(dk, 0, sizeof(double) * (size_t)(B * Hkv * N * d));
    memset(dv, 0, sizeof(double) * (size_t)(B * Hkv * N * d));
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    /* one (batch, KV head) per task: its dk and dv are written by that task only */
#pragma omp parallel
    {
        double* M = (double*)malloc(sizeof(double) * (size_t)N);
        double* z = (double*)malloc(sizeof(double) * (size_t)N);
        double* a = (double*)malloc(sizeof(double) * (size_t)N);
        double* da = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < B * Hkv; ++t) {
            const int64_t b = t / Hkv, hk = t % Hkv;
            const size_t koff = (size_t)((b * Hkv + hk) * N * d);
            for (int64_t h = hk * g; h < (hk + 1) * g; ++h) {
                for (int64_t r = 0; r < nrows; ++r) {
                    const int64_t i = rows ? rows[r] : r;
                    const size_t qoff = (size_t)(((b * Hq + h) * N + i) * d);
                    mask_row(kind, i, W, stride, M);
                    softmax_row(q + qoff, k + koff, d, i, scale, M, z, a);
                    double delta = 0.0;
                    for (int64_t j = 0; j <= i; ++j) {
                        da[j] = 0.0;
                        if (M[j] != 0.0) continue;  /* masked */
                        const double* vj = v + koff + (size_t)(j * d);
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += dout[qoff + c] * vj[c];
                        da[j] = dot;
                        delta += a[j] * dot;
                    }
                    for (int64_t j = 0; j <= i; ++j) {
                        if (M[j] != 0.0) continue;
                        const double dzj = a[j] * (da[j] - delta);
                        const size_t jo = koff + (size_t)(j * d);
                        for (int64_t c = 0; c < d; ++c) {
                            dq[qoff + c] += scale * dzj * k[jo + c];
                            dk[jo + c] += scale * dzj * q[qoff + c];
                            dv[jo + c] += a[j] * dout[qoff + c];
                        }
                    }
                }
            }
        }
        free(M);
        free(z);
        free(a);
        free(da);
    }
    return 0;
}

/*
 * Gradients of the differential attention forward ([AVpt] "Atenção Diferencial",
 * out = (A1 - lambda_h A2) V, both maps under the window mask of width W, W >= N causal),
 * with one lambda per query head (lams[h]), for an upstream gradient dout.  The chain rule
 * row by row, with da_ij = dout_i . v_j:
 *   dv_j   += (a1_ij - lambda a2_ij) dout_i               (out is linear in v)
 *   dz1_ij  = a1_ij (da_ij - sum_j' a1_ij' da_ij')        (the softmax Jacobian of map 1)
 *   dz2_ij  = a2_ij (-lambda da_ij + lambda sum_j' a2_ij' da_ij')   (map 2 enters with -lambda)
 *   dq1_i  += scale sum_j dz1_ij k1_j,   dk1_j += scale dz1_ij q1_i   (map 2 likewise)
 *   dlam_h += -sum_j a2_ij da_ij                          (d out_i / d lambda = -(A2 V)_i)
 * dk1, dk2, dv of a KV head sum over its query heads; dlam[h] sums over batches and rows.
 */
int oracle_diff_bwd(const double* q1, const double* k1, const double* q2, const double* k2,
                    const double* v, const double* lams, const double* dout, double* dq1,
                    double* dk1, double* dq2, double* dk2, double* dv, double* dlam, int64_t B,
                    int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int64_t W, double scale,
                    int nthreads) {
    if (check_shape(B, Hq, Hkv, N, d)) return 2;
    if (W < 1) return 2;
    const int64_t g = Hq / Hkv;
    const size_t nq = (size_t)(B * Hq * N * d), nk = (size_t)(B * Hkv * N * d);
    memset(dq1, 0, sizeof(double) * nq);
    memset(dq2, 0, sizeof(double) * nq);
    memset(dk1, 0, sizeof(double) * nk);
    memset(dk2, 0, sizeof(double) * nk);
    memset(dv, 0, sizeof(double) * nk);
    double* dlam_bh = (double*)calloc((size_t)(B * Hq), sizeof(double));
    if (!dlam_bh) return 3;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    /* one (batch, KV head) per task: its dk1, dk2, dv and its heads' dlam_bh are its own */
#pragma omp parallel
    {
        double* M = (double*)malloc(sizeof(double) * (size_t)N);
        double* z = (double*)malloc(sizeof(double) * (size_t)N);
        double* a1 = (double*)malloc(sizeof(double) * (size_t)N);
        double* a2 = (double*)malloc(sizeof(double) * (size_t)N);
        double* da = (double*)malloc(sizeof(double) * (size_t)N);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < B * Hkv; ++t) {
            const int64_t b = t / Hkv, hk = t % Hkv;
            const size_t koff = (size_t)((b * Hkv + hk) * N * d);
            for (int64_t h = hk * g; h < (hk + 1) * g; ++h) {
                const double lam = lams[h];
                for (int64_t i = 0; i < N; ++i) {
                    const size_t qoff = (size_t)(((b * Hq + h) * N + i) * d);
                    mask_row(MASK_WINDOW, i, W, 0, M);
                    softmax_row(q1 + qoff, k1 + koff, d, i, scale, M, z, a1);
                    softmax_row(q2 + qoff, k2 + koff, d, i, scale, M, z, a2);
                    double s1 = 0.0, s2 = 0.0;
                    for (int64_t j = 0; j <= i; ++j) {
                        da[j] = 0.0;
                        if (M[j] != 0.0) continue;
                        const double* vj = v + koff + (size_t)(j * d);
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += dout[qoff + c] * vj[c];
                        da[j] = dot;
                        s1 += a1[j] * dot;
                        s2 += a2[j] * dot;
                    }
                    dlam_bh[b * Hq + h] -= s2;
                    for (int64_t j = 0; j <= i; ++j) {
                        if (M[j] != 0.0) continue;
                        const double dz1 = a1[j] * (da[j] - s1);
                        const double dz2 = a2[j] * (-lam * da[j] + lam * s2);
                        const size_t jo = koff + (size_t)(j * d);
                        for (int64_t c = 0; c < d; ++c) {
                            dq1[qoff + c] += scale * dz1 * k1[jo + c];
                            dk1[jo + c] += scale * dz1 * q1[qoff + c];
                            dq2[qoff + c] += scale * dz2 * k2[jo + c];
                            dk2[jo + c] += scale * dz2 * q2[qoff + c];
                            dv[jo + c] += (a1[j] - lam * a2[j]) * dout[qoff + c];
                        }
                    }
                }
            }
        }
        free(M);
        free(z);
        free(a1);
        free(a2);
        free(da);
    }
    for (int64_t h = 0; h < Hq; ++h) {
        dlam[h] = 0.0;
        for (int64_t b = 0; b < B; ++b) dlam[h] += dlam_bh[b * Hq + h];
    }
    free(dlam_bh);
    return 0;
}

/* Slot of absolute position j in a W-slot rolling cache ([SWA] §4.2, 0-indexed). */
int64_t oracle_cache_slot(int64_t j, int64_t W) { return (W < 1 || j < 0) ? -1 : j % W; }

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
