/*
 * FP64 CPU oracle for triangle attention, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (TurboPairFormer, arXiv 2610.05854v1, Abstract): every
 * row-slice i of the N x N pair tensor runs ordinary multi-head attention over
 * its N positions, with a pair bias B[h,j,k] that is the same for all slices.
 * Because the bias is shared, its gradient is the sum over slices of the
 * per-slice score gradient, on top of the usual reductions over queries (dK,
 * dV) and keys (dQ).  The oracle is that definition written out plainly in
 * double precision: for each (batch b, slice i, head h) it materialises the
 * score matrix S, the probabilities P, dP and the score gradient dS, with no
 * tiling, fusion or reordering.
 *
 *   S[j,k]  = scale * sum_c Q[j,c] K[k,c] + bias[b,h,j,k] + mask[b,i,k]
 *   P[j,:]  = softmax_k S[j,:],          LSE[j] = log sum_k exp S[j,k]
 *   O[j,c]  = sum_k P[j,k] V[k,c]
 *   dP[j,k] = sum_c dO[j,c] V[k,c],      D[j] = sum_c dO[j,c] O[j,c]   (exact O)
 *   dS[j,k] = P[j,k] (dP[j,k] - D[j])
 *   dQ = scale dS K,   dK = scale dS^T Q,   dV = P^T dO,   dBias[b,h] = sum_i dS_i
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - scale multiplies Q K^T only, not the bias;
 *  - mask is an additive key mask [B,S,N] (0 or -inf), broadcast over h and j;
 *  - bias is [B,H,N,N]; dBias sums over slices only, never over the batch;
 *  - a row whose keys are all masked has P = 0, O = 0, LSE = -inf and
 *    contributes nothing to any gradient;
 *  - D is formed from the exact (unrounded) forward output: that is the
 *    quantity the residual compensation approximates.
 *
 * Layouts (all contiguous, row-major): Q K V dO O dQ dK dV [B,S,N,H,d];
 * bias dBias [B,H,N,N]; mask [B,S,N]; LSE D [B,S,H,N].
 *
 * Parallelism: OpenMP over independent (b,i,h) work items. dBias is summed in
 * a fixed order (a fixed partition of the slices into chunks, each chunk summed
 * in slice order, then the chunks in chunk order), so results do not depend on
 * the thread count.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

/* Number of slice chunks used for the fixed-order dBias sum. */
#define DBIAS_CHUNKS 16

typedef struct {
    int B, S, N, H, d;
    double scale;
} shape_t;

static size_t x_index(const shape_t *s, int b, int i, int n, int h, int c) {
    return ((((size_t)b * s->S + i) * s->N + n) * s->H + h) * s->d + c;
}

/* Copies the (b,i,h) slice of a [B,S,N,H,d] tensor into a dense [N][d] array. */
static void gather(const shape_t *s, const double *x, int b, int i, int h, double *out) {
    for (int n = 0; n < s->N; ++n)
        for (int c = 0; c < s->d; ++c)
            out[(size_t)n * s->d + c] = x[x_index(s, b, i, n, h, c)];
}

static void scatter(const shape_t *s, double *x, int b, int i, int h, const double *in) {
    for (int n = 0; n < s->N; ++n)
        for (int c = 0; c < s->d; ++c)
            x[x_index(s, b, i, n, h, c)] = in[(size_t)n * s->d + c];
}

/*
 * Forward of one (b,i,h): fills P [N][N], o [N][d] and lse [N].
 * q, k, v are dense [N][d] copies of the slice.
 */
static void slice_forward(const shape_t *s, int b, int i, int h,
                          const double *q, const double *k, const double *v,
                          const double *bias, const double *mask,
                          double *P, double *o, double *lse) {
    const int N = s->N, d = s->d;
    const double *bias_bh = bias + ((size_t)b * s->H + h) * N * N;
    const double *mask_bi = mask ? mask + ((size_t)b * s->S + i) * N : NULL;
    for (int j = 0; j < N; ++j) {
        double *row = P + (size_t)j * N;
        double m = -INFINITY;
        for (int kk = 0; kk < N; ++kk) {
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += q[(size_t)j * d + c] * k[(size_t)kk * d + c];
            double sc = s->scale * dot + bias_bh[(size_t)j * N + kk];
            if (mask_bi) sc += mask_bi[kk];
            row[kk] = sc;
            if (sc > m) m = sc;
        }
        if (m == -INFINITY) {
            /* every key of this row is masked */
            for (int kk = 0; kk < N; ++kk) row[kk] = 0.0;
            lse[j] = -INFINITY;
        } else {
            double l = 0.0;
            for (int kk = 0; kk < N; ++kk) {
                row[kk] = exp(row[kk] - m);
                l += row[kk];
            }
            for (int kk = 0; kk < N; ++kk) row[kk] /= l;
            lse[j] = m + log(l);
        }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int kk = 0; kk < N; ++kk) acc += row[kk] * v[(size_t)kk * d + c];
            o[(size_t)j * d + c] = acc;
        }
    }
}

/*
 * Backward of one (b,i,h) given P and o from slice_forward: fills dS [N][N],
 * dq, dk, dv [N][d] and Dvec [N].
 */
static void slice_backward(const shape_t *s, const double *q, const double *k,
                           const double *v, const double *P, const double *o,
                           const double *dout, double *dS, double *dq, double *dk,
                           double *dv, double *Dvec) {
    const int N = s->N, d = s->d;
    for (int j = 0; j < N; ++j) {
        double Dj = 0.0;
        for (int c = 0; c < d; ++c) Dj += dout[(size_t)j * d + c] * o[(size_t)j * d + c];
        Dvec[j] = Dj;
        for (int kk = 0; kk < N; ++kk) {
            double dp = 0.0;
            for (int c = 0; c < d; ++c) dp += dout[(size_t)j * d + c] * v[(size_t)kk * d + c];
            dS[(size_t)j * N + kk] = P[(size_t)j * N + kk] * (dp - Dj);
        }
    }
    for (int j = 0; j < N; ++j)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int kk = 0; kk < N; ++kk) acc += dS[(size_t)j * N + kk] * k[(size_t)kk * d + c];
            dq[(size_t)j * d + c] = s->scale * acc;
        }
    for (int kk = 0; kk < N; ++kk)
        for (int c = 0; c < d; ++c) {
            double acck = 0.0, accv = 0.0;
            for (int j = 0; j < N; ++j) {
                acck += dS[(size_t)j * N + kk] * q[(size_t)j * d + c];
                accv += P[(size_t)j * N + kk] * dout[(size_t)j * d + c];
            }
            dk[(size_t)kk * d + c] = s->scale * acck;
            dv[(size_t)kk * d + c] = accv;
        }
}

static int check_shape(const shape_t *s) {
    if (s->B <= 0 || s->S <= 0 || s->N <= 0 || s->H <= 0 || s->d <= 0) return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* Forward over the whole tensor: O [B,S,N,H,d] and LSE [B,S,H,N]. */
int oracle_tri_attn_fwd(int B, int S, int N, int H, int d, double scale,
                        const double *Q, const double *K, const double *V,
                        const double *bias, const double *mask,
                        double *O, double *LSE, int nthreads) {
    shape_t s = {B, S, N, H, d, scale};
    if (check_shape(&s) || !Q || !K || !V || !bias || !O || !LSE) return ORACLE_EINVAL;
    if (nthreads > 0) omp_set_num_threads(nthreads);
    const long items = (long)B * S * H;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *q = malloc(sizeof(double) * N * d), *k = malloc(sizeof(double) * N * d);
        double *v = malloc(sizeof(double) * N * d), *o = malloc(sizeof(double) * N * d);
        double *P = malloc(sizeof(double) * (size_t)N * N);
        if (!q || !k || !v || !o || !P) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long it = 0; it < items; ++it) {
                int h = (int)(it % H), i = (int)((it / H) % S), b = (int)(it / ((long)H * S));
                gather(&s, Q, b, i, h, q);
                gather(&s, K, b, i, h, k);
                gather(&s, V, b, i, h, v);
                double *lse = LSE + (((size_t)b * S + i) * H + h) * N;
                slice_forward(&s, b, i, h, q, k, v, bias, mask, P, o, lse);
                scatter(&s, O, b, i, h, o);
            }
        }
        free(q); free(k); free(v); free(o); free(P);
    }
    return err;
}

/*
 * Backward over the whole tensor. Recomputes the forward internally and
 * returns dQ dK dV [B,S,N,H,d], dBias [B,H,N,N] and, when D is not NULL, the
 * exact softmax-backward correction D [B,S,H,N].
 */
int oracle_tri_attn_bwd(int B, int S, int N, int H, int d, double scale,
                        const double *Q, const double *K, const double *V,
                        const double *bias, const double *mask, const double *dO,
                        double *dQ, double *dK, double *dV, double *dBias, double *D,
                        int nthreads) {
    shape_t s = {B, S, N, H, d, scale};
    if (check_shape(&s) || !Q || !K || !V || !bias || !dO || !dQ || !dK || !dV || !dBias)
        return ORACLE_EINVAL;
    if (nthreads > 0) omp_set_num_threads(nthreads);
    const int chunks = S < DBIAS_CHUNKS ? S : DBIAS_CHUNKS;
    const size_t nbias = (size_t)B * H * N * N;
    double *partial = calloc((size_t)chunks * nbias, sizeof(double));
    if (!partial) return ORACLE_ENOMEM;
    /* chunk c holds slices [c*S/chunks, (c+1)*S/chunks) */
    const long items = (long)B * H * chunks;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        size_t nd = (size_t)N * d, nn = (size_t)N * N;
        double *q = malloc(sizeof(double) * nd), *k = malloc(sizeof(double) * nd);
        double *v = malloc(sizeof(double) * nd), *o = malloc(sizeof(double) * nd);
        double *dout = malloc(sizeof(double) * nd), *dq = malloc(sizeof(double) * nd);
        double *dk = malloc(sizeof(double) * nd), *dv = malloc(sizeof(double) * nd);
        double *P = malloc(sizeof(double) * nn), *dS = malloc(sizeof(double) * nn);
        double *lse = malloc(sizeof(double) * N), *Dvec = malloc(sizeof(double) * N);
        if (!q || !k || !v || !o || !dout || !dq || !dk || !dv || !P || !dS || !lse || !Dvec) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long it = 0; it < items; ++it) {
                int c = (int)(it % chunks), h = (int)((it / chunks) % H);
                int b = (int)(it / ((long)chunks * H));
                int i0 = (int)((long)c * S / chunks), i1 = (int)((long)(c + 1) * S / chunks);
                double *acc = partial + (size_t)c * nbias + ((size_t)b * H + h) * nn;
                for (int i = i0; i < i1; ++i) {
                    gather(&s, Q, b, i, h, q);
                    gather(&s, K, b, i, h, k);
                    gather(&s, V, b, i, h, v);
                    gather(&s, dO, b, i, h, dout);
                    slice_forward(&s, b, i, h, q, k, v, bias, mask, P, o, lse);
                    slice_backward(&s, q, k, v, P, o, dout, dS, dq, dk, dv, Dvec);
                    scatter(&s, dQ, b, i, h, dq);
                    scatter(&s, dK, b, i, h, dk);
                    scatter(&s, dV, b, i, h, dv);
                    if (D) memcpy(D + (((size_t)b * S + i) * H + h) * N, Dvec, sizeof(double) * N);
                    for (size_t e = 0; e < nn; ++e) acc[e] += dS[e];
                }
            }
        }
        free(q); free(k); free(v); free(o); free(dout); free(dq); free(dk); free(dv);
        free(P); free(dS); free(lse); free(Dvec);
    }
    if (err == ORACLE_OK) {
        for (size_t e = 0; e < nbias; ++e) {
            double sum = 0.0;
            for (int c = 0; c < chunks; ++c) sum += partial[(size_t)c * nbias + e];
            dBias[e] = sum;
        }
    }
    free(partial);
    return err;
}

/*
 * One (b,i,h) slice, exposing the materialised matrices: P [N][N], dS [N][N]
 * (NULL dO skips the backward and leaves dS untouched).
 */
int oracle_tri_attn_slice(int B, int S, int N, int H, int d, double scale,
                          int b, int i, int h,
                          const double *Q, const double *K, const double *V,
                          const double *bias, const double *mask, const double *dO,
                          double *P, double *dS) {
    shape_t s = {B, S, N, H, d, scale};
    if (check_shape(&s) || b < 0 || b >= B || i < 0 || i >= S || h < 0 || h >= H) return ORACLE_EINVAL;
    if (!Q || !K || !V || !bias || !P) return ORACLE_EINVAL;
    size_t nd = (size_t)N * d;
    double *q = malloc(sizeof(double) * nd), *k = malloc(sizeof(double) * nd);
    double *v = malloc(sizeof(double) * nd), *o = malloc(sizeof(double) * nd);
    double *dout = malloc(sizeof(double) * nd), *dq = malloc(sizeof(double) * nd);
    double *dk = malloc(sizeof(double) * nd), *dv = malloc(sizeof(double) * nd);
    double *lse = malloc(sizeof(double) * N), *Dvec = malloc(sizeof(double) * N);
    int err = ORACLE_OK;
    if (!q || !k || !v || !o || !dout || !dq || !dk || !dv || !lse || !Dvec) {
        err = ORACLE_ENOMEM;
    } else {
        gather(&s, Q, b, i, h, q);
        gather(&s, K, b, i, h, k);
        gather(&s, V, b, i, h, v);
        slice_forward(&s, b, i, h, q, k, v, bias, mask, P, o, lse);
        if (dO && dS) {
            gather(&s, dO, b, i, h, dout);
            slice_backward(&s, q, k, v, P, o, dout, dS, dq, dk, dv, Dvec);
        }
    }
    free(q); free(k); free(v); free(o); free(dout); free(dq); free(dk); free(dv);
    free(lse); free(Dvec);
    return err;
}

/* Threads an OpenMP parallel region uses with the given request (<=0: default). */
int oracle_num_threads(int nthreads) {
    if (nthreads > 0) omp_set_num_threads(nthreads);
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
}

/*
 * dBias for selected rows: for each requested (b, h, j), returns
 * dBias[b,h,j,:] = sum over all slices i of dS_i[j,:], computed directly from
 * query row j of every slice (one row of S, P, dP per slice). Used to check
 * the bias gradient at sizes where the full backward is too slow to run.
 * rows holds nrows triples (b, h, j); out is [nrows][N].
 */
int oracle_tri_attn_dbias_rows(int B, int S, int N, int H, int d, double scale,
                               const double *Q, const double *K, const double *V,
                               const double *bias, const double *mask, const double *dO,
                               const int *rows, int nrows, double *out, int nthreads) {
    shape_t s = {B, S, N, H, d, scale};
    if (check_shape(&s) || !Q || !K || !V || !bias || !dO || !rows || !out || nrows < 0)
        return ORACLE_EINVAL;
    for (int r = 0; r < nrows; ++r)
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= H ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= N)
            return ORACLE_EINVAL;
    if (nthreads > 0) omp_set_num_threads(nthreads);
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double *srow = malloc(sizeof(double) * N), *o = malloc(sizeof(double) * d);
        if (!srow || !o) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int r = 0; r < nrows; ++r) {
                const int b = rows[3 * r], h = rows[3 * r + 1], j = rows[3 * r + 2];
                double *acc = out + (size_t)r * N;
                for (int kk = 0; kk < N; ++kk) acc[kk] = 0.0;
                const double *brow = bias + (((size_t)b * H + h) * N + j) * N;
                for (int i = 0; i < S; ++i) {
                    const double *mrow = mask ? mask + ((size_t)b * S + i) * N : NULL;
                    double m = -INFINITY;
                    for (int kk = 0; kk < N; ++kk) {
                        double dot = 0.0;
                        for (int c = 0; c < d; ++c)
                            dot += Q[x_index(&s, b, i, j, h, c)] * K[x_index(&s, b, i, kk, h, c)];
                        double sc = scale * dot + brow[kk];
                        if (mrow) sc += mrow[kk];
                        srow[kk] = sc;
                        if (sc > m) m = sc;
                    }
                    if (m == -INFINITY) continue; /* fully masked row: no contribution */
                    double l = 0.0;
                    for (int kk = 0; kk < N; ++kk) { srow[kk] = exp(srow[kk] - m); l += srow[kk]; }
                    for (int kk = 0; kk < N; ++kk) srow[kk] /= l; /* srow is now P[j,:] */
                    for (int c = 0; c < d; ++c) {
                        double a = 0.0;
                        for (int kk = 0; kk < N; ++kk) a += srow[kk] * V[x_index(&s, b, i, kk, h, c)];
                        o[c] = a;
                    }
                    double Dj = 0.0;
                    for (int c = 0; c < d; ++c) Dj += dO[x_index(&s, b, i, j, h, c)] * o[c];
                    for (int kk = 0; kk < N; ++kk) {
                        double dp = 0.0;
                        for (int c = 0; c < d; ++c)
                            dp += dO[x_index(&s, b, i, j, h, c)] * V[x_index(&s, b, i, kk, h, c)];
                        acc[kk] += srow[kk] * (dp - Dj);
                    }
                }
            }
        }
        free(srow); free(o);
    }
    return err;
}
