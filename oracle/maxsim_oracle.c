/*
 * CPU oracle for the MaxSim operator -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct restatement of what the operator computes,
 * accumulated in double (int64 for the INT8 variant). It shares no code,
 * header, table or helper with the CUDA library; only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it. Nothing in the
 * product path calls it.
 *
 * Sources (page title, section / equation):
 *  - "Flash-MaxSim" paper, Sec. 1 Eq. (1): score = sum over query tokens of the
 *    max over document tokens of <Q_s, D_t>.
 *  - "late-interaction-kernels" design notes, "Problem": score[i,j] over
 *    batches Q [Nq,Lq,d], D [Nd,Ld,d]; q_mask drops query rows from the sum,
 *    d_mask hides document tokens from the inner max.
 *  - same notes, "Forward" and "Mask handling": masked positions become -inf
 *    before the max; after the max, a non-finite m or an inactive query row
 *    contributes 0; argmax keeps the lowest index among ties.
 *  - same notes, "Varlen / packed path": packed tokens with cu_seqlens offsets;
 *    an empty sequence contributes zero.
 *  - "Flash-MaxSim" Sec. 4.3.1: per-token symmetric INT8 quantisation with the
 *    dequantisation applied to the scores.
 *  - "Flash-MaxSim" Sec. 4.2.1 Eqs. (2)-(3): gradient gather for Q and scatter
 *    for D through the saved argmax, multiplied by q_mask (design notes,
 *    "Backward"); Sec. 4.2.2: inverse map as a CSR built by bincount, cumsum
 *    and a stable ordering of sources; Sec. 4.2.3: destination-owned sums.
 *
 * Readings where the pages are silent (each also listed in the design notes of
 * this repository):
 *  - A query row with no valid document token (empty document or all tokens
 *    masked) contributes 0 and reports argmax -1 (not 0), so that the
 *    backward routes no gradient through it.
 *  - The argmax of an inactive query row (q_mask = 0) is still computed.
 *  - INT8: the max is taken over dequantised values dot * d_scale[t]; the
 *    positive q_scale[s] multiplies the row maximum.
 *  - Masked query rows still enter the CSR (their weight is 0).
 *  - Chamfer: with an empty point set both terms are 0 and every point
 *    reports nearest index -1 (distance 0).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- exact decoding of the storage formats (IEEE 754 definitions) -------- */

/* binary16: sign, 5-bit exponent with bias 15, 10-bit fraction. */
static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);            /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f | 0x400), e - 25); /* (1024 + f) * 2^(e-15-10) */
    }
    return sign ? -v : v;
}

/* bfloat16: sign, 8-bit exponent with bias 127, 7-bit fraction. */
static double decode_bf16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int f = h & 0x7F;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);           /* subnormal: f * 2^(-126-7) */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f | 0x80), e - 134); /* (128 + f) * 2^(e-127-7) */
    }
    return sign ? -v : v;
}

/* dtype: 0 = binary16, 1 = bfloat16, 2 = float64 (the last is for pins). */
static double load_elem(const void *base, int dtype, int64_t idx) {
    switch (dtype) {
    case 0: return decode_f16(((const uint16_t *)base)[idx]);
    case 1: return decode_bf16(((const uint16_t *)base)[idx]);
    default: return ((const double *)base)[idx];
    }
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Forward MaxSim over packed token rows.
 *
 *   Q rows of query i:   q_off[i] .. q_off[i+1]-1  (dim values each)
 *   D rows of doc j:     d_off[j] .. d_off[j+1]-1
 *   q_mask / d_mask:     one byte per packed row (nonzero = active), or NULL
 *   docs:                the documents to score (n_sel of them), or NULL = all
 *
 * Outputs for query i and selected document c (doc j = docs[c]):
 *   scores[i*n_sel + c]               sum over active rows of the row maximum
 *   argmax[(i*n_sel + c)*lq_stride+s] lowest t attaining the maximum, or -1
 *   gap[(i*n_sel + c)*lq_stride + s]  maximum minus the second largest value
 *                                     (+inf with fewer than two valid tokens)
 * argmax and gap may be NULL. Rows s >= Lq_i are filled with -1 / +inf.
 */
int oracle_fwd(const void *Q, const void *D, int dtype, int64_t Nq, const int64_t *q_off,
               int64_t Nd, const int64_t *d_off, int64_t dim, const uint8_t *q_mask,
               const uint8_t *d_mask, const int64_t *docs, int64_t n_sel, double *scores,
               int32_t *argmax, double *gap, int64_t lq_stride, int nthreads) {
    if (Nq < 0 || Nd < 0 || dim <= 0 || n_sel < 0) return 1;
    set_threads(nthreads);
    int64_t npairs = Nq * n_sel;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int64_t pair = 0; pair < npairs; ++pair) {
        int64_t i = pair / n_sel;
        int64_t c = pair % n_sel;
        int64_t j = docs ? docs[c] : c;
        int64_t lq = q_off[i + 1] - q_off[i];
        int64_t ld = d_off[j + 1] - d_off[j];
        /* decode this pair's rows once into doubles */
        double *qv = (double *)malloc((size_t)(lq > 0 ? lq : 1) * (size_t)dim * sizeof(double));
        double *dv = (double *)malloc((size_t)(ld > 0 ? ld : 1) * (size_t)dim * sizeof(double));
        if (!qv || !dv) { free(qv); free(dv); failed = 1; continue; }
        for (int64_t s = 0; s < lq; ++s)
            for (int64_t k = 0; k < dim; ++k) qv[s * dim + k] = load_elem(Q, dtype, (q_off[i] + s) * dim + k);
        for (int64_t t = 0; t < ld; ++t)
            for (int64_t k = 0; k < dim; ++k) dv[t * dim + k] = load_elem(D, dtype, (d_off[j] + t) * dim + k);
        double score = 0.0;
        for (int64_t s = 0; s < lq; ++s) {
            double best = -INFINITY, second = -INFINITY;
            int32_t best_t = -1;
            for (int64_t t = 0; t < ld; ++t) {
                if (d_mask && !d_mask[d_off[j] + t]) continue;
                double v = 0.0;
                for (int64_t k = 0; k < dim; ++k) v += qv[s * dim + k] * dv[t * dim + k];
                if (best_t < 0 || v > best) {
                    second = best;
                    best = v;
                    best_t = (int32_t)t;
                } else if (v > second) {
                    second = v;
                }
            }
            int active = q_mask ? (q_mask[q_off[i] + s] != 0) : 1;
            if (active && best_t >= 0) score += best;
            if (argmax) argmax[pair * lq_stride + s] = best_t;
            if (gap) gap[pair * lq_stride + s] = (best_t >= 0 && second > -INFINITY) ? best - second : INFINITY;
        }
        for (int64_t s = lq; s < lq_stride; ++s) {
            if (argmax) argmax[pair * lq_stride + s] = -1;
            if (gap) gap[pair * lq_stride + s] = INFINITY;
        }
        scores[pair] = score;
        free(qv);
        free(dv);
    }
    return failed ? 4 : 0;
}

/*
 * INT8 x INT8 forward, dense layout Q [Nq,Lq,dim], D [Nd,Ld,dim] (int8) with
 * one float scale per token. For each (i,j,s):
 *   dot_t = sum_k q8[i,s,k] * d8[j,t,k]                (exact, int64)
 *   v_t   = dot_t * d_scale[j,t]                       (double)
 *   m_s   = max over valid t of v_t, lowest t on ties
 *   score = sum over active s with a valid t of q_scale[i,s] * m_s
 * win_dot[(i*n_sel+c)*Lq + s] receives dot at the argmax (0 if none); returns
 * 2 if any dot does not fit int32.
 */
int oracle_fwd_int8(const int8_t *Q, const float *q_scale, const int8_t *D, const float *d_scale,
                    int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld, int64_t dim,
                    const uint8_t *q_mask, const uint8_t *d_mask, const int64_t *docs,
                    int64_t n_sel, double *scores, int32_t *argmax, int32_t *win_dot, double *gap,
                    int nthreads) {
    if (Nq < 0 || Nd < 0 || Lq < 0 || Ld < 0 || dim <= 0 || n_sel < 0) return 1;
    set_threads(nthreads);
    int64_t npairs = Nq * n_sel;
    int overflow = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : overflow)
    for (int64_t pair = 0; pair < npairs; ++pair) {
        int64_t i = pair / n_sel;
        int64_t c = pair % n_sel;
        int64_t j = docs ? docs[c] : c;
        double score = 0.0;
        for (int64_t s = 0; s < Lq; ++s) {
            int64_t qrow = i * Lq + s;
            double best = -INFINITY, second = -INFINITY;
            int32_t best_t = -1;
            int64_t best_dot = 0;
            for (int64_t t = 0; t < Ld; ++t) {
                int64_t drow = j * Ld + t;
                if (d_mask && !d_mask[drow]) continue;
                int64_t dot = 0;
                for (int64_t k = 0; k < dim; ++k)
                    dot += (int64_t)Q[qrow * dim + k] * (int64_t)D[drow * dim + k];
                if (dot > INT32_MAX || dot < INT32_MIN) overflow = 1;
                double v = (double)dot * (double)d_scale[drow];
                if (best_t < 0 || v > best) {
                    second = best;
                    best = v;
                    best_t = (int32_t)t;
                    best_dot = dot;
                } else if (v > second) {
                    second = v;
                }
            }
            int active = q_mask ? (q_mask[qrow] != 0) : 1;
            if (active && best_t >= 0) score += (double)q_scale[qrow] * best;
            if (argmax) argmax[pair * Lq + s] = best_t;
            if (win_dot) win_dot[pair * Lq + s] = (int32_t)best_dot;
            if (gap) gap[pair * Lq + s] = (best_t >= 0 && second > -INFINITY) ? best - second : INFINITY;
        }
        scores[pair] = score;
    }
    return overflow ? 2 : 0;
}

/*
 * Inverse-argmax CSR (Flash-MaxSim Sec. 4.2.2). Source p = (i*Nd + j)*Lq + s
 * with a = argmax[p] != -1 points at destination row j*Ld + a.
 *   row_ptr = exclusive prefix sum of the per-destination counts (bincount,
 *             then cumsum), length Nd*Ld + 1
 *   col     = the sources of each destination in ascending p (a stable
 *             ordering of the flattened destinations)
 * Returns 3 if an argmax lies outside [-1, Ld).
 */
int oracle_csr(const int32_t *argmax, int64_t Nq, int64_t Lq, int64_t Nd, int64_t Ld,
               int32_t *row_ptr, int32_t *col) {
    int64_t nsrc = Nq * Nd * Lq;
    int64_t ndst = Nd * Ld;
    int64_t *count = (int64_t *)calloc((size_t)ndst + 1, sizeof(int64_t));
    int64_t *fill = (int64_t *)calloc((size_t)ndst + 1, sizeof(int64_t));
    if (!count || !fill) { free(count); free(fill); return 4; }
    for (int64_t p = 0; p < nsrc; ++p) {
        int32_t a = argmax[p];
        if (a == -1) continue;
        if (a < -1 || a >= Ld) { free(count); free(fill); return 3; }
        int64_t j = (p / Lq) % Nd;
        count[j * Ld + a] += 1;
    }
    int64_t run = 0;
    for (int64_t r = 0; r < ndst; ++r) {
        row_ptr[r] = (int32_t)run;
        run += count[r];
    }
    row_ptr[ndst] = (int32_t)run;
    for (int64_t p = 0; p < nsrc; ++p) { /* ascending p: stable */
        int32_t a = argmax[p];
        if (a == -1) continue;
        int64_t j = (p / Lq) % Nd;
        int64_t r = j * Ld + a;
        col[row_ptr[r] + fill[r]] = (int32_t)p;
        fill[r] += 1;
    }
    free(count);
    free(fill);
    return 0;
}

/*
 * Backward through the saved argmax (Flash-MaxSim Eqs. (2)-(3); design notes
 * "Backward"), dense layout, g = dL/dscore [Nq, Nd]:
 *   dQ[i,s] = q_mask[i,s] * sum_j g[i,j] * D[j, argmax[i,j,s]]   (ascending j)
 *   dD[j,t] = sum over CSR row (j,t) of q_mask[i,s] * g[i,j] * Q[i,s]
 * dD is formed destination by destination from the CSR (ascending sources).
 * Sources with argmax -1 contribute nothing. row_ptr / col may be NULL.
 */
int oracle_bwd(const void *Q, const void *D, int dtype, int64_t Nq, int64_t Lq, int64_t Nd,
               int64_t Ld, int64_t dim, const uint8_t *q_mask, const int32_t *argmax,
               const float *g, double *dQ, double *dD, int32_t *row_ptr_out, int32_t *col_out,
               int nthreads) {
    if (Nq < 0 || Nd < 0 || Lq < 0 || Ld < 0 || dim <= 0) return 1;
    set_threads(nthreads);
    int64_t nsrc = Nq * Nd * Lq;
    int64_t ndst = Nd * Ld;
    int32_t *row_ptr = row_ptr_out ? row_ptr_out : (int32_t *)malloc(((size_t)ndst + 1) * sizeof(int32_t));
    int32_t *col = col_out ? col_out : (int32_t *)malloc(((size_t)nsrc + 1) * sizeof(int32_t));
    if (!row_ptr || !col) return 4;
    int rc = oracle_csr(argmax, Nq, Lq, Nd, Ld, row_ptr, col);
    if (rc == 0) {
        /* dQ: one row (i,s) at a time, gathering D at the winners */
#pragma omp parallel for schedule(static)
        for (int64_t is = 0; is < Nq * Lq; ++is) {
            int64_t i = is / Lq, s = is % Lq;
            double *out = dQ + is * dim;
            for (int64_t k = 0; k < dim; ++k) out[k] = 0.0;
            double w = q_mask ? (q_mask[is] ? 1.0 : 0.0) : 1.0;
            for (int64_t j = 0; j < Nd; ++j) {
                int32_t a = argmax[(i * Nd + j) * Lq + s];
                if (a < 0) continue;
                double gij = (double)g[i * Nd + j];
                for (int64_t k = 0; k < dim; ++k)
                    out[k] += w * gij * load_elem(D, dtype, (j * Ld + a) * dim + k);
            }
        }
        /* dD: one destination row at a time, walking its CSR sources */
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < ndst; ++r) {
            double *out = dD + r * dim;
            for (int64_t k = 0; k < dim; ++k) out[k] = 0.0;
            for (int64_t e = row_ptr[r]; e < row_ptr[r + 1]; ++e) {
                int64_t p = col[e];
                int64_t s = p % Lq;
                int64_t ij = p / Lq;
                int64_t i = ij / Nd, j = ij % Nd;
                double w = q_mask ? (q_mask[i * Lq + s] ? 1.0 : 0.0) : 1.0;
                double gij = (double)g[i * Nd + j];
                for (int64_t k = 0; k < dim; ++k)
                    out[k] += w * gij * load_elem(Q, dtype, (i * Lq + s) * dim + k);
            }
        }
    }
    if (!row_ptr_out) free(row_ptr);
    if (!col_out) free(col);
    return rc;
}

/*
 * Chamfer distance ("Flash-MaxSim" paper, Sec. 4.2.4): for B independent
 * pairs of point sets P [B, N, dim] and Q [B, M, dim],
 *   CD(P, Q) = (1/N) sum_p min_q ||p - q||^2 + (1/M) sum_q min_p ||q - p||^2.
 * float32 inputs, double arithmetic. Per point: the squared distance to its
 * nearest point of the other set, that point's index (lowest index among
 * ties) and the gap to the second-nearest distance (+inf if there is none).
 * Reading where the page is silent: with an empty set (N or M = 0) both
 * terms are 0 and every point reports index -1 and distance 0.
 */
static void chamfer_dir(const float *X, int64_t nx, const float *Y, int64_t ny, int64_t dim, double *dist,
                        int32_t *idx, double *gap) {
    for (int64_t x = 0; x < nx; ++x) {
        double best = INFINITY, second = INFINITY;
        int32_t arg = -1;
        for (int64_t y = 0; y < ny; ++y) {
            double d2 = 0.0;
            for (int64_t k = 0; k < dim; ++k) {
                double diff = (double)X[x * dim + k] - (double)Y[y * dim + k];
                d2 += diff * diff;
            }
            if (d2 < best) { second = best; best = d2; arg = (int32_t)y; }
            else if (d2 < second) { second = d2; }
        }
        dist[x] = arg < 0 ? 0.0 : best;
        idx[x] = arg;
        gap[x] = second - best;
    }
}

int oracle_chamfer_fwd(const float *P, const float *Q, int64_t B, int64_t N, int64_t M, int64_t dim,
                       double *dist_p, int32_t *idx_p, double *gap_p, double *dist_q, int32_t *idx_q,
                       double *gap_q, double *loss, int nthreads) {
    if (B < 0 || N < 0 || M < 0 || dim <= 0) return 1;
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t b = 0; b < B; ++b) {
        const float *Pb = P + b * N * dim, *Qb = Q + b * M * dim;
        chamfer_dir(Pb, N, Qb, M, dim, dist_p + b * N, idx_p + b * N, gap_p + b * N);
        chamfer_dir(Qb, M, Pb, N, dim, dist_q + b * M, idx_q + b * M, gap_q + b * M);
        double sp = 0.0, sq = 0.0;
        for (int64_t x = 0; x < N; ++x) sp += dist_p[b * N + x];
        for (int64_t y = 0; y < M; ++y) sq += dist_q[b * M + y];
        loss[b] = (N > 0 && M > 0) ? sp / (double)N + sq / (double)M : 0.0;
    }
    return 0;
}

/*
 * Gradient of sum_b g[b] * CD(P_b, Q_b) through the saved nearest indices
 * a = idx_p (P -> Q) and c = idx_q (Q -> P) (Sec. 4.2.4 with the inverse
 * index of Sec. 4.2.2-4.2.3):
 *   dP[p] = g (2/N) (p - Q[a_p]) - g (2/M) sum over q with c_q = p of (q - p)
 *   dQ[q] = g (2/M) (q - P[c_q]) - g (2/N) sum over p with a_p = q of (p - q)
 * The sums over an inverse index run in ascending source order (a CSR by
 * counting sort). Points with index -1 contribute nothing. Returns 3 for an
 * index outside [-1, size of the other set).
 */
int oracle_chamfer_bwd(const float *P, const float *Q, int64_t B, int64_t N, int64_t M, int64_t dim,
                       const int32_t *idx_p, const int32_t *idx_q, const float *g, double *dP, double *dQ) {
    if (B < 0 || N < 0 || M < 0 || dim <= 0) return 1;
    for (int64_t b = 0; b < B; ++b) {
        const float *Pb = P + b * N * dim, *Qb = Q + b * M * dim;
        const int32_t *a = idx_p + b * N, *c = idx_q + b * M;
        double *dPb = dP + b * N * dim, *dQb = dQ + b * M * dim;
        const double gb = (double)g[b];
        const double wn = N > 0 ? 2.0 * gb / (double)N : 0.0, wm = M > 0 ? 2.0 * gb / (double)M : 0.0;
        for (int64_t x = 0; x < N; ++x)
            if (a[x] < -1 || a[x] >= M) return 3;
        for (int64_t y = 0; y < M; ++y)
            if (c[y] < -1 || c[y] >= N) return 3;
        /* inverse of a (destinations = Q points) and of c (destinations = P points) as CSRs */
        int64_t *cnt_q = (int64_t *)calloc((size_t)M + 1, sizeof(int64_t));
        int64_t *cnt_p = (int64_t *)calloc((size_t)N + 1, sizeof(int64_t));
        int64_t *col_q = (int64_t *)malloc(((size_t)N + 1) * sizeof(int64_t));
        int64_t *col_p = (int64_t *)malloc(((size_t)M + 1) * sizeof(int64_t));
        int64_t *fill_q = (int64_t *)calloc((size_t)M + 1, sizeof(int64_t));
        int64_t *fill_p = (int64_t *)calloc((size_t)N + 1, sizeof(int64_t));
        if (!cnt_q || !cnt_p || !col_q || !col_p || !fill_q || !fill_p) {
            free(cnt_q); free(cnt_p); free(col_q); free(col_p); free(fill_q); free(fill_p);
            return 4;
        }
        for (int64_t x = 0; x < N; ++x) if (a[x] >= 0) cnt_q[a[x] + 1] += 1;
        for (int64_t y = 0; y < M; ++y) if (c[y] >= 0) cnt_p[c[y] + 1] += 1;
        for (int64_t y = 0; y < M; ++y) cnt_q[y + 1] += cnt_q[y];
        for (int64_t x = 0; x < N; ++x) cnt_p[x + 1] += cnt_p[x];
        for (int64_t x = 0; x < N; ++x)
            if (a[x] >= 0) { col_q[cnt_q[a[x]] + fill_q[a[x]]] = x; fill_q[a[x]] += 1; }
        for (int64_t y = 0; y < M; ++y)
            if (c[y] >= 0) { col_p[cnt_p[c[y]] + fill_p[c[y]]] = y; fill_p[c[y]] += 1; }
        for (int64_t x = 0; x < N; ++x) {
            for (int64_t k = 0; k < dim; ++k) {
                const double px = (double)Pb[x * dim + k];
                double v = a[x] >= 0 ? wn * (px - (double)Qb[(int64_t)a[x] * dim + k]) : 0.0;
                double inv = 0.0;
                for (int64_t e = cnt_p[x]; e < cnt_p[x + 1]; ++e) inv += (double)Qb[col_p[e] * dim + k] - px;
                dPb[x * dim + k] = v - wm * inv;
            }
        }
        for (int64_t y = 0; y < M; ++y) {
            for (int64_t k = 0; k < dim; ++k) {
                const double qy = (double)Qb[y * dim + k];
                double v = c[y] >= 0 ? wm * (qy - (double)Pb[(int64_t)c[y] * dim + k]) : 0.0;
                double inv = 0.0;
                for (int64_t e = cnt_q[y]; e < cnt_q[y + 1]; ++e) inv += (double)Pb[col_q[e] * dim + k] - qy;
                dQb[y * dim + k] = v - wn * inv;
            }
        }
        free(cnt_q); free(cnt_p); free(col_q); free(col_p); free(fill_q); free(fill_p);
    }
    return 0;
}

int oracle_version(void) { return 1; }
