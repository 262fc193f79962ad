/*
 * df_oracle.c -- plain fp64 CPU oracle for exact DeBERTa-v2/v3 disentangled
 * self-attention (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file.  The product path (the
 * CUDA library) shares no code, header, table or constant with it.
 *
 * What it computes, per sequence s and head h (tokens i, j of that sequence,
 * positions counted inside the sequence):
 *
 *   bucket(r)  DeBERTa log bucketing of the relative position r = i - j
 *   delta(r)   = clamp(bucket(r) + span, 0, 2*span - 1)          (R = 2*span)
 *   Z[i,j]     = Q_i.K_j + Q_i.Kr[delta(i-j)] + K_j.Qr[delta(i-j)]
 *   S[i,j]     = c * Z[i,j]   (c = 1/sqrt(3D) unless given),  -inf where the
 *                query or the key is masked
 *   LSE_i      = log sum_j exp(S[i,j])   (natural log)
 *   P          = exp(S - LSE);  dropout: Pd = P * keep / (1 - p)
 *   O          = Pd V
 *
 * Sources: "DisentangledFlash" (pypi disentangled-flash 1.1.1), sections
 * "Status" (C2P/P2C DeBERTa-v2/v3 attention, factorised 2-D padding masks,
 * packed cu_seqlens, Philox dropout regenerated in backward) and
 * "Performance" (the FLOP count names the C2P and P2C relative-position
 * products over R relative rows); the score formula, the log bucketing and
 * the clamp are DeBERTa's published definitions, restated here as plain math.
 *
 * Backward (plain calculus of the forward above):
 *   dV   = Pd^T dO
 *   dPd  = dO V^T ;  dP = dPd * keep / (1 - p)
 *   Dl_i = sum_j P[i,j] dP[i,j]
 *   dZ   = c * P * (dP - Dl)
 *   dQ_i = sum_j dZ[i,j] (K_j + Kr[delta(i-j)])
 *   dK_j = sum_i dZ[i,j] (Q_i + Qr[delta(i-j)])
 *   dKr[r] = sum over (s, i, j) with delta(i-j) = r of dZ[i,j] Q_i
 *   dQr[r] = sum over (s, i, j) with delta(i-j) = r of dZ[i,j] K_j
 *
 * Rows with no attendable key (masked query, or every key masked) get O = 0,
 * LSE = +inf and zero gradients (the reading of the silent mask case).
 *
 * Dropout draws come from Philox4x32-10 (Salmon, Moraes, Dror, Shaw,
 * "Parallel random numbers: as easy as 1, 2, 3", SC'11): key = (seed_lo,
 * seed_hi), counter = (j >> 2, i, s*H + h, offset); the word j & 3 of the
 * output decides keep[i,j] = (word < floor((1 - p) * 2^32)).
 *
 * Layouts: Q, K, V, dO, O, dQ, dK, dV are [T, H, D] (token-major, T tokens
 * of all sequences back to back, cu[s]..cu[s+1] the tokens of sequence s);
 * Qr, Kr, dQr, dKr are [H, R, D]; LSE is [H, T]; masks are [T] bytes.
 *
 * Parity pins: see the tests that call this file (tests/test_oracle_pins.py):
 * brute-force evaluation, library attention with Kr = Qr = 0, invariants,
 * finite differences and an autograd formulation.  Philox is pinned only by
 * statistics on the CPU ("parity unpinned" against a known-answer vector:
 * the pages print none).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int nseq;                    /* number of sequences                      */
    const int *cu;               /* [nseq+1] token offsets                    */
    int T, H, D;                 /* total tokens, heads, head dim             */
    int span, nb, mp;            /* att_span, position_buckets, max_rel_pos   */
    const unsigned char *qmask;  /* [T] or NULL                               */
    const unsigned char *kmask;  /* [T] or NULL                               */
    double scale;                /* c; <= 0 means 1/sqrt(3D)                  */
    double p_drop;               /* attention-probability dropout             */
    uint64_t seed;
    uint32_t offset;
} orc_cfg;

/* ---------------------------------------------------------------- buckets */

/* DeBERTa log bucketing of a relative position r.  Positions within
 * +-(nb/2) keep their value; farther ones are compressed logarithmically so
 * that |r| = mp - 1 lands on nb/2 + (nb/2 - 1).  No bucketing when nb <= 0
 * or mp <= 0. */
long orc_bucket(long r, int nb, int mp)
{
    if (nb <= 0 || mp <= 0) return r;
    long mid = nb / 2;
    long a = r < 0 ? -r : r;
    if (a <= mid) return r;
    double x = log((double)a / (double)mid) / log((double)(mp - 1) / (double)mid)
               * (double)(mid - 1);
    long b = mid + (long)ceil(x);
    return r < 0 ? -b : b;
}

long orc_delta(long r, int span, int nb, int mp)
{
    long d = orc_bucket(r, nb, mp) + span;
    if (d < 0) d = 0;
    if (d > 2L * span - 1) d = 2L * span - 1;
    return d;
}

/* delta for every r in [-(L-1), L-1]; out[r + L - 1]. */
int orc_delta_table(int L, int span, int nb, int mp, int32_t *out)
{
    if (L <= 0 || span <= 0) return -1;
    for (long r = -(long)(L - 1); r <= (long)(L - 1); ++r)
        out[r + L - 1] = (int32_t)orc_delta(r, span, nb, mp);
    return 0;
}

/* ---------------------------------------------------------------- Philox */

static void mulhilo32(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo)
{
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

/* Philox4x32 with 10 rounds.  Each round multiplies words 0 and 2 by the two
 * Philox multipliers and mixes the high halves with words 1 and 3 and the
 * round key; the key advances by the two Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint32_t hi0, lo0, hi1, lo1;
        mulhilo32(M0, x0, &hi0, &lo0);
        mulhilo32(M1, x2, &hi1, &lo1);
        uint32_t y0 = hi1 ^ x1 ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x3 ^ k1;
        uint32_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += W0; k1 += W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

uint64_t orc_keep_threshold(double p)
{
    if (p <= 0.0) return (uint64_t)1 << 32;
    double t = floor((1.0 - p) * 4294967296.0);
    if (t < 0.0) t = 0.0;
    return (uint64_t)t;
}

/* keep bit for token pair (i, j) of sequence s, head h (positions inside the
 * sequence). */
static int keep_bit(const orc_cfg *c, int s, int h, int i, int j, uint64_t thr)
{
    uint32_t ctr[4] = {(uint32_t)j >> 2, (uint32_t)i, (uint32_t)(s * c->H + h), c->offset};
    uint32_t key[2] = {(uint32_t)c->seed, (uint32_t)(c->seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    return (uint64_t)w[j & 3] < thr;
}

/* keep mask of one (s, h) pair, row-major [n, n]; exposed for tests. */
int orc_keep_mask(const orc_cfg *c, int s, int h, unsigned char *out)
{
    int n = c->cu[s + 1] - c->cu[s];
    uint64_t thr = orc_keep_threshold(c->p_drop);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) out[(size_t)i * n + j] = (unsigned char)keep_bit(c, s, h, i, j, thr);
    return 0;
}

/* ------------------------------------------------------------ score rows */

static double scale_of(const orc_cfg *c)
{
    return c->scale > 0.0 ? c->scale : 1.0 / sqrt(3.0 * (double)c->D);
}

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int k = 0; k < n; ++k) s += a[k] * b[k];
    return s;
}

/* Row i of S for pair (s, h): fills srow[0..n).  Returns 1 if the row has at
 * least one finite entry. */
static int score_row(const orc_cfg *c, int s, int h, int i, const double *q, const double *k,
                     const double *qr, const double *kr, double *srow)
{
    const int H = c->H, D = c->D, R = 2 * c->span;
    const int t0 = c->cu[s], n = c->cu[s + 1] - t0;
    const double cs = scale_of(c);
    const double *qi = q + ((size_t)(t0 + i) * H + h) * D;
    int any = 0;
    int qvalid = c->qmask ? c->qmask[t0 + i] != 0 : 1;
    for (int j = 0; j < n; ++j) {
        int kvalid = c->kmask ? c->kmask[t0 + j] != 0 : 1;
        if (!qvalid || !kvalid) { srow[j] = -INFINITY; continue; }
        const double *kj = k + ((size_t)(t0 + j) * H + h) * D;
        long d = orc_delta((long)i - (long)j, c->span, c->nb, c->mp);
        const double *krd = kr + ((size_t)h * R + d) * D;
        const double *qrd = qr + ((size_t)h * R + d) * D;
        double z = dot(qi, kj, D) + dot(qi, krd, D) + dot(kj, qrd, D);
        srow[j] = cs * z;
        any = 1;
    }
    return any;
}

/* log-sum-exp of a row; +inf when the row is entirely -inf */
static double row_lse(const double *srow, int n)
{
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) if (srow[j] > m) m = srow[j];
    if (m == -INFINITY) return INFINITY;
    double acc = 0.0;
    for (int j = 0; j < n; ++j) acc += exp(srow[j] - m);
    return m + log(acc);
}

/* ---------------------------------------------------------------- forward */

/* forward of one (s, h) pair; rows == NULL means all rows, else nrows rows
 * listed in rows[] (positions inside the sequence).  o is [T, H, D], lse is
 * [H, T]; only the selected rows are written. */
int orc_forward_pair(const orc_cfg *c, int s, int h, const double *q, const double *k, const double *v,
                     const double *qr, const double *kr, double *o, double *lse, int nrows, const int *rows)
{
    const int H = c->H, D = c->D, T = c->T;
    const int t0 = c->cu[s], n = c->cu[s + 1] - t0;
    const uint64_t thr = orc_keep_threshold(c->p_drop);
    const double dscale = c->p_drop > 0.0 ? 1.0 / (1.0 - c->p_drop) : 1.0;
    double *srow = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!srow) return -2;
    int cnt = rows ? nrows : n;
    for (int ri = 0; ri < cnt; ++ri) {
        int i = rows ? rows[ri] : ri;
        if (i < 0 || i >= n) { free(srow); return -1; }
        double *oi = o + ((size_t)(t0 + i) * H + h) * D;
        for (int d = 0; d < D; ++d) oi[d] = 0.0;
        int any = score_row(c, s, h, i, q, k, qr, kr, srow);
        double L = any ? row_lse(srow, n) : INFINITY;
        lse[(size_t)h * T + t0 + i] = L;
        if (!any) continue;
        for (int j = 0; j < n; ++j) {
            double p = exp(srow[j] - L);
            if (p == 0.0) continue;
            if (c->p_drop > 0.0) p = keep_bit(c, s, h, i, j, thr) ? p * dscale : 0.0;
            const double *vj = v + ((size_t)(t0 + j) * H + h) * D;
            for (int d = 0; d < D; ++d) oi[d] += p * vj[d];
        }
    }
    free(srow);
    return 0;
}

int orc_forward(const orc_cfg *c, const double *q, const double *k, const double *v, const double *qr,
                const double *kr, double *o, double *lse, int nthreads)
{
    int npair = c->nseq * c->H, err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (int pidx = 0; pidx < npair; ++pidx)
        err |= orc_forward_pair(c, pidx / c->H, pidx % c->H, q, k, v, qr, kr, o, lse, 0, NULL) != 0;
    (void)nthreads;
    return err ? -1 : 0;
}

/* --------------------------------------------------------------- backward */

/* Backward of one (s, h) pair.  Writes dq, dk, dv rows of this pair into the
 * [T, H, D] outputs and the pair's own contribution to dKr / dQr into
 * dkr_part / dqr_part ([R, D], overwritten).  All accumulation runs in a fixed
 * order (rows ascending, keys ascending). */
int orc_backward_pair(const orc_cfg *c, int s, int h, const double *q, const double *k, const double *v,
                      const double *qr, const double *kr, const double *dout, double *dq, double *dk,
                      double *dv, double *dkr_part, double *dqr_part)
{
    const int H = c->H, D = c->D, R = 2 * c->span;
    const int t0 = c->cu[s], n = c->cu[s + 1] - t0;
    const double cs = scale_of(c);
    const uint64_t thr = orc_keep_threshold(c->p_drop);
    const double dscale = c->p_drop > 0.0 ? 1.0 / (1.0 - c->p_drop) : 1.0;
    double *srow = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * 3);
    if (!srow) return -2;
    double *prow = srow + n, *dzrow = prow + n;
    memset(dkr_part, 0, sizeof(double) * (size_t)R * D);
    memset(dqr_part, 0, sizeof(double) * (size_t)R * D);
    for (int j = 0; j < n; ++j) {
        memset(dk + ((size_t)(t0 + j) * H + h) * D, 0, sizeof(double) * D);
        memset(dv + ((size_t)(t0 + j) * H + h) * D, 0, sizeof(double) * D);
    }
    for (int i = 0; i < n; ++i) {
        const double *qi = q + ((size_t)(t0 + i) * H + h) * D;
        const double *doi = dout + ((size_t)(t0 + i) * H + h) * D;
        double *dqi = dq + ((size_t)(t0 + i) * H + h) * D;
        for (int d = 0; d < D; ++d) dqi[d] = 0.0;
        int any = score_row(c, s, h, i, q, k, qr, kr, srow);
        if (!any) continue;
        double L = row_lse(srow, n);
        /* P row, dP row and the row constant Dl_i = sum_j P dP */
        double dl = 0.0;
        for (int j = 0; j < n; ++j) {
            double p = exp(srow[j] - L);
            prow[j] = p;
            const double *vj = v + ((size_t)(t0 + j) * H + h) * D;
            double dpd = dot(doi, vj, D);
            double keep = 1.0;
            if (c->p_drop > 0.0) keep = keep_bit(c, s, h, i, j, thr) ? dscale : 0.0;
            /* dV_j += Pd[i,j] dO_i */
            if (p != 0.0 && keep != 0.0) {
                double *dvj = dv + ((size_t)(t0 + j) * H + h) * D;
                for (int d = 0; d < D; ++d) dvj[d] += p * keep * doi[d];
            }
            dzrow[j] = dpd * keep; /* dP for now */
            dl += p * dzrow[j];
        }
        for (int j = 0; j < n; ++j) dzrow[j] = cs * prow[j] * (dzrow[j] - dl);
        for (int j = 0; j < n; ++j) {
            double g = dzrow[j];
            if (g == 0.0) continue;
            const double *kj = k + ((size_t)(t0 + j) * H + h) * D;
            long dd = orc_delta((long)i - (long)j, c->span, c->nb, c->mp);
            const double *krd = kr + ((size_t)h * R + dd) * D;
            const double *qrd = qr + ((size_t)h * R + dd) * D;
            double *dkj = dk + ((size_t)(t0 + j) * H + h) * D;
            double *dkr_d = dkr_part + (size_t)dd * D;
            double *dqr_d = dqr_part + (size_t)dd * D;
            for (int d = 0; d < D; ++d) {
                dqi[d] += g * (kj[d] + krd[d]);
                dkj[d] += g * (qi[d] + qrd[d]);
                dkr_d[d] += g * qi[d];
                dqr_d[d] += g * kj[d];
            }
        }
    }
    free(srow);
    return 0;
}

/* Full backward over all pairs; dkr / dqr ([H, R, D]) are the sums over the
 * sequences, taken in ascending sequence order for every head. */
int orc_backward(const orc_cfg *c, const double *q, const double *k, const double *v, const double *qr,
                 const double *kr, const double *dout, double *dq, double *dk, double *dv, double *dqr,
                 double *dkr, int nthreads)
{
    const int H = c->H, D = c->D, R = 2 * c->span;
    const size_t rd = (size_t)R * D;
    int err = 0;
    memset(dkr, 0, sizeof(double) * (size_t)H * rd);
    memset(dqr, 0, sizeof(double) * (size_t)H * rd);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
#endif
    for (int h = 0; h < H; ++h) {
        double *pk = (double *)malloc(sizeof(double) * rd * 2);
        if (!pk) { err |= 1; continue; }
        double *pq = pk + rd;
        for (int s = 0; s < c->nseq; ++s) {
            err |= orc_backward_pair(c, s, h, q, k, v, qr, kr, dout, dq, dk, dv, pk, pq) != 0;
            double *hk = dkr + (size_t)h * rd, *hq = dqr + (size_t)h * rd;
            for (size_t x = 0; x < rd; ++x) { hk[x] += pk[x]; hq[x] += pq[x]; }
        }
        free(pk);
    }
    (void)nthreads;
    return err ? -1 : 0;
}

/* Sampled backward of one (s, h) pair for full-size checks: dQ of the rows
 * listed in rows[] and dK, dV of the keys listed in cols[] (positions inside
 * the sequence), each computed from the plain definition.  The per-row
 * constants LSE_i and Dl_i that the key gradients need are computed for every
 * row (rows in parallel).  Outputs: dq_rows [nrows, D], dk_cols, dv_cols
 * [ncols, D]. */
int orc_backward_sample(const orc_cfg *c, int s, int h, const double *q, const double *k, const double *v,
                        const double *qr, const double *kr, const double *dout, int nrows, const int *rows,
                        int ncols, const int *cols, double *dq_rows, double *dk_cols, double *dv_cols)
{
    const int H = c->H, D = c->D, R = 2 * c->span;
    const int t0 = c->cu[s], n = c->cu[s + 1] - t0;
    const double cs = scale_of(c);
    const uint64_t thr = orc_keep_threshold(c->p_drop);
    const double dscale = c->p_drop > 0.0 ? 1.0 / (1.0 - c->p_drop) : 1.0;
    double *lse = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * 2);
    if (!lse) return -2;
    double *dl = lse + n;
    int err = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16) reduction(| : err)
#endif
    for (int i = 0; i < n; ++i) {
        double *srow = (double *)malloc(sizeof(double) * (size_t)n);
        if (!srow) { err |= 1; continue; }
        int any = score_row(c, s, h, i, q, k, qr, kr, srow);
        lse[i] = any ? row_lse(srow, n) : INFINITY;
        double acc = 0.0;
        if (any) {
            const double *doi = dout + ((size_t)(t0 + i) * H + h) * D;
            for (int j = 0; j < n; ++j) {
                double p = exp(srow[j] - lse[i]);
                if (p == 0.0) continue;
                double keep = 1.0;
                if (c->p_drop > 0.0) keep = keep_bit(c, s, h, i, j, thr) ? dscale : 0.0;
                acc += p * dot(doi, v + ((size_t)(t0 + j) * H + h) * D, D) * keep;
            }
        }
        dl[i] = acc;
        free(srow);
    }
    if (err) { free(lse); return -2; }
    double *srow = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int ri = 0; ri < nrows; ++ri) {
        const int i = rows[ri];
        double *o = dq_rows + (size_t)ri * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (i < 0 || i >= n || lse[i] == INFINITY) continue;
        score_row(c, s, h, i, q, k, qr, kr, srow);
        const double *doi = dout + ((size_t)(t0 + i) * H + h) * D;
        for (int j = 0; j < n; ++j) {
            double p = exp(srow[j] - lse[i]);
            if (p == 0.0) continue;
            double keep = 1.0;
            if (c->p_drop > 0.0) keep = keep_bit(c, s, h, i, j, thr) ? dscale : 0.0;
            const double *kj = k + ((size_t)(t0 + j) * H + h) * D;
            double g = cs * p * (dot(doi, v + ((size_t)(t0 + j) * H + h) * D, D) * keep - dl[i]);
            long dd = orc_delta((long)i - (long)j, c->span, c->nb, c->mp);
            const double *krd = kr + ((size_t)h * R + dd) * D;
            for (int d = 0; d < D; ++d) o[d] += g * (kj[d] + krd[d]);
        }
    }
    for (int cj = 0; cj < ncols; ++cj) {
        const int j = cols[cj];
        double *ok = dk_cols + (size_t)cj * D, *ov = dv_cols + (size_t)cj * D;
        for (int d = 0; d < D; ++d) { ok[d] = 0.0; ov[d] = 0.0; }
        if (j < 0 || j >= n) continue;
        if (c->kmask && !c->kmask[t0 + j]) continue;
        const double *kj = k + ((size_t)(t0 + j) * H + h) * D;
        const double *vj = v + ((size_t)(t0 + j) * H + h) * D;
        for (int i = 0; i < n; ++i) {
            if (lse[i] == INFINITY) continue;
            if (c->qmask && !c->qmask[t0 + i]) continue;
            const double *qi = q + ((size_t)(t0 + i) * H + h) * D;
            const double *doi = dout + ((size_t)(t0 + i) * H + h) * D;
            long dd = orc_delta((long)i - (long)j, c->span, c->nb, c->mp);
            const double *krd = kr + ((size_t)h * R + dd) * D;
            const double *qrd = qr + ((size_t)h * R + dd) * D;
            double z = dot(qi, kj, D) + dot(qi, krd, D) + dot(kj, qrd, D);
            double p = exp(cs * z - lse[i]);
            double keep = 1.0;
            if (c->p_drop > 0.0) keep = keep_bit(c, s, h, i, j, thr) ? dscale : 0.0;
            double g = cs * p * (dot(doi, vj, D) * keep - dl[i]);
            for (int d = 0; d < D; ++d) {
                ov[d] += p * keep * doi[d];
                ok[d] += g * (qi[d] + qrd[d]);
            }
        }
    }
    free(srow);
    free(lse);
    return 0;
}

/* Forward and backward work of the query rows [r0, r1) of `npairs` (s, h)
 * pairs (one pair per OpenMP thread), exactly as orc_forward_pair /
 * orc_backward_pair do it row by row, with private accumulators.  Used to
 * time the oracle on a bounded sample of a large workload.  Returns a
 * checksum of the outputs (so the work cannot be skipped). */
double orc_step_rows_sample(const orc_cfg *c, int npairs, const int *pairs, int r0, int r1, const double *q,
                            const double *k, const double *v, const double *qr, const double *kr,
                            const double *dout, int nthreads)
{
    double total = 0.0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : total)
#endif
    for (int x = 0; x < npairs; ++x) {
        const int s = pairs[2 * x], h = pairs[2 * x + 1];
        const int H = c->H, D = c->D, R = 2 * c->span;
        const int t0 = c->cu[s], n = c->cu[s + 1] - t0;
        const double cs = scale_of(c);
        const uint64_t thr = orc_keep_threshold(c->p_drop);
        const double dscale = c->p_drop > 0.0 ? 1.0 / (1.0 - c->p_drop) : 1.0;
        double *buf = (double *)calloc((size_t)3 * n + (size_t)2 * n * D + (size_t)2 * R * D + 2 * (size_t)D, sizeof(double));
        if (!buf) continue;
        double *srow = buf, *prow = srow + n, *dzrow = prow + n;
        double *dk = dzrow + n, *dv = dk + (size_t)n * D, *dkr = dv + (size_t)n * D, *dqr = dkr + (size_t)R * D;
        double *o = dqr + (size_t)R * D, *dq = o + D;
        for (int i = r0; i < r1 && i < n; ++i) {
            const double *qi = q + ((size_t)(t0 + i) * H + h) * D;
            const double *doi = dout + ((size_t)(t0 + i) * H + h) * D;
            if (!score_row(c, s, h, i, q, k, qr, kr, srow)) continue;
            const double L = row_lse(srow, n);
            for (int d = 0; d < D; ++d) { o[d] = 0.0; dq[d] = 0.0; }
            double dl = 0.0;
            for (int j = 0; j < n; ++j) {
                const double p = exp(srow[j] - L);
                prow[j] = p;
                double keep = 1.0;
                if (c->p_drop > 0.0) keep = keep_bit(c, s, h, i, j, thr) ? dscale : 0.0;
                const double *vj = v + ((size_t)(t0 + j) * H + h) * D;
                for (int d = 0; d < D; ++d) o[d] += p * keep * vj[d];
                for (int d = 0; d < D; ++d) dv[(size_t)j * D + d] += p * keep * doi[d];
                dzrow[j] = dot(doi, vj, D) * keep;
                dl += p * dzrow[j];
            }
            for (int j = 0; j < n; ++j) {
                const double g = cs * prow[j] * (dzrow[j] - dl);
                const double *kj = k + ((size_t)(t0 + j) * H + h) * D;
                const long dd = orc_delta((long)i - (long)j, c->span, c->nb, c->mp);
                const double *krd = kr + ((size_t)h * R + dd) * D;
                const double *qrd = qr + ((size_t)h * R + dd) * D;
                for (int d = 0; d < D; ++d) {
                    dq[d] += g * (kj[d] + krd[d]);
                    dk[(size_t)j * D + d] += g * (qi[d] + qrd[d]);
                    dkr[(size_t)dd * D + d] += g * qi[d];
                    dqr[(size_t)dd * D + d] += g * kj[d];
                }
            }
            for (int d = 0; d < D; ++d) total += o[d] + dq[d];
        }
        for (size_t x2 = 0; x2 < (size_t)2 * n * D + (size_t)2 * R * D; ++x2) total += dk[x2];
        free(buf);
    }
    return total;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
