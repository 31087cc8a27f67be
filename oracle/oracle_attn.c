/*
 * oracle_attn.c -- plain fp64 CPU oracle for shifted-schedule sharded attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA library; it builds its own shift table from the formula.
 *
 * What it computes (sources are the three pages on Mercury, SOSP 2025):
 *
 *  - Attention "patch": Mercury keeps a known-good local attention kernel
 *    (FlashAttention) fixed and only schedules around it (Silicon & Systems,
 *    "CommIR makes communication transformable"; paper notes "核心方法").
 *    Its result is plain softmax attention, the thing the artifact's numerical
 *    checks compare against (Silicon & Systems, "The tuning bill").  Here that
 *    is written out by definition, per query row, in fp64, two passes:
 *        x_k   = <Q[b,h,q,:], K[b,g,k,:]> / sqrt(d)      g = h / (Hq/Hkv)
 *        LSE   = M + ln(sum_k exp(x_k - M)),   M = max_k x_k
 *        O     = sum_k exp(x_k - LSE) V[b,g,k,:]
 *    over the allowed keys k (causal: k <= q + (Skv - Sq)).
 *
 *  - shard: queries split into R contiguous blocks, keys/values into R
 *    contiguous shards; virtual rank i owns block i and shard i
 *    (Silicon & Systems, "The hidden cost of synchronized operators";
 *    paper notes "核心方法", shard primitive).
 *
 *  - shift: rank i reads shard (i + j) mod R at step j, the "(j+i)%J" access
 *    of the shift primitive (paper notes "核心方法"), so ranks consume the
 *    shared KV in a staggered order (Silicon & Systems, "The hidden cost of
 *    synchronized operators").  Nested two-level order for an Ro x Ri mesh
 *    (hierarchical topologies, Silicon & Systems "What Mercury finds that
 *    templates miss"): rank i = a*Ri + b, step j = s*Ri + t,
 *    shard = ((a+s) mod Ro)*Ri + (b+t) mod Ri.  The pages give no formula for
 *    the nested order; this is the reading used throughout.
 *
 *  - partial + merge: per (rank, step) a partial (O_j, LSE_j) over one shard,
 *    normalised within the shard, and the log-sum-exp merge
 *        L = ln sum_j exp(LSE_j),   O = sum_j exp(LSE_j - L) O_j,
 *    taken in step order.  A shard with no allowed key gives O_j = 0 and
 *    LSE_j = -inf, and contributes nothing.  The pages name no formula for
 *    the combine; this is the standard exact one that RingAttention uses and
 *    Mercury reproduces (paper notes, one-line summary and "实验与结果").
 *
 * Inputs are bf16 bit patterns (uint16); widening bf16 -> fp64 is exact.
 * Layouts: q [B,Hq,Sq,d], k/v [B,Hkv,Skv,d], outputs row-major doubles.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Shift table, built here from the formula (independent of the library's
 * planner).  shift 0: unshifted, order[i][j] = j.  shift 1: flat,
 * (i + j) mod R.  shift k >= 2: nested with inner size Ri = k, outer size
 * Ro = R / k.  Returns 0, or -1 for an invalid (R, shift). */
int oracle_shift_order(int R, int shift, int *order)
{
    if (R < 1 || shift < 0 || order == NULL)
        return -1;
    if (shift >= 2 && (shift > R || R % shift != 0))
        return -1;
    for (int i = 0; i < R; ++i) {
        for (int j = 0; j < R; ++j) {
            int s;
            if (shift == 0) {
                s = j;
            } else if (shift == 1) {
                s = (i + j) % R;
            } else {
                int Ri = shift, Ro = R / shift;
                int a = i / Ri, b = i % Ri;   /* rank = (outer a, inner b) */
                int so = j / Ri, t = j % Ri;  /* step = (outer s, inner t) */
                s = ((a + so) % Ro) * Ri + (b + t) % Ri;
            }
            order[i * R + j] = s;
        }
    }
    return 0;
}

/* Last allowed key (inclusive) for query row q: causal alignment puts the
 * last query on the last key, k <= q + (Skv - Sq). */
static int64_t last_allowed_key(int64_t q, int64_t Sq, int64_t Skv, int causal)
{
    if (!causal)
        return Skv - 1;
    int64_t lim = q + (Skv - Sq);
    return lim < Skv - 1 ? lim : Skv - 1;
}

/* Attention of one query row over keys [k_lo, k_hi] (inclusive; empty when
 * k_hi < k_lo).  scores: scratch of at least (k_hi - k_lo + 1) doubles. */
static void attend_row(const double *qrow, const uint16_t *Kg, const uint16_t *Vg,
                       int d, int64_t k_lo, int64_t k_hi, double *scores,
                       double *o, double *lse)
{
    for (int t = 0; t < d; ++t)
        o[t] = 0.0;
    if (k_hi < k_lo) {
        *lse = -INFINITY;
        return;
    }
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    int64_t n = k_hi - k_lo + 1;
    double M = -INFINITY;
    for (int64_t c = 0; c < n; ++c) {
        const uint16_t *kr = Kg + (k_lo + c) * (int64_t)d;
        double acc = 0.0;
        for (int t = 0; t < d; ++t)
            acc += qrow[t] * bf16_to_f64(kr[t]);
        scores[c] = acc * inv_sqrt_d;
        if (scores[c] > M)
            M = scores[c];
    }
    double Z = 0.0;
    for (int64_t c = 0; c < n; ++c)
        Z += exp(scores[c] - M);
    double L = M + log(Z);
    for (int64_t c = 0; c < n; ++c) {
        double w = exp(scores[c] - L);
        const uint16_t *vr = Vg + (k_lo + c) * (int64_t)d;
        for (int t = 0; t < d; ++t)
            o[t] += w * bf16_to_f64(vr[t]);
    }
    *lse = L;
}

static int check_shape(int B, int Hq, int Hkv, int Sq, int Skv, int d)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 0 || Skv < 0 || d < 1)
        return -1;
    if (Hq % Hkv != 0)
        return -1;
    return 0;
}

/* Full (unsharded) attention for selected rows.
 * rows[r] = (b*Hq + h)*Sq + q.  out [n_rows][d], lse [n_rows]. */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                     int64_t n_rows, const int64_t *rows, double *out, double *lse)
{
    if (check_shape(B, Hq, Hkv, Sq, Skv, d))
        return -1;
    const int G = Hq / Hkv;
    int err = 0;
#pragma omp parallel
    {
        double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
        double *scores = (double *)malloc(sizeof(double) * (size_t)(Skv > 0 ? Skv : 1));
        if (!qrow || !scores) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < n_rows; ++r) {
                int64_t row = rows[r];
                int64_t qi = row % Sq;
                int64_t bh = row / Sq;
                int64_t b = bh / Hq, h = bh % Hq;
                int64_t g = h / G;
                const uint16_t *qr = q + row * (int64_t)d;
                for (int t = 0; t < d; ++t)
                    qrow[t] = bf16_to_f64(qr[t]);
                const uint16_t *Kg = k + (b * Hkv + g) * (int64_t)Skv * d;
                const uint16_t *Vg = v + (b * Hkv + g) * (int64_t)Skv * d;
                int64_t hi = last_allowed_key(qi, Sq, Skv, causal);
                attend_row(qrow, Kg, Vg, d, 0, hi, scores, out + r * (int64_t)d, lse + r);
            }
        }
        free(qrow);
        free(scores);
    }
    return err;
}

/* Per-step partials of the sharded schedule for selected rows.
 * Row q belongs to virtual rank i = q / (Sq/R); at step j it attends to shard
 * s = order[i][j], keys [s*Bk, (s+1)*Bk), intersected with the causal limit.
 * o_part [R][n_rows][d], lse_part [R][n_rows]; slot j = step j. */
int oracle_attn_partial_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             int B, int Hq, int Hkv, int Sq, int Skv, int d,
                             int R, int shift, int causal,
                             int64_t n_rows, const int64_t *rows,
                             double *o_part, double *lse_part)
{
    if (check_shape(B, Hq, Hkv, Sq, Skv, d))
        return -1;
    if (R < 1 || Sq % R != 0 || Skv % R != 0)
        return -1;
    int *order = (int *)malloc(sizeof(int) * (size_t)R * R);
    if (!order)
        return -2;
    if (oracle_shift_order(R, shift, order)) {
        free(order);
        return -1;
    }
    const int G = Hq / Hkv;
    const int64_t Bq = Sq / R, Bk = Skv / R;
    int err = 0;
#pragma omp parallel
    {
        double *qrow = (double *)malloc(sizeof(double) * (size_t)d);
        double *scores = (double *)malloc(sizeof(double) * (size_t)(Bk > 0 ? Bk : 1));
        if (!qrow || !scores) {
#pragma omp atomic write
            err = -2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < n_rows; ++r) {
                int64_t row = rows[r];
                int64_t qi = row % Sq;
                int64_t bh = row / Sq;
                int64_t b = bh / Hq, h = bh % Hq;
                int64_t g = h / G;
                int64_t rank = qi / Bq;
                const uint16_t *qr = q + row * (int64_t)d;
                for (int t = 0; t < d; ++t)
                    qrow[t] = bf16_to_f64(qr[t]);
                const uint16_t *Kg = k + (b * Hkv + g) * (int64_t)Skv * d;
                const uint16_t *Vg = v + (b * Hkv + g) * (int64_t)Skv * d;
                int64_t lim = last_allowed_key(qi, Sq, Skv, causal);
                for (int j = 0; j < R; ++j) {
                    int64_t s = order[rank * R + j];
                    int64_t lo = s * Bk, hi = (s + 1) * Bk - 1;
                    if (hi > lim)
                        hi = lim;
                    attend_row(qrow, Kg, Vg, d, lo, hi, scores,
                               o_part + ((int64_t)j * n_rows + r) * d,
                               lse_part + (int64_t)j * n_rows + r);
                }
            }
        }
        free(qrow);
        free(scores);
    }
    free(order);
    return err;
}

/* Log-sum-exp merge of n_parts partials, taken in part order.
 * o_part [n_parts][rows][d], lse_part [n_parts][rows] -> out [rows][d], lse [rows].
 * All parts at -inf: O = 0, L = -inf. */
int oracle_lse_merge(const double *o_part, const double *lse_part, int n_parts,
                     int64_t rows, int d, double *out, double *lse)
{
    if (n_parts < 1 || rows < 0 || d < 1)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int j = 0; j < n_parts; ++j) {
            double l = lse_part[(int64_t)j * rows + r];
            if (l > M)
                M = l;
        }
        double *o = out + r * d;
        for (int t = 0; t < d; ++t)
            o[t] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double Z = 0.0;
        for (int j = 0; j < n_parts; ++j)
            Z += exp(lse_part[(int64_t)j * rows + r] - M);
        double L = M + log(Z);
        for (int j = 0; j < n_parts; ++j) {
            double w = exp(lse_part[(int64_t)j * rows + r] - L);
            if (w == 0.0)
                continue;
            const double *op = o_part + ((int64_t)j * rows + r) * d;
            for (int t = 0; t < d; ++t)
                o[t] += w * op[t];
        }
        lse[r] = L;
    }
    return 0;
}

/* Sharded attention = per-step partials merged in step order. */
int oracle_attn_sharded_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             int B, int Hq, int Hkv, int Sq, int Skv, int d,
                             int R, int shift, int causal,
                             int64_t n_rows, const int64_t *rows,
                             double *out, double *lse)
{
    double *op = (double *)malloc(sizeof(double) * (size_t)R * (size_t)(n_rows > 0 ? n_rows : 1) * d);
    double *lp = (double *)malloc(sizeof(double) * (size_t)R * (size_t)(n_rows > 0 ? n_rows : 1));
    int rc = -2;
    if (op && lp) {
        rc = oracle_attn_partial_rows(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal,
                                      n_rows, rows, op, lp);
        if (rc == 0)
            rc = oracle_lse_merge(op, lp, R, n_rows, d, out, lse);
    }
    free(op);
    free(lp);
    return rc;
}

/* Number of unmasked (query, key) pairs of one (b, h): the algorithmic work
 * unit (4*d flops per pair: 2*d for the score, 2*d for the value sum). */
int64_t oracle_unmasked_pairs(int Sq, int Skv, int causal)
{
    int64_t n = 0;
    for (int64_t q = 0; q < Sq; ++q) {
        int64_t hi = last_allowed_key(q, Sq, Skv, causal);
        if (hi >= 0)
            n += hi + 1;
    }
    return n;
}
