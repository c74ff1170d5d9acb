/*
 * fa_oracle.c -- plain, slow, fp64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes is the plain definition of attention, written out without
 * any tiling:
 *   S = scale * Q K^T, masked (causal: key c visible to query r iff c <= r;
 *   sliding window of W keys: visible iff r - c < W, in addition),
 *   P = softmax_rows(S), O = P V, L = rowwise log-sum-exp of S (natural log).
 * The window is the attention-mask change that sliding-window attention
 * makes (FlashAttention-3 summary, discussion of GQA and sliding-window
 * attention): it only restricts which keys a query sees; window 0 = none.
 * "FlashAttention-2 ... (blog.csdn.net, 3.1.1 forward formula analysis)" shows
 * that the tiled online-softmax recurrence with a single final diag(l)^-1
 * rescale reaches exactly this O and L = m + log(l); "6.2 FlashAttention V2 chi
 * tiet", section 6.1 gives the same forward as pseudocode.  So the oracle is
 * the definition, not the recurrence.
 *
 * The backward is the analytic gradient listed step by step in "3.1.2 backward
 * formula analysis" of the blog.csdn.net page:
 *   D = rowsum(dO o O), P = exp(S - L), dV = P^T dO, dP = dO V^T,
 *   dS = P o (dP - D), dQ = scale * dS K, dK = scale * dS^T Q.
 * The scale factor is carried by the chain rule because the forward scores are
 * scale * Q K^T (section 6.1 of the Vietnamese page divides by sqrt(d)); the
 * blog's backward list omits it, and the chain rule puts it back.
 * Grouped-query heads: query head h reads key/value head h / (Hq / Hkv), and
 * dK, dV sum over the query heads of a group ("multi-query and grouped-query
 * attention" paragraph at the end of the blog.csdn.net page).
 *
 * Layout of every tensor: [B][H][N][d], d contiguous, fp64.  L and D: [B][Hq][N].
 *
 * The FP8 helpers model incoherent processing from the FlashAttention-3
 * summary (vi.news.hada.io, "Do chinh xac thap FP8 va incoherent processing"):
 * a random-sign Sylvester-Hadamard rotation, applied here as a dense d x d
 * matrix product (no fast transform), and round-to-nearest-even to the OCP
 * e4m3 ("fn") grid with saturation at +-448.
 */
#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include <string.h>

/* Threads of the OpenMP loops below, for timing baselines (n < 1: one per
 * host processor, the default).  No effect on any result. */
void oracle_set_threads(int n) { omp_set_num_threads(n >= 1 ? n : omp_get_num_procs()); }
int oracle_get_threads(void) { return omp_get_max_threads(); }

#define IDX4(b, h, n, H, N) ((((long)(b) * (H) + (h)) * (N) + (n)))

static int args_ok(long B, long Hq, long Hkv, long N, long d) {
    if (B < 1 || Hq < 1 || Hkv < 1 || N < 1 || d < 1) return 0;
    if (Hq % Hkv != 0) return 0;
    return 1;
}

/* Keys visible to query row r: c0 <= c < c1. */
static void visible_keys(long r, long N, int causal, long window, long *c0,
                         long *c1) {
    *c1 = causal ? (r + 1 < N ? r + 1 : N) : N;
    *c0 = (window > 0 && r - window + 1 > 0) ? r - window + 1 : 0;
}

/* Query rows that see key c: r0 <= r < r1. */
static void visible_rows(long c, long N, int causal, long window, long *r0,
                         long *r1) {
    *r0 = causal ? c : 0;
    *r1 = (window > 0 && c + window < N) ? c + window : N;
}

/* One query row: s[c - c0] = scale * q.k_c for c0 <= c < c1. */
static void score_row(const double *qr, const double *kh, long c0, long c1,
                      long d, double scale, double *s) {
    for (long c = c0; c < c1; ++c) {
        const double *kc = kh + c * d;
        double acc = 0.0;
        for (long t = 0; t < d; ++t) acc += qr[t] * kc[t];
        s[c - c0] = scale * acc;
    }
}

/* Forward for one (b, hq, r): writes o_row[d] and *lse. s is scratch of N. */
static void fwd_one_row(const double *q, const double *k, const double *v,
                        long b, long hq, long r, long Hq, long Hkv, long N,
                        long d, int causal, long window, double scale,
                        double *s, double *o_row, double *lse) {
    long G = Hq / Hkv, hk = hq / G;
    const double *qr = q + IDX4(b, hq, r, Hq, N) * d;
    const double *kh = k + IDX4(b, hk, 0, Hkv, N) * d;
    const double *vh = v + IDX4(b, hk, 0, Hkv, N) * d;
    long c0, c1;
    visible_keys(r, N, causal, window, &c0, &c1);
    long nvis = c1 - c0;
    score_row(qr, kh, c0, c1, d, scale, s);
    double m = -INFINITY;
    for (long c = 0; c < nvis; ++c) if (s[c] > m) m = s[c];
    double l = 0.0;
    for (long c = 0; c < nvis; ++c) { s[c] = exp(s[c] - m); l += s[c]; }
    for (long t = 0; t < d; ++t) o_row[t] = 0.0;
    for (long c = 0; c < nvis; ++c) {
        const double *vc = vh + (c0 + c) * d;
        double p = s[c] / l;
        for (long t = 0; t < d; ++t) o_row[t] += p * vc[t];
    }
    *lse = m + log(l);
}

/* O[B][Hq][N][d], lse[B][Hq][N] for the whole problem. */
int oracle_fwd(const double *q, const double *k, const double *v, double *o,
               double *lse, long B, long Hq, long Hkv, long N, long d,
               int causal, long window, double scale) {
    if (!args_ok(B, Hq, Hkv, N, d)) return 1;
    long total = B * Hq * N;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * N);
#pragma omp for schedule(dynamic, 16)
        for (long idx = 0; idx < total; ++idx) {
            long r = idx % N, bh = idx / N, hq = bh % Hq, b = bh / Hq;
            fwd_one_row(q, k, v, b, hq, r, Hq, Hkv, N, d, causal, window,
                        scale, s, o + idx * d, lse + idx);
        }
        free(s);
    }
    return 0;
}

/* Selected rows only: rows[3*i .. 3*i+2] = (b, hq, r).  o_rows[nrows][d]. */
int oracle_fwd_rows(const double *q, const double *k, const double *v,
                    const long *rows, long nrows, double *o_rows,
                    double *lse_rows, long B, long Hq, long Hkv, long N, long d,
                    int causal, long window, double scale) {
    if (!args_ok(B, Hq, Hkv, N, d)) return 1;
    for (long i = 0; i < nrows; ++i) {
        long b = rows[3 * i], h = rows[3 * i + 1], r = rows[3 * i + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || r < 0 || r >= N) return 2;
    }
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * N);
#pragma omp for schedule(dynamic, 1)
        for (long i = 0; i < nrows; ++i)
            fwd_one_row(q, k, v, rows[3 * i], rows[3 * i + 1], rows[3 * i + 2],
                        Hq, Hkv, N, d, causal, window, scale, s, o_rows + i * d,
                        lse_rows + i);
        free(s);
    }
    return 0;
}

/*
 * Backward for one (batch b, key/value head g) group.  Writes
 *   dq_g[G][N][d]  for query heads g*G .. g*G+G-1,
 *   dk_g[N][d], dv_g[N][d]  summed over those G query heads.
 * Three passes, each recomputing the scores it needs:
 *   1. O, L and D = rowsum(dO o O) for every row of every head in the group;
 *   2. dQ_r = scale * sum_c dS_rc K_c (parallel over rows);
 *   3. dV_c = sum_{h,r} P_rc dO_r and dK_c = scale * sum_{h,r} dS_rc Q_r
 *      (parallel over key rows c).
 */
int oracle_bwd_group(const double *q, const double *k, const double *v,
                     const double *dO, long b, long g, double *dq_g,
                     double *dk_g, double *dv_g, long B, long Hq, long Hkv,
                     long N, long d, int causal, long window, double scale) {
    if (!args_ok(B, Hq, Hkv, N, d)) return 1;
    if (b < 0 || b >= B || g < 0 || g >= Hkv) return 2;
    long G = Hq / Hkv;
    double *Og = (double *)malloc(sizeof(double) * G * N * d);
    double *Lg = (double *)malloc(sizeof(double) * G * N);
    double *Dg = (double *)malloc(sizeof(double) * G * N);
    if (!Og || !Lg || !Dg) { free(Og); free(Lg); free(Dg); return 3; }
    const double *kh = k + IDX4(b, g, 0, Hkv, N) * d;
    const double *vh = v + IDX4(b, g, 0, Hkv, N) * d;

    /* pass 1 */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * N);
#pragma omp for schedule(dynamic, 16)
        for (long idx = 0; idx < G * N; ++idx) {
            long j = idx / N, r = idx % N, hq = g * G + j;
            fwd_one_row(q, k, v, b, hq, r, Hq, Hkv, N, d, causal, window,
                        scale, s, Og + idx * d, Lg + idx);
            const double *dor = dO + IDX4(b, hq, r, Hq, N) * d;
            double acc = 0.0;
            for (long t = 0; t < d; ++t) acc += dor[t] * Og[idx * d + t];
            Dg[idx] = acc;
        }
        free(s);
    }

    /* pass 2: dQ */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * N);
#pragma omp for schedule(dynamic, 16)
        for (long idx = 0; idx < G * N; ++idx) {
            long j = idx / N, r = idx % N, hq = g * G + j;
            const double *qr = q + IDX4(b, hq, r, Hq, N) * d;
            const double *dor = dO + IDX4(b, hq, r, Hq, N) * d;
            double *dqr = dq_g + idx * d;
            long c0, c1;
            visible_keys(r, N, causal, window, &c0, &c1);
            score_row(qr, kh, c0, c1, d, scale, s);
            for (long t = 0; t < d; ++t) dqr[t] = 0.0;
            for (long c = c0; c < c1; ++c) {
                double p = exp(s[c - c0] - Lg[idx]);
                const double *vc = vh + c * d;
                double dp = 0.0;
                for (long t = 0; t < d; ++t) dp += dor[t] * vc[t];
                double ds = p * (dp - Dg[idx]);
                const double *kc = kh + c * d;
                for (long t = 0; t < d; ++t) dqr[t] += scale * ds * kc[t];
            }
        }
        free(s);
    }

    /* pass 3: dK, dV */
#pragma omp parallel for schedule(dynamic, 4)
    for (long c = 0; c < N; ++c) {
        const double *kc = kh + c * d;
        const double *vc = vh + c * d;
        double *dkc = dk_g + c * d;
        double *dvc = dv_g + c * d;
        for (long t = 0; t < d; ++t) { dkc[t] = 0.0; dvc[t] = 0.0; }
        for (long j = 0; j < G; ++j) {
            long hq = g * G + j;
            long r0, r1;
            visible_rows(c, N, causal, window, &r0, &r1);
            for (long r = r0; r < r1; ++r) {
                long idx = j * N + r;
                const double *qr = q + IDX4(b, hq, r, Hq, N) * d;
                const double *dor = dO + IDX4(b, hq, r, Hq, N) * d;
                double sc = 0.0, dp = 0.0;
                for (long t = 0; t < d; ++t) { sc += qr[t] * kc[t]; dp += dor[t] * vc[t]; }
                double p = exp(scale * sc - Lg[idx]);
                double ds = p * (dp - Dg[idx]);
                for (long t = 0; t < d; ++t) {
                    dvc[t] += p * dor[t];
                    dkc[t] += scale * ds * qr[t];
                }
            }
        }
    }
    free(Og); free(Lg); free(Dg);
    return 0;
}

/* Whole-problem backward: dq [B][Hq][N][d], dk/dv [B][Hkv][N][d]. */
int oracle_bwd(const double *q, const double *k, const double *v,
               const double *dO, double *dq, double *dk, double *dv, long B,
               long Hq, long Hkv, long N, long d, int causal, long window,
               double scale) {
    if (!args_ok(B, Hq, Hkv, N, d)) return 1;
    long G = Hq / Hkv;
    for (long b = 0; b < B; ++b)
        for (long g = 0; g < Hkv; ++g) {
            int rc = oracle_bwd_group(q, k, v, dO, b, g,
                                      dq + IDX4(b, g * G, 0, Hq, N) * d,
                                      dk + IDX4(b, g, 0, Hkv, N) * d,
                                      dv + IDX4(b, g, 0, Hkv, N) * d, B, Hq,
                                      Hkv, N, d, causal, window, scale);
            if (rc) return rc;
        }
    return 0;
}

/* ---------------------------------------------------------------- FP8 model */

/* Sylvester Hadamard entry H_d[i][j] = (-1)^popcount(i & j), d a power of 2. */
static double sylvester(long i, long j) {
    long x = i & j, par = 0;
    while (x) { par ^= (x & 1); x >>= 1; }
    return par ? -1.0 : 1.0;
}

/* out[r] = (x[r] o s) H_d / sqrt(d) as a dense product; signs may be NULL
 * (then s = 1 and only the orthonormal Hadamard is applied). */
int oracle_hadamard(const double *x, const double *signs, double *out,
                    long rows, long d) {
    if (rows < 0 || d < 1 || (d & (d - 1))) return 1;
    double inv = 1.0 / sqrt((double)d);
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        const double *xr = x + r * d;
        double *orow = out + r * d;
        for (long j = 0; j < d; ++j) {
            double acc = 0.0;
            for (long i = 0; i < d; ++i)
                acc += xr[i] * (signs ? signs[i] : 1.0) * sylvester(i, j);
            orow[j] = acc * inv;
        }
    }
    return 0;
}

/* Round to the nearest e4m3fn value, ties to even, saturating at +-448.
 * Grid: normal numbers (1 + m/8) 2^e for e in [-6, 8], subnormals m 2^-9. */
static double e4m3_round(double x) {
    if (x != x) return x;
    double a = fabs(x);
    double quantum;
    if (a < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9);
    } else {
        int e;
        frexp(a, &e);          /* a = f 2^e with f in [0.5, 1) */
        e -= 1;                /* a in [2^e, 2^(e+1)) */
        if (e > 8) e = 8;
        quantum = ldexp(1.0, e - 3);
    }
    double r = nearbyint(a / quantum) * quantum; /* default mode: ties to even */
    if (r > 448.0) r = 448.0;
    return x < 0 ? -r : r;
}

int oracle_e4m3_round(const double *x, double *out, long n) {
    for (long i = 0; i < n; ++i) out[i] = e4m3_round(x[i]);
    return 0;
}
