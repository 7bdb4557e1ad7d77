/*
 * CPU oracle for the k-means Lloyd iteration and greedy k-means++ seeding.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU library computes.  Only the test-suite, the smoke
 * check and the CPU-baseline leg of the benchmark load it.  It shares no code,
 * header, table or constant with the CUDA library, and it never calls it.
 *
 * Arithmetic is IEEE binary64 throughout: every difference x_f - c_f of two
 * binary32 inputs is exact in binary64, and so is its square, so the only
 * rounding is in the accumulation.  Build with -ffp-contract=off so that the
 * same source gives the same bits on x86-64 and on aarch64.
 *
 * Sources (three pages of one benchmarking journal):
 *  - "Three shapes that fit an eager Gram assignment", section "Gram
 *    assignment": the nearest centroid is the argmin over c of ||x - c||^2.
 *  - same page, section "Running argmin, one centroid": the assignment state is
 *    an int64 label and a float32 winning distance per sample.
 *  - same page, section "Full Lloyd step": the update is the mean of each
 *    centroid's members (the one-hot membership times X, over the counts).
 *  - "004 — tile sizes, a Cython Lloyd step, and k-means++", section
 *    "k-means++": greedy D^2 seeding with 2 + log(n_clusters) candidate trials
 *    per new center.
 *  - Philox4x32-10: Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers:
 *    As Easy as 1, 2, 3", SC'11 (the counter-based generator both sides
 *    implement from that definition for the k-means++ draws).
 *
 * Readings where the pages are silent (each is also listed with the design
 * notes): ties go to the lowest centroid index; an empty cluster keeps its old
 * centroid; the log in the trial count is natural and floored; the first
 * center is uniform; a D^2 draw takes the first sample whose running sum
 * exceeds the target (strictly), and the last sample when none does; equal
 * candidate potentials go to the lowest trial.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 (SC'11 definition): 10 rounds of two 32x32->64 multiplies,  */
/* key schedule bumped by the Weyl constants between rounds.                 */
/* ------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Uniform double in [0,1) for draw number `draw` under `seed`: the top 53 of
 * the first two 32-bit outputs, counter (draw_lo, draw_hi, 0, 0), key (seed_lo,
 * seed_hi). */
double oracle_uniform(uint64_t seed, uint64_t draw) {
    uint32_t ctr[4] = {(uint32_t)draw, (uint32_t)(draw >> 32), 0u, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t r[4];
    oracle_philox4x32_10(ctr, key, r);
    uint64_t bits = (((uint64_t)r[0] << 32) | (uint64_t)r[1]) >> 11;
    return (double)bits * (1.0 / 9007199254740992.0); /* 2^-53 */
}

/* ------------------------------------------------------------------------- */
/* Squared Euclidean distance, by definition: sum over features of the       */
/* squared difference.  Four running partial sums in a fixed order.          */
/* ------------------------------------------------------------------------- */
static double sqdist(const float *x, const float *c, int64_t d) {
    double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
    int64_t f = 0;
    for (; f + 4 <= d; f += 4) {
        double t0 = (double)x[f] - (double)c[f];
        double t1 = (double)x[f + 1] - (double)c[f + 1];
        double t2 = (double)x[f + 2] - (double)c[f + 2];
        double t3 = (double)x[f + 3] - (double)c[f + 3];
        a0 += t0 * t0;
        a1 += t1 * t1;
        a2 += t2 * t2;
        a3 += t3 * t3;
    }
    for (; f < d; ++f) {
        double t = (double)x[f] - (double)c[f];
        a0 += t * t;
    }
    return (a0 + a1) + (a2 + a3);
}

static void set_threads(int nthreads) {
    if (nthreads > 0) omp_set_num_threads(nthreads);
}

int oracle_max_threads(void) { return omp_get_max_threads(); }

double oracle_sqdist(const float *x, const float *c, int64_t d) {
    return sqdist(x, c, d);
}

/* ------------------------------------------------------------------------- */
/* Assignment ("Gram assignment" section): for every sample, the centroid    */
/* with the smallest squared distance; ties go to the lowest index (strict   */
/* '<' while scanning j upward).  Also returns the runner-up distance so a   */
/* caller can tell a near tie from a wrong answer.  Returns the inertia      */
/* (sum of the winning distances, in sample order).                          */
/* ------------------------------------------------------------------------- */
double oracle_assign(const float *X, const float *C, int64_t n, int64_t k,
                     int64_t d, int64_t *labels, double *best, double *second,
                     int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < n; ++i) {
        const float *x = X + i * d;
        double b = INFINITY, s = INFINITY;
        int64_t arg = 0;
        for (int64_t j = 0; j < k; ++j) {
            double dist = sqdist(x, C + j * d, d);
            if (dist < b) {
                s = b;
                b = dist;
                arg = j;
            } else if (dist < s) {
                s = dist;
            }
        }
        labels[i] = arg;
        if (best) best[i] = b;
        if (second) second[i] = s;
    }
    double inertia = 0.0;
    if (best)
        for (int64_t i = 0; i < n; ++i) inertia += best[i];
    return inertia;
}

/* ------------------------------------------------------------------------- */
/* Update ("Full Lloyd step" section): each centroid becomes the mean of the */
/* samples labelled with it, summed in sample order in binary64 and rounded  */
/* once to binary32.  A centroid with no members keeps its old row.          */
/* Columns are split across threads; each column is still summed over the    */
/* samples in index order, so the result does not depend on the thread count.*/
/* ------------------------------------------------------------------------- */
int oracle_update(const float *X, const int64_t *labels, const float *C_old,
                  int64_t n, int64_t k, int64_t d, float *C_new,
                  int64_t *counts, int nthreads) {
    for (int64_t i = 0; i < n; ++i)
        if (labels[i] < 0 || labels[i] >= k) return 1;
    int64_t *cnt = (int64_t *)calloc((size_t)k, sizeof(int64_t));
    if (!cnt) return 2;
    for (int64_t i = 0; i < n; ++i) cnt[labels[i]] += 1;
    set_threads(nthreads);
    const int64_t CB = 64; /* column block per task */
    int64_t nblocks = (d + CB - 1) / CB;
    int err = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)k * CB * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            err = 2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t b = 0; b < nblocks; ++b) {
            if (!acc) continue;
            int64_t f0 = b * CB;
            int64_t w = (d - f0) < CB ? (d - f0) : CB;
            memset(acc, 0, (size_t)k * CB * sizeof(double));
            for (int64_t i = 0; i < n; ++i) {
                double *a = acc + labels[i] * CB;
                const float *x = X + i * d + f0;
                for (int64_t f = 0; f < w; ++f) a[f] += (double)x[f];
            }
            for (int64_t j = 0; j < k; ++j) {
                for (int64_t f = 0; f < w; ++f) {
                    if (cnt[j] == 0)
                        C_new[j * d + f0 + f] = C_old[j * d + f0 + f];
                    else
                        C_new[j * d + f0 + f] =
                            (float)(acc[j * CB + f] / (double)cnt[j]);
                }
            }
        }
        free(acc);
    }
    if (counts)
        for (int64_t j = 0; j < k; ++j) counts[j] = cnt[j];
    free(cnt);
    return err;
}

/* ------------------------------------------------------------------------- */
/* Greedy k-means++ ("k-means++" section of the tile-tradeoff page).         */
/*   draw 0           -> first center, uniform over the samples              */
/*   draw 1+(c-1)*T+t -> trial t of center c                                 */
/* For each new center: every trial samples a candidate with probability     */
/* proportional to D^2 (the squared distance to the nearest chosen center),  */
/* scores it by the potential sum_i min(D^2_i, ||x_i - cand||^2), and the    */
/* lowest-potential trial is kept.  D^2 is then lowered by the new center.   */
/* `margins` (nullable) receives, per draw, the distance of the target from  */
/* the nearest running-sum boundary over the total: how close the draw came  */
/* to picking a neighbouring sample.                                         */
/* ------------------------------------------------------------------------- */
int oracle_kmeanspp(const float *X, int64_t n, int64_t d, int64_t k,
                    int n_trials, uint64_t seed, int64_t *indices,
                    float *centers, double *margins, double *potentials,
                    int nthreads) {
    if (n < 1 || k < 1 || k > n || d < 1) return 1;
    int T = n_trials > 0 ? n_trials : 2 + (int)floor(log((double)k));
    set_threads(nthreads);
    double *D2 = (double *)malloc((size_t)n * sizeof(double));
    double *cum = (double *)malloc((size_t)n * sizeof(double));
    double *dist = (double *)malloc((size_t)n * (size_t)T * sizeof(double));
    int64_t *cand = (int64_t *)malloc((size_t)T * sizeof(int64_t));
    double *pot = (double *)malloc((size_t)T * sizeof(double));
    if (!D2 || !cum || !dist || !cand || !pot) {
        free(D2); free(cum); free(dist); free(cand); free(pot);
        return 2;
    }

    double u0 = oracle_uniform(seed, 0);
    int64_t first = (int64_t)floor(u0 * (double)n);
    if (first > n - 1) first = n - 1;
    indices[0] = first;
    if (margins) {
        double pos = u0 * (double)n;
        double lo = pos - floor(pos), hi = 1.0 - lo;
        margins[0] = (lo < hi ? lo : hi) / (double)n;
    }
    {
        const float *c = X + first * d;
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) D2[i] = sqdist(X + i * d, c, d);
    }
    if (potentials) {
        double tot = 0.0;
        for (int64_t i = 0; i < n; ++i) tot += D2[i];
        potentials[0] = tot;
    }

    for (int64_t cidx = 1; cidx < k; ++cidx) {
        /* running sum of D^2, sequential */
        double run = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            run += D2[i];
            cum[i] = run;
        }
        double total = run;
        for (int t = 0; t < T; ++t) {
            uint64_t draw = 1 + (uint64_t)(cidx - 1) * (uint64_t)T + (uint64_t)t;
            double target = oracle_uniform(seed, draw) * total;
            /* first i with cum[i] > target; binary search on the sorted sums */
            int64_t lo = 0, hi = n; /* answer in [lo, hi] */
            while (lo < hi) {
                int64_t mid = lo + (hi - lo) / 2;
                if (cum[mid] > target) hi = mid; else lo = mid + 1;
            }
            int64_t pick = lo < n ? lo : n - 1;
            cand[t] = pick;
            if (margins) {
                double below = pick > 0 ? cum[pick - 1] : 0.0;
                double m1 = target - below, m2 = cum[pick] - target;
                double m = m1 < m2 ? m1 : m2;
                margins[draw] = total > 0.0 ? fabs(m) / total : 0.0;
            }
        }
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i)
            for (int t = 0; t < T; ++t)
                dist[i * T + t] = sqdist(X + i * d, X + cand[t] * d, d);
        for (int t = 0; t < T; ++t) {
            double p = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                double v = dist[i * T + t];
                p += v < D2[i] ? v : D2[i];
            }
            pot[t] = p;
        }
        int bt = 0;
        for (int t = 1; t < T; ++t)
            if (pot[t] < pot[bt]) bt = t;
        indices[cidx] = cand[bt];
        if (potentials) potentials[cidx] = pot[bt];
        for (int64_t i = 0; i < n; ++i) {
            double v = dist[i * T + bt];
            if (v < D2[i]) D2[i] = v;
        }
    }
    if (centers)
        for (int64_t c = 0; c < k; ++c)
            memcpy(centers + c * d, X + indices[c] * d, (size_t)d * sizeof(float));
    free(D2); free(cum); free(dist); free(cand); free(pot);
    return 0;
}
