/*
 * oracle.c — plain, slow, double-precision CPU oracle for the embedding
 * similarity scan.  TEST INFRASTRUCTURE ONLY: the CUDA library never links,
 * loads or calls this file; only the tests, the smoke check and the CPU
 * baseline leg of the benchmark do.
 *
 * Two computations are restated here, each from its plain definition, in
 * double precision, with every sum taken in ascending index order and no
 * blocking, fusion or reordering:
 *
 *  1. Greedy diversity sequences ("Issue 9-014: Tile Diversity Shader Inner
 *     Loop For L2 Cache Locality", sections Current Behavior and Intended
 *     Behavior).  Each sequence repeatedly picks the unmasked candidate that
 *     is farthest from what it already holds.  The running criterion
 *     is the max-min (farthest-first) reading: every candidate keeps the
 *     smallest cosine distance to any row picked so far, and the pick is the
 *     candidate whose kept distance is largest, lowest index on ties.  The
 *     scan may walk the candidates in tiles of T with the running
 *     (best, index) carried from tile to tile; by associativity of max the
 *     result equals one pass (same issue, Intended Behavior; Suggested
 *     Implementation Steps, the tile loop, whose running maximum carries
 *     over from tile to tile; Risks, the last partial tile).
 *
 *  1b. The centroid criterion named in the same issue (FP16 storage
 *     section, where a candidate is judged by its distance from the
 *     centroid of the held rows): each sequence picks the unmasked
 *     candidate at the largest cosine distance from the centroid (plain
 *     mean) of the rows it holds, lowest index on ties.  A zero centroid
 *     makes every distance 1 (cosine taken as 0).
 *
 *  2. Best-matching-unit search ("From 80x to 385x: A Best-Matching-Unit
 *     Search at the L2 Roof", section 3, Background): for each sample the
 *     index of the codebook row at the smallest squared Euclidean distance,
 *     taken in the direct form sum_k (x_k - w_k)^2, lowest index on ties.
 *
 *  3. The neighbourhood update of a SOM epoch (same page, sections 3
 *     Background and 6, the epoch's composition: every sample's closest
 *     neuron is found first, then that neuron and its neighbours on the map
 *     are updated).  Since the update follows a search over all samples it
 *     is read as the batch map: each neuron becomes the mean of all samples
 *     weighted by the neighbourhood function between the neuron and each
 *     sample's BMU on the grid.
 *
 * Readings where the pages are silent:
 *   - cosine distance d(p, c) = 1 - <e_p, e_c> / (|e_p| |e_c|), in [0, 2];
 *   - the start row seeds the running minimum and is masked; L counts the
 *     picks after the start; the running minimum starts at +infinity;
 *   - the BMU distance is the squared distance (no square root);
 *   - the map is a planar rectangular grid of side_x x side_y neurons,
 *     neuron j at column j % side_x and row j / side_x; the neighbourhood
 *     weight between grid points a and b is exp(-|a - b|^2 / (2 sigma^2))
 *     inside the square window |dx| <= R, |dy| <= R and 0 outside it
 *     (sigma = 0: 1 for a == b, else 0); a neuron whose weights sum to 0
 *     keeps its weights.
 *
 * Parallelism: OpenMP only across independent units (sequences, samples);
 * the arithmetic inside one unit is strictly sequential.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void set_threads(int threads) {
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

/* Threads an OpenMP parallel region will use with this setting. */
int oracle_threads(int threads) {
#ifdef _OPENMP
    set_threads(threads);
    return omp_get_max_threads();
#else
    (void)threads;
    return 1;
#endif
}

/* |e_c| = sqrt(sum_k E[c,k]^2), k ascending, for every row c. */
void oracle_row_norms(const float *E, int64_t N, int32_t D, double *nrm) {
    for (int64_t c = 0; c < N; ++c) {
        double s = 0.0;
        for (int32_t k = 0; k < D; ++k) {
            double v = (double)E[c * (int64_t)D + k];
            s += v * v;
        }
        nrm[c] = sqrt(s);
    }
}

/* Cosine distance between rows p and c. */
static double cosine_distance(const float *E, int32_t D, const double *nrm,
                              int64_t p, int64_t c) {
    double s = 0.0;
    const float *ep = E + p * (int64_t)D;
    const float *ec = E + c * (int64_t)D;
    for (int32_t k = 0; k < D; ++k) s += (double)ep[k] * (double)ec[k];
    return 1.0 - s / (nrm[p] * nrm[c]);
}

/* The fold of the newest pick p into the running minimum:
 * m[c] <- min(m[c], d(p, c)) for every candidate c. */
void oracle_fold(const float *E, int64_t N, int32_t D, const double *nrm,
                 int64_t p, double *m) {
    for (int64_t c = 0; c < N; ++c) {
        double d = cosine_distance(E, D, nrm, p, c);
        if (d < m[c]) m[c] = d;
    }
}

/* The fold for R independent sequences at once (teacher forcing):
 * row r of m (length N) takes the fold of pick p[r]. */
void oracle_fold_batch(const float *E, int64_t N, int32_t D, const double *nrm,
                       const int64_t *p, int32_t R, double *m, int threads) {
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < R; ++r) oracle_fold(E, N, D, nrm, p[r], m + (int64_t)r * N);
}

/* Argmax of m over the unmasked candidates, scanning c ascending in tiles of
 * T candidates ([t*T, min((t+1)*T, N))); T <= 0 means one pass over all N.
 * The running (best, index) is carried across tiles and a candidate replaces
 * it only when strictly larger, so ties go to the lowest index.
 * Returns -1 when every candidate is masked. */
int64_t oracle_argmax(const double *m, const uint8_t *masked, int64_t N, int64_t T) {
    if (T <= 0) T = N;
    double best = -INFINITY;
    int64_t best_idx = -1;
    for (int64_t t0 = 0; t0 < N; t0 += T) {
        int64_t t1 = t0 + T < N ? t0 + T : N;
        for (int64_t c = t0; c < t1; ++c) {
            if (masked[c]) continue;
            if (best_idx < 0 || m[c] > best) {
                best = m[c];
                best_idx = c;
            }
        }
    }
    return best_idx;
}

/* Greedy max-min diversity sequences.
 * E: N x D row-major; starts[B]; mask[N] (NULL = none) excludes candidates
 * from every sequence; picks[B*L] receives the L picks after each start;
 * radius[B*L] (NULL = not wanted) receives the running minimum distance of
 * each pick at the time it was picked.  T is the scan tile (<= 0: one pass).
 * Returns 0, or -1 if a sequence runs out of candidates (its remaining picks
 * are set to -1). */
int oracle_dseq(const float *E, int64_t N, int32_t D, const int32_t *starts,
                int32_t B, int32_t L, const uint8_t *mask, int64_t T,
                int32_t *picks, double *radius, int threads) {
    double *nrm = (double *)malloc(sizeof(double) * (size_t)N);
    if (!nrm) return -2;
    oracle_row_norms(E, N, D, nrm);
    int status = 0;
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(min : status)
    for (int32_t b = 0; b < B; ++b) {
        double *m = (double *)malloc(sizeof(double) * (size_t)N);
        uint8_t *masked = (uint8_t *)malloc((size_t)N);
        if (!m || !masked) {
            free(m);
            free(masked);
            status = -2;
            continue;
        }
        for (int64_t c = 0; c < N; ++c) {
            m[c] = INFINITY;
            masked[c] = mask ? (mask[c] != 0) : 0;
        }
        int64_t p = starts[b];
        masked[p] = 1;
        for (int32_t t = 0; t < L; ++t) {
            oracle_fold(E, N, D, nrm, p, m);
            int64_t w = oracle_argmax(m, masked, N, T);
            picks[(int64_t)b * L + t] = (int32_t)w;
            if (w < 0) {
                for (int32_t u = t; u < L; ++u) picks[(int64_t)b * L + u] = -1;
                status = -1;
                break;
            }
            if (radius) radius[(int64_t)b * L + t] = m[w];
            masked[w] = 1;
            p = w;
        }
        free(m);
        free(masked);
    }
    free(nrm);
    return status;
}

/* Cosine distances of every row to the centroid (plain mean, double) of the
 * rows listed in members[0..n_members): d[c] = 1 - <C, e_c> / (|C| |e_c|),
 * or 1 for every c when the centroid is zero. */
void oracle_centroid_dist(const float *E, int64_t N, int32_t D, const double *nrm,
                          const int64_t *members, int32_t n_members, double *d) {
    double *C = (double *)calloc((size_t)D, sizeof(double));
    if (!C) return;
    for (int32_t i = 0; i < n_members; ++i)
        for (int32_t k = 0; k < D; ++k) C[k] += (double)E[members[i] * (int64_t)D + k];
    double cn = 0.0;
    for (int32_t k = 0; k < D; ++k) {
        C[k] /= (double)n_members;
        cn += C[k] * C[k];
    }
    cn = sqrt(cn);
    for (int64_t c = 0; c < N; ++c) {
        if (cn == 0.0) {
            d[c] = 1.0;
            continue;
        }
        double s = 0.0;
        for (int32_t k = 0; k < D; ++k) s += C[k] * (double)E[c * (int64_t)D + k];
        d[c] = 1.0 - s / (cn * nrm[c]);
    }
    free(C);
}

/* oracle_centroid_dist for R sequences at once (teacher forcing): row r of
 * members (R x n_members) lists sequence r's rows; d is R x N. */
void oracle_centroid_dist_batch(const float *E, int64_t N, int32_t D, const double *nrm,
                                const int64_t *members, int32_t R, int32_t n_members, double *d,
                                int threads) {
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t r = 0; r < R; ++r)
        oracle_centroid_dist(E, N, D, nrm, members + (int64_t)r * n_members, n_members,
                             d + (int64_t)r * N);
}

/* Greedy centroid-criterion sequences (arguments as oracle_dseq); radius
 * receives the centroid distance of each pick. */
int oracle_dseq_centroid(const float *E, int64_t N, int32_t D, const int32_t *starts, int32_t B,
                         int32_t L, const uint8_t *mask, int64_t T, int32_t *picks,
                         double *radius, int threads) {
    double *nrm = (double *)malloc(sizeof(double) * (size_t)N);
    if (!nrm) return -2;
    oracle_row_norms(E, N, D, nrm);
    int status = 0;
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(min : status)
    for (int32_t b = 0; b < B; ++b) {
        double *d = (double *)malloc(sizeof(double) * (size_t)N);
        uint8_t *masked = (uint8_t *)malloc((size_t)N);
        int64_t *members = (int64_t *)malloc(sizeof(int64_t) * (size_t)(L + 1));
        if (!d || !masked || !members) {
            free(d);
            free(masked);
            free(members);
            status = -2;
            continue;
        }
        for (int64_t c = 0; c < N; ++c) masked[c] = mask ? (mask[c] != 0) : 0;
        members[0] = starts[b];
        masked[starts[b]] = 1;
        for (int32_t t = 0; t < L; ++t) {
            oracle_centroid_dist(E, N, D, nrm, members, t + 1, d);
            int64_t w = oracle_argmax(d, masked, N, T);
            picks[(int64_t)b * L + t] = (int32_t)w;
            if (w < 0) {
                for (int32_t u = t; u < L; ++u) picks[(int64_t)b * L + u] = -1;
                status = -1;
                break;
            }
            if (radius) radius[(int64_t)b * L + t] = d[w];
            masked[w] = 1;
            members[t + 1] = w;
        }
        free(d);
        free(masked);
        free(members);
    }
    free(nrm);
    return status;
}

/* Squared Euclidean distance in the direct form, k ascending. */
static double sqdist(const float *x, const float *w, int32_t D) {
    double s = 0.0;
    for (int32_t k = 0; k < D; ++k) {
        double diff = (double)x[k] - (double)w[k];
        s += diff * diff;
    }
    return s;
}

/* Best-matching unit of every sample.
 * X: n x D, W: M x D, both row-major.  idx[i] = the first j reaching the
 * minimum of sqdist(X_i, W_j) (strict '<' while scanning j ascending);
 * dist[i] = that minimum; second[i] (NULL = not wanted) = the smallest
 * distance over j != idx[i], used to recognise near-ties. */
void oracle_bmu(const float *X, int64_t n, const float *W, int64_t M, int32_t D,
                int32_t *idx, double *dist, double *second, int threads) {
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < n; ++i) {
        const float *x = X + i * (int64_t)D;
        double best = INFINITY, runner = INFINITY;
        int64_t best_j = -1;
        for (int64_t j = 0; j < M; ++j) {
            double d = sqdist(x, W + j * (int64_t)D, D);
            if (best_j < 0 || d < best) {
                runner = best;
                best = d;
                best_j = j;
            } else if (d < runner) {
                runner = d;
            }
        }
        idx[i] = (int32_t)best_j;
        dist[i] = best;
        if (second) second[i] = runner;
    }
}

/* sqdist(X_{ii[r]}, W_{jj[r]}) for R given (sample, neuron) pairs. */
void oracle_sqdist_pairs(const float *X, const float *W, int32_t D, const int64_t *ii,
                         const int64_t *jj, int64_t R, double *out) {
    for (int64_t r = 0; r < R; ++r)
        out[r] = sqdist(X + ii[r] * (int64_t)D, W + jj[r] * (int64_t)D, D);
}

/* Batch-map update of the listed neurons.
 * X: n x D samples, bmu[i] their BMUs, W: M x D codebook (M = side_x *
 * side_y).  For each listed neuron j, visiting the samples in ascending
 * order, num = sum_i h(j, bmu[i]) X_i and den = sum_i h(j, bmu[i]); the
 * row out[r] (neuron neurons[r]) is num / den, or W_j when den is 0. */
void oracle_som_update(const float *X, int64_t n, int32_t D, const int32_t *bmu, const float *W,
                       int32_t side_x, int32_t side_y, double sigma, int32_t radius,
                       const int64_t *neurons, int64_t n_neurons, double *out, int threads) {
    (void)side_y;
    set_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_neurons; ++r) {
        const int64_t j = neurons[r];
        const int64_t xj = j % side_x, yj = j / side_x;
        double *num = out + r * (int64_t)D;
        double den = 0.0;
        for (int32_t k = 0; k < D; ++k) num[k] = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            const int64_t c = bmu[i];
            const int64_t dx = c % side_x - xj, dy = c / side_x - yj;
            if (dx > radius || dx < -radius || dy > radius || dy < -radius) continue;
            double h;
            if (sigma > 0.0)
                h = exp(-(double)(dx * dx + dy * dy) / (2.0 * sigma * sigma));
            else
                h = (dx == 0 && dy == 0) ? 1.0 : 0.0;
            if (h == 0.0) continue;
            den += h;
            const float *x = X + i * (int64_t)D;
            for (int32_t k = 0; k < D; ++k) num[k] += h * (double)x[k];
        }
        const float *w = W + j * (int64_t)D;
        for (int32_t k = 0; k < D; ++k) num[k] = den > 0.0 ? num[k] / den : (double)w[k];
    }
}
