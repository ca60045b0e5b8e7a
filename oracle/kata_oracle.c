/*
 * kata_oracle.c -- plain CPU oracle for causal kernelized linear attention with
 * the rank-one PSD feature map (KATA).  TEST INFRASTRUCTURE ONLY: the product
 * path never links, loads or calls this file; only the tests, the smoke check
 * and the benchmark's CPU-baseline leg do.
 *
 * Everything here is computed in double precision with no blocking, fusion or
 * reordering beyond what the cited definitions state, so that each function can
 * be checked against the paper by eye.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Source: "Kernelized Linear Attention: Breaking the Capacity Wall with
 * Symmetric Cones" (KATA, arXiv 2607.17419v1):
 *   - Sec. 2, Eq. 2: normalised linear attention
 *       o_t = psi(q_t)^T S_t / psi(q_t)^T Z_t,
 *       S_t = sum_{i<=t} psi(k_i) v_i^T,  Z_t = sum_{i<=t} psi(k_i),
 *     with the additive recurrence S_t = S_{t-1} + psi(k_t) v_t^T,
 *     Z_t = Z_{t-1} + psi(k_t); the readout is defined when the denominator
 *     is positive.
 *   - Sec. 3.1: rank-one PSD lift psi(u) = u u^T with
 *     <u u^T, v v^T>_F = (u^T v)^2, in the n = p(p+1)/2 dimensional ambient
 *     space of symmetric matrices under the Frobenius inner product.
 *   - Sec. 4.1: n = d(d+1)/2 unique coordinates after symmetry packing;
 *     chunkwise forward Eq. 17-20.
 *   - App. D.2, Algorithm 1: chunkwise forward for one head (pad the final
 *     chunk, S_0 = 0, Z_0 = 0, per chunk: expand psi, output via Eq. 20, then
 *     update the state via Eq. 17, truncate to T).
 *   - App. D.1 "Plain KATA": the additive recurrence (used for decoding).
 *
 * Readings where the paper is silent (each is listed with its reason in the
 * design notes of the repository):
 *   - packing: upper triangle (i <= j), row-major order
 *       f(i,j) = i*d - i*(i-1)/2 + (j - i),
 *     diagonal entries x_i^2, off-diagonal entries sqrt(2) x_i x_j, which makes
 *     the packed vector an isometric image of x x^T under the Frobenius norm.
 *   - the causal sum is inclusive (s <= t), as in Eq. 1-2;
 *   - no 1/sqrt(d) or temperature is applied;
 *   - a zero denominator gives a zero output row.
 *
 * Layouts: q, k are [B*H][T][d], v and out are [B*H][T][dv], all contiguous
 * double.  The decode state is S [B*H][n][dv] and z [B*H][n].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 0; /* 0: OpenMP default */

void kata_oracle_set_threads(int n) { g_threads = n; }

int kata_oracle_get_threads(void) {
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

/* n = d(d+1)/2: the packed width of a symmetric d x d matrix (Sec. 4.1). */
int kata_oracle_feature_dim(int d) { return d * (d + 1) / 2; }

/* Rank-one PSD lift of one vector x in R^d (Sec. 3.1, packed as Sec. 4.1). */
static void lift_one(const double *x, int d, double *phi) {
    const double r2 = sqrt(2.0);
    int f = 0;
    for (int i = 0; i < d; ++i) {
        for (int j = i; j < d; ++j) {
            phi[f] = (i == j) ? x[i] * x[i] : r2 * x[i] * x[j];
            ++f;
        }
    }
}

/* Lift `rows` vectors: x [rows][d] -> phi [rows][n]. */
void kata_oracle_lift(const double *x, int64_t rows, int d, double *phi) {
    const int n = kata_oracle_feature_dim(d);
    for (int64_t r = 0; r < rows; ++r) lift_one(x + r * d, d, phi + r * n);
}

/* The direct definition (Eq. 2 with psi the rank-one lift) for one output row:
 * w_s = (q_t . k_s)^2 for s <= t, o_t = sum_s w_s v_s / sum_s w_s. */
static void direct_row(const double *q, const double *k, const double *v, int t, int d,
                       int dv, double *o) {
    const double *qt = q + (int64_t)t * d;
    double den = 0.0;
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int s = 0; s <= t; ++s) {
        const double *ks = k + (int64_t)s * d;
        double dot = 0.0;
        for (int i = 0; i < d; ++i) dot += qt[i] * ks[i];
        const double w = dot * dot;
        den += w;
        const double *vs = v + (int64_t)s * dv;
        for (int j = 0; j < dv; ++j) o[j] += w * vs[j];
    }
    for (int j = 0; j < dv; ++j) o[j] = den > 0.0 ? o[j] / den : 0.0;
}

/* Full causal forward by the direct O(T^2) definition. */
void kata_oracle_forward(const double *q, const double *k, const double *v, double *out,
                         int BH, int T, int d, int dv) {
    const int64_t total = (int64_t)BH * T;
#pragma omp parallel for schedule(dynamic, 16) num_threads(kata_oracle_get_threads())
    for (int64_t r = 0; r < total; ++r) {
        const int64_t bh = r / T;
        const int t = (int)(r % T);
        direct_row(q + bh * T * d, k + bh * T * d, v + bh * T * dv, t, d, dv,
                   out + r * dv);
    }
}

/* The same definition evaluated only at sampled rows.  rows[i] = bh*T + t;
 * out is [nrows][dv]. */
void kata_oracle_forward_rows(const double *q, const double *k, const double *v,
                              const int64_t *rows, int64_t nrows, double *out, int BH,
                              int T, int d, int dv) {
    (void)BH;
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t bh = rows[i] / T;
        const int t = (int)(rows[i] % T);
        direct_row(q + bh * T * d, k + bh * T * d, v + bh * T * dv, t, d, dv,
                   out + i * dv);
    }
}

/* Self-check form 1: the explicit feature-state recurrence of Eq. 2,
 * S_t = S_{t-1} + psi(k_t) v_t^T, Z_t = Z_{t-1} + psi(k_t),
 * o_t = psi(q_t)^T S_t / psi(q_t)^T Z_t. */
void kata_oracle_recurrent(const double *q, const double *k, const double *v,
                           double *out, int BH, int T, int d, int dv) {
    const int n = kata_oracle_feature_dim(d);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *S = calloc((size_t)n * dv, sizeof(double));
        double *Z = calloc((size_t)n, sizeof(double));
        double *pk = malloc((size_t)n * sizeof(double));
        double *pq = malloc((size_t)n * sizeof(double));
        for (int t = 0; t < T; ++t) {
            const int64_t row = (int64_t)bh * T + t;
            lift_one(k + row * d, d, pk);
            lift_one(q + row * d, d, pq);
            const double *vt = v + row * dv;
            for (int f = 0; f < n; ++f) {
                for (int j = 0; j < dv; ++j) S[(size_t)f * dv + j] += pk[f] * vt[j];
                Z[f] += pk[f];
            }
            double den = 0.0;
            for (int f = 0; f < n; ++f) den += pq[f] * Z[f];
            double *o = out + row * dv;
            for (int j = 0; j < dv; ++j) {
                double num = 0.0;
                for (int f = 0; f < n; ++f) num += pq[f] * S[(size_t)f * dv + j];
                o[j] = den > 0.0 ? num / den : 0.0;
            }
        }
        free(S);
        free(Z);
        free(pk);
        free(pq);
    }
}

/* Self-check form 2: Algorithm 1 (App. D.2) with the chunk equations 17-20.
 * N_C = ceil(T/C); the final chunk is padded with zero rows; S = 0, Z = 0;
 * per chunk: Psi(Q), Psi(K); P = (Psi(Q) Psi(K)^T) .* M (M lower-triangular,
 * diagonal included); N = Psi(Q) S + P V; D = Psi(Q) Z + P 1; O = diag(D)^-1 N;
 * then S += Psi(K)^T V, Z += Psi(K)^T 1; finally truncate to T rows. */
void kata_oracle_chunked(const double *q, const double *k, const double *v, double *out,
                         int BH, int T, int d, int dv, int C) {
    const int n = kata_oracle_feature_dim(d);
    const int NC = (T + C - 1) / C;
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *S = calloc((size_t)n * dv, sizeof(double));
        double *Z = calloc((size_t)n, sizeof(double));
        double *PQ = calloc((size_t)C * n, sizeof(double));
        double *PK = calloc((size_t)C * n, sizeof(double));
        double *Vc = calloc((size_t)C * dv, sizeof(double));
        double *P = calloc((size_t)C * C, sizeof(double));
        double *N = calloc((size_t)C * dv, sizeof(double));
        double *D = calloc((size_t)C, sizeof(double));
        for (int c = 0; c < NC; ++c) {
            /* load the chunk, zero-padding rows past T */
            for (int r = 0; r < C; ++r) {
                const int t = c * C + r;
                if (t < T) {
                    const int64_t row = (int64_t)bh * T + t;
                    lift_one(q + row * d, d, PQ + (size_t)r * n);
                    lift_one(k + row * d, d, PK + (size_t)r * n);
                    memcpy(Vc + (size_t)r * dv, v + row * dv, sizeof(double) * dv);
                } else {
                    memset(PQ + (size_t)r * n, 0, sizeof(double) * n);
                    memset(PK + (size_t)r * n, 0, sizeof(double) * n);
                    memset(Vc + (size_t)r * dv, 0, sizeof(double) * dv);
                }
            }
            /* P = (Psi(Q) Psi(K)^T) .* M */
            for (int r = 0; r < C; ++r)
                for (int s = 0; s < C; ++s) {
                    double acc = 0.0;
                    if (s <= r)
                        for (int f = 0; f < n; ++f)
                            acc += PQ[(size_t)r * n + f] * PK[(size_t)s * n + f];
                    P[(size_t)r * C + s] = acc;
                }
            /* Eq. 18-19 */
            for (int r = 0; r < C; ++r) {
                double dacc = 0.0;
                for (int f = 0; f < n; ++f) dacc += PQ[(size_t)r * n + f] * Z[f];
                for (int s = 0; s < C; ++s) dacc += P[(size_t)r * C + s];
                D[r] = dacc;
                for (int j = 0; j < dv; ++j) {
                    double nacc = 0.0;
                    for (int f = 0; f < n; ++f)
                        nacc += PQ[(size_t)r * n + f] * S[(size_t)f * dv + j];
                    for (int s = 0; s < C; ++s)
                        nacc += P[(size_t)r * C + s] * Vc[(size_t)s * dv + j];
                    N[(size_t)r * dv + j] = nacc;
                }
            }
            /* Eq. 20, truncated to T */
            for (int r = 0; r < C; ++r) {
                const int t = c * C + r;
                if (t >= T) break;
                double *o = out + ((int64_t)bh * T + t) * dv;
                for (int j = 0; j < dv; ++j)
                    o[j] = D[r] > 0.0 ? N[(size_t)r * dv + j] / D[r] : 0.0;
            }
            /* Eq. 17 */
            for (int f = 0; f < n; ++f) {
                for (int j = 0; j < dv; ++j) {
                    double acc = 0.0;
                    for (int s = 0; s < C; ++s)
                        acc += PK[(size_t)s * n + f] * Vc[(size_t)s * dv + j];
                    S[(size_t)f * dv + j] += acc;
                }
                double zacc = 0.0;
                for (int s = 0; s < C; ++s) zacc += PK[(size_t)s * n + f];
                Z[f] += zacc;
            }
        }
        free(S);
        free(Z);
        free(PQ);
        free(PK);
        free(Vc);
        free(P);
        free(N);
        free(D);
    }
}

/* The state pair (S_T, Z_T) after T tokens, by the additive recurrence of
 * Eq. 2 / App. D.1.  S is [BH][n][dv], z is [BH][n]. */
void kata_oracle_prefix_state(const double *k, const double *v, double *S, double *z,
                              int BH, int T, int d, int dv) {
    const int n = kata_oracle_feature_dim(d);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * n * dv;
        double *zb = z + (size_t)bh * n;
        double *pk = malloc((size_t)n * sizeof(double));
        memset(Sb, 0, sizeof(double) * n * dv);
        memset(zb, 0, sizeof(double) * n);
        for (int t = 0; t < T; ++t) {
            const int64_t row = (int64_t)bh * T + t;
            lift_one(k + row * d, d, pk);
            for (int f = 0; f < n; ++f) {
                for (int j = 0; j < dv; ++j)
                    Sb[(size_t)f * dv + j] += pk[f] * v[row * dv + j];
                zb[f] += pk[f];
            }
        }
        free(pk);
    }
}

/* One recurrent decode step (App. D.1, Plain KATA), in place:
 * S += psi(k) v^T, z += psi(k), then o = psi(q)^T S / psi(q)^T z
 * (update, then read: the step's own key is included, as in Eq. 2).
 * q, k are [BH][d], v and out are [BH][dv]. */
void kata_oracle_decode_step(double *S, double *z, const double *q, const double *k,
                             const double *v, double *out, int BH, int d, int dv) {
    const int n = kata_oracle_feature_dim(d);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * n * dv;
        double *zb = z + (size_t)bh * n;
        double *pk = malloc((size_t)n * sizeof(double));
        double *pq = malloc((size_t)n * sizeof(double));
        lift_one(k + (size_t)bh * d, d, pk);
        lift_one(q + (size_t)bh * d, d, pq);
        const double *vb = v + (size_t)bh * dv;
        for (int f = 0; f < n; ++f) {
            for (int j = 0; j < dv; ++j) Sb[(size_t)f * dv + j] += pk[f] * vb[j];
            zb[f] += pk[f];
        }
        double den = 0.0;
        for (int f = 0; f < n; ++f) den += pq[f] * zb[f];
        for (int j = 0; j < dv; ++j) {
            double num = 0.0;
            for (int f = 0; f < n; ++f) num += pq[f] * Sb[(size_t)f * dv + j];
            out[(size_t)bh * dv + j] = den > 0.0 ? num / den : 0.0;
        }
        free(pk);
        free(pq);
    }
}

/* ---------------------------------------------------------------------------
 * Reduced PSD families (Sec. 4.1, "two reduced PSD families"; the
 * configuration appendix for the Sigma maps' eps I term and scale).  The
 * vector u in R^d is cut into g blocks u_a of width m = d / g:
 *   map 1, KATA-M_g:     psi(u) = (u_1 u_1^T, ..., u_g u_g^T), g matrices m x m,
 *                        <psi(q), psi(k)> = sum_a (q_a . k_a)^2;
 *   map 2, KATA-Sigma_g: psi(u) = eps I + s * sum_a u_a u_a^T, one m x m matrix
 *                        (eps: a numerical safeguard the Sigma configuration
 *                        sets to 1e-4; s: 1/4 in its reported Sigma_4 setup);
 *   map 0: the full rank-one map (g = 1);
 *   map 3, orthant (the linear-state family of the pages' kernel appendix, one
 *                        feature per coordinate): psi(u)_i = max(u_i, 0) + eps,
 *                        n = d (eps: 1e-6 in the pages' configuration).
 * Both families give the full map at g = 1 (eps = 0, s = 1).  Inner products
 * are Frobenius; each matrix is packed like the full map (upper triangle,
 * row-major, sqrt(2) off the diagonal), the g matrices of M_g in block order.
 * ------------------------------------------------------------------------- */

/* Packed feature width of a map (the pages' dominant state size over d_v). */
int kata_oracle_map_dim(int map, int d, int g) {
    const int m = d / g;
    if (map == 3) return d;
    if (map == 1) return g * m * (m + 1) / 2;
    if (map == 2) return m * (m + 1) / 2;
    return d * (d + 1) / 2;
}

/* The map's matrices for one vector u, written out from the definitions:
 * A[a][i][j] for a < count, each w x w.  Returns count; *w_out = w. */
static int map_matrices(const double *u, int d, int map, int g, double eps, double s,
                        double *A, int *w_out) {
    if (map == 1) {
        const int m = d / g;
        *w_out = m;
        for (int a = 0; a < g; ++a)
            for (int i = 0; i < m; ++i)
                for (int j = 0; j < m; ++j)
                    A[((size_t)a * m + i) * m + j] = u[a * m + i] * u[a * m + j];
        return g;
    }
    if (map == 2) {
        const int m = d / g;
        *w_out = m;
        for (int i = 0; i < m; ++i)
            for (int j = 0; j < m; ++j) {
                double acc = 0.0;
                for (int a = 0; a < g; ++a) acc += u[a * m + i] * u[a * m + j];
                A[(size_t)i * m + j] = (i == j ? eps : 0.0) + s * acc;
            }
        return 1;
    }
    *w_out = d;
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) A[(size_t)i * d + j] = u[i] * u[j];
    return 1;
}

/* Packed lift of one vector under a map; A is scratch of at least d*d. */
static void lift_map_one(const double *x, int d, int map, int g, double eps, double s,
                         double *phi, double *A) {
    if (map == 3) {   /* orthant: coordinatewise */
        for (int i = 0; i < d; ++i) phi[i] = (x[i] > 0.0 ? x[i] : 0.0) + eps;
        return;
    }
    const double r2 = sqrt(2.0);
    int w = 0;
    const int count = map_matrices(x, d, map, g, eps, s, A, &w);
    int f = 0;
    for (int a = 0; a < count; ++a)
        for (int i = 0; i < w; ++i)
            for (int j = i; j < w; ++j) {
                const double e = A[((size_t)a * w + i) * w + j];
                phi[f++] = (i == j) ? e : r2 * e;
            }
}

void kata_oracle_lift_map(const double *x, int64_t rows, int d, int map, int g, double eps,
                          double s, double *phi) {
    const int n = kata_oracle_map_dim(map, d, g);
    double *A = malloc(sizeof(double) * (size_t)d * d);
    for (int64_t r = 0; r < rows; ++r) lift_map_one(x + r * d, d, map, g, eps, s, phi + r * n, A);
    free(A);
}

/* <psi(q), psi(k)>_F as the entrywise sum over the map's matrices. */
static double map_weight(const double *q, const double *k, int d, int map, int g, double eps,
                         double s, double *Aq, double *Ak) {
    if (map == 3) {   /* orthant: the dot product of the two feature vectors */
        double acc = 0.0;
        for (int i = 0; i < d; ++i)
            acc += ((q[i] > 0.0 ? q[i] : 0.0) + eps) * ((k[i] > 0.0 ? k[i] : 0.0) + eps);
        return acc;
    }
    int w = 0;
    const int count = map_matrices(q, d, map, g, eps, s, Aq, &w);
    map_matrices(k, d, map, g, eps, s, Ak, &w);
    double acc = 0.0;
    for (size_t e = 0; e < (size_t)count * w * w; ++e) acc += Aq[e] * Ak[e];
    return acc;
}

/* Eq. 2 with the map's psi, one output row t (direct O(T) sum over s <= t). */
static void direct_row_map(const double *q, const double *k, const double *v, int t, int d,
                           int dv, int map, int g, double eps, double s, double *o) {
    double *Aq = malloc(sizeof(double) * (size_t)d * d);
    double *Ak = malloc(sizeof(double) * (size_t)d * d);
    const double *qt = q + (int64_t)t * d;
    double den = 0.0;
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int si = 0; si <= t; ++si) {
        const double w = map_weight(qt, k + (int64_t)si * d, d, map, g, eps, s, Aq, Ak);
        den += w;
        const double *vs = v + (int64_t)si * dv;
        for (int j = 0; j < dv; ++j) o[j] += w * vs[j];
    }
    for (int j = 0; j < dv; ++j) o[j] = den > 0.0 ? o[j] / den : 0.0;
    free(Aq);
    free(Ak);
}

void kata_oracle_forward_map(const double *q, const double *k, const double *v, double *out,
                             int BH, int T, int d, int dv, int map, int g, double eps,
                             double s) {
    const int64_t total = (int64_t)BH * T;
#pragma omp parallel for schedule(dynamic, 16) num_threads(kata_oracle_get_threads())
    for (int64_t r = 0; r < total; ++r) {
        const int64_t bh = r / T;
        const int t = (int)(r % T);
        direct_row_map(q + bh * T * d, k + bh * T * d, v + bh * T * dv, t, d, dv, map, g, eps,
                       s, out + r * dv);
    }
}

void kata_oracle_forward_rows_map(const double *q, const double *k, const double *v,
                                  const int64_t *rows, int64_t nrows, double *out, int BH,
                                  int T, int d, int dv, int map, int g, double eps, double s) {
    (void)BH;
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t bh = rows[i] / T;
        const int t = (int)(rows[i] % T);
        direct_row_map(q + bh * T * d, k + bh * T * d, v + bh * T * dv, t, d, dv, map, g, eps,
                       s, out + i * dv);
    }
}

/* Self-check form: the packed-feature recurrence of Eq. 2 under the map. */
void kata_oracle_recurrent_map(const double *q, const double *k, const double *v, double *out,
                               int BH, int T, int d, int dv, int map, int g, double eps,
                               double s) {
    const int n = kata_oracle_map_dim(map, d, g);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *S = calloc((size_t)n * dv, sizeof(double));
        double *Z = calloc((size_t)n, sizeof(double));
        double *pk = malloc((size_t)n * sizeof(double));
        double *pq = malloc((size_t)n * sizeof(double));
        double *A = malloc(sizeof(double) * (size_t)d * d);
        for (int t = 0; t < T; ++t) {
            const int64_t row = (int64_t)bh * T + t;
            lift_map_one(k + row * d, d, map, g, eps, s, pk, A);
            lift_map_one(q + row * d, d, map, g, eps, s, pq, A);
            const double *vt = v + row * dv;
            for (int f = 0; f < n; ++f) {
                for (int j = 0; j < dv; ++j) S[(size_t)f * dv + j] += pk[f] * vt[j];
                Z[f] += pk[f];
            }
            double den = 0.0;
            for (int f = 0; f < n; ++f) den += pq[f] * Z[f];
            double *o = out + row * dv;
            for (int j = 0; j < dv; ++j) {
                double num = 0.0;
                for (int f = 0; f < n; ++f) num += pq[f] * S[(size_t)f * dv + j];
                o[j] = den > 0.0 ? num / den : 0.0;
            }
        }
        free(S);
        free(Z);
        free(pk);
        free(pq);
        free(A);
    }
}

/* The state pair after T tokens under a map (Eq. 2's additive recurrence with
 * the map's psi): S = sum_t psi(k_t) v_t^T [BH][n][dv], z = sum_t psi(k_t)
 * [BH][n], features in the packed order of kata_oracle_lift_map. */
void kata_oracle_prefix_state_map(const double *k, const double *v, double *S, double *z,
                                  int BH, int T, int d, int dv, int map, int g, double eps,
                                  double s) {
    const int n = kata_oracle_map_dim(map, d, g);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * n * dv;
        double *zb = z + (size_t)bh * n;
        double *pk = malloc((size_t)n * sizeof(double));
        double *A = malloc(sizeof(double) * (size_t)d * d);
        memset(Sb, 0, sizeof(double) * n * dv);
        memset(zb, 0, sizeof(double) * n);
        for (int t = 0; t < T; ++t) {
            const int64_t row = (int64_t)bh * T + t;
            lift_map_one(k + row * d, d, map, g, eps, s, pk, A);
            for (int f = 0; f < n; ++f) {
                for (int j = 0; j < dv; ++j) Sb[(size_t)f * dv + j] += pk[f] * v[row * dv + j];
                zb[f] += pk[f];
            }
        }
        free(pk);
        free(A);
    }
}

/* One decode step under a map, in place: S += psi(k) v^T, z += psi(k), then
 * o = psi(q)^T S / psi(q)^T z (0 where the denominator is not positive). */
void kata_oracle_decode_step_map(double *S, double *z, const double *q, const double *k,
                                 const double *v, double *out, int BH, int d, int dv, int map,
                                 int g, double eps, double s) {
    const int n = kata_oracle_map_dim(map, d, g);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * n * dv;
        double *zb = z + (size_t)bh * n;
        double *pk = malloc((size_t)n * sizeof(double));
        double *pq = malloc((size_t)n * sizeof(double));
        double *A = malloc(sizeof(double) * (size_t)d * d);
        lift_map_one(k + (size_t)bh * d, d, map, g, eps, s, pk, A);
        lift_map_one(q + (size_t)bh * d, d, map, g, eps, s, pq, A);
        const double *vb = v + (size_t)bh * dv;
        for (int f = 0; f < n; ++f) {
            for (int j = 0; j < dv; ++j) Sb[(size_t)f * dv + j] += pk[f] * vb[j];
            zb[f] += pk[f];
        }
        double den = 0.0;
        for (int f = 0; f < n; ++f) den += pq[f] * zb[f];
        for (int j = 0; j < dv; ++j) {
            double num = 0.0;
            for (int f = 0; f < n; ++f) num += pq[f] * Sb[(size_t)f * dv + j];
            out[(size_t)bh * dv + j] = den > 0.0 ? num / den : 0.0;
        }
        free(pk);
        free(pq);
        free(A);
    }
}

/* ---------------------------------------------------------------------------
 * GatedKATA (the appendix on recurrent variants, "multiplicative scalar state
 * gate", and Sec. 5.2): a scalar gate gamma_t in [0, 1] inside the recurrence,
 *   S_t = gamma_t S_{t-1} + psi(k_t) v_t^T,
 * which unrolls to S_t = sum_{s<=t} (prod_{r=s+1}^{t} gamma_r) psi(k_s) v_s^T:
 * write s is weighted by the gates of the later tokens only.  Readings (each
 * listed with its reason in the design notes of the repository):
 *   - Z_t carries the same gate, Z_t = gamma_t Z_{t-1} + psi(k_t), so the
 *     readout psi(q_t)^T S_t / psi(q_t)^T Z_t is the convex output gate of
 *     Prop. 1 over the gated weights (normalize = 1);
 *   - normalize = 0 gives the no-denominator readout o_t = psi(q_t)^T S_t of the
 *     MQAR configuration appendix;
 *   - gamma is given per (head, token) as a value in [0, 1]: gamma [BH][T] for
 *     the forward, gamma [BH] for one decode step. */

/* The direct definition for one output row: weights a_ts (q_t . k_s)^2 with
 * a_tt = 1 and a_t,s-1 = a_ts gamma_s (the product over r = s .. t). */
static void gated_row(const double *q, const double *k, const double *v, const double *gamma,
                      int t, int d, int dv, int normalize, double *o) {
    const double *qt = q + (int64_t)t * d;
    double den = 0.0, a = 1.0;
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int s = t; s >= 0; --s) {
        const double *ks = k + (int64_t)s * d;
        double dot = 0.0;
        for (int i = 0; i < d; ++i) dot += qt[i] * ks[i];
        const double w = a * dot * dot;
        den += w;
        const double *vs = v + (int64_t)s * dv;
        for (int j = 0; j < dv; ++j) o[j] += w * vs[j];
        a *= gamma[s];
    }
    if (normalize)
        for (int j = 0; j < dv; ++j) o[j] = den > 0.0 ? o[j] / den : 0.0;
}

/* Full causal gated forward by the direct O(T^2) definition. */
void kata_oracle_forward_gated(const double *q, const double *k, const double *v,
                               const double *gamma, double *out, int BH, int T, int d, int dv,
                               int normalize) {
    const int64_t total = (int64_t)BH * T;
#pragma omp parallel for schedule(dynamic, 16) num_threads(kata_oracle_get_threads())
    for (int64_t r = 0; r < total; ++r) {
        const int64_t bh = r / T;
        const int t = (int)(r % T);
        gated_row(q + bh * T * d, k + bh * T * d, v + bh * T * dv, gamma + bh * T, t, d, dv,
                  normalize, out + r * dv);
    }
}

/* The same at sampled rows: rows[i] = bh*T + t, out [nrows][dv]. */
void kata_oracle_forward_rows_gated(const double *q, const double *k, const double *v,
                                    const double *gamma, const int64_t *rows, int64_t nrows,
                                    double *out, int BH, int T, int d, int dv, int normalize) {
    (void)BH;
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t bh = rows[i] / T;
        const int t = (int)(rows[i] % T);
        gated_row(q + bh * T * d, k + bh * T * d, v + bh * T * dv, gamma + bh * T, t, d, dv,
                  normalize, out + i * dv);
    }
}

/* Self-check form: the gated feature-state recurrence itself,
 * S_t = gamma_t S_{t-1} + psi(k_t) v_t^T, Z_t = gamma_t Z_{t-1} + psi(k_t),
 * read out as psi(q_t)^T S_t (/ psi(q_t)^T Z_t when normalize). */
void kata_oracle_recurrent_gated(const double *q, const double *k, const double *v,
                                 const double *gamma, double *out, int BH, int T, int d, int dv,
                                 int normalize) {
    const int n = kata_oracle_feature_dim(d);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *S = calloc((size_t)n * dv, sizeof(double));
        double *Z = calloc((size_t)n, sizeof(double));
        double *pk = malloc((size_t)n * sizeof(double));
        double *pq = malloc((size_t)n * sizeof(double));
        for (int t = 0; t < T; ++t) {
            const int64_t row = (int64_t)bh * T + t;
            const double g = gamma[row];
            lift_one(k + row * d, d, pk);
            lift_one(q + row * d, d, pq);
            const double *vt = v + row * dv;
            for (int f = 0; f < n; ++f) {
                for (int j = 0; j < dv; ++j)
                    S[(size_t)f * dv + j] = g * S[(size_t)f * dv + j] + pk[f] * vt[j];
                Z[f] = g * Z[f] + pk[f];
            }
            double den = 0.0;
            for (int f = 0; f < n; ++f) den += pq[f] * Z[f];
            double *o = out + row * dv;
            for (int j = 0; j < dv; ++j) {
                double num = 0.0;
                for (int f = 0; f < n; ++f) num += pq[f] * S[(size_t)f * dv + j];
                o[j] = normalize ? (den > 0.0 ? num / den : 0.0) : num;
            }
        }
        free(S);
        free(Z);
        free(pk);
        free(pq);
    }
}

/* (S_T, Z_T) after T tokens under the gated recurrence.  S [BH][n][dv], z [BH][n]. */
void kata_oracle_prefix_state_gated(const double *k, const double *v, const double *gamma,
                                    double *S, double *z, int BH, int T, int d, int dv) {
    const int n = kata_oracle_feature_dim(d);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * n * dv;
        double *zb = z + (size_t)bh * n;
        double *pk = malloc((size_t)n * sizeof(double));
        memset(Sb, 0, sizeof(double) * n * dv);
        memset(zb, 0, sizeof(double) * n);
        for (int t = 0; t < T; ++t) {
            const int64_t row = (int64_t)bh * T + t;
            const double g = gamma[row];
            lift_one(k + row * d, d, pk);
            for (int f = 0; f < n; ++f) {
                for (int j = 0; j < dv; ++j)
                    Sb[(size_t)f * dv + j] = g * Sb[(size_t)f * dv + j] + pk[f] * v[row * dv + j];
                zb[f] = g * zb[f] + pk[f];
            }
        }
        free(pk);
    }
}

/* One gated decode step, in place: S = gamma S + psi(k) v^T, z = gamma z + psi(k),
 * then the readout (update, then read).  gamma is [BH]. */
void kata_oracle_decode_step_gated(double *S, double *z, const double *q, const double *k,
                                   const double *v, const double *gamma, double *out, int BH,
                                   int d, int dv, int normalize) {
    const int n = kata_oracle_feature_dim(d);
#pragma omp parallel for schedule(dynamic, 1) num_threads(kata_oracle_get_threads())
    for (int bh = 0; bh < BH; ++bh) {
        double *Sb = S + (size_t)bh * n * dv;
        double *zb = z + (size_t)bh * n;
        double *pk = malloc((size_t)n * sizeof(double));
        double *pq = malloc((size_t)n * sizeof(double));
        const double g = gamma[bh];
        lift_one(k + (size_t)bh * d, d, pk);
        lift_one(q + (size_t)bh * d, d, pq);
        const double *vb = v + (size_t)bh * dv;
        for (int f = 0; f < n; ++f) {
            for (int j = 0; j < dv; ++j)
                Sb[(size_t)f * dv + j] = g * Sb[(size_t)f * dv + j] + pk[f] * vb[j];
            zb[f] = g * zb[f] + pk[f];
        }
        double den = 0.0;
        for (int f = 0; f < n; ++f) den += pq[f] * zb[f];
        for (int j = 0; j < dv; ++j) {
            double num = 0.0;
            for (int f = 0; f < n; ++f) num += pq[f] * Sb[(size_t)f * dv + j];
            out[(size_t)bh * dv + j] = normalize ? (den > 0.0 ? num / den : 0.0) : num;
        }
        free(pk);
        free(pq);
    }
}
