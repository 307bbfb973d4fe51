/*
 * Parallax attention oracle: plain fp64 CPU loops (TEST INFRASTRUCTURE ONLY).
 *
 * Only the tests, the smoke check and the bench's CPU-baseline / reference arm
 * may load this library.  The product path (the CUDA library) never calls it
 * and shares no code, header or constant with it.
 *
 * What it computes (Parallax, "Parallax mantem softmax" news page, paragraph 2,
 * and its French twin "Parallax garde softmax", paragraph 2: the layer output is
 * softmax attention minus a covariance term, the key/value covariance
 * multiplied by a learned probe rho_i = W_R x_i; W_R = 0 gives plain softmax):
 *
 *   for one query row i with key set J(i):
 *     s_j   = scale * (q_i . k_j)                               j in J(i)
 *     p_j   = exp(s_j - max s) / sum_j' exp(s_j' - max s)        (softmax)
 *     mu_v  = sum_j p_j v_j ,   mu_k = sum_j p_j k_j
 *     C     = sum_j p_j (k_j - mu_k)(v_j - mu_v)^T              (d x d, keys on rows)
 *     o_i   = mu_v - C^T rho_i,  i.e. o[c] = mu_v[c] - sum_a rho[a] C[a][c]
 *
 * The pages print no formula; the reading above (rho lives in key space, the
 * scale multiplies only q.k, r = rho.k is unscaled) is the plainest one the
 * prose supports and is listed with the other readings in the design notes.
 *
 * Three algebraic forms are provided so that they can be checked against one
 * another:
 *   ORACLE_EXPLICIT    (0) the explicit d x d covariance, two centered passes;
 *   ORACLE_CONTRACTED  (1) the same centered formula with rho contracted into
 *                          the key side first: o = mu_v - sum_j p_j t_j (v_j - mu_v),
 *                          t_j = rho . (k_j - mu_k)   -- O(n d) per row;
 *   ORACLE_UNCENTERED  (2) one pass of raw moments: with w_j = exp(s_j - max s),
 *                          r_j = rho . k_j,  l = sum w, A = sum w r, U = sum w v,
 *                          W = sum w r v:  o = U/l - (W/l - (A/l)(U/l)).
 * Conventions: an empty key set gives o = 0; rho == NULL means rho = 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_EXPLICIT = 0, ORACLE_CONTRACTED = 1, ORACLE_UNCENTERED = 2 };

/* Scratch for one row: p[n] plus, for the explicit form, C[d*d] and mu_k[d]. */
typedef struct {
    double* p;
    int64_t p_cap;
    double* cov;
    double* mu_k;
    double* mu_v;
    double* t;
} row_scratch;

static int scratch_reserve(row_scratch* s, int64_t n, int64_t d) {
    if (n > s->p_cap) {
        free(s->p);
        free(s->t);
        s->p = (double*)malloc(sizeof(double) * (size_t)n);
        s->t = (double*)malloc(sizeof(double) * (size_t)n);
        if (!s->p || !s->t) return -1;
        s->p_cap = n;
    }
    if (!s->cov) {
        s->cov = (double*)malloc(sizeof(double) * (size_t)(d * d));
        s->mu_k = (double*)malloc(sizeof(double) * (size_t)d);
        s->mu_v = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s->cov || !s->mu_k || !s->mu_v) return -1;
    }
    return 0;
}

static void scratch_free(row_scratch* s) {
    free(s->p);
    free(s->t);
    free(s->cov);
    free(s->mu_k);
    free(s->mu_v);
    memset(s, 0, sizeof(*s));
}

/* Softmax weights p_j over keys 0..n-1 of K (row stride d). */
static void softmax_weights(const double* q, const double* K, int64_t n, int64_t d,
                            double scale, double* p) {
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int64_t a = 0; a < d; ++a) dot += q[a] * K[j * d + a];
        p[j] = scale * dot;
        if (p[j] > mx) mx = p[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        p[j] = exp(p[j] - mx);
        z += p[j];
    }
    for (int64_t j = 0; j < n; ++j) p[j] /= z;
}

/* One output row; returns 0 on success. */
static int parallax_row(const double* q, const double* rho, const double* K, const double* V,
                        int64_t n, int64_t d, double scale, int form, double* out,
                        row_scratch* s) {
    if (n <= 0) {
        for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
        return 0;
    }
    if (scratch_reserve(s, n, d) != 0) return -1;
    double* p = s->p;

    if (form == ORACLE_UNCENTERED) {
        /* raw moments with unnormalised weights w_j = exp(s_j - max s) */
        double mx = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int64_t a = 0; a < d; ++a) dot += q[a] * K[j * d + a];
            p[j] = scale * dot;
            if (p[j] > mx) mx = p[j];
        }
        double l = 0.0, A = 0.0;
        double* U = s->mu_v;
        double* W = s->mu_k;
        for (int64_t c = 0; c < d; ++c) U[c] = W[c] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double w = exp(p[j] - mx);
            double r = 0.0;
            if (rho)
                for (int64_t a = 0; a < d; ++a) r += rho[a] * K[j * d + a];
            l += w;
            A += w * r;
            for (int64_t c = 0; c < d; ++c) {
                U[c] += w * V[j * d + c];
                W[c] += w * r * V[j * d + c];
            }
        }
        for (int64_t c = 0; c < d; ++c) {
            double mu = U[c] / l;
            out[c] = mu - (W[c] / l - (A / l) * mu);
        }
        return 0;
    }

    softmax_weights(q, K, n, d, scale, p);
    double* mu_v = s->mu_v;
    double* mu_k = s->mu_k;
    for (int64_t c = 0; c < d; ++c) mu_v[c] = mu_k[c] = 0.0;
    for (int64_t j = 0; j < n; ++j)
        for (int64_t c = 0; c < d; ++c) {
            mu_v[c] += p[j] * V[j * d + c];
            mu_k[c] += p[j] * K[j * d + c];
        }

    if (!rho) {
        for (int64_t c = 0; c < d; ++c) out[c] = mu_v[c];
        return 0;
    }

    if (form == ORACLE_EXPLICIT) {
        double* C = s->cov; /* C[a*d + c] = sum_j p_j (k_ja - mu_k a)(v_jc - mu_v c) */
        for (int64_t x = 0; x < d * d; ++x) C[x] = 0.0;
        for (int64_t j = 0; j < n; ++j)
            for (int64_t a = 0; a < d; ++a) {
                double ka = p[j] * (K[j * d + a] - mu_k[a]);
                for (int64_t c = 0; c < d; ++c) C[a * d + c] += ka * (V[j * d + c] - mu_v[c]);
            }
        for (int64_t c = 0; c < d; ++c) {
            double corr = 0.0;
            for (int64_t a = 0; a < d; ++a) corr += rho[a] * C[a * d + c];
            out[c] = mu_v[c] - corr;
        }
        return 0;
    }

    if (form == ORACLE_CONTRACTED) {
        double* t = s->t; /* t_j = rho . (k_j - mu_k) */
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int64_t a = 0; a < d; ++a) acc += rho[a] * (K[j * d + a] - mu_k[a]);
            t[j] = acc;
        }
        for (int64_t c = 0; c < d; ++c) {
            double corr = 0.0;
            for (int64_t j = 0; j < n; ++j) corr += p[j] * t[j] * (V[j * d + c] - mu_v[c]);
            out[c] = mu_v[c] - corr;
        }
        return 0;
    }
    return -2;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * nq query rows that share one key/value set K, V ([nk x d] row-major);
 * row i attends to keys 0..nkeys[i]-1 (nkeys[i] must lie in [0, nk]).
 * q, rho, o are [nq x d].  rho may be NULL.
 */
int oracle_rows(const double* q, const double* rho, const double* k, const double* v,
                const int64_t* nkeys, int64_t nq, int64_t nk, int64_t d, double scale,
                int form, double* o) {
    if (!q || !k || !v || !nkeys || !o || nq < 0 || nk < 0 || d <= 0) return -1;
    for (int64_t i = 0; i < nq; ++i)
        if (nkeys[i] < 0 || nkeys[i] > nk) return -1;
    int err = 0;
#pragma omp parallel
    {
        row_scratch s;
        memset(&s, 0, sizeof(s));
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < nq; ++i) {
            int e = parallax_row(q + i * d, rho ? rho + i * d : NULL, k, v, nkeys[i], d, scale,
                                 form, o + i * d, &s);
            if (e) {
#pragma omp atomic write
                err = e;
            }
        }
        scratch_free(&s);
    }
    return err;
}

/*
 * Prefill: q, rho, k, v, o are [B, H, L, d] row-major; rho may be NULL.
 * causal = 1: query i sees keys 0..i; causal = 0: keys 0..L-1.
 */
int oracle_prefill(const double* q, const double* rho, const double* k, const double* v,
                   int64_t B, int64_t H, int64_t L, int64_t d, int causal, double scale,
                   int form, double* o) {
    if (!q || !k || !v || !o || B < 0 || H < 0 || L < 0 || d <= 0) return -1;
    if (causal != 0 && causal != 1) return -1;
    const int64_t nrows = B * H * L;
    int err = 0;
#pragma omp parallel
    {
        row_scratch s;
        memset(&s, 0, sizeof(s));
#pragma omp for schedule(dynamic, 16)
        for (int64_t row = 0; row < nrows; ++row) {
            const int64_t bh = row / L, i = row % L;
            const int64_t head = bh * L * d;
            const int64_t n = causal ? i + 1 : L;
            int e = parallax_row(q + row * d, rho ? rho + row * d : NULL, k + head, v + head, n,
                                 d, scale, form, o + row * d, &s);
            if (e) {
#pragma omp atomic write
                err = e;
            }
        }
        scratch_free(&s);
    }
    return err;
}

/*
 * Decode: q, rho, o are [B, H, d]; k_cache, v_cache are [B, H, Lmax, d];
 * sequence b uses cache rows 0..seqlens[b]-1 (seqlens[b] must lie in [0, Lmax]).
 */
int oracle_decode(const double* q, const double* rho, const double* k_cache,
                  const double* v_cache, const int32_t* seqlens, int64_t B, int64_t H,
                  int64_t Lmax, int64_t d, double scale, int form, double* o) {
    if (!q || !k_cache || !v_cache || !seqlens || !o || B < 0 || H < 0 || Lmax < 0 || d <= 0)
        return -1;
    for (int64_t b = 0; b < B; ++b)
        if (seqlens[b] < 0 || seqlens[b] > Lmax) return -1;
    const int64_t nheads = B * H;
    int err = 0;
#pragma omp parallel
    {
        row_scratch s;
        memset(&s, 0, sizeof(s));
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < nheads; ++bh) {
            const int64_t b = bh / H;
            const int64_t head = bh * Lmax * d;
            int e = parallax_row(q + bh * d, rho ? rho + bh * d : NULL, k_cache + head,
                                 v_cache + head, seqlens[b], d, scale, form, o + bh * d, &s);
            if (e) {
#pragma omp atomic write
                err = e;
            }
        }
        scratch_free(&s);
    }
    return err;
}
