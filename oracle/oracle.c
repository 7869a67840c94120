/*
 * Dynamic Bifocal RoPE attention -- fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * statement of what the GPU library computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares
 * no code, header, table or constant with the CUDA library.
 *
 * Source: "Jet-Long: Efficient Long-Context Extension with Dynamic Bifocal
 * RoPE" (arXiv 2607.07740), as described on the engineersofai.com abstract
 * page (Abstract), the researchpod.app summary (Summary paragraph 2 and the
 * transcript on caching and prefill) and the seventnews.com / transform-ai
 * articles ("How bifocal attention sidesteps the fixed-scaling trap",
 * "How Jet-Long works").  The pages print no formulas; every concrete
 * choice below is a reading of their prose and is listed as such.
 *
 * Notation (all positions are 0-based token indices):
 *   D          head dimension (even), tau = 1/sqrt(D)
 *   theta_d    = theta^(-2d/D), d in [0, D/2)
 *   R_p(x)     rotates every pair (x_d, x_{d+D/2}) by the angle p*theta_d
 *              (half-split pair layout -- a reading; the pages name none)
 *   g(s, L)    smallest integer g >= 1 such that floor((s-1)/g) <= L-1,
 *              i.e. every grouped position of a length-s sequence lies in
 *              the pretrained window [0, L)  (researchpod Summary: "smallest
 *              integer grouping that keeps remote rotation angles within the
 *              pretrained distribution"; abstract: factor adapts to the
 *              current length s)
 *   delta_p    = floor(p/g) - p   (position aliasing, researchpod transcript:
 *              a distant position is mapped onto the known grid)
 *
 * Query i (exact-RoPE vector q_i = R_i(q~_i)) attends to keys j <= i:
 *   local (exact) score   for 0 <= i-j < w :  tau * <q_i, k_j>
 *   remote (grouped) score for i-j >= w    :  tau * <R_{delta_i} q_i, R_{delta_j} k_j>
 * The remote vectors come from correcting the exact-RoPE inputs (abstract:
 * "on-the-fly RoPE correction rotation"; researchpod transcript: the cache
 * keeps original positions and the remapping is applied at lookup time).
 * Softmax over the union of both key sets gives out_i and
 * lse_i = ln sum_j exp(score_ij).
 *
 * oracle_bifocal_rows_3pass() computes the same thing the way the abstract
 * and the researchpod summary describe it: three attention passes --
 * local(window, exact), remote(all, grouped), remote(window, grouped) --
 * merged by inclusion-exclusion on their log-sum-exp statistics.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Group factor (researchpod Summary: smallest integer grouping).      */
/* Written as the literal search over g = 1, 2, ... so that the closed */
/* form ceil(s/L) used elsewhere is checked against it, not assumed.   */
/* ------------------------------------------------------------------ */
int64_t oracle_group_factor(int64_t s, int64_t L)
{
    if (s < 1 || L < 1) return -1;
    int64_t g = 1;
    while ((s - 1) / g > L - 1) g++;
    return g;
}

static int64_t floor_div(int64_t a, int64_t b)
{
    int64_t q = a / b;
    if ((a % b != 0) && ((a < 0) != (b < 0))) q--;
    return q;
}

/* Aliased position floor(p/g) (researchpod transcript, position aliasing). */
int64_t oracle_grouped_position(int64_t p, int64_t g)
{
    return floor_div(p, g);
}

/* theta_d = theta^(-2d/D) */
static double freq(int64_t d, int64_t D, double theta)
{
    return pow(theta, -2.0 * (double)d / (double)D);
}

/* y = R_p(x) for one head vector of length D (half-split pairs). */
static void rotate(const double *x, double *y, int64_t D, int64_t p, double theta)
{
    int64_t h = D / 2;
    for (int64_t d = 0; d < h; d++) {
        double a = (double)p * freq(d, D, theta);
        double c = cos(a), s = sin(a);
        double x0 = x[d], x1 = x[d + h];
        y[d] = x0 * c - x1 * s;
        y[d + h] = x1 * c + x0 * s;
    }
}

static double dot(const double *a, const double *b, int64_t D)
{
    double acc = 0.0;
    for (int64_t d = 0; d < D; d++) acc += a[d] * b[d];
    return acc;
}

/* ------------------------------------------------------------------ */
/* Exact RoPE (local, "original, unscaled" frequencies):               */
/* out[b,s,h,:] = R_{pos0+s}(x[b,s,h,:]), x laid out [B,S,H,D].        */
/* ------------------------------------------------------------------ */
void oracle_rope(const double *x, double *out, int64_t B, int64_t S, int64_t H,
                 int64_t D, int64_t pos0, double theta)
{
    int64_t rows = B * S * H;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        int64_t s = (r / H) % S;
        rotate(x + r * D, out + r * D, D, pos0 + s, theta);
    }
}

/* ------------------------------------------------------------------ */
/* Shared argument layout of the attention entry points:               */
/*   q    [B, Sq, Hq, D]   exact-RoPE queries at positions qpos[0..Sq) */
/*   k, v [B, Sk, Hkv, D]  exact-RoPE keys / values at positions 0..Sk) */
/*   s_len   the current length s that fixes g                         */
/*   L       pretrained window, w local window                         */
/*   out  [B, Sq, Hq, D],  lse [B, Hq, Sq]                             */
/* GQA: query head h reads kv head h / (Hq/Hkv).                       */
/* Query at position i attends to keys j <= min(i, Sk-1).              */
/* Returns 0, or -1 on bad arguments.                                  */
/* ------------------------------------------------------------------ */

static int check_args(int64_t B, int64_t Sq, int64_t Hq, int64_t Hkv, int64_t Sk,
                      int64_t D, int64_t s_len, int64_t L, int64_t w, double theta)
{
    if (B < 1 || Sq < 0 || Hq < 1 || Hkv < 1 || Sk < 1 || D < 2 || (D % 2) != 0)
        return -1;
    if (Hq % Hkv != 0 || s_len < 1 || L < 1 || w < 1 || !(theta > 0.0)) return -1;
    return 0;
}

/* Grouped (remote-view) keys: kg_j = R_{delta_j}(k_j) for every key of one
 * (b, kv-head); this is step "correct the key" done once per key. */
static double *grouped_keys(const double *k, int64_t b, int64_t hk, int64_t Sk,
                            int64_t Hkv, int64_t D, int64_t g, double theta)
{
    double *kg = (double *)malloc((size_t)(Sk * D) * sizeof(double));
    if (!kg) return NULL;
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < Sk; j++) {
        const double *kj = k + ((b * Sk + j) * Hkv + hk) * D;
        rotate(kj, kg + j * D, D, floor_div(j, g) - j, theta);
    }
    return kg;
}

/* Single masked pass: every key is scored once, with the view its distance
 * selects, and one softmax is taken over the union. */
int oracle_bifocal_rows(const double *q, const double *k, const double *v,
                        int64_t B, int64_t Sq, int64_t Hq, int64_t Hkv, int64_t Sk,
                        int64_t D, const int64_t *qpos, int64_t s_len, int64_t L,
                        int64_t w, double theta, double *out, double *lse)
{
    if (check_args(B, Sq, Hq, Hkv, Sk, D, s_len, L, w, theta)) return -1;
    const int64_t grp = Hq / Hkv;
    const int64_t g = oracle_group_factor(s_len, L);
    const double tau = 1.0 / sqrt((double)D);

    for (int64_t b = 0; b < B; b++) {
        for (int64_t hk = 0; hk < Hkv; hk++) {
            double *kg = grouped_keys(k, b, hk, Sk, Hkv, D, g, theta);
            if (!kg) return -1;
            int64_t nrow = Sq * grp;
#pragma omp parallel
            {
                double *sc = (double *)malloc((size_t)Sk * sizeof(double));
                double *qg = (double *)malloc((size_t)D * sizeof(double));
#pragma omp for schedule(dynamic, 1)
                for (int64_t t = 0; t < nrow; t++) {
                    int64_t r = t / grp, h = hk * grp + t % grp;
                    int64_t i = qpos[r];
                    const double *qi = q + ((b * Sq + r) * Hq + h) * D;
                    rotate(qi, qg, D, floor_div(i, g) - i, theta);
                    int64_t jmax = i < Sk - 1 ? i : Sk - 1;
                    double m = -INFINITY;
                    for (int64_t j = 0; j <= jmax; j++) {
                        const double *kj = k + ((b * Sk + j) * Hkv + hk) * D;
                        double s = (i - j < w) ? tau * dot(qi, kj, D)
                                               : tau * dot(qg, kg + j * D, D);
                        sc[j] = s;
                        if (s > m) m = s;
                    }
                    double *o = out + ((b * Sq + r) * Hq + h) * D;
                    for (int64_t d = 0; d < D; d++) o[d] = 0.0;
                    double Z = 0.0;
                    for (int64_t j = 0; j <= jmax; j++) {
                        double p = exp(sc[j] - m);
                        Z += p;
                        const double *vj = v + ((b * Sk + j) * Hkv + hk) * D;
                        for (int64_t d = 0; d < D; d++) o[d] += p * vj[d];
                    }
                    for (int64_t d = 0; d < D; d++) o[d] /= Z;
                    lse[(b * Hq + h) * Sq + r] = (jmax >= 0) ? m + log(Z) : -INFINITY;
                }
                free(sc);
                free(qg);
            }
            free(kg);
        }
    }
    return 0;
}

/* One softmax pass over the keys j in [jlo, jhi] of one query row, with
 * either the exact vectors (qv, k) or the grouped ones (qv, kg).
 * Writes o[D] and returns the pass's log-sum-exp (-inf if the set is empty). */
static double softmax_pass(const double *qv, const double *keys, int64_t key_stride,
                           const double *v, int64_t v_stride, int64_t jlo, int64_t jhi,
                           int64_t D, double tau, double *sc, double *o)
{
    for (int64_t d = 0; d < D; d++) o[d] = 0.0;
    if (jhi < jlo) return -INFINITY;
    double m = -INFINITY;
    for (int64_t j = jlo; j <= jhi; j++) {
        double s = tau * dot(qv, keys + j * key_stride, D);
        sc[j - jlo] = s;
        if (s > m) m = s;
    }
    double Z = 0.0;
    for (int64_t j = jlo; j <= jhi; j++) {
        double p = exp(sc[j - jlo] - m);
        Z += p;
        for (int64_t d = 0; d < D; d++) o[d] += p * v[j * v_stride + d];
    }
    for (int64_t d = 0; d < D; d++) o[d] /= Z;
    return m + log(Z);
}

/* Three passes merged by inclusion-exclusion:
 *   local(window) + remote(all) - remote(window)
 * with each pass reduced to (O, lse) and merged on lse statistics. */
int oracle_bifocal_rows_3pass(const double *q, const double *k, const double *v,
                              int64_t B, int64_t Sq, int64_t Hq, int64_t Hkv, int64_t Sk,
                              int64_t D, const int64_t *qpos, int64_t s_len, int64_t L,
                              int64_t w, double theta, double *out, double *lse)
{
    if (check_args(B, Sq, Hq, Hkv, Sk, D, s_len, L, w, theta)) return -1;
    const int64_t grp = Hq / Hkv;
    const int64_t g = oracle_group_factor(s_len, L);
    const double tau = 1.0 / sqrt((double)D);
    const int64_t kstride = Hkv * D;

    for (int64_t b = 0; b < B; b++) {
        for (int64_t hk = 0; hk < Hkv; hk++) {
            double *kg = grouped_keys(k, b, hk, Sk, Hkv, D, g, theta);
            if (!kg) return -1;
            const double *kb = k + (b * Sk * Hkv + hk) * D;
            const double *vb = v + (b * Sk * Hkv + hk) * D;
            int64_t nrow = Sq * grp;
#pragma omp parallel
            {
                double *sc = (double *)malloc((size_t)Sk * sizeof(double));
                double *qg = (double *)malloc((size_t)D * sizeof(double));
                double *oL = (double *)malloc((size_t)(3 * D) * sizeof(double));
                double *oA = oL + D, *oW = oL + 2 * D;
#pragma omp for schedule(dynamic, 1)
                for (int64_t t = 0; t < nrow; t++) {
                    int64_t r = t / grp, h = hk * grp + t % grp;
                    int64_t i = qpos[r];
                    const double *qi = q + ((b * Sq + r) * Hq + h) * D;
                    rotate(qi, qg, D, floor_div(i, g) - i, theta);
                    int64_t jmax = i < Sk - 1 ? i : Sk - 1;
                    int64_t jwin = i - w + 1; /* first key of the local window */
                    if (jwin < 0) jwin = 0;
                    /* local view: exact scores over the window */
                    double lL = softmax_pass(qi, kb, kstride, vb, kstride, jwin, jmax, D,
                                             tau, sc, oL);
                    /* remote view over all causal keys, grouped scores */
                    double lA = softmax_pass(qg, kg, D, vb, kstride, 0, jmax, D, tau, sc, oA);
                    /* remote view restricted to the window (the overlap) */
                    double lW = softmax_pass(qg, kg, D, vb, kstride, jwin, jmax, D, tau, sc,
                                             oW);
                    double M = lL > lA ? lL : lA;
                    double eL = exp(lL - M), eA = exp(lA - M), eW = exp(lW - M);
                    double Z = eL + eA - eW;
                    double *o = out + ((b * Sq + r) * Hq + h) * D;
                    for (int64_t d = 0; d < D; d++)
                        o[d] = (eL * oL[d] + eA * oA[d] - eW * oW[d]) / Z;
                    lse[(b * Hq + h) * Sq + r] = M + log(Z);
                }
                free(sc);
                free(qg);
                free(oL);
            }
            free(kg);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Variants (the method's optional forms, one flag each):              */
/*                                                                     */
/*  ORACLE_PER_QUERY_G  query i uses its own current length s = i + 1, */
/*      so g = g(i + 1) changes inside one prefill (abstract: the      */
/*      factor adapts to the current length s; a causal model at       */
/*      token i has seen i + 1 tokens).                                */
/*  ORACLE_SLIDING      a sliding-window layer of a hybrid model: keys */
/*      with i - j >= w are not attended at all and no key is aliased  */
/*      (seventnews.com, "Generalization to hybrid attention           */
/*      architectures": local-window layers keep their own window).    */
/*  ORACLE_QUERY_SHIFT  Self-Extend-style shift: the aliased query     */
/*      position is floor(i/g) + (w - floor(w/g)), which makes the     */
/*      aliased distance continuous with the exact one at i - j = w;   */
/*      g is then the smallest integer with                            */
/*      floor((s-1)/g) + w - floor(w/g) <= L - 1 (ResearchPod summary  */
/*      names Self-Extend as a baseline; the shift is its grouping).   */
/* ------------------------------------------------------------------ */
#define ORACLE_PER_QUERY_G 1
#define ORACLE_SLIDING 2
#define ORACLE_QUERY_SHIFT 4

/* Smallest g >= 1 whose largest aliased distance, with the query shifted by
 * w - floor(w/g), stays inside the pretrained window: literal search.
 * -1 when no g does (w >= L). */
int64_t oracle_group_factor_shift(int64_t s, int64_t L, int64_t w)
{
    if (s < 1 || L < 1 || w < 1) return -1;
    int64_t gmax = (s > w ? s : w) + 1;
    for (int64_t g = 1; g <= gmax; g++)
        if ((s - 1) / g + (w - w / g) <= L - 1) return g;
    return -1;
}

/* g of a row of current length s under the flags (-1: no valid g). */
int64_t oracle_row_group(int64_t s, int64_t L, int64_t w, int64_t flags)
{
    return (flags & ORACLE_QUERY_SHIFT) ? oracle_group_factor_shift(s, L, w)
                                        : oracle_group_factor(s, L);
}

/* Single masked pass with variant flags; same layout and result convention as
 * oracle_bifocal_rows (which this equals when flags == 0).  The grouped keys
 * are built once per distinct g that some row uses. */
int oracle_bifocal_rows_ex(const double *q, const double *k, const double *v,
                           int64_t B, int64_t Sq, int64_t Hq, int64_t Hkv, int64_t Sk,
                           int64_t D, const int64_t *qpos, int64_t s_len, int64_t L,
                           int64_t w, double theta, int64_t flags, double *out, double *lse)
{
    if (check_args(B, Sq, Hq, Hkv, Sk, D, s_len, L, w, theta)) return -1;
    if (flags & ~(int64_t)(ORACLE_PER_QUERY_G | ORACLE_SLIDING | ORACLE_QUERY_SHIFT)) return -1;
    const int64_t grp = Hq / Hkv;
    const double tau = 1.0 / sqrt((double)D);
    /* g of every row */
    int64_t *grow = (int64_t *)malloc((size_t)(Sq > 0 ? Sq : 1) * sizeof(int64_t));
    if (!grow) return -1;
    for (int64_t r = 0; r < Sq; r++) {
        int64_t s_row = (flags & ORACLE_PER_QUERY_G) ? qpos[r] + 1 : s_len;
        grow[r] = oracle_row_group(s_row, L, w, flags);
        if (grow[r] < 1) {
            free(grow);
            return -1;
        }
    }
    for (int64_t b = 0; b < B; b++) {
        for (int64_t hk = 0; hk < Hkv; hk++) {
            /* rows are handled in groups of equal g */
            int64_t done_g = 0;
            for (;;) {
                int64_t g = -1;
                for (int64_t r = 0; r < Sq; r++)
                    if (grow[r] > done_g && (g < 0 || grow[r] < g)) g = grow[r];
                if (g < 0) break;
                done_g = g;
                double *kg = grouped_keys(k, b, hk, Sk, Hkv, D, g, theta);
                if (!kg) {
                    free(grow);
                    return -1;
                }
                const int64_t shift = (flags & ORACLE_QUERY_SHIFT) ? w - w / g : 0;
                int64_t nrow = Sq * grp;
#pragma omp parallel
                {
                    double *sc = (double *)malloc((size_t)Sk * sizeof(double));
                    double *qg = (double *)malloc((size_t)D * sizeof(double));
                    unsigned char *use = (unsigned char *)malloc((size_t)Sk);
#pragma omp for schedule(dynamic, 1)
                    for (int64_t t = 0; t < nrow; t++) {
                        int64_t r = t / grp, h = hk * grp + t % grp;
                        if (grow[r] != g) continue;
                        int64_t i = qpos[r];
                        const double *qi = q + ((b * Sq + r) * Hq + h) * D;
                        rotate(qi, qg, D, floor_div(i, g) + shift - i, theta);
                        int64_t jmax = i < Sk - 1 ? i : Sk - 1;
                        double m = -INFINITY;
                        for (int64_t j = 0; j <= jmax; j++) {
                            const double *kj = k + ((b * Sk + j) * Hkv + hk) * D;
                            use[j] = 1;
                            if (i - j < w) {
                                sc[j] = tau * dot(qi, kj, D);
                            } else if (flags & ORACLE_SLIDING) {
                                use[j] = 0; /* outside a sliding window: not attended */
                                continue;
                            } else {
                                sc[j] = tau * dot(qg, kg + j * D, D);
                            }
                            if (sc[j] > m) m = sc[j];
                        }
                        double *o = out + ((b * Sq + r) * Hq + h) * D;
                        for (int64_t d = 0; d < D; d++) o[d] = 0.0;
                        double Z = 0.0;
                        for (int64_t j = 0; j <= jmax; j++) {
                            if (!use[j]) continue;
                            double p = exp(sc[j] - m);
                            Z += p;
                            const double *vj = v + ((b * Sk + j) * Hkv + hk) * D;
                            for (int64_t d = 0; d < D; d++) o[d] += p * vj[d];
                        }
                        for (int64_t d = 0; d < D; d++) o[d] /= Z;
                        lse[(b * Hq + h) * Sq + r] = (jmax >= 0) ? m + log(Z) : -INFINITY;
                    }
                    free(sc);
                    free(qg);
                    free(use);
                }
                free(kg);
            }
        }
    }
    free(grow);
    return 0;
}

/* Number of OpenMP threads the oracle runs on (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
