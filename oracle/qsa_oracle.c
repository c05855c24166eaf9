/*
 * QSA oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU statement of what one Qwen Sparse
 * Attention (QSA) layer computes.  Only the test-suite, the package smoke
 * check and the benchmark's CPU-baseline leg may load this library; the CUDA
 * product path never does.  It shares no code, header, table or constant
 * generator with the CUDA library: every constant below is restated here from
 * the sources.
 *
 * Sources (web pages about the Qwen3.8-Flash-Next release):
 *   [LP]  launch post, section "Model Architecture / Attention: GDN + QSA for
 *         Efficient Memory and Precise Retrieval": a lightweight indexer groups
 *         the sequence into micro-blocks, scores importance per block and the
 *         attention then runs only over the selected regions; compression is
 *         done independently in every layer.
 *   [MC]  model card (Qwen3.8-Flash-Next-GGUF), section "Model Overview /
 *         Qwen Sparse Attention": 24 query heads, 2 KV heads, head dim 256,
 *         rotary dim 64, indexer = MQA with 4 query heads and 1 shared key
 *         head of dim 128, budget 512 blocks or 2048 tokens.
 *   [MCR] model card, section "Processing Ultra-Long Texts" (rope_parameters):
 *         rope_theta = 10000000, partial_rotary_factor = 0.25; beyond 262,144
 *         positions the card enables YaRN with factor 4 over an original
 *         context of 262,144.
 *   [YaRN] the published YaRN method (Peng et al., 2023, "YaRN: Efficient
 *         Context Window Extension of Large Language Models", sections 3.2 to
 *         3.4), which [MCR] names but does not restate: per rotary frequency
 *         w_d with wavelength lambda_d = 2 pi / w_d and r_d = L_orig /
 *         lambda_d, a ramp gamma(r) = 0 below alpha, 1 above beta, linear in
 *         between (alpha = 1, beta = 32), and w'_d = (1 - gamma) w_d / s +
 *         gamma w_d; the attention logits get the temperature 1/t with
 *         sqrt(1/t) = 0.1 ln s + 1.
 *
 * Readings taken where the pages leave a step open (all are listed in the
 * design notes of the repository):
 *   R1  a micro-block is 4 tokens (512 blocks <-> 2048 tokens, [MC]);
 *   R2  the block key is the mean of the block's 4 indexer keys, evaluated as
 *       ((k0 + k1) + k2) + k3 in fp64, times 1/4, rounded to bf16
 *       (round-to-nearest-even) -- bf16 is what the tensor cores consume;
 *   R3  block score s[t,b] = sum_h w[t,h] * max(0, qi[t,h] . kblk[b]),
 *       no scale factor;
 *   R4  the query at position t sits in block c = floor(t/4), which is always
 *       selected (and causally masked inside); among the past blocks b < c
 *       the (budget-1) best by (score descending, block index ascending) are
 *       selected; if there are fewer past blocks, all of them are;
 *   R5  RoPE on the first 64 of 256 dims, rotate-half pairing (i, i+32),
 *       w_i = theta^(-2i/64) (or its YaRN rescaling, [YaRN] with factor s),
 *       angle = pos * w_i; the rotated values are rounded to bf16 (the point
 *       where the GPU rounds before its tensor cores); the indexer tensors get
 *       no RoPE;
 *   R6  attention over keys j with floor(j/4) selected and j <= t; query head
 *       h reads KV head floor(h/12); softmax scale 1/sqrt(256) unless given;
 *       everything after the bf16 inputs is kept in fp64;
 *   R7  with YaRN on, the temperature multiplies the whole attention logit
 *       (all 256 dims), as [YaRN] defines it: a temperature on the softmax of
 *       q.k.  Implementations written for fully rotary models fold
 *       sqrt(1/t) into the cos/sin tables, which here, with only 64 of 256
 *       dims rotary, would scale the rotary part of the logit alone; the
 *       method's definition is followed rather than that folding.
 *
 * Parity unpinned: qo_yarn_logit_factor.  Its constant (0.1 ln s + 1,
 * squared) is [YaRN]'s recommended fit; the pages print no value of it, and
 * no property of the method fixes it, so the tests pin only how it is used
 * (the temperature scales the logits and nothing else), not its value.
 * Every other function here is pinned by the tests against closed forms,
 * invariants, library routines or brute force.
 *
 * All tensors are row-major, bf16 passed as raw uint16 bit patterns.
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QO_BS 4      /* tokens per micro-block (R1)            */
#define QO_HQ 24     /* query heads [MC]                       */
#define QO_HKV 2     /* KV heads [MC]                          */
#define QO_D 256     /* head dim [MC]                          */
#define QO_RD 64     /* rotary dims [MC], 0.25 * 256 [MCR]     */
#define QO_HI 4      /* indexer query heads [MC]               */
#define QO_DI 128    /* indexer head dim [MC]                  */

/* ---------------------------------------------------------------- bf16 -- */

double qo_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), directly from the
 * double: bf16 keeps 8 significant bits, so scale the value to an integer
 * with 8 bits, round that with rint() (the default rounding mode is
 * round-to-nearest-even), and scale back.  Exact in double. */
uint16_t qo_f64_to_bf16(double x)
{
    if (isnan(x)) return 0x7FC0;
    double ax = fabs(x);
    double r;
    if (ax < ldexp(1.0, -126)) {
        /* subnormal bf16 range: fixed quantum 2^-133 */
        r = rint(x * ldexp(1.0, 133)) * ldexp(1.0, -133);
    } else {
        int e;
        double m = frexp(x, &e);           /* x = m * 2^e, 0.5 <= |m| < 1 */
        r = ldexp(rint(ldexp(m, 8)), e - 8);
    }
    /* largest finite bf16 is (2 - 2^-7) * 2^127 */
    if (fabs(r) > ldexp(255.0, 120)) r = copysign(INFINITY, x);
    float f = (float)r;                    /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* -------------------------------------------------------- micro-blocks -- */

/* R2: kblk[b, :] for the floor(L/4) complete blocks. */
void qo_block_keys(int64_t L, const uint16_t *ki, uint16_t *kblk)
{
    int64_t nb = L / QO_BS;
    for (int64_t b = 0; b < nb; ++b)
        for (int d = 0; d < QO_DI; ++d) {
            double sum = 0.0;
            for (int i = 0; i < QO_BS; ++i)
                sum = sum + qo_bf16_to_f64(ki[(b * QO_BS + i) * QO_DI + d]);
            kblk[b * QO_DI + d] = qo_f64_to_bf16(sum * 0.25);
        }
}

/* ---------------------------------------------------------------- RoPE -- */

/* R5: the 32 rotary frequencies w_i = theta^(-2i/64); with a YaRN factor
 * s > 1, each is rescaled as [YaRN] states: r = L_orig / (2 pi / w_i),
 * gamma(r) = clamp((r - alpha) / (beta - alpha), 0, 1),
 * w'_i = (1 - gamma) w_i / s + gamma w_i. */
void qo_rope_inv_freq(double theta, double s, double l_orig, double alpha, double beta, double *out)
{
    const int half = QO_RD / 2;
    for (int i = 0; i < half; ++i) {
        double w = pow(theta, -2.0 * (double)i / (double)QO_RD);
        if (s > 1.0) {
            double lambda = 2.0 * M_PI / w;
            double r = l_orig / lambda;
            double gamma = r < alpha ? 0.0 : (r > beta ? 1.0 : (r - alpha) / (beta - alpha));
            w = (1.0 - gamma) * w / s + gamma * w;
        }
        out[i] = w;
    }
}

/* [YaRN]: the factor the attention logits are multiplied by, (0.1 ln s + 1)^2
 * (both query and key carry sqrt(1/t)); 1 without YaRN.  Parity unpinned:
 * the constant is the method's fitted value, printed on none of the pages. */
double qo_yarn_logit_factor(double s)
{
    if (s <= 1.0) return 1.0;
    double m = 0.1 * log(s) + 1.0;
    return m * m;
}

/* R5, exact part: the 64 rotated values of one head row, in fp64. */
void qo_rope_exact(const uint16_t *x, const double *inv_freq, int64_t pos, double *out)
{
    const int half = QO_RD / 2;
    for (int i = 0; i < half; ++i) {
        double ang = (double)pos * inv_freq[i];
        double c = cos(ang), s = sin(ang);
        double x1 = qo_bf16_to_f64(x[i]);
        double x2 = qo_bf16_to_f64(x[i + half]);
        out[i] = x1 * c - x2 * s;
        out[i + half] = x2 * c + x1 * s;
    }
}

/* R5: one full head row (256 dims) after RoPE, as the bf16 the tensor cores
 * see: dims [0,64) rotated and rounded, dims [64,256) passed through. */
void qo_rope_row_bf16(const uint16_t *x, const double *inv_freq, int64_t pos, uint16_t *out)
{
    double rot[QO_RD];
    qo_rope_exact(x, inv_freq, pos, rot);
    for (int i = 0; i < QO_RD; ++i) out[i] = qo_f64_to_bf16(rot[i]);
    for (int i = QO_RD; i < QO_D; ++i) out[i] = x[i];
}

/* K' for a whole [rows, 2, 256] key tensor at positions 0..rows-1. */
void qo_rope_keys(int64_t rows, const double *inv_freq, const uint16_t *k, uint16_t *k_rot)
{
    for (int64_t j = 0; j < rows; ++j)
        for (int g = 0; g < QO_HKV; ++g)
            qo_rope_row_bf16(k + (j * QO_HKV + g) * QO_D, inv_freq, j,
                             k_rot + (j * QO_HKV + g) * QO_D);
}

/* -------------------------------------------------------------- scores -- */

/* R3: scores of one query (qi_t [4,128], w_t [4]) against blocks 0..nb-1. */
void qo_block_scores(const uint16_t *qi_t, const uint16_t *w_t,
                     const uint16_t *kblk, int64_t nb, double *s)
{
    for (int64_t b = 0; b < nb; ++b) {
        double total = 0.0;
        for (int h = 0; h < QO_HI; ++h) {
            double dot = 0.0;
            for (int d = 0; d < QO_DI; ++d)
                dot += qo_bf16_to_f64(qi_t[h * QO_DI + d]) *
                       qo_bf16_to_f64(kblk[b * QO_DI + d]);
            double relu = dot > 0.0 ? dot : 0.0;
            total += qo_bf16_to_f64(w_t[h]) * relu;
        }
        s[b] = total;
    }
}

/* ----------------------------------------------------------- selection -- */

typedef struct { double s; int64_t b; } qo_pair;

/* order: score descending, then block index ascending (R4) */
static int qo_cmp_rank(const void *pa, const void *pb)
{
    const qo_pair *a = (const qo_pair *)pa, *b = (const qo_pair *)pb;
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
    return (a->b < b->b) ? -1 : (a->b > b->b);
}

static int qo_cmp_i64(const void *pa, const void *pb)
{
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    return (a > b) - (a < b);
}

/* R4: s[0..c-1] are the past-block scores of a query in block c.
 * Writes the selected blocks ascending into sel[0..budget-1] (-1 padded)
 * and their scores into sel_s (current block +inf, padding -inf) if given.
 * Returns the number selected. */
int qo_select(const double *s, int64_t c, int budget, int32_t *sel, double *sel_s)
{
    int64_t want = budget - 1;
    int64_t npast = c < want ? c : want;
    qo_pair *p = (qo_pair *)malloc(sizeof(qo_pair) * (size_t)(c > 0 ? c : 1));
    int64_t *chosen = (int64_t *)malloc(sizeof(int64_t) * (size_t)(npast + 1));
    for (int64_t b = 0; b < c; ++b) { p[b].s = s[b]; p[b].b = b; }
    qsort(p, (size_t)c, sizeof(qo_pair), qo_cmp_rank);
    for (int64_t i = 0; i < npast; ++i) chosen[i] = p[i].b;
    qsort(chosen, (size_t)npast, sizeof(int64_t), qo_cmp_i64);
    for (int64_t i = 0; i < npast; ++i) {
        sel[i] = (int32_t)chosen[i];
        if (sel_s) sel_s[i] = s[chosen[i]];
    }
    sel[npast] = (int32_t)c;
    if (sel_s) sel_s[npast] = INFINITY;
    for (int64_t i = npast + 1; i < budget; ++i) {
        sel[i] = -1;
        if (sel_s) sel_s[i] = -INFINITY;
    }
    free(p);
    free(chosen);
    return (int)(npast + 1);
}

/* ----------------------------------------------------------- attention -- */

/* R6 for one query row.
 *   q_t   [24,256] pre-RoPE query at position pos
 *   k, v  [rows,2,256] pre-RoPE keys / values of the sequence (row j = position j)
 *   sel   selected blocks (entries < 0 ignored), nsel entries
 *   o     [24,256] output, lse [24] natural-log log-sum-exp of the scaled logits */
void qo_attend(const uint16_t *q_t, int64_t pos, const uint16_t *k, const uint16_t *v,
               const int32_t *sel, int nsel, const double *inv_freq, double scale,
               double *o, double *lse)
{
    /* gather the attended key positions */
    int64_t nkeys = 0;
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nsel * QO_BS + 1));
    for (int i = 0; i < nsel; ++i) {
        if (sel[i] < 0) continue;
        for (int r = 0; r < QO_BS; ++r) {
            int64_t j = (int64_t)sel[i] * QO_BS + r;
            if (j <= pos) keys[nkeys++] = j;
        }
    }
    uint16_t qrot[QO_HQ][QO_D];
    for (int h = 0; h < QO_HQ; ++h) qo_rope_row_bf16(q_t + h * QO_D, inv_freq, pos, qrot[h]);

    double *z = (double *)malloc(sizeof(double) * (size_t)(QO_HQ * (nkeys > 0 ? nkeys : 1)));
    uint16_t krot[QO_D];
    for (int64_t jj = 0; jj < nkeys; ++jj) {
        int64_t j = keys[jj];
        for (int g = 0; g < QO_HKV; ++g) {
            qo_rope_row_bf16(k + (j * QO_HKV + g) * QO_D, inv_freq, j, krot);
            for (int h = g * (QO_HQ / QO_HKV); h < (g + 1) * (QO_HQ / QO_HKV); ++h) {
                double dot = 0.0;
                for (int d = 0; d < QO_D; ++d)
                    dot += qo_bf16_to_f64(qrot[h][d]) * qo_bf16_to_f64(krot[d]);
                z[h * nkeys + jj] = dot * scale;
            }
        }
    }
    for (int h = 0; h < QO_HQ; ++h) {
        int g = h / (QO_HQ / QO_HKV);
        double m = -INFINITY;
        for (int64_t jj = 0; jj < nkeys; ++jj) if (z[h * nkeys + jj] > m) m = z[h * nkeys + jj];
        double l = 0.0;
        for (int64_t jj = 0; jj < nkeys; ++jj) l += exp(z[h * nkeys + jj] - m);
        for (int d = 0; d < QO_D; ++d) o[h * QO_D + d] = 0.0;
        for (int64_t jj = 0; jj < nkeys; ++jj) {
            double p = exp(z[h * nkeys + jj] - m) / l;
            const uint16_t *vr = v + (keys[jj] * QO_HKV + g) * QO_D;
            for (int d = 0; d < QO_D; ++d) o[h * QO_D + d] += p * qo_bf16_to_f64(vr[d]);
        }
        lse[h] = m + log(l);
    }
    free(z);
    free(keys);
}

/* --------------------------------------------------------- whole layer -- */

/* Prefill: the QSA layer for the query rows listed in rows[] of a sequence
 * of L tokens (positions 0..L-1).
 *   q [L,24,256], k [L,2,256], v [L,2,256] (k pre-RoPE)
 *   qi [L,4,128], w [L,4], ki [L,128]
 * Outputs are per listed row (any may be NULL):
 *   idx [nrows,budget], sel_score [nrows,budget], o [nrows,24,256], lse [nrows,24].
 * If idx_given is non-NULL ([nrows,budget]), the selection step is skipped
 * and attention runs over the given blocks (used to compare attention on
 * one and the same selection). */
void qo_prefill_rows(int64_t L, int budget, const double *inv_freq, double scale,
                     const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const uint16_t *qi, const uint16_t *w, const uint16_t *ki,
                     const int64_t *rows, int64_t nrows, const int32_t *idx_given,
                     int32_t *idx, double *sel_score, double *o, double *lse,
                     int nthreads)
{
    int64_t nb = L / QO_BS;
    uint16_t *kblk = NULL;
    if (!idx_given) {
        kblk = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)((nb > 0 ? nb : 1) * QO_DI));
        qo_block_keys(L, ki, kblk);
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t t = rows[r];
        int64_t c = t / QO_BS;
        int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)budget);
        double *ss = (double *)malloc(sizeof(double) * (size_t)budget);
        int nsel;
        if (idx_given) {
            memcpy(sel, idx_given + r * budget, sizeof(int32_t) * (size_t)budget);
            nsel = budget;
        } else {
            double *s = (double *)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1));
            qo_block_scores(qi + t * QO_HI * QO_DI, w + t * QO_HI, kblk, c, s);
            qo_select(s, c, budget, sel, ss);
            nsel = budget;
            free(s);
        }
        if (idx) memcpy(idx + r * budget, sel, sizeof(int32_t) * (size_t)budget);
        if (sel_score) memcpy(sel_score + r * budget, ss, sizeof(double) * (size_t)budget);
        if (o || lse) {
            double ob[QO_HQ * QO_D], lb[QO_HQ];
            qo_attend(q + t * QO_HQ * QO_D, t, k, v, sel, nsel, inv_freq, scale, ob, lb);
            if (o) memcpy(o + r * QO_HQ * QO_D, ob, sizeof ob);
            if (lse) memcpy(lse + r * QO_HQ, lb, sizeof lb);
        }
        free(sel);
        free(ss);
    }
    free(kblk);
}

/* Prefill scores without selection: s[r, b] for b < c(rows[r]); entries
 * b >= c are set to NaN.  out is [nrows, L/4]. */
void qo_prefill_scores(int64_t L, const uint16_t *qi, const uint16_t *w, const uint16_t *ki,
                       const int64_t *rows, int64_t nrows, double *out, int nthreads)
{
    int64_t nb = L / QO_BS;
    uint16_t *kblk = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)((nb > 0 ? nb : 1) * QO_DI));
    qo_block_keys(L, ki, kblk);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t t = rows[r];
        int64_t c = t / QO_BS;
        double *row = out + r * nb;
        qo_block_scores(qi + t * QO_HI * QO_DI, w + t * QO_HI, kblk, c < nb ? c : nb, row);
        for (int64_t b = c; b < nb; ++b) row[b] = NAN;
    }
    free(kblk);
}

/* Decode: one new token per sequence.  Sequence s holds seq_lens[s] = T
 * tokens (the new one included, at position T-1) in caches laid out
 * [B, Tmax, ...]:
 *   k_raw, v [B,Tmax,2,256] (k pre-RoPE), ki_raw [B,Tmax,128]
 *   q [B,24,256] pre-RoPE, qi [B,4,128], w [B,4]
 * Outputs [B,budget] / [B,24,256] / [B,24]; idx_given as for prefill. */
void qo_decode(int B, int64_t Tmax, const int64_t *seq_lens, int budget, const double *inv_freq,
               double scale, const uint16_t *q, const uint16_t *qi, const uint16_t *w,
               const uint16_t *k_raw, const uint16_t *v, const uint16_t *ki_raw,
               const int32_t *idx_given, int32_t *idx, double *sel_score, double *o,
               double *lse, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel for schedule(dynamic, 1)
    for (int s = 0; s < B; ++s) {
        int64_t T = seq_lens[s];
        int64_t t = T - 1;
        int64_t c = t / QO_BS;
        const uint16_t *ks = k_raw + (int64_t)s * Tmax * QO_HKV * QO_D;
        const uint16_t *vs = v + (int64_t)s * Tmax * QO_HKV * QO_D;
        int32_t *sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)budget);
        double *ss = (double *)malloc(sizeof(double) * (size_t)budget);
        if (idx_given) {
            memcpy(sel, idx_given + (int64_t)s * budget, sizeof(int32_t) * (size_t)budget);
        } else {
            /* block keys of the complete past blocks 0..c-1 */
            uint16_t *kblk = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)((c > 0 ? c : 1) * QO_DI));
            qo_block_keys(c * QO_BS, ki_raw + (int64_t)s * Tmax * QO_DI, kblk);
            double *sc = (double *)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1));
            qo_block_scores(qi + (int64_t)s * QO_HI * QO_DI, w + (int64_t)s * QO_HI, kblk, c, sc);
            qo_select(sc, c, budget, sel, ss);
            free(sc);
            free(kblk);
        }
        if (idx) memcpy(idx + (int64_t)s * budget, sel, sizeof(int32_t) * (size_t)budget);
        if (sel_score) memcpy(sel_score + (int64_t)s * budget, ss, sizeof(double) * (size_t)budget);
        if (o || lse) {
            double ob[QO_HQ * QO_D], lb[QO_HQ];
            qo_attend(q + (int64_t)s * QO_HQ * QO_D, t, ks, vs, sel, budget, inv_freq, scale, ob, lb);
            if (o) memcpy(o + (int64_t)s * QO_HQ * QO_D, ob, sizeof ob);
            if (lse) memcpy(lse + (int64_t)s * QO_HQ, lb, sizeof lb);
        }
        free(sel);
        free(ss);
    }
}

int qo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
