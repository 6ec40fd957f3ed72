/*
 * oracle.c -- plain CPU oracle (fp64) for the prerouted MoE decode layer.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, __graft_entry__.smoke() and
 * bench.py's CPU baseline leg.  The product never links, loads or calls it.
 * See oracle.h for the definitions and the pages each function follows.
 *
 * Style: every function is the plain definition, written out.  Sums run in
 * ascending index order in double; no blocking, fusion or reordering.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================== */
/* Storage formats                                                          */
/* ======================================================================== */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)frac, -24);                 /* zero / subnormal */
    else if (e == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), e - 25);     /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

/* Rounds |v| to an integer count of the unit 2^unit_exp, ties to even. */
static double round_units(double a, int unit_exp)
{
    return nearbyint(ldexp(a, -unit_exp));   /* default mode: nearest-even */
}

uint16_t orc_f64_to_f16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7e00;
    if (isinf(v))
        return sign | 0x7c00;
    if (a >= 65520.0)                 /* midpoint of 65504 and 2^16 -> inf */
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {        /* subnormal range: unit 2^-24 */
        double n = round_units(a, -24);      /* 0 .. 1024; 1024 = min normal */
        return sign | (uint16_t)n;
    }
    int ex;
    frexp(a, &ex);                    /* a in [2^(ex-1), 2^ex) */
    int E = ex - 1;
    double n = round_units(a, E - 10);       /* 1024 .. 2048 */
    if (n >= 2048.0) {
        n = 1024.0;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)n - 1024));
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double orc_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)frac, -133);                /* 2^-126 * f/128 */
    else if (e == 255)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + frac), e - 134);     /* (1.f) * 2^(e-127) */
    return sign ? -v : v;
}

uint16_t orc_f64_to_bf16(double v)
{
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v))
        return 0x7fc0;
    if (isinf(v))
        return sign | 0x7f80;
    if (a < ldexp(1.0, -126)) {       /* subnormal range: unit 2^-133 */
        double n = round_units(a, -133);     /* 0 .. 128; 128 = min normal */
        return sign | (uint16_t)n;
    }
    int ex;
    frexp(a, &ex);
    int E = ex - 1;
    double n = round_units(a, E - 7);        /* 128 .. 256 */
    if (n >= 256.0) {
        n = 128.0;
        E += 1;
    }
    if (E > 127)
        return sign | 0x7f80;
    return sign | (uint16_t)(((E + 127) << 7) | ((int)n - 128));
}

/* ======================================================================== */
/* Weight matrices                                                          */
/* ======================================================================== */

double orc_weight(const orc_mat *m, int o, int k)
{
    if (m->kind == ORC_F16)
        return orc_f16_to_f64(m->f16[(size_t)o * m->cols + k]);
    int per_word = 32 / m->bits;
    int words_per_row = m->cols / per_word;
    uint32_t word = m->q[(size_t)o * words_per_row + k / per_word];
    uint32_t mask = (1u << m->bits) - 1u;
    uint32_t n = (word >> (m->bits * (k % per_word))) & mask;
    int groups = m->cols / m->group;
    double s = orc_f16_to_f64(m->s[(size_t)o * groups + k / m->group]);
    double b = orc_f16_to_f64(m->b[(size_t)o * groups + k / m->group]);
    return (double)n * s + b;
}

void orc_dequant(const orc_mat *m, double *w)
{
    for (int o = 0; o < m->rows; o++)
        for (int k = 0; k < m->cols; k++)
            w[(size_t)o * m->cols + k] = orc_weight(m, o, k);
}

/* Threads the row loops of orc_gemv and orc_head_logits may use (1 unless
 * orc_set_threads raised it; only when built with OpenMP).  A row is always
 * summed by one thread in ascending index order, so results are the same
 * bits at any count. */
static int orc_threads = 1;

void orc_set_threads(int n) { orc_threads = n > 0 ? n : 1; }

int orc_openmp(void)
{
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

void orc_gemv(const orc_mat *m, const double *x, double *y)
{
#pragma omp parallel for num_threads(orc_threads) schedule(static) if (orc_threads > 1)
    for (int o = 0; o < m->rows; o++) {
        double acc = 0.0;
        for (int k = 0; k < m->cols; k++)
            acc += orc_weight(m, o, k) * x[k];
        y[o] = acc;
    }
}

/* ======================================================================== */
/* LoRA and activations                                                     */
/* ======================================================================== */

void orc_lora_apply(const orc_lora *l, int in, int out, const double *x,
                    double *y)
{
    if (l == NULL || l->r == 0)
        return;
    double *v = (double *)calloc((size_t)l->r, sizeof(double));
    for (int i = 0; i < l->r; i++) {                  /* v = A x */
        double acc = 0.0;
        for (int k = 0; k < in; k++)
            acc += orc_f16_to_f64(l->A[(size_t)i * in + k]) * x[k];
        v[i] = acc;
    }
    for (int o = 0; o < out; o++) {                   /* y += scale * B v */
        double acc = 0.0;
        for (int i = 0; i < l->r; i++)
            acc += orc_f16_to_f64(l->B[(size_t)o * l->r + i]) * v[i];
        y[o] += l->scale * acc;
    }
    free(v);
}

double orc_silu(double g) { return g / (1.0 + exp(-g)); }

double orc_gelu_erf(double a) { return 0.5 * a * (1.0 + erf(a / sqrt(2.0))); }

/* ======================================================================== */
/* Experts                                                                  */
/* ======================================================================== */

void orc_expert_forward(const orc_expert *ex, const double *x,
                        int round_h_bf16, double *h_out, double *y)
{
    int F = ex->gate.rows, d = ex->gate.cols;
    double *g = (double *)calloc((size_t)F, sizeof(double));
    double *u = (double *)calloc((size_t)F, sizeof(double));
    double *h = (double *)calloc((size_t)F, sizeof(double));
    orc_gemv(&ex->gate, x, g);
    orc_lora_apply(&ex->lg, d, F, x, g);
    orc_gemv(&ex->up, x, u);
    orc_lora_apply(&ex->lu, d, F, x, u);
    for (int f = 0; f < F; f++) {
        h[f] = orc_silu(g[f]) * u[f];
        if (round_h_bf16)
            h[f] = orc_bf16_to_f64(orc_f64_to_bf16(h[f]));
    }
    orc_gemv(&ex->down, h, y);
    orc_lora_apply(&ex->ld, F, ex->down.rows, h, y);
    if (h_out)
        memcpy(h_out, h, (size_t)F * sizeof(double));
    free(g);
    free(u);
    free(h);
}

void orc_expert_ffn(const orc_expert *experts, int E, const orc_expert *shared,
                    int d, const double *x, const int32_t *idx, int T, int K,
                    int round_h_bf16, double *y_slots)
{
    int slots = K + (shared != NULL);
    for (int t = 0; t < T; t++) {
        for (int k = 0; k < K; k++) {
            int e = idx[(size_t)t * K + k];
            if (e < 0 || e >= E)
                abort();
            orc_expert_forward(&experts[e], x + (size_t)t * d, round_h_bf16,
                               NULL, y_slots + ((size_t)t * slots + k) * d);
        }
        if (shared)
            orc_expert_forward(shared, x + (size_t)t * d, round_h_bf16, NULL,
                               y_slots + ((size_t)t * slots + K) * d);
    }
}

/* ======================================================================== */
/* Prerouter head                                                           */
/* ======================================================================== */

void orc_head_features(int d, int E, const double *x, const int32_t *cur,
                       const int32_t *prev, int K, double *f)
{
    for (int k = 0; k < d; k++)
        f[k] = x[k];
    for (int c = 0; c < 2 * E; c++)
        f[d + c] = 0.0;
    for (int k = 0; k < K; k++) {
        if (cur)
            f[d + cur[k]] = 1.0;           /* K-hot of the current route  */
        if (prev)
            f[d + E + prev[k]] = 1.0;      /* K-hot of the previous route */
    }
}

static double bias_or_zero(const uint16_t *b, int i)
{
    return b ? orc_f16_to_f64(b[i]) : 0.0;
}

/* Element (o, c) of a matrix whose first d columns are `dense` and whose
 * last 2E columns are the transposed table tab[2E][rows]. */
static double split_weight(const orc_mat *dense, const uint16_t *tab,
                           int rows, int d, int o, int c)
{
    if (c < d)
        return orc_weight(dense, o, c);
    return tab ? orc_f16_to_f64(tab[(size_t)(c - d) * rows + o]) : 0.0;
}

void orc_head_logits(const orc_head *hd, const double *x, const int32_t *cur,
                     const int32_t *prev, int K, double *z)
{
    int d = hd->d, E = hd->E, H = hd->H, width = d + 2 * E;
    double *f = (double *)calloc((size_t)width, sizeof(double));
    orc_head_features(d, E, x, cur, prev, K, f);

    double *g = (double *)calloc((size_t)(H > 0 ? H : 1), sizeof(double));
#pragma omp parallel for num_threads(orc_threads) schedule(static) if (orc_threads > 1)
    for (int o = 0; o < H; o++) {                     /* a = fc1 f + b1 */
        double acc = 0.0;
        for (int c = 0; c < width; c++)
            acc += split_weight(&hd->fc1x, hd->fc1_tab, H, d, o, c) * f[c];
        g[o] = orc_gelu_erf(acc + bias_or_zero(hd->b1, o));
    }
#pragma omp parallel for num_threads(orc_threads) schedule(static) if (orc_threads > 1)
    for (int e = 0; e < E; e++) {
        double acc = 0.0;
        for (int o = 0; o < H; o++)                   /* fc2 gelu(a) */
            acc += orc_weight(&hd->fc2, e, o) * g[o];
        acc += bias_or_zero(hd->b2, e);
        double lin = 0.0;
        for (int c = 0; c < width; c++)               /* l f */
            lin += split_weight(&hd->lx, hd->l_tab, E, d, e, c) * f[c];
        z[e] = acc + lin + bias_or_zero(hd->bl, e);
    }
    free(f);
    free(g);
}

/* ======================================================================== */
/* Top-K and weights                                                        */
/* ======================================================================== */

typedef struct {
    double v;
    int i;
} vi_pair;

static int by_value_desc_index_asc(const void *pa, const void *pb)
{
    const vi_pair *a = (const vi_pair *)pa, *b = (const vi_pair *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->i > b->i) - (a->i < b->i);
}

void orc_route_weights(const double *z, const int32_t *idx, int K, double *w)
{
    double zmax = -INFINITY;
    for (int k = 0; k < K; k++)
        if (z[idx[k]] > zmax)
            zmax = z[idx[k]];
    double sum = 0.0;
    for (int k = 0; k < K; k++)
        sum += exp(z[idx[k]] - zmax);
    for (int k = 0; k < K; k++)
        w[k] = exp(z[idx[k]] - zmax) / sum;
}

void orc_topk(const double *z, int E, int K, int32_t *idx, double *w,
              double *margin)
{
    vi_pair *p = (vi_pair *)malloc((size_t)E * sizeof(vi_pair));
    for (int e = 0; e < E; e++) {
        p[e].v = z[e];
        p[e].i = e;
    }
    qsort(p, (size_t)E, sizeof(vi_pair), by_value_desc_index_asc);
    for (int k = 0; k < K; k++)
        idx[k] = p[k].i;
    if (w)
        orc_route_weights(z, idx, K, w);
    if (margin)
        *margin = (K < E) ? p[K - 1].v - p[K].v : INFINITY;
    free(p);
}

/* ======================================================================== */
/* Combine                                                                  */
/* ======================================================================== */

void orc_combine(const double *y_slots, const double *w, int K, int has_shared,
                 int d, const double *residual, double *out, double *x_next)
{
    for (int i = 0; i < d; i++) {
        double acc = residual[i];
        for (int k = 0; k < K; k++)
            acc += w[k] * y_slots[(size_t)k * d + i];
        if (has_shared)
            acc += y_slots[(size_t)K * d + i];
        out[i] = acc;
    }
    if (x_next) {
        double ss = 0.0;
        for (int i = 0; i < d; i++)
            ss += out[i] * out[i];
        double inv = 1.0 / sqrt(ss / d + 1e-6);
        for (int i = 0; i < d; i++)
            x_next[i] = out[i] * inv;
    }
}

/* ======================================================================== */
/* Stack step                                                               */
/* ======================================================================== */

/* Route for layer N from logits z; adopts ext (if given) at near-ties. */
static void take_route(const double *z, int E, int K, const int32_t *chosen,
                       double chosen_margin, const int32_t *ext,
                       double tie_margin, int32_t *idx, double *w,
                       double *margin_out, uint8_t *forced)
{
    for (int k = 0; k < K; k++)
        idx[k] = chosen[k];
    *forced = 0;
    if (ext && chosen_margin <= tie_margin) {
        for (int k = 0; k < K; k++)
            idx[k] = ext[k];
        *forced = 1;
    }
    orc_route_weights(z, idx, K, w);
    *margin_out = chosen_margin;
    (void)E;
}

void orc_stack_step(const orc_stack *st, orc_stack_state *state,
                    const double *x0, const int32_t *ext_idx,
                    double tie_margin, double *out_last, int32_t *used_idx,
                    double *used_w, double *used_margin, uint8_t *forced)
{
    int L = st->L, d = st->d, E = st->E, K = st->K;
    int t = state->t;
    double *stream = (double *)malloc((size_t)d * sizeof(double));
    double *x = (double *)malloc((size_t)d * sizeof(double));
    double *out = (double *)malloc((size_t)d * sizeof(double));
    double *xn = (double *)malloc((size_t)d * sizeof(double));
    double *z = (double *)malloc((size_t)E * sizeof(double));
    int32_t *cur = (int32_t *)malloc((size_t)L * K * sizeof(int32_t));
    double *w = (double *)malloc((size_t)K * sizeof(double));
    int32_t *own = (int32_t *)malloc((size_t)K * sizeof(int32_t));
    int slots_max = K + 1;
    double *y = (double *)malloc((size_t)slots_max * d * sizeof(double));
    /* predictions made during this step are for the next one: keep them
       apart from the ones this step consumes */
    int32_t *nx_idx = (int32_t *)malloc((size_t)L * K * sizeof(int32_t));
    double *nx_z = (double *)malloc((size_t)L * E * sizeof(double));
    double *nx_margin = (double *)malloc((size_t)L * sizeof(double));
    memcpy(nx_idx, state->pred_idx, (size_t)L * K * sizeof(int32_t));
    memcpy(nx_z, state->pred_z, (size_t)L * E * sizeof(double));
    memcpy(nx_margin, state->pred_margin, (size_t)L * sizeof(double));

    memcpy(stream, x0, (size_t)d * sizeof(double));
    memcpy(x, x0, (size_t)d * sizeof(double));

    for (int N = 0; N < L; N++) {
        const orc_layer *ly = &st->layers[N];
        int32_t *idx = cur + (size_t)N * K;
        double margin;
        uint8_t fz;
        const int32_t *ext = ext_idx ? ext_idx + (size_t)N * K : NULL;

        int use_prediction = (t > 0) &&
            (N > 0 || (L == 1 && st->single_layer_self_predict));
        if (use_prediction) {
            const double *pz = state->pred_z + (size_t)N * E;
            take_route(pz, E, K, state->pred_idx + (size_t)N * K,
                       state->pred_margin[N], ext, tie_margin, idx, w,
                       &margin, &fz);
        } else {
            double m;
            orc_head_logits(&ly->router, x, NULL, NULL, K, z);
            orc_topk(z, E, K, own, NULL, &m);
            take_route(z, E, K, own, m, ext, tie_margin, idx, w, &margin,
                       &fz);
        }
        if (used_idx)
            memcpy(used_idx + (size_t)N * K, idx, (size_t)K * sizeof(int32_t));
        if (used_w)
            memcpy(used_w + (size_t)N * K, w, (size_t)K * sizeof(double));
        if (used_margin)
            used_margin[N] = margin;
        if (forced)
            forced[N] = fz;

        /* experts, then combine with the residual stream */
        orc_expert_ffn(ly->experts, E, ly->shared, d, x, idx, 1, K, 0, y);
        orc_combine(y, w, K, ly->shared != NULL, d, stream, out, xn);

        /* head N on x_N predicts the next step's route of layer N+1
           (or of layer 0 itself for a single self-predicting layer) */
        int target = (N + 1 < L) ? N + 1 : (st->single_layer_self_predict ? 0 : -1);
        if (target >= 0) {
            const int32_t *prev = t > 0 ? state->prev_idx + (size_t)N * K : NULL;
            double *pz = nx_z + (size_t)target * E;
            orc_head_logits(&ly->head, x, idx, prev, K, pz);
            orc_topk(pz, E, K, nx_idx + (size_t)target * K, NULL,
                     &nx_margin[target]);
        }

        memcpy(stream, out, (size_t)d * sizeof(double));
        memcpy(x, xn, (size_t)d * sizeof(double));
    }
    memcpy(state->prev_idx, cur, (size_t)L * K * sizeof(int32_t));
    memcpy(state->pred_idx, nx_idx, (size_t)L * K * sizeof(int32_t));
    memcpy(state->pred_z, nx_z, (size_t)L * E * sizeof(double));
    memcpy(state->pred_margin, nx_margin, (size_t)L * sizeof(double));
    memcpy(out_last, stream, (size_t)d * sizeof(double));
    state->t = t + 1;

    free(stream);
    free(x);
    free(out);
    free(xn);
    free(z);
    free(cur);
    free(w);
    free(own);
    free(y);
    free(nx_idx);
    free(nx_z);
    free(nx_margin);
}

/* ======================================================================== */
/* Merging a LoRA delta into the quantised weights (fp64, see oracle.h)      */
/* ======================================================================== */

void orc_merge_weights(const orc_mat *m, const orc_lora *l, double *w)
{
    orc_dequant(m, w);
    if (!l || l->r == 0)
        return;
    for (int o = 0; o < m->rows; o++)
        for (int k = 0; k < m->cols; k++) {
            double d = 0.0;
            for (int j = 0; j < l->r; j++)
                d += orc_f16_to_f64(l->B[(size_t)o * l->r + j]) *
                     orc_f16_to_f64(l->A[(size_t)j * m->cols + k]);
            w[(size_t)o * m->cols + k] += l->scale * d;
        }
}

void orc_quant_codes(const double *w, int rows, int cols, int bits, int group,
                     const uint16_t *s, const uint16_t *b, uint32_t *q_out,
                     double *t_pre)
{
    const int per = 32 / bits, ng = cols / group;
    const double qmax = (double)((1 << bits) - 1);
    memset(q_out, 0, sizeof(uint32_t) * (size_t)rows * (cols / per));
    for (int o = 0; o < rows; o++)
        for (int k = 0; k < cols; k++) {
            const double sv = orc_f16_to_f64(s[(size_t)o * ng + k / group]);
            const double bv = orc_f16_to_f64(b[(size_t)o * ng + k / group]);
            double t = 0.0, q = 0.0;
            if (sv != 0.0) {
                t = (w[(size_t)o * cols + k] - bv) / sv;
                q = nearbyint(t);                     /* nearest, ties even */
                q = q < 0.0 ? 0.0 : (q > qmax ? qmax : q);
            }
            if (t_pre)
                t_pre[(size_t)o * cols + k] = t;
            q_out[(size_t)o * (cols / per) + k / per] |=
                (uint32_t)q << (bits * (k % per));
        }
}

void orc_requantise(const double *w, int rows, int cols, int bits, int group,
                    uint32_t *q_out, uint16_t *s_out, uint16_t *b_out,
                    double *s_pre, double *b_pre, double *t_pre)
{
    const int ng = cols / group;
    const double qmax = (double)((1 << bits) - 1);
    for (int o = 0; o < rows; o++)
        for (int g = 0; g < ng; g++) {
            const double *wg = w + (size_t)o * cols + (size_t)g * group;
            double lo = wg[0], hi = wg[0];
            for (int i = 1; i < group; i++) {
                if (wg[i] < lo) lo = wg[i];
                if (wg[i] > hi) hi = wg[i];
            }
            const double span = (hi - lo) / qmax;
            s_out[(size_t)o * ng + g] = orc_f64_to_f16(span);
            b_out[(size_t)o * ng + g] = orc_f64_to_f16(lo);
            if (s_pre)
                s_pre[(size_t)o * ng + g] = span;
            if (b_pre)
                b_pre[(size_t)o * ng + g] = lo;
        }
    orc_quant_codes(w, rows, cols, bits, group, s_out, b_out, q_out, t_pre);
}

void orc_merge_lora(const orc_mat *m, const orc_lora *l, uint32_t *q_out,
                    uint16_t *s_out, uint16_t *b_out, double *s_pre,
                    double *b_pre, double *t_pre)
{
    double *w = malloc(sizeof(double) * (size_t)m->rows * m->cols);
    orc_merge_weights(m, l, w);
    orc_requantise(w, m->rows, m->cols, m->bits, m->group, q_out, s_out,
                   b_out, s_pre, b_pre, t_pre);
    free(w);
}
