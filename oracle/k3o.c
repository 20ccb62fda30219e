/*
 * k3o.c -- ORACLE of the MXFP4 routed-expert MoE layer.  TEST INFRASTRUCTURE ONLY.
 *
 * Plain scalar fp64 C99 (+ optional OpenMP over independent rows and tokens).  It is the
 * plain definition of the layer written out; no blocking, fusion or reordering beyond the
 * group-wise summation the README's MXFP4 mat-vec states.  It shares nothing with the CUDA
 * library.  See k3o.h for the sources and the meaning of every argument.
 */
#include "k3o.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- number formats (README Part II section 4) ------------------------------------ */

/* E2M1: one sign bit, two exponent bits, one mantissa bit.  The sixteen values in code
 * order, as the README's code table prints them (codes 8..15 are the negatives). */
static const double E2M1_VALUES[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

double k3o_e2m1(int code) { return E2M1_VALUES[code & 15]; }

/* E8M0: a bare biased exponent.  The MX spec reserves 0xFF for NaN; the README maps it to
 * zero so that one corrupt byte silences its group instead of poisoning the row. */
double k3o_e8m0(int byte)
{
    byte &= 255;
    if (byte == 255) return 0.0;
    return ldexp(1.0, byte - 127);
}

double k3o_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

uint16_t k3o_bf16_from_f32(float v)
{
    uint32_t u;
    memcpy(&u, &v, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) /* NaN: keep it a NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb; /* round half to even on the 16 dropped bits */
    return (uint16_t)(u >> 16);
}

/* ---- MXFP4 mat-vec (README Part II section 4) -------------------------------------- */

/* Nibble of logical column col in one packed row: byte col/2, low nibble for the even
 * column and high nibble for the odd one. */
static int nibble_at(const uint8_t *row, int col)
{
    int byte = row[col / 2];
    return (col % 2 == 0) ? (byte & 15) : (byte >> 4);
}

void k3o_matvec_mxfp4(double *y, const double *x, const uint8_t *packed,
                      const uint8_t *scales, int in, int rows, int group)
{
    const int ngroup = (in + group - 1) / group;
    const size_t rowbytes = (size_t)(in + 1) / 2;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int r = 0; r < rows; r++) {
        const uint8_t *prow = packed + (size_t)r * rowbytes;
        const uint8_t *srow = scales + (size_t)r * ngroup;
        double acc = 0.0;
        for (int g = 0; g < ngroup; g++) {
            const double s = k3o_e8m0(srow[g]);
            if (s == 0.0) continue; /* a NaN scale silences the whole group */
            const int c0 = g * group;
            const int c1 = (c0 + group < in) ? c0 + group : in;
            double part = 0.0;
            for (int col = c0; col < c1; col++)
                part += x[col] * k3o_e2m1(nibble_at(prow, col));
            acc += part * s;
        }
        y[r] = acc;
    }
}

/* The whole matrix W[r][c] = E2M1[nibble(r, c)] * 2^(scale(r, c / group) - 127) in fp64,
 * a NaN scale (255) giving a zero group: the same definition as the mat-vec above, written
 * out element by element so that a library matmul can take the multiply-adds. */
void k3o_dequant_mxfp4(double *w, const uint8_t *packed, const uint8_t *scales, int in,
                       int rows, int group)
{
    const int ngroup = (in + group - 1) / group;
    const size_t rowbytes = (size_t)(in + 1) / 2;
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int r = 0; r < rows; r++) {
        const uint8_t *prow = packed + (size_t)r * rowbytes;
        const uint8_t *srow = scales + (size_t)r * ngroup;
        double *wr = w + (size_t)r * in;
        for (int col = 0; col < in; col++)
            wr[col] = k3o_e2m1(nibble_at(prow, col)) * k3o_e8m0(srow[col / group]);
    }
}

/* ---- router (README Part II section 9) --------------------------------------------- */

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

void k3o_gates_for(const k3o_cfg *c, const double *sc, const int32_t *idx, double *gate)
{
    double sum = 0.0;
    for (int j = 0; j < c->topk; j++) {
        gate[j] = sc[idx[j]]; /* the unbiased score, never the selection score */
        sum += gate[j];
    }
    if (c->renorm && sum > 0.0)
        for (int j = 0; j < c->topk; j++) gate[j] /= sum;
    for (int j = 0; j < c->topk; j++) gate[j] *= c->routed_scale;
}

int k3o_route(const k3o_cfg *c, const uint16_t *h, const uint16_t *wr, const float *bias,
              int T, int32_t *idx, double *gate, double *gap, double *sc_out,
              double *ch_out)
{
    if (!c || !h || !wr || !idx || !gate || T < 0) return K3O_ERR_ARG;
    const int H = c->hidden, E = c->n_experts, K = c->topk;
    if (H <= 0 || E <= 0 || K <= 0 || K > E) return K3O_ERR_ARG;
    const size_t TE = (size_t)T * (size_t)E;
    double *sc = (double *)malloc(sizeof(double) * (TE ? TE : 1));
    double *ch = (double *)malloc(sizeof(double) * (TE ? TE : 1));
    if (!sc || !ch) {
        free(sc); free(ch);
        return K3O_ERR_NOMEM;
    }
    /* scores: one independent dot product per (token, expert) */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (long long te = 0; te < (long long)TE; te++) {
        const int t = (int)(te / E), e = (int)(te % E);
        const uint16_t *ht = h + (size_t)t * H;
        const uint16_t *we = wr + (size_t)e * H;
        double logit = 0.0;
        for (int i = 0; i < H; i++) logit += k3o_bf16_value(ht[i]) * k3o_bf16_value(we[i]);
        sc[te] = sigmoid(logit);                          /* the unbiased score  */
        ch[te] = sc[te] + (bias ? (double)bias[e] : 0.0); /* the selection score */
    }
    int err = 0;
    /* selection: top-k by repeated arg-max, strict '>' so the lower index wins a tie */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int t = 0; t < T; t++) {
        const double *cht = ch + (size_t)t * E;
        char *taken = (char *)calloc((size_t)E, 1);
        if (!taken) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = 1;
            continue;
        }
        int32_t *it = idx + (size_t)t * K;
        for (int j = 0; j < K; j++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || cht[e] > cht[best])) best = e;
            taken[best] = 1;
            it[j] = best;
        }
        if (gap) {
            int rest = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (rest < 0 || cht[e] > cht[rest])) rest = e;
            gap[t] = (rest < 0) ? INFINITY : cht[it[K - 1]] - cht[rest];
        }
        k3o_gates_for(c, sc + (size_t)t * E, it, gate + (size_t)t * K);
        free(taken);
    }
    if (sc_out) memcpy(sc_out, sc, sizeof(double) * TE);
    if (ch_out) memcpy(ch_out, ch, sizeof(double) * TE);
    free(sc); free(ch);
    return err ? K3O_ERR_NOMEM : K3O_OK;
}

/* ---- expert FFN and the routed sum (README Part II section 9, step 3) -------------- */

void k3o_activation(const k3o_cfg *c, const double *g, const double *u, double *act, int n)
{
    for (int i = 0; i < n; i++) {
        if (c->act == 1) {
            /* SiTU-GLU: the sigmoid takes the uncapped gate */
            const double a = c->situ_b1 * tanh(g[i] / c->situ_b1) * sigmoid(g[i]);
            const double b = c->situ_b2 * tanh(u[i] / c->situ_b2);
            act[i] = a * b;
        } else {
            act[i] = g[i] * sigmoid(g[i]) * u[i]; /* SwiGLU: silu(g) * u */
        }
    }
}

int k3o_expert_ffn(const k3o_cfg *c, const k3o_expert *ex, const double *x, double *o)
{
    if (!c) return K3O_ERR_ARG;
    const int L = c->latent, I = c->inter, G = c->group;
    if (!ex || !ex->w1p || !ex->w1s || !ex->w3p || !ex->w3s || !ex->w2p || !ex->w2s)
        return K3O_ERR_MISSING_EXPERT;
    double *g = (double *)malloc(sizeof(double) * (size_t)I);
    double *u = (double *)malloc(sizeof(double) * (size_t)I);
    double *a = (double *)malloc(sizeof(double) * (size_t)I);
    if (!g || !u || !a) {
        free(g); free(u); free(a);
        return K3O_ERR_NOMEM;
    }
    k3o_matvec_mxfp4(g, x, ex->w1p, ex->w1s, L, I, G);
    k3o_matvec_mxfp4(u, x, ex->w3p, ex->w3s, L, I, G);
    k3o_activation(c, g, u, a, I);
    k3o_matvec_mxfp4(o, a, ex->w2p, ex->w2s, I, L, G);
    free(g); free(u); free(a);
    return K3O_OK;
}

int k3o_experts(const k3o_cfg *c, const k3o_expert *table, int n_table, const uint16_t *x,
                const int32_t *idx, const double *gate, int T, double *y)
{
    if (!c || !table || !x || !idx || !gate || !y || T < 0) return K3O_ERR_ARG;
    const int L = c->latent, K = c->topk;
    if (L <= 0 || K <= 0) return K3O_ERR_ARG;
    double *xd = (double *)malloc(sizeof(double) * (size_t)L);
    double *o = (double *)malloc(sizeof(double) * (size_t)L);
    if (!xd || !o) {
        free(xd); free(o);
        return K3O_ERR_NOMEM;
    }
    int rc = K3O_OK;
    for (int t = 0; t < T && rc == K3O_OK; t++) {
        double *yt = y + (size_t)t * L;
        for (int i = 0; i < L; i++) {
            xd[i] = k3o_bf16_value(x[(size_t)t * L + i]);
            yt[i] = 0.0;
        }
        for (int j = 0; j < K; j++) {
            const int e = idx[(size_t)t * K + j];
            if (e < 0 || e >= n_table) { rc = K3O_ERR_MISSING_EXPERT; break; }
            rc = k3o_expert_ffn(c, &table[e], xd, o);
            if (rc != K3O_OK) break;
            const double w = gate[(size_t)t * K + j];
            for (int i = 0; i < L; i++) yt[i] += w * o[i];
        }
    }
    free(xd); free(o);
    return rc;
}

/* ---- RMSNorm (README Part II section 5) -------------------------------------------- */

void k3o_rmsnorm(double *out, const double *x, int n, double eps)
{
    k3o_rmsnorm_w(out, x, NULL, n, eps);
}

void k3o_rmsnorm_w(double *out, const double *x, const float *w, int n, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += x[i] * x[i];
    const double inv = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; i++) out[i] = x[i] * inv * (w ? (double)w[i] : 1.0);
}

/* ---- the LatentMoE wrapper (README Part II section 9, k3_moe) ----------------------- */

void k3o_matvec_bf16(double *y, const double *x, const uint16_t *W, int in, int rows)
{
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int r = 0; r < rows; r++) {
        const uint16_t *wr = W + (size_t)r * in;
        double acc = 0.0;
        for (int c = 0; c < in; c++) acc += k3o_bf16_value(wr[c]) * x[c];
        y[r] = acc;
    }
}

int k3o_latent_moe(const k3o_cfg *c, const k3o_latent *lw, const uint16_t *h,
                   const uint16_t *wr, const float *bias, const k3o_expert *table, int n_table,
                   int T, int32_t *idx, double *gate, double *out)
{
    if (!c || !lw || !h || !wr || !table || !idx || !gate || !out || T < 0) return K3O_ERR_ARG;
    if (!lw->down || !lw->up || lw->n_shared < 0) return K3O_ERR_ARG;
    if (lw->n_shared > 0 && (!lw->sh1 || !lw->sh3 || !lw->sh2)) return K3O_ERR_ARG;
    const int H = c->hidden, L = c->latent, SI = c->inter * lw->n_shared;
    int rc = k3o_route(c, h, wr, bias, T, idx, gate, NULL, NULL, NULL);
    if (rc != K3O_OK) return rc;
    const size_t nh = (size_t)H, nl = (size_t)L, ns = (size_t)(SI > 0 ? SI : 1);
    double *hd = malloc(nh * sizeof *hd), *zd = malloc(nl * sizeof *zd);
    double *acc = malloc(nl * sizeof *acc), *a = malloc(nl * sizeof *a);
    double *g = malloc(ns * sizeof *g), *u = malloc(ns * sizeof *u), *act = malloc(ns * sizeof *act);
    double *o = malloc(nh * sizeof *o);
    uint16_t *zb = malloc(nl * sizeof *zb);
    if (!hd || !zd || !acc || !a || !g || !u || !act || !o || !zb) {
        rc = K3O_ERR_NOMEM;
        goto done;
    }
    for (int t = 0; t < T && rc == K3O_OK; t++) {
        const uint16_t *ht = h + (size_t)t * H;
        for (int i = 0; i < H; i++) hd[i] = k3o_bf16_value(ht[i]);
        /* down-projection into the latent, rounded to the experts' bf16 input */
        k3o_matvec_bf16(zd, hd, lw->down, H, L);
        for (int i = 0; i < L; i++) zb[i] = k3o_bf16_from_f32((float)zd[i]);
        /* the routed experts on z, with this token's choice and gates */
        rc = k3o_experts(c, table, n_table, zb, idx + (size_t)t * c->topk,
                         gate + (size_t)t * c->topk, 1, acc);
        if (rc != K3O_OK) break;
        /* the aggregate's norm, then back up to full width */
        if (lw->latent_norm) k3o_rmsnorm_w(a, acc, lw->norm_w, L, lw->rms_eps);
        else memcpy(a, acc, nl * sizeof *a);
        double *ot = out + (size_t)t * H;
        k3o_matvec_bf16(ot, a, lw->up, L, H);
        /* shared experts on the full-width input, added unweighted */
        if (SI > 0) {
            k3o_matvec_bf16(g, hd, lw->sh1, H, SI);
            k3o_matvec_bf16(u, hd, lw->sh3, H, SI);
            k3o_activation(c, g, u, act, SI);
            k3o_matvec_bf16(o, act, lw->sh2, SI, H);
            for (int i = 0; i < H; i++) ot[i] += o[i];
        }
    }
done:
    free(hd); free(zd); free(acc); free(a); free(g); free(u); free(act); free(o); free(zb);
    return rc;
}

int k3o_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
