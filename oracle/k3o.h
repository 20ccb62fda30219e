/*
 * k3o.h -- the ORACLE of the MXFP4 routed-expert MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, scalar fp64 CPU statement of what the
 * layer computes.  Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no code, header, table or constant with the CUDA library
 * (mxfp4_routed_expert_gemv_gb300/csrc), and it includes nothing from there.
 *
 * Sources (web pages, cited by title and section):
 *   [README]  "kimi-k3-in-c" README (runchr.com English edition; shilu.ai Chinese edition)
 *             Part II section 4 "Reduction one: the experts already ship at half a byte"
 *             Part II section 5 "Kernels with a floating point contract"
 *             Part II section 9 "Picking 16 experts of 896"
 *   [AUDIT]   "K3_ARTIFACT_AUDIT" (llm-atlas), section 4.3 (one routed expert's MXFP4
 *             tensors: shapes, byte counts, group size 32)
 *
 * Every floating-point step is fp64.  bf16 inputs widen to fp64 exactly.  Products of a
 * bf16 value, an E2M1 value and a power of two are exact in fp64, so the MXFP4 mat-vec
 * below equals the exact dot product up to the rounding of its fp64 additions.
 */
#ifndef K3O_H
#define K3O_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Layer configuration.  Field meanings follow the README's config struct
 * (hidden, n_experts, topk, moe_renorm, routed_scale, situ_b1/b2) and the audit's
 * expert shapes (latent 3584, inter 3072, group 32). */
typedef struct k3o_cfg {
    int hidden;          /* router input width H                                   */
    int n_experts;       /* E                                                      */
    int topk;            /* k                                                      */
    int latent;          /* L: expert input and output width                       */
    int inter;           /* I: expert intermediate width                           */
    int group;           /* MX group: consecutive weights sharing one E8M0 scale   */
    int renorm;          /* 1: gates renormalised to sum 1 over the chosen k       */
    double routed_scale; /* gates are multiplied by this after renormalisation     */
    int act;             /* 0: SwiGLU  silu(g)*u ;  1: SiTU-GLU (README section 9) */
    double situ_b1;      /* SiTU gate cap b1                                       */
    double situ_b2;      /* SiTU up cap b2                                         */
} k3o_cfg;

/* One expert's six tensors in checkpoint row layout (host memory):
 *   w1p, w3p: [inter][ceil(latent/2)]  packed E2M1, low nibble = even column
 *   w1s, w3s: [inter][ceil(latent/group)] E8M0 scale bytes
 *   w2p:      [latent][ceil(inter/2)]
 *   w2s:      [latent][ceil(inter/group)]                                           */
typedef struct k3o_expert {
    const uint8_t *w1p, *w1s, *w3p, *w3s, *w2p, *w2s;
} k3o_expert;

enum { K3O_OK = 0, K3O_ERR_ARG = 1, K3O_ERR_MISSING_EXPERT = 2, K3O_ERR_NOMEM = 3 };

/* E2M1 code (0..15) -> value.  README section 4 code table. */
double k3o_e2m1(int code);
/* E8M0 scale byte -> 2^(b-127); byte 255 (NaN in the MX spec) -> 0.  README section 4. */
double k3o_e8m0(int byte);
/* bf16 bit pattern -> its exact value. */
double k3o_bf16_value(uint16_t bits);
/* fp32 -> bf16 bit pattern, round to nearest, ties to even (NaN kept quiet). */
uint16_t k3o_bf16_from_f32(float v);

/* y[r] = sum_c W[r][c] x[c] for an MXFP4 matrix W[rows][in] (README section 4 mat-vec).
 * Per group: part = sum of x*E2M1 in fp64, acc += part*scale; a zero scale skips the group. */
void k3o_matvec_mxfp4(double *y, const double *x, const uint8_t *packed,
                      const uint8_t *scales, int in, int rows, int group);

/* The dense fp64 matrix W [rows][in] of an MXFP4 matrix (packed [rows][ceil(in/2)],
 * scales [rows][ceil(in/group)]): W[r][c] = E2M1[nibble] * 2^(s - 127), s = 255 -> 0
 * (README Part II section 4). */
void k3o_dequant_mxfp4(double *w, const uint8_t *packed, const uint8_t *scales, int in,
                       int rows, int group);

/* Router for T tokens (README section 9):
 *   logit[t][e] = sum_i h[t][i]*Wr[e][i]            (bf16 inputs, fp64 sum)
 *   sc = 1/(1+exp(-logit))                           unbiased score
 *   ch = sc + bias[e]  (bias may be NULL)            selection score
 *   top-k over ch by repeated arg-max, strict '>' (the lower index wins a tie)
 *   gate_j = sc[idx_j]; renormalised by their sum when renorm and the sum is > 0;
 *   then multiplied by routed_scale.
 * Outputs: idx[T][k], gate[T][k], gap[T] = ch[idx_{k-1}] - max over unchosen ch
 * (+inf when k == E).  sc_out[T][E] and ch_out[T][E] are optional (NULL to skip).
 * Returns K3O_OK or K3O_ERR_ARG. */
int k3o_route(const k3o_cfg *c, const uint16_t *h, const uint16_t *wr, const float *bias,
              int T, int32_t *idx, double *gate, double *gap, double *sc_out,
              double *ch_out);

/* Gates for a given index list from one token's unbiased scores sc[E] (the last two
 * steps of the router).  Used to score a different but equally valid top-k choice. */
void k3o_gates_for(const k3o_cfg *c, const double *sc, const int32_t *idx, double *gate);

/* Expert activation (n values): SwiGLU act = g*sigmoid(g)*u, or SiTU-GLU
 * act = b1*tanh(g/b1)*sigmoid(g) * b2*tanh(u/b2)  (README section 9). */
void k3o_activation(const k3o_cfg *c, const double *g, const double *u, double *act, int n);

/* One expert FFN on one latent vector x[L]: g = W1 x, u = W3 x, a = act(g,u),
 * o = W2 a.  o has L entries.  Returns K3O_OK, K3O_ERR_ARG or K3O_ERR_NOMEM. */
int k3o_expert_ffn(const k3o_cfg *c, const k3o_expert *ex, const double *x, double *o);

/* The routed-expert sum for T tokens (steps 3 of the README's per-token MoE):
 *   y[t] = sum_j gate[t][j] * FFN_{idx[t][j]}(x[t])
 * x is bf16 [T][L]; table[e] holds expert e (entries not referenced by idx may be
 * all-NULL).  Returns K3O_ERR_MISSING_EXPERT if a referenced expert is absent or an
 * index is out of [0, n_table). */
int k3o_experts(const k3o_cfg *c, const k3o_expert *table, int n_table, const uint16_t *x,
                const int32_t *idx, const double *gate, int T, double *y);

/* RMSNorm with unit weight, eps inside the square root, fp64 throughout
 * (README section 5): out = x / sqrt(mean(x^2) + eps). */
void k3o_rmsnorm(double *out, const double *x, int n, double eps);

/* RMSNorm with a per-element weight (NULL: unit weight), eps inside the square root, fp64
 * throughout (README section 5): out[i] = x[i] / sqrt(mean(x^2) + eps) * w[i]. */
void k3o_rmsnorm_w(double *out, const double *x, const float *w, int n, double eps);

/* Dense mat-vec with bf16 weights W[rows][in] (row-major): y[r] = sum_c W[r][c] x[c], fp64.
 * The README's dense matmul of the LatentMoE wrapper (section 9, k3_moe's k3_mmw). */
void k3o_matvec_bf16(double *y, const double *x, const uint16_t *W, int in, int rows);

/* The dense tensors of the LatentMoE wrapper around the routed experts (README Part II
 * section 9, k3_moe), bf16 row-major unless noted:
 *   down [latent][hidden]     z = down . h          (routed experts run on z)
 *   up   [hidden][latent]     out = up . norm(acc)  (acc = the routed-expert sum)
 *   norm_w [latent] fp32 or NULL (unit); latent_norm = 1 applies the RMSNorm to acc
 *   sh1, sh3 [n_shared*inter][hidden], sh2 [hidden][n_shared*inter]: the shared experts,
 *   on the full-width h, added unweighted; n_shared = 0 for none. */
typedef struct k3o_latent {
    const uint16_t *down, *up;
    const float *norm_w;
    int latent_norm;
    double rms_eps;
    int n_shared;
    const uint16_t *sh1, *sh3, *sh2;
} k3o_latent;

/* The LatentMoE layer for T tokens, per token t (README Part II section 9, k3_moe):
 *   route on h[t] (k3o_route: idx, gate);
 *   z = bf16(down . h[t])                  (the latent enters the experts as bf16: the
 *                                           library's expert input type; fp64 -> fp32 ->
 *                                           bf16 round to nearest even);
 *   acc = sum_j gate_j FFN_{idx_j}(z)      (k3o_experts);
 *   a = latent_norm ? rmsnorm_w(acc) : acc;
 *   out[t] = up . a  +  sh2 . act(sh1 . h[t], sh3 . h[t])   (act: cfg->act, as the experts).
 * h is bf16 [T][hidden]; out fp64 [T][hidden]; idx [T][k], gate [T][k] are written.
 * Returns K3O_OK, K3O_ERR_ARG, K3O_ERR_MISSING_EXPERT or K3O_ERR_NOMEM. */
int k3o_latent_moe(const k3o_cfg *c, const k3o_latent *lw, const uint16_t *h,
                   const uint16_t *wr, const float *bias, const k3o_expert *table, int n_table,
                   int T, int32_t *idx, double *gate, double *out);

/* Number of OpenMP threads the oracle will use (1 when built without OpenMP). */
int k3o_threads(void);

#ifdef __cplusplus
}
#endif
#endif /* K3O_H */
