/*
 * oracle.h -- plain CPU oracle for one decode step of a fine-grained MoE FFN
 * layer whose routing is predicted a token ahead.
 *
 * TEST INFRASTRUCTURE ONLY.  This code exists to check the CUDA path.  It is
 * loaded by the tests, by __graft_entry__.smoke() and by bench.py's CPU
 * baseline leg; the product library never links, loads or calls it, and it
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Every floating-point value is carried in double (fp64).  Stored fp16/bf16
 * values are widened exactly; every sum runs in ascending index order.
 * Nothing is blocked, fused or reordered beyond what the definitions state.
 *
 * Sources (the three pages the method is taken from):
 *  - "La otra mitad del muro de la memoria: Servir MoEs de 35B desde SSD con
 *    prediccion de enrutamiento entrenada" (xyznot.com/es/paper/2609.18063),
 *    section "Arquitectura del cabezal Prerouter" (head features, dim = d+2E,
 *    head equation) and "Ejecucion del adaptador no fusionado" (LoRA delta).
 *    "Ideas clave": the prediction is used as the real routing.
 *  - "Inferencia de LLM MoE en MacBook Pro: Streaming de Expertos desde SSD
 *    con Metal" (kerneldigest.dev), section "Arquitectura del Sistema"
 *    (4-/2-bit dequant matvec, fused SwiGLU, RMS norm, fused combine +
 *    residual) and its Metal fragment (affine dequant  nibble*scale + bias).
 *  - "Arquitecturas nativas para device: MoE de grano fino y pre-attention
 *    router" (blog.lo0.es), section "Dos niveles de sparsity" (top-k of many
 *    small experts).
 *
 * Pins: every function here is checked by the "not gpu" tests against
 * closed forms, brute force, library routines or printed values.  The whole
 * layer/stack outputs have no printed end-to-end value on the pages; they are
 * pinned only through the per-function pins (see the tests).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- half-precision storage formats (IEEE binary16, bfloat16) ---------- */
double   orc_f16_to_f64(uint16_t h);
uint16_t orc_f64_to_f16(double v);      /* round to nearest, ties to even */
double   orc_bf16_to_f64(uint16_t h);
uint16_t orc_f64_to_bf16(double v);     /* round to nearest, ties to even */

/* ---- weight matrices ----------------------------------------------------
 * ORC_AFFINE: group-quantised affine weights.  Row o, column k:
 *     word = q[o*(cols*bits/32) + k/(32/bits)]
 *     n    = (word >> (bits * (k % (32/bits)))) & (2^bits - 1)   (LSB first)
 *     W    = n * s[o][k/group] + b[o][k/group]        (s, b stored fp16)
 * ORC_F16: plain fp16 row-major [rows][cols] in f16.                        */
enum { ORC_AFFINE = 0, ORC_F16 = 1 };

typedef struct {
    int kind;              /* ORC_AFFINE or ORC_F16                          */
    int rows, cols;
    int bits, group;       /* ORC_AFFINE only: bits in {2,4}; group 64       */
    const uint32_t *q;     /* ORC_AFFINE: [rows][cols*bits/32]               */
    const uint16_t *s;     /* ORC_AFFINE: [rows][cols/group] fp16 scales     */
    const uint16_t *b;     /* ORC_AFFINE: [rows][cols/group] fp16 biases     */
    const uint16_t *f16;   /* ORC_F16:    [rows][cols]                       */
} orc_mat;

/* One weight, decoded exactly (the product n*s is exact in double). */
double orc_weight(const orc_mat *m, int o, int k);
/* Whole matrix, decoded into w[rows*cols] (row-major). */
void   orc_dequant(const orc_mat *m, double *w);
/* y[o] = sum_k W[o][k] * x[k]. */
void   orc_gemv(const orc_mat *m, const double *x, double *y);

/* Threads for the row loops of orc_gemv and orc_head_logits (default 1; the
 * library is built with OpenMP where the compiler has it).  Each row is one
 * thread's ascending-order sum: the results do not depend on n. */
void   orc_set_threads(int n);
int    orc_openmp(void);                /* 1 when built with OpenMP */

/* ---- recovery LoRA:  y += (alpha/r) * B (A x)  ---------------------------
 * A fp16 [r][in], B fp16 [out][r]; r == 0 means no adapter.                 */
typedef struct {
    int r;
    double scale;          /* alpha / r                                      */
    const uint16_t *A;
    const uint16_t *B;
} orc_lora;

void orc_lora_apply(const orc_lora *l, int in, int out, const double *x,
                    double *y);

/* ---- activations --------------------------------------------------------*/
double orc_silu(double g);        /* g / (1 + exp(-g))                       */
double orc_gelu_erf(double a);    /* a/2 * (1 + erf(a / sqrt 2))             */

/* ---- one expert:  h = silu(W_g x) * (W_u x),  y = W_d h  -----------------
 * gate, up: [F][d]; down: [d][F].  Each projection may carry a LoRA.
 * round_h_bf16: round h to bfloat16 (RNE) before the down projection
 * (batched path, bf16 activations).                                          */
typedef struct {
    orc_mat gate, up, down;
    orc_lora lg, lu, ld;
} orc_expert;

void orc_expert_forward(const orc_expert *ex, const double *x,
                        int round_h_bf16, double *h /* [F] or NULL */,
                        double *y /* [d] */);

/* ---- expert FFN over T tokens --------------------------------------------
 * experts[E] routed experts, shared (may be NULL).  x [T][d]; idx [T][K].
 * y_slots [T][K + (shared != NULL)][d]: slot k < K is expert idx[t][k], the
 * last slot (if any) is the shared expert.                                    */
void orc_expert_ffn(const orc_expert *experts, int E, const orc_expert *shared,
                    int d, const double *x, const int32_t *idx, int T, int K,
                    int round_h_bf16, double *y_slots);

/* ---- prerouter head ------------------------------------------------------
 * Features f = [x ; khot(cur) ; khot(prev)], width d + 2E.
 *   a = fc1 f + b1,   z = fc2 gelu_erf(a) + b2 + l f + bl
 * fc1 is stored as its first d columns (fc1x, [H][d]) plus its last 2E
 * columns transposed (fc1_tab, fp16 [2E][H]); l likewise (lx [E][d],
 * l_tab fp16 [2E][E]).  H == 0 means no fc1/fc2 branch: z = l f + bl (a plain
 * router).  Biases are fp16 and may be NULL (zero).  The oracle assembles the
 * whole fc1 / l rows and multiplies the dense feature vector; it never takes
 * a shortcut through the one-hot structure.                                  */
typedef struct {
    int d, E, H;
    orc_mat fc1x;                 /* [H][d]                                 */
    const uint16_t *fc1_tab;      /* [2E][H]                                */
    const uint16_t *b1;           /* [H]                                    */
    orc_mat fc2;                  /* [E][H]                                 */
    const uint16_t *b2;           /* [E]                                    */
    orc_mat lx;                   /* [E][d]                                 */
    const uint16_t *l_tab;        /* [2E][E]                                */
    const uint16_t *bl;           /* [E]                                    */
} orc_head;

/* Builds the dense feature vector f [d+2E] (cur/prev may be NULL = zero). */
void orc_head_features(int d, int E, const double *x, const int32_t *cur,
                       const int32_t *prev, int K, double *f);
void orc_head_logits(const orc_head *hd, const double *x, const int32_t *cur,
                     const int32_t *prev, int K, double *z /* [E] */);

/* ---- top-K and combine weights -------------------------------------------
 * Sort all E logits by (value descending, index ascending); keep the first
 * K.  w_k = exp(z_k - z_max) / sum_{j in top-K} exp(z_j - z_max).
 * margin = z_(K) - z_(K+1)  (+infinity when K == E).                         */
void orc_topk(const double *z, int E, int K, int32_t *idx, double *w,
              double *margin);
/* Weights at a given index set (used when the route is taken from outside). */
void orc_route_weights(const double *z, const int32_t *idx, int K, double *w);

/* ---- combine + residual ----------------------------------------------------
 * out = residual + sum_k w_k y_k (+ y_shared).  If x_next != NULL:
 * x_next = out / sqrt(mean(out^2) + 1e-6).                                    */
void orc_combine(const double *y_slots, const double *w, int K, int has_shared,
                 int d, const double *residual, double *out, double *x_next);

/* ---- a decode stack of L layers (driver semantics) ------------------------
 * Layer N holds experts [E], an optional shared expert and a router
 * (a head with H == 0).  Heads exist for N = 0 .. L-2; head N predicts layer
 * N+1's route for the next token.  With L == 1 the single head predicts the
 * layer's own route for the next token.
 *
 * One step at token t (stream is the residual stream, x_0 = input):
 *   layer 0 routes with its own router on x_0 (every step);
 *   layer N >= 1 uses the route head N-1 predicted at t-1, or, at t == 0
 *   (no prediction yet), its own router on x_N;
 *   y = experts(x_N); out_N = stream_N + combine; x_{N+1} = rms(out_N);
 *   head N runs on x_N with cur = layer N's route at t and prev = layer N's
 *   route at t-1 (none at t == 0), and its top-K becomes the route used at
 *   t+1 (by layer N+1, or by layer 0 itself when L == 1 and use_head_l0).  */
typedef struct {
    const orc_expert *experts;    /* [E]                                    */
    const orc_expert *shared;     /* NULL: none                             */
    orc_head router;              /* H == 0                                 */
    orc_head head;                /* predicts the next layer; unused for L-1 */
} orc_layer;

typedef struct {
    int L, d, E, K;
    const orc_layer *layers;
    int single_layer_self_predict;  /* L == 1: the head predicts layer 0 */
} orc_stack;

/* Route state carried from step to step (caller-allocated). */
typedef struct {
    int32_t *pred_idx;    /* [L][K]  route predicted for the next step      */
    double  *pred_z;      /* [L][E]  logits that prediction came from       */
    double  *pred_margin; /* [L]                                            */
    int32_t *prev_idx;    /* [L][K]  route each layer used at the last step */
    int      t;           /* steps taken so far                             */
} orc_stack_state;

/* One decode step.  If ext_idx != NULL it holds, per layer, the route some
 * other implementation used at this step; wherever the oracle's own route
 * was chosen with margin <= tie_margin, the oracle adopts ext_idx[N] instead
 * (teacher forcing at near-ties) and recomputes the weights from its own
 * logits at those indices.  used_* report, per layer, the route the oracle
 * used, its weights, the margin of the logits it came from and whether it
 * was adopted from ext_idx.                                                  */
void orc_stack_step(const orc_stack *st, orc_stack_state *state,
                    const double *x0,
                    const int32_t *ext_idx, double tie_margin,
                    double *out_last    /* [d] final residual stream      */,
                    int32_t *used_idx   /* [L][K] or NULL                 */,
                    double *used_w      /* [L][K] or NULL                 */,
                    double *used_margin /* [L] or NULL                    */,
                    uint8_t *forced     /* [L] or NULL                    */);

/* ---- merging a LoRA delta into the quantised weights ---------------------
 * The alternative to the unfused adapter: W' = requantise(W + (alpha/r) B A),
 * group by group, in the same affine form (the pages run the adapter unfused
 * because merging and requantising keeps only a small part of its delta:
 * "Ejecucion del adaptador no fusionado", xyznot.com/es/paper/2609.18063).
 *
 * orc_merge_weights: the merged weights, from the definition, in fp64:
 *     w[o][k] = W[o][k] + scale * sum_{j<r} B[o][j] * A[j][k]   (j ascending)
 * orc_quant_codes: the codes of w under a given fp16 scale s and bias b per
 *     (row, group) -- the affine quantiser's code rule:
 *     q = s == 0 ? 0 : clamp(rint((w - b) / s), 0, 2^bits - 1)  (ties even)
 *     t_pre (nullable) receives (w - b) / s before rounding (0 where s == 0).
 * orc_requantise: the min/max affine quantiser applied to w, per (row, group):
 *     lo = min w, hi = max w, s = f16((hi - lo) / (2^bits - 1)), b = f16(lo)
 *     (RNE), then the codes as above.  s_pre / b_pre (nullable) receive
 *     (hi - lo) / (2^bits - 1) and lo before the fp16 rounding, t_pre the
 *     code values before rint -- so a caller can see which decisions lie
 *     near a rounding boundary.
 * orc_merge_lora = orc_merge_weights then orc_requantise.  m: ORC_AFFINE;
 * r == 0 requantises W itself.  Outputs in m's layout: q [rows][cols*bits/32],
 * s, b [rows][cols/group] fp16 bit patterns, s_pre/b_pre [rows][cols/group],
 * t_pre [rows][cols].                                                         */
void orc_merge_weights(const orc_mat *m, const orc_lora *l, double *w);
void orc_quant_codes(const double *w, int rows, int cols, int bits, int group,
                     const uint16_t *s, const uint16_t *b, uint32_t *q_out,
                     double *t_pre);
void orc_requantise(const double *w, int rows, int cols, int bits, int group,
                    uint32_t *q_out, uint16_t *s_out, uint16_t *b_out,
                    double *s_pre, double *b_pre, double *t_pre);
void orc_merge_lora(const orc_mat *m, const orc_lora *l, uint32_t *q_out,
                    uint16_t *s_out, uint16_t *b_out, double *s_pre,
                    double *b_pre, double *t_pre);

#ifdef __cplusplus
}
#endif
#endif
