/*
 * moe.h -- C ABI of the GB300 (sm_103a) decode MoE layer with routing
 * predicted a token ahead.
 *
 * One decode step of a fine-grained Mixture-of-Experts FFN layer is split into
 * four calls, in the order a decoder issues them:
 *
 *   moe_prerouter_head    head(x) = fc2(erf-GELU(fc1(f))) + l(f) on the
 *                         features f = [x ; K-hot(cur) ; K-hot(prev)] of width
 *                         d_model + 2E; predicts the next layer's routing.
 *                         Source: "La otra mitad del muro de la memoria:
 *                         Servir MoEs de 35B desde SSD con prediccion de
 *                         enrutamiento entrenada" (xyznot.com/es/paper/
 *                         2609.18063), section "Arquitectura del cabezal
 *                         Prerouter" (dim = d_model + 2E; head equation; l is
 *                         a linear path started from the next layer's router).
 *   moe_topk_route        top-K of the logits with softmax weights
 *                         renormalised over the K kept experts.  The same page,
 *                         "Ideas clave": the prediction is used as the real
 *                         routing (no fallback, no dropped tokens).
 *   moe_expert_ffn_int4   per selected expert (and the shared expert) the
 *                         group-quantised affine int4 / 2-bit gate/up GEMV with
 *                         SwiGLU, then the down GEMV, each with an optional
 *                         unfused LoRA delta y = W x + (alpha/r) B A x.
 *                         Sources: "Inferencia de LLM MoE en MacBook Pro:
 *                         Streaming de Expertos desde SSD con Metal"
 *                         (kerneldigest.dev), section "Arquitectura del
 *                         Sistema" (4-/2-bit dequant matvec, fused SwiGLU) and
 *                         its Metal fragment (w = nibble*scale + bias, taken as
 *                         fma(nibble, scale*x, bias*x)); the LoRA form is the
 *                         xyznot page, "Ejecucion del adaptador no fusionado".
 *   moe_combine_residual  out = residual + sum_k w_k y_k + y_shared, with an
 *                         optional RMS-normalised copy of out (kerneldigest
 *                         page, "Arquitectura del Sistema": fused expert
 *                         combine + residual, RMS normalisation).
 *
 * Whole decode steps over a stack of layers (every layer's calls above, with
 * all routes known at the start of the step): moe_decode_step (one persistent
 * kernel) and moe_decode_step_chain (two kernels per layer chained by
 * programmatic dependent launch; the faster of the two).  Around them:
 * moe_merge_lora (the adapter merged into the int4 weights and requantised,
 * the alternative the xyznot page argues against), moe_gather_experts (a
 * route's experts from a host-memory pool into HBM slots, for an expert tier
 * outside HBM), packing, sizes and test hooks.
 *
 * Conventions shared by every call
 *  - Memory: every pointer argument is a DEVICE pointer unless stated
 *    otherwise; the caller owns all memory.  The library never allocates,
 *    frees or synchronises (the *_status readers synchronise the stream
 *    they are given).  Scratch memory comes from a caller-provided workspace
 *    whose size the matching *_workspace_bytes() call returns -- except for
 *    moe_expert_ffn_int4_noalloc, whose scratch is one static 4 MiB device
 *    array that every GPU loading the library holds until exit, shared by
 *    all calls on that device.
 *  - Alignment: device pointers must be 16-byte aligned; expert pools and
 *    packed matrices 256-byte aligned.
 *  - Streams: every call only enqueues work on `stream` (asynchronous).
 *    Descriptors are read during the call and not retained.
 *  - Errors: calls return a moe_status.  Arguments are validated before any
 *    work is enqueued; a rejected call enqueues nothing.  moe_last_error()
 *    returns a human-readable detail of the last failure on the calling host
 *    thread.  Launch failures are reported as MOE_ECUDA.
 *  - Determinism: no floating-point atomics; reductions run in a fixed order,
 *    so results are bitwise reproducible run to run.
 *
 * Packed weight format ("records").  A weight matrix [rows][cols] of affine
 * group-quantised weights is stored as `rows` records of
 * moe_record_bytes(cols, bits) bytes each: first the row's packed codes
 * (cols*bits/8 bytes, uint32 words little-endian, element j of a word at bits
 * [bits*j, bits*j+bits)), then one {fp16 scale, fp16 bias} pair per group of
 * 64 columns, then zero padding to a multiple of 16 bytes.  Decoded weight:
 * w = code*scale + bias.
 *
 * Expert blob.  One expert is one contiguous blob of
 * moe_pool_expert_bytes(d, F, bits, 64) bytes: a gate/up section of 2F
 * records of d columns (record 2f is gate row f, record 2f+1 is up row f),
 * then a down section of d records of F columns; each section starts on a
 * 256-byte boundary.  An expert pool is E blobs, expert_stride bytes apart.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
typedef enum {
    MOE_OK = 0,
    MOE_EINVAL = 1,         /* an argument is out of range, null or misaligned */
    MOE_EUNSUPPORTED = 2,   /* valid, but a shape this build has no kernel for */
    MOE_ECUDA = 3,          /* a CUDA runtime call or kernel launch failed     */
    MOE_ETIMEOUT = 4,       /* a bounded device-side wait expired              */
    MOE_ENOSPACE = 5        /* the workspace is smaller than required          */
} moe_status;

/* Static string naming a status code ("MOE_OK", ...). */
const char *moe_status_string(int status);
/* Detail of the last failing call on this host thread ("" if none).  The
 * string stays valid until the next failing call on the same thread. */
const char *moe_last_error(void);

/* ---------------------------------------------------------------- enums */
enum {
    MOE_DTYPE_F32 = 0,      /* activations in fp32                             */
    MOE_DTYPE_BF16 = 1      /* activations in bfloat16                         */
};

enum {
    MOE_PREC_AFFINE4 = 4,   /* affine int4, group 64, packed records           */
    MOE_PREC_FP16 = 16      /* plain fp16 row-major [rows][cols]               */
};

/* ---------------------------------------------------------------- sizes */
/* Bytes of one packed record (one row of `cols` weights); 0 if invalid. */
size_t moe_record_bytes(int cols, int bits);
/* Bytes of a packed matrix: rows * moe_record_bytes(cols, bits). */
size_t moe_packed_matrix_bytes(int rows, int cols, int bits);
/* Bytes of one expert blob (gate/up and down sections, see above); 0 if the
 * shape is invalid (bits not in {2,4}, group != 64, d or F not multiples of
 * 64).  At d=4096, F=1024, bits=4 this is 7,077,888 bytes (6.75 MiB). */
size_t moe_pool_expert_bytes(int d, int F, int bits, int group);

/* ---------------------------------------------------------------- packing */
/* Packs one logical matrix into records.  q: uint32 [rows][cols*bits/32],
 * s, b: fp16 bit patterns [rows][cols/64]; out: moe_packed_matrix_bytes()
 * bytes.  All device pointers; enqueued on `stream`. */
int moe_pack_matrix(const uint32_t *q, const uint16_t *s, const uint16_t *b,
                    int rows, int cols, int bits, void *out,
                    cudaStream_t stream);

/* Packs E experts into a pool.  Logical inputs, contiguous per expert:
 * gate_q/up_q [E][F][d*bits/32], gate_s/b, up_s/b [E][F][d/64],
 * down_q [E][d][F*bits/32], down_s/b [E][d][F/64].  pool: E blobs,
 * expert_stride bytes apart (>= moe_pool_expert_bytes, multiple of 256). */
int moe_pack_experts(int d, int F, int E, int bits,
                     const uint32_t *gate_q, const uint16_t *gate_s,
                     const uint16_t *gate_b, const uint32_t *up_q,
                     const uint16_t *up_s, const uint16_t *up_b,
                     const uint32_t *down_q, const uint16_t *down_s,
                     const uint16_t *down_b, void *pool, size_t expert_stride,
                     cudaStream_t stream);

/* Test hook: decodes matrix `which` (0 gate [F][d], 1 up [F][d], 2 down
 * [d][F]) of one expert blob into fp32 out[rows][cols] as
 * fmaf(code, scale, bias), the same decode the GEMV kernels use. */
int moe_debug_dequant(const void *blob, int d, int F, int bits, int which,
                      float *out, cudaStream_t stream);

/* Test hook, process-wide: the bound of every device-side wait of the
 * batched tensor-core engine (moe_expert_ffn_int4 and moe_prerouter_head with
 * T > 1 bf16 tokens), timeout_ns (0 = 1 second), read at each launch.
 * stall != 0 adds to every later launch one wait for bytes that no copy
 * sends: it runs out after timeout_ns, MOE_ETIMEOUT lands in the call's
 * status word (ws word 0) and the launch returns with invalid outputs.
 * moe_debug_batched_waits(0, 0) restores the defaults. */
int moe_debug_batched_waits(unsigned long long timeout_ns, int stall);

/* Test and measurement hook, process-wide: which engine runs the batched
 * path's grouped GEMMs.  0 (default) or 1: the register engine (mma.sync,
 * fp32 accumulators in registers); 2: the tensor-memory engine (tcgen05.mma,
 * fp32 accumulators in TMEM) when its shared memory fits and the GEMM's
 * columns are a multiple of 128, else the register engine.  Both give
 * results within the same tolerance of the exact sums (the per-group affine
 * terms are applied in fp32 to exact bf16 partial sums either way); the
 * register engine is the faster of the two on GB300 at every batch size
 * measured (8 to 4096 tokens), hence the default. */
int moe_debug_batched_engine(int mode);

/* Profiling hook, process-wide: a device buffer of 64 * 16 u64 that CTA 0 of
 * the next tensor-memory engine launch fills with %globaltimer stamps of
 * its first 64 chunks (per chunk: producer issue, converters see / release
 * groups 0-3, MMA warp sees the stage / issues groups 0-3, epilogue sees
 * accumulators 0-3, epilogue releases the stage); NULL turns it off.  The
 * hook is cleared by that launch. */
int moe_debug_batched_trace(unsigned long long *buf);

/* ---------------------------------------------------------------- head */
typedef struct {
    int d;                    /* d_model                                      */
    int E;                    /* experts of the predicted layer               */
    int H;                    /* head hidden size; 0 = plain router l(x) only  */
    int prec;                 /* MOE_PREC_AFFINE4 or MOE_PREC_FP16 for the
                                 dense matrices fc1x, fc2, lx                 */
    const void *fc1x;         /* [H][d]  fc1 columns that multiply x          */
    const uint16_t *fc1_tab;  /* [2E][H] fp16: fc1 columns of the two K-hot
                                 vectors, transposed (row c = column d+c)     */
    const uint16_t *b1;       /* [H] fp16, or NULL (zero)                     */
    const void *fc2;          /* [E][H]                                       */
    const uint16_t *b2;       /* [E] fp16, or NULL                            */
    const void *lx;           /* [E][d]  l columns that multiply x            */
    const uint16_t *l_tab;    /* [2E][E] fp16, or NULL (zero)                 */
    const uint16_t *bl;       /* [E] fp16, or NULL                            */
} moe_head_desc;

size_t moe_prerouter_head_workspace_bytes(const moe_head_desc *hd, int T);

/* Logits of the prerouter head for T tokens.
 * x: [T][d] in x_dtype.  cur_idx / prev_idx: int32 [T][K] expert indices in
 * [0, E) of the current / previous token's route (the K-hot vectors); either
 * may be NULL (an all-zero vector).  logits: fp32 [T][E].
 *   a = fc1x x + sum_{c in cur} fc1_tab[c] + sum_{c in prev} fc1_tab[E+c] + b1
 *   logits = fc2 gelu_erf(a) + b2 + lx x + sum l_tab rows (same rule) + bl
 * With H == 0 only the l branch is computed (a plain linear router).
 * T > 1 tokens in bf16 with an int4 head run fc1 + l and fc2 as tensor-core
 * GEMMs over all tokens (fc2's input g carried as bf16 hi + lo parts, so the
 * logits keep fp32 accuracy); ws word 0 then holds the status of their
 * bounded device-side waits (MOE_OK or MOE_ETIMEOUT) once the stream
 * completes. */
int moe_prerouter_head(const moe_head_desc *hd, const void *x, int x_dtype,
                       const int32_t *cur_idx, const int32_t *prev_idx, int K,
                       int T, float *logits, void *ws, size_t ws_bytes,
                       cudaStream_t stream);

/* ---------------------------------------------------------------- route */
/* Top-K of logits [T][E] ordered by (value descending, index ascending).
 * idx: int32 [T][K]; w: fp32 [T][K], w_k = exp(z_k - z_1) / sum_j exp(z_j - z_1)
 * over the kept K; margin: fp32 [T] (may be NULL), z_(K) - z_(K+1) (+inf if
 * K == E).  1 <= K <= 16, K <= E <= 1024. */
int moe_topk_route(const float *logits, int T, int E, int K, int32_t *idx,
                   float *w, float *margin, cudaStream_t stream);

/* ---------------------------------------------------------------- experts */
typedef struct {
    int r;                    /* rank; 0 = no adapter                         */
    float scale;              /* alpha / r                                    */
    const uint16_t *A;        /* fp16 [r][in]  (expert e: A + e*a_stride)     */
    const uint16_t *B;        /* fp16 [out][r] (expert e: B + e*b_stride)     */
    size_t a_stride;          /* elements between experts' A (routed only)    */
    size_t b_stride;          /* elements between experts' B (routed only)    */
} moe_lora_desc;

typedef struct {
    int d;                    /* d_model (multiple of 64)                     */
    int F;                    /* expert SwiGLU hidden size (multiple of 64)   */
    int E;                    /* routed experts in the pool                   */
    int bits;                 /* 4 or 2                                       */
    const void *pool;         /* E expert blobs                               */
    size_t expert_stride;     /* bytes between blobs (multiple of 256)        */
    const void *shared;       /* blob of the always-on shared expert, or NULL */
    moe_lora_desc lora[3];    /* routed experts: gate, up, down               */
    moe_lora_desc shared_lora[3]; /* shared expert: gate, up, down            */
} moe_experts_desc;

size_t moe_expert_ffn_workspace_bytes(const moe_experts_desc *ed, int T, int K);

/* Expert outputs for T tokens routed to idx [T][K] (int32, in [0, E)).
 * x: [T][d] in x_dtype.  y_slots: fp32 [T][K + (shared != NULL)][d]; slot
 * k < K holds expert idx[t][k]'s output y = W_d h (+ LoRA), the last slot the
 * shared expert's.  h = silu(W_g x + LoRA) * (W_u x + LoRA) is kept in fp32
 * for x_dtype == MOE_DTYPE_F32 and rounded to bf16 for MOE_DTYPE_BF16.
 * An index outside [0, E) is never read: that slot's output is NaN.
 * T == 1, or fp32 x, is the decode path (per-token GEMVs).  T > 1 with bf16 x
 * is the batched path: the (token, slot) entries are sorted by expert (a
 * stable counting sort, "tokens sorted/grouped by expert" of the batched
 * configuration in xyznot.com/es/paper/2609.18063's workload list) and each
 * expert's tokens run as grouped tensor-core GEMMs that read its weights
 * once.  Results are deterministic.  The batched path's device-side waits
 * are bounded: after the stream completes, int32 word 0 of ws holds MOE_OK,
 * or MOE_ETIMEOUT if one expired (the outputs are then invalid). */
int moe_expert_ffn_int4(const moe_experts_desc *ed, const void *x, int x_dtype,
                        const int32_t *idx, int T, int K, float *y_slots,
                        void *ws, size_t ws_bytes, cudaStream_t stream);

/* Bytes of the static device scratch behind moe_expert_ffn_int4_noalloc. */
#define MOE_FFN_STATIC_SCRATCH_BYTES ((size_t)4 << 20)

/* moe_expert_ffn_int4 without a workspace argument.  The pages have no
 * counterpart to this call; it exists for callers that are handed only their
 * input and output buffers and cannot allocate device memory or carve a
 * workspace -- for example a plugin or custom operator hosted by a framework
 * that owns the device allocator, or a fixed-budget real-time loop that
 * forbids allocation once it has started.
 *
 * Arguments and results are those of moe_expert_ffn_int4.  The scratch the
 * call needs comes from one fixed array of MOE_FFN_STATIC_SCRATCH_BYTES
 * (4 MiB) in the library's device memory, which every GPU that loads the
 * library holds until the process exits.  Calls whose scratch need
 * (moe_expert_ffn_workspace_bytes(ed, T, K)) exceeds it return MOE_ENOSPACE.
 * The call allocates and frees nothing.
 *
 * The first call on a device (with that device current) looks up the array's
 * device address (cudaGetSymbolAddress) and caches it; make that first call
 * before any stream capture on the device.  All calls on a device share the
 * one array, which keeps the last call's contents: calls that may overlap on
 * the GPU (e.g. issued on different streams without ordering) race with each
 * other and must be serialised by the caller.  Each call clears the array's
 * status word (word 0) on `stream`; the rest needs no clearing between
 * calls.  Bad arguments get the same status as from moe_expert_ffn_int4.
 *
 * The batched path's bounded device-side waits record MOE_ETIMEOUT in that
 * status word (the outputs are then invalid); the caller has no workspace to
 * read it from, so it reads it with moe_expert_ffn_noalloc_status. */
int moe_expert_ffn_int4_noalloc(const moe_experts_desc *ed, const void *x,
                                int x_dtype, const int32_t *idx, int T, int K,
                                float *y_slots, cudaStream_t stream);

/* Waits for `stream` and stores in *status (host) the status word of the last
 * moe_expert_ffn_int4_noalloc call on the current device that `stream` has
 * finished: MOE_OK, or MOE_ETIMEOUT if one of its batched-path waits expired.
 * Synchronises `stream`. */
int moe_expert_ffn_noalloc_status(int *status, cudaStream_t stream);

/* ---------------------------------------------------------------- combine */
/* out[t] = residual[t] + sum_k w[t][k] * y_slots[t][k] (+ y_slots[t][K] if
 * has_shared), all fp32, y_slots [T][K + has_shared][d].  If x_next is not
 * NULL it receives out[t] / sqrt(mean(out[t]^2) + 1e-6).  out may alias
 * residual. */
int moe_combine_residual(const float *y_slots, const float *w, int T, int K,
                         int has_shared, int d, const float *residual,
                         float *out, float *x_next, cudaStream_t stream);

/* ---------------------------------------------------------------- merge */
/* Merges a LoRA delta into packed records: W' = requantise(W + scale B A),
 * group by group (64 columns) in the same affine form -- the merged
 * alternative to the unfused adapter (xyznot.com/es/paper/2609.18063,
 * "Ejecucion del adaptador no fusionado": the adapter stays unfused because
 * requantising keeps little of its delta; this call measures how little).
 * src: `rows` records of moe_record_bytes(cols, bits) bytes, src_stride
 * bytes apart (e.g. 2 * record for the gate or up rows of an expert blob);
 * A fp16 [r][cols], B fp16 [rows][r] (r == 0: W is only requantised);
 * dst: the merged records, dst_stride apart -- dst == src with equal
 * strides merges in place (any other overlap is undefined).  Arithmetic,
 * binary32 with every operation rounded to nearest even: per row o, group,
 * column k: d_k = sum_j B[o][j] A[j][k] (fma chain, j ascending),
 * w_k = fma(scale, d_k, fma(code_k, s, b)); s' = f16((max w - min w) /
 * (2^bits - 1)), b' = f16(min w); code'_k = s' == 0 ? 0 :
 * clamp(rint((w_k - b') / s'), 0, 2^bits - 1).  Records and strides 16-byte
 * aligned, A 4-byte aligned; all device memory; enqueued on `stream`.
 * rows == 0 is a no-op. */
int moe_merge_lora(const void *src, size_t src_stride, int rows, int cols, int bits,
                   const uint16_t *A, const uint16_t *B, int r, float scale,
                   void *dst, size_t dst_stride, cudaStream_t stream);

/* ---------------------------------------------------------------- tiers */
/* Copies the blobs of experts idx[0..n-1] (a device array: a route) of a
 * pool of E experts, expert_stride bytes apart, into n slots slot_stride
 * bytes apart, and writes slot_idx[i] = i -- or n where idx[i] is outside
 * [0, E): that blob is not copied and an expert call reading slot_idx gives
 * NaN for it, as it would for idx.  The pool may live outside HBM: pinned
 * host memory is read directly by the GPU (over NVLink-C2C on a Grace
 * machine), so the routed experts of a layer can be brought into HBM a token
 * ahead from the predicted route without a host round trip (the predicted
 * route is the routing: xyznot.com/es/paper/2609.18063, "Ideas clave").
 * blob_bytes, strides: multiples of 16 (blob_bytes <= both strides); pool and
 * slots 16-byte aligned; n <= 17; enqueued on `stream`. */
int moe_gather_experts(const void *pool, size_t expert_stride, int E, const int32_t *idx,
                       int n, size_t blob_bytes, void *slots, size_t slot_stride,
                       int32_t *slot_idx, cudaStream_t stream);

/* An HBM cache of C expert slots in front of a pool (host or device memory)
 * of one layer -- the expert cache of the xyznot page's streaming design
 * ("Ideas clave": the predicted route is known a token ahead), kept on the
 * GPU.  cache: C slots, slot_stride bytes apart (device); tags [C] (device):
 * the expert in each slot, -1 for none (the caller sets every tag to -1 once);
 * ages [C] (device): the step each slot was last used at; clock (device, one
 * int32): the cache's step counter, advanced by one by every call (on the
 * device, so calls replayed from a captured graph age the slots too).  For
 * the route idx[0..n-1] (device): an expert already in a slot is a hit;
 * any other valid one takes the least recently used slot this route does not
 * use (empty slots first, then the oldest step, then the lowest index) and its
 * blob is copied there from pool.  slot_idx[i] (device) receives idx[i]'s
 * slot, or C for an index outside [0, E) (not copied); this is the slot map
 * moe_decode_step_chain reads (moe_stack_desc.slot_map).  plan [n] (device):
 * scratch between the call's two launches (the decision, one warp; the
 * copies).  stats (device int32 [2], or NULL): += distinct hits, += misses.
 * 1 <= n <= 17, n <= C <= 1024; strides and blob 16-byte multiples. */
int moe_cache_experts(const void *pool, size_t expert_stride, int E, const int32_t *idx,
                      int n, size_t blob_bytes, void *cache, size_t slot_stride, int C,
                      int32_t *tags, int32_t *ages, int32_t *clock, int32_t *slot_idx,
                      int32_t *plan, int32_t *stats, cudaStream_t stream);

/* ---------------------------------------------------------------- stack */
/* A decode stack: depth layers per step, layer N using resident layer
 * N % n_layers (all of one shape).  Layer 0 routes with its own router every
 * step (unless self_predict); layer N >= 1 uses the route head N-1 predicted
 * at the previous step; head N (N < depth-1) runs on layer N's input with the
 * K-hot routes of layer N at this and the previous step and predicts layer
 * N+1's route for the next step.  self_predict (depth 1 only): the single
 * layer's head predicts its own next route and the layer routes with it. */
typedef struct {
    const moe_experts_desc *experts;  /* [n_layers]                            */
    const moe_head_desc *routers;     /* [n_layers] H == 0 heads (l = router)  */
    const moe_head_desc *heads;       /* [n_layers] int4 heads, or NULL when no
                                         head runs (depth 1, no self_predict)  */
    int n_layers;                     /* resident layers (<= 48)               */
    int depth;                        /* layers per decode step (<= 48)        */
    int K;                            /* experts per token (<= 16)             */
    int self_predict;
    unsigned long long timeout_ns;    /* bound of every device-side wait;
                                         0 = 1 second                          */
    int debug_unset_wait;             /* test hook: 1 makes the kernel wait on
                                         a flag nothing sets (-> MOE_ETIMEOUT) */
    unsigned long long *debug_trace;  /* profiling hook: NULL, or a device
                                         buffer of %globaltimer stamps.
                                         moe_decode_step: n_SM * depth * 16
                                         u64, per CTA and layer at phase
                                         boundaries.  moe_decode_step_chain:
                                         2048 + 65536 u64, 8 stamps of CTA 0
                                         per launch, then every CTA's end
                                         (256 per launch)                     */
    unsigned inflight_bytes;          /* tuning: weight-copy bytes in flight
                                         per SM (0 = 32 KiB; at least 16 KiB) */
    const int32_t *slot_map;          /* moe_decode_step_chain only (NULL for
                                         moe_decode_step): NULL, or a device
                                         array [depth][K] -- layer N's route
                                         position k then reads the routed
                                         expert blob at experts[N % n_layers]
                                         .pool + slot_map[N * K + k] *
                                         expert_stride instead of the one its
                                         route index names (an expert cache or
                                         staging area the caller filled, e.g.
                                         with moe_gather_experts); the route
                                         indices still feed the heads and the
                                         routed adapters.  Not used for layer
                                         0 when it routes itself in the step */
    void *const *layer_ready;         /* moe_decode_step_chain only: NULL, or
                                         [depth] cudaEvent_t (NULL entries
                                         allowed); the step's stream waits on
                                         layer_ready[N] before layer N's first
                                         kernel (e.g. the copy of its experts
                                         on another stream) */
    int free_sms;                     /* moe_decode_step_chain only: SMs the
                                         step leaves free (its kernels run one
                                         CTA on each of the others; 0 = every
                                         SM), e.g. for copy kernels running on
                                         another stream beside it; the
                                         workspace size depends on it */
} moe_stack_desc;

/* Workspace bytes of moe_decode_step; 0 if the descriptor is invalid. */
size_t moe_decode_step_workspace_bytes(const moe_stack_desc *sd);

/* One decode step (token t >= 1) of the whole stack in one persistent kernel
 * (one CTA per SM, cooperative launch): per layer the expert FFN, combine +
 * residual + RMS, the prerouter head and its top-K -- the same operations as
 * the four calls above, fused across layers.
 * x0: fp32 [d] layer-0 input (also its residual); out: fp32 [d] final
 * residual stream.  Route state (caller-owned, device): route_idx int32
 * [3][depth][K], route_w fp32 [3][depth][K], route_margin fp32 [3][depth],
 * rotating by t % 3: set t % 3 holds the routes used at t (written by the
 * previous step, or by this one for layer 0's own route), set (t+1) % 3
 * receives the predictions for t+1, set (t+2) % 3 holds the routes of t-1 (the
 * "previous token" K-hot input of the heads).  Step 0 (every layer routing
 * with its own router) is run with the per-call functions.
 * ws: moe_decode_step_workspace_bytes() bytes, 256-byte aligned, ZEROED before
 * the first call (never again, unless a call reports an error).  Device-side
 * waits are bounded; a step that timed out or found a bad route records the
 * status in the workspace (read it with moe_decode_step_status) and every
 * later step on that workspace returns immediately until it is zeroed. */
int moe_decode_step(const moe_stack_desc *sd, const float *x0, float *out,
                    int32_t *route_idx, float *route_w, float *route_margin,
                    int t, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Reads the status word of a decode-step workspace into *status (host):
 * MOE_OK, MOE_ETIMEOUT (a bounded wait expired) or MOE_EINVAL (a route index
 * out of range).  Synchronises `stream`. */
int moe_decode_step_status(const void *ws, int *status, cudaStream_t stream);

/* The same decode step as moe_decode_step (same arguments, routes, results
 * and step-0 rule), run as two kernels per layer chained by programmatic
 * dependent launch instead of one persistent kernel: kernel A takes an even
 * share of every layer's gate/up row pairs and head rows per SM (h,
 * gelu(fc1 f), l f), kernel B a share of the output rows (the down GEMV of
 * every slot, combine + residual, down LoRA), of the head's fc2 logits and of
 * the next layer's gate/up LoRA partials.  Each kernel copies its weights into
 * shared memory before it waits for the one before (the step's routes are
 * known when it starts).  The heads' top-K (the routes of t+1) run in one
 * launch at the end of the step.  No kernel waits on another's CTAs: the only
 * device-side wait is a CTA's on its own copies (bounded by sd->timeout_ns,
 * 0 = 1 second; on expiry MOE_ETIMEOUT lands in the status word and the CTA
 * returns: the step's outputs are then invalid).  sd->debug_unset_wait = 1
 * makes CTA 0 of layer 0's first kernel wait, once its own copies have
 * landed, for bytes no copy sends: a test of that path.
 * ws: moe_decode_step_chain_workspace_bytes() bytes, 256-byte aligned (no
 * clearing needed); its status reads with moe_decode_step_status.  The step
 * enqueues 2 * depth launches, + 2 for layer 0's own router and its top-K
 * (+ 1 for its router alone when only the shared expert's gate/up adapters
 * need layer 0's partials), + 1 for the heads' top-K; under stream capture
 * they form one graph. */
size_t moe_decode_step_chain_workspace_bytes(const moe_stack_desc *sd);

/* How the two per-layer kernels of moe_decode_step_chain sit on an SM of the
 * current device for the stack sd (host struct, filled by the call below). */
typedef struct {
    size_t smem_a, smem_b;       /* dynamic shared memory per CTA of A and B  */
    int threads;                 /* threads per CTA                           */
    int regs_a, regs_b;          /* registers per thread                      */
    int local_bytes_a, local_bytes_b; /* local memory per thread (spills)     */
    int ctas_a, ctas_b;          /* CTAs of A (of B) an SM holds on its own   */
    int coresident;              /* 1: an SM holds a CTA of A beside one of B
                                    (shared memory incl. the per-CTA
                                    reservation, and registers) -- so that
                                    A(N+1) copies its weights while B(N) runs */
} moe_chain_info;

/* Fills *info for sd on the current device (the occupancy API and the
 * kernels' attributes); MOE_EUNSUPPORTED when a kernel does not fit an SM at
 * all (moe_decode_step_chain then fails the same way).  The step runs when
 * coresident is 0, with each kernel's copies starting only when the previous
 * one's CTAs have left. */
int moe_decode_step_chain_info(const moe_stack_desc *sd, moe_chain_info *info);

/* Which form moe_decode_step_chain takes (process-wide, read at each call):
 * variant 0 the library's choice (two kernels per layer), 1 two kernels per
 * layer, 2 one kernel per layer with a thread-block cluster of 16 CTAs per
 * expert slot and one for the head: CTA j of a slot takes gate/up row pairs
 * [F j/16, F (j+1)/16) and output rows [d j/16, d (j+1)/16), h is exchanged
 * inside the cluster through distributed shared memory, and each slot's
 * weighted output goes to a per-slot vector that the next layer sums onto
 * the residual (one global exchange per layer).  Two CTAs per SM: gate/up
 * rows are copied into shared memory, down rows read into registers.
 * Variant 2 returns MOE_EUNSUPPORTED from the step when a CTA's share of a
 * slot does not fit (shared memory, or F / (128 / bits) not dividing 32, or
 * more than 4 passes of a warp over its down rows, or F > 1024, or an
 * adapter rank above 16).  prefetch_l2: variant 2 prefetches its down rows
 * into L2 in its prologue.  Same arguments, routes and results as variant 1;
 * workspace from moe_decode_step_chain_workspace_bytes (sized for both).
 * MOE_EINVAL for another variant. */
int moe_decode_step_chain_variant(int variant, int prefetch_l2);

/* Graph cache of moe_decode_step_chain (process-wide).  A call's launches
 * depend only on the descriptor's values, the call's pointers, t mod 3, the
 * device and the variant, so a call not made under stream capture is
 * recorded once into a CUDA graph (on an internal stream, thread-local
 * capture mode) and later calls with the same key launch that graph on the
 * caller's stream: one host launch per step instead of about two per layer.
 * Calls with layer_ready events, debug_unset_wait or debug_trace are never
 * cached.  max_graphs: graphs kept (least recently used dropped first;
 * default 16); 0 disables the cache.  Every call empties the cache.
 * The graphs belong to the device's current context: call
 * moe_decode_step_chain_cache(0) before resetting the device (a graph of a
 * destroyed context fails to launch with MOE_ECUDA).
 * MOE_EINVAL outside 0 .. 1024. */
int moe_decode_step_chain_cache(int max_graphs);
int moe_decode_step_chain(const moe_stack_desc *sd, const float *x0, float *out,
                          int32_t *route_idx, float *route_w, float *route_margin,
                          int t, void *ws, size_t ws_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
