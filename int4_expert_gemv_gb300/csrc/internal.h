// internal.h -- launcher interfaces between the C ABI (abi.cu) and the kernel
// translation units.  Every launcher assumes validated arguments and only
// enqueues work; it returns a moe_status.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {

struct LoraDev {
    int r;
    float scale;
    const uint16_t *A;
    const uint16_t *B;
    size_t a_stride, b_stride;
};

struct FfnParams {
    const uint8_t *pool;
    size_t stride;
    const uint8_t *shared;
    const int32_t *idx;          // [T][K]
    int T, K, slots, d, F, E, bits;
    const void *x;               // [T][d]
    int x_dtype;
    int round_h_bf16;
    float *h;                    // workspace [T*slots][F]
    float *v;                    // workspace [T*slots][3][kMaxLoraRank]
    float *y;                    // [T*slots][d]
    LoraDev lora[3];
    LoraDev shared_lora[3];
    BlobLayout L;
    int any_gu_lora;             // some slot carries a gate or up adapter
    // grouped (T > 1, bf16) path
    int32_t *counts;             // workspace [E+1]: entries per expert, then invalid ones
    int32_t *offsets;            // workspace [E+2]
    int32_t *perm;               // workspace [T*K] (token*K + k), by expert, in token order
    const __nv_bfloat16 *xb;     // = x, [T][d]
    __nv_bfloat16 *xg;           // workspace [T*K + T][d]: x rows in sorted order (shared: T*K + t)
    float *xsum;                 // workspace [T*K + T][ld]: sum of xg per group
    __nv_bfloat16 *h16;          // workspace [T*K + T][F]: h at sorted positions (shared: T*K + t)
    float *hsum;                 // workspace [T*K + T][ld]: sum of h per group
    float *vd;                   // workspace [T*K + T][kMaxLoraRank]: A_d h
    int32_t *item_off;           // workspace [2][E+2]: work-item offsets per group (gate/up, down)
    int32_t *err;                // workspace word 0: status of the device-side waits
};

struct HeadParams {
    int d, E, H, K, T, prec;
    const uint8_t *fc1x;
    const uint16_t *fc1_tab, *b1;
    const uint8_t *fc2;
    const uint16_t *b2;
    const uint8_t *lx;
    const uint16_t *l_tab, *bl;
    const void *x;
    int x_dtype;
    const int32_t *cur, *prev;
    float *g;                    // workspace [T][H]
    float *zl;                   // workspace [T][E]
    float *xsum;                 // workspace [T][ld]: sum of x per group (batched path)
    __nv_bfloat16 *gg;           // workspace [2T][H]: g split as bf16 hi (row 2t) + lo (row 2t+1)
    float *ggsum;                // workspace [2T][ld]: sum of gg per group
    int32_t *err;                // workspace word 0: status of the device-side waits
    float *logits;               // [T][E]
};

int launch_expert_ffn(const FfnParams &p, cudaStream_t st);
int launch_expert_ffn_grouped(const FfnParams &p, cudaStream_t st);
void lora_ax_kernel_launch(const FfnParams &p, cudaStream_t st);
int launch_prerouter_head(const HeadParams &p, cudaStream_t st);
int launch_topk(const float *logits, int T, int E, int K, int32_t *idx, float *w,
                float *margin, cudaStream_t st);
int launch_combine(const float *y, const float *w, int T, int K, int has_shared, int d,
                   const float *res, float *out, float *xn, cudaStream_t st);
int launch_pack_rows(const uint32_t *q, const uint16_t *s, const uint16_t *b, int rows,
                     int cols, int bits, int nmat, size_t src_q_stride,
                     size_t src_sb_stride, uint8_t *dst, size_t dst_mat_stride,
                     size_t first_record, size_t record_step, cudaStream_t st);
int launch_debug_dequant(const uint8_t *sec, size_t rec, size_t first_record,
                         size_t record_step, int rows, int cols, int bits, float *out,
                         cudaStream_t st);

int num_sms();

// Validation of a decode-stack descriptor shared by the decode-step paths.
int check_decode_stack(const moe_stack_desc *sd);

}  // namespace moe
