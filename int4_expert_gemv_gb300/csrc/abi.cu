// abi.cu -- the extern "C" boundary: argument validation, workspace carving,
// dispatch to the kernel launchers.  Nothing is enqueued unless every argument
// passed validation.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "internal.h"

namespace moe {

static thread_local char g_last_error[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return code;
}

int check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(MOE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    return MOE_OK;
}

int num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

static bool aligned(const void *p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

static bool shape_ok(int d, int F, int bits) {
    return d > 0 && F > 0 && d % kGroup == 0 && F % kGroup == 0 && (bits == 2 || bits == 4);
}

// Workspace carving for the expert FFN.  The LoRA partials, the histogram,
// the offsets, the permutation and the work-item offsets are common; the
// per-token path's h and the grouped path's {x in sorted order, its group
// sums, h (bf16), sum h, A_d h} share one region, since a call takes one
// path or the other.
struct FfnWs {
    size_t err, h, v, counts, offsets, perm, item_off, xg, xsum, h16, hsum, vd, total;
};

// Row stride (floats) of the per-group sums the batched kernels read through
// tensor maps: padded to 16 bytes.
static size_t gsum_ld(int cols) { return (size_t)((cols / kGroup + 3) / 4 * 4); }

static FfnWs ffn_ws(const moe_experts_desc *ed, int T, int K) {
    FfnWs w;
    const size_t slots = (size_t)K + (ed->shared ? 1 : 0);
    const size_t npos = (size_t)T * K + (ed->shared ? T : 0);
    size_t off = 0;
    w.err = off;
    off = 256;
    w.v = off;
    off = align_up(off + (size_t)T * slots * 3 * kMaxLoraRank * sizeof(float), 256);
    w.counts = off;
    off = align_up(off + (size_t)(ed->E + 1) * sizeof(int32_t), 256);
    w.offsets = off;
    off = align_up(off + (size_t)(ed->E + 2) * sizeof(int32_t), 256);
    w.perm = off;
    off = align_up(off + (size_t)T * K * sizeof(int32_t), 256);
    w.item_off = off;
    off = align_up(off + 2 * (size_t)(ed->E + 2) * sizeof(int32_t), 256);
    const size_t region = off;
    w.h = region;
    const size_t end_tok = align_up(region + (size_t)T * slots * ed->F * sizeof(float), 256);
    size_t g = region;
    w.xg = g;
    g = align_up(g + npos * ed->d * sizeof(uint16_t), 256);
    w.xsum = g;
    g = align_up(g + npos * gsum_ld(ed->d) * sizeof(float), 256);
    w.h16 = g;
    g = align_up(g + npos * ed->F * sizeof(uint16_t), 256);
    w.hsum = g;
    g = align_up(g + npos * gsum_ld(ed->F) * sizeof(float), 256);
    w.vd = g;
    g = align_up(g + npos * kMaxLoraRank * sizeof(float), 256);
    w.total = end_tok > g ? end_tok : g;
    return w;
}

static int check_lora(const moe_lora_desc &l, const char *name) {
    if (l.r < 0 || l.r > kMaxLoraRank)
        return fail(MOE_EINVAL, "%s: LoRA rank %d outside [0, %d]", name, l.r, kMaxLoraRank);
    if (l.r > 0 && (l.A == nullptr || l.B == nullptr))
        return fail(MOE_EINVAL, "%s: LoRA rank %d with a null A or B", name, l.r);
    return MOE_OK;
}

static int check_experts(const moe_experts_desc *ed) {
    if (ed == nullptr) return fail(MOE_EINVAL, "experts descriptor is NULL");
    if (!shape_ok(ed->d, ed->F, ed->bits))
        return fail(MOE_EINVAL, "experts: d=%d F=%d bits=%d (need d, F multiples of 64, bits 2 or 4)",
                    ed->d, ed->F, ed->bits);
    if (ed->E < 1) return fail(MOE_EINVAL, "experts: E=%d", ed->E);
    if (ed->pool == nullptr || !aligned(ed->pool, 256))
        return fail(MOE_EINVAL, "experts: pool is NULL or not 256-byte aligned");
    const size_t blob = blob_layout(ed->d, ed->F, ed->bits).bytes;
    if (ed->expert_stride < blob || ed->expert_stride % 256)
        return fail(MOE_EINVAL, "experts: expert_stride %zu (need >= %zu, multiple of 256)",
                    ed->expert_stride, blob);
    if (ed->shared && !aligned(ed->shared, 256))
        return fail(MOE_EINVAL, "experts: shared blob not 256-byte aligned");
    static const char *names[3] = {"gate", "up", "down"};
    for (int i = 0; i < 3; i++) {
        if (int rc = check_lora(ed->lora[i], names[i])) return rc;
        if (int rc = check_lora(ed->shared_lora[i], names[i])) return rc;
    }
    return MOE_OK;
}

static LoraDev lora_dev(const moe_lora_desc &l) {
    return LoraDev{l.r, l.scale, l.A, l.B, l.a_stride, l.b_stride};
}

static int check_head(const moe_head_desc *hd) {
    if (hd == nullptr) return fail(MOE_EINVAL, "head descriptor is NULL");
    if (hd->d <= 0 || hd->d % kGroup)
        return fail(MOE_EINVAL, "head: d=%d is not a positive multiple of 64", hd->d);
    if (hd->E < 1 || hd->E > 1024) return fail(MOE_EINVAL, "head: E=%d outside [1, 1024]", hd->E);
    if (hd->H < 0 || hd->H % kGroup)
        return fail(MOE_EINVAL, "head: H=%d is not a non-negative multiple of 64", hd->H);
    if (hd->prec != MOE_PREC_AFFINE4 && hd->prec != MOE_PREC_FP16)
        return fail(MOE_EINVAL, "head: prec=%d (need MOE_PREC_AFFINE4 or MOE_PREC_FP16)", hd->prec);
    if (hd->lx == nullptr || !aligned(hd->lx, 16)) return fail(MOE_EINVAL, "head: lx is NULL or misaligned");
    if (hd->H > 0) {
        if (hd->fc1x == nullptr || hd->fc2 == nullptr || !aligned(hd->fc1x, 16) ||
            !aligned(hd->fc2, 16))
            return fail(MOE_EINVAL, "head: H=%d with a NULL or misaligned fc1x/fc2", hd->H);
    }
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_EINVAL: return "MOE_EINVAL";
        case MOE_EUNSUPPORTED: return "MOE_EUNSUPPORTED";
        case MOE_ECUDA: return "MOE_ECUDA";
        case MOE_ETIMEOUT: return "MOE_ETIMEOUT";
        case MOE_ENOSPACE: return "MOE_ENOSPACE";
        default: return "MOE_UNKNOWN";
    }
}

const char *moe_last_error(void) { return g_last_error; }

size_t moe_record_bytes(int cols, int bits) {
    if (cols <= 0 || cols % kGroup || (bits != 2 && bits != 4)) return 0;
    return record_bytes(cols, bits);
}

size_t moe_packed_matrix_bytes(int rows, int cols, int bits) {
    if (rows <= 0) return 0;
    return (size_t)rows * moe_record_bytes(cols, bits);
}

size_t moe_pool_expert_bytes(int d, int F, int bits, int group) {
    if (group != kGroup || !shape_ok(d, F, bits)) return 0;
    return blob_layout(d, F, bits).bytes;
}

int moe_pack_matrix(const uint32_t *q, const uint16_t *s, const uint16_t *b, int rows,
                    int cols, int bits, void *out, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0 || cols % kGroup || (bits != 2 && bits != 4))
        return fail(MOE_EINVAL, "pack_matrix: rows=%d cols=%d bits=%d", rows, cols, bits);
    if (!q || !s || !b || !out) return fail(MOE_EINVAL, "pack_matrix: NULL pointer");
    if (!aligned(q, 4) || !aligned(s, 2) || !aligned(b, 2) || !aligned(out, 256))
        return fail(MOE_EINVAL, "pack_matrix: misaligned pointer (out needs 256 bytes)");
    return launch_pack_rows(q, s, b, rows, cols, bits, 1, 0, 0, static_cast<uint8_t *>(out), 0,
                            0, 1, stream);
}

int moe_pack_experts(int d, int F, int E, int bits, const uint32_t *gate_q,
                     const uint16_t *gate_s, const uint16_t *gate_b, const uint32_t *up_q,
                     const uint16_t *up_s, const uint16_t *up_b, const uint32_t *down_q,
                     const uint16_t *down_s, const uint16_t *down_b, void *pool,
                     size_t expert_stride, cudaStream_t stream) {
    if (!shape_ok(d, F, bits) || E < 1)
        return fail(MOE_EINVAL, "pack_experts: d=%d F=%d E=%d bits=%d", d, F, E, bits);
    if (!gate_q || !gate_s || !gate_b || !up_q || !up_s || !up_b || !down_q || !down_s ||
        !down_b || !pool)
        return fail(MOE_EINVAL, "pack_experts: NULL pointer");
    const BlobLayout L = blob_layout(d, F, bits);
    if (!aligned(pool, 256) || expert_stride < L.bytes || expert_stride % 256)
        return fail(MOE_EINVAL, "pack_experts: pool alignment or expert_stride %zu (need >= %zu, multiple of 256)",
                    expert_stride, L.bytes);
    uint8_t *dst = static_cast<uint8_t *>(pool);
    const size_t gq = (size_t)F * d * bits / 32, gsb = (size_t)F * d / kGroup;
    int rc = launch_pack_rows(gate_q, gate_s, gate_b, F, d, bits, E, gq, gsb, dst + L.gu_off,
                              expert_stride, 0, 2, stream);
    if (rc) return rc;
    rc = launch_pack_rows(up_q, up_s, up_b, F, d, bits, E, gq, gsb, dst + L.gu_off,
                          expert_stride, 1, 2, stream);
    if (rc) return rc;
    const size_t dq = (size_t)d * F * bits / 32, dsb = (size_t)d * F / kGroup;
    return launch_pack_rows(down_q, down_s, down_b, d, F, bits, E, dq, dsb, dst + L.down_off,
                            expert_stride, 0, 1, stream);
}

int moe_debug_dequant(const void *blob, int d, int F, int bits, int which, float *out,
                      cudaStream_t stream) {
    if (!shape_ok(d, F, bits) || which < 0 || which > 2)
        return fail(MOE_EINVAL, "debug_dequant: d=%d F=%d bits=%d which=%d", d, F, bits, which);
    if (!blob || !out || !aligned(blob, 256))
        return fail(MOE_EINVAL, "debug_dequant: NULL or misaligned pointer");
    const BlobLayout L = blob_layout(d, F, bits);
    const uint8_t *b = static_cast<const uint8_t *>(blob);
    if (which < 2)
        return launch_debug_dequant(b + L.gu_off, L.gu_rec, which, 2, F, d, bits, out, stream);
    return launch_debug_dequant(b + L.down_off, L.down_rec, 0, 1, d, F, bits, out, stream);
}

size_t moe_prerouter_head_workspace_bytes(const moe_head_desc *hd, int T) {
    if (hd == nullptr || T < 0) return 0;
    return 256 + align_up((size_t)T * hd->H * sizeof(float), 256) +
           align_up((size_t)T * hd->E * sizeof(float), 256) +
           align_up((size_t)T * gsum_ld(hd->d) * sizeof(float), 256) +
           align_up((size_t)2 * T * hd->H * sizeof(uint16_t), 256) +
           align_up((size_t)2 * T * gsum_ld(hd->H) * sizeof(float), 256);
}

int moe_prerouter_head(const moe_head_desc *hd, const void *x, int x_dtype,
                       const int32_t *cur_idx, const int32_t *prev_idx, int K, int T,
                       float *logits, void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (int rc = check_head(hd)) return rc;
    if (T < 0) return fail(MOE_EINVAL, "prerouter_head: T=%d", T);
    if (x_dtype != MOE_DTYPE_F32 && x_dtype != MOE_DTYPE_BF16)
        return fail(MOE_EINVAL, "prerouter_head: x_dtype=%d", x_dtype);
    if ((cur_idx || prev_idx) && (K < 1 || K > 16 || K > hd->E))
        return fail(MOE_EINVAL, "prerouter_head: K=%d with E=%d", K, hd->E);
    if (T == 0) return MOE_OK;
    if (!x || !logits || !aligned(x, 16) || !aligned(logits, 16))
        return fail(MOE_EINVAL, "prerouter_head: NULL or misaligned x/logits");
    const size_t need = moe_prerouter_head_workspace_bytes(hd, T);
    if (need && (ws == nullptr || ws_bytes < need || !aligned(ws, 256)))
        return fail(MOE_ENOSPACE, "prerouter_head: workspace %zu bytes, need %zu (256-aligned)",
                    ws_bytes, need);
    HeadParams p{};
    p.d = hd->d;
    p.E = hd->E;
    p.H = hd->H;
    p.K = K;
    p.T = T;
    p.prec = hd->prec;
    p.fc1x = static_cast<const uint8_t *>(hd->fc1x);
    p.fc1_tab = hd->fc1_tab;
    p.b1 = hd->b1;
    p.fc2 = static_cast<const uint8_t *>(hd->fc2);
    p.b2 = hd->b2;
    p.lx = static_cast<const uint8_t *>(hd->lx);
    p.l_tab = hd->l_tab;
    p.bl = hd->bl;
    p.x = x;
    p.x_dtype = x_dtype;
    p.cur = cur_idx;
    p.prev = prev_idx;
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.err = reinterpret_cast<int32_t *>(w);
    p.g = reinterpret_cast<float *>(w + 256);
    const size_t zl_off = 256 + align_up((size_t)T * hd->H * sizeof(float), 256);
    p.zl = reinterpret_cast<float *>(w + zl_off);
    const size_t xs_off = zl_off + align_up((size_t)T * hd->E * sizeof(float), 256);
    p.xsum = reinterpret_cast<float *>(w + xs_off);
    const size_t gg_off = xs_off + align_up((size_t)T * gsum_ld(hd->d) * sizeof(float), 256);
    p.gg = reinterpret_cast<__nv_bfloat16 *>(w + gg_off);
    p.ggsum = reinterpret_cast<float *>(w + gg_off + align_up((size_t)2 * T * hd->H * sizeof(uint16_t), 256));
    p.logits = logits;
    return launch_prerouter_head(p, stream);
}

int moe_topk_route(const float *logits, int T, int E, int K, int32_t *idx, float *w,
                   float *margin, cudaStream_t stream) {
    if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 16 || K > E)
        return fail(MOE_EINVAL, "topk_route: T=%d E=%d K=%d (need 1<=K<=16, K<=E<=1024)", T, E, K);
    if (T == 0) return MOE_OK;
    if (!logits || !idx || !w) return fail(MOE_EINVAL, "topk_route: NULL pointer");
    if (!aligned(logits, 4) || !aligned(idx, 4) || !aligned(w, 4) || (margin && !aligned(margin, 4)))
        return fail(MOE_EINVAL, "topk_route: misaligned pointer");
    return launch_topk(logits, T, E, K, idx, w, margin, stream);
}

size_t moe_expert_ffn_workspace_bytes(const moe_experts_desc *ed, int T, int K) {
    if (ed == nullptr || T < 0 || K < 0) return 0;
    return ffn_ws(ed, T, K).total;
}

int moe_expert_ffn_int4(const moe_experts_desc *ed, const void *x, int x_dtype,
                        const int32_t *idx, int T, int K, float *y_slots, void *ws,
                        size_t ws_bytes, cudaStream_t stream) {
    if (int rc = check_experts(ed)) return rc;
    if (T < 0 || K < 1 || K > 16 || K > ed->E)
        return fail(MOE_EINVAL, "expert_ffn: T=%d K=%d E=%d (need 1<=K<=16, K<=E)", T, K, ed->E);
    if (x_dtype != MOE_DTYPE_F32 && x_dtype != MOE_DTYPE_BF16)
        return fail(MOE_EINVAL, "expert_ffn: x_dtype=%d", x_dtype);
    if (T == 0) return MOE_OK;
    if (!x || !idx || !y_slots || !aligned(x, 16) || !aligned(idx, 4) || !aligned(y_slots, 16))
        return fail(MOE_EINVAL, "expert_ffn: NULL or misaligned x/idx/y_slots");
    const FfnWs wl = ffn_ws(ed, T, K);
    if (ws == nullptr || ws_bytes < wl.total || !aligned(ws, 256))
        return fail(MOE_ENOSPACE, "expert_ffn: workspace %zu bytes, need %zu (256-aligned)",
                    ws_bytes, wl.total);
    FfnParams p{};
    p.pool = static_cast<const uint8_t *>(ed->pool);
    p.stride = ed->expert_stride;
    p.shared = static_cast<const uint8_t *>(ed->shared);
    p.idx = idx;
    p.T = T;
    p.K = K;
    p.slots = K + (ed->shared ? 1 : 0);
    p.d = ed->d;
    p.F = ed->F;
    p.E = ed->E;
    p.bits = ed->bits;
    p.x = x;
    p.x_dtype = x_dtype;
    p.round_h_bf16 = x_dtype == MOE_DTYPE_BF16;
    uint8_t *w = static_cast<uint8_t *>(ws);
    p.h = reinterpret_cast<float *>(w + wl.h);
    p.v = reinterpret_cast<float *>(w + wl.v);
    p.counts = reinterpret_cast<int32_t *>(w + wl.counts);
    p.offsets = reinterpret_cast<int32_t *>(w + wl.offsets);
    p.perm = reinterpret_cast<int32_t *>(w + wl.perm);
    p.xb = static_cast<const __nv_bfloat16 *>(x);
    p.xg = reinterpret_cast<__nv_bfloat16 *>(w + wl.xg);
    p.xsum = reinterpret_cast<float *>(w + wl.xsum);
    p.h16 = reinterpret_cast<__nv_bfloat16 *>(w + wl.h16);
    p.hsum = reinterpret_cast<float *>(w + wl.hsum);
    p.vd = reinterpret_cast<float *>(w + wl.vd);
    p.item_off = reinterpret_cast<int32_t *>(w + wl.item_off);
    p.err = reinterpret_cast<int32_t *>(w + wl.err);
    p.y = y_slots;
    for (int i = 0; i < 3; i++) {
        p.lora[i] = lora_dev(ed->lora[i]);
        p.shared_lora[i] = lora_dev(ed->shared ? ed->shared_lora[i] : moe_lora_desc{});
    }
    p.any_gu_lora = ed->lora[0].r || ed->lora[1].r ||
                    (ed->shared && (ed->shared_lora[0].r || ed->shared_lora[1].r));
    p.L = blob_layout(ed->d, ed->F, ed->bits);
    // Several tokens in bf16 (prefill, batched decode): sorted by expert and
    // run as grouped GEMMs.  One token, or fp32 activations: per-token GEMVs.
    if (T > 1 && x_dtype == MOE_DTYPE_BF16) return launch_expert_ffn_grouped(p, stream);
    return launch_expert_ffn(p, stream);
}

int moe_combine_residual(const float *y_slots, const float *w, int T, int K, int has_shared,
                         int d, const float *residual, float *out, float *x_next,
                         cudaStream_t stream) {
    if (T < 0 || K < 0 || K > 16 || d < 1 || (K == 0 && !has_shared))
        return fail(MOE_EINVAL, "combine_residual: T=%d K=%d d=%d has_shared=%d", T, K, d, has_shared);
    if (T == 0) return MOE_OK;
    if (!y_slots || (K > 0 && !w) || !residual || !out)
        return fail(MOE_EINVAL, "combine_residual: NULL pointer");
    if (!aligned(y_slots, 4) || (w && !aligned(w, 4)) || !aligned(residual, 4) ||
        !aligned(out, 4) || (x_next && !aligned(x_next, 4)))
        return fail(MOE_EINVAL, "combine_residual: misaligned pointer");
    return launch_combine(y_slots, w, T, K, has_shared ? 1 : 0, d, residual, out, x_next, stream);
}

}  // extern "C"
