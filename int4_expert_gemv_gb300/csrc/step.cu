// step.cu -- one decode step of a whole layer stack in one persistent kernel.
//
// The four per-layer operations of the prerouted MoE layer -- expert FFN
// (gate/up + SwiGLU, down, unfused LoRA), combine + residual (+ RMS for the
// next layer's input), prerouter head and its top-K -- run for every layer of
// the stack inside one launch of one CTA per SM.  What makes this pay on GB300:
//
//  * Every expert a step reads is known when the step starts (the route of
//    layer N+1 for token t+1 is predicted by head N at token t: "Ideas clave"
//    and "Arquitectura del cabezal Prerouter" of xyznot.com/es/paper/
//    2609.18063), so weight fetches never wait for the activations.  A
//    producer warp streams each CTA's share of every layer's weights into a
//    byte ring in shared memory with bulk copies (cp.async.bulk + mbarrier),
//    as far ahead as the ring allows, across layer boundaries.
//  * Dependencies between CTAs (h after gate/up, out after down, head values,
//    LoRA products) travel as 64-bit (tag, value) words in global memory: a
//    reader polls the words it needs until their tag is the current one.
//    There is no grid-wide barrier; each value is its own ready flag.  All
//    polls of a phase are issued together, so a layer costs two dependent
//    round trips: x (the previous layer's out) and h.
//  * x enters the GEMVs unnormalised; 1/rms is applied to each finished row
//    dot, so a CTA can start on x as soon as it has polled it.
//  * Every wait is bounded (globaltimer); on expiry the kernel records
//    MOE_ETIMEOUT in the workspace status word, waits (bounded) for its own
//    copies in flight and returns.
//
// Work per layer.  Phase A (needs x): LoRA A-rows on x, gate/up row pairs of
// every slot (slots with gate/up LoRA first), head fc1 rows and l rows --
// split across CTAs by bytes.  The owners of a down-LoRA slot's gate/up rows
// also publish their partial A_d h.  Phase B (needs h): down rows (CTA c owns
// outputs [c*d/n, (c+1)*d/n) of every slot, adds their LoRA terms and
// combines them), then head fc2 rows (split by count).  Phase R (layer 0,
// when it routes with its own router): router rows.
#include <algorithm>

#include "step_common.cuh"

namespace moe {
namespace step {

constexpr int kMaxLayers = 48;
constexpr int kNW = 12;                        // consumer warps
constexpr int kProducerWarp = 0, kRouteWarp = 1, kCons0 = 2;
constexpr int kThreads = (kCons0 + kNW) * 32;  // 448
constexpr int kMaxPiece = 16384;               // bytes per bulk copy
constexpr int kNB = 32;                        // pieces in flight (barrier pairs)
constexpr int kMaxK = 16;
constexpr int kMaxGroups = 40;
constexpr int kMaxOwnE = 64;                   // fc2 rows one CTA may own
constexpr int kMaxVdp = 4096;                  // floats of polled A_d h partials
constexpr int kTrace = 16;                     // stamps per (CTA, layer), debug trace

enum Kind : uint8_t { KLA = 0, KGU, KFC1, KLX, KROUTER, KDOWN, KFC2 };
enum Tmpl : int { T_R = 0, T_A_HEAD, T_A_NOHEAD, T_B_HEAD, T_B_NOHEAD, T_COUNT };

// control words at the start of the workspace
enum Ctrl : int { C_STATUS = 0, C_EPOCH = 1, C_DONE = 2, C_ABORT = 3, C_NEVER = 4 };
constexpr size_t kCtrlBytes = 256;

struct LoraP {
    int r;
    float scale;
    const uint16_t *A, *B;
    size_t as, bs;
};

struct LayerP {
    const uint8_t *pool, *shared;
    LoraP lora[3], slora[3];
    const uint8_t *router;
    const uint8_t *fc1x;
    const uint16_t *fc1_tab, *b1;
    const uint8_t *fc2;
    const uint16_t *b2;
    const uint8_t *lx;
    const uint16_t *l_tab, *bl;
};

struct Params {
    int d, F, E, K, H, S, depth, n_res, self_predict, own0, t, n_cta, max_orows, rd;
    uint32_t ring_bytes;
    size_t stride;
    uint32_t gu_off, down_off, rec_d, rec_F, rec_dh, rec_H;
    const float *x0;
    float *out;
    int32_t *ridx;
    float *rw, *rmargin;
    uint8_t *ws;
    uint32_t off_h, off_v, off_vdp, off_ga, off_zl, off_zr, off_z, off_out;
    uint64_t timeout_ns;
    int debug_unset_wait;
    unsigned long long *trace;   // debug: [n_cta][depth][kTrace] globaltimer stamps
    // shared-memory layout (byte offsets from the dynamic base)
    uint32_t sm_ring, sm_bar, sm_pend, sm_tmpl, sm_xf, sm_xsc, sm_xhat, sm_xf4, sm_xsc4, sm_xhat4,
        sm_stream, sm_hf, sm_hsc, sm_hhat, sm_gf, sm_gsc, sm_ghat, sm_zl, sm_y, sm_bd, sm_vdp,
        sm_vd, sm_rcur, sm_rprev, sm_rw, sm_misc;
    LayerP layer[kMaxLayers];
};

// A group of equal items, contiguous in memory; [lo, hi) = this CTA's items.
struct Grp {
    uint32_t item_bytes;
    int n, lo, hi, cols;
    uint8_t kind, slot, aux, pad;
};

// A phase's groups, identical for every layer of the same kind (only the
// source addresses depend on the layer and its route).
struct Tmplt {
    Grp g[kMaxGroups];
    int n;
    int o_lo, o_hi, e_lo, e_hi;
    // phase A: owners [own0[s], own1[s]] of the gate/up rows of slot s
    int own0[kMaxK + 1], own1[kMaxK + 1];
};

// ---------------------------------------------------------------- control
__device__ __forceinline__ int *ctrl(const Params &p) { return reinterpret_cast<int *>(p.ws); }

__device__ __forceinline__ void raise_error(const Params &p, int code) {
    atomicCAS(ctrl(p) + C_STATUS, 0, code);
    atomicExch(ctrl(p) + C_ABORT, 1);
}

__device__ __forceinline__ bool aborted(const Params &p) { return ld_flag(ctrl(p) + C_ABORT) != 0; }

// Warp-collective bounded wait on an mbarrier phase: every lane observes the
// phase and the warp leaves together; false (error recorded) on timeout or
// when another CTA has aborted.
__device__ bool wait_bar_warp(const Params &p, uint64_t *bar, uint32_t parity) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    if (lane == 0) t0 = now_ns();
    for (int it = 1;; it++) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((it & 63) == 0) {
            int stop = 0;
            if (lane == 0) {
                if (aborted(p)) stop = 1;
                else if (now_ns() - t0 > p.timeout_ns) {
                    raise_error(p, MOE_ETIMEOUT);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        }
    }
}

// Single-thread bounded wait (producer lane, end of kernel).
__device__ bool wait_bar(const Params &p, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    for (int it = 1;; it++) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (aborted(p)) return false;
            if (now_ns() - t0 > p.timeout_ns) {
                raise_error(p, MOE_ETIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ uint64_t *tagged(const Params &p, uint32_t off) {
    return reinterpret_cast<uint64_t *>(p.ws + off);
}

// Per-thread bounded poll of `cnt` (<= 8) tagged words at w + idx[k], all
// loads in flight together; values to val[k].  False on timeout or abort.
__device__ __forceinline__ bool poll_set(const Params &p, const uint64_t *w, const int *idx,
                                         int cnt, uint32_t tag, float *val) {
    uint32_t pend = (1u << cnt) - 1u;
    uint64_t t0 = 0;
    for (int it = 0; pend; it++) {
        uint64_t v[8];
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (pend >> k & 1u) v[k] = get_word(w + idx[k]);
#pragma unroll
        for (int k = 0; k < 8; k++)
            if ((pend >> k & 1u) && (uint32_t)(v[k] >> 32) == tag) {
                val[k] = __uint_as_float((uint32_t)v[k]);
                pend &= ~(1u << k);
            }
        if (pend) {
            // back off so that waiting warps leave issue slots to working ones
            __nanosleep(32u << (it < 3 ? it : 3));
            if ((it & 7) == 7) {
                if (it == 7) t0 = now_ns();
                else if (aborted(p)) return false;
                else if (now_ns() - t0 > p.timeout_ns) {
                    raise_error(p, MOE_ETIMEOUT);
                    return false;
                }
            }
        }
    }
    return true;
}

// Warp poll of E logits, lane-strided (vals[i] = logit lane + 32 i), all in
// flight together.  Warp-uniform result.
__device__ __noinline__ bool poll_logits(const Params &p, const uint64_t *z, int E, uint32_t tag, int lane,
                            float (&vals)[32]) {
    uint32_t pend = 0;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        vals[i] = -INFINITY;
        if (lane + 32 * i < E) pend |= 1u << i;
    }
    uint64_t t0 = 0;
    bool lok = true;
    for (int it = 0; pend && lok; it++) {
#pragma unroll
        for (int i = 0; i < 32; i++)
            if (pend >> i & 1u) {
                const uint64_t v = get_word(z + lane + 32 * i);
                if ((uint32_t)(v >> 32) == tag) {
                    vals[i] = __uint_as_float((uint32_t)v);
                    pend &= ~(1u << i);
                }
            }
        if (pend) {
            __nanosleep(64u << (it < 2 ? it : 2));
            if ((it & 7) == 7) {
                if (it == 7) t0 = now_ns();
                else if (aborted(p)) lok = false;
                else if (now_ns() - t0 > p.timeout_ns) {
                    raise_error(p, MOE_ETIMEOUT);
                    lok = false;
                }
            }
        }
    }
    return __all_sync(0xffffffffu, lok);
}

// ---------------------------------------------------------------- layers
__device__ __forceinline__ const LayerP &layer_of(const Params &p, int N) {
    return p.layer[N % p.n_res];
}

__device__ __forceinline__ bool head_runs(const Params &p, int N) {
    return N + 1 < p.depth || p.self_predict;
}

__device__ __forceinline__ const LoraP &slot_lora(const Params &p, const LayerP &L, int s, int w) {
    return s < p.K ? L.lora[w] : L.slora[w];
}

__device__ __forceinline__ const uint8_t *slot_blob(const Params &p, const LayerP &L,
                                                    const int *route, int s) {
    return s < p.K ? L.pool + (size_t)route[s] * p.stride : L.shared;
}

__device__ __forceinline__ const uint16_t *lora_a(const Params &p, const LayerP &L, const int *route,
                                                  int s, int w) {
    const LoraP &l = slot_lora(p, L, s, w);
    return l.A + (s < p.K ? (size_t)route[s] * l.as : 0);
}

__device__ __forceinline__ const uint16_t *lora_bm(const Params &p, const LayerP &L,
                                                   const int *route, int s, int w) {
    const LoraP &l = slot_lora(p, L, s, w);
    return l.B + (s < p.K ? (size_t)route[s] * l.bs : 0);
}

// Address of item 0 of group g in layer N.
__device__ __forceinline__ const uint8_t *group_src(const Params &p, int N, const Grp &g,
                                                    const int *route) {
    const LayerP &L = layer_of(p, N);
    switch (g.kind) {
        case KLA: return reinterpret_cast<const uint8_t *>(lora_a(p, L, route, g.slot, g.aux));
        case KGU: return slot_blob(p, L, route, g.slot) + p.gu_off;
        case KFC1: return L.fc1x;
        case KLX: return L.lx;
        case KROUTER: return L.router;
        case KDOWN: return slot_blob(p, L, route, g.slot) + p.down_off;
        default: return L.fc2;
    }
}

__device__ __forceinline__ bool gu_lora(const Params &p, const LayerP &L, int s) {
    return slot_lora(p, L, s, 0).r || slot_lora(p, L, s, 1).r;
}

// ---------------------------------------------------------------- templates
__device__ void add_group(Tmplt &t, uint32_t ib, int n, int kind, int slot, int aux, int cols,
                          int lo = 0, int hi = 0) {
    Grp &g = t.g[t.n++];
    g.item_bytes = ib;
    g.n = n;
    g.lo = lo;
    g.hi = hi;
    g.cols = cols;
    g.kind = (uint8_t)kind;
    g.slot = (uint8_t)slot;
    g.aux = (uint8_t)aux;
    g.pad = 0;
}

__device__ __forceinline__ long long split_at(long long total, int c, int n) {
    return total * c / n;
}

// CTA owning the item that starts at byte `pos` of a phase of `total` bytes.
__device__ int owner_of(long long pos, long long total, int n) {
    int c = (int)(pos * n / total);
    if (c > n - 1) c = n - 1;
    while (c + 1 < n && split_at(total, c + 1, n) <= pos) c++;
    while (c > 0 && split_at(total, c, n) > pos) c--;
    return c;
}

// Item ranges of all groups of t under an even split of their bytes; also the
// owner CTAs of each gate/up group.
__device__ void split_bytes(Tmplt &t, int c, int n_cta) {
    long long total = 0;
    for (int i = 0; i < t.n; i++) total += (long long)t.g[i].n * t.g[i].item_bytes;
    const long long a = split_at(total, c, n_cta), b = split_at(total, c + 1, n_cta);
    long long base = 0;
    for (int i = 0; i < t.n; i++) {
        Grp &g = t.g[i];
        const long long ib = g.item_bytes;
        const long long lo = a <= base ? 0 : (a - base + ib - 1) / ib;
        const long long hi = b <= base ? 0 : (b - base + ib - 1) / ib;
        g.lo = (int)(lo < g.n ? lo : g.n);
        g.hi = (int)(hi < g.n ? hi : g.n);
        if (g.kind == KGU) {
            t.own0[g.slot] = owner_of(base, total, n_cta);
            t.own1[g.slot] = owner_of(base + (long long)(g.n - 1) * ib, total, n_cta);
        }
        base += (long long)g.n * ib;
    }
}

// The CTA's phase templates (built once per launch by one thread).
__device__ __noinline__ void build_templates(const Params &p, int c, Tmplt *T) {
    const LayerP &L = p.layer[0];
    {
        Tmplt &t = T[T_R];
        t.n = 0;
        add_group(t, p.rec_dh, p.E, KROUTER, 0, 0, p.d);
        split_bytes(t, c, p.n_cta);
    }
    for (int head = 1; head >= 0; head--) {
        Tmplt &t = T[head ? T_A_HEAD : T_A_NOHEAD];
        t.n = 0;
        for (int s = 0; s < p.S; s++)
            for (int w = 0; w < 2; w++)
                if (slot_lora(p, L, s, w).r)
                    add_group(t, 2u * p.d, slot_lora(p, L, s, w).r, KLA, s, w, p.d);
        for (int pass = 0; pass < 2; pass++)              // LoRA slots first
            for (int s = 0; s < p.S; s++)
                if (gu_lora(p, L, s) == (pass == 0)) add_group(t, 2u * p.rec_d, p.F, KGU, s, 0, p.d);
        if (head) {
            if (p.H) add_group(t, p.rec_dh, p.H, KFC1, 0, 0, p.d);
            add_group(t, p.rec_dh, p.E, KLX, 0, 0, p.d);
        }
        split_bytes(t, c, p.n_cta);
    }
    const int o_lo = (int)((long long)p.d * c / p.n_cta);
    const int o_hi = (int)((long long)p.d * (c + 1) / p.n_cta);
    const int e_lo = (int)((long long)p.E * c / p.n_cta);
    const int e_hi = (int)((long long)p.E * (c + 1) / p.n_cta);
    for (int head = 1; head >= 0; head--) {
        Tmplt &t = T[head ? T_B_HEAD : T_B_NOHEAD];
        t.n = 0;
        t.o_lo = o_lo;
        t.o_hi = o_hi;
        t.e_lo = e_lo;
        t.e_hi = e_hi;
        for (int s = 0; s < p.S; s++) add_group(t, p.rec_F, p.d, KDOWN, s, 0, p.F, o_lo, o_hi);
        if (head && p.H > 0) add_group(t, p.rec_H, p.E, KFC2, 0, 0, p.H, e_lo, e_hi);
    }
}

__device__ __forceinline__ const Tmplt &tmpl_A(const Params &p, const Tmplt *T, int N) {
    return T[head_runs(p, N) ? T_A_HEAD : T_A_NOHEAD];
}

__device__ __forceinline__ const Tmplt &tmpl_B(const Params &p, const Tmplt *T, int N) {
    return T[head_runs(p, N) ? T_B_HEAD : T_B_NOHEAD];
}

__host__ __device__ __forceinline__ int pow2_floor32(int n) {
    int l = 1;
    while (l * 2 <= n && l < 32) l *= 2;
    return l;
}

// 16-byte chunks per item row (what the lanes of a row split).
template <int BITS>
__device__ __forceinline__ int item_chunks(const Grp &g) {
    switch (g.kind) {
        case KGU:
        case KDOWN: return g.cols * BITS / 128;
        case KLA: return g.cols / 8;
        default: return g.cols / 32;              // int4 head rows
    }
}

// ---------------------------------------------------------------- ring
// Byte ring of pieces: a piece never straddles the end of the ring; producer
// and consumers place pieces with the same rule, so they agree on offsets.
struct RingPos {
    uint64_t head = 0;
    uint32_t q = 0;
    __device__ __forceinline__ uint64_t place(uint32_t bytes, uint32_t rb) {
        uint64_t start = head;
        if ((uint32_t)(start % rb) + bytes > rb) start = (start / rb + 1) * rb;
        head = start + bytes;
        return start;
    }
};

// ---------------------------------------------------------------- smem views
struct Smem {
    uint8_t *ring;
    uint64_t *full, *empty, *route_bar, *cons_bar, *end_bar, *pend;
    Tmplt *T;
    uint8_t *xf, *xf4, *hf, *gf;          // staged fixed-point vectors
    float *xsc, *xhat, *xsc4, *xhat4, *hsc, *hhat, *gsc, *ghat;
    float *stream, *zl, *y, *bd, *vdp, *vd;
    int *rcur, *rprev;
    float *rw, *misc;
};

__device__ __forceinline__ Smem smem_views(const Params &p, uint8_t *base) {
    Smem s;
    s.ring = base + p.sm_ring;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + p.sm_bar);
    s.full = bars;
    s.empty = bars + kNB;
    s.route_bar = bars + 2 * kNB;
    s.cons_bar = s.route_bar + 1;
    s.end_bar = s.route_bar + 2;
    s.pend = reinterpret_cast<uint64_t *>(base + p.sm_pend);
    s.T = reinterpret_cast<Tmplt *>(base + p.sm_tmpl);
    auto f = [&](uint32_t o) { return reinterpret_cast<float *>(base + o); };
    s.xf = base + p.sm_xf;
    s.xf4 = base + p.sm_xf4;
    s.hf = base + p.sm_hf;
    s.gf = base + p.sm_gf;
    s.xsc = f(p.sm_xsc);
    s.xhat = f(p.sm_xhat);
    s.xsc4 = f(p.sm_xsc4);
    s.xhat4 = f(p.sm_xhat4);
    s.hsc = f(p.sm_hsc);
    s.hhat = f(p.sm_hhat);
    s.gsc = f(p.sm_gsc);
    s.ghat = f(p.sm_ghat);
    s.stream = f(p.sm_stream);
    s.zl = f(p.sm_zl);
    s.y = f(p.sm_y);
    s.bd = f(p.sm_bd);
    s.vdp = f(p.sm_vdp);
    s.vd = f(p.sm_vd);
    s.rcur = reinterpret_cast<int *>(base + p.sm_rcur);
    s.rprev = reinterpret_cast<int *>(base + p.sm_rprev);
    s.rw = f(p.sm_rw);
    s.misc = f(p.sm_misc);
    return s;
}

// ---------------------------------------------------------------- math helpers
// Dot products of R rows (records at rec + r*stride) with a staged vector
// (xf, per-chunk scale and xhat) over the chunks this lane owns; reduced over
// the lpr lanes of each row group.  Per chunk: exact integer codes . x^, then
// fma(scale, that, bias * xhat) -- the affine dequantisation applied once per
// chunk instead of per weight.
template <int BITS, int R>
__device__ __forceinline__ void rows_dot(const uint8_t *rec, uint32_t stride, int cols,
                                         const uint8_t *xf, const float *xsc, const float *xhat,
                                         int sub, int lpr, float *out) {
    constexpr int VALS = 128 / BITS;
    const int nch = cols / VALS;
    const int cb = cols * BITS / 8;
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; r++) acc[r] = 0.0f;
    const uint4 *xq = reinterpret_cast<const uint4 *>(xf);
    for (int c = sub; c < nch; c += lpr) {
        uint4 q[R];
        uint32_t sbw[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            q[r] = *reinterpret_cast<const uint4 *>(rec + (size_t)r * stride + (size_t)kChunk * c);
            sbw[r] = *reinterpret_cast<const uint32_t *>(rec + (size_t)r * stride + cb +
                                                         4 * ((c * VALS) / kGroup));
        }
        int dq[R];
        chunk_dot_fix<BITS, R>(q, xq, nch, c, dq);
        const float sc = xsc[c], X = xhat[c];
#pragma unroll
        for (int r = 0; r < R; r++) {
            const float2 sb = sb_f(sbw[r]);
            acc[r] += fmaf(sb.x, (float)dq[r] * sc, sb.y * X);
        }
    }
#pragma unroll
    for (int r = 0; r < R; r++) out[r] = warp_sum(acc[r], lpr);
}

// Dot product of one fp16 row (in smem) with a plain float vector (smem),
// reduced over the lpr lanes of the row group.
__device__ __forceinline__ float f16_row_dot_s(const uint8_t *row, int cols, const float *v,
                                               int sub, int lpr) {
    float acc = 0.0f;
    for (int c = sub; c < cols / 8; c += lpr)
        acc += chunk_dot_f16(*reinterpret_cast<const uint4 *>(row + (size_t)kChunk * c), v + 8 * c);
    return warp_sum(acc, lpr);
}

// Warp top-K over E logits (value desc, index asc) -> idx, softmax weights,
// margin (lane 0's copies are the ones used).  vals[i]: logit of expert
// lane + 32 i (-inf beyond E).
__device__ __noinline__ void warp_topk(const float (&vals)[32], int E, int K, int lane, int *idx, float *w,
                          float *margin) {
    uint32_t taken = 0;
    float topv[kMaxK + 1];
    int topi[kMaxK + 1];
    const int rounds = K < E ? K + 1 : K;
    for (int k = 0; k < rounds; k++) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 32; i++) {
            const int e = lane + 32 * i;
            const float v = vals[i] == vals[i] ? vals[i] : -INFINITY;
            if (e < E && !(taken >> i & 1u) && (v > bv || (v == bv && e < bi))) {
                bv = v;
                bi = e;
            }
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        topv[k] = bv;
        topi[k] = bi;
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    float sum = 0.0f;
    for (int k = 0; k < K; k++) sum += expf(topv[k] - topv[0]);
    for (int k = 0; k < K; k++) {
        idx[k] = topi[k];
        w[k] = expf(topv[k] - topv[0]) / sum;
    }
    *margin = K < E ? topv[K - 1] - topv[K] : INFINITY;
}

// ---------------------------------------------------------------- producer
template <int BITS>
__device__ __noinline__ void producer(const Params &p, const Smem &s) {
    RingPos rp;
    uint32_t rel = 0;       // pieces [rel, rp.q) are not yet released
    uint64_t tail = 0;      // ring bytes before `tail` are free
    bool ok = true;
    auto issue = [&](int N, const Tmplt &t) -> bool {
        const int *route = s.rcur + N * p.K;
        for (int gi = 0; gi < t.n; gi++) {
            const Grp &g = t.g[gi];
            const uint8_t *src = group_src(p, N, g, route);
            const int per = max(1, kMaxPiece / (int)g.item_bytes);
            for (int i0 = g.lo; i0 < g.hi; i0 += per) {
                const uint32_t bytes = (uint32_t)min(per, g.hi - i0) * g.item_bytes;
                const uint64_t start = rp.place(bytes, p.ring_bytes);
                const uint32_t q = rp.q++;
                while (rel < q && (start + bytes - tail > p.ring_bytes || q - rel >= (uint32_t)kNB)) {
                    if (!wait_bar(p, s.empty + rel % kNB, (rel / kNB) & 1)) return false;
                    tail = s.pend[rel % kNB];
                    rel++;
                }
                s.pend[q % kNB] = start + bytes;
                mbar_arrive_expect_tx(s.full + q % kNB, bytes);
                bulk_g2s(s.ring + start % p.ring_bytes, src + (size_t)i0 * g.item_bytes, bytes,
                         s.full + q % kNB);
            }
        }
        return true;
    };
    for (int N = 0; N < p.depth && ok; N++) {
        if (N == 0 && p.own0) {
            if (!(ok = issue(0, s.T[T_R]))) break;
            if (!(ok = wait_bar(p, s.route_bar, 0))) break;
        }
        // validate the route before it turns into addresses
        for (int k = 0; k < p.K; k++)
            if ((unsigned)s.rcur[N * p.K + k] >= (unsigned)p.E) {
                raise_error(p, MOE_EINVAL);
                ok = false;
            }
        if (!ok) break;
        if (p.trace) p.trace[((size_t)blockIdx.x * p.depth + N) * kTrace + 9] = now_ns();
        if (!(ok = issue(N, tmpl_A(p, s.T, N)))) break;
        if (p.trace) p.trace[((size_t)blockIdx.x * p.depth + N) * kTrace + 10] = now_ns();
        if (!(ok = issue(N, tmpl_B(p, s.T, N)))) break;
        if (p.trace) p.trace[((size_t)blockIdx.x * p.depth + N) * kTrace + 11] = now_ns();
    }
    // never leave the CTA with copies in flight: wait (bounded) for every
    // piece not yet released
    for (uint32_t q = rel; q < rp.q; q++) {
        if (!mbar_try_wait(s.full + q % kNB, (q / kNB) & 1)) {
            const uint64_t t0 = now_ns();
            while (!mbar_try_wait(s.full + q % kNB, (q / kNB) & 1) && now_ns() - t0 < p.timeout_ns) {
            }
        }
    }
}

// ---------------------------------------------------------------- route warp
// Top-K of the heads' logits of the layers this CTA is responsible for;
// writes the predicted routes for the next step.
__device__ __noinline__ void route_warp(const Params &p, int c, int lane) {
    const int nxt = (p.t + 1) % 3;
    const uint32_t epoch = (uint32_t)ld_flag(ctrl(p) + C_EPOCH);
    for (int N = c; N < p.depth; N += p.n_cta) {
        if (!head_runs(p, N)) continue;
        float vals[32];
        if (!poll_logits(p, tagged(p, p.off_z) + (size_t)N * p.E, p.E, epoch * 64u + N + 1, lane,
                         vals))
            return;
        int idx[kMaxK];
        float w[kMaxK], margin;
        warp_topk(vals, p.E, p.K, lane, idx, w, &margin);
        const int tgt = N + 1 < p.depth ? N + 1 : 0;
        if (lane == 0) {
            for (int k = 0; k < p.K; k++) {
                p.ridx[((size_t)nxt * p.depth + tgt) * p.K + k] = idx[k];
                p.rw[((size_t)nxt * p.depth + tgt) * p.K + k] = w[k];
            }
            p.rmargin[(size_t)nxt * p.depth + tgt] = margin;
        }
    }
}

// ---------------------------------------------------------------- consumers
template <int BITS>
struct Consumer {
    const Params &p;
    const Smem &s;
    int c, warp, lane;   // warp: 0 .. kNW-1
    uint32_t epoch;
    RingPos rp;
    uint32_t nsync = 0;
    float inv = 1.0f;    // 1/rms of this layer's input
    float vdp0 = 0.0f, vdp1 = 0.0f;   // partial A_d h, by slot parity
    int trace_gu = 0;

    static constexpr int kT = kNW * 32;
    static constexpr int VALS = 128 / BITS;
    __device__ uint32_t tag(int N) const { return epoch * 64u + (uint32_t)N + 1u; }
    __device__ uint32_t tag_router() const { return epoch * 64u + 63u; }
    __device__ int tid() const { return warp * 32 + lane; }
    __device__ void stamp(int N, int k) const {
        if (p.trace && warp == 0 && lane == 0)
            p.trace[((size_t)c * p.depth + N) * kTrace + k] = now_ns();
    }

    // barrier among the consumer warps (bounded)
    __device__ bool sync() {
        __syncwarp();
        if (lane == 0) mbar_arrive(s.cons_bar);
        const bool ok = wait_bar_warp(p, s.cons_bar, nsync & 1);
        nsync++;
        __syncwarp();
        return ok;
    }

    // Polls the tagged words of `nvec` vectors of `vec` values at w and stages
    // them chunk by chunk (VB-bit chunks of vb values): warp w takes chunks
    // w, w+kNW, ...; lane j polls values j, j+32, ... of a chunk.  Vector vi is
    // staged at xf + vi*vec*2 bytes with scales/xhat at sc/hat + vi*(vec/vb).
    // Plain values go to plain[] if not null; ss accumulates their squares.
    template <int VB>
    __device__ __noinline__ bool poll_chunks(const uint64_t *w, int nvec, int vec, uint32_t tg,
                                             uint8_t *xf, float *sc, float *hat, float *plain,
                                             float *ss) {
        constexpr int vb = 128 / VB;              // values per chunk
        constexpr int per = vb / 32;              // values per lane per chunk
        const int cpv = vec / vb;                 // chunks per vector
        const int nchunks = nvec * cpv;
        constexpr int CB = 8 / per;               // chunks per poll batch
        bool lok = true;
        for (int ch0 = warp; ch0 < nchunks; ch0 += kNW * CB) {
            int idx[8];
            float val[8];
            int cnt = 0;
#pragma unroll
            for (int b = 0; b < CB; b++) {
                const int ch = ch0 + b * kNW;
#pragma unroll
                for (int m = 0; m < per; m++) {
                    idx[b * per + m] = ch * vb + lane + 32 * m;
                    val[b * per + m] = 0.0f;
                }
                if (ch < nchunks) cnt = (b + 1) * per;
            }
            if (lok) lok = poll_set(p, w, idx, cnt, tg, val);
#pragma unroll
            for (int b = 0; b < CB; b++) {
                const int ch = ch0 + b * kNW;
                if (ch >= nchunks) break;             // warp-uniform
                const int vi = ch / cpv, cl = ch % cpv;
                stage_chunk<VB>(val + b * per, lane, xf + (size_t)vi * vec * 2, cl, cpv,
                                sc + vi * cpv, hat + vi * cpv);
#pragma unroll
                for (int m = 0; m < per; m++) {
                    const float v = val[b * per + m];
                    if (plain) plain[vi * vec + cl * vb + lane + 32 * m] = v;
                    *ss = fmaf(v, v, *ss);
                }
            }
        }
        return __all_sync(0xffffffffu, lok);
    }

    // Stages a plain vector in smem (n values) in the VB-bit layout.
    template <int VB>
    __device__ void stage_plain(const float *v, int n, uint8_t *xf, float *sc, float *hat) {
        constexpr int vb = 128 / VB, per = vb / 32;
        for (int ch = warp; ch < n / vb; ch += kNW) {
            float val[per];
#pragma unroll
            for (int m = 0; m < per; m++) val[m] = v[ch * vb + lane + 32 * m];
            stage_chunk<VB>(val, lane, xf, ch, n / vb, sc, hat);
        }
    }

    // x of layer N (unnormalised: the previous layer's out, or x0), staged for
    // the expert GEMVs (and, with 2-bit experts, for the int4 heads too);
    // inv = 1/rms (1 for layer 0).
    __device__ __noinline__ bool prologue_A(int N) {
        const int d = p.d;
        float ss = 0.0f;
        if (N == 0) {
            for (int i = tid(); i < d; i += kT) s.stream[i] = p.x0[i];
            if (!sync()) return false;
            stage_plain<BITS>(s.stream, d, s.xf, s.xsc, s.xhat);
            if (BITS != 4) stage_plain<4>(s.stream, d, s.xf4, s.xsc4, s.xhat4);
            inv = 1.0f;
            return sync();
        }
        const uint64_t *out = tagged(p, p.off_out);
        if (!poll_chunks<BITS>(out, 1, d, tag(N - 1), s.xf, s.xsc, s.xhat, s.stream, &ss))
            return false;
        ss = warp_sum(ss, 32);
        if (lane == 0) s.misc[warp] = ss;
        if (!sync()) return false;
        if (BITS != 4) stage_plain<4>(s.stream, d, s.xf4, s.xsc4, s.xhat4);
        float tot = 0.0f;
        for (int w = 0; w < kNW; w++) tot += s.misc[w];
        inv = 1.0f / sqrtf(tot / d + 1e-6f);
        if (BITS != 4) return sync();
        return true;
    }

    // Everything phase B needs from other CTAs, polled together: h of every
    // slot, gelu(fc1 f), l f of this CTA's fc2 rows, and the partial A_d h of
    // down-LoRA slots; plus this CTA's rows of the down-LoRA B matrices.
    __device__ __noinline__ bool prologue_B(int N, const Tmplt &ta, const Tmplt &tb) {
        const uint32_t tg = tag(N);
        const LayerP &L = layer_of(p, N);
        const int *route = s.rcur + N * p.K;
        float ss = 0.0f;
        // B_d rows of this CTA's outputs (plain loads, issued first)
        if (p.rd) {
            const int no = tb.o_hi - tb.o_lo;
            for (int sl = 0; sl < p.S; sl++) {
                const LoraP &l = slot_lora(p, L, sl, 2);
                if (!l.r) continue;
                const uint16_t *B = lora_bm(p, L, route, sl, 2);
                for (int i = tid(); i < no * l.r; i += kT)
                    s.bd[(sl * p.max_orows + i / l.r) * p.rd + i % l.r] =
                        half_f(B[(size_t)(tb.o_lo + i / l.r) * l.r + i % l.r]);
            }
        }
        bool lok = poll_chunks<BITS>(tagged(p, p.off_h), p.S, p.F, tg, s.hf, s.hsc, s.hhat, nullptr, &ss);
        const bool fc2 = head_runs(p, N) && p.H > 0;
        if (fc2 && lok)
            lok = poll_chunks<4>(tagged(p, p.off_ga), 1, p.H, tg, s.gf, s.gsc, s.ghat, nullptr, &ss);
        if (fc2 && lok && tb.e_hi > tb.e_lo) {
            const int n = tb.e_hi - tb.e_lo;
            for (int i0 = tid(); i0 < n && lok; i0 += 8 * kT) {
                int idx[8];
                float val[8];
                int cnt = 0;
                for (int k = 0; k < 8; k++) {
                    const int i = i0 + k * kT;
                    idx[k] = tb.e_lo + (i < n ? i : 0);
                    if (i < n) cnt = k + 1;
                }
                lok = poll_set(p, tagged(p, p.off_zl), idx, cnt, tg, val);
                for (int k = 0; k < cnt; k++) s.zl[i0 + k * kT] = val[k];
            }
        }
        if (p.rd && lok) {
            // partial A_d h of down-LoRA slots from their gate/up owners
            int base = 0;
            for (int sl = 0; sl < p.S && lok; sl++) {
                const int r = slot_lora(p, L, sl, 2).r;
                if (!r) continue;
                const int n = (ta.own1[sl] - ta.own0[sl] + 1) * r;
                const uint64_t *w = tagged(p, p.off_vdp) + (size_t)sl * p.n_cta * kMaxLoraRank;
                for (int i0 = tid(); i0 < n && lok; i0 += 8 * kT) {
                    int idx[8];
                    float val[8];
                    int cnt = 0;
                    for (int k = 0; k < 8; k++) {
                        const int i = i0 + k * kT;
                        const int ii = i < n ? i : 0;
                        idx[k] = (ta.own0[sl] + ii / r) * kMaxLoraRank + ii % r;
                        if (i < n) cnt = k + 1;
                    }
                    lok = poll_set(p, w, idx, cnt, tg, val);
                    for (int k = 0; k < cnt; k++) s.vdp[base + i0 + k * kT] = val[k];
                }
                base += n;
            }
        }
        if (!__all_sync(0xffffffffu, lok)) return false;
        if (!sync()) return false;
        if (p.rd && warp == 0) {
            // vd[s][k] = sum over owners (ascending) of the partials
            int base = 0;
            for (int sl = 0; sl < p.S; sl++) {
                const int r = slot_lora(p, L, sl, 2).r;
                if (!r) continue;
                const int no = ta.own1[sl] - ta.own0[sl] + 1;
                for (int k = lane; k < r; k += 32) {
                    float a = 0.0f;
                    for (int o = 0; o < no; o++) a += s.vdp[base + o * r + k];
                    s.vd[sl * kMaxLoraRank + k] = a;
                }
                base += no * r;
            }
        }
        return true;
    }

    // ---- tasks -------------------------------------------------------
    // Gate/up row pairs: h = silu(g) * u (+ gate/up LoRA), published; the
    // partial A_d h of down-LoRA slots accumulates in vdp_acc (lane k of
    // every row group holds component k).
    __device__ __noinline__ void task_gu(int N, const Grp &g, const uint8_t *base, int i, int cnt, int lpr) {
        const int sub = lane % lpr, rsub = lane / lpr;
        const int f = i + rsub;
        const bool ok = rsub < cnt;
        const LayerP &L = layer_of(p, N);
        const int *route = s.rcur + N * p.K;
        const int sl = g.slot;
        const uint32_t tg = tag(N);
        const LoraP &lg = slot_lora(p, L, sl, 0), &lu = slot_lora(p, L, sl, 1),
                    &ld = slot_lora(p, L, sl, 2);
        // LoRA operands for this row, loaded before the dot product
        float bg = 0.0f, bu = 0.0f, ad = 0.0f;
        if (ok && sub < lg.r) bg = half_f(lora_bm(p, L, route, sl, 0)[(size_t)f * lg.r + sub]);
        if (ok && sub < lu.r) bu = half_f(lora_bm(p, L, route, sl, 1)[(size_t)f * lu.r + sub]);
        if (ok && sub < ld.r) ad = half_f(lora_a(p, L, route, sl, 2)[(size_t)sub * p.F + f]);
        float r2[2];
        rows_dot<BITS, 2>(base + (size_t)(rsub < cnt ? rsub : 0) * g.item_bytes, p.rec_d, p.d, s.xf,
                          s.xsc, s.xhat, sub, lpr, r2);
        float gg = r2[0] * inv, uu = r2[1] * inv;
        if (lg.r || lu.r) {
            // this lane's components of A_g x and A_u x
            int idx[2];
            float val[2] = {0.0f, 0.0f};
            int n = 0, at_g = -1, at_u = -1;
            if (ok && sub < lg.r) {
                at_g = n;
                idx[n++] = (sl * 2 + 0) * kMaxLoraRank + sub;
            }
            if (ok && sub < lu.r) {
                at_u = n;
                idx[n++] = (sl * 2 + 1) * kMaxLoraRank + sub;
            }
            if (n) poll_set(p, tagged(p, p.off_v), idx, n, tg, val);
            const float vg = at_g >= 0 ? val[at_g] : 0.0f;
            const float vu = at_u >= 0 ? val[at_u] : 0.0f;
            gg += lg.scale * warp_sum(bg * vg, lpr);
            uu += lu.scale * warp_sum(bu * vu, lpr);
        }
        const float h = silu_f(gg) * uu;
        if (ok && sub == 0) put_tagged(tagged(p, p.off_h) + (size_t)sl * p.F + f, tg, h);
        if (ld.r) {
            const float hf = __shfl_sync(0xffffffffu, h, rsub * lpr);
            if (ok) {
                if (sl & 1) vdp1 = fmaf(ad, hf, vdp1);
                else vdp0 = fmaf(ad, hf, vdp0);
            }
        }
    }

    // fc1 / l / router rows on x, with the K-hot table rows and the bias.
    __device__ __noinline__ void task_head(int N, const Grp &g, const uint8_t *base, int i, int cnt, int lpr) {
        const int sub = lane % lpr, rsub = lane / lpr;
        const int row = i + rsub;
        const bool ok = rsub < cnt;
        const LayerP &L = layer_of(p, N);
        const int *cur = s.rcur + N * p.K;
        const int *prev = p.t > 0 ? s.rprev + N * p.K : nullptr;
        const uint16_t *tab = g.kind == KFC1 ? L.fc1_tab : (g.kind == KLX ? L.l_tab : nullptr);
        const int width = g.kind == KFC1 ? p.H : p.E;
        const uint16_t *bias = g.kind == KFC1 ? L.b1 : (g.kind == KLX ? L.bl : nullptr);
        // table rows of the 2K active one-hot columns: lanes of the row group
        float gv = 0.0f;
        if (ok && tab)
            for (int k = sub; k < 2 * p.K; k += lpr) {
                const int e = k < p.K ? cur[k] : (prev ? prev[k - p.K] : -1);
                if ((unsigned)e < (unsigned)p.E)
                    gv += half_f(tab[(size_t)(k < p.K ? e : p.E + e) * width + row]);
            }
        const float b = (ok && sub == 0 && bias) ? half_f(bias[row]) : 0.0f;
        const uint8_t *xf = BITS == 4 ? s.xf : s.xf4;
        const float *xsc = BITS == 4 ? s.xsc : s.xsc4;
        const float *xhat = BITS == 4 ? s.xhat : s.xhat4;
        float a;
        rows_dot<4, 1>(base + (size_t)(rsub < cnt ? rsub : 0) * g.item_bytes, 0, p.d, xf, xsc, xhat,
                       sub, lpr, &a);
        const float gsum = tab ? warp_sum(gv, lpr) : 0.0f;
        if (ok && sub == 0) {
            a = a * inv + gsum + b;
            const uint32_t tg = tag(N);
            if (g.kind == KFC1) put_tagged(tagged(p, p.off_ga) + row, tg, gelu_erf_f(a));
            else if (g.kind == KLX) {
                if (p.H > 0) put_tagged(tagged(p, p.off_zl) + row, tg, a);
                else put_tagged(tagged(p, p.off_z) + (size_t)N * p.E + row, tg, a);
            } else
                put_tagged(tagged(p, p.off_zr) + row, tag_router(), a);
        }
    }

    // LoRA A rows on x: v = A x, published.
    __device__ __noinline__ void task_la(int N, const Grp &g, const uint8_t *base, int i, int cnt, int lpr) {
        const int sub = lane % lpr, rsub = lane / lpr;
        const float a = f16_row_dot_s(base + (size_t)(rsub < cnt ? rsub : 0) * g.item_bytes, p.d, s.stream, sub, lpr);
        if (rsub < cnt && sub == 0)
            put_tagged(tagged(p, p.off_v) + ((size_t)g.slot * 2 + g.aux) * kMaxLoraRank + i + rsub,
                       tag(N), a * inv);
    }

    __device__ __noinline__ void task_down(int N, const Grp &g, const Tmplt &t, const uint8_t *base, int i,
                              int cnt, int lpr) {
        const int sub = lane % lpr, rsub = lane / lpr;
        float a;
        rows_dot<BITS, 1>(base + (size_t)(rsub < cnt ? rsub : 0) * g.item_bytes, 0, p.F,
                          s.hf + (size_t)g.slot * p.F * 2, s.hsc + g.slot * (p.F / VALS),
                          s.hhat + g.slot * (p.F / VALS), sub, lpr, &a);
        if (rsub < cnt && sub == 0) s.y[g.slot * p.max_orows + (i + rsub - t.o_lo)] = a;
    }

    __device__ __noinline__ void task_fc2(int N, const Grp &g, const Tmplt &t, const uint8_t *base, int i,
                             int cnt, int lpr) {
        const int sub = lane % lpr, rsub = lane / lpr;
        const int e = i + rsub;
        const LayerP &L = layer_of(p, N);
        const float b = (rsub < cnt && sub == 0 && L.b2) ? half_f(L.b2[e]) : 0.0f;
        float a;
        rows_dot<4, 1>(base + (size_t)(rsub < cnt ? rsub : 0) * g.item_bytes, 0, p.H, s.gf, s.gsc,
                       s.ghat, sub, lpr, &a);
        if (rsub < cnt && sub == 0)
            put_tagged(tagged(p, p.off_z) + (size_t)N * p.E + e, tag(N), a + b + s.zl[e - t.e_lo]);
    }

    // Consumes this CTA's pieces of groups [g0, g1) of t, in the producer's
    // order; warp tasks of rpw items go round-robin to the consumer warps.
    __device__ __noinline__ bool run(int N, const Tmplt &t, int g0, int g1) {
        uint32_t tasks = 0;
        for (int gi = g0; gi < g1; gi++) {
            const Grp &g = t.g[gi];
            const int per = max(1, kMaxPiece / (int)g.item_bytes);
            const int lpr = pow2_floor32(item_chunks<BITS>(g));
            const int rpw = 32 / lpr;
            for (int i0 = g.lo; i0 < g.hi; i0 += per) {
                const int cnt = min(per, g.hi - i0);
                const uint64_t start = rp.place((uint32_t)cnt * g.item_bytes, p.ring_bytes);
                const uint32_t q = rp.q++;
                if (!wait_bar_warp(p, s.full + q % kNB, (q / kNB) & 1)) return false;
                const uint8_t *base = s.ring + start % p.ring_bytes;
                const int ntask = (cnt + rpw - 1) / rpw;
                for (int k = (int)((kNW + warp - tasks % kNW) % kNW); k < ntask; k += kNW) {
                    const int li = k * rpw;
                    const uint8_t *b = base + (size_t)li * g.item_bytes;
                    const int n = min(rpw, cnt - li);
                    const bool tr = g.kind == KGU && trace_gu == 0 && p.trace;
                    if (tr) stamp(N, 15);
                    switch (g.kind) {
                        case KGU: task_gu(N, g, b, i0 + li, n, lpr); break;
                        case KFC1:
                        case KLX:
                        case KROUTER: task_head(N, g, b, i0 + li, n, lpr); break;
                        case KLA: task_la(N, g, b, i0 + li, n, lpr); break;
                        case KDOWN: task_down(N, g, t, b, i0 + li, n, lpr); break;
                        default: task_fc2(N, g, t, b, i0 + li, n, lpr); break;
                    }
                    if (tr) {
                        trace_gu = 1;
                        if (warp == 0 && lane == 0) {
                            const size_t at = ((size_t)c * p.depth + N) * kTrace + 15;
                            p.trace[at] = now_ns() - p.trace[at];
                        }
                    }
                }
                tasks += ntask;
                __syncwarp();
                if (lane == 0) mbar_arrive(s.empty + q % kNB);
            }
        }
        return true;
    }

    // Layer 0's own route: poll the router logits, top-K (every CTA alike).
    __device__ __noinline__ bool route0() {
        if (warp == 0) {
            float vals[32];
            if (!poll_logits(p, tagged(p, p.off_zr), p.E, tag_router(), lane, vals)) return false;
            int idx[kMaxK];
            float w[kMaxK], margin;
            warp_topk(vals, p.E, p.K, lane, idx, w, &margin);
            if (lane == 0) {
                const int use = p.t % 3;
                for (int k = 0; k < p.K; k++) {
                    s.rcur[k] = idx[k];
                    s.rw[k] = w[k];
                    if (c == 0) {
                        p.ridx[(size_t)use * p.depth * p.K + k] = idx[k];
                        p.rw[(size_t)use * p.depth * p.K + k] = w[k];
                    }
                }
                if (c == 0) p.rmargin[(size_t)use * p.depth] = margin;
                mbar_arrive(s.route_bar);
            }
        }
        return sync();
    }

    // Publishes this CTA's partial A_d h for every down-LoRA slot whose
    // gate/up rows it helps own (zeros if it owns none of them).
    __device__ __noinline__ bool publish_vdp(int N, const Tmplt &ta) {
        const LayerP &L = layer_of(p, N);
        // per-warp partials: lane k of row group 0 after folding the row
        // groups (every row group of a gate/up task has the lpr of d); a CTA
        // spans at most two down-LoRA slots, kept apart by slot parity
        const int lpr = pow2_floor32(p.d * BITS / 128);
        for (int par = 0; par < 2; par++) {
            float v = par ? vdp1 : vdp0;
            for (int o = lpr; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane < lpr) s.misc[16 + (par * kNW + warp) * 32 + lane] = v;
        }
        vdp0 = vdp1 = 0.0f;
        if (!sync()) return false;
        const uint32_t tg = tag(N);
        for (int sl = 0; sl < p.S; sl++) {
            const int r = slot_lora(p, L, sl, 2).r;
            if (!r || c < ta.own0[sl] || c > ta.own1[sl]) continue;
            for (int k = tid(); k < r; k += kT) {
                float a = 0.0f;
                for (int w = 0; w < kNW; w++) a += s.misc[16 + ((sl & 1) * kNW + w) * 32 + k];
                put_tagged(tagged(p, p.off_vdp) + ((size_t)sl * p.n_cta + c) * kMaxLoraRank + k, tg,
                           a);
            }
        }
        return true;
    }

    // Combine + residual over this CTA's output rows; publishes out.
    __device__ __noinline__ void combine(int N, const Tmplt &t) {
        const uint32_t tg = tag(N);
        const float *w = s.rw + N * p.K;
        const LayerP &L = layer_of(p, N);
        for (int o = t.o_lo + tid(); o < t.o_hi; o += kT) {
            const int li = o - t.o_lo;
            float v = s.stream[o];
            for (int sl = 0; sl < p.S; sl++) {
                float ys = s.y[sl * p.max_orows + li];
                const LoraP &l = slot_lora(p, L, sl, 2);
                if (l.r) {
                    float a = 0.0f;
                    for (int k = 0; k < l.r; k++)
                        a = fmaf(s.bd[(sl * p.max_orows + li) * p.rd + k], s.vd[sl * kMaxLoraRank + k], a);
                    ys += l.scale * a;
                }
                v = sl < p.K ? fmaf(w[sl], ys, v) : v + ys;
            }
            put_tagged(tagged(p, p.off_out) + o, tg, v);
            if (N == p.depth - 1) p.out[o] = v;
        }
    }

    __device__ bool layer(int N) {
        trace_gu = 0;
        stamp(N, 0);
        if (!prologue_A(N)) return false;
        stamp(N, 1);
        if (N == 0 && p.own0) {
            if (!run(0, s.T[T_R], 0, s.T[T_R].n)) return false;
            if (!route0()) return false;
        }
        const Tmplt &ta = tmpl_A(p, s.T, N), &tb = tmpl_B(p, s.T, N);
        if (!run(N, ta, 0, ta.n)) return false;
        stamp(N, 2);
        if (p.rd && !publish_vdp(N, ta)) return false;
        if (!prologue_B(N, ta, tb)) return false;
        stamp(N, 3);
        if (!sync()) return false;              // h, ga and vd visible to all warps
        stamp(N, 4);
        const int nd = head_runs(p, N) && p.H > 0 ? tb.n - 1 : tb.n;
        if (!run(N, tb, 0, nd)) return false;   // down rows
        stamp(N, 6);
        if (!sync()) return false;
        combine(N, tb);
        stamp(N, 7);
        if (!run(N, tb, nd, tb.n)) return false;  // head fc2 rows
        stamp(N, 8);
        return true;
    }

    __device__ bool run_all() {
        if (p.debug_unset_wait && c == 0 && warp == 0) {
            // test hook: a flag nothing ever sets, so this wait runs out
            float v;
            int idx = 0;
            const bool lok = poll_set(p, tagged(p, C_NEVER * 4), &idx, 1, 0xFFFFFFFFu, &v);
            if (!__all_sync(0xffffffffu, lok)) return false;
        }
        for (int N = 0; N < p.depth; N++)
            if (!layer(N)) return false;
        return true;
    }
};

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const Smem s = smem_views(p, smem);
    const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // routes of this step (layer 0's own route is filled in later)
    const int use = p.t % 3, prv = (p.t + 2) % 3;
    for (int i = threadIdx.x; i < p.depth * p.K; i += blockDim.x) {
        s.rcur[i] = p.ridx[(size_t)use * p.depth * p.K + i];
        s.rw[i] = p.rw[(size_t)use * p.depth * p.K + i];
        s.rprev[i] = p.ridx[(size_t)prv * p.depth * p.K + i];
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNB; i++) {
            mbar_init(s.full + i, 1);
            mbar_init(s.empty + i, kNW);
        }
        mbar_init(s.route_bar, 1);
        mbar_init(s.cons_bar, kNW);
        mbar_init(s.end_bar, kCons0 + kNW);
        mbar_fence_init();
        build_templates(p, c, s.T);
    }
    __syncthreads();

    if (warp == kProducerWarp) {
        if (lane == 0) producer<BITS>(p, s);
    } else if (warp == kRouteWarp) {
        route_warp(p, c, lane);
    } else {
        Consumer<BITS> cons{p, s, c, warp - kCons0, lane, (uint32_t)ld_flag(ctrl(p) + C_EPOCH)};
        cons.run_all();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(s.end_bar);
    if (threadIdx.x == 0) {
        // the step is complete in this CTA once every warp has arrived
        if (wait_bar(p, s.end_bar, 0) && !aborted(p)) {
            __threadfence();
            const int prev = atomicAdd(ctrl(p) + C_DONE, 1);
            if (prev == p.n_cta - 1) {
                atomicExch(ctrl(p) + C_DONE, 0);
                atomicAdd(ctrl(p) + C_EPOCH, 1);
            }
        }
    }
}

}  // namespace step

// ---------------------------------------------------------------- host side
using namespace step;

static size_t al(size_t v, size_t a) { return (v + a - 1) / a * a; }

static void step_ws_layout(int d, int F, int E, int H, int S, int depth, int n_cta,
                           uint32_t *offs, size_t *total) {
    size_t off = kCtrlBytes;
    auto take = [&](size_t n) {
        const size_t o = off;
        off = al(off + n * sizeof(uint64_t), 256);
        return (uint32_t)o;
    };
    offs[0] = take((size_t)S * F);                          // h
    offs[1] = take((size_t)S * 2 * kMaxLoraRank);           // LoRA A x (gate, up)
    offs[2] = take((size_t)S * n_cta * kMaxLoraRank);       // partial A_d h per owner CTA
    offs[3] = take((size_t)(H > 0 ? H : 1));                // gelu(fc1 f)
    offs[4] = take((size_t)E);                              // l f
    offs[5] = take((size_t)E);                              // router logits
    offs[6] = take((size_t)depth * E);                      // head logits per layer
    offs[7] = take((size_t)d);                              // out
    *total = off;
}

static int launch_decode_step(const moe_stack_desc *sd, const float *x0, float *out,
                              int32_t *ridx, float *rw, float *rmargin, int t, void *ws,
                              cudaStream_t st);

static int device_sms() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

}  // namespace moe

using namespace moe;

static int check_stack(const moe_stack_desc *sd) {
    if (sd == nullptr || sd->experts == nullptr || sd->routers == nullptr)
        return fail(MOE_EINVAL, "decode_step: NULL descriptor");
    if (sd->n_layers < 1 || sd->n_layers > kMaxLayers || sd->depth < 1 || sd->depth > kMaxLayers)
        return fail(MOE_EINVAL, "decode_step: n_layers=%d depth=%d (1..%d)", sd->n_layers, sd->depth,
                    kMaxLayers);
    if (sd->K < 1 || sd->K > kMaxK) return fail(MOE_EINVAL, "decode_step: K=%d", sd->K);
    if (sd->self_predict && sd->depth != 1)
        return fail(MOE_EINVAL, "decode_step: self_predict needs depth 1");
    const bool heads = sd->depth > 1 || sd->self_predict;
    if (heads && sd->heads == nullptr) return fail(MOE_EINVAL, "decode_step: heads are NULL");
    const moe_experts_desc &e0 = sd->experts[0];
    if (e0.d <= 0 || e0.d % 64 || e0.F <= 0 || e0.F % 64 || (e0.bits != 2 && e0.bits != 4) ||
        e0.E < sd->K || e0.E > 1024)
        return fail(MOE_EINVAL, "decode_step: expert shape d=%d F=%d E=%d bits=%d", e0.d, e0.F,
                    e0.E, e0.bits);
    const int H = heads ? sd->heads[0].H : 0;
    int down_lora_slots = 0;
    for (int i = 0; i < sd->n_layers; i++) {
        const moe_experts_desc &e = sd->experts[i];
        if (e.d != e0.d || e.F != e0.F || e.E != e0.E || e.bits != e0.bits ||
            (e.shared == nullptr) != (e0.shared == nullptr) || e.pool == nullptr ||
            e.expert_stride != e0.expert_stride)
            return fail(MOE_EINVAL, "decode_step: layer %d differs in shape from layer 0", i);
        if (e.expert_stride < blob_layout(e.d, e.F, e.bits).bytes || e.expert_stride % 256)
            return fail(MOE_EINVAL, "decode_step: expert_stride %zu", e.expert_stride);
        for (int j = 0; j < 3; j++) {
            const int r0 = e.lora[j].r, r1 = e.shared ? e.shared_lora[j].r : 0;
            const int q0 = e0.lora[j].r, q1 = e0.shared ? e0.shared_lora[j].r : 0;
            if (r0 != q0 || r1 != q1 || r0 < 0 || r0 > 32 || r1 < 0 || r1 > 32)
                return fail(MOE_EUNSUPPORTED,
                            "decode_step: LoRA ranks must match across layers and be <= 32");
            if ((r0 && (!e.lora[j].A || !e.lora[j].B)) ||
                (r1 && (!e.shared_lora[j].A || !e.shared_lora[j].B)))
                return fail(MOE_EINVAL, "decode_step: LoRA with NULL A or B");
        }
        const moe_head_desc &r = sd->routers[i];
        if (r.d != e0.d || r.E != e0.E || r.lx == nullptr)
            return fail(MOE_EINVAL, "decode_step: router %d shape", i);
        if (r.prec != MOE_PREC_AFFINE4)
            return fail(MOE_EUNSUPPORTED, "decode_step: fp16 routers run through the per-call path");
        if (heads) {
            const moe_head_desc &h = sd->heads[i];
            if (h.d != e0.d || h.E != e0.E || h.H != H || h.H < 0 || h.H % 64 || h.lx == nullptr ||
                (h.H > 0 && (h.fc1x == nullptr || h.fc2 == nullptr)))
                return fail(MOE_EINVAL, "decode_step: head %d shape", i);
            if (h.prec != MOE_PREC_AFFINE4)
                return fail(MOE_EUNSUPPORTED, "decode_step: fp16 heads run through the per-call path");
        }
    }
    down_lora_slots = (e0.lora[2].r ? sd->K : 0) + (e0.shared && e0.shared_lora[2].r ? 1 : 0);
    if (down_lora_slots > 1 && (e0.lora[2].r || e0.shared_lora[2].r)) {
        // one CTA owning gate/up rows of two down-LoRA slots would mix their
        // partials; the split keeps slots apart only when each slot's rows
        // span whole CTAs, which the host cannot promise in general
        if (e0.d < 64) return fail(MOE_EUNSUPPORTED, "decode_step: down-LoRA layout");
    }
    return MOE_OK;
}

extern "C" size_t moe_decode_step_workspace_bytes(const moe_stack_desc *sd) {
    if (check_stack(sd) != MOE_OK) return 0;
    const moe_experts_desc &e0 = sd->experts[0];
    const int H = (sd->depth > 1 || sd->self_predict) ? sd->heads[0].H : 0;
    uint32_t offs[8];
    size_t total = 0;
    const int sms = device_sms();
    step_ws_layout(e0.d, e0.F, e0.E, H, sd->K + (e0.shared ? 1 : 0), sd->depth,
                   sms > 0 ? sms : 256, offs, &total);
    return total;
}

extern "C" int moe_decode_step(const moe_stack_desc *sd, const float *x0, float *out,
                               int32_t *route_idx, float *route_w, float *route_margin, int t,
                               void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (int rc = check_stack(sd)) return rc;
    if (t < 1)
        return fail(MOE_EINVAL, "decode_step: t=%d (step 0 routes every layer with its own router; "
                                "run it with the per-call functions)", t);
    if (!x0 || !out || !route_idx || !route_w || !route_margin || !ws)
        return fail(MOE_EINVAL, "decode_step: NULL pointer");
    const size_t need = moe_decode_step_workspace_bytes(sd);
    if (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 256))
        return fail(MOE_ENOSPACE, "decode_step: workspace %zu bytes, need %zu (256-aligned)",
                    ws_bytes, need);
    return launch_decode_step(sd, x0, out, route_idx, route_w, route_margin, t, ws, stream);
}

extern "C" int moe_decode_step_status(const void *ws, int *status, cudaStream_t stream) {
    if (ws == nullptr || status == nullptr)
        return fail(MOE_EINVAL, "decode_step_status: NULL pointer");
    int st[1] = {0};
    cudaError_t e = cudaMemcpyAsync(st, ws, sizeof(int), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step_status: %s", cudaGetErrorString(e));
    *status = st[0];
    return MOE_OK;
}

namespace moe {

template <int BITS>
static int launch_bits(const Params &p, size_t smem, cudaStream_t st) {
    static thread_local int configured_dev = -1;
    static thread_local size_t configured_smem = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev || configured_smem < smem) {
        cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return fail(MOE_ECUDA, "decode_step: smem attribute: %s", cudaGetErrorString(e));
        configured_dev = dev;
        configured_smem = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_cta);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_step_kernel<BITS>, p);
    if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step launch: %s", cudaGetErrorString(e));
    return MOE_OK;
}

static int launch_decode_step(const moe_stack_desc *sd, const float *x0, float *out,
                              int32_t *ridx, float *rw, float *rmargin, int t, void *ws,
                              cudaStream_t st) {
    static thread_local Params p;   // large (layer table); built per call, passed by value
    const moe_experts_desc &e0 = sd->experts[0];
    const bool heads = sd->depth > 1 || sd->self_predict;
    p = Params{};
    p.d = e0.d;
    p.F = e0.F;
    p.E = e0.E;
    p.K = sd->K;
    p.H = heads ? sd->heads[0].H : 0;
    p.S = sd->K + (e0.shared ? 1 : 0);
    p.depth = sd->depth;
    p.n_res = sd->n_layers;
    p.self_predict = sd->self_predict;
    p.own0 = !sd->self_predict;
    p.t = t;
    const int bits = e0.bits;
    const BlobLayout L = blob_layout(p.d, p.F, bits);
    p.stride = e0.expert_stride;
    p.gu_off = (uint32_t)L.gu_off;
    p.down_off = (uint32_t)L.down_off;
    p.rec_d = (uint32_t)L.gu_rec;
    p.rec_F = (uint32_t)L.down_rec;
    p.rec_dh = (uint32_t)record_bytes(p.d, 4);
    p.rec_H = p.H ? (uint32_t)record_bytes(p.H, 4) : 0;
    p.rd = std::max(e0.lora[2].r, e0.shared ? e0.shared_lora[2].r : 0);
    p.x0 = x0;
    p.out = out;
    p.ridx = ridx;
    p.rw = rw;
    p.rmargin = rmargin;
    p.ws = static_cast<uint8_t *>(ws);
    const int sms = device_sms();
    int dev = 0, smem_max = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (sms <= 0 || smem_max <= 0) return fail(MOE_ECUDA, "decode_step: no device attributes");
    p.n_cta = sms;
    uint32_t offs[8];
    size_t total = 0;
    step_ws_layout(p.d, p.F, p.E, p.H, p.S, p.depth, sms, offs, &total);
    p.off_h = offs[0];
    p.off_v = offs[1];
    p.off_vdp = offs[2];
    p.off_ga = offs[3];
    p.off_zl = offs[4];
    p.off_zr = offs[5];
    p.off_z = offs[6];
    p.off_out = offs[7];
    p.timeout_ns = sd->timeout_ns ? sd->timeout_ns : 1000000000ull;
    p.debug_unset_wait = sd->debug_unset_wait;
    p.trace = sd->debug_trace;
    for (int i = 0; i < sd->n_layers; i++) {
        const moe_experts_desc &e = sd->experts[i];
        LayerP &lp = p.layer[i];
        lp.pool = static_cast<const uint8_t *>(e.pool);
        lp.shared = static_cast<const uint8_t *>(e.shared);
        for (int j = 0; j < 3; j++) {
            lp.lora[j] = LoraP{e.lora[j].r, e.lora[j].scale, e.lora[j].A, e.lora[j].B,
                               e.lora[j].a_stride, e.lora[j].b_stride};
            lp.slora[j] = e.shared ? LoraP{e.shared_lora[j].r, e.shared_lora[j].scale,
                                          e.shared_lora[j].A, e.shared_lora[j].B, 0, 0}
                                   : LoraP{};
        }
        lp.router = static_cast<const uint8_t *>(sd->routers[i].lx);
        if (heads) {
            const moe_head_desc &h = sd->heads[i];
            lp.fc1x = static_cast<const uint8_t *>(h.fc1x);
            lp.fc1_tab = h.fc1_tab;
            lp.b1 = h.b1;
            lp.fc2 = static_cast<const uint8_t *>(h.fc2);
            lp.b2 = h.b2;
            lp.lx = static_cast<const uint8_t *>(h.lx);
            lp.l_tab = h.l_tab;
            lp.bl = h.bl;
        }
    }

    p.max_orows = (p.d + sms - 1) / sms;
    if ((p.E + sms - 1) / sms > kMaxOwnE)
        return fail(MOE_EUNSUPPORTED, "decode_step: E=%d too large for %d SMs", p.E, sms);

    // shared-memory layout
    const int VALS = 128 / bits;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        off = al(off, 16);
        const size_t o = off;
        off += bytes;
        return (uint32_t)o;
    };
    p.sm_bar = take((size_t)(2 * kNB + 3) * 8);
    p.sm_pend = take((size_t)kNB * 8);
    p.sm_tmpl = take(T_COUNT * sizeof(Tmplt));
    p.sm_xf = take((size_t)p.d * 2);
    p.sm_xsc = take((size_t)(p.d / VALS) * 4);
    p.sm_xhat = take((size_t)(p.d / VALS) * 4);
    p.sm_xf4 = bits == 4 ? p.sm_xf : take((size_t)p.d * 2);
    p.sm_xsc4 = bits == 4 ? p.sm_xsc : take((size_t)(p.d / 32) * 4);
    p.sm_xhat4 = bits == 4 ? p.sm_xhat : take((size_t)(p.d / 32) * 4);
    p.sm_stream = take((size_t)p.d * 4);
    p.sm_hf = take((size_t)p.S * p.F * 2);
    p.sm_hsc = take((size_t)p.S * (p.F / VALS) * 4);
    p.sm_hhat = take((size_t)p.S * (p.F / VALS) * 4);
    p.sm_gf = take((size_t)(p.H ? p.H : 64) * 2);
    p.sm_gsc = take((size_t)(p.H ? p.H / 32 : 2) * 4);
    p.sm_ghat = take((size_t)(p.H ? p.H / 32 : 2) * 4);
    p.sm_zl = take((size_t)kMaxOwnE * 4);
    p.sm_y = take((size_t)p.S * p.max_orows * 4);
    p.sm_bd = take((size_t)p.S * p.max_orows * (p.rd ? p.rd : 1) * 4);
    p.sm_vdp = take((size_t)(p.rd ? kMaxVdp : 1) * 4);
    p.sm_vd = take((size_t)p.S * kMaxLoraRank * 4);
    p.sm_rcur = take((size_t)p.depth * p.K * 4);
    p.sm_rprev = take((size_t)p.depth * p.K * 4);
    p.sm_rw = take((size_t)p.depth * p.K * 4);
    p.sm_misc = take((size_t)(16 + 2 * kNW * 32) * 4);
    p.sm_ring = (uint32_t)al(off, 1024);
    long long room = (long long)smem_max - (long long)p.sm_ring;
    room = room / 1024 * 1024;
    if (room < 3 * kMaxPiece)
        return fail(MOE_EUNSUPPORTED, "decode_step: shapes leave a %lld-byte ring (< 48 KiB)", room);
    p.ring_bytes = (uint32_t)room;
    const size_t smem = (size_t)p.sm_ring + p.ring_bytes;

    // every item must fit a piece; the down-LoRA partials must fit their
    // buffer (each slot's owners x rank)
    if (2 * p.rec_d > (uint32_t)kMaxPiece || 2u * p.d > (uint32_t)kMaxPiece)
        return fail(MOE_EUNSUPPORTED, "decode_step: d=%d rows exceed a %d-byte piece", p.d,
                    kMaxPiece);
    if (3 * p.S + 2 > kMaxGroups)
        return fail(MOE_EUNSUPPORTED, "decode_step: K=%d needs too many work groups", p.K);
    if (p.rd) {
        // CTAs owning gate/up rows of a slot: about the slot's share of the
        // phase bytes plus one on each side
        const long long gu_bytes = 2LL * p.rec_d * p.F;
        long long total = (long long)p.S * gu_bytes +
                          (p.H ? (long long)p.H * p.rec_dh : 0) + (long long)p.E * p.rec_dh;
        for (int sl = 0; sl < p.S; sl++)
            for (int w = 0; w < 2; w++) {
                const int r = sl < p.K ? e0.lora[w].r : (e0.shared ? e0.shared_lora[w].r : 0);
                total += 2LL * p.d * r;
            }
        const long long owners = gu_bytes * sms / total + 3;
        const int slots = (e0.lora[2].r ? p.K : 0) + (e0.shared && e0.shared_lora[2].r ? 1 : 0);
        if (owners * slots * p.rd > kMaxVdp)
            return fail(MOE_EUNSUPPORTED, "decode_step: down-LoRA partials exceed %d floats", kMaxVdp);
        // a CTA may span the gate/up rows of at most two down-LoRA slots (two
        // accumulators): each slot's rows must be at least one CTA's share
        if (slots > 1 && gu_bytes * sms < total)
            return fail(MOE_EUNSUPPORTED, "decode_step: down-LoRA slots too small to split");
        // lane k of a gate/up row group holds component k of A_d h
        if (p.rd > pow2_floor32(p.d * bits / 128))
            return fail(MOE_EUNSUPPORTED, "decode_step: down-LoRA rank %d above lanes per row", p.rd);
    }

    return bits == 4 ? launch_bits<4>(p, smem, st) : launch_bits<2>(p, smem, st);
}

}  // namespace moe
