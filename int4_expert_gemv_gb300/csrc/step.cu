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
//    ring of shared-memory slots with bulk copies (cp.async.bulk + mbarrier)
//    as far ahead as the ring allows, across layer boundaries.
//  * Dependencies between CTAs (h after gate/up, out after down, logits,
//    LoRA A-products) travel as 64-bit (tag, value) words in global memory:
//    a reader polls the words it needs until their tag is the current one.
//    There is no grid-wide barrier; each value is its own ready flag.
//  * Every CTA computes the RMS of the residual stream, and layer 0's top-K,
//    itself from the full vectors, so no reduction round trip is needed.
//  * Every wait is bounded (globaltimer); on expiry the kernel records
//    MOE_ETIMEOUT in the workspace status word, waits (bounded) for its own
//    copies in flight and returns.
//
// Work split per layer: phase A (needs x_N) = LoRA A-rows on x, gate/up row
// pairs of every slot, head fc1 rows and l rows; phase B (needs h) = LoRA
// A-rows on h, down rows (CTA c owns output rows [c*d/n, (c+1)*d/n) of every
// slot and combines them), head fc2 rows.  Phase R (layer 0 only, when it
// routes with its own router) = router rows.  A and B are split across CTAs
// by bytes; within a CTA, warp tasks go round-robin to the consumer warps.
#include <algorithm>

#include "step_common.cuh"

namespace moe {
namespace step {

constexpr int kMaxLayers = 48;
constexpr int kNW = 12;                        // consumer warps
constexpr int kProducerWarp = 0, kRouteWarp = 1, kCons0 = 2;
constexpr int kThreads = (kCons0 + kNW) * 32;  // 448
constexpr int kSlotBytes = 16384;
constexpr int kMaxRing = 16;
constexpr int kMaxK = 16;
constexpr int kMaxS = kMaxK + 1;
constexpr int kMaxGroups = 64;

enum Kind : uint8_t { KLA = 0, KGU, KFC1, KLX, KROUTER, KLD, KDOWN, KFC2 };
enum PhaseId : int { PR = 0, PA = 1, PB = 2 };

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
    int d, F, E, K, H, S, depth, n_res, self_predict, own0, t, n_cta, n_slots, max_orows;
    size_t stride;
    uint32_t gu_off, down_off, rec_d, rec_F, rec_dh, rec_H;
    const float *x0;
    float *out;
    int32_t *ridx;
    float *rw, *rmargin;
    uint8_t *ws;
    uint32_t off_h, off_v, off_vd, off_ga, off_zl, off_zr, off_z, off_out;
    uint64_t timeout_ns;
    int debug_unset_wait;
    // shared-memory layout (byte offsets from the dynamic base)
    uint32_t sm_ring, sm_bar, sm_plan, sm_x, sm_xps, sm_xps4, sm_xsum, sm_xsum4, sm_stream,
        sm_h, sm_hps, sm_hsum, sm_ga, sm_gps, sm_gsum, sm_y, sm_rcur, sm_rprev, sm_rw, sm_misc;
    LayerP layer[kMaxLayers];
};

struct Grp {
    const uint8_t *src;    // address of item 0
    uint32_t item_bytes;
    int n;                 // items in the group
    int lo, hi;            // this CTA's item range
    uint8_t kind, slot, aux, pad;
    int cols;
};

struct Plan {
    Grp g[kMaxGroups];
    int n;
    int o_lo, o_hi;        // phase B: this CTA's output rows
};

// ---------------------------------------------------------------- control
__device__ __forceinline__ int *ctrl(const Params &p) { return reinterpret_cast<int *>(p.ws); }

__device__ __forceinline__ void raise_error(const Params &p, int code) {
    atomicCAS(ctrl(p) + C_STATUS, 0, code);
    atomicExch(ctrl(p) + C_ABORT, 1);
}

__device__ __forceinline__ bool aborted(const Params &p) { return ld_flag(ctrl(p) + C_ABORT) != 0; }

// Warp-collective bounded wait on an mbarrier phase: every lane observes the
// phase, and the warp leaves together; false (error recorded) on timeout or
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

// Bounded poll of one tagged word; returns false on timeout/abort.
__device__ __forceinline__ bool poll_tag(const Params &p, const uint64_t *w, uint32_t tag,
                                         float *v) {
    uint64_t x = get_word(w);
    if ((uint32_t)(x >> 32) == tag) {
        *v = __uint_as_float((uint32_t)x);
        return true;
    }
    const uint64_t t0 = now_ns();
    for (int it = 1;; it++) {
        x = get_word(w);
        if ((uint32_t)(x >> 32) == tag) {
            *v = __uint_as_float((uint32_t)x);
            return true;
        }
        if ((it & 15) == 0) {
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

// ---------------------------------------------------------------- plans
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

__device__ __forceinline__ void add_group(Plan &pl, const uint8_t *src, uint32_t ib, int n, int kind,
                                          int slot, int aux, int cols) {
    Grp &g = pl.g[pl.n++];
    g.src = src;
    g.item_bytes = ib;
    g.n = n;
    g.lo = 0;
    g.hi = 0;
    g.kind = (uint8_t)kind;
    g.slot = (uint8_t)slot;
    g.aux = (uint8_t)aux;
    g.cols = cols;
}

// Item ranges of groups [first, last) under an even split of their bytes.
__device__ void split_bytes(Plan &pl, int first, int last, int c, int n_cta) {
    long long total = 0;
    for (int i = first; i < last; i++) total += (long long)pl.g[i].n * pl.g[i].item_bytes;
    const long long a = total * c / n_cta, b = total * (c + 1) / n_cta;
    long long base = 0;
    for (int i = first; i < last; i++) {
        Grp &g = pl.g[i];
        const long long ib = g.item_bytes;
        auto first_at = [&](long long x) -> int {
            if (x <= base) return 0;
            long long k = (x - base + ib - 1) / ib;
            return (int)(k < g.n ? k : g.n);
        };
        g.lo = first_at(a);
        g.hi = first_at(b);
        base += (long long)g.n * ib;
    }
}

// Builds this CTA's plan of phase `ph` of layer N.  `route` = layer N's route.
__device__ void make_plan(const Params &p, int N, int ph, const int *route, int c, Plan &pl) {
    const LayerP &L = layer_of(p, N);
    pl.n = 0;
    pl.o_lo = pl.o_hi = 0;
    if (ph == PR) {
        add_group(pl, L.router, p.rec_dh, p.E, KROUTER, 0, 0, p.d);
        split_bytes(pl, 0, pl.n, c, p.n_cta);
        return;
    }
    if (ph == PA) {
        for (int s = 0; s < p.S; s++)
            for (int w = 0; w < 2; w++) {
                const LoraP &l = slot_lora(p, L, s, w);
                if (l.r)
                    add_group(pl,
                              reinterpret_cast<const uint8_t *>(
                                  l.A + (s < p.K ? (size_t)route[s] * l.as : 0)),
                              2u * p.d, l.r, KLA, s, w, p.d);
            }
        for (int s = 0; s < p.S; s++)
            add_group(pl, slot_blob(p, L, route, s) + p.gu_off, 2u * p.rec_d, p.F, KGU, s, 0, p.d);
        if (head_runs(p, N)) {
            if (p.H) add_group(pl, L.fc1x, p.rec_dh, p.H, KFC1, 0, 0, p.d);
            add_group(pl, L.lx, p.rec_dh, p.E, KLX, 0, 0, p.d);
        }
        split_bytes(pl, 0, pl.n, c, p.n_cta);
        return;
    }
    // phase B: LoRA A-rows on h, then down rows of every slot, then fc2 rows.
    for (int s = 0; s < p.S; s++) {
        const LoraP &l = slot_lora(p, L, s, 2);
        if (l.r)
            add_group(pl,
                      reinterpret_cast<const uint8_t *>(l.A + (s < p.K ? (size_t)route[s] * l.as : 0)),
                      2u * p.F, l.r, KLD, s, 0, p.F);
    }
    const int n_ld = pl.n;
    const bool fc2 = head_runs(p, N) && p.H > 0;
    if (fc2) add_group(pl, L.fc2, p.rec_H, p.E, KFC2, 0, 0, p.H);
    split_bytes(pl, 0, pl.n, c, p.n_cta);
    Grp fc2g;
    if (fc2) fc2g = pl.g[--pl.n];
    pl.o_lo = (int)((long long)p.d * c / p.n_cta);
    pl.o_hi = (int)((long long)p.d * (c + 1) / p.n_cta);
    for (int s = 0; s < p.S; s++) {
        add_group(pl, slot_blob(p, L, route, s) + p.down_off, p.rec_F, p.d, KDOWN, s, 0, p.F);
        pl.g[pl.n - 1].lo = pl.o_lo;
        pl.g[pl.n - 1].hi = pl.o_hi;
    }
    if (fc2) pl.g[pl.n++] = fc2g;
    (void)n_ld;
}

__device__ __forceinline__ int pow2_floor32(int n) {
    int l = 1;
    while (l * 2 <= n && l < 32) l *= 2;
    return l;
}

template <int BITS>
__device__ __forceinline__ int item_chunks(const Grp &g) {
    switch (g.kind) {
        case KGU:
        case KDOWN: return g.cols * BITS / 128;
        case KLA:
        case KLD: return g.cols / 8;
        default: return g.cols / 32;              // int4 head rows
    }
}

// ---------------------------------------------------------------- smem views
struct Smem {
    uint8_t *ring;
    uint64_t *full, *empty, *route_bar, *cons_bar, *end_bar;
    Plan *plan_c, *plan_p;
    float *x, *xps, *xps4, *xsum, *xsum4, *stream;
    float *h, *hps, *hsum, *ga, *gps, *gsum, *y;
    int *rcur, *rprev;
    float *rw, *misc;
};

__device__ __forceinline__ Smem smem_views(const Params &p, uint8_t *base) {
    Smem s;
    s.ring = base + p.sm_ring;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + p.sm_bar);
    s.full = bars;
    s.empty = bars + p.n_slots;
    s.route_bar = bars + 2 * p.n_slots;
    s.cons_bar = s.route_bar + 1;
    s.end_bar = s.route_bar + 2;
    s.plan_c = reinterpret_cast<Plan *>(base + p.sm_plan);
    s.plan_p = s.plan_c + 1;
    s.x = reinterpret_cast<float *>(base + p.sm_x);
    s.xps = reinterpret_cast<float *>(base + p.sm_xps);
    s.xps4 = reinterpret_cast<float *>(base + p.sm_xps4);
    s.xsum = reinterpret_cast<float *>(base + p.sm_xsum);
    s.xsum4 = reinterpret_cast<float *>(base + p.sm_xsum4);
    s.stream = reinterpret_cast<float *>(base + p.sm_stream);
    s.h = reinterpret_cast<float *>(base + p.sm_h);
    s.hps = reinterpret_cast<float *>(base + p.sm_hps);
    s.hsum = reinterpret_cast<float *>(base + p.sm_hsum);
    s.ga = reinterpret_cast<float *>(base + p.sm_ga);
    s.gps = reinterpret_cast<float *>(base + p.sm_gps);
    s.gsum = reinterpret_cast<float *>(base + p.sm_gsum);
    s.y = reinterpret_cast<float *>(base + p.sm_y);
    s.rcur = reinterpret_cast<int *>(base + p.sm_rcur);
    s.rprev = reinterpret_cast<int *>(base + p.sm_rprev);
    s.rw = reinterpret_cast<float *>(base + p.sm_rw);
    s.misc = reinterpret_cast<float *>(base + p.sm_misc);
    return s;
}

// Consumer-warp barrier (an mbarrier with kNW arrivals, bounded wait).
struct ConsSync {
    uint32_t n = 0;
    __device__ bool sync(const Params &p, const Smem &s, int lane) {
        __syncwarp();
        if (lane == 0) mbar_arrive(s.cons_bar);
        const bool ok = wait_bar_warp(p, s.cons_bar, n & 1);
        n++;
        __syncwarp();
        return ok;
    }
};

// ---------------------------------------------------------------- math helpers
// Dot products of R rows (records at rec + r*stride) with a pre-scaled vector
// over the chunks this lane owns; reduced over the lpr lanes of each row group.
template <int BITS, int R>
__device__ __forceinline__ void rows_dot(const uint8_t *rec, uint32_t stride, int cols,
                                         const float *vps, const float *vsum, int sub, int lpr,
                                         float *out) {
    constexpr int VALS = 128 / BITS;
    const int nch = cols / VALS;
    const int cb = cols * BITS / 8;
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; r++) acc[r] = 0.0f;
    const float4 *v4 = reinterpret_cast<const float4 *>(vps);
    for (int c = sub; c < nch; c += lpr) {
        uint4 q[R];
        uint32_t sbw[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            q[r] = *reinterpret_cast<const uint4 *>(rec + (size_t)r * stride + (size_t)kChunk * c);
            sbw[r] = *reinterpret_cast<const uint32_t *>(rec + (size_t)r * stride + cb +
                                                         4 * ((c * VALS) / kGroup));
        }
        uint64_t a[R];
#pragma unroll
        for (int r = 0; r < R; r++) a[r] = 0;
        chunk_dot_ps<BITS, R>(q, v4 + c, nch, a);
        const float X = vsum[c];
#pragma unroll
        for (int r = 0; r < R; r++) {
            const float2 sb = sb_f(sbw[r]);
            acc[r] += fmaf(sb.x, f2_sum(a[r]), sb.y * X);
        }
    }
#pragma unroll
    for (int r = 0; r < R; r++) out[r] = warp_sum(acc[r], lpr);
}

// Dot product of one fp16 row with a plain float vector, reduced over lpr lanes.
__device__ __forceinline__ float f16_row_dot_s(const uint8_t *row, int cols, const float *v,
                                               int sub, int lpr) {
    float acc = 0.0f;
    for (int c = sub; c < cols / 8; c += lpr)
        acc += chunk_dot_f16(*reinterpret_cast<const uint4 *>(row + (size_t)kChunk * c), v + 8 * c);
    return warp_sum(acc, lpr);
}

__device__ __forceinline__ float gather2k(const uint16_t *tab, int width, int E, const int *cur,
                                          const int *prev, int K, int col) {
    float a = 0.0f;
    if (tab == nullptr) return a;
    if (cur)
        for (int k = 0; k < K; k++)
            if ((unsigned)cur[k] < (unsigned)E) a += half_f(tab[(size_t)cur[k] * width + col]);
    if (prev)
        for (int k = 0; k < K; k++)
            if ((unsigned)prev[k] < (unsigned)E)
                a += half_f(tab[(size_t)(E + prev[k]) * width + col]);
    return a;
}

__device__ __forceinline__ float lora_b(const LoraP &l, int s, int K, int e, int row,
                                        const float *v) {
    const uint16_t *B = l.B + (s < K ? (size_t)e * l.bs : 0) + (size_t)row * l.r;
    float a = 0.0f;
    for (int i = 0; i < l.r; i++) a = fmaf(half_f(B[i]), v[i], a);
    return l.scale * a;
}

// Writes vector v (n floats, plain, in smem) into the pre-scaled layout for
// BITS and its per-chunk sums; threads [t0, t0+nt) cooperate.
template <int BITS>
__device__ __forceinline__ void prescale(const float *v, int n, float *ps, int t, int nt) {
    const int nch = n / (128 / BITS);
    for (int i = t; i < n; i += nt) ps[ps_index<BITS>(i, nch)] = v[i] * ps_scale<BITS>(i);
}

template <int BITS>
__device__ __forceinline__ void chunk_sums(const float *v, int n, float *sums, int t, int nt) {
    constexpr int VALS = 128 / BITS;
    for (int c = t; c < n / VALS; c += nt) {
        float a = 0.0f;
        for (int j = 0; j < VALS; j++) a += v[c * VALS + j];
        sums[c] = a;
    }
}

// Warp top-K over E logits (value desc, index asc) -> idx, softmax weights,
// margin.  vals: per-lane logits for e = lane + 32 i.
__device__ void warp_topk(const float *vals_in, int E, int K, int lane, int *idx, float *w,
                          float *margin) {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; i++) {
        const float z = vals_in[i];
        v[i] = z == z ? z : -INFINITY;
    }
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
            if (e < E && !(taken >> i & 1u) &&
                (v[i] > bv || (v[i] == bv && e < bi))) {
                bv = v[i];
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
__device__ void producer(const Params &p, const Smem &s, int c) {
    uint32_t piece = 0;
    bool ok = true;
    auto issue_plan = [&](const Plan &pl) -> bool {
        for (int gi = 0; gi < pl.n; gi++) {
            const Grp &g = pl.g[gi];
            const int per = max(1, kSlotBytes / (int)g.item_bytes);
            for (int i0 = g.lo; i0 < g.hi; i0 += per) {
                const int cnt = min(per, g.hi - i0);
                const uint32_t slot = piece % p.n_slots, round = piece / p.n_slots;
                if (round > 0 && !wait_bar(p, s.empty + slot, (round - 1) & 1)) return false;
                const uint32_t bytes = (uint32_t)cnt * g.item_bytes;
                mbar_arrive_expect_tx(s.full + slot, bytes);
                bulk_g2s(s.ring + (size_t)slot * kSlotBytes, g.src + (size_t)i0 * g.item_bytes,
                         bytes, s.full + slot);
                piece++;
            }
        }
        return true;
    };
    for (int N = 0; N < p.depth && ok; N++) {
        if (N == 0 && p.own0) {
            make_plan(p, 0, PR, s.rcur, c, *s.plan_p);
            if (!(ok = issue_plan(*s.plan_p))) break;
            if (!(ok = wait_bar(p, s.route_bar, 0))) break;
        }
        // validate the route before it turns into addresses
        for (int k = 0; k < p.K; k++)
            if ((unsigned)s.rcur[N * p.K + k] >= (unsigned)p.E) {
                raise_error(p, MOE_EINVAL);
                ok = false;
            }
        if (!ok) break;
        make_plan(p, N, PA, s.rcur + N * p.K, c, *s.plan_p);
        if (!(ok = issue_plan(*s.plan_p))) break;
        make_plan(p, N, PB, s.rcur + N * p.K, c, *s.plan_p);
        if (!(ok = issue_plan(*s.plan_p))) break;
    }
    // never leave the CTA with copies in flight: wait (bounded) for the last
    // pieces issued
    const uint32_t first = piece > (uint32_t)p.n_slots ? piece - p.n_slots : 0;
    for (uint32_t q = first; q < piece; q++) {
        const uint32_t slot = q % p.n_slots, round = q / p.n_slots;
        if (!mbar_try_wait(s.full + slot, round & 1)) {
            const uint64_t t0 = now_ns();
            while (!mbar_try_wait(s.full + slot, round & 1) && now_ns() - t0 < p.timeout_ns) {
            }
        }
    }
}

// ---------------------------------------------------------------- route warp
// Top-K of the heads' logits of the layers this CTA is responsible for;
// writes the predicted routes for the next step.
__device__ void route_warp(const Params &p, int c, int lane) {
    const int nxt = (p.t + 1) % 3;
    for (int N = c; N < p.depth; N += p.n_cta) {
        if (!head_runs(p, N)) continue;
        const uint32_t tag = (uint32_t)ld_flag(ctrl(p) + C_EPOCH) * 64u + N + 1;
        const uint64_t *z = tagged(p, p.off_z) + (size_t)N * p.E;
        float vals[32];
        bool lok = true;
#pragma unroll
        for (int i = 0; i < 32; i++) {
            const int e = lane + 32 * i;
            vals[i] = -INFINITY;
            if (lok && e < p.E) lok = poll_tag(p, z + e, tag, &vals[i]);
        }
        if (!__all_sync(0xffffffffu, lok)) return;
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
    uint32_t piece = 0;
    ConsSync cs;
    uint32_t epoch;

    __device__ uint32_t tag(int N) const { return epoch * 64u + (uint32_t)N + 1u; }
    __device__ uint32_t tag_router() const { return epoch * 64u + 63u; }
    __device__ int tid() const { return warp * 32 + lane; }
    static constexpr int kT = kNW * 32;

    // x of layer N: poll out of layer N-1 (or take x0), RMS-normalise,
    // build the plain / pre-scaled copies and chunk sums.
    __device__ bool prologue_A(int N) {
        const int d = p.d;
        float ss = 0.0f;
        if (N == 0) {
            for (int i = tid(); i < d; i += kT) {
                const float v = p.x0[i];
                s.stream[i] = v;
                s.x[i] = v;
            }
        } else {
            const uint64_t *out = tagged(p, p.off_out);
            const uint32_t tg = tag(N - 1);
            bool lok = true;
            for (int i = tid(); i < d && lok; i += kT) {
                float v;
                lok = poll_tag(p, out + i, tg, &v);
                s.stream[i] = v;
                ss = fmaf(v, v, ss);
            }
            if (!__all_sync(0xffffffffu, lok)) return false;
            ss = warp_sum(ss, 32);
            if (lane == 0) s.misc[warp] = ss;
        }
        if (!cs.sync(p, s, lane)) return false;
        if (N > 0) {
            float tot = 0.0f;
            for (int w = 0; w < kNW; w++) tot += s.misc[w];
            const float inv = 1.0f / sqrtf(tot / d + 1e-6f);
            for (int i = tid(); i < d; i += kT) s.x[i] = s.stream[i] * inv;
            if (!cs.sync(p, s, lane)) return false;
        }
        prescale<BITS>(s.x, d, s.xps, tid(), kT);
        chunk_sums<BITS>(s.x, d, s.xsum, tid(), kT);
        if (BITS != 4) {
            prescale<4>(s.x, d, s.xps4, tid(), kT);
            chunk_sums<4>(s.x, d, s.xsum4, tid(), kT);
        }
        return cs.sync(p, s, lane);
    }

    // h of every slot and gelu(fc1 f) of the head: poll, pre-scale, sum.
    __device__ bool prologue_B(int N) {
        const uint32_t tg = tag(N);
        const int SF = p.S * p.F;
        const uint64_t *h = tagged(p, p.off_h);
        bool lok = true;
        for (int i = tid(); i < SF && lok; i += kT) {
            float v;
            lok = poll_tag(p, h + i, tg, &v);
            s.h[i] = v;
        }
        const bool fc2 = head_runs(p, N) && p.H > 0;
        if (fc2) {
            const uint64_t *ga = tagged(p, p.off_ga);
            for (int i = tid(); i < p.H && lok; i += kT) {
                float v;
                lok = poll_tag(p, ga + i, tg, &v);
                s.ga[i] = v;
            }
        }
        if (!__all_sync(0xffffffffu, lok)) return false;
        if (!cs.sync(p, s, lane)) return false;
        constexpr int VALS = 128 / BITS;
        for (int sl = 0; sl < p.S; sl++) {
            prescale<BITS>(s.h + sl * p.F, p.F, s.hps + sl * p.F, tid(), kT);
            chunk_sums<BITS>(s.h + sl * p.F, p.F, s.hsum + sl * (p.F / VALS), tid(), kT);
        }
        if (fc2) {
            prescale<4>(s.ga, p.H, s.gps, tid(), kT);
            chunk_sums<4>(s.ga, p.H, s.gsum, tid(), kT);
        }
        return cs.sync(p, s, lane);
    }

    // One warp task: `cnt` items of group g starting at item i (local index
    // `li` into the slot), records at `base`.
    __device__ bool task(int N, const Grp &g, const uint8_t *base, int i, int cnt, int lpr) {
        const int sub = lane % lpr, rsub = lane / lpr;
        const int item = i + rsub;
        const bool ok = rsub < cnt;
        const uint8_t *rec = base + (size_t)rsub * g.item_bytes;
        const LayerP &L = layer_of(p, N);
        const int *route = s.rcur + N * p.K;
        const uint32_t tg = tag(N);
        bool lok = true;
        switch (g.kind) {
            case KGU: {
                float r2[2];
                rows_dot<BITS, 2>(rec, p.rec_d, p.d, s.xps, s.xsum, sub, lpr, r2);
                if (ok && sub == 0) {
                    float gg = r2[0], uu = r2[1];
                    const LoraP &lg = slot_lora(p, L, g.slot, 0), &lu = slot_lora(p, L, g.slot, 1);
                    const int e = g.slot < p.K ? route[g.slot] : 0;
                    if (lg.r || lu.r) {
                        float v[kMaxLoraRank];
                        const uint64_t *vv = tagged(p, p.off_v) + (size_t)g.slot * 2 * kMaxLoraRank;
                        if (lg.r) {
                            for (int k = 0; k < lg.r && lok; k++)
                                lok = poll_tag(p, vv + k, tg, &v[k]);
                            gg += lora_b(lg, g.slot, p.K, e, item, v);
                        }
                        if (lu.r && lok) {
                            for (int k = 0; k < lu.r && lok; k++)
                                lok = poll_tag(p, vv + kMaxLoraRank + k, tg, &v[k]);
                            uu += lora_b(lu, g.slot, p.K, e, item, v);
                        }
                    }
                    if (lok)
                        put_tagged(tagged(p, p.off_h) + (size_t)g.slot * p.F + item, tg,
                                   silu_f(gg) * uu);
                }
                break;
            }
            case KFC1:
            case KLX:
            case KROUTER: {
                const float *xp = BITS == 4 ? s.xps : s.xps4;
                const float *xsm = BITS == 4 ? s.xsum : s.xsum4;
                float a;
                rows_dot<4, 1>(rec, 0, p.d, xp, xsm, sub, lpr, &a);
                if (ok && sub == 0) {
                    const int *cur = route;
                    const int *prev = p.t > 0 ? s.rprev + N * p.K : nullptr;
                    if (g.kind == KFC1) {
                        a += gather2k(L.fc1_tab, p.H, p.E, cur, prev, p.K, item) +
                             (L.b1 ? half_f(L.b1[item]) : 0.0f);
                        put_tagged(tagged(p, p.off_ga) + item, tg, gelu_erf_f(a));
                    } else if (g.kind == KLX) {
                        a += gather2k(L.l_tab, p.E, p.E, cur, prev, p.K, item) +
                             (L.bl ? half_f(L.bl[item]) : 0.0f);
                        if (p.H > 0) put_tagged(tagged(p, p.off_zl) + item, tg, a);
                        else put_tagged(tagged(p, p.off_z) + (size_t)N * p.E + item, tg, a);
                    } else {
                        put_tagged(tagged(p, p.off_zr) + item, tag_router(), a);
                    }
                }
                break;
            }
            case KLA: {
                const float a = f16_row_dot_s(rec, p.d, s.x, sub, lpr);
                if (ok && sub == 0)
                    put_tagged(tagged(p, p.off_v) + ((size_t)g.slot * 2 + g.aux) * kMaxLoraRank + item,
                               tg, a);
                break;
            }
            case KLD: {
                const float a = f16_row_dot_s(rec, p.F, s.h + g.slot * p.F, sub, lpr);
                if (ok && sub == 0)
                    put_tagged(tagged(p, p.off_vd) + (size_t)g.slot * kMaxLoraRank + item, tg, a);
                break;
            }
            case KDOWN: {
                constexpr int VALS = 128 / BITS;
                float a;
                rows_dot<BITS, 1>(rec, 0, p.F, s.hps + g.slot * p.F,
                                  s.hsum + g.slot * (p.F / VALS), sub, lpr, &a);
                if (ok && sub == 0) {
                    const LoraP &ld = slot_lora(p, L, g.slot, 2);
                    if (ld.r) {
                        float v[kMaxLoraRank];
                        const uint64_t *vv = tagged(p, p.off_vd) + (size_t)g.slot * kMaxLoraRank;
                        for (int k = 0; k < ld.r && lok; k++)
                            lok = poll_tag(p, vv + k, tg, &v[k]);
                        const int e = g.slot < p.K ? route[g.slot] : 0;
                        a += lora_b(ld, g.slot, p.K, e, item, v);
                    }
                    s.y[g.slot * p.max_orows + (item - g.lo)] = a;
                }
                break;
            }
            case KFC2: {
                float a;
                rows_dot<4, 1>(rec, 0, p.H, s.gps, s.gsum, sub, lpr, &a);
                if (ok && sub == 0) {
                    float zl = 0.0f;
                    lok = poll_tag(p, tagged(p, p.off_zl) + item, tg, &zl);
                    a += (L.b2 ? half_f(L.b2[item]) : 0.0f) + zl;
                    if (lok) put_tagged(tagged(p, p.off_z) + (size_t)N * p.E + item, tg, a);
                }
                break;
            }
        }
        return __all_sync(0xffffffffu, lok);
    }

    // Consumes this CTA's pieces of one phase, in the producer's order.
    __device__ bool run_plan(int N, const Plan &pl) {
        uint32_t tasks = 0;
        for (int gi = 0; gi < pl.n; gi++) {
            const Grp &g = pl.g[gi];
            const int per = max(1, kSlotBytes / (int)g.item_bytes);
            const int lpr = pow2_floor32(item_chunks<BITS>(g));
            const int rpw = 32 / lpr;
            for (int i0 = g.lo; i0 < g.hi; i0 += per) {
                const int cnt = min(per, g.hi - i0);
                const uint32_t slot = piece % p.n_slots, round = piece / p.n_slots;
                if (!wait_bar_warp(p, s.full + slot, round & 1)) return false;
                const uint8_t *base = s.ring + (size_t)slot * kSlotBytes;
                const int ntask = (cnt + rpw - 1) / rpw;
                for (int k = 0; k < ntask; k++) {
                    if ((int)((tasks + k) % kNW) != warp) continue;
                    const int li = k * rpw;
                    if (!task(N, g, base + (size_t)li * g.item_bytes, i0 + li, min(rpw, cnt - li), lpr))
                        return false;
                }
                tasks += ntask;
                __syncwarp();
                if (lane == 0) mbar_arrive(s.empty + slot);
                piece++;
            }
        }
        return true;
    }

    // Layer 0's own route: poll the router logits, top-K (every CTA alike).
    __device__ bool route0() {
        if (warp == 0) {
            const uint64_t *zr = tagged(p, p.off_zr);
            float vals[32];
            bool lok = true;
#pragma unroll
            for (int i = 0; i < 32; i++) {
                const int e = lane + 32 * i;
                vals[i] = -INFINITY;
                if (lok && e < p.E) lok = poll_tag(p, zr + e, tag_router(), &vals[i]);
            }
            if (!__all_sync(0xffffffffu, lok)) return false;
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
        return cs.sync(p, s, lane);
    }

    // Combine + residual over this CTA's output rows; publishes out.
    __device__ bool epilogue_B(int N, const Plan &pl) {
        if (!cs.sync(p, s, lane)) return false;
        const uint32_t tg = tag(N);
        const float *w = s.rw + N * p.K;
        for (int o = pl.o_lo + tid(); o < pl.o_hi; o += kT) {
            const int li = o - pl.o_lo;
            float v = s.stream[o];
            for (int k = 0; k < p.K; k++) v = fmaf(w[k], s.y[k * p.max_orows + li], v);
            if (p.S > p.K) v += s.y[p.K * p.max_orows + li];
            put_tagged(tagged(p, p.off_out) + o, tg, v);
            if (N == p.depth - 1) p.out[o] = v;
        }
        return true;
    }

    __device__ bool run() {
        if (p.debug_unset_wait && c == 0 && warp == 0) {
            // test hook: a flag nothing ever sets, so this wait runs out
            float v;
            const bool lok = poll_tag(p, tagged(p, C_NEVER * 4), 0xFFFFFFFFu, &v);
            if (!__all_sync(0xffffffffu, lok)) return false;
        }
        for (int N = 0; N < p.depth; N++) {
            if (!prologue_A(N)) return false;
            if (N == 0 && p.own0) {
                if (warp == 0 && lane == 0) make_plan(p, 0, PR, s.rcur, c, *s.plan_c);
                if (!cs.sync(p, s, lane)) return false;
                if (!run_plan(0, *s.plan_c)) return false;
                if (!route0()) return false;
            }
            if (warp == 0 && lane == 0) make_plan(p, N, PA, s.rcur + N * p.K, c, *s.plan_c);
            if (!cs.sync(p, s, lane)) return false;
            if (!run_plan(N, *s.plan_c)) return false;
            if (!cs.sync(p, s, lane)) return false;
            if (!prologue_B(N)) return false;
            if (warp == 0 && lane == 0) make_plan(p, N, PB, s.rcur + N * p.K, c, *s.plan_c);
            if (!cs.sync(p, s, lane)) return false;
            if (!run_plan(N, *s.plan_c)) return false;
            if (!epilogue_B(N, *s.plan_c)) return false;
        }
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
        for (int i = 0; i < p.n_slots; i++) {
            mbar_init(s.full + i, 1);
            mbar_init(s.empty + i, kNW);
        }
        mbar_init(s.route_bar, 1);
        mbar_init(s.cons_bar, kNW);
        mbar_init(s.end_bar, kCons0 + kNW);
        mbar_fence_init();
    }
    __syncthreads();

    bool ok = true;
    if (warp == kProducerWarp) {
        if (lane == 0) producer<BITS>(p, s, c);
    } else if (warp == kRouteWarp) {
        route_warp(p, c, lane);
    } else {
        Consumer<BITS> cons{p, s, c, warp - kCons0, lane};
        cons.epoch = (uint32_t)ld_flag(ctrl(p) + C_EPOCH);
        ok = cons.run();
    }
    (void)ok;
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

struct StepLayout {
    Params p;
    size_t smem;
};

static size_t al(size_t v, size_t a) { return (v + a - 1) / a * a; }

int decode_step_workspace_layout(int d, int F, int E, int H, int S, int depth, uint32_t *offs,
                                 size_t *total) {
    size_t off = kCtrlBytes;
    auto take = [&](size_t n) {
        const size_t o = off;
        off = al(off + n * sizeof(uint64_t), 256);
        return (uint32_t)o;
    };
    offs[0] = take((size_t)S * F);                    // h
    offs[1] = take((size_t)S * 2 * kMaxLoraRank);     // v (gate/up A x)
    offs[2] = take((size_t)S * kMaxLoraRank);         // vd (down A h)
    offs[3] = take((size_t)(H > 0 ? H : 1));          // gelu(fc1 f)
    offs[4] = take((size_t)E);                        // zl (l f)
    offs[5] = take((size_t)E);                        // router logits
    offs[6] = take((size_t)depth * E);                // head logits per layer
    offs[7] = take((size_t)d);                        // out
    *total = off;
    return 0;
}

int launch_decode_step(const moe_stack_desc *sd, const float *x0, float *out, int32_t *ridx,
                       float *rw, float *rmargin, int t, void *ws, size_t ws_bytes,
                       cudaStream_t st);

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
    for (int i = 0; i < sd->n_layers; i++) {
        const moe_experts_desc &e = sd->experts[i];
        if (e.d != e0.d || e.F != e0.F || e.E != e0.E || e.bits != e0.bits ||
            (e.shared == nullptr) != (e0.shared == nullptr) || e.pool == nullptr ||
            e.expert_stride != e0.expert_stride)
            return fail(MOE_EINVAL, "decode_step: layer %d differs in shape from layer 0", i);
        if (e.expert_stride < blob_layout(e.d, e.F, e.bits).bytes || e.expert_stride % 256)
            return fail(MOE_EINVAL, "decode_step: expert_stride %zu", e.expert_stride);
        for (int j = 0; j < 3; j++) {
            if (e.lora[j].r != e0.lora[j].r || e.shared_lora[j].r != e0.shared_lora[j].r ||
                e.lora[j].r < 0 || e.lora[j].r > kMaxLoraRank || e.shared_lora[j].r < 0 ||
                e.shared_lora[j].r > kMaxLoraRank)
                return fail(MOE_EINVAL, "decode_step: LoRA ranks must match across layers (<= 64)");
            if ((e.lora[j].r && (!e.lora[j].A || !e.lora[j].B)) ||
                (e.shared_lora[j].r && (!e.shared_lora[j].A || !e.shared_lora[j].B)))
                return fail(MOE_EINVAL, "decode_step: LoRA with NULL A or B");
        }
        const moe_head_desc &r = sd->routers[i];
        if (r.d != e0.d || r.E != e0.E || r.lx == nullptr || r.prec != MOE_PREC_AFFINE4)
            return fail(r.prec != MOE_PREC_AFFINE4 ? MOE_EUNSUPPORTED : MOE_EINVAL,
                        "decode_step: router %d (needs int4 l rows of [E][d])", i);
        if (heads) {
            const moe_head_desc &h = sd->heads[i];
            if (h.d != e0.d || h.E != e0.E || h.H != H || h.H < 0 || h.H % 64 || h.lx == nullptr ||
                (h.H > 0 && (h.fc1x == nullptr || h.fc2 == nullptr)))
                return fail(MOE_EINVAL, "decode_step: head %d shape", i);
            if (h.prec != MOE_PREC_AFFINE4)
                return fail(MOE_EUNSUPPORTED, "decode_step: fp16 heads run through the per-call path");
        }
    }
    return MOE_OK;
}

extern "C" size_t moe_decode_step_workspace_bytes(const moe_stack_desc *sd) {
    if (check_stack(sd) != MOE_OK) return 0;
    const moe_experts_desc &e0 = sd->experts[0];
    const int H = (sd->depth > 1 || sd->self_predict) ? sd->heads[0].H : 0;
    uint32_t offs[8];
    size_t total = 0;
    decode_step_workspace_layout(e0.d, e0.F, e0.E, H, sd->K + (e0.shared ? 1 : 0), sd->depth,
                                 offs, &total);
    return total;
}

extern "C" int moe_decode_step(const moe_stack_desc *sd, const float *x0, float *out,
                               int32_t *route_idx, float *route_w, float *route_margin, int t,
                               void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (int rc = check_stack(sd)) return rc;
    if (t < 1) return fail(MOE_EINVAL, "decode_step: t=%d (step 0 routes every layer with its own router; use the per-call path)", t);
    if (!x0 || !out || !route_idx || !route_w || !route_margin || !ws)
        return fail(MOE_EINVAL, "decode_step: NULL pointer");
    const size_t need = moe_decode_step_workspace_bytes(sd);
    if (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 256))
        return fail(MOE_ENOSPACE, "decode_step: workspace %zu bytes, need %zu (256-aligned)", ws_bytes, need);
    return launch_decode_step(sd, x0, out, route_idx, route_w, route_margin, t, ws, ws_bytes,
                              stream);
}

extern "C" int moe_decode_step_status(const void *ws, int *status, cudaStream_t stream) {
    if (ws == nullptr || status == nullptr) return fail(MOE_EINVAL, "decode_step_status: NULL pointer");
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
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step: smem attribute: %s", cudaGetErrorString(e));
        configured_dev = dev;
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

int launch_decode_step(const moe_stack_desc *sd, const float *x0, float *out, int32_t *ridx,
                       float *rw, float *rmargin, int t, void *ws, size_t ws_bytes,
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
    p.x0 = x0;
    p.out = out;
    p.ridx = ridx;
    p.rw = rw;
    p.rmargin = rmargin;
    p.ws = static_cast<uint8_t *>(ws);
    uint32_t offs[8];
    size_t total = 0;
    decode_step_workspace_layout(p.d, p.F, p.E, p.H, p.S, p.depth, offs, &total);
    p.off_h = offs[0];
    p.off_v = offs[1];
    p.off_vd = offs[2];
    p.off_ga = offs[3];
    p.off_zl = offs[4];
    p.off_zr = offs[5];
    p.off_z = offs[6];
    p.off_out = offs[7];
    p.timeout_ns = sd->timeout_ns ? sd->timeout_ns : 1000000000ull;
    p.debug_unset_wait = sd->debug_unset_wait;
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

    // grid: one CTA per SM (all co-resident: cooperative launch)
    int dev = 0, sms = 0, smem_max = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    p.n_cta = sms;
    p.max_orows = (p.d + sms - 1) / sms;

    // shared-memory layout
    const int VALS = 128 / bits;
    size_t off = 0;
    auto take = [&](size_t bytes, size_t a = 16) {
        off = al(off, a);
        const size_t o = off;
        off += bytes;
        return (uint32_t)o;
    };
    p.sm_plan = take(2 * sizeof(Plan), 16);
    p.sm_x = take(p.d * 4);
    p.sm_xps = take(p.d * 4);
    p.sm_xps4 = bits == 4 ? p.sm_xps : take(p.d * 4);
    p.sm_xsum = take((p.d / VALS) * 4);
    p.sm_xsum4 = bits == 4 ? p.sm_xsum : take((p.d / 32) * 4);
    p.sm_stream = take(p.d * 4);
    p.sm_h = take((size_t)p.S * p.F * 4);
    p.sm_hps = take((size_t)p.S * p.F * 4);
    p.sm_hsum = take((size_t)p.S * (p.F / VALS) * 4);
    p.sm_ga = take((size_t)(p.H ? p.H : 1) * 4);
    p.sm_gps = take((size_t)(p.H ? p.H : 1) * 4);
    p.sm_gsum = take((size_t)(p.H ? p.H / 32 : 1) * 4);
    p.sm_y = take((size_t)p.S * p.max_orows * 4);
    p.sm_rcur = take((size_t)p.depth * p.K * 4);
    p.sm_rprev = take((size_t)p.depth * p.K * 4);
    p.sm_rw = take((size_t)p.depth * p.K * 4);
    p.sm_misc = take(64 * 4);
    const size_t fixed_end = al(off, 1024);
    int slots = (int)(((size_t)smem_max - fixed_end - (size_t)(2 * kMaxRing + 3) * 8 - 64) / kSlotBytes);
    slots = std::min(slots, kMaxRing);
    if (slots < 3)
        return fail(MOE_EUNSUPPORTED, "decode_step: shapes leave room for %d ring slots (< 3)", slots);
    p.n_slots = slots;
    p.sm_ring = (uint32_t)fixed_end;
    p.sm_bar = (uint32_t)(fixed_end + (size_t)slots * kSlotBytes);
    const size_t smem = p.sm_bar + (size_t)(2 * slots + 3) * 8;

    // every item must fit a ring slot
    if (2 * p.rec_d > (uint32_t)kSlotBytes || 2u * p.d > (uint32_t)kSlotBytes)
        return fail(MOE_EUNSUPPORTED, "decode_step: d=%d rows exceed a %d-byte ring slot", p.d, kSlotBytes);

    int occ = 0;
    if (bits == 4)
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_step_kernel<4>, kThreads, 0);
    else
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_step_kernel<2>, kThreads, 0);
    if (occ < 1) return fail(MOE_EUNSUPPORTED, "decode_step: kernel does not fit an SM");

    return bits == 4 ? launch_bits<4>(p, smem, st) : launch_bits<2>(p, smem, st);
}

}  // namespace moe
