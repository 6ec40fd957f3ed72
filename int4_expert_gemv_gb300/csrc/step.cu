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
//    as far ahead as the ring allows, across layer boundaries.  All 32 lanes
//    issue copies together (one thread issues about one copy per 200 ns), and
//    the bytes in flight per SM are capped: a deep queue of weight copies
//    delays every load that shares the return path, including the polls of
//    the exchanges below (measured on GB300: an all-to-all exchange takes
//    1.3 us with 32 KB in flight per SM, 8 us with 192 KB).
//  * Dependencies between CTAs travel as 64-bit (tag, value) words in global
//    memory, gated by one ready flag per CTA and exchange: one warp of a CTA
//    polls the flags while the others sleep on an mbarrier, then every warp
//    reads its words once (their tags are checked).  There is no grid-wide
//    barrier.  A layer has exactly two exchanges on its critical path: x (the
//    previous layer's out) and h.  The LoRA products ride on them: each CTA
//    publishes, with its rows of out, its partial A x over those rows for the
//    next layer's gate/up LoRA, and the owners of a down-LoRA slot's gate/up
//    rows publish their partial A_d h with h.
//  * The prerouter head's first layer (fc1, l) reads x like the gate/up rows
//    do and is split with them; its second layer (fc2) and the top-K only feed
//    the next token, so an auxiliary warp runs them off the critical path, and
//    also prepares each layer's small operands (K-hot table sums, LoRA B rows,
//    A columns and scales) in shared memory a layer ahead.
//  * The launch context lives in shared memory (read with plain shared loads
//    by every function) and per-thread state in registers: nothing of the hot
//    path goes through local memory, whose misses would cost an L2 round trip
//    each.
//  * x enters the GEMVs unnormalised; 1/rms is applied to each finished row
//    dot.  Activations are staged per 16-byte code chunk as 16-bit fixed
//    point, and each chunk's code dot is an exact integer sum (dp4a).
//  * Every wait is bounded (globaltimer); on expiry the kernel records
//    MOE_ETIMEOUT in the workspace status word, waits (bounded) for its own
//    copies in flight and returns.
//
// Work per layer and CTA.  Phase A (needs x): gate/up row pairs of every slot,
// head fc1 rows and l rows -- split across CTAs by bytes.  Phase B (needs h):
// down rows of CTA c's outputs [c*d/n, (c+1)*d/n) for every slot; the warp
// that owns an output row in one slot owns it in all, so it combines the row
// itself.  Phase R (layer 0, when it routes with its own router): router rows.
#include <algorithm>

#include "step_common.cuh"

namespace moe {
namespace step {

constexpr int kMaxLayers = 48;
constexpr int kNW = 12;                        // consumer warps
constexpr int kProducerWarp = 0, kAuxWarp = 1, kCons0 = 2;
constexpr int kThreads = (kCons0 + kNW) * 32;  // 448
constexpr int kMaxPiece = 16384;               // bytes per bulk copy
constexpr int kNB = 64;                        // pieces in the ring at once (barrier pairs)
constexpr int kMaxK = 16;
constexpr int kMaxGroups = 24;
constexpr int kMaxR = 32;                      // LoRA rank bound of the fused kernel
constexpr int kPollW = 20;                     // tagged words one lane polls at once
constexpr int kTrace = 16;                     // stamps per (CTA, layer), debug trace
constexpr uint32_t kDefaultInflight = 32768;   // weight bytes in flight per SM
constexpr uint32_t kSleepHint = 20000;         // ns a thread may sleep in one mbarrier wait

enum Kind : uint8_t { KGU = 0, KFC1, KLX, KROUTER, KDOWN };
enum Tmpl : int { T_R = 0, T_A_HEAD, T_A_NOHEAD, T_B, T_COUNT };

// control words at the start of the workspace
enum Ctrl : int { C_STATUS = 0, C_EPOCH = 1, C_DONE = 2, C_ABORT = 3, C_NEVER = 4 };
constexpr size_t kCtrlBytes = 256;

// mbarriers after the kNB full / kNB empty pairs
enum Bar : int {
    B_ROUTE = 0, B_CONS, B_END, B_PREP_FULL0, B_PREP_FULL1, B_PREP_EMPTY0, B_PREP_EMPTY1, B_X, B_H,
    B_AUX, B_COUNT
};

// last-warp counters and small values in the misc area (ints / floats)
enum Misc : int {
    M_SS = 0, M_INV = 12, M_CNT_A = 16, M_CNT_X, M_CNT_H, M_CNT_D, M_TMPL_OK, M_VDP_N0, M_VDP_N1,
    M_COUNT
};

// debug trace stamps (per CTA and layer)
enum Stamp : int {
    ST_L0 = 0, ST_X = 1, ST_A = 2, ST_H = 3, ST_D = 4,
    ST_PA = 8, ST_PB = 9, ST_PE = 10, ST_AUXP = 12, ST_AUXF = 13
};

// per-layer LoRA scales in the prep buffer
enum Scale : int { SC_G = 0, SC_U, SC_DR, SC_DS, SC_COUNT };

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

// Everything the device code reads besides the layer table; copied into
// shared memory at the start of the kernel.
struct Ctx {
    int d, F, E, K, H, S, depth, n_res, self_predict, own0, t, n_cta;
    int max_orows, max_erows, max_pairs, max_hrows, max_owners;
    int rg, ru, rd, rdr, rds, gu_slot, n_dl;   // LoRA ranks: gate, up (on gu_slot), down (max,
                                               // routed, shared); down-LoRA slot count
    uint32_t dl_mask;                          // slots with a down LoRA
    uint32_t ring_bytes, inflight, epoch;
    uint32_t gu_off, down_off, rec_d, rec_F, rec_dh, rec_H;
    size_t stride;
    uint64_t timeout_ns;
    int debug_unset_wait;
    uint8_t *ws;
    const float *x0;
    float *out;
    int32_t *ridx;
    float *rw, *rmargin;
    unsigned long long *trace;                 // debug: [n_cta][depth][kTrace] globaltimer stamps
    uint32_t off_h, off_vp, off_vdp, off_ga, off_zl, off_zr, off_z, off_out, off_xflag, off_hflag;
    // shared-memory layout (byte offsets from the dynamic base)
    uint32_t sm_ring, sm_bar, sm_pend, sm_tmpl, sm_xf, sm_xsc, sm_xhat, sm_xf4, sm_xsc4, sm_xhat4,
        sm_stream, sm_hf, sm_hsc, sm_hhat, sm_vpw, sm_vx, sm_vdw, sm_vd, sm_vdacc, sm_vnw, sm_comb,
        sm_prep, sm_gf, sm_gsc, sm_ghat, sm_frec, sm_rcur, sm_rprev, sm_rw, sm_misc, sm_stage, sm_graw,
        sm_poff;
    // one prep buffer: bytes, and float offsets of its parts
    uint32_t prep_bytes, pp_tsum, pp_bgu, pp_adn, pp_bd, pp_agu, pp_scale;
};

struct Params {
    Ctx cx;
    LayerP layer[kMaxLayers];
};

// A group of equal items, contiguous in memory; [lo, hi) = this CTA's items.
struct Grp {
    uint32_t item_bytes;
    int n, lo, hi, cols;
    uint8_t kind, slot, pad0, pad1;
};

// A phase's groups, identical for every layer of the same kind (only the
// source addresses depend on the layer and its route).
struct Tmplt {
    Grp g[kMaxGroups];
    int n;
    int o_lo, o_hi, e_lo, e_hi;
    int own0[kMaxSlots], own1[kMaxSlots];   // CTAs owning the slot's gate/up rows
    int plo[kMaxSlots], phi[kMaxSlots];     // this CTA's gate/up pairs of the slot
    int pbase[kMaxSlots];                   // CTA-local index of the slot's first own pair
    int f1lo, f1hi, llo, lhi;               // this CTA's fc1 and l rows
};

// ---------------------------------------------------------------- context
extern __shared__ __align__(1024) uint8_t g_smem[];

__device__ __forceinline__ const Ctx &CX() { return *reinterpret_cast<const Ctx *>(g_smem); }

template <typename T>
__device__ __forceinline__ T *SM(uint32_t off) {
    return reinterpret_cast<T *>(g_smem + off);
}

__device__ __forceinline__ uint64_t *bar_full(int i) { return SM<uint64_t>(CX().sm_bar) + i; }
__device__ __forceinline__ uint64_t *bar_empty(int i) { return SM<uint64_t>(CX().sm_bar) + kNB + i; }
__device__ __forceinline__ uint64_t *bar(int b) { return SM<uint64_t>(CX().sm_bar) + 2 * kNB + b; }
__device__ __forceinline__ const Tmplt *tmpls() { return SM<Tmplt>(CX().sm_tmpl); }
__device__ __forceinline__ int *misc_i() { return SM<int>(CX().sm_misc); }
__device__ __forceinline__ float *misc_f() { return SM<float>(CX().sm_misc); }

__device__ __forceinline__ float *prep_of(int N, uint32_t part) {
    const Ctx &cx = CX();
    return reinterpret_cast<float *>(g_smem + cx.sm_prep + (size_t)(N & 1) * cx.prep_bytes) + part;
}

// ---------------------------------------------------------------- control
__device__ __forceinline__ int *ctrl() { return reinterpret_cast<int *>(CX().ws); }

__device__ __forceinline__ void raise_error(int code) {
    atomicCAS(ctrl() + C_STATUS, 0, code);
    atomicExch(ctrl() + C_ABORT, 1);
}

__device__ __forceinline__ bool aborted() { return ld_flag(ctrl() + C_ABORT) != 0; }

// Warp-collective bounded wait on an mbarrier phase (inlined copy for the
// piece loop; wait_bar_warp is the out-of-line one): every lane observes the
// phase and the warp leaves together; false (error recorded) on timeout or
// when another CTA has aborted.
__device__ __forceinline__ bool wait_bar_warp_inl(uint64_t *b, uint32_t parity) {
    if (__all_sync(0xffffffffu, mbar_test_wait(b, parity))) return true;
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    if (lane == 0) t0 = now_ns();
    for (int it = 1;; it++) {
        const bool ok = mbar_try_wait_sleep(b, parity, kSleepHint);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((it & 7) == 0) {
            int stop = 0;
            if (lane == 0) {
                if (aborted()) stop = 1;
                else if (now_ns() - t0 > CX().timeout_ns) {
                    raise_error(MOE_ETIMEOUT);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        }
    }
}

__device__ __noinline__ bool wait_bar_warp(uint64_t *b, uint32_t parity) {
    return wait_bar_warp_inl(b, parity);
}

// Single-thread bounded wait (end of kernel).
__device__ bool wait_bar(uint64_t *b, uint32_t parity) {
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = now_ns();
    for (int it = 1;; it++) {
        if (mbar_try_wait_sleep(b, parity, kSleepHint)) return true;
        if ((it & 7) == 0) {
            if (aborted()) return false;
            if (now_ns() - t0 > CX().timeout_ns) {
                raise_error(MOE_ETIMEOUT);
                return false;
            }
        }
    }
}

__device__ __forceinline__ uint64_t *tagged(uint32_t off) {
    return reinterpret_cast<uint64_t *>(CX().ws + off);
}

// the workspace as 64-bit words (tagged words are indexed from here)
__device__ __forceinline__ const uint64_t *ws_words() {
    return reinterpret_cast<const uint64_t *>(CX().ws);
}

// A word the staged copy held with an old tag (its writer's data became
// visible after its flag): read again from global memory until current
// (bounded; NaN and the error recorded on expiry, which ends the step).
__device__ __noinline__ float refetch_word(uint32_t widx, uint32_t tag) {
    const uint64_t *w = ws_words() + widx;
    const uint64_t t0 = now_ns();
#pragma unroll 1
    for (int it = 0;; it++) {
        const uint64_t v = get_word(w);
        if ((uint32_t)(v >> 32) == tag) return __uint_as_float((uint32_t)v);
        if ((it & 7) == 7 && (aborted() || now_ns() - t0 > CX().timeout_ns)) {
            if (!aborted()) raise_error(MOE_ETIMEOUT);
            return __int_as_float(0x7fc00000);
        }
        __nanosleep(128);
    }
}

// Value of tagged word widx, copied into stage[i]; refetched if stale.
__device__ __forceinline__ float staged(const uint64_t *stage, int i, uint32_t widx, uint32_t tag) {
    const uint64_t v = stage[i];
    return (uint32_t)(v >> 32) == tag ? __uint_as_float((uint32_t)v) : refetch_word(widx, tag);
}

__device__ __forceinline__ uint32_t *flag_of(uint32_t off, int c) {
    return reinterpret_cast<uint32_t *>(CX().ws + off) + c;
}

// Per-lane bounded poll of the tagged words base[idx[k]] for the bits k set
// in `pend`, all loads in flight together; word k must carry tagB if bit k of
// selB is set, else tagA.  Values to val[k].  False on timeout or abort.
template <int W>
__device__ __forceinline__ bool poll_vals(const uint64_t *base, const uint32_t (&idx)[W],
                                          uint32_t pend, uint32_t selB, uint32_t tagA,
                                          uint32_t tagB, float (&val)[W]) {
    uint64_t t0 = 0;
    for (int it = 0; pend; it++) {
        uint64_t v[W];
#pragma unroll
        for (int k = 0; k < W; k++) v[k] = (pend >> k & 1u) ? get_word(base + idx[k]) : 0ull;
#pragma unroll
        for (int k = 0; k < W; k++) {
            const uint32_t tg = (selB >> k & 1u) ? tagB : tagA;
            if ((pend >> k & 1u) && (uint32_t)(v[k] >> 32) == tg) {
                val[k] = __uint_as_float((uint32_t)v[k]);
                pend &= ~(1u << k);
            }
        }
        if (pend && (it & 7) == 7) {
            if (it == 7) t0 = now_ns();
            else if (aborted()) return false;
            else if (now_ns() - t0 > CX().timeout_ns) {
                raise_error(MOE_ETIMEOUT);
                return false;
            }
        }
    }
    return true;
}

// Reads the tagged words base[idx(i)], i < n, of this lane and hands their
// values to sink(i, value) in order.  Called after the flags of the words'
// writers, so their tags are normally current: the first pass uses plain L2
// loads, eight in flight at a time.  If any word still carried an old tag,
// the whole read is repeated (reset() first) with strong loads after a short
// sleep, bounded.  Warp-uniform result.
template <typename Idx, typename Sink, typename Reset>
__device__ __forceinline__ bool read_words(const uint64_t *base, int n, uint32_t tag, Idx idx,
                                           Sink sink, Reset reset) {
    bool stale = false;
#pragma unroll 1
    for (int i0 = 0; i0 < n; i0 += 8) {
        uint64_t w[8];
#pragma unroll
        for (int k = 0; k < 8; k++)
            w[k] = i0 + k < n ? __ldcg(reinterpret_cast<const unsigned long long *>(base + idx(i0 + k)))
                              : 0ull;
#pragma unroll
        for (int k = 0; k < 8; k++)
            if (i0 + k < n) {
                stale |= (uint32_t)(w[k] >> 32) != tag;
                sink(i0 + k, __uint_as_float((uint32_t)w[k]));
            }
    }
    if (!__any_sync(0xffffffffu, stale)) return true;
    const uint64_t t0 = now_ns();
#pragma unroll 1
    for (;;) {
        __nanosleep(256);
        reset();
        stale = false;
#pragma unroll 1
        for (int i = 0; i < n; i++) {
            const uint64_t w = get_word(base + idx(i));
            stale |= (uint32_t)(w >> 32) != tag;
            sink(i, __uint_as_float((uint32_t)w));
        }
        if (!__any_sync(0xffffffffu, stale)) return true;
        if (aborted() || now_ns() - t0 > CX().timeout_ns) {
            if (!aborted()) raise_error(MOE_ETIMEOUT);
            return false;
        }
    }
}

// Warp-collective bounded wait until every CTA's flag at workspace offset
// `off` has reached `tag` (flags only grow within a step); lane j polls flags
// j, j+32, ...
__device__ __noinline__ bool poll_flags(uint32_t off, uint32_t tag, int lane, uint32_t sleep_ns) {
    const uint32_t *f = flag_of(off, 0);
    const int n_cta = CX().n_cta;
    uint32_t pend = 0;
#pragma unroll
    for (int i = 0; i < 8; i++)
        if (lane + 32 * i < n_cta) pend |= 1u << i;
    uint64_t t0 = 0;
    for (int it = 0;; it++) {
#pragma unroll
        for (int i = 0; i < 8; i++)
            if ((pend >> i & 1u) && (int)(ld_acquire(f + lane + 32 * i) - tag) >= 0)
                pend &= ~(1u << i);
        if (__all_sync(0xffffffffu, pend == 0)) return true;
        if (sleep_ns) __nanosleep(sleep_ns);
        if ((it & 7) == 7) {
            int stop = 0;
            if (lane == 0) {
                if (it == 7) t0 = now_ns();
                else if (aborted()) stop = 1;
                else if (now_ns() - t0 > CX().timeout_ns) {
                    raise_error(MOE_ETIMEOUT);
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) return false;
        }
    }
}

// Warp poll of E logits, lane-strided (vals[i] = logit lane + 32 i), all in
// flight together.  Warp-uniform result.
__device__ __forceinline__ bool poll_logits(const uint64_t *z, int E, uint32_t tag, int lane,
                                            float (&vals)[32], uint32_t sleep_ns) {
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
        if (pend && sleep_ns) __nanosleep(sleep_ns);
        if (pend && (it & 7) == 7) {
            if (it == 7) t0 = now_ns();
            else if (aborted()) lok = false;
            else if (now_ns() - t0 > CX().timeout_ns) {
                raise_error(MOE_ETIMEOUT);
                lok = false;
            }
        }
    }
    return __all_sync(0xffffffffu, lok);
}

__device__ __forceinline__ void stamp_at(int c, int N, int k) {
    const Ctx &cx = CX();
    if (cx.trace) cx.trace[((size_t)c * cx.depth + N) * kTrace + k] = now_ns();
}

// ---------------------------------------------------------------- layers
__device__ __forceinline__ bool head_runs(int N) {
    const Ctx &cx = CX();
    return N + 1 < cx.depth || cx.self_predict;
}

__device__ __forceinline__ const LayerP &layer_of(const Params &p, int N) {
    return p.layer[N % p.cx.n_res];
}

__device__ __forceinline__ const LoraP &slot_lora(const LayerP &L, int K, int s, int w) {
    return s < K ? L.lora[w] : L.slora[w];
}

__device__ __forceinline__ const uint16_t *lora_a(const LayerP &L, int K, const int *route, int s,
                                                  int w) {
    const LoraP &l = slot_lora(L, K, s, w);
    return l.A + (s < K ? (size_t)route[s] * l.as : 0);
}

__device__ __forceinline__ const uint16_t *lora_bm(const LayerP &L, int K, const int *route, int s,
                                                   int w) {
    const LoraP &l = slot_lora(L, K, s, w);
    return l.B + (s < K ? (size_t)route[s] * l.bs : 0);
}

// rank of slot s's down LoRA
__device__ __forceinline__ int dl_rank(int s) {
    const Ctx &cx = CX();
    return s < cx.K ? cx.rdr : cx.rds;
}

// index of slot s among the down-LoRA slots
__device__ __forceinline__ int dl_index(int s) { return __popc(CX().dl_mask & ((1u << s) - 1u)); }

// ---------------------------------------------------------------- templates
__device__ void add_group(Tmplt &t, uint32_t ib, int n, int kind, int slot, int cols, int lo = 0,
                          int hi = 0) {
    Grp &g = t.g[t.n++];
    g.item_bytes = ib;
    g.n = n;
    g.lo = lo;
    g.hi = hi;
    g.cols = cols;
    g.kind = (uint8_t)kind;
    g.slot = (uint8_t)slot;
    g.pad0 = g.pad1 = 0;
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

// Item ranges of all groups of t under an even split of their bytes (an item
// belongs to the CTA whose share holds its first byte); also the owner CTAs
// of each gate/up group and this CTA's own ranges.
__device__ void split_bytes(Tmplt &t, int c, int n_cta) {
    long long total = 0;
#pragma unroll 1
    for (int i = 0; i < t.n; i++) total += (long long)t.g[i].n * t.g[i].item_bytes;
    const long long a = split_at(total, c, n_cta), b = split_at(total, c + 1, n_cta);
    long long base = 0;
    int pairs = 0;
#pragma unroll 1
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
            t.plo[g.slot] = g.lo;
            t.phi[g.slot] = g.hi;
            t.pbase[g.slot] = pairs;
            pairs += g.hi - g.lo;
        } else if (g.kind == KFC1) {
            t.f1lo = g.lo;
            t.f1hi = g.hi;
        } else if (g.kind == KLX) {
            t.llo = g.lo;
            t.lhi = g.hi;
        }
        base += (long long)g.n * ib;
    }
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
        default: return g.cols / 32;              // int4 head rows
    }
}

// Items per bulk copy of a group: as many as fit kMaxPiece, a multiple of the
// rows one warp task takes; a slot's down rows of this CTA are one piece (the
// host checks that they fit).
template <int BITS>
__device__ __forceinline__ int piece_items(const Grp &g) {
    if (g.kind == KDOWN) return g.hi > g.lo ? g.hi - g.lo : 1;   // one piece per slot
    const int rpw = 32 / pow2_floor32(item_chunks<BITS>(g));
    int per = kMaxPiece / (int)g.item_bytes;
    if (per < 1) per = 1;
    if (per >= rpw) per -= per % rpw;
    return per;
}

// The CTA's phase templates (built once per launch by one thread); false if a
// per-CTA bound of the shared-memory layout is exceeded.
__device__ __noinline__ bool build_templates(int c, Tmplt *T) {
    const Ctx &cx = CX();
    {
        Tmplt &t = T[T_R];
        t.n = 0;
        add_group(t, cx.rec_dh, cx.E, KROUTER, 0, cx.d);
        split_bytes(t, c, cx.n_cta);
    }
    bool ok = true;
#pragma unroll 1
    for (int head = 1; head >= 0; head--) {
        Tmplt &t = T[head ? T_A_HEAD : T_A_NOHEAD];
        t.n = 0;
        t.f1lo = t.f1hi = t.llo = t.lhi = 0;
        #pragma unroll 1
        for (int s = 0; s < cx.S; s++) add_group(t, 2u * cx.rec_d, cx.F, KGU, s, cx.d);
        if (head) {
            if (cx.H) add_group(t, cx.rec_dh, cx.H, KFC1, 0, cx.d);
            add_group(t, cx.rec_dh, cx.E, KLX, 0, cx.d);
        }
        split_bytes(t, c, cx.n_cta);
        // the down-LoRA owner partials must fit the stage
#pragma unroll 1
        for (int s = 0; s < cx.S; s++)
            if ((cx.dl_mask >> s & 1u) && t.own1[s] - t.own0[s] + 1 > cx.max_owners) ok = false;
        int pairs = 0;
        #pragma unroll 1
        for (int s = 0; s < cx.S; s++) pairs += t.phi[s] - t.plo[s];
        ok = ok && pairs <= cx.max_pairs && (t.f1hi - t.f1lo) + (t.lhi - t.llo) <= cx.max_hrows;
    }
    Tmplt &t = T[T_B];
    t.n = 0;
    t.o_lo = (int)((long long)cx.d * c / cx.n_cta);
    t.o_hi = (int)((long long)cx.d * (c + 1) / cx.n_cta);
    t.e_lo = (int)((long long)cx.E * c / cx.n_cta);
    t.e_hi = (int)((long long)cx.E * (c + 1) / cx.n_cta);
#pragma unroll 1
    for (int s = 0; s < cx.S; s++) add_group(t, cx.rec_F, cx.d, KDOWN, s, cx.F, t.o_lo, t.o_hi);
    return ok && t.o_hi - t.o_lo <= cx.max_orows && t.e_hi - t.e_lo <= cx.max_erows;
}

__device__ __forceinline__ int tmpl_A_index(int N) { return head_runs(N) ? T_A_HEAD : T_A_NOHEAD; }

// ---------------------------------------------------------------- ring
// Byte ring of pieces: a piece never straddles the end of the ring; producer
// and consumers place pieces with the same rule, so they agree on offsets.
// head: absolute position (monotonic; for the producer's space accounting),
// off: head within the ring (kept alongside, so no division is needed).
struct RingPos {
    uint64_t head = 0;
    uint32_t off = 0, q = 0;
    // places a piece; returns its absolute start, its ring offset in *at
    __device__ __forceinline__ uint64_t place(uint32_t bytes, uint32_t rb, uint32_t *at) {
        if (off + bytes > rb) {
            head += rb - off;
            off = 0;
        }
        *at = off;
        const uint64_t start = head;
        head += bytes;
        off += bytes;
        if (off == rb) off = 0;
        return start;
    }
};

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
#pragma unroll 1
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

// Warp top-K over E logits (value desc, index asc) -> idx, softmax weights,
// margin (lane 0's copies are the ones used).  vals[i]: logit of expert
// lane + 32 i (-inf beyond E).
__device__ __forceinline__ void warp_topk(const float (&vals)[32], int E, int K, int lane,
                                          int (&idx)[kMaxK], float (&w)[kMaxK], float *margin) {
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

// Polls the E logits at z (tag), top-K, and writes the route of layer `tgt`
// into route set `set` of the caller's buffers (lane 0, with to_global) and
// into the CTA's current routes (with to_smem).  Warp-uniform result.
__device__ __noinline__ bool route_from_logits(const uint64_t *z, uint32_t tag, int set, int tgt,
                                               bool to_global, bool to_smem, uint32_t sleep_ns) {
    const Ctx &cx = CX();
    const int lane = threadIdx.x & 31;
    float vals[32];
    if (!poll_logits(z, cx.E, tag, lane, vals, sleep_ns)) return false;
    int idx[kMaxK];
    float w[kMaxK], margin;
    warp_topk(vals, cx.E, cx.K, lane, idx, w, &margin);
    if (lane == 0) {
        for (int k = 0; k < cx.K; k++) {
            if (to_global) {
                cx.ridx[((size_t)set * cx.depth + tgt) * cx.K + k] = idx[k];
                cx.rw[((size_t)set * cx.depth + tgt) * cx.K + k] = w[k];
            }
            if (to_smem) {
                SM<int>(cx.sm_rcur)[tgt * cx.K + k] = idx[k];
                SM<float>(cx.sm_rw)[tgt * cx.K + k] = w[k];
            }
        }
        if (to_global) cx.rmargin[(size_t)set * cx.depth + tgt] = margin;
    }
    return true;
}

// ---------------------------------------------------------------- producer
// All 32 lanes walk the same piece sequence; pieces are issued in batches of
// up to 32 (lane i issues piece i of the batch) under three limits: ring
// space, barrier pairs, and the bytes in flight (issued, not yet landed).
template <int BITS>
struct Producer {
    const Params &p;
    int lane;
    RingPos rp;
    uint32_t rel = 0, landed = 0;   // pieces [rel, q) not yet released; [landed, q) maybe in flight
    uint64_t tail = 0;              // ring bytes before `tail` are free
    uint64_t landed_end = 0;        // ring position up to which copies have landed
    uint64_t issued_end = 0;        // ring position up to which copies were issued
    uint32_t qb = 0;                // first piece of the open batch
    int nb = 0;                     // pieces in the open batch
    uint32_t bbytes = 0;
    uint64_t bend = 0;
    const uint8_t *my_src = nullptr;
    uint32_t my_bytes = 0, my_off = 0;
    uint64_t my_start = 0;

    __device__ __forceinline__ bool flush() {
        if (nb == 0) return true;
        const Ctx &cx = CX();
        uint64_t *pend = SM<uint64_t>(cx.sm_pend);
        const uint32_t qe = qb + nb;
        // ring space and barrier pairs for the whole batch
        while (rel < qe && (bend - tail > cx.ring_bytes || qe - 1 - rel >= (uint32_t)kNB)) {
            if (!wait_bar_warp(bar_empty(rel % kNB), (rel / kNB) & 1)) return false;
            tail = pend[rel % kNB];
            rel++;
            if (landed < rel) {
                landed = rel;
                landed_end = tail;
            }
        }
        // bytes in flight
        while (landed < qb && issued_end - landed_end + bbytes > cx.inflight) {
            if (!wait_bar_warp(bar_full(landed % kNB), (landed / kNB) & 1)) return false;
            landed_end = pend[landed % kNB];
            landed++;
        }
        if (lane < nb) {
            const uint32_t q = qb + lane;
            pend[q % kNB] = my_start + my_bytes;
            mbar_arrive_expect_tx(bar_full(q % kNB), my_bytes);
            bulk_g2s(SM<uint8_t>(cx.sm_ring) + my_off, my_src, my_bytes,
                     bar_full(q % kNB));
        }
        __syncwarp();
        issued_end = bend;
        qb = qe;
        nb = 0;
        bbytes = 0;
        return true;
    }

    __device__ __forceinline__ bool add(const uint8_t *src, uint32_t bytes) {
        const Ctx &cx = CX();
        const uint32_t cap = cx.inflight / 2 > bytes ? cx.inflight / 2 : bytes;
        if (nb == 32 || (nb > 0 && bbytes + bytes > cap))
            if (!flush()) return false;
        uint32_t at;
        const uint64_t start = rp.place(bytes, cx.ring_bytes, &at);
        rp.q++;
        if (lane == nb) {
            my_src = src;
            my_bytes = bytes;
            my_start = start;
            my_off = at;
        }
        nb++;
        bbytes += bytes;
        bend = start + bytes;
        return true;
    }

    // address of item 0 of group g in layer N
    __device__ __forceinline__ const uint8_t *group_src(int N, const Grp &g, const int *route) {
        const Ctx &cx = CX();
        const LayerP &L = layer_of(p, N);
        const uint8_t *blob = g.slot < cx.K ? L.pool + (size_t)route[g.slot] * cx.stride : L.shared;
        switch (g.kind) {
            case KGU: return blob + cx.gu_off;
            case KFC1: return L.fc1x;
            case KLX: return L.lx;
            case KROUTER: return L.router;
            default: return blob + cx.down_off;
        }
    }

    __device__ __forceinline__ bool issue(int N, int ti) {
        const Ctx &cx = CX();
        const Tmplt &t = tmpls()[ti];
        const int *route = SM<int>(cx.sm_rcur) + N * cx.K;
        #pragma unroll 1
        for (int gi = 0; gi < t.n; gi++) {
            const Grp &g = t.g[gi];
            const uint8_t *src = group_src(N, g, route);
            const int per = piece_items<BITS>(g);
            #pragma unroll 1
            for (int i0 = g.lo; i0 < g.hi; i0 += per) {
                const uint32_t bytes = (uint32_t)min(per, g.hi - i0) * g.item_bytes;
                if (!add(src + (size_t)i0 * g.item_bytes, bytes)) return false;
            }
        }
        return true;
    }

    __device__ __forceinline__ bool routes_valid(int N) {
        const Ctx &cx = CX();
        bool ok = true;
        #pragma unroll 1
        for (int k = 0; k < cx.K; k++)
            if ((unsigned)SM<int>(cx.sm_rcur)[N * cx.K + k] >= (unsigned)cx.E) ok = false;
        if (!ok && lane == 0) raise_error(MOE_EINVAL);
        return ok;
    }

    __device__ __forceinline__ void run() {
        const Ctx &cx = CX();
        const int c = blockIdx.x;
        bool ok = true;
#pragma unroll 1
        for (int N = 0; N < cx.depth && ok; N++) {
            // phase 0: router rows (layer 0 routing with its own router; the
            // producer then waits for the route), 1: phase A, 2: phase B
#pragma unroll 1
            for (int ph = N == 0 && cx.own0 ? 0 : 1; ph < 3 && ok; ph++) {
                // validate the route before it turns into addresses
                if (ph == 1 && !(ok = routes_valid(N))) break;
                if (lane == 0) stamp_at(c, N, ST_PA + ph - 1 + (ph == 0));
                ok = issue(N, ph == 0 ? T_R : ph == 1 ? tmpl_A_index(N) : T_B);
                if (ok && ph == 0) ok = flush() && wait_bar_warp(bar(B_ROUTE), 0);
            }
            if (ok && lane == 0) stamp_at(c, N, ST_PE);
        }
        if (ok) flush();
        // never leave the CTA with copies in flight: wait (bounded) for every
        // piece that may not have landed (a barrier pair is reused only after
        // its piece was released, hence landed)
        if (lane == 0) {
            const uint32_t q_end = qb;
            const uint32_t from = q_end > (uint32_t)kNB && landed < q_end - kNB ? q_end - kNB : landed;
            #pragma unroll 1
            for (uint32_t q = from; q < q_end; q++) {
                if (!mbar_try_wait(bar_full(q % kNB), (q / kNB) & 1)) {
                    const uint64_t t0 = now_ns();
                    while (!mbar_try_wait(bar_full(q % kNB), (q / kNB) & 1) &&
                           now_ns() - t0 < cx.timeout_ns) {
                    }
                }
            }
        }
        __syncwarp();
    }
};

// ---------------------------------------------------------------- aux warp
// Prepares each layer's small operands in shared memory (double-buffered by
// layer parity), runs head fc2 of every layer once gelu(fc1 f) is complete,
// and finally the top-K of the heads this CTA owns.
__device__ __forceinline__ uint32_t tag_of(int N) { return CX().epoch * 64u + (uint32_t)N + 1u; }
__device__ __forceinline__ uint32_t tag_router() { return CX().epoch * 64u + 63u; }

// A columns of layer M's gate/up LoRA for this CTA's rows of x
__device__ __noinline__ void aux_load_agu(const LayerP *L, float *agu, int lane) {
    const Ctx &cx = CX();
    const Tmplt &tb = tmpls()[T_B];
    const int r2 = cx.rg + cx.ru, no = tb.o_hi - tb.o_lo;
    const uint16_t *Ag = L->slora[0].A, *Au = L->slora[1].A;
#pragma unroll 1
    for (int i = lane; i < no * r2; i += 32) {
        const int o = tb.o_lo + i / r2, k = i % r2;
        agu[i] = k < cx.rg ? half_f(Ag[(size_t)k * cx.d + o]) : half_f(Au[(size_t)(k - cx.rg) * cx.d + o]);
    }
}

// layer 0's x partials for the gate/up LoRA over this CTA's rows of x0
__device__ __noinline__ void aux_vp0(const LayerP *L0, int c, int lane) {
    const Ctx &cx = CX();
    float *agu = prep_of(1, cx.pp_agu);           // buffer 1 is free until layer 1 is prepared
    aux_load_agu(L0, agu, lane);
    __syncwarp();
    const Tmplt &tb = tmpls()[T_B];
    const int r2 = cx.rg + cx.ru;
    for (int k = lane; k < r2; k += 32) {
        float a = 0.0f;
        #pragma unroll 1
        for (int o = tb.o_lo; o < tb.o_hi; o++) a = fmaf(agu[(o - tb.o_lo) * r2 + k], cx.x0[o], a);
        put_tagged(tagged(cx.off_vp) + (size_t)c * 2 * kMaxR + k, tag_of(0), a);
    }
    __syncwarp();
}

// the routes of layer N (this step's and the previous one's) index the tables
// and the routed LoRA matrices: check them before any use
__device__ __forceinline__ bool aux_routes_ok(int N) {
    const Ctx &cx = CX();
    bool ok = true;
#pragma unroll 1
    for (int k = 0; k < cx.K; k++)
        ok = ok && (unsigned)SM<int>(cx.sm_rcur)[N * cx.K + k] < (unsigned)cx.E &&
             (unsigned)SM<int>(cx.sm_rprev)[N * cx.K + k] < (unsigned)cx.E;
    return ok;
}

__device__ __noinline__ void aux_prep(const LayerP *Lp, const LayerP *Lnext, int N, int lane) {
    const Ctx &cx = CX();
    const LayerP &L = *Lp;
    const Tmplt &ta = tmpls()[tmpl_A_index(N)], &tb = tmpls()[T_B];
    const int *cur = SM<int>(cx.sm_rcur) + N * cx.K, *prev = SM<int>(cx.sm_rprev) + N * cx.K;
    // LoRA scales of this layer
    if (lane == 0) {
        float *sc = prep_of(N, cx.pp_scale);
        sc[SC_G] = L.slora[0].scale;
        sc[SC_U] = L.slora[1].scale;
        sc[SC_DR] = L.lora[2].scale;
        sc[SC_DS] = L.slora[2].scale;
    }
    // K-hot table sums (+ bias) of this CTA's fc1 and l rows
    if (head_runs(N)) {
        float *ts = prep_of(N, cx.pp_tsum);
        const int n1 = ta.f1hi - ta.f1lo, nl = ta.lhi - ta.llo;
        #pragma unroll 1
        for (int i = lane; i < n1 + nl; i += 32) {
            const bool fc1 = i < n1;
            const int row = fc1 ? ta.f1lo + i : ta.llo + (i - n1);
            const int width = fc1 ? cx.H : cx.E;
            const uint16_t *tab = fc1 ? L.fc1_tab : L.l_tab;
            const uint16_t *bias = fc1 ? L.b1 : L.bl;
            float a = 0.0f;
            if (tab) {
                #pragma unroll 1
                for (int k = 0; k < cx.K; k++) a += half_f(tab[(size_t)cur[k] * width + row]);
                #pragma unroll 1
                for (int k = 0; k < cx.K; k++) a += half_f(tab[(size_t)(cx.E + prev[k]) * width + row]);
            }
            if (bias) a += half_f(bias[row]);
            ts[i] = a;
        }
    }
    // B rows of this CTA's gate/up LoRA rows
    if (cx.gu_slot >= 0) {
        float *bgu = prep_of(N, cx.pp_bgu);
        const int gs = cx.gu_slot, r2 = cx.rg + cx.ru;
        const int np = ta.phi[gs] - ta.plo[gs];
        const uint16_t *Bg = L.slora[0].B, *Bu = L.slora[1].B;
        #pragma unroll 1
        for (int i = lane; i < np * r2; i += 32) {
            const int f = ta.plo[gs] + i / r2, k = i % r2;
            bgu[i] = k < cx.rg ? half_f(Bg[(size_t)f * cx.rg + k]) : half_f(Bu[(size_t)f * cx.ru + (k - cx.rg)]);
        }
    }
    // down LoRA: A_d columns of this CTA's gate/up rows, B_d rows of its outputs
    if (cx.dl_mask) {
        float *adn = prep_of(N, cx.pp_adn), *bd = prep_of(N, cx.pp_bd);
        const int no = tb.o_hi - tb.o_lo;
        for (int sl = 0; sl < cx.S; sl++) {
            if (!(cx.dl_mask >> sl & 1u)) continue;
            const int r = dl_rank(sl), j = dl_index(sl);
            const uint16_t *A = lora_a(L, cx.K, cur, sl, 2), *B = lora_bm(L, cx.K, cur, sl, 2);
            const int np = ta.phi[sl] - ta.plo[sl];
            #pragma unroll 1
            for (int i = lane; i < np * r; i += 32) {
                const int f = ta.plo[sl] + i / r, k = i % r;
                adn[(ta.pbase[sl] + i / r) * cx.rd + k] = half_f(A[(size_t)k * cx.F + f]);
            }
            #pragma unroll 1
            for (int i = lane; i < no * r; i += 32) {
                const int o = tb.o_lo + i / r, k = i % r;
                bd[(j * cx.max_orows + i / r) * cx.rd + k] = half_f(B[(size_t)o * r + k]);
            }
        }
    }
    // A columns of the next layer's gate/up LoRA (for its x partials)
    if (cx.gu_slot >= 0 && Lnext) aux_load_agu(Lnext, prep_of(N, cx.pp_agu), lane);
}

// fc2 rows of head N: z = fc2 gelu(fc1 f) + b2 + l f, published per row
__device__ __noinline__ bool aux_fc2(const LayerP *Lp, int N, int lane) {
    const Ctx &cx = CX();
    const Tmplt &tb = tmpls()[T_B];
    const int ne = tb.e_hi - tb.e_lo;
    const uint32_t tg = tag_of(N);
    if (cx.H == 0 || ne <= 0) return true;
    uint8_t *frec = SM<uint8_t>(cx.sm_frec);
    // records of this CTA's rows (plain 16-byte loads)
    const int q16 = cx.rec_H / 16;
#pragma unroll 1
    for (int i = lane; i < ne * q16; i += 32)
        reinterpret_cast<uint4 *>(frec)[i] =
            *reinterpret_cast<const uint4 *>(Lp->fc2 + (size_t)tb.e_lo * cx.rec_H + (size_t)i * 16);
    // every CTA has finished phase A of layer N (fc1 and l rows published):
    // gelu(fc1 f) in one bulk copy (into graw), l f of this CTA's rows (lane
    // i: row i) with plain loads, then gelu(fc1 f) staged chunk by chunk
    if (!poll_flags(cx.off_hflag, tg, lane, 128)) return false;
    const int nch = cx.H / 32;
    uint8_t *gf = SM<uint8_t>(cx.sm_gf);
    float *gsc = SM<float>(cx.sm_gsc), *ghat = SM<float>(cx.sm_ghat);
    const uint64_t *graw = SM<uint64_t>(cx.sm_graw);
    const uint32_t gw = cx.off_ga / 8 + (uint32_t)(N * cx.H);
    if (lane == 0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(bar(B_AUX), (uint32_t)cx.H * 8);
        bulk_g2s(SM<uint8_t>(cx.sm_graw), cx.ws + (size_t)gw * 8, (uint32_t)cx.H * 8, bar(B_AUX));
    }
    float zl = 0.0f;
    if (lane < ne) {
        const uint32_t zw = cx.off_zl / 8 + (uint32_t)(N * cx.E + tb.e_lo + lane);
        const uint64_t v = get_word(ws_words() + zw);
        zl = (uint32_t)(v >> 32) == tg ? __uint_as_float((uint32_t)v) : refetch_word(zw, tg);
    }
    // the k-th fc2 call is for head k (heads run for N = 0, 1, ...)
    if (!wait_bar_warp(bar(B_AUX), (uint32_t)N & 1u)) return false;
#pragma unroll 1
    for (int ch = 0; ch < nch; ch++) {
        const float v = staged(graw, ch * 32 + lane, gw + ch * 32 + lane, tg);
        stage_chunk<4>(&v, lane, gf, ch, nch, gsc, ghat);
    }
    __syncwarp();
    const int lpr = pow2_floor32(nch), rpw = 32 / lpr;
    const int sub = lane % lpr, rsub = lane / lpr;
#pragma unroll 1
    for (int i0 = 0; i0 < ne; i0 += rpw) {
        const int i = i0 + rsub;
        float a;
        rows_dot<4, 1>(frec + (size_t)(i < ne ? i : 0) * cx.rec_H, 0, cx.H, gf, gsc, ghat, sub, lpr, &a);
        const float zli = __shfl_sync(0xffffffffu, zl, i & 31);
        if (i < ne && sub == 0) {
            const int e = tb.e_lo + i;
            const float b = Lp->b2 ? half_f(Lp->b2[e]) : 0.0f;
            put_tagged(tagged(cx.off_z) + (size_t)N * cx.E + e, tg, a + b + zli);
        }
    }
    __syncwarp();
    return true;
}

template <int BITS>
__device__ __noinline__ void aux_main(const Params &p, int c, int lane) {
    const Ctx &cx = CX();
    if (cx.gu_slot >= 0) aux_vp0(&p.layer[0], c, lane);
#pragma unroll 1
    for (int N = 0; N < cx.depth; N++) {
        if (N >= 2 && !wait_bar_warp(bar(B_PREP_EMPTY0 + (N & 1)), ((N >> 1) - 1) & 1)) return;
        if (N == 0 && cx.own0 && !wait_bar_warp(bar(B_ROUTE), 0)) return;
        if (!aux_routes_ok(N)) {
            if (lane == 0) raise_error(MOE_EINVAL);
            return;
        }
        aux_prep(&layer_of(p, N), N + 1 < cx.depth ? &layer_of(p, N + 1) : nullptr, N, lane);
        __syncwarp();
        if (lane == 0) {
            stamp_at(c, N, ST_AUXP);
            mbar_arrive(bar(B_PREP_FULL0 + (N & 1)));
        }
        if (N >= 1 && head_runs(N - 1)) {
            if (!aux_fc2(&layer_of(p, N - 1), N - 1, lane)) return;
            if (lane == 0) stamp_at(c, N - 1, ST_AUXF);
        }
    }
    if (head_runs(cx.depth - 1) && !aux_fc2(&layer_of(p, cx.depth - 1), cx.depth - 1, lane)) return;
    // top-K of the heads this CTA owns: routes for the next step
    const int nxt = (cx.t + 1) % 3;
#pragma unroll 1
    for (int N = c; N < cx.depth; N += cx.n_cta) {
        if (!head_runs(N)) continue;
        const int tgt = N + 1 < cx.depth ? N + 1 : 0;
        if (!route_from_logits(tagged(cx.off_z) + (size_t)N * cx.E, tag_of(N), nxt, tgt, true,
                               false, 256))
            return;
    }
}

// ---------------------------------------------------------------- consumers
// true in the warp that arrives last at counter `cnt` (reset for reuse);
// every warp's shared-memory writes before the call are visible to it
__device__ __forceinline__ bool last_warp(int *cnt) {
    const int lane = threadIdx.x & 31;
    __syncwarp();
    int old = 0;
    if (lane == 0) {
        __threadfence_block();
        old = atomicAdd(cnt, 1);
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != kNW - 1) return false;
    __threadfence_block();
    if (lane == 0) *cnt = 0;
    return true;
}

// x of layer N, staged for the GEMVs (and, with 2-bit experts, in the int4
// layout for the heads); the raw values go to the residual stream.  x is the
// previous layer's out (already copied into the stage with its tags) or x0.
// Warp w stages chunks w, w+kNW, ... (lane j: values j, j+32 of a chunk).
// With want_vp also the partial A x of every CTA for the gate/up LoRA (lane
// k: component k, warp w: CTAs w, w+kNW, ...), summed per lane in CTA order;
// the last warp sums the warps' sums into vx and the sums of squares into
// 1/rms.
template <int BITS>
__device__ __noinline__ bool phase_x(int N, bool want_x, bool want_vp, int warp, int lane) {
    constexpr int VALS = 128 / BITS, PER = VALS / 32;
    const Ctx &cx = CX();
    const int d = cx.d, nch = d / VALS;
    float *stream = SM<float>(cx.sm_stream) + (size_t)(N & 1) * d;
    const uint64_t *stage = SM<uint64_t>(cx.sm_stage);
    const uint32_t tx = N > 0 ? tag_of(N - 1) : 0u;
    const int ncw = want_x && warp < nch ? (nch - warp + kNW - 1) / kNW : 0;   // chunks of this warp
    uint8_t *xf = SM<uint8_t>(cx.sm_xf), *xf4 = SM<uint8_t>(cx.sm_xf4);
    float *xsc = SM<float>(cx.sm_xsc), *xhat = SM<float>(cx.sm_xhat);
    float *xsc4 = SM<float>(cx.sm_xsc4), *xhat4 = SM<float>(cx.sm_xhat4);
    float ss = 0.0f;
#pragma unroll 1
    for (int i = 0; i < ncw; i++) {
        const int ch = warp + kNW * i;
        float v[PER];
#pragma unroll
        for (int m = 0; m < PER; m++) {
            const int pos = ch * VALS + lane + 32 * m;
            v[m] = N == 0 ? cx.x0[pos] : staged(stage, pos, cx.off_out / 8 + pos, tx);
            stream[pos] = v[m];
            ss = fmaf(v[m], v[m], ss);
        }
        stage_chunk<BITS>(v, lane, xf, ch, nch, xsc, xhat);
        if (BITS != 4) {
#pragma unroll
            for (int m = 0; m < PER; m++)
                stage_chunk<4>(&v[m], lane, xf4, ch * PER + m, d / 32, xsc4, xhat4);
        }
    }
    float va = 0.0f;
    if (want_vp) {
        const int nvo = (cx.n_cta - warp + kNW - 1) / kNW;               // CTAs of this warp
        const int n = lane < cx.rg + cx.ru ? nvo : 0;
        if (!read_words(ws_words(), n, tag_of(N),
                        [&](int j) { return cx.off_vp / 8 + (uint32_t)((warp + kNW * j) * 2 * kMaxR + lane); },
                        [&](int, float v) { va += v; }, [&] { va = 0.0f; }))
            return false;
    }
    float *mf = misc_f();
    float *vpw = SM<float>(cx.sm_vpw);
    if (want_x) {
        ss = warp_sum(ss, 32);
        if (lane == 0) mf[M_SS + warp] = ss;
    }
    if (want_vp) vpw[warp * 2 * kMaxR + lane] = va;
    if (last_warp(misc_i() + M_CNT_X)) {
        if (want_x && lane == 0) {
            float tot = 0.0f;
#pragma unroll 1
            for (int w = 0; w < kNW; w++) tot += mf[M_SS + w];
            mf[M_INV] = N > 0 ? 1.0f / sqrtf(tot / d + 1e-6f) : 1.0f;
        }
        if (want_vp) {
            float a = 0.0f;
#pragma unroll 1
            for (int w = 0; w < kNW; w++) a += vpw[w * 2 * kMaxR + lane];
            SM<float>(cx.sm_vx)[lane] = a;
        }
    }
    return true;
}

// h of every slot, staged per slot (warp w takes chunks w, w+kNW, ... of the
// concatenated slots), from the stage: the h words, then for each down-LoRA
// slot the partial A_d h words of its owner CTAs (32 per owner, lane k:
// component k), which warp w sums for owners w, w+kNW, ... in order into vdw;
// the last warp sums the warps' sums into vd.
template <int BITS>
__device__ __noinline__ bool phase_h(int N, int warp, int lane) {
    constexpr int VALS = 128 / BITS, PER = VALS / 32;
    const Ctx &cx = CX();
    const Tmplt &ta = tmpls()[tmpl_A_index(N)];
    const int cps = cx.F / VALS;                    // chunks per slot
    const int nch = cx.S * cps;
    const int ncw = warp < nch ? (nch - warp + kNW - 1) / kNW : 0;
    const uint32_t tg = tag_of(N);
    const uint64_t *stage = SM<uint64_t>(cx.sm_stage);
    uint8_t *hf = SM<uint8_t>(cx.sm_hf);
    float *hsc = SM<float>(cx.sm_hsc), *hhat = SM<float>(cx.sm_hhat);
#pragma unroll 1
    for (int i = 0; i < ncw; i++) {
        const int ch = warp + kNW * i, sc = ch / cps, cl = ch % cps;
        float v[PER];
#pragma unroll
        for (int m = 0; m < PER; m++) {
            const int pos = ch * VALS + lane + 32 * m;
            v[m] = staged(stage, pos, cx.off_h / 8 + pos, tg);
        }
        stage_chunk<BITS>(v, lane, hf + (size_t)sc * cx.F * 2, cl, cps, hsc + sc * cps, hhat + sc * cps);
    }
    if (cx.dl_mask) {
        float *vdw = SM<float>(cx.sm_vdw) + warp * cx.n_dl * kMaxR;
        int base = cx.S * cx.F;
#pragma unroll 1
        for (int sl = 0; sl < cx.S; sl++) {
            if (!(cx.dl_mask >> sl & 1u)) continue;
            const int no = ta.own1[sl] - ta.own0[sl] + 1, j = dl_index(sl);
            float a = 0.0f;
            if (lane < dl_rank(sl)) {
#pragma unroll 1
                for (int i = warp; i < no; i += kNW)
                    a += staged(stage, base + i * kMaxR + lane,
                                cx.off_vdp / 8 + (uint32_t)((sl * cx.n_cta + ta.own0[sl] + i) * kMaxR + lane), tg);
            }
            vdw[j * kMaxR + lane] = a;
            base += no * kMaxR;
        }
        if (last_warp(misc_i() + M_CNT_H)) {
            float *vd = SM<float>(cx.sm_vd), *vdw0 = SM<float>(cx.sm_vdw);
#pragma unroll 1
            for (int j = 0; j < cx.n_dl; j++) {
                float a = 0.0f;
#pragma unroll 1
                for (int w = 0; w < kNW; w++) a += vdw0[(w * cx.n_dl + j) * kMaxR + lane];
                vd[j * kMaxR + lane] = a;
            }
        }
    }
    return true;
}

// ---- tasks -----------------------------------------------------------
// Gate/up row pairs: h = silu(g) * u (+ gate/up LoRA), published; the
// partial A_d h of a down-LoRA slot accumulates in vdacc[warp].
template <int BITS>
__device__ __forceinline__ void task_gu(int N, int gi, const uint8_t *base, int i, int cnt, int lpr,
                                     float inv, int warp, int lane) {
    const Ctx &cx = CX();
    const Tmplt &t = tmpls()[tmpl_A_index(N)];
    const Grp &g = t.g[gi];
    const int sub = lane % lpr, rsub = lane / lpr;
    const int f = i + rsub;
    const bool ok = rsub < cnt;
    const int sl = g.slot;
    float r2v[2];
    rows_dot<BITS, 2>(base + (size_t)(ok ? rsub : 0) * g.item_bytes, cx.rec_d, cx.d,
                      SM<uint8_t>(cx.sm_xf), SM<float>(cx.sm_xsc), SM<float>(cx.sm_xhat), sub, lpr,
                      r2v);
    float gg = r2v[0] * inv, uu = r2v[1] * inv;
    if (sl == cx.gu_slot) {
        const float *sc = prep_of(N, cx.pp_scale);
        const float *bgu = prep_of(N, cx.pp_bgu) + (ok ? f - t.plo[sl] : 0) * (cx.rg + cx.ru);
        const float *vx = SM<float>(cx.sm_vx);
        float a = 0.0f, b = 0.0f;
        if (ok) {
            #pragma unroll 1
            for (int k = sub; k < cx.rg; k += lpr) a = fmaf(bgu[k], vx[k], a);
            #pragma unroll 1
            for (int k = sub; k < cx.ru; k += lpr) b = fmaf(bgu[cx.rg + k], vx[cx.rg + k], b);
        }
        gg += sc[SC_G] * inv * warp_sum(a, lpr);
        uu += sc[SC_U] * inv * warp_sum(b, lpr);
    }
    const float h = silu_f(gg) * uu;
    if (ok && sub == 0) put_tagged(tagged(cx.off_h) + (size_t)sl * cx.F + f, tag_of(N), h);
    if (cx.dl_mask >> sl & 1u) {
        const int r = dl_rank(sl), j = dl_index(sl);
        const float *adn = prep_of(N, cx.pp_adn) + (t.pbase[sl] + (ok ? f - t.plo[sl] : 0)) * cx.rd;
        float *vdacc = SM<float>(cx.sm_vdacc) + (warp * cx.n_dl + j) * kMaxR;
        #pragma unroll 1
        for (int k0 = 0; k0 < r; k0 += lpr) {
            const int k = k0 + sub;
            float a = (ok && k < r) ? adn[k] * h : 0.0f;
            #pragma unroll 1
            for (int o = lpr; o < 32; o <<= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (rsub == 0 && k < r) vdacc[k] += a;
        }
    }
}

// fc1 / l / router rows on x, with the K-hot table sums and the bias.
template <int BITS>
__device__ __forceinline__ void task_head(int N, int ti, int gi, const uint8_t *base, int i, int cnt,
                                       int lpr, float inv, int lane) {
    const Ctx &cx = CX();
    const Tmplt &t = tmpls()[ti];
    const Grp &g = t.g[gi];
    const int sub = lane % lpr, rsub = lane / lpr;
    const int row = i + rsub;
    const bool ok = rsub < cnt;
    float a;
    rows_dot<4, 1>(base + (size_t)(ok ? rsub : 0) * g.item_bytes, 0, cx.d, SM<uint8_t>(cx.sm_xf4),
                   SM<float>(cx.sm_xsc4), SM<float>(cx.sm_xhat4), sub, lpr, &a);
    if (ok && sub == 0) {
        a *= inv;
        const uint32_t tg = tag_of(N);
        if (g.kind == KFC1) {
            a += prep_of(N, cx.pp_tsum)[row - t.f1lo];
            put_tagged(tagged(cx.off_ga) + (size_t)N * cx.H + row, tg, gelu_erf_f(a));
        } else if (g.kind == KLX) {
            a += prep_of(N, cx.pp_tsum)[(t.f1hi - t.f1lo) + row - t.llo];
            if (cx.H > 0) put_tagged(tagged(cx.off_zl) + (size_t)N * cx.E + row, tg, a);
            else put_tagged(tagged(cx.off_z) + (size_t)N * cx.E + row, tg, a);
        } else {
            put_tagged(tagged(cx.off_zr) + row, tag_router(), a);
        }
    }
}

// End of phase A: this CTA's h rows (and fc1 / l rows) are out.  The last warp
// to get here publishes, for the owners of a down-LoRA slot's gate/up rows,
// the partial A_d h (sum of the warps' partials), then the CTA's flag with a
// release store: the other warps' writes reach it through the CTA-scope
// hand-over of last_warp, and the release orders them all before the flag (a
// reader that still finds an old tag reads again).
__device__ __noinline__ void publish_a(int N, int c, int lane) {
    if (!last_warp(misc_i() + M_CNT_A)) return;
    const Ctx &cx = CX();
    const Tmplt &ta = tmpls()[tmpl_A_index(N)];
    const uint32_t tg = tag_of(N);
#pragma unroll 1
    for (int sl = 0; sl < cx.S; sl++) {
        if (!(cx.dl_mask >> sl & 1u) || c < ta.own0[sl] || c > ta.own1[sl]) continue;
        const int r = dl_rank(sl), j = dl_index(sl);
        if (lane < r) {
            float a = 0.0f;
            #pragma unroll 1
            for (int w = 0; w < kNW; w++) {
                float *v = SM<float>(cx.sm_vdacc) + (w * cx.n_dl + j) * kMaxR + lane;
                a += *v;
                *v = 0.0f;
            }
            put_tagged(tagged(cx.off_vdp) + ((size_t)sl * cx.n_cta + c) * kMaxR + lane, tg, a);
        }
    }
    __syncwarp();
    if (lane == 0) put_flag(flag_of(cx.off_hflag, c), tg);
}

// End of phase B: this CTA's rows of out are published.  The last warp
// publishes the next layer's gate/up LoRA partial over those rows (sum of the
// warps' partials), then the CTA's flag (release store, as in publish_a).
__device__ __noinline__ void publish_d(int N, int c, int lane) {
    const Ctx &cx = CX();
    if (!last_warp(misc_i() + M_CNT_D)) return;
    const uint32_t tg = tag_of(N);
    if (cx.gu_slot >= 0) {
        const int r2 = cx.rg + cx.ru;
        float *vnw = SM<float>(cx.sm_vnw);
        float a = 0.0f;
        #pragma unroll 1
        for (int w = 0; w < kNW; w++) {
            a += vnw[w * 2 * kMaxR + lane];
            vnw[w * 2 * kMaxR + lane] = 0.0f;
        }
        if (lane < r2) put_tagged(tagged(cx.off_vp) + (size_t)c * 2 * kMaxR + lane, tag_of(N + 1), a);
    }
    __syncwarp();
    if (lane == 0) put_flag(flag_of(cx.off_xflag, c), tg);
}

// Ring position and task rotation of a consumer warp, carried from one
// template's pieces to the next.
struct RunState {
    uint64_t head;
    uint32_t off, q, tasks, ok;
};

// Consumes this CTA's pieces of template ti (phase R or A), in the producer's
// order; warp tasks of rpw items go round-robin to the consumer warps.  A
// leaf function: the tasks are inlined, so no loop state is saved around
// calls.
template <int BITS>
__device__ __noinline__ RunState run_tmpl(int N, int ti, float inv, int warp, int lane, RunState st) {
    const Ctx &cx = CX();
    const Tmplt &t = tmpls()[ti];
    const uint8_t *ring = SM<uint8_t>(cx.sm_ring);
    RingPos rp;
    rp.head = st.head;
    rp.off = st.off;
    rp.q = st.q;
    uint32_t tasks = st.tasks;
#pragma unroll 1
    for (int gi = 0; gi < t.n; gi++) {
        const Grp &g = t.g[gi];
        const int kind = g.kind, lo = g.lo, hi = g.hi;
        const uint32_t ib = g.item_bytes;
        const int per = piece_items<BITS>(g);
        const int lpr = pow2_floor32(item_chunks<BITS>(g));
        const int rpw = 32 / lpr;
        #pragma unroll 1
        for (int i0 = lo; i0 < hi; i0 += per) {
            const int cnt = min(per, hi - i0);
            uint32_t at;
            rp.place((uint32_t)cnt * ib, cx.ring_bytes, &at);
            const uint32_t q = rp.q++;
            if (!wait_bar_warp_inl(bar_full(q % kNB), (q / kNB) & 1)) return RunState{rp.head, rp.off, rp.q, tasks, 0u};
            const uint8_t *base = ring + at;
            const int ntask = (cnt + rpw - 1) / rpw;
            const int k0 = (int)((kNW + warp - tasks % kNW) % kNW);
            #pragma unroll 1
            for (int k = k0; k < ntask; k += kNW) {
                const int li = k * rpw;
                const uint8_t *b = base + (size_t)li * ib;
                const int n = min(rpw, cnt - li);
                if (kind == KGU) task_gu<BITS>(N, gi, b, i0 + li, n, lpr, inv, warp, lane);
                else task_head<BITS>(N, ti, gi, b, i0 + li, n, lpr, inv, lane);
            }
            tasks += ntask;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty(q % kNB));
        }
    }
    return RunState{rp.head, rp.off, rp.q, tasks, 1u};
}

// Phase B in one pass per output row: the S pieces (one per slot) are waited
// for, then the warp owning output o (o - o_lo = warp mod kNW) spreads the
// S * cps (slot, chunk) pairs of the row over its lanes, weights each slot's
// part by its combine weight, adds the down-LoRA terms, reduces once and
// writes out = residual + sum (published, with its share of the next layer's
// gate/up LoRA partial in vnw[warp]).  Then the pieces are released.
template <int BITS>
__device__ __noinline__ RunState run_down(int N, int warp, int lane, RunState st) {
    constexpr int VALS = 128 / BITS;
    const Ctx &cx = CX();
    const Tmplt &t = tmpls()[T_B];
    const uint8_t *ring = SM<uint8_t>(cx.sm_ring);
    uint32_t *poff = SM<uint32_t>(cx.sm_poff) + warp * kMaxSlots;
    RingPos rp;
    rp.head = st.head;
    rp.off = st.off;
    rp.q = st.q;
    const int no = t.o_hi - t.o_lo;
    const uint32_t q0 = rp.q;
#pragma unroll 1
    for (int sl = 0; sl < cx.S; sl++) {
        uint32_t at;
        rp.place((uint32_t)(no > 0 ? no : 1) * cx.rec_F, cx.ring_bytes, &at);
        const uint32_t q = rp.q++;
        if (lane == 0) poff[sl] = at;
        if (!wait_bar_warp_inl(bar_full(q % kNB), (q / kNB) & 1)) return RunState{rp.head, rp.off, rp.q, st.tasks, 0u};
    }
    __syncwarp();
    const int cps = cx.F / VALS, npair = cx.S * cps, cb = cx.F * BITS / 8;
    const uint8_t *hf = SM<uint8_t>(cx.sm_hf);
    const float *hsc = SM<float>(cx.sm_hsc), *hhat = SM<float>(cx.sm_hhat);
    const float *rw = SM<float>(cx.sm_rw) + N * cx.K;
    const float *stream = SM<float>(cx.sm_stream) + (size_t)(N & 1) * cx.d;
    const float *sc = prep_of(N, cx.pp_scale);
    const bool last = N + 1 >= cx.depth;
    const bool vp = cx.gu_slot >= 0 && !last;
    const int r2 = cx.rg + cx.ru;
    float vn = 0.0f;
#pragma unroll 1
    for (int ol = warp; ol < no; ol += kNW) {
        const int o = t.o_lo + ol;
        float acc = 0.0f;
        // the lane's (slot, chunk) pairs: lane, lane + 32, ...
        int sl = lane / cps, c = lane - sl * cps;
#pragma unroll 1
        for (int pi = lane; pi < npair; pi += 32) {
            const uint8_t *rec = ring + poff[sl] + (size_t)ol * cx.rec_F;
            const uint4 q = *reinterpret_cast<const uint4 *>(rec + (size_t)kChunk * c);
            const uint32_t sbw = *reinterpret_cast<const uint32_t *>(rec + cb + 4 * ((c * VALS) / kGroup));
            int dq;
            chunk_dot_fix<BITS, 1>(&q, reinterpret_cast<const uint4 *>(hf + (size_t)sl * cx.F * 2), cps, c, &dq);
            const float2 sb = sb_f(sbw);
            const float y = fmaf(sb.x, (float)dq * hsc[sl * cps + c], sb.y * hhat[sl * cps + c]);
            acc = fmaf(sl < cx.K ? rw[sl] : 1.0f, y, acc);
            c += 32;
            while (c >= cps && sl < cx.S) {
                c -= cps;
                sl++;
            }
        }
        // down LoRA of the slots that have one: lane k holds component k
        if (cx.dl_mask) {
            const float *bd = prep_of(N, cx.pp_bd);
            const float *vd = SM<float>(cx.sm_vd);
#pragma unroll 1
            for (int s2 = 0; s2 < cx.S; s2++) {
                if (!(cx.dl_mask >> s2 & 1u)) continue;
                const int j = dl_index(s2);
                if (lane < dl_rank(s2))
                    acc = fmaf((s2 < cx.K ? rw[s2] : 1.0f) * sc[s2 < cx.K ? SC_DR : SC_DS] *
                                   bd[(j * cx.max_orows + ol) * cx.rd + lane],
                               vd[j * kMaxR + lane], acc);
            }
        }
        const float outv = stream[o] + warp_sum(acc, 32);
        if (lane == 0) {
            if (!last) put_tagged(tagged(cx.off_out) + o, tag_of(N), outv);
            else cx.out[o] = outv;
        }
        if (vp && lane < r2) vn = fmaf(prep_of(N, cx.pp_agu)[ol * r2 + lane], outv, vn);
    }
    if (vp) SM<float>(cx.sm_vnw)[warp * 2 * kMaxR + lane] += vn;
    __syncwarp();
    if (lane < cx.S) mbar_arrive(bar_empty((q0 + lane) % kNB));
    return RunState{rp.head, rp.off, rp.q, st.tasks, 1u};
}

template <int BITS>
struct Consumer {
    int c, warp, lane;   // warp: 0 .. kNW-1
    RingPos rp;
    uint32_t nsync = 0, xuses = 0, huses = 0, tasks = 0;

    // barrier among the consumer warps (bounded)
    __device__ __forceinline__ bool sync() {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_CONS));
        const bool ok = wait_bar_warp(bar(B_CONS), nsync & 1);
        nsync++;
        __syncwarp();
        return ok;
    }

    // Waits until every CTA's flag at `off` has reached `tg` (warp 0 polls the
    // flags), then warp 0 lane 0 copies the exchanged words into the stage
    // with bulk copies completing on mbarrier `b` (issue(b) arms its byte
    // count and starts them); every warp sleeps on `b` until they land.
    template <typename Issue>
    __device__ __forceinline__ bool flag_copy(uint32_t off, uint32_t tg, uint64_t *b, uint32_t &uses,
                                              Issue issue) {
        if (warp == 0) {
            if (!poll_flags(off, tg, lane, 0)) return false;
            if (lane == 0) {
                fence_proxy_async();
                issue(b);
            }
        }
        const bool ok = wait_bar_warp(b, uses & 1);
        uses++;
        return ok;
    }

    __device__ __forceinline__ bool gu_lora_here(int N) const {
        const Ctx &cx = CX();
        if (cx.gu_slot < 0) return false;
        const Tmplt &ta = tmpls()[tmpl_A_index(N)];
        return ta.phi[cx.gu_slot] > ta.plo[cx.gu_slot];
    }

    __device__ __forceinline__ bool run(int N, int ti, float inv) {
        const RunState st = run_tmpl<BITS>(N, ti, inv, warp, lane, RunState{rp.head, rp.off, rp.q, tasks, 1u});
        rp.head = st.head;
        rp.off = st.off;
        rp.q = st.q;
        tasks = st.tasks;
        return st.ok != 0;
    }

    __device__ __forceinline__ bool layer(int N) {
        const Ctx &cx = CX();
        if (warp == 0 && lane == 0) stamp_at(c, N, ST_L0);
        const bool r0 = N == 0 && cx.own0;
        const bool vp = gu_lora_here(N);
        // every CTA's rows of the previous layer's out: one bulk copy
        if (N > 0 && !flag_copy(cx.off_xflag, tag_of(N - 1), bar(B_X), xuses, [&](uint64_t *b) {
                const uint32_t bytes = (uint32_t)cx.d * 8;
                mbar_arrive_expect_tx(b, bytes);
                bulk_g2s(SM<uint8_t>(cx.sm_stage), cx.ws + cx.off_out, bytes, b);
            }))
            return false;
        if (!phase_x<BITS>(N, true, vp && !r0, warp, lane)) return false;
        if (!sync()) return false;
        const float inv = misc_f()[M_INV];
        if (warp == 0 && lane == 0) stamp_at(c, N, ST_X);
        if (r0) {
            if (!run(0, T_R, inv)) return false;
            // layer 0's own route (every CTA alike)
            if (warp == 0) {
                if (!route_from_logits(tagged(cx.off_zr), tag_router(), cx.t % 3, 0, c == 0, true, 0))
                    return false;
                if (lane == 0) mbar_arrive(bar(B_ROUTE));
            }
            if (vp && !phase_x<BITS>(0, false, true, warp, lane)) return false;
            if (!sync()) return false;
        }
        if (!wait_bar_warp(bar(B_PREP_FULL0 + (N & 1)), (N >> 1) & 1)) return false;
        if (!run(N, tmpl_A_index(N), inv)) return false;
        publish_a(N, c, lane);
        if (warp == 0 && lane == 0) stamp_at(c, N, ST_A);
        // every CTA's h rows, then each down-LoRA slot's owner partials
        if (!flag_copy(cx.off_hflag, tag_of(N), bar(B_H), huses, [&](uint64_t *b) {
                const Tmplt &ta = tmpls()[tmpl_A_index(N)];
                uint32_t bytes = (uint32_t)cx.S * cx.F * 8;
#pragma unroll 1
                for (int sl = 0; sl < cx.S; sl++)
                    if (cx.dl_mask >> sl & 1u) bytes += (uint32_t)(ta.own1[sl] - ta.own0[sl] + 1) * kMaxR * 8;
                mbar_arrive_expect_tx(b, bytes);
                uint8_t *stage = SM<uint8_t>(cx.sm_stage);
                bulk_g2s(stage, cx.ws + cx.off_h, (uint32_t)cx.S * cx.F * 8, b);
                uint32_t at = (uint32_t)cx.S * cx.F * 8;
#pragma unroll 1
                for (int sl = 0; sl < cx.S; sl++) {
                    if (!(cx.dl_mask >> sl & 1u)) continue;
                    const uint32_t nb = (uint32_t)(ta.own1[sl] - ta.own0[sl] + 1) * kMaxR * 8;
                    bulk_g2s(stage + at,
                             cx.ws + cx.off_vdp + ((size_t)sl * cx.n_cta + ta.own0[sl]) * kMaxR * 8, nb, b);
                    at += nb;
                }
            }))
            return false;
        if (!phase_h<BITS>(N, warp, lane)) return false;
        if (!sync()) return false;               // h and vd visible to all warps
        if (warp == 0 && lane == 0) stamp_at(c, N, ST_H);
        {                                        // down rows + combine
            const RunState rs = run_down<BITS>(N, warp, lane, RunState{rp.head, rp.off, rp.q, tasks, 1u});
            rp.head = rs.head;
            rp.off = rs.off;
            rp.q = rs.q;
            if (!rs.ok) return false;
        }
        if (N + 1 < cx.depth) publish_d(N, c, lane);
        if (warp == 0 && lane == 0) stamp_at(c, N, ST_D);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PREP_EMPTY0 + (N & 1)));
        return true;
    }

    __device__ __forceinline__ void run_all() {
        const Ctx &cx = CX();
        if (cx.debug_unset_wait && c == 0 && warp == 0) {
            // test hook: a flag nothing ever sets, so this wait runs out
            const uint32_t idx[1] = {C_NEVER / 2};
            float v[1];
            if (!__all_sync(0xffffffffu, poll_vals<1>(reinterpret_cast<const uint64_t *>(cx.ws), idx,
                                                      1u, 0u, 0xFFFFFFFFu, 0xFFFFFFFFu, v)))
                return;
        }
        #pragma unroll 1
        for (int N = 0; N < cx.depth; N++)
            if (!layer(N)) return;
    }
};

// The three roles, each in a function of its own (its own registers: no
// spills of one role's loop state into local memory because of another's).
template <int BITS>
__device__ __noinline__ void producer_main(const Params &p, int lane) {
    Producer<BITS> pr{p, lane};
    pr.run();
}

template <int BITS>
__device__ __noinline__ void consumer_main(int c, int warp, int lane) {
    Consumer<BITS> cons{c, warp, lane};
    cons.run_all();
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const __grid_constant__ Params p) {
    const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the context: copied into shared memory (its first bytes), read from there
    {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(&p.cx);
        uint32_t *dst = reinterpret_cast<uint32_t *>(g_smem);
        #pragma unroll 1
        for (int i = threadIdx.x; i < (int)(sizeof(Ctx) / 4); i += blockDim.x) dst[i] = src[i];
    }
    __syncthreads();
    if (threadIdx.x == 0)
        reinterpret_cast<Ctx *>(g_smem)->epoch =
            (uint32_t)ld_flag(reinterpret_cast<const int *>(p.cx.ws) + C_EPOCH);
    const Ctx &cx = CX();

    // routes of this step (layer 0's own route is filled in later)
    const int use = p.cx.t % 3, prv = (p.cx.t + 2) % 3;
#pragma unroll 1
    for (int i = threadIdx.x; i < p.cx.depth * p.cx.K; i += blockDim.x) {
        SM<int>(p.cx.sm_rcur)[i] = p.cx.ridx[(size_t)use * p.cx.depth * p.cx.K + i];
        SM<float>(p.cx.sm_rw)[i] = p.cx.rw[(size_t)use * p.cx.depth * p.cx.K + i];
        SM<int>(p.cx.sm_rprev)[i] = p.cx.ridx[(size_t)prv * p.cx.depth * p.cx.K + i];
    }
#pragma unroll 1
    for (int i = threadIdx.x; i < kNW * p.cx.n_dl * kMaxR; i += blockDim.x)
        SM<float>(p.cx.sm_vdacc)[i] = 0.0f;
#pragma unroll 1
    for (int i = threadIdx.x; i < kNW * 2 * kMaxR; i += blockDim.x) SM<float>(p.cx.sm_vnw)[i] = 0.0f;
    if (threadIdx.x == 0) {
        uint64_t *bars = SM<uint64_t>(p.cx.sm_bar);
        #pragma unroll 1
        for (int i = 0; i < kNB; i++) {
            mbar_init(bars + i, 1);
            mbar_init(bars + kNB + i, kNW);
        }
        uint64_t *b = bars + 2 * kNB;
        mbar_init(b + B_ROUTE, 1);
        mbar_init(b + B_CONS, kNW);
        mbar_init(b + B_END, kCons0 + kNW);
        mbar_init(b + B_X, 1);
        mbar_init(b + B_H, 1);
        mbar_init(b + B_AUX, 1);
        #pragma unroll 1
        for (int k = 0; k < 2; k++) {
            mbar_init(b + B_PREP_FULL0 + k, 1);
            mbar_init(b + B_PREP_EMPTY0 + k, kNW);
        }
        int *mi = SM<int>(p.cx.sm_misc);
        #pragma unroll 1
        for (int i = M_CNT_A; i <= M_CNT_D; i++) mi[i] = 0;
        mbar_fence_init();
        mi[M_TMPL_OK] = build_templates(c, SM<Tmplt>(p.cx.sm_tmpl)) ? 1 : 0;
        if (!mi[M_TMPL_OK]) raise_error(MOE_EINVAL);
    }
    __syncthreads();

    if (misc_i()[M_TMPL_OK] && !aborted()) {
        if (warp == kProducerWarp) producer_main<BITS>(p, lane);
        else if (warp == kAuxWarp) aux_main<BITS>(p, c, lane);
        else consumer_main<BITS>(c, warp - kCons0, lane);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(B_END));
    if (threadIdx.x == 0) {
        // the step is complete in this CTA once every warp has arrived
        if (wait_bar(bar(B_END), 0) && !aborted()) {
            __threadfence();
            const int prev = atomicAdd(ctrl() + C_DONE, 1);
            if (prev == cx.n_cta - 1) {
                atomicExch(ctrl() + C_DONE, 0);
                atomicAdd(ctrl() + C_EPOCH, 1);
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
    offs[1] = take((size_t)n_cta * 2 * kMaxR);              // partial A x per CTA (gate/up LoRA)
    offs[2] = take((size_t)S * n_cta * kMaxR);              // partial A_d h per owner CTA
    offs[3] = take((size_t)depth * (H > 0 ? H : 1));        // gelu(fc1 f) per layer
    offs[4] = take((size_t)depth * E);                      // l f per layer
    offs[5] = take((size_t)E);                              // router logits
    offs[6] = take((size_t)depth * E);                      // head logits per layer
    offs[7] = take((size_t)d);                              // out
    offs[8] = take((size_t)(n_cta + 1) / 2);                // per-CTA flag: out (+ partials) published
    offs[9] = take((size_t)(n_cta + 1) / 2);                // per-CTA flag: phase A published
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
            if (r0 != q0 || r1 != q1 || r0 < 0 || r0 > kMaxR || r1 < 0 || r1 > kMaxR)
                return fail(MOE_EUNSUPPORTED,
                            "decode_step: LoRA ranks must match across layers and be <= %d", kMaxR);
            if ((r0 && (!e.lora[j].A || !e.lora[j].B)) ||
                (r1 && (!e.shared_lora[j].A || !e.shared_lora[j].B)))
                return fail(MOE_EINVAL, "decode_step: LoRA with NULL A or B");
        }
        // the shared gate and up adapters' A x share one 32-lane vector
        if (e.shared && e.shared_lora[0].r + e.shared_lora[1].r > kMaxR)
            return fail(MOE_EUNSUPPORTED, "decode_step: shared gate + up LoRA ranks %d + %d above %d",
                        e.shared_lora[0].r, e.shared_lora[1].r, kMaxR);
        if (e.lora[0].r || e.lora[1].r)
            return fail(MOE_EUNSUPPORTED,
                        "decode_step: gate/up LoRA on routed experts runs through the per-call path");
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
    return MOE_OK;
}

namespace moe {
int check_decode_stack(const moe_stack_desc *sd) { return check_stack(sd); }
}  // namespace moe

extern "C" size_t moe_decode_step_workspace_bytes(const moe_stack_desc *sd) {
    if (check_stack(sd) != MOE_OK) return 0;
    const moe_experts_desc &e0 = sd->experts[0];
    const int H = (sd->depth > 1 || sd->self_predict) ? sd->heads[0].H : 0;
    uint32_t offs[10];
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
    if (sd->slot_map || sd->layer_ready)
        return fail(MOE_EUNSUPPORTED, "decode_step: slot_map / layer_ready are for moe_decode_step_chain");
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
    cfg.gridDim = dim3(p.cx.n_cta);
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
    Ctx &cx = p.cx;
    cx.d = e0.d;
    cx.F = e0.F;
    cx.E = e0.E;
    cx.K = sd->K;
    cx.H = heads ? sd->heads[0].H : 0;
    cx.S = sd->K + (e0.shared ? 1 : 0);
    cx.depth = sd->depth;
    cx.n_res = sd->n_layers;
    cx.self_predict = sd->self_predict;
    cx.own0 = !sd->self_predict;
    cx.t = t;
    const int bits = e0.bits;
    const BlobLayout L = blob_layout(cx.d, cx.F, bits);
    cx.stride = e0.expert_stride;
    cx.gu_off = (uint32_t)L.gu_off;
    cx.down_off = (uint32_t)L.down_off;
    cx.rec_d = (uint32_t)L.gu_rec;
    cx.rec_F = (uint32_t)L.down_rec;
    cx.rec_dh = (uint32_t)record_bytes(cx.d, 4);
    cx.rec_H = cx.H ? (uint32_t)record_bytes(cx.H, 4) : 0;
    // LoRA: gate/up only on the shared slot; down on routed and/or shared
    const moe_lora_desc *sl = e0.shared ? e0.shared_lora : nullptr;
    cx.rg = sl ? sl[0].r : 0;
    cx.ru = sl ? sl[1].r : 0;
    cx.gu_slot = (cx.rg || cx.ru) ? cx.S - 1 : -1;
    if (cx.rg + cx.ru > 32)
        return fail(MOE_EUNSUPPORTED, "decode_step: gate + up LoRA ranks %d + %d exceed 32", cx.rg,
                    cx.ru);
    cx.rdr = e0.lora[2].r;
    cx.rds = sl ? sl[2].r : 0;
    cx.dl_mask = 0;
    if (cx.rdr)
        for (int s = 0; s < cx.K; s++) cx.dl_mask |= 1u << s;
    if (cx.rds) cx.dl_mask |= 1u << (cx.S - 1);
    cx.n_dl = __builtin_popcount(cx.dl_mask);
    cx.rd = std::max(cx.rdr, cx.rds);
    cx.x0 = x0;
    cx.out = out;
    cx.ridx = ridx;
    cx.rw = rw;
    cx.rmargin = rmargin;
    cx.ws = static_cast<uint8_t *>(ws);
    const int sms = device_sms();
    int dev = 0, smem_max = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (sms <= 0 || smem_max <= 0) return fail(MOE_ECUDA, "decode_step: no device attributes");
    if (sms > 256) return fail(MOE_EUNSUPPORTED, "decode_step: %d SMs (at most 256)", sms);
    cx.n_cta = sms;
    uint32_t offs[10];
    size_t total = 0;
    step_ws_layout(cx.d, cx.F, cx.E, cx.H, cx.S, cx.depth, sms, offs, &total);
    cx.off_h = offs[0];
    cx.off_vp = offs[1];
    cx.off_vdp = offs[2];
    cx.off_ga = offs[3];
    cx.off_zl = offs[4];
    cx.off_zr = offs[5];
    cx.off_z = offs[6];
    cx.off_out = offs[7];
    cx.off_xflag = offs[8];
    cx.off_hflag = offs[9];
    cx.timeout_ns = sd->timeout_ns ? sd->timeout_ns : 1000000000ull;
    cx.debug_unset_wait = sd->debug_unset_wait;
    cx.trace = sd->debug_trace;
    cx.inflight = sd->inflight_bytes ? sd->inflight_bytes : kDefaultInflight;
    if (cx.inflight < (uint32_t)kMaxPiece) cx.inflight = kMaxPiece;
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

    // per-CTA bounds of the byte split (checked again on the device)
    {
        const long long gu = (long long)cx.S * cx.F * 2 * cx.rec_d;
        const long long total_a = gu + (heads ? (long long)(cx.H + cx.E) * cx.rec_dh : 0);
        const long long share = (total_a + sms - 1) / sms;
        cx.max_pairs = (int)(share / (2 * cx.rec_d)) + cx.S + 1;
        cx.max_hrows = (int)(share / cx.rec_dh) + 3;
        // CTAs whose share holds some of one slot's gate/up rows: at most the
        // slot's part of the phase without head rows (the smaller total)
        cx.max_owners = sms / cx.S + 3;
        if (cx.max_owners > sms) cx.max_owners = sms;
    }
    cx.max_orows = (cx.d + sms - 1) / sms;
    cx.max_erows = (cx.E + sms - 1) / sms;
    if (cx.max_erows > 32 || cx.max_erows * (int)cx.rec_H > 16384)
        return fail(MOE_EUNSUPPORTED, "decode_step: E=%d too large for %d SMs", cx.E, sms);

    // shared-memory layout: the context first
    const int VALS = 128 / bits;
    size_t off = sizeof(Ctx);
    auto take = [&](size_t bytes) {
        off = al(off, 16);
        const size_t o = off;
        off += bytes;
        return (uint32_t)o;
    };
    const int r2 = cx.rg + cx.ru;
    const int ndl = std::max(cx.n_dl, 1);
    cx.sm_bar = take((size_t)(2 * kNB + B_COUNT) * 8);
    cx.sm_pend = take((size_t)kNB * 8);
    cx.sm_tmpl = take(T_COUNT * sizeof(Tmplt));
    cx.sm_xf = take((size_t)cx.d * 2);
    cx.sm_xsc = take((size_t)(cx.d / VALS) * 4);
    cx.sm_xhat = take((size_t)(cx.d / VALS) * 4);
    cx.sm_xf4 = bits == 4 ? cx.sm_xf : take((size_t)cx.d * 2);
    cx.sm_xsc4 = bits == 4 ? cx.sm_xsc : take((size_t)(cx.d / 32) * 4);
    cx.sm_xhat4 = bits == 4 ? cx.sm_xhat : take((size_t)(cx.d / 32) * 4);
    cx.sm_stream = take((size_t)2 * cx.d * 4);
    cx.sm_hf = take((size_t)cx.S * cx.F * 2);
    cx.sm_hsc = take((size_t)cx.S * (cx.F / VALS) * 4);
    cx.sm_hhat = take((size_t)cx.S * (cx.F / VALS) * 4);
    cx.sm_vpw = take((size_t)kNW * 2 * kMaxR * 4);
    cx.sm_vx = take((size_t)2 * kMaxR * 4);
    cx.sm_vdw = take((size_t)kNW * ndl * kMaxR * 4);
    cx.sm_vd = take((size_t)ndl * kMaxR * 4);
    cx.sm_vdacc = take((size_t)kNW * ndl * kMaxR * 4);
    cx.sm_vnw = take((size_t)kNW * 2 * kMaxR * 4);
    cx.sm_comb = take((size_t)cx.max_orows * 4);
    // prep buffer (floats): scales | tsum | bgu | adn | bd | agu
    {
        uint32_t f = 0;
        cx.pp_scale = f;
        f += SC_COUNT;
        cx.pp_tsum = f;
        f += (uint32_t)cx.max_hrows;
        cx.pp_bgu = f;
        f += (uint32_t)(cx.gu_slot >= 0 ? cx.max_pairs * r2 : 0);
        cx.pp_adn = f;
        f += (uint32_t)(cx.dl_mask ? cx.max_pairs * cx.rd : 0);
        cx.pp_bd = f;
        f += (uint32_t)(cx.n_dl * cx.max_orows * cx.rd);
        cx.pp_agu = f;
        f += (uint32_t)(cx.gu_slot >= 0 ? cx.max_orows * r2 : 0);
        cx.prep_bytes = (uint32_t)al((size_t)f * 4, 16);
    }
    cx.sm_prep = take((size_t)2 * cx.prep_bytes);
    cx.sm_gf = take((size_t)(cx.H ? cx.H : 64) * 2);
    cx.sm_gsc = take((size_t)(cx.H ? cx.H / 32 : 2) * 4);
    cx.sm_ghat = take((size_t)(cx.H ? cx.H / 32 : 2) * 4);
    cx.sm_frec = take((size_t)std::max(cx.max_erows * (int)cx.rec_H, 16));
    cx.sm_rcur = take((size_t)cx.depth * cx.K * 4);
    cx.sm_rprev = take((size_t)cx.depth * cx.K * 4);
    cx.sm_rw = take((size_t)cx.depth * cx.K * 4);
    cx.sm_misc = take((size_t)M_COUNT * 4);
    // the stage: tagged words of one exchange (x; or h and the down-LoRA
    // owner partials), 8 bytes each
    cx.sm_stage = take((size_t)std::max((long long)cx.d, (long long)cx.S * cx.F +
                                                           (long long)cx.n_dl * cx.max_owners * kMaxR) *
                       8);
    cx.sm_graw = take((size_t)(cx.H ? cx.H : 32) * 8);
    cx.sm_poff = take((size_t)kNW * kMaxSlots * 4);
    cx.sm_ring = (uint32_t)al(off, 1024);
    long long room = (long long)smem_max - (long long)cx.sm_ring;
    room = room / 1024 * 1024;
    if (room < 3 * kMaxPiece)
        return fail(MOE_EUNSUPPORTED, "decode_step: shapes leave a %lld-byte ring (< 48 KiB)", room);
    cx.ring_bytes = (uint32_t)room;
    const size_t smem = (size_t)cx.sm_ring + cx.ring_bytes;
    // a batch of copies (at most half the in-flight bytes, or one piece) must
    // always fit the ring with room to spare
    cx.inflight = std::min(cx.inflight, cx.ring_bytes / 2);

    // a slot's down rows of one CTA are one piece
    if ((size_t)cx.max_orows * cx.rec_F > (size_t)kMaxPiece)
        return fail(MOE_EUNSUPPORTED, "decode_step: %d down rows of %u bytes exceed a %d-byte piece",
                    cx.max_orows, cx.rec_F, kMaxPiece);
    // every item must fit a piece
    if (2 * cx.rec_d > (uint32_t)kMaxPiece || cx.rec_dh > (uint32_t)kMaxPiece)
        return fail(MOE_EUNSUPPORTED, "decode_step: d=%d rows exceed a %d-byte piece", cx.d,
                    kMaxPiece);
    if (cx.S + 2 > kMaxGroups)
        return fail(MOE_EUNSUPPORTED, "decode_step: K=%d needs too many work groups", cx.K);

    return bits == 4 ? launch_bits<4>(p, smem, st) : launch_bits<2>(p, smem, st);
}

}  // namespace moe
