// chain.cu -- the decode step as a chain of per-layer kernels joined by
// programmatic dependent launch (moe_decode_step_chain).
//
// Per layer N (the same math as the per-call path and the persistent kernel:
// experts of "Arquitectura del Sistema" on kerneldigest.dev, prerouter head of
// "Arquitectura del cabezal Prerouter" on xyznot.com/es/paper/2609.18063):
//
//   A(N): x = out(N-1) / rms (x0 for N = 0); every CTA takes a byte-balanced
//         share of the layer's gate/up row pairs (all slots) and head rows
//         (fc1, l): h = silu(g) * u (+ gate/up LoRA on the shared expert),
//         gelu(fc1 f), l f.  CTA 0 also ranks head N-1's logits (the route
//         of layer N for the next token).
//   B(N): every CTA takes a share of the output rows: out = residual +
//         sum_k w_k y_k + y_shared (down GEMV of every slot + down LoRA), a
//         share of head N's fc2 logits, and its partial A x of the next
//         layer's gate/up LoRA over its rows.
//
// The routes of every layer are known when the step starts (they were
// predicted by the previous token's heads), so each kernel copies its
// weights into shared memory in its prologue -- before griddepcontrol.wait,
// while the previous kernel still runs -- and reads its activations after
// it.  Every global write follows the wait, so a kernel never races the one
// before it.  The only wait inside a kernel is on its own bulk copies
// (bounded: on expiry the status word records MOE_ETIMEOUT and the kernel
// returns).  No CTA waits on another.
#include <algorithm>
#include <cfloat>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "step_common.cuh"

namespace moe {
namespace chain {

using step::chunk_dot_fix;
using step::Fix;
using step::fix_place;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxR = 32;                 // LoRA rank bound
constexpr int kMaxK = 16;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;   // a wait's bound when the caller sets none
constexpr int kMaxHPass = 8;              // h of all slots: at most 8 * 512 float4 (16 Ki floats)

struct CLayer {
    const uint8_t *pool, *shared;
    const uint16_t *la_d, *lb_d;          // routed down LoRA (expert e: + e * stride)
    size_t la_ds, lb_ds;
    int r_d;
    float s_d;
    const uint16_t *sa[3], *sb[3];        // shared expert LoRA: gate, up, down
    int sr[3];
    float ss[3];
    const uint8_t *router, *fc1x, *fc2, *lx;
    const uint16_t *fc1_tab, *b1, *b2, *l_tab, *bl;
};

// One launch's parameters (one layer, one kernel).
struct CP {
    int d, F, E, K, H, S, N, n_cta, depth;
    int head;                 // layer N's head runs (A: fc1, l rows; B: fc2 rows)
    int route_late;           // layer N's route is made in this step (read it after the wait)
    int cur, prv;             // route sets of this step and the previous one
    size_t stride;
    uint32_t gu_off, down_off, rec_d, rec_F, rec_dh, rec_H;
    int gu_lora;              // the shared expert has a gate or up adapter
    CLayer L;
    const int32_t *smap;      // this layer's slot map [K] (route position -> pool blob), or null
    const uint16_t *nA[2];    // the next layer's shared gate / up A (for its LoRA partials)
    int nr[2];
    const float *x_in;        // out(N - 1), or x0
    int x_is_out;             // x_in is an out (normalise it) rather than x0
    float *out;               // out(N)
    int32_t *ridx;
    float *rw, *rmargin;
    float *h;                 // [S][F] of layer N
    float *g, *zl, *z;        // [H], [E], [E] of layer N
    const float *vp;          // [n_cta][2 kMaxR] partials of layer N's gate/up LoRA
    float *vp_next;           // [n_cta][2 kMaxR] the next layer's
    const float *topk_z;      // logits the router top-K ranks
    int topk_set, topk_tgt;   // where the route goes
    int32_t *err;
    uint64_t timeout_ns;      // bound of every mbarrier wait
    int debug_unset_wait;     // test hook: CTA 0 of this launch waits on bytes nobody sends
    unsigned long long *trace;   // debug: per launch 8 stamps of CTA 0 (start, waited, end, ...)
    int launch_id;
};

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ uint32_t saddr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;");
}

// Weight copies stream each byte once per step: L2 evict-first, so that they
// do not push the small exchanged vectors (x, h, g) out of L2.
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(saddr(dst)), "l"(src), "r"(bytes), "r"(saddr(bar)), "l"(pol) : "memory");
}

__device__ __forceinline__ void bar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void bar_expect(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)),
                 "r"(bytes) : "memory");
}

// Bounded wait for phase 0 of bar (this kernel's one use of it): false, with
// MOE_ETIMEOUT in *err, once timeout_ns have passed.
__device__ __forceinline__ bool bar_wait(uint64_t *bar, int32_t *err, uint64_t timeout_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; it++) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0; "
            "selp.u32 %0, 1, 0, p; }"
            : "=r"(ok) : "r"(saddr(bar)) : "memory");
        if (ok) return true;
        uint64_t now;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
        if (it == 0) t0 = now;
        else if (now - t0 > timeout_ns) {
            atomicExch(err, MOE_ETIMEOUT);
            return false;
        }
    }
}

// Debug stamp k of this launch (CTA 0, thread 0), when tracing.
__device__ __forceinline__ void stamp(const CP &p, int k) {
    if (p.trace && blockIdx.x == 0 && threadIdx.x == 0) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        p.trace[(size_t)p.launch_id * 8 + k] = t;
    }
}

// Debug: every CTA's end, after 256 launches x 8 stamps of CTA 0.
__device__ __forceinline__ void stamp_end(const CP &p) {
    if (p.trace && threadIdx.x == 0 && blockIdx.x < 256) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        p.trace[2048 + (size_t)p.launch_id * 256 + blockIdx.x] = t;
    }
}

__device__ __forceinline__ float block_sum(float v, float *red) {
    v = warp_sum(v, 32);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float a = 0.0f;
    if (lane < kWarps) a = red[lane];
    a = warp_sum(a, 32);
    return a;      // every thread
}

// Dot of a packed record (cols columns) with x staged padded per chunk
// (stage_vec) and xs (per 16-byte chunk sums of x), over this lane's chunks.
template <int BITS>
__device__ __forceinline__ float rec_dot(const uint8_t *rec, int cols, const float *x,
                                         const float *xs, int lane) {
    constexpr int VALS = 128 / BITS;
    const int nch = cols / VALS;
    const size_t cb = code_bytes(cols, BITS);
    float acc = 0.0f;
    for (int c = lane; c < nch; c += 32) {
        const uint4 q = *reinterpret_cast<const uint4 *>(rec + (size_t)kChunk * c);
        const float2 sb = sb_f(*reinterpret_cast<const uint32_t *>(rec + cb + 4 * ((c * VALS) / kGroup)));
        acc += fmaf(sb.x, chunk_dot<BITS>(q, x + c * (VALS + 1)), sb.y * xs[c]);
    }
    return acc;
}

// Stages n floats (global) into shared memory in chunks of `vals` values,
// chunk c at dst + c * (vals + 1): the lanes of a warp each take one chunk,
// and the one-float pad puts lane l's j-th value in bank (l + j) mod 32 (no
// conflicts).  The per-chunk sums come from the same pass: a chunk's vals / 4
// float4 loads sit in consecutive lanes, reduced with shuffles (in a fixed
// order).  Returns the sum of squares (every thread).  n: a multiple of 4 *
// blockDim.x is not needed, vals: 32 or 64.
__device__ __forceinline__ float stage_vec(const float *src, int n, int vals, float *dst,
                                           float *sums, float *red) {
    float ss = 0.0f;
    const int per = vals / 4;                                 // lanes per chunk (8 or 16)
    for (int base = 0; base < n / 4; base += blockDim.x) {    // whole warps per pass (shuffles)
        const int i = base + threadIdx.x;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (i < n / 4) v = reinterpret_cast<const float4 *>(src)[i];
        const int c = (4 * i) / vals, j = 4 * i - c * vals;
        if (i < n / 4) {
            float *d = dst + c * (vals + 1) + j;
            d[0] = v.x;
            d[1] = v.y;
            d[2] = v.z;
            d[3] = v.w;
        }
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        float a = (v.x + v.y) + (v.z + v.w);
        for (int o = 1; o < per; o <<= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (i < n / 4 && (i & (per - 1)) == 0) sums[c] = a;
    }
    return block_sum(ss, red);
}

__host__ __device__ inline size_t padded(int n, int vals) { return (size_t)(n / vals) * (vals + 1); }

// Issues this thread's float4 loads of an n-float vector (at most MAXP passes
// of the block) so that several vectors' loads are in flight together.
template <int MAXP>
__device__ __forceinline__ void load_vec(const float *src, int n, float4 (&v)[MAXP]) {
#pragma unroll
    for (int k = 0; k < MAXP; k++) {
        const int i = k * blockDim.x + threadIdx.x;
        v[k] = i < n / 4 ? reinterpret_cast<const float4 *>(src)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Stages a vector as 16-bit fixed point per chunk of 128 / BITS values for
// the dp4a dot, straight from registers: thread i holds positions 4i .. 4i+3
// (v), the 128 / BITS / 4 consecutive lanes of a chunk find its max |x| and
// its sum with shuffles, and each lane writes its four fixed-point values --
// xf bytes in the layout chunk_dot_fix reads, the chunk scale 2^(e-15) and
// xhat = sum of the fixed-point values times the scale (scale, rounding and
// layout as the persistent decode kernel's stage_chunk).  Every
// lane of the warp calls it (in: whether position 4i exists).
template <int BITS>
__device__ __forceinline__ void quant4(const float4 &v, int i, bool in, uint8_t *xf, int nch,
                                       float *xsc, float *xhat) {
    constexpr int VALS = 128 / BITS, PER = VALS / 4;
    uint32_t mb = max(max(__float_as_uint(fabsf(v.x)), __float_as_uint(fabsf(v.y))),
                      max(__float_as_uint(fabsf(v.z)), __float_as_uint(fabsf(v.w))));
#pragma unroll
    for (int o = 1; o < PER; o <<= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const bool nz = (mb >> 23) != 0;
    const int e = nz ? (int)((mb >> 23) & 0xff) - 126 : 0;
    const float f = nz ? __uint_as_float((uint32_t)(127 + 15 - e) << 23) : 0.0f;
    int q[4];
    const float vv[4] = {v.x, v.y, v.z, v.w};
    int sum = 0;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        q[k] = max(-32767, min(32767, (int)rintf(vv[k] * f)));
        sum += q[k];
    }
#pragma unroll
    for (int o = 1; o < PER; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (!in) return;
    const int c = (4 * i) / VALS, pos = 4 * i - c * VALS;
    if (BITS == 4) {
        // positions 8j + 4b + {0..3}: (q0, q2) are high/low bytes 2b, 2b+1 of
        // the A words, (q1, q3) of the B words
        const int j = pos >> 3, b = (pos >> 2) & 1;
        uint8_t *w = xf + ((size_t)j * nch + c) * 16 + 2 * b;
        const auto hi = [](int x) { return (uint32_t)((x >> 8) & 0xff); };
        const auto lo = [](int x) { return (uint32_t)(x & 0xff); };
        *reinterpret_cast<uint16_t *>(w) = (uint16_t)(hi(q[0]) | hi(q[2]) << 8);
        *reinterpret_cast<uint16_t *>(w + 4) = (uint16_t)(lo(q[0]) | lo(q[2]) << 8);
        *reinterpret_cast<uint16_t *>(w + 8) = (uint16_t)(hi(q[1]) | hi(q[3]) << 8);
        *reinterpret_cast<uint16_t *>(w + 12) = (uint16_t)(lo(q[1]) | lo(q[3]) << 8);
    } else {
#pragma unroll
        for (int k = 0; k < 4; k++) {
            int slot, byte;
            fix_place<BITS>(pos + k, slot, byte);
            uint8_t *w = xf + ((size_t)slot * nch + c) * 16;
            w[byte] = (uint8_t)((q[k] >> 8) & 0xff);
            w[byte + 4] = (uint8_t)(q[k] & 0xff);
        }
    }
    if ((i & (PER - 1)) == 0) {
        const float sc = nz ? __uint_as_float((uint32_t)(127 + e - 15) << 23) : 0.0f;
        xsc[c] = sc;
        xhat[c] = (float)sum * sc;
    }
}

__host__ __device__ inline size_t fix_bytes(int n, int bits) {
    return (size_t)(n / (128 / bits)) * (bits == 4 ? 4 : 8) * 16;
}

// Dots of R consecutive records (rec0, rec0 + stride, ...; cols columns) with
// a vector staged by quant4, over this lane's chunks (exact integer chunk
// dots, then fma(scale, dot * 2^(e-15), bias * xhat)).
template <int BITS, int R>
__device__ __forceinline__ void fix_dot(const uint8_t *rec0, uint32_t stride, int cols,
                                        const uint8_t *xf, const float *xsc, const float *xhat,
                                        int lane, float (&out)[R]) {
    constexpr int VALS = 128 / BITS;
    const int nch = cols / VALS;
    const size_t cb = code_bytes(cols, BITS);
    const uint4 *xq = reinterpret_cast<const uint4 *>(xf);
#pragma unroll
    for (int r = 0; r < R; r++) out[r] = 0.0f;
    for (int c = lane; c < nch; c += 32) {
        uint4 q[R];
        uint32_t sbw[R];
#pragma unroll
        for (int r = 0; r < R; r++) {
            q[r] = *reinterpret_cast<const uint4 *>(rec0 + (size_t)r * stride + (size_t)kChunk * c);
            sbw[r] = *reinterpret_cast<const uint32_t *>(rec0 + (size_t)r * stride + cb + 4 * ((c * VALS) / kGroup));
        }
        int dq[R];
        chunk_dot_fix<BITS, R>(q, xq, nch, c, dq);
        const float sc = xsc[c], X = xhat[c];
#pragma unroll
        for (int r = 0; r < R; r++) {
            const float2 sb = sb_f(sbw[r]);
            out[r] += fmaf(sb.x, (float)dq[r] * sc, sb.y * X);
        }
    }
}

__device__ __forceinline__ float half_at(const uint16_t *p, size_t i) { return half_f(p[i]); }

// Ranks E <= 1024 logits (value desc, index asc; NaN last) in one warp:
// route of layer tgt in set `set` (indices, softmax weights over the kept K,
// margin z_(K) - z_(K+1)).  Lane l holds logits l, l + 32, ..., NV of them
// (NV * 32 >= E); each lane keeps its best remaining one (a pairwise tree
// over its values), every round takes the warp's best of those (ties: lower
// index) and only the winning lane rescans.  The k-th winner ends in lane k
// (registers only).
template <int NV>
struct Logits {
    float v[NV];
};

template <int NV>
__device__ __forceinline__ void load_logits(const float *z, int E, Logits<NV> &L) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        const float x = e < E ? z[e] : -INFINITY;
        L.v[i] = x == x ? x : -INFINITY;
    }
}

// (value, index) a ranks before b
__device__ __forceinline__ bool ranks_before(float av, int ai, float bv, int bi) {
    return av > bv || (av == bv && ai < bi);
}

template <int NV>
__device__ void warp_route(const Logits<NV> &L, int E, int K, int32_t *ridx, float *rw,
                           float *rmargin, int set, int depth, int tgt) {
    const int lane = threadIdx.x & 31;
    uint32_t taken = 0;
    // this lane's best remaining entry: taken and absent entries become
    // (-inf, INT_MAX), after every real one
    auto best_of_lane = [&](float &bv, int &bi) {
        float tv[NV];
        int ti[NV];
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int e = lane + 32 * i;
            const bool ok = e < E && !(taken >> i & 1u);
            tv[i] = ok ? L.v[i] : -INFINITY;
            ti[i] = ok ? e : 0x7fffffff;
        }
#pragma unroll
        for (int w = 1; w < NV; w <<= 1)
#pragma unroll
            for (int i = 0; i + w < NV; i += 2 * w)
                if (ranks_before(tv[i + w], ti[i + w], tv[i], ti[i])) {
                    tv[i] = tv[i + w];
                    ti[i] = ti[i + w];
                }
        bv = tv[0];
        bi = ti[0];
    };
    float lv, mv = -INFINITY;       // this lane's best remaining; my winner's value (lane k)
    int li, mi = 0;
    best_of_lane(lv, li);
    const int rounds = K < E ? K + 1 : K;
    for (int k = 0; k < rounds; k++) {
        float bv = lv;
        int bi = li;
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ranks_before(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == k) {
            mv = bv;
            mi = bi;
        }
        if (bi < E && (bi & 31) == lane) {      // the winner's lane takes it and rescans
            taken |= 1u << (bi >> 5);
            best_of_lane(lv, li);
        }
    }
    // softmax over the kept K (lane k < K), margin from lanes K - 1 and K
    const float top = __shfl_sync(0xffffffffu, mv, 0);
    const float ex = lane < K ? expf(mv - top) : 0.0f;
    const float sum = warp_sum(ex, 32);
    const float vk1 = __shfl_sync(0xffffffffu, mv, K - 1);
    const float vk = __shfl_sync(0xffffffffu, mv, K < 32 ? K : 0);
    if (lane < K) {
        ridx[((size_t)set * depth + tgt) * K + lane] = mi;
        rw[((size_t)set * depth + tgt) * K + lane] = ex / sum;
    }
    if (lane == 0) rmargin[(size_t)set * depth + tgt] = K < E ? vk1 - vk : INFINITY;
}

// The route of layer tgt from the E logits at z, by one warp.
__device__ __forceinline__ void route_one(const CP &p, const float *z, int set, int tgt) {
    if (p.E <= 256) {
        Logits<8> zv;
        load_logits(z, p.E, zv);
        warp_route(zv, p.E, p.K, p.ridx, p.rw, p.rmargin, set, p.depth, tgt);
    } else if (p.E <= 512) {
        Logits<16> zv;
        load_logits(z, p.E, zv);
        warp_route(zv, p.E, p.K, p.ridx, p.rw, p.rmargin, set, p.depth, tgt);
    } else {
        Logits<32> zv;
        load_logits(z, p.E, zv);
        warp_route(zv, p.E, p.K, p.ridx, p.rw, p.rmargin, set, p.depth, tgt);
    }
}

// ---------------------------------------------------------------- A work split
// CTA c takes an even share of the gate/up row pairs of every slot
// (slot-major, P bytes each) and an even share of the head rows (fc1 rows,
// then l rows, R bytes each; none when the head does not run): the same mix
// of work on every CTA.  Its units, in order: its pairs, then its head rows.
struct ASplit {
    long long gu_units, P, R;
    int head_rows;
    __host__ __device__ void range(int c, int n, long long &g0, long long &g1, int &r0, int &r1) const {
        g0 = gu_units * c / n;
        g1 = gu_units * (c + 1) / n;
        r0 = (int)((long long)head_rows * c / n);
        r1 = (int)((long long)head_rows * (c + 1) / n);
    }
};

__host__ __device__ inline ASplit a_split(int S, int F, int H, int E, int head, uint32_t rec_d,
                                          uint32_t rec_dh) {
    ASplit s;
    s.gu_units = (long long)S * F;
    s.P = 2LL * rec_d;
    s.R = rec_dh;
    s.head_rows = head ? H + E : 0;
    return s;
}

// The blob of route position s: the shared expert, the routed expert the
// route names, or -- with a slot map -- the pool blob the map names for it.
__device__ __forceinline__ const uint8_t *slot_blob(const CP &p, const int32_t *route, int s,
                                                    bool &bad) {
    if (s >= p.K) return p.L.shared;
    const int e = route[s];
    const int b = p.smap ? p.smap[s] : e;
    if ((unsigned)e >= (unsigned)p.E || b < 0) {
        bad = true;
        return p.L.pool;
    }
    return p.L.pool + (size_t)b * p.stride;
}

// ---------------------------------------------------------------- kernel A
template <int BITS>
__global__ void __launch_bounds__(kThreads, 2) chain_a_kernel(const __grid_constant__ CP p) {
    constexpr int VALS = 128 / BITS;
    extern __shared__ __align__(128) uint8_t sm[];
    const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ASplit sp = a_split(p.S, p.F, p.H, p.E, p.head, p.rec_d, p.rec_dh);
    long long g0, g1;
    int r0, r1;
    sp.range(c, p.n_cta, g0, g1, r0, r1);
    const int ng = (int)(g1 - g0), nh = r1 - r0;
    const uint32_t gbytes = (uint32_t)(ng * sp.P);
    const uint32_t wbytes = gbytes + (uint32_t)(nh * sp.R);
    // shared memory: weights, x as fixed point (and in 4-bit chunks for the
    // head), table sums of the head rows, LoRA v, misc
    uint8_t *wts = sm;
    size_t off = (wbytes + 127) / 128 * 128;
    uint8_t *xf = sm + off;                                   // x as fixed point (BITS chunks)
    off += fix_bytes(p.d, BITS);
    float *xsc = reinterpret_cast<float *>(sm + off);
    off += (size_t)(p.d / VALS) * 4;
    float *xhat = reinterpret_cast<float *>(sm + off);
    off += (size_t)(p.d / VALS) * 4;
    uint8_t *xf4 = BITS == 4 ? xf : sm + off;                 // ... and in 4-bit chunks (head)
    if (BITS != 4) off += fix_bytes(p.d, 4);
    float *xsc4 = BITS == 4 ? xsc : reinterpret_cast<float *>(sm + off);
    if (BITS != 4) off += (size_t)(p.d / 32) * 4;
    float *xhat4 = BITS == 4 ? xhat : reinterpret_cast<float *>(sm + off);
    if (BITS != 4) off += (size_t)(p.d / 32) * 4;
    float *tsum = reinterpret_cast<float *>(sm + off);
    off += (size_t)(nh + 1) * 4;
    float *tterm = reinterpret_cast<float *>(sm + off);       // [nh][2K + 1] table terms
    off += (size_t)(nh * (2 * p.K + 1) + 1) * 4;
    float *vx = reinterpret_cast<float *>(sm + off);          // gate/up LoRA A x
    off += 2 * kMaxR * 4;
    float *vwarp = reinterpret_cast<float *>(sm + off);       // per-warp sums of the partials
    off += kWarps * 32 * 4;
    // the shared expert's gate / up B rows of this CTA's units of that slot
    const int gs = p.S - 1;
    const long long f_lo = max(g0, (long long)gs * p.F), f_hi = min(g1, (long long)(gs + 1) * p.F);
    const int nlf = p.gu_lora && f_hi > f_lo ? (int)(f_hi - f_lo) : 0;
    float *bgu = reinterpret_cast<float *>(sm + off);         // [nlf][2 kMaxR]
    off += (size_t)(nlf * 2 * kMaxR + 1) * 4;
    float *red = reinterpret_cast<float *>(sm + off);
    off += 32 * 4;
    int32_t *route = reinterpret_cast<int32_t *>(sm + off);
    off += (kMaxK + 1) * 4;
    off = (off + 7) / 8 * 8;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + off);

    stamp(p, 0);
    const int32_t *rcur = p.ridx + ((size_t)p.cur * p.depth + p.N) * p.K;
    const int32_t *rprv = p.ridx + ((size_t)p.prv * p.depth + p.N) * p.K;
    auto issue = [&]() {
        // segments: per slot a run of pairs, then fc1 rows, then l rows
        if (threadIdx.x == 0) {
            bool bad = false;
            bar_expect(bar, wbytes);
            uint32_t at = 0;
            for (long long u = g0; u < g1;) {
                const int s = (int)(u / p.F), f = (int)(u % p.F);
                const long long n = min((long long)(p.F - f), g1 - u);
                bulk_copy(wts + at, slot_blob(p, route, s, bad) + p.gu_off + (size_t)f * sp.P,
                          (uint32_t)(n * sp.P), bar);
                at += (uint32_t)(n * sp.P);
                u += n;
            }
            const int f1 = min(r1, p.H);
            if (f1 > r0) {
                bulk_copy(wts + at, p.L.fc1x + (size_t)r0 * sp.R, (uint32_t)((f1 - r0) * sp.R), bar);
                at += (uint32_t)((f1 - r0) * sp.R);
            }
            const int l0 = max(r0, p.H);
            if (r1 > l0) bulk_copy(wts + at, p.L.lx + (size_t)(l0 - p.H) * sp.R, (uint32_t)((r1 - l0) * sp.R), bar);
            if (bad) atomicExch(p.err, MOE_EINVAL);
        }
    };
    if (threadIdx.x == 0) bar_init(bar);
    if (threadIdx.x < p.K && !p.route_late) route[threadIdx.x] = rcur[threadIdx.x];
    __syncthreads();
    if (!p.route_late) issue();
    stamp(p, 5);
    // table sums of this CTA's head rows (the routes of layer N at t and t - 1)
    auto tables = [&]() {
        // item (row i, term j): j < K the current route's table row, then the
        // previous route's, then the bias -- one load each, in parallel; row
        // i's terms are then summed in that order
        const int nt = 2 * p.K + 1;
        for (int it = threadIdx.x; it < nh * nt; it += blockDim.x) {
            const int i = it / nt, j = it - i * nt;
            const int r = r0 + i;
            const bool fc1 = r < p.H;
            const int row = fc1 ? (int)r : (int)(r - p.H);
            const int width = fc1 ? p.H : p.E;
            const uint16_t *tab = fc1 ? p.L.fc1_tab : p.L.l_tab;
            const uint16_t *bias = fc1 ? p.L.b1 : p.L.bl;
            float a = 0.0f;
            if (j == 2 * p.K) a = bias ? half_at(bias, row) : 0.0f;
            else if (tab) {
                const int e = j < p.K ? route[j] : rprv[j - p.K];
                if ((unsigned)e < (unsigned)p.E)
                    a = half_at(tab, (size_t)(j < p.K ? e : p.E + e) * width + row);
            }
            tterm[it] = a;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nh; i += blockDim.x) {
            float a = 0.0f;
            for (int j = 0; j < nt; j++) a += tterm[i * nt + j];
            tsum[i] = a;
        }
    };
    if (!p.route_late) tables();
    // B rows of the shared gate / up adapters for this CTA's rows of that slot
    // (entries 0..31 of a row: lane k reads entry k)
    for (int it = threadIdx.x; it < nlf * 32; it += blockDim.x) {
        const int i = it >> 5, k = it & 31;
        const int f = (int)(f_lo - (long long)gs * p.F) + i, rg = p.L.sr[0], ru = p.L.sr[1];
        float v = 0.0f;
        if (k < rg) v = half_at(p.L.sb[0], (size_t)f * rg + k);
        else if (k < rg + ru) v = half_at(p.L.sb[1], (size_t)f * ru + (k - rg));
        bgu[(size_t)i * 2 * kMaxR + k] = v;
    }
    stamp(p, 7);
    grid_launch_dependents();
    grid_wait();
    stamp(p, 1);
    // the partials of the shared gate/up LoRA's A x: loads first (they
    // overlap the staging of x)
    const bool lora_here = nlf > 0;
    constexpr int kPer = 16;                    // up to 256 CTAs
    float vpl[kPer];
    if (lora_here) {
#pragma unroll
        for (int j = 0; j < kPer; j++) {
            const int q = warp + j * kWarps;
            vpl[j] = q < p.n_cta ? p.vp[(size_t)q * 2 * kMaxR + lane] : 0.0f;
        }
    }
    if (p.route_late) {
        if (threadIdx.x < p.K) route[threadIdx.x] = rcur[threadIdx.x];
        __syncthreads();
        issue();
        tables();
    }
    // x as fixed point straight from the loads; per-warp sums of x^2 (1/rms
    // when x is an out, summed over the warps in order after the barrier)
    float ss = 0.0f;
    for (int base = 0; base < p.d / 4; base += blockDim.x) {     // uniform over the block
        const int i = base + threadIdx.x;
        const bool in = i < p.d / 4;
        const float4 v = in ? reinterpret_cast<const float4 *>(p.x_in)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        quant4<BITS>(v, i, in, xf, p.d / VALS, xsc, xhat);
        if (BITS != 4) quant4<4>(v, i, in, xf4, p.d / 32, xsc4, xhat4);
    }
    ss = warp_sum(ss, 32);
    if (lane == 0) red[warp] = ss;
    stamp(p, 3);
    // the shared expert's gate/up LoRA: A x from the previous layer's
    // partials (warp w summed CTAs w, w + kWarps, ... in order; warp 0 sums
    // the warps')
    if (lora_here) {
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < kPer; j++) a += vpl[j];
        vwarp[warp * 32 + lane] = a;
    }
    __syncthreads();
    float inv = 1.0f;
    if (p.x_is_out) {
        float t = 0.0f;
        for (int w = 0; w < kWarps; w++) t += red[w];
        inv = 1.0f / sqrtf(t / p.d + 1e-6f);
    }
    if (lora_here && warp == 0) {
        float a = 0.0f;
        for (int w = 0; w < kWarps; w++) a += vwarp[w * 32 + lane];
        vx[lane] = a * inv;
    }
    __syncthreads();
    if (!bar_wait(bar, p.err, p.timeout_ns)) return;
    if (p.debug_unset_wait && c == 0) {
        // test hook: a wait for 16 bytes no copy delivers, on a barrier of its
        // own once this CTA's copies have landed: it runs out after
        // timeout_ns, records MOE_ETIMEOUT and the CTA returns
        if (threadIdx.x == 0) {
            bar_init(bar + 1);
            bar_expect(bar + 1, 16);
        }
        __syncthreads();
        if (!bar_wait(bar + 1, p.err, p.timeout_ns)) return;
    }
    // units v = w, w + kWarps, ... of the CTA's list (its pairs, then its head rows)
    stamp(p, 4);
    for (int v = warp; v < ng + nh; v += kWarps) {
        const uint8_t *rec = wts + (v < ng ? (size_t)v * sp.P : gbytes + (size_t)(v - ng) * sp.R);
        const long long u = v < ng ? g0 + v : sp.gu_units + r0 + (v - ng);
        if (v < ng) {
            const int s = (int)u / p.F, f = (int)u - s * p.F;
            float gu[2];
            fix_dot<BITS, 2>(rec, p.rec_d, p.d, xf, xsc, xhat, lane, gu);
            float a0 = gu[0] * inv, a1 = gu[1] * inv;
            if (s == gs && p.gu_lora) {
                // lane k < rg: gate term k; rg <= k < rg + ru: up term k - rg
                // (added to the lanes' partials: one sum per projection)
                const int rg = p.L.sr[0];
                const float t = bgu[(size_t)(u - f_lo) * 2 * kMaxR + lane] * vx[lane];
                a0 = fmaf(p.L.ss[0], lane < rg ? t : 0.0f, a0);
                a1 = fmaf(p.L.ss[1], lane < rg ? 0.0f : t, a1);
            }
            const float gg = warp_sum(a0, 32), uu = warp_sum(a1, 32);
            if (lane == 0) p.h[(size_t)s * p.F + f] = silu_f(gg) * uu;
        } else {
            const long long r = u - sp.gu_units;
            float hd[1];
            fix_dot<4, 1>(rec, 0, p.d, xf4, xsc4, xhat4, lane, hd);
            const float a = warp_sum(hd[0], 32) * inv + tsum[v - ng];
            if (lane == 0) {
                if (r < p.H) p.g[r] = gelu_erf_f(a);
                else if (p.H > 0) p.zl[r - p.H] = a;
                else p.z[r - p.H] = a;
            }
        }
    }
    stamp(p, 6);
    if (p.trace) __syncthreads();          // debug: the stamp marks the whole CTA's end
    stamp(p, 2);
    stamp_end(p);
}

// ---------------------------------------------------------------- kernel B
// Output rows [o0, o1) and logit rows [e0, e1) of CTA c (even splits).
template <int BITS>
__global__ void __launch_bounds__(kThreads, 2) chain_b_kernel(const __grid_constant__ CP p) {
    constexpr int VALS = 128 / BITS;
    extern __shared__ __align__(128) uint8_t sm[];
    const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int o0 = (int)((long long)p.d * c / p.n_cta), o1 = (int)((long long)p.d * (c + 1) / p.n_cta);
    const int no = o1 - o0;
    const int e0 = p.head ? (int)((long long)p.E * c / p.n_cta) : 0;
    const int e1 = p.head ? (int)((long long)p.E * (c + 1) / p.n_cta) : 0;
    const int ne = e1 - e0;
    const uint32_t dbytes = (uint32_t)no * p.rec_F;           // per slot
    const uint32_t fbytes = p.H ? (uint32_t)ne * p.rec_H : 0u;
    uint8_t *wts = sm;                                        // [S][no] down records, then fc2 rows
    size_t off = ((size_t)p.S * dbytes + fbytes + 127) / 128 * 128;
    float *hs = reinterpret_cast<float *>(sm + off);          // [S][F] padded per chunk (LoRA)
    off += padded(p.S * p.F, VALS) * 4;
    uint8_t *hf = sm + off;                                   // h as fixed point per chunk
    off += fix_bytes(p.S * p.F, BITS);
    float *hsc = reinterpret_cast<float *>(sm + off);
    off += (size_t)(p.S * p.F / VALS) * 4;
    float *hhat = reinterpret_cast<float *>(sm + off);
    off += (size_t)(p.S * p.F / VALS) * 4;
    uint8_t *gf = sm + off;                                   // g as fixed point (4-bit chunks)
    off += p.H > 0 ? fix_bytes(p.H, 4) : 16;
    float *gsc = reinterpret_cast<float *>(sm + off);
    off += (size_t)(p.H > 0 ? p.H / 32 : 1) * 4;
    float *ghat = reinterpret_cast<float *>(sm + off);
    off += (size_t)(p.H > 0 ? p.H / 32 : 1) * 4;
    float *vd = reinterpret_cast<float *>(sm + off);          // [S][kMaxR] down LoRA A_d h
    off += (size_t)p.S * kMaxR * 4;
    // the down adapters' A (fp16 [r][F] per adapter slot), copied with the weights
    uint16_t *adn = reinterpret_cast<uint16_t *>(sm + off);
    const int nrd = p.L.r_d ? p.K : 0;                        // routed slots with an adapter
    const uint32_t abytes = (uint32_t)(nrd * p.L.r_d + (p.S > p.K ? p.L.sr[2] : 0)) * p.F * 2;
    off += (abytes + 15) / 16 * 16;
    // the next layer's gate/up A columns of this CTA's rows: [2 kMaxR][no]
    float *anext = reinterpret_cast<float *>(sm + off);
    off += (size_t)2 * kMaxR * (no + 1) * 4;
    float *outs = reinterpret_cast<float *>(sm + off);        // [no] this CTA's out rows
    off += (size_t)(no + 1) * 4;
    float *resid = reinterpret_cast<float *>(sm + off);       // [no] residual rows
    off += (size_t)(no + 1) * 4;
    float *zls = reinterpret_cast<float *>(sm + off);         // [ne] l f rows
    off += (size_t)(ne + 1) * 4;
    float *b2s = reinterpret_cast<float *>(sm + off);         // [ne] fc2 bias rows
    off += (size_t)(ne + 1) * 4;
    float *bdn = reinterpret_cast<float *>(sm + off);         // [S][no][kMaxR] down B rows
    off += (size_t)p.S * (no + 1) * kMaxR * 4;
    float *wk = reinterpret_cast<float *>(sm + off);          // combine weights
    off += (kMaxK + 1) * 4;
    int32_t *route = reinterpret_cast<int32_t *>(sm + off);
    off += (kMaxK + 1) * 4;
    off = (off + 7) / 8 * 8;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + off);

    stamp(p, 0);
    const int32_t *rcur = p.ridx + ((size_t)p.cur * p.depth + p.N) * p.K;
    const float *wcur = p.rw + ((size_t)p.cur * p.depth + p.N) * p.K;
    auto issue = [&]() {
        if (threadIdx.x == 0) {
            bool bad = false;
            bar_expect(bar, (uint32_t)p.S * dbytes + fbytes + abytes);
            for (int s = 0; s < p.S; s++)
                if (dbytes)
                    bulk_copy(wts + (size_t)s * dbytes,
                              slot_blob(p, route, s, bad) + p.down_off + (size_t)o0 * p.rec_F, dbytes, bar);
            if (fbytes) bulk_copy(wts + (size_t)p.S * dbytes, p.L.fc2 + (size_t)e0 * p.rec_H, fbytes, bar);
            uint32_t at = 0;
            for (int s = 0; s < nrd; s++) {                   // routed adapters (valid routes only)
                const uint32_t nb = (uint32_t)p.L.r_d * p.F * 2;
                const int e = route[s];
                bulk_copy(reinterpret_cast<uint8_t *>(adn) + at,
                          p.L.la_d + (size_t)((unsigned)e < (unsigned)p.E ? e : 0) * p.L.la_ds, nb, bar);
                at += nb;
            }
            if (p.S > p.K && p.L.sr[2])
                bulk_copy(reinterpret_cast<uint8_t *>(adn) + at, p.L.sa[2], (uint32_t)p.L.sr[2] * p.F * 2, bar);
            if (bad) atomicExch(p.err, MOE_EINVAL);
        }
    };
    if (threadIdx.x == 0) bar_init(bar);
    if (threadIdx.x < p.K && !p.route_late) {
        route[threadIdx.x] = rcur[threadIdx.x];
        wk[threadIdx.x] = wcur[threadIdx.x];
    }
    __syncthreads();
    if (!p.route_late) issue();
    // fc2 biases, down B rows of this CTA's outputs (the routed adapters' need
    // the route: with it, or after the wait)
    // (only the slots with an adapter, k < r: the only entries read)
    auto load_b = [&]() {
        for (int s = 0; s < p.S; s++) {
            const bool shared = s >= p.K;
            const int r = shared ? p.L.sr[2] : p.L.r_d;
            if (r == 0) continue;
            const int e = shared ? 0 : route[s];
            const bool ok = shared || (unsigned)e < (unsigned)p.E;
            const uint16_t *B = shared ? p.L.sb[2] : p.L.lb_d + (size_t)(ok ? e : 0) * p.L.lb_ds;
            for (int it = threadIdx.x; it < no * r; it += blockDim.x) {
                const int i = it / r, k = it - i * r;
                bdn[((size_t)s * no + i) * kMaxR + k] = ok ? half_at(B, (size_t)(o0 + i) * r + k) : 0.0f;
            }
        }
    };
    for (int i = threadIdx.x; i < ne; i += blockDim.x) b2s[i] = p.L.b2 ? half_at(p.L.b2, e0 + i) : 0.0f;
    if (!p.route_late) load_b();
    // the next layer's gate/up A columns of this CTA's rows (static data)
    const int r2n = p.vp_next ? p.nr[0] + p.nr[1] : 0;
    for (int it = threadIdx.x; it < r2n * no; it += blockDim.x) {
        const int k = it / no, i = it - k * no;
        const uint16_t *A = k < p.nr[0] ? p.nA[0] + (size_t)k * p.d : p.nA[1] + (size_t)(k - p.nr[0]) * p.d;
        anext[k * no + i] = half_at(A, o0 + i);
    }
    grid_launch_dependents();
    grid_wait();
    stamp(p, 1);
    if (p.route_late) {
        if (threadIdx.x < p.K) {
            route[threadIdx.x] = rcur[threadIdx.x];
            wk[threadIdx.x] = wcur[threadIdx.x];
        }
        __syncthreads();
        issue();
        load_b();
    }
    // h of every slot, g (head fc2 input), this CTA's residual rows and l f
    // rows: every load issued before any is used
    float4 hv[kMaxHPass], gv[1];
    load_vec<kMaxHPass>(p.h, p.S * p.F, hv);
    const bool gh = p.head && p.H > 0;
    if (gh) load_vec<1>(p.g, p.H, gv);
    float resv = 0.0f, zlv = 0.0f;
    if (threadIdx.x < no) resv = p.x_in[o0 + threadIdx.x];
    if (threadIdx.x >= 32 && threadIdx.x < 32 + ne) zlv = p.zl[e0 + threadIdx.x - 32];
    // fixed point straight from the loads (h also padded as floats, for the
    // down LoRA)
    const int nh4 = p.S * p.F / 4;
#pragma unroll
    for (int k = 0; k < kMaxHPass; k++) {
        if (k * (int)blockDim.x >= nh4) break;                   // whole block: uniform
        const int i = k * blockDim.x + threadIdx.x;
        const bool in = i < nh4;
        if (in) {
            const int ch = (4 * i) / VALS;
            float *d = hs + ch * (VALS + 1) + (4 * i - ch * VALS);
            d[0] = hv[k].x;
            d[1] = hv[k].y;
            d[2] = hv[k].z;
            d[3] = hv[k].w;
        }
        quant4<BITS>(hv[k], i, in, hf, p.S * p.F / VALS, hsc, hhat);
    }
    stamp(p, 7);
    if (gh) quant4<4>(gv[0], threadIdx.x, (int)threadIdx.x < p.H / 4, gf, p.H / 32, gsc, ghat);
    if (threadIdx.x < no) resid[threadIdx.x] = resv;
    if (threadIdx.x >= 32 && threadIdx.x < 32 + ne) zls[threadIdx.x - 32] = zlv;
    __syncthreads();
    stamp(p, 3);
    if (!bar_wait(bar, p.err, p.timeout_ns)) return;
    stamp(p, 4);
    // down LoRA: vd[s][k] = A_d[k] h_s (routed adapter slots, then the shared
    // one), one (slot, k) row per warp, A from shared memory
    {
        const int rs = p.S > p.K ? p.L.sr[2] : 0;
        const int nrow = nrd * p.L.r_d + rs;
        for (int it = warp; it < nrow; it += kWarps) {
            const bool shared = it >= nrd * p.L.r_d;
            const int s = shared ? p.S - 1 : it / p.L.r_d;
            const int k = shared ? it - nrd * p.L.r_d : it - s * p.L.r_d;
            const uint16_t *A = adn + (size_t)it * p.F;
            float a = 0.0f;
            const float *hrow = hs + (size_t)s * (p.F / VALS) * (VALS + 1);
#pragma unroll 4
            for (int f = lane; f < p.F; f += 32) a = fmaf(half_f(A[f]), hrow[f + f / VALS], a);
            a = warp_sum(a, 32);
            if (lane == 0) vd[s * kMaxR + k] = (!shared && (unsigned)route[s] >= (unsigned)p.E) ? 0.0f : a;
        }
    }
    __syncthreads();
    stamp(p, 5);
    // out rows: warp per row; lanes over the (slot, chunk) pairs
    const int cps = p.F / VALS, npair = p.S * cps;
    const size_t cb = code_bytes(p.F, BITS);
    for (int i = warp; i < no; i += kWarps) {
        const int o = o0 + i;
        float acc = 0.0f;
        for (int q = lane; q < npair; q += 32) {
            const int s = q / cps, ch = q - s * cps;
            const uint8_t *rec = wts + (size_t)s * dbytes + (size_t)i * p.rec_F;
            const uint4 w4[1] = {*reinterpret_cast<const uint4 *>(rec + (size_t)kChunk * ch)};
            const float2 sb = sb_f(*reinterpret_cast<const uint32_t *>(rec + cb + 4 * ((ch * VALS) / kGroup)));
            int dq[1];
            const int hc = s * cps + ch;
            chunk_dot_fix<BITS, 1>(w4, reinterpret_cast<const uint4 *>(hf), npair, hc, dq);
            const float y = fmaf(sb.x, (float)dq[0] * hsc[hc], sb.y * hhat[hc]);
            acc = fmaf(s < p.K ? wk[s] : 1.0f, y, acc);
        }
        // down LoRA: lane k < r of each adapter slot (B rows from shared memory)
        for (int s = 0; s < p.S; s++) {
            const bool shared = s >= p.K;
            const int r = shared ? p.L.sr[2] : p.L.r_d;
            if (r == 0 || lane >= r) continue;
            const float sc = shared ? p.L.ss[2] : p.L.s_d;
            acc = fmaf((shared ? 1.0f : wk[s]) * sc,
                       bdn[((size_t)s * no + i) * kMaxR + lane] * vd[s * kMaxR + lane], acc);
        }
        acc = warp_sum(acc, 32);
        if (lane == 0) {
            const float v = resid[i] + acc;
            outs[i] = v;
            p.out[o] = v;
        }
    }
    stamp(p, 6);
    // head N's fc2 rows: z = fc2 g + b2 + l f (row i on warp (no + i) mod
    // 16: the warps without an out row first)
    for (int i = (warp - no % kWarps + kWarps) % kWarps; i < ne; i += kWarps) {
        const int e = e0 + i;
        float a = 0.0f;
        if (p.H > 0) {
            float f2[1];
            fix_dot<4, 1>(wts + (size_t)p.S * dbytes + (size_t)i * p.rec_H, 0, p.H, gf, gsc, ghat, lane, f2);
            a = warp_sum(f2[0], 32);
        }
        if (lane == 0) p.z[e] = a + b2s[i] + zls[i];
    }
    // the next layer's gate/up LoRA partial over this CTA's rows of out
    if (p.vp_next) {
        __syncthreads();
        if (warp == 0) {
            float a = 0.0f;
            if (lane < r2n)
                for (int i = 0; i < no; i++) a = fmaf(anext[lane * no + i], outs[i], a);
            p.vp_next[(size_t)c * 2 * kMaxR + lane] = a;
        }
    }
    if (p.trace) __syncthreads();          // debug: the stamp marks the whole CTA's end
    stamp(p, 2);
    stamp_end(p);
}

// ---------------------------------------------------------------- router kernel
// Layer 0's own router on x0 (rows split over the CTAs) and/or layer 0's
// gate/up LoRA partials over each CTA's rows of x0.
__global__ void __launch_bounds__(kThreads, 1) chain_r_kernel(const __grid_constant__ CP p,
                                                              int do_router, float *zr) {
    extern __shared__ __align__(128) uint8_t sm[];
    const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *x = reinterpret_cast<float *>(sm);                 // padded per 4-bit chunk
    float *xs = x + padded(p.d, 32);
    float *red = xs + p.d / 32;
    stamp(p, 0);
    grid_wait();
    stamp(p, 1);
    stage_vec(p.x_in, p.d, 32, x, xs, red);
    __syncthreads();
    if (do_router) {
        const int e0 = (int)((long long)p.E * c / p.n_cta), e1 = (int)((long long)p.E * (c + 1) / p.n_cta);
        for (int e = e0 + warp; e < e1; e += kWarps) {
            const float a = warp_sum(rec_dot<4>(p.L.router + (size_t)e * p.rec_dh, p.d, x, xs, lane), 32);
            if (lane == 0) zr[e] = a;
        }
    }
    if (p.vp_next && warp == 0) {
        const int o0 = (int)((long long)p.d * c / p.n_cta), o1 = (int)((long long)p.d * (c + 1) / p.n_cta);
        const int rg = p.nr[0], ru = p.nr[1];
        float a = 0.0f;
        if (lane < rg + ru) {
            const uint16_t *A = lane < rg ? p.nA[0] + (size_t)lane * p.d : p.nA[1] + (size_t)(lane - rg) * p.d;
            for (int o = o0; o < o1; o++) a = fmaf(half_at(A, o), x[o + o / 32], a);
        }
        p.vp_next[(size_t)c * 2 * kMaxR + lane] = a;
    }
}

// The next token's routes from every head of the step: warp w of CTA b
// ranks head N = b * kRankWarps + w (heads 0 .. n_heads - 1; head N's logits
// at z + N * E, its target layer N + 1, or 0 for the last one).  Small CTAs,
// so that they fit beside the last layer's kernel B.
constexpr int kRankWarps = 4;
__global__ void __launch_bounds__(kRankWarps * 32) chain_rank_kernel(const __grid_constant__ CP p,
                                                                     const float *z, int n_heads) {
    stamp(p, 0);
    grid_wait();
    stamp(p, 1);
    const int N = blockIdx.x * kRankWarps + (threadIdx.x >> 5);
    if (N < n_heads) route_one(p, z + (size_t)N * p.E, p.topk_set, N + 1 < p.depth ? N + 1 : 0);
    stamp(p, 2);
}

// One warp: the route of layer tgt from logits z.
__global__ void __launch_bounds__(32) chain_topk_kernel(const __grid_constant__ CP p) {
    stamp(p, 0);
    grid_wait();
    stamp(p, 1);
    route_one(p, p.topk_z, p.topk_set, p.topk_tgt);
    stamp(p, 2);
}

// ---------------------------------------------------------------- kernel C
// The cluster variant of a layer: one launch per layer, one thread-block
// cluster of kCluster CTAs per expert slot and one for the head.  CTA j of
// slot s takes gate/up row pairs [F j / C, F (j+1) / C) of that slot and
// output rows [d j / C, d (j+1) / C) of its down projection; h of the slot
// is all-gathered inside the cluster through distributed shared memory, so
// the layer has one global exchange (its input x) instead of two.  Each slot
// cluster writes its weighted output w_s y_s (down LoRA included) to a
// per-slot vector; the next launch sums them onto the residual while it
// stages its x (out(N) = out(N-1) + sum_s w_s y_s), and slot cluster 0
// stores that sum as out(N).  The head cluster takes fc1 rows [H j / C, ...)
// and logit rows [E j / C, ...) (l and fc2), with gelu(fc1 f) all-gathered
// the same way.
//
// Residency: two CTAs per SM, so that the next layer's clusters sit beside
// this layer's and copy their gate/up rows while it runs.  Only the gate/up
// rows go to shared memory (bulk copies); the down rows are prefetched into
// L2 in the prologue and loaded into registers while h is exchanged, and so
// are the rows of the down adapter's A.
//
// Exchanges: a CTA writes its values into every peer's shared memory
// (st.shared::cluster) and then arrives on that peer's mbarrier with release
// semantics at cluster scope (each writing thread arrives itself, so each
// arrive covers the writes before it); the reader waits on its own mbarrier
// (acquire, bounded).  No CTA returns early: a wait that runs out records
// MOE_ETIMEOUT and the CTA carries on (its results are then invalid), so
// every CTA reaches the cluster barrier before exit, after which no peer
// touches its shared memory.
constexpr int kCThreads = 512;
constexpr int kCWarps = kCThreads / 32;
constexpr int kCluster = 16;
constexpr int kDPass = 4;      // down: a warp's passes over its rows (32 / chunks-per-row rows each)
constexpr int kAPass = 4;      // down adapter A: 16-byte pieces of a row per lane (F <= 1024)

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory address of `p` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void peer_store(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void peer_arrive(uint32_t bar_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_addr) : "memory");
}

__device__ __forceinline__ void bar_init_n(uint64_t *bar, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(n));
}

// Bounded wait for phase 0 of a barrier that peers arrive on (acquire at
// cluster scope): false, with MOE_ETIMEOUT in *err, after timeout_ns.
__device__ __forceinline__ bool cbar_wait(uint64_t *bar, int32_t *err, uint64_t timeout_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; it++) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0; "
            "selp.u32 %0, 1, 0, p; }"
            : "=r"(ok) : "r"(saddr(bar)) : "memory");
        if (ok) return true;
        uint64_t now;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
        if (it == 0) t0 = now;
        else if (now - t0 > timeout_ns) {
            atomicExch(err, MOE_ETIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    if (bytes) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Even split [n j / C, n (j+1) / C).
__host__ __device__ inline void csplit(int n, int j, int C, int &a, int &b) {
    a = (int)((long long)n * j / C);
    b = (int)((long long)n * (j + 1) / C);
}

// Shared-memory layout of kernel C (byte offsets; the same for every CTA of
// a launch, sized for the largest share of either role).
struct CLay {
    uint32_t wts, xr, xf, xsc, xhat, agu, bgu, bdn, hs, hf, hsc, hhat, vpart, vd, tterm, tsum, zls,
        b2s, red, route, wk, bars, total;
};

__host__ __device__ inline CLay c_layout(int d, int F, int E, int H, int K, int bits, int C, int rmax) {
    const int VALS = 128 / bits;
    const uint32_t rec_d = (uint32_t)record_bytes(d, bits);
    const uint32_t rec_dh = (uint32_t)record_bytes(d, 4), rec_H = H ? (uint32_t)record_bytes(H, 4) : 0u;
    const int np = (F + C - 1) / C, no = (d + C - 1) / C, nh = (H + C - 1) / C, ne = (E + C - 1) / C;
    const size_t slot_w = (size_t)np * 2 * rec_d;
    const size_t head_w = (size_t)(nh + ne) * rec_dh + (size_t)ne * rec_H;
    CLay L;
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) {
        off = (off + align - 1) / align * align;
        const uint32_t at = (uint32_t)off;
        off += bytes;
        return at;
    };
    L.wts = take(slot_w > head_w ? slot_w : head_w, 128);
    L.xr = take((size_t)no * 4, 16);                         // this CTA's rows of x (raw)
    L.xf = take(fix_bytes(d, 4) > fix_bytes(d, bits) ? fix_bytes(d, 4) : fix_bytes(d, bits), 16);
    L.xsc = take((size_t)(d / 32) * 4, 16);
    L.xhat = take((size_t)(d / 32) * 4, 16);
    L.agu = take((size_t)32 * no * 2, 16);                   // [32][no] fp16 gate/up A columns
    L.bgu = take((size_t)np * 32 * 4, 16);                   // [np][32] gate/up B rows
    L.bdn = take((size_t)no * rmax * 4 + 4, 16);             // [no][rmax] down B rows
    const size_t hpad = padded(F, VALS) > (size_t)H ? padded(F, VALS) : (size_t)H;
    L.hs = take(hpad * 4, 16);                               // h padded per chunk / g
    L.hf = take(fix_bytes(F, bits) > (H ? fix_bytes(H, 4) : 0) ? fix_bytes(F, bits) : fix_bytes(H, 4), 16);
    const int nq = F / VALS > (H ? H / 32 : 0) ? F / VALS : H / 32;
    L.hsc = take((size_t)nq * 4, 16);
    L.hhat = take((size_t)nq * 4, 16);
    L.vpart = take((size_t)C * 32 * 4, 16);                  // [C][32] gate/up LoRA partials
    L.vd = take(kMaxR * 4, 16);
    L.tterm = take((size_t)(nh + ne) * (2 * K + 1) * 4 + 4, 16);
    L.tsum = take((size_t)(nh + ne) * 4 + 4, 16);
    L.zls = take((size_t)ne * 4 + 4, 16);
    L.b2s = take((size_t)ne * 4 + 4, 16);
    L.red = take((size_t)kCWarps * 32 * 4, 16);
    L.route = take((kMaxK + 1) * 4, 16);
    L.wk = take((kMaxK + 1) * 4, 16);
    L.bars = take(4 * 8, 8);
    L.total = (uint32_t)off;
    return L;
}

// Extra parameters of kernel C (beside the layer's CP).
struct CX {
    int C;                     // cluster size
    int rmax;                  // largest down adapter rank of the stack
    int prefetch;              // prefetch the down rows into L2 in the prologue
    const float *base;         // out(N-2) (or x0): the residual the partials add onto
    const float *part_in;      // [S][d] weighted slot outputs of layer N-1, or null (layer 0)
    float *part;               // [S][d] this layer's
    float *x_out;              // where out(N-1) is stored (slot cluster 0), or null
};

template <int BITS>
__global__ void __launch_bounds__(kCThreads, 2) chain_c_kernel(const __grid_constant__ CP p,
                                                                const __grid_constant__ CX q) {
    constexpr int VALS = 128 / BITS;
    extern __shared__ __align__(128) uint8_t sm[];
    const int C = q.C;
    const int j = (int)cluster_rank(), cl = blockIdx.x / C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool head = cl >= p.S;
    const int s = cl;                                           // slot (slot clusters)
    const CLay Lo = c_layout(p.d, p.F, p.E, p.H, p.K, BITS, C, q.rmax);
    uint8_t *wts = sm + Lo.wts;
    float *xr = reinterpret_cast<float *>(sm + Lo.xr);
    uint8_t *xf = sm + Lo.xf;
    float *xsc = reinterpret_cast<float *>(sm + Lo.xsc);
    float *xhat = reinterpret_cast<float *>(sm + Lo.xhat);
    uint16_t *agu = reinterpret_cast<uint16_t *>(sm + Lo.agu);
    float *bgu = reinterpret_cast<float *>(sm + Lo.bgu);
    float *bdn = reinterpret_cast<float *>(sm + Lo.bdn);
    float *hs = reinterpret_cast<float *>(sm + Lo.hs);
    uint8_t *hf = sm + Lo.hf;
    float *hsc = reinterpret_cast<float *>(sm + Lo.hsc);
    float *hhat = reinterpret_cast<float *>(sm + Lo.hhat);
    float *vpart = reinterpret_cast<float *>(sm + Lo.vpart);
    float *vd = reinterpret_cast<float *>(sm + Lo.vd);
    float *tterm = reinterpret_cast<float *>(sm + Lo.tterm);
    float *tsum = reinterpret_cast<float *>(sm + Lo.tsum);
    float *zls = reinterpret_cast<float *>(sm + Lo.zls);
    float *b2s = reinterpret_cast<float *>(sm + Lo.b2s);
    float *red = reinterpret_cast<float *>(sm + Lo.red);
    int32_t *route = reinterpret_cast<int32_t *>(sm + Lo.route);
    float *wk = reinterpret_cast<float *>(sm + Lo.wk);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + Lo.bars);   // copies, LoRA v, h / g, test hook

    // this CTA's shares
    int f0, f1, o0, o1, h0, h1, e0, e1;
    csplit(p.F, j, C, f0, f1);
    csplit(p.d, j, C, o0, o1);
    csplit(p.H, j, C, h0, h1);
    csplit(p.E, j, C, e0, e1);
    const int np = f1 - f0, no = o1 - o0, nh = h1 - h0, ne = e1 - e0;
    const uint32_t P = 2 * p.rec_d;
    const uint32_t gbytes = head ? 0u : (uint32_t)np * P;
    const uint32_t dbytes = head ? 0u : (uint32_t)no * p.rec_F;
    const bool shared = !head && s >= p.K;
    // this slot's down adapter (routed: the route's; shared: its own)
    const int rd = head ? 0 : shared ? p.L.sr[2] : p.L.r_d;
    const int rg = shared ? p.L.sr[0] : 0, ru = shared ? p.L.sr[1] : 0;
    const bool gul = rg + ru > 0;
    const int32_t *rcur = p.ridx + ((size_t)p.cur * p.depth + p.N) * p.K;
    const float *wcur = p.rw + ((size_t)p.cur * p.depth + p.N) * p.K;
    const int32_t *rprv = p.ridx + ((size_t)p.prv * p.depth + p.N) * p.K;

    stamp(p, 0);
    if (threadIdx.x == 0) {
        bar_init_n(bar, 1);
        bar_init_n(bar + 1, (uint32_t)C);             // one lane of every CTA
        bar_init_n(bar + 2, (uint32_t)kCWarps * C);   // every warp of every CTA
        bar_init_n(bar + 3, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    auto load_route = [&]() {
        if (threadIdx.x < p.K) {
            route[threadIdx.x] = rcur[threadIdx.x];
            wk[threadIdx.x] = wcur[threadIdx.x];
        }
    };
    if (!p.route_late) load_route();
    __syncthreads();
    cluster_sync();             // every peer's barriers initialised before any remote arrive
    bool bad = false;
    const uint8_t *blob = p.L.pool;   // this slot's expert blob (slot CTAs)
    auto issue = [&]() {
        if (!head) blob = slot_blob(p, route, s, bad);        // every thread
        if (threadIdx.x != 0) return;
        if (!head) {
            bar_expect(bar, gbytes);
            if (gbytes) bulk_copy(wts, blob + p.gu_off + (size_t)f0 * P, gbytes, bar);
            if (q.prefetch) prefetch_l2(blob + p.down_off + (size_t)o0 * p.rec_F, dbytes);
        } else {
            const uint32_t b1 = (uint32_t)nh * p.rec_dh, b2 = (uint32_t)ne * p.rec_dh, b3 = (uint32_t)ne * p.rec_H;
            bar_expect(bar, b1 + b2 + b3);
            if (b1) bulk_copy(wts, p.L.fc1x + (size_t)h0 * p.rec_dh, b1, bar);
            if (b2) bulk_copy(wts + b1, p.L.lx + (size_t)e0 * p.rec_dh, b2, bar);
            if (b3) bulk_copy(wts + b1 + b2, p.L.fc2 + (size_t)e0 * p.rec_H, b3, bar);
        }
        if (bad) atomicExch(p.err, MOE_EINVAL);
    };
    if (!p.route_late) issue();
    // static side data: gate/up adapters' A columns of this CTA's rows and B
    // rows of its pairs (shared slot)
    if (!head && gul) {
        for (int it = threadIdx.x; it < (rg + ru) * no; it += blockDim.x) {
            const int k = it / no, i = it - k * no;
            const uint16_t *A = k < rg ? p.L.sa[0] + (size_t)k * p.d : p.L.sa[1] + (size_t)(k - rg) * p.d;
            agu[k * no + i] = A[o0 + i];
        }
        for (int it = threadIdx.x; it < np * 32; it += blockDim.x) {
            const int i = it >> 5, k = it & 31, f = f0 + i;
            float v = 0.0f;
            if (k < rg) v = half_at(p.L.sb[0], (size_t)f * rg + k);
            else if (k < rg + ru) v = half_at(p.L.sb[1], (size_t)f * ru + (k - rg));
            bgu[i * 32 + k] = v;
        }
    }
    // route-dependent side data: down B rows of this CTA's outputs; the head's
    // table sums (routes of layer N now and at t - 1) and fc2 biases
    auto side = [&]() {
        if (!head && rd) {
            const bool ok = shared || (unsigned)route[s] < (unsigned)p.E;
            const uint16_t *B = shared ? p.L.sb[2] : p.L.lb_d + (size_t)(ok ? route[s] : 0) * p.L.lb_ds;
            for (int it = threadIdx.x; it < no * rd; it += blockDim.x) {
                const int i = it / rd, k = it - i * rd;
                bdn[i * q.rmax + k] = ok ? half_at(B, (size_t)(o0 + i) * rd + k) : 0.0f;
            }
        }
        if (head) {
            const int nt = 2 * p.K + 1, nr = nh + ne;
            for (int it = threadIdx.x; it < nr * nt; it += blockDim.x) {
                const int i = it / nt, t = it - i * nt;
                const bool fc1 = i < nh;
                const int row = fc1 ? h0 + i : e0 + (i - nh);
                const int width = fc1 ? p.H : p.E;
                const uint16_t *tab = fc1 ? p.L.fc1_tab : p.L.l_tab;
                const uint16_t *bias = fc1 ? p.L.b1 : p.L.bl;
                float a = 0.0f;
                if (t == 2 * p.K) a = bias ? half_at(bias, row) : 0.0f;
                else if (tab) {
                    const int e = t < p.K ? route[t] : rprv[t - p.K];
                    if ((unsigned)e < (unsigned)p.E) a = half_at(tab, (size_t)(t < p.K ? e : p.E + e) * width + row);
                }
                tterm[it] = a;
            }
            for (int i = threadIdx.x; i < ne; i += blockDim.x) b2s[i] = p.L.b2 ? half_at(p.L.b2, e0 + i) : 0.0f;
            __syncthreads();
            for (int i = threadIdx.x; i < nr; i += blockDim.x) {
                float a = 0.0f;
                for (int t = 0; t < nt; t++) a += tterm[i * nt + t];
                tsum[i] = a;
            }
        }
    };
    if (!p.route_late) side();
    stamp(p, 5);
    grid_launch_dependents();
    grid_wait();
    stamp(p, 1);
    if (p.route_late) {
        load_route();
        __syncthreads();
        issue();
        side();
    }
    // x = out(N-1) = base + sum_s part_in[s] (or x0): this CTA's rows kept
    // raw, the whole vector staged as fixed point (slot: BITS chunks; head:
    // 4-bit chunks); 1/rms of it when it is an out.  The slot vectors' loads
    // are issued eight at a time, unconditionally, before their sum.
    float ss = 0.0f;
    for (int b0 = 0; b0 < p.d / 4; b0 += blockDim.x) {          // uniform over the block
        const int i = b0 + threadIdx.x;
        const bool in = i < p.d / 4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (in) {
            v = reinterpret_cast<const float4 *>(q.base)[i];
            if (q.part_in)
                for (int k0 = 0; k0 < p.S; k0 += 8) {
                    float4 t[8];
#pragma unroll
                    for (int u = 0; u < 8; u++)
                        t[u] = reinterpret_cast<const float4 *>(q.part_in + (size_t)min(k0 + u, p.S - 1) * p.d)[i];
#pragma unroll
                    for (int u = 0; u < 8; u++)
                        if (k0 + u < p.S) {
                            v.x += t[u].x;
                            v.y += t[u].y;
                            v.z += t[u].z;
                            v.w += t[u].w;
                        }
                }
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int u = 0; u < 4; u++)
                if (4 * i + u >= o0 && 4 * i + u < o1) xr[4 * i + u - o0] = vv[u];
        }
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        if (head) quant4<4>(v, i, in, xf, p.d / 32, xsc, xhat);
        else quant4<BITS>(v, i, in, xf, p.d / VALS, xsc, xhat);
    }
    ss = warp_sum(ss, 32);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float inv = 1.0f;
    if (p.x_is_out) {
        float t = 0.0f;
        for (int w = 0; w < kCWarps; w++) t += red[w];
        inv = 1.0f / sqrtf(t / p.d + 1e-6f);
    }
    stamp(p, 3);
    // slot cluster 0 stores out(N-1)
    if (!head && s == 0 && q.x_out)
        for (int i = threadIdx.x; i < no; i += blockDim.x) q.x_out[o0 + i] = xr[i];
    // shared gate/up LoRA: this CTA's partial of A x over its rows, to every
    // peer (warp 0; lane k holds entry k)
    if (!head && gul) {
        __syncthreads();                                         // red reused below
        float a = 0.0f;
        if (lane < rg + ru)
            for (int i = warp; i < no; i += kCWarps) a = fmaf(half_f(agu[lane * no + i]), xr[i], a);
        red[warp * 32 + lane] = a;
        __syncthreads();
        if (warp == 0) {
            // lane r sends the 32 entries to peer r and arrives once there
            // (one release per lane, all lanes at once)
            float v = 0.0f;
            for (int w = 0; w < kCWarps; w++) v += red[w * 32 + lane];
            vd[lane] = v;
            __syncwarp();
            if (lane < C) {
                for (int k = 0; k < 32; k++) peer_store(peer_addr(vpart + j * 32 + k, lane), vd[k]);
                peer_arrive(peer_addr(bar + 1, lane));
            }
        }
    }
    bar_wait(bar, p.err, p.timeout_ns);
    if (p.debug_unset_wait && blockIdx.x == 0) {
        // test hook: a wait for 16 bytes no copy delivers; it runs out after
        // timeout_ns and records MOE_ETIMEOUT (the CTA carries on)
        if (threadIdx.x == 0) bar_expect(bar + 3, 16);
        __syncthreads();
        bar_wait(bar + 3, p.err, p.timeout_ns);
    }
    stamp(p, 4);
    if (!head) {
        // gate/up pairs, two per warp (records g, u, g', u') -> h, pushed to
        // every peer
        float vxl = 0.0f;                 // lane k: entry k of the adapters' A x
        bool vready = false;
        auto emit = [&](int v, float g, float u) {
            float a0 = g * inv, a1 = u * inv;
            if (gul) {
                if (!vready) {
                    cbar_wait(bar + 1, p.err, p.timeout_ns);
                    for (int r = 0; r < C; r++) vxl += vpart[r * 32 + lane];
                    vxl *= inv;
                    vready = true;
                }
                const float t = bgu[v * 32 + lane] * vxl;
                a0 = fmaf(p.L.ss[0], lane < rg ? t : 0.0f, a0);
                a1 = fmaf(p.L.ss[1], lane < rg ? 0.0f : t, a1);
            }
            const float gg = warp_sum(a0, 32), uu = warp_sum(a1, 32);
            const float hv = silu_f(gg) * uu;
            const int f = f0 + v;
            if (lane < C) peer_store(peer_addr(hs + f + f / VALS, lane), hv);
        };
        const int np2 = np / 2 * 2;
        for (int v = 2 * warp; v < np2; v += 2 * kCWarps) {
            float gu[4];
            fix_dot<BITS, 4>(wts + (size_t)v * P, p.rec_d, p.d, xf, xsc, xhat, lane, gu);
            emit(v, gu[0], gu[1]);
            emit(v + 1, gu[2], gu[3]);
        }
        for (int v = np2 + warp; v < np; v += kCWarps) {
            float gu[2];
            fix_dot<BITS, 2>(wts + (size_t)v * P, p.rec_d, p.d, xf, xsc, xhat, lane, gu);
            emit(v, gu[0], gu[1]);
        }
        // this warp's down rows into registers while h is exchanged: rows
        // [warp rw, (warp + 1) rw) of the CTA's, pass k lane l: row
        // k G + l / nch, chunk l % nch
        const int nch = p.F / VALS, G = 32 / nch;
        const int rw = (no + kCWarps - 1) / kCWarps;
        const int gl = lane / nch, c = lane - gl * nch;
        const size_t cbF = code_bytes(p.F, BITS);
        const uint8_t *down = blob + p.down_off + (size_t)o0 * p.rec_F;
        uint4 dw[kDPass];
        uint32_t dsb[kDPass];
#pragma unroll
        for (int k = 0; k < kDPass; k++) {
            const int r = k * G + gl, i = warp * rw + r;
            const bool okr = r < rw && i < no;
            const uint8_t *rec = down + (size_t)(okr ? i : 0) * p.rec_F;
            dw[k] = okr ? __ldg(reinterpret_cast<const uint4 *>(rec + (size_t)kChunk * c)) : make_uint4(0, 0, 0, 0);
            dsb[k] = okr ? __ldg(reinterpret_cast<const unsigned int *>(rec + cbF + 4 * ((c * VALS) / kGroup))) : 0u;
        }
        // ... and the down adapter's A row `warp` (k < rd)
        uint4 av[kAPass];
        const uint16_t *Ad = nullptr;
        if (warp < rd)
            Ad = (shared ? p.L.sa[2]
                         : p.L.la_d + (size_t)((unsigned)route[s] < (unsigned)p.E ? route[s] : 0) * p.L.la_ds) +
                 (size_t)warp * p.F;
#pragma unroll
        for (int k = 0; k < kAPass; k++) {
            const int f = (k * 32 + lane) * 8;
            av[k] = Ad && f < p.F ? __ldg(reinterpret_cast<const uint4 *>(Ad + f)) : make_uint4(0, 0, 0, 0);
        }
        if (lane < C) peer_arrive(peer_addr(bar + 2, lane));
        cbar_wait(bar + 2, p.err, p.timeout_ns);
        stamp(p, 6);
        // h as fixed point per chunk (from the padded floats)
        for (int b0 = 0; b0 < p.F / 4; b0 += blockDim.x) {
            const int i = b0 + threadIdx.x;
            const bool in = i < p.F / 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (in) {
                const int ch = (4 * i) / VALS;
                const float *src = hs + ch * (VALS + 1) + (4 * i - ch * VALS);
                v = make_float4(src[0], src[1], src[2], src[3]);
            }
            quant4<BITS>(v, i, in, hf, nch, hsc, hhat);
        }
        // down LoRA: vd[k] = A_d[k] h (warp k)
        if (warp < rd) {
            float a = 0.0f;
#pragma unroll
            for (int k = 0; k < kAPass; k++) {
                const int f = (k * 32 + lane) * 8;
                if (f < p.F) {
                    const uint32_t w[4] = {av[k].x, av[k].y, av[k].z, av[k].w};
#pragma unroll
                    for (int u = 0; u < 8; u++) {
                        const int g = f + u;
                        a = fmaf(half_f((uint16_t)(w[u >> 1] >> (16 * (u & 1)))), hs[g + g / VALS], a);
                    }
                }
            }
            a = warp_sum(a, 32);
            if (lane == 0) vd[warp] = a;
        }
        __syncthreads();
        // down rows: w_s (y + s_d B_d vd), the nch lanes of a row summed by
        // shuffles
        const bool valid = shared || (unsigned)route[s] < (unsigned)p.E;
        const float ws = shared ? 1.0f : wk[s];
        const float sc = shared ? p.L.ss[2] : p.L.s_d;
#pragma unroll
        for (int k = 0; k < kDPass; k++) {
            if (k * G >= rw) break;                              // uniform over the warp
            const int r = k * G + gl, i = warp * rw + r;
            const bool okr = r < rw && i < no;
            const uint4 w1[1] = {dw[k]};
            int dq[1];
            chunk_dot_fix<BITS, 1>(w1, reinterpret_cast<const uint4 *>(hf), nch, c, dq);
            const float2 sb = sb_f(dsb[k]);
            float y = fmaf(sb.x, (float)dq[0] * hsc[c], sb.y * hhat[c]);
            if (okr) {
                float l = 0.0f;
                for (int kk = c; kk < rd; kk += nch) l = fmaf(bdn[i * q.rmax + kk], vd[kk], l);
                y = fmaf(sc, l, y);
            } else {
                y = 0.0f;
            }
            for (int o = 1; o < nch; o <<= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
            if (c == 0 && okr) q.part[(size_t)s * p.d + o0 + i] = valid ? ws * y : 0.0f;
        }
    } else {
        // fc1 rows (warp per row) -> gelu -> pushed to every peer; l rows
        for (int v = warp; v < nh; v += kCWarps) {
            float hd[1];
            fix_dot<4, 1>(wts + (size_t)v * p.rec_dh, 0, p.d, xf, xsc, xhat, lane, hd);
            const float gv = gelu_erf_f(warp_sum(hd[0], 32) * inv + tsum[v]);
            if (lane < C) peer_store(peer_addr(hs + h0 + v, lane), gv);
        }
        if (lane < C) peer_arrive(peer_addr(bar + 2, lane));
        for (int v = warp; v < ne; v += kCWarps) {
            float hd[1];
            fix_dot<4, 1>(wts + (size_t)(nh + v) * p.rec_dh, 0, p.d, xf, xsc, xhat, lane, hd);
            const float a = warp_sum(hd[0], 32) * inv + tsum[nh + v];
            if (lane == 0) zls[v] = a;
        }
        cbar_wait(bar + 2, p.err, p.timeout_ns);
        stamp(p, 6);
        // g as fixed point (4-bit chunks), then the fc2 rows: z = fc2 g + b2 + l f
        for (int b0 = 0; b0 < p.H / 4; b0 += blockDim.x) {
            const int i = b0 + threadIdx.x;
            const bool in = i < p.H / 4;
            const float4 v = in ? reinterpret_cast<const float4 *>(hs)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            quant4<4>(v, i, in, hf, p.H / 32, hsc, hhat);
        }
        __syncthreads();
        const uint8_t *w2 = wts + (size_t)(nh + ne) * p.rec_dh;
        for (int v = warp; v < ne; v += kCWarps) {
            float f2[1];
            fix_dot<4, 1>(w2 + (size_t)v * p.rec_H, 0, p.H, hf, hsc, hhat, lane, f2);
            const float a = warp_sum(f2[0], 32);
            if (lane == 0) p.z[e0 + v] = a + b2s[v] + zls[v];
        }
    }
    stamp(p, 2);
    stamp_end(p);
    cluster_sync();             // no peer reads or writes this CTA's shared memory after this
}

// out = base + sum_s part[s] (the last layer's outputs onto its residual).
__global__ void __launch_bounds__(256) chain_fin_kernel(const __grid_constant__ CP p,
                                                        const __grid_constant__ CX q) {
    grid_launch_dependents();
    grid_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.d / 4) return;
    float4 v = reinterpret_cast<const float4 *>(q.base)[i];
    for (int k = 0; k < p.S; k++) {
        const float4 t = reinterpret_cast<const float4 *>(q.part_in + (size_t)k * p.d)[i];
        v.x += t.x;
        v.y += t.y;
        v.z += t.z;
        v.w += t.w;
    }
    reinterpret_cast<float4 *>(p.out)[i] = v;
}

}  // namespace chain
}  // namespace moe

// ====================================================================== host
namespace moe {
namespace chain {

static size_t al256(size_t v) { return (v + 255) / 256 * 256; }

// Workspace: status word | out per layer [depth][d] | h [depth][S][F] |
// gelu(fc1 f) [depth][H] | l f [depth][E] | head logits [depth][E] | router
// logits [E] | LoRA partials [depth][n_cta][2 kMaxR].
struct Ws {
    size_t outs, h, g, zl, z, zr, vp, total;
};

static Ws ws_layout(int d, int F, int E, int H, int S, int depth, int n_cta) {
    Ws w;
    size_t off = 256;
    w.outs = off;
    off = al256(off + (size_t)depth * d * 4);
    w.h = off;
    off = al256(off + (size_t)depth * S * F * 4);
    w.g = off;
    off = al256(off + (size_t)depth * (H > 0 ? H : 1) * 4);
    w.zl = off;
    off = al256(off + (size_t)depth * E * 4);
    w.z = off;
    off = al256(off + (size_t)depth * E * 4);
    w.zr = off;
    off = al256(off + (size_t)E * 4);
    w.vp = off;
    off = al256(off + (size_t)depth * n_cta * 2 * kMaxR * 4);
    w.total = off;
    return w;
}

static int sms_of_device() {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

struct Shapes {
    int d, F, E, K, H, S, bits, depth, n_res, self_predict, own0;
    int rd_routed, rd_shared;      // down adapter ranks
    bool heads;
};

static Shapes shapes_of(const moe_stack_desc *sd) {
    const moe_experts_desc &e0 = sd->experts[0];
    Shapes s;
    s.d = e0.d;
    s.F = e0.F;
    s.E = e0.E;
    s.K = sd->K;
    s.heads = sd->depth > 1 || sd->self_predict;
    s.H = s.heads ? sd->heads[0].H : 0;
    s.S = sd->K + (e0.shared ? 1 : 0);
    s.bits = e0.bits;
    s.depth = sd->depth;
    s.n_res = sd->n_layers;
    s.self_predict = sd->self_predict;
    s.own0 = !sd->self_predict;
    s.rd_routed = e0.lora[2].r;
    s.rd_shared = e0.shared ? e0.shared_lora[2].r : 0;
    return s;
}

static bool head_runs(const Shapes &s, int N) { return N + 1 < s.depth || s.self_predict; }

// Shared-memory bytes of kernel A and B (the largest CTA share).
static void smem_need(const Shapes &s, int n_cta, size_t *sa, size_t *sb) {
    const int VALS = 128 / s.bits;
    const uint32_t rec_d = (uint32_t)record_bytes(s.d, s.bits), rec_dh = (uint32_t)record_bytes(s.d, 4);
    const uint32_t rec_F = (uint32_t)record_bytes(s.F, s.bits);
    const uint32_t rec_H = s.H ? (uint32_t)record_bytes(s.H, 4) : 0u;
    size_t a = 0;
    for (int head = 0; head < 2; head++) {
        const ASplit sp = a_split(s.S, s.F, s.H, s.E, head, rec_d, rec_dh);
        for (int c = 0; c < n_cta; c++) {
            long long g0, g1;
            int r0, r1;
            sp.range(c, n_cta, g0, g1, r0, r1);
            const size_t wb = (size_t)((g1 - g0) * sp.P + (long long)(r1 - r0) * sp.R);
            const size_t nh = (size_t)(r1 - r0);
            size_t need = (wb + 127) / 128 * 128 +
                          fix_bytes(s.d, s.bits) + (size_t)(s.d / VALS) * 8 +
                          (s.bits != 4 ? fix_bytes(s.d, 4) + (size_t)(s.d / 32) * 8 : 0) +
                          (nh + 1) * 4 + (nh * (2 * s.K + 1) + 1) * 4 +
                          2 * kMaxR * 4 + kWarps * 32 * 4 + ((wb / sp.P + 2) * 2 * kMaxR + 1) * 4 +
                          32 * 4 + (kMaxK + 1) * 4 + 24;      // two mbarriers (8-aligned)
            if (need > a) a = need;
        }
    }
    const int no = (s.d + n_cta - 1) / n_cta, ne = (s.E + n_cta - 1) / n_cta;
    *sa = a;
    *sb = ((size_t)s.S * no * rec_F + (size_t)ne * rec_H + 127) / 128 * 128 + padded(s.S * s.F, VALS) * 4 +
          fix_bytes(s.S * s.F, s.bits) +
          (size_t)(s.S * s.F / VALS) * 8 + (s.H > 0 ? fix_bytes(s.H, 4) : 16) +
          (size_t)(s.H > 0 ? s.H / 32 : 1) * 8 + (size_t)s.S * kMaxR * 4 +
          ((size_t)(s.K * s.rd_routed + s.rd_shared) * s.F * 2 + 15) / 16 * 16 +
          (size_t)2 * kMaxR * (no + 1) * 4 + (size_t)(no + 1) * 12 + (size_t)(ne + 1) * 8 +
          (size_t)s.S * (no + 1) * kMaxR * 4 +
          2 * (kMaxK + 1) * 4 + 16;
}

static CLayer layer_of(const moe_stack_desc *sd, int N, const Shapes &s) {
    const int i = N % s.n_res;
    const moe_experts_desc &e = sd->experts[i];
    CLayer L{};
    L.pool = static_cast<const uint8_t *>(e.pool);
    L.shared = static_cast<const uint8_t *>(e.shared);
    L.la_d = e.lora[2].A;
    L.lb_d = e.lora[2].B;
    L.la_ds = e.lora[2].a_stride;
    L.lb_ds = e.lora[2].b_stride;
    L.r_d = e.lora[2].r;
    L.s_d = e.lora[2].scale;
    for (int j = 0; j < 3; j++) {
        L.sa[j] = e.shared ? e.shared_lora[j].A : nullptr;
        L.sb[j] = e.shared ? e.shared_lora[j].B : nullptr;
        L.sr[j] = e.shared ? e.shared_lora[j].r : 0;
        L.ss[j] = e.shared ? e.shared_lora[j].scale : 0.0f;
    }
    L.router = static_cast<const uint8_t *>(sd->routers[i].lx);
    if (s.heads) {
        const moe_head_desc &h = sd->heads[i];
        L.fc1x = static_cast<const uint8_t *>(h.fc1x);
        L.fc2 = static_cast<const uint8_t *>(h.fc2);
        L.lx = static_cast<const uint8_t *>(h.lx);
        L.fc1_tab = h.fc1_tab;
        L.b1 = h.b1;
        L.b2 = h.b2;
        L.l_tab = h.l_tab;
        L.bl = h.bl;
    }
    return L;
}

template <typename Kern>
static int launch(Kern k, const CP &p, int grid, int threads, size_t smem, bool pdl, cudaStream_t st,
                  const char *what) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, p);
    if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step_chain: %s launch: %s", what, cudaGetErrorString(e));
    return MOE_OK;
}

// Once per (device, BITS) and host thread: every chain kernel may use the
// device's largest dynamic shared memory and asks for the same (largest)
// carveout -- an SM only holds CTAs of one carveout at a time, and a kernel
// with a smaller one would wait for the SM to drain instead of starting
// beside its predecessor.
template <int BITS>
static int configure(int dev, int smem_max) {
    static thread_local int done_dev = -1;
    if (done_dev == dev) return MOE_OK;
    const int co = cudaSharedmemCarveoutMaxShared;
    if (cudaFuncSetAttribute(chain_a_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) != cudaSuccess ||
        cudaFuncSetAttribute(chain_b_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) != cudaSuccess ||
        cudaFuncSetAttribute(chain_a_kernel<BITS>, cudaFuncAttributePreferredSharedMemoryCarveout, co) != cudaSuccess ||
        cudaFuncSetAttribute(chain_b_kernel<BITS>, cudaFuncAttributePreferredSharedMemoryCarveout, co) != cudaSuccess ||
        cudaFuncSetAttribute(chain_r_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, co) != cudaSuccess ||
        cudaFuncSetAttribute(chain_topk_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, co) != cudaSuccess ||
        cudaFuncSetAttribute(chain_rank_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, co) != cudaSuccess)
        return fail(MOE_ECUDA, "decode_step_chain: shared-memory attribute");
    done_dev = dev;
    return MOE_OK;
}

// Residency of the two per-layer kernels on the current device: CTAs of each
// an SM holds alone (occupancy API), and whether an SM holds a CTA of A
// beside one of B (shared memory incl. the per-CTA reservation, registers
// in their allocation granules) -- what lets A(N+1) stream its weights
// while B(N) runs.
template <int BITS>
static int residency(const Shapes &s, int n_cta, moe_chain_info *info) {
    size_t sa, sb;
    smem_need(s, n_cta, &sa, &sb);
    int dev = 0, smem_max = 0, smem_sm = 0, reserved = 0, regs_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    *info = moe_chain_info{};
    info->smem_a = sa;
    info->smem_b = sb;
    info->threads = kThreads;
    if (sa > (size_t)smem_max || sb > (size_t)smem_max)
        return fail(MOE_EUNSUPPORTED, "decode_step_chain: %zu / %zu bytes of shared memory (at most %d)",
                    sa, sb, smem_max);
    if (int rc = configure<BITS>(dev, smem_max)) return rc;
    cudaFuncAttributes fa{}, fb{};
    if (cudaFuncGetAttributes(&fa, chain_a_kernel<BITS>) != cudaSuccess ||
        cudaFuncGetAttributes(&fb, chain_b_kernel<BITS>) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&info->ctas_a, chain_a_kernel<BITS>, kThreads, sa) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&info->ctas_b, chain_b_kernel<BITS>, kThreads, sb) != cudaSuccess)
        return fail(MOE_ECUDA, "decode_step_chain: kernel attributes / occupancy");
    info->regs_a = fa.numRegs;
    info->regs_b = fb.numRegs;
    info->local_bytes_a = (int)fa.localSizeBytes;
    info->local_bytes_b = (int)fb.localSizeBytes;
    const auto granule = [](int r) { return (r + 7) / 8 * 8; };
    info->coresident = sa + sb + 2 * (size_t)reserved <= (size_t)smem_sm &&
                       (granule(fa.numRegs) + granule(fb.numRegs)) * kThreads <= regs_sm &&
                       info->ctas_a >= 1 && info->ctas_b >= 1;
    if (info->ctas_a < 1 || info->ctas_b < 1)
        return fail(MOE_EUNSUPPORTED, "decode_step_chain: a kernel does not fit an SM (%d / %d CTAs)",
                    info->ctas_a, info->ctas_b);
    return MOE_OK;
}

// CTAs per kernel of the step: one per SM, less the SMs the caller leaves
// free (at least one).
static int chain_ctas(const moe_stack_desc *sd) {
    const int sms = sms_of_device();
    if (sms <= 0) return sms;
    return std::max(1, sms - std::max(0, sd->free_sms));
}

template <int BITS>
static int run(const moe_stack_desc *sd, const Shapes &s, const float *x0, float *out,
               int32_t *ridx, float *rw, float *rmargin, int t, uint8_t *ws, cudaStream_t st) {
    const int n_cta = chain_ctas(sd);
    const Ws W = ws_layout(s.d, s.F, s.E, s.H, s.S, s.depth, n_cta);
    moe_chain_info info;
    if (int rc = residency<BITS>(s, n_cta, &info)) return rc;
    const size_t sa = info.smem_a, sb = info.smem_b;
    const size_t sr = padded(s.d, 32) * 4 + (size_t)(s.d / 32) * 4 + 32 * 4 + 16;
    int32_t *err = reinterpret_cast<int32_t *>(ws);
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), st) != cudaSuccess)
        return fail(MOE_ECUDA, "decode_step_chain: status reset");
    float *outs = reinterpret_cast<float *>(ws + W.outs), *h = reinterpret_cast<float *>(ws + W.h);
    float *g = reinterpret_cast<float *>(ws + W.g), *zl = reinterpret_cast<float *>(ws + W.zl);
    float *z = reinterpret_cast<float *>(ws + W.z), *zr = reinterpret_cast<float *>(ws + W.zr);
    float *vp = reinterpret_cast<float *>(ws + W.vp);
    const int Hs = s.H > 0 ? s.H : 1;
    const size_t vps = (size_t)n_cta * 2 * kMaxR;
    const int cur = t % 3, nxt = (t + 1) % 3, prv = (t + 2) % 3;

    CP b{};
    b.d = s.d;
    b.F = s.F;
    b.E = s.E;
    b.K = s.K;
    b.H = s.H;
    b.S = s.S;
    b.n_cta = n_cta;
    b.depth = s.depth;
    b.cur = cur;
    b.prv = prv;
    const BlobLayout BL = blob_layout(s.d, s.F, s.bits);
    b.stride = sd->experts[0].expert_stride;
    b.gu_off = (uint32_t)BL.gu_off;
    b.down_off = (uint32_t)BL.down_off;
    b.rec_d = (uint32_t)BL.gu_rec;
    b.rec_F = (uint32_t)BL.down_rec;
    b.rec_dh = (uint32_t)record_bytes(s.d, 4);
    b.rec_H = s.H ? (uint32_t)record_bytes(s.H, 4) : 0u;
    b.ridx = ridx;
    b.rw = rw;
    b.rmargin = rmargin;
    b.err = err;
    b.timeout_ns = sd->timeout_ns ? sd->timeout_ns : kDefaultWaitNs;
    b.trace = sd->debug_trace;
    int lid = 0;
    const moe_experts_desc &e0 = sd->experts[0];
    b.gu_lora = e0.shared && (e0.shared_lora[0].r || e0.shared_lora[1].r);
    auto next_lora = [&](CP &p, int M) {       // layer M's shared gate / up A, its partials
        if (!b.gu_lora || M >= s.depth) return;
        const moe_experts_desc &e = sd->experts[M % s.n_res];
        p.nA[0] = e.shared_lora[0].A;
        p.nA[1] = e.shared_lora[1].A;
        p.nr[0] = e.shared_lora[0].r;
        p.nr[1] = e.shared_lora[1].r;
        p.vp_next = vp + (size_t)M * vps;
    };
    bool first = true;
    // layer 0: its own router on x0 (every step) and its gate/up LoRA partials
    if (s.own0 || b.gu_lora) {
        CP p = b;
        p.N = 0;
        p.launch_id = lid++;
        p.L = layer_of(sd, 0, s);
        p.x_in = x0;
        next_lora(p, 0);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n_cta);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = sr;
        cfg.stream = st;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, chain_r_kernel, p, s.own0 ? 1 : 0, zr);
        if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step_chain: router launch: %s", cudaGetErrorString(e));
        first = false;
        if (s.own0) {
            CP q = b;
            q.launch_id = lid++;
            q.topk_z = zr;
            q.topk_set = cur;
            q.topk_tgt = 0;
            if (int rc = launch(chain_topk_kernel, q, 1, 32, 0, true, st, "router top-K")) return rc;
        }
    }
    for (int N = 0; N < s.depth; N++) {
        CP p = b;
        p.N = N;
        p.L = layer_of(sd, N, s);
        p.head = head_runs(s, N) ? 1 : 0;
        p.route_late = N == 0 && s.own0;
        p.x_in = N == 0 ? x0 : outs + (size_t)(N - 1) * s.d;
        p.x_is_out = N > 0;
        p.out = N + 1 == s.depth ? out : outs + (size_t)N * s.d;
        p.h = h + (size_t)N * s.S * s.F;
        p.g = g + (size_t)N * Hs;
        p.zl = zl + (size_t)N * s.E;
        p.z = z + (size_t)N * s.E;
        p.vp = vp + (size_t)N * vps;
        next_lora(p, N + 1);
        p.smap = sd->slot_map && !p.route_late ? sd->slot_map + (size_t)N * s.K : nullptr;
        if (sd->layer_ready && sd->layer_ready[N]) {
            const cudaError_t e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(sd->layer_ready[N]), 0);
            if (e != cudaSuccess)
                return fail(MOE_ECUDA, "decode_step_chain: wait for layer %d: %s", N, cudaGetErrorString(e));
        }
        p.launch_id = lid++;
        p.debug_unset_wait = N == 0 ? sd->debug_unset_wait : 0;
        if (int rc = launch(chain_a_kernel<BITS>, p, n_cta, kThreads, sa, !first, st, "A")) return rc;
        first = false;
        p.debug_unset_wait = 0;
        p.launch_id = lid++;
        if (int rc = launch(chain_b_kernel<BITS>, p, n_cta, kThreads, sb, true, st, "B")) return rc;
    }
    // the next token's routes: every head that ran (heads 0 .. depth - 2, and
    // the last one for a single self-predicting layer)
    const int n_heads = head_runs(s, s.depth - 1) ? s.depth : s.depth - 1;
    if (n_heads > 0) {
        CP q = b;
        q.launch_id = lid++;
        q.topk_set = nxt;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((n_heads + kRankWarps - 1) / kRankWarps);
        cfg.blockDim = dim3(kRankWarps * 32);
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, chain_rank_kernel, q, (const float *)z, n_heads);
        if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step_chain: ranking launch: %s", cudaGetErrorString(e));
    }
    return MOE_OK;
}

// ---------------------------------------------------------------- cluster variant (host)
// Which variant moe_decode_step_chain runs: 0 the library's choice, 1 two
// kernels per layer, 2 one cluster kernel per layer; and whether the cluster
// kernel prefetches its down rows into L2 in its prologue.
static int g_variant = 0;
static int g_prefetch = 1;

// Workspace of the cluster variant: status word | out per layer [depth][d] |
// weighted slot outputs [depth][S][d] | head logits [depth][E] | router
// logits [E].
struct CWs {
    size_t outs, part, z, zr, total;
};

static CWs cws_layout(int d, int E, int S, int depth) {
    CWs w;
    size_t off = 256;
    w.outs = off;
    off = al256(off + (size_t)depth * d * 4);
    w.part = off;
    off = al256(off + (size_t)depth * S * d * 4);
    w.z = off;
    off = al256(off + (size_t)depth * E * 4);
    w.zr = off;
    off = al256(off + (size_t)E * 4);
    w.total = off;
    return w;
}

static int c_rmax(const Shapes &s) { return std::max(s.rd_routed, s.rd_shared); }

// Whether the cluster variant takes this stack (a message in *why if not).
template <int BITS>
static bool c_fits(const moe_stack_desc *sd, const Shapes &s, const char **why) {
    const moe_experts_desc &e0 = sd->experts[0];
    const int rg = e0.shared ? e0.shared_lora[0].r : 0, ru = e0.shared ? e0.shared_lora[1].r : 0;
    if (s.heads && (s.H <= 0 || s.H % 32)) {
        *why = "the head width must be a positive multiple of 32";
        return false;
    }
    if (rg + ru > 32 || c_rmax(s) > kCWarps) {
        *why = "adapter ranks too large";
        return false;
    }
    const int nch = s.F / (128 / s.bits), no = (s.d + kCluster - 1) / kCluster;
    const int rw = (no + kCWarps - 1) / kCWarps;
    if (32 % nch || (rw + 32 / nch - 1) / (32 / nch) > kDPass || s.F > kAPass * 256) {
        *why = "the down rows of a warp do not fit its registers";
        return false;
    }
    const CLay Lo = c_layout(s.d, s.F, s.E, s.H, s.K, s.bits, kCluster, c_rmax(s));
    int dev = 0, smem_max = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (Lo.total > (uint32_t)smem_max) {
        *why = "a CTA's share of a slot does not fit shared memory";
        return false;
    }
    return true;
}

template <int BITS>
static int c_configure(int dev, uint32_t smem) {
    static thread_local int done_dev = -1;
    static thread_local uint32_t done_smem = 0;
    if (done_dev == dev && done_smem >= smem) return MOE_OK;
    int smem_max = 0;
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (cudaFuncSetAttribute(chain_c_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) != cudaSuccess ||
        cudaFuncSetAttribute(chain_c_kernel<BITS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
        cudaFuncSetAttribute(chain_c_kernel<BITS>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaFuncSetAttribute(chain_fin_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return fail(MOE_ECUDA, "decode_step_chain: cluster kernel attributes");
    done_dev = dev;
    done_smem = smem;
    return MOE_OK;
}

// Clusters of the layer kernel an SM set can hold at once (occupancy API).
template <int BITS>
static int c_clusters(int grid, uint32_t smem, int *n) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kCluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(n, chain_c_kernel<BITS>, &cfg) != cudaSuccess)
        return fail(MOE_ECUDA, "decode_step_chain: cluster occupancy");
    return MOE_OK;
}

template <int BITS>
static int run_c(const moe_stack_desc *sd, const Shapes &s, const float *x0, float *out, int32_t *ridx,
                 float *rw, float *rmargin, int t, uint8_t *ws, cudaStream_t st) {
    const int C = kCluster, rmax = c_rmax(s);
    const CLay Lo = c_layout(s.d, s.F, s.E, s.H, s.K, s.bits, C, rmax);
    int dev = 0, smem_max = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (int rc = configure<BITS>(dev, smem_max)) return rc;
    if (int rc = c_configure<BITS>(dev, Lo.total)) return rc;
    int ncl = 0;
    if (int rc = c_clusters<BITS>((s.S + 1) * C, Lo.total, &ncl)) return rc;
    if (ncl < 1)
        return fail(MOE_EUNSUPPORTED, "decode_step_chain: no cluster of %d CTAs with %u bytes fits", C, Lo.total);
    const CWs W = cws_layout(s.d, s.E, s.S, s.depth);
    int32_t *err = reinterpret_cast<int32_t *>(ws);
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), st) != cudaSuccess)
        return fail(MOE_ECUDA, "decode_step_chain: status reset");
    float *outs = reinterpret_cast<float *>(ws + W.outs), *part = reinterpret_cast<float *>(ws + W.part);
    float *z = reinterpret_cast<float *>(ws + W.z), *zr = reinterpret_cast<float *>(ws + W.zr);
    const int cur = t % 3, nxt = (t + 1) % 3, prv = (t + 2) % 3;
    const size_t ps = (size_t)s.S * s.d;

    CP b{};
    b.d = s.d;
    b.F = s.F;
    b.E = s.E;
    b.K = s.K;
    b.H = s.H;
    b.S = s.S;
    b.n_cta = (s.S + 1) * C;
    b.depth = s.depth;
    b.cur = cur;
    b.prv = prv;
    const BlobLayout BL = blob_layout(s.d, s.F, s.bits);
    b.stride = sd->experts[0].expert_stride;
    b.gu_off = (uint32_t)BL.gu_off;
    b.down_off = (uint32_t)BL.down_off;
    b.rec_d = (uint32_t)BL.gu_rec;
    b.rec_F = (uint32_t)BL.down_rec;
    b.rec_dh = (uint32_t)record_bytes(s.d, 4);
    b.rec_H = s.H ? (uint32_t)record_bytes(s.H, 4) : 0u;
    b.ridx = ridx;
    b.rw = rw;
    b.rmargin = rmargin;
    b.err = err;
    b.timeout_ns = sd->timeout_ns ? sd->timeout_ns : kDefaultWaitNs;
    b.trace = sd->debug_trace;
    int lid = 0;
    bool first = true;
    if (s.own0) {
        // layer 0 routes itself on x0 (router logits, then its top-K)
        CP p = b;
        p.N = 0;
        p.n_cta = sms_of_device();
        p.launch_id = lid++;
        p.L = layer_of(sd, 0, s);
        p.x_in = x0;
        const size_t sr = padded(s.d, 32) * 4 + (size_t)(s.d / 32) * 4 + 32 * 4 + 16;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(p.n_cta);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = sr;
        cfg.stream = st;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, chain_r_kernel, p, 1, zr);
        if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step_chain: router launch: %s", cudaGetErrorString(e));
        CP q = b;
        q.launch_id = lid++;
        q.topk_z = zr;
        q.topk_set = cur;
        q.topk_tgt = 0;
        if (int rc = launch(chain_topk_kernel, q, 1, 32, 0, true, st, "router top-K")) return rc;
        first = false;
    }
    for (int N = 0; N < s.depth; N++) {
        CP p = b;
        p.N = N;
        p.L = layer_of(sd, N, s);
        p.head = head_runs(s, N) ? 1 : 0;
        p.route_late = N == 0 && s.own0;
        p.x_is_out = N > 0;
        p.z = z + (size_t)N * s.E;
        p.smap = sd->slot_map && !p.route_late ? sd->slot_map + (size_t)N * s.K : nullptr;
        p.debug_unset_wait = N == 0 ? sd->debug_unset_wait : 0;
        p.launch_id = lid++;
        CX x{};
        x.C = C;
        x.rmax = rmax;
        x.prefetch = g_prefetch;
        x.base = N <= 1 ? x0 : outs + (size_t)(N - 2) * s.d;
        x.part_in = N == 0 ? nullptr : part + (size_t)(N - 1) * ps;
        x.part = part + (size_t)N * ps;
        x.x_out = N >= 1 ? outs + (size_t)(N - 1) * s.d : nullptr;
        if (sd->layer_ready && sd->layer_ready[N]) {
            const cudaError_t e = cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(sd->layer_ready[N]), 0);
            if (e != cudaSuccess)
                return fail(MOE_ECUDA, "decode_step_chain: wait for layer %d: %s", N, cudaGetErrorString(e));
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((s.S + p.head) * C);
        cfg.blockDim = dim3(kCThreads);
        cfg.dynamicSmemBytes = Lo.total;
        cfg.stream = st;
        cudaLaunchAttribute at[2];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = C;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = first ? 1 : 2;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, chain_c_kernel<BITS>, p, x);
        if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step_chain: layer launch: %s", cudaGetErrorString(e));
        first = false;
    }
    {
        // the last layer's outputs onto its residual
        CP p = b;
        p.out = out;
        p.launch_id = lid++;
        CX x{};
        x.base = s.depth == 1 ? x0 : outs + (size_t)(s.depth - 2) * s.d;
        x.part_in = part + (size_t)(s.depth - 1) * ps;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((s.d / 4 + 255) / 256);
        cfg.blockDim = dim3(256);
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, chain_fin_kernel, p, x);
        if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step_chain: output launch: %s", cudaGetErrorString(e));
    }
    const int n_heads = head_runs(s, s.depth - 1) ? s.depth : s.depth - 1;
    if (n_heads > 0) {
        CP q = b;
        q.launch_id = lid++;
        q.topk_set = nxt;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((n_heads + kRankWarps - 1) / kRankWarps);
        cfg.blockDim = dim3(kRankWarps * 32);
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, chain_rank_kernel, q, (const float *)z, n_heads);
        if (e != cudaSuccess) return fail(MOE_ECUDA, "decode_step_chain: ranking launch: %s", cudaGetErrorString(e));
    }
    return MOE_OK;
}


// ---------------------------------------------------------------- graph cache
// A call's launches depend only on the descriptor's values, the call's
// pointers, t mod 3, the device and the form chosen -- not on the contents
// of any buffer.  So a call not made under stream capture is recorded once
// into a CUDA graph (captured on an internal stream of the calling thread,
// in thread-local capture mode) and later calls with the same key launch
// that graph on the caller's stream: one host launch instead of two per
// layer.  Calls with ready events or debug hooks are never cached.  At most
// g_cache_max graphs (least recently used out first; 0 disables).
static std::mutex g_gmu;
static int g_cache_max = 16;
struct GEntry {
    std::vector<uint8_t> key;
    cudaGraphExec_t exec;      // null: the call could not be captured (run directly)
    unsigned long long used;
};
static std::vector<GEntry> g_graphs;
static unsigned long long g_tick = 0;

template <class T>
static void put(std::vector<uint8_t> &k, const T &v) {
    const uint8_t *b = reinterpret_cast<const uint8_t *>(&v);
    k.insert(k.end(), b, b + sizeof(T));
}

static std::vector<uint8_t> step_key(const moe_stack_desc *sd, const Shapes &s, const float *x0,
                                     const float *out, const int32_t *ridx, const float *rw,
                                     const float *rmg, int t, const void *ws) {
    std::vector<uint8_t> k;
    k.reserve(256 + 256 * (size_t)s.n_res);
    int dev = 0;
    cudaGetDevice(&dev);
    put(k, dev);
    put(k, g_variant);
    put(k, g_prefetch);
    put(k, t % 3);
    put(k, x0);
    put(k, out);
    put(k, ridx);
    put(k, rw);
    put(k, rmg);
    put(k, ws);
    const int sh[] = {s.d, s.F, s.E, s.K, s.H, s.S, s.bits, s.depth, s.n_res, s.self_predict, s.own0,
                      s.rd_routed, s.rd_shared, s.heads ? 1 : 0, sd->free_sms};
    put(k, sh);
    put(k, sd->experts[0].expert_stride);
    put(k, sd->timeout_ns);
    put(k, sd->slot_map);
    for (int i = 0; i < s.n_res; i++) {
        const CLayer L = layer_of(sd, i, s);
        const void *ptrs[] = {L.pool, L.shared, L.la_d, L.lb_d, L.sa[0], L.sa[1], L.sa[2], L.sb[0], L.sb[1],
                              L.sb[2], L.router, L.fc1x, L.fc2, L.lx, L.fc1_tab, L.b1, L.b2, L.l_tab, L.bl};
        put(k, ptrs);
        const size_t strides[] = {L.la_ds, L.lb_ds};
        put(k, strides);
        const int ranks[] = {L.r_d, L.sr[0], L.sr[1], L.sr[2]};
        put(k, ranks);
        const float scales[] = {L.s_d, L.ss[0], L.ss[1], L.ss[2]};
        put(k, scales);
    }
    return k;
}

static cudaStream_t capture_stream() {
    static thread_local cudaStream_t caps[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return nullptr;
    if (!caps[dev] && cudaStreamCreateWithFlags(&caps[dev], cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        caps[dev] = nullptr;
    }
    return caps[dev];
}

template <class Direct>
static int run_cached(const std::vector<uint8_t> &key, Direct direct, cudaStream_t st) {
    {
        std::lock_guard<std::mutex> g(g_gmu);
        for (GEntry &e : g_graphs)
            if (e.key == key) {
                e.used = ++g_tick;
                if (!e.exec) return direct(st);
                const cudaError_t r = cudaGraphLaunch(e.exec, st);
                if (r != cudaSuccess) return fail(MOE_ECUDA, "decode_step_chain: graph launch: %s", cudaGetErrorString(r));
                return MOE_OK;
            }
    }
    // a new key: this call runs directly (which also sets the kernels'
    // attributes up), then its launches are recorded for the next calls
    if (int rc = direct(st)) return rc;
    cudaGraphExec_t exec = nullptr;
    cudaStream_t cap = capture_stream();
    if (cap && cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
        const int rc = direct(cap);
        cudaGraph_t graph = nullptr;
        const cudaError_t ec = cudaStreamEndCapture(cap, &graph);
        if (rc == MOE_OK && ec == cudaSuccess && graph && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
            exec = nullptr;
        if (graph) cudaGraphDestroy(graph);
    }
    cudaGetLastError();       // a failed capture leaves no sticky error (the key then runs directly)
    {
        std::lock_guard<std::mutex> g(g_gmu);
        if ((int)g_graphs.size() >= g_cache_max) {
            size_t old = 0;
            for (size_t i = 1; i < g_graphs.size(); i++)
                if (g_graphs[i].used < g_graphs[old].used) old = i;
            if (g_graphs[old].exec) cudaGraphExecDestroy(g_graphs[old].exec);   // freed when it completes
            g_graphs.erase(g_graphs.begin() + (long)old);
        }
        g_graphs.push_back(GEntry{key, exec, ++g_tick});
    }
    return MOE_OK;
}

static void clear_cache() {
    std::lock_guard<std::mutex> g(g_gmu);
    for (GEntry &e : g_graphs)
        if (e.exec) cudaGraphExecDestroy(e.exec);
    g_graphs.clear();
}

}  // namespace chain
}  // namespace moe

using namespace moe;

extern "C" size_t moe_decode_step_chain_workspace_bytes(const moe_stack_desc *sd) {
    if (check_decode_stack(sd) != MOE_OK) return 0;
    const chain::Shapes s = chain::shapes_of(sd);
    const int sms = chain::chain_ctas(sd);
    return std::max(chain::ws_layout(s.d, s.F, s.E, s.H, s.S, s.depth, sms > 0 ? sms : 256).total,
                    chain::cws_layout(s.d, s.E, s.S, s.depth).total);
}

extern "C" int moe_decode_step_chain_variant(int variant, int prefetch_l2) {
    if (variant < 0 || variant > 2) return fail(MOE_EINVAL, "decode_step_chain_variant: variant %d", variant);
    chain::g_variant = variant;
    chain::g_prefetch = prefetch_l2 ? 1 : 0;
    return MOE_OK;
}

extern "C" int moe_decode_step_chain_info(const moe_stack_desc *sd, moe_chain_info *info) {
    if (info == nullptr) return fail(MOE_EINVAL, "decode_step_chain_info: NULL info");
    if (int rc = check_decode_stack(sd)) return rc;
    const chain::Shapes s = chain::shapes_of(sd);
    const int n = chain::chain_ctas(sd);
    if (n <= 0) return fail(MOE_ECUDA, "decode_step_chain_info: no device");
    return s.bits == 4 ? chain::residency<4>(s, n, info) : chain::residency<2>(s, n, info);
}

extern "C" int moe_decode_step_chain(const moe_stack_desc *sd, const float *x0, float *out,
                                     int32_t *route_idx, float *route_w, float *route_margin, int t,
                                     void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (int rc = check_decode_stack(sd)) return rc;
    if (t < 1)
        return fail(MOE_EINVAL, "decode_step_chain: t=%d (step 0 routes every layer with its own "
                                "router; run it with the per-call functions)", t);
    if (!x0 || !out || !route_idx || !route_w || !route_margin || !ws)
        return fail(MOE_EINVAL, "decode_step_chain: NULL pointer");
    const size_t need = moe_decode_step_chain_workspace_bytes(sd);
    if (ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) % 256))
        return fail(MOE_ENOSPACE, "decode_step_chain: workspace %zu bytes, need %zu (256-aligned)",
                    ws_bytes, need);
    const chain::Shapes s = chain::shapes_of(sd);
    if (s.d % 256 && s.bits == 2)
        return fail(MOE_EUNSUPPORTED, "decode_step_chain: 2-bit needs d a multiple of 256");
    const int n = chain::chain_ctas(sd);
    if (n <= 0) return fail(MOE_ECUDA, "decode_step_chain: no device");
    if ((long long)s.S * s.F > (long long)chain::kMaxHPass * chain::kThreads * 4 ||
        (s.d + n - 1) / n > chain::kThreads || (s.E + n - 1) / n > chain::kThreads - 32)
        return fail(MOE_EUNSUPPORTED, "decode_step_chain: slots x F = %d x %d (or d, E) too large "
                                      "for %d SMs", s.S, s.F, n);
    uint8_t *w = static_cast<uint8_t *>(ws);
    if (chain::g_variant == 2) {
        const char *why = "";
        if (!(s.bits == 4 ? chain::c_fits<4>(sd, s, &why) : chain::c_fits<2>(sd, s, &why)))
            return fail(MOE_EUNSUPPORTED, "decode_step_chain: cluster variant: %s", why);
    }
    const int variant = chain::g_variant;
    auto direct = [&](cudaStream_t st) {
        if (variant == 2)
            return s.bits == 4 ? chain::run_c<4>(sd, s, x0, out, route_idx, route_w, route_margin, t, w, st)
                               : chain::run_c<2>(sd, s, x0, out, route_idx, route_w, route_margin, t, w, st);
        return s.bits == 4 ? chain::run<4>(sd, s, x0, out, route_idx, route_w, route_margin, t, w, st)
                           : chain::run<2>(sd, s, x0, out, route_idx, route_w, route_margin, t, w, st);
    };
    if (chain::g_cache_max > 0 && !sd->layer_ready && !sd->debug_unset_wait && !sd->debug_trace) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone)
            return chain::run_cached(chain::step_key(sd, s, x0, out, route_idx, route_w, route_margin, t, ws),
                                     direct, stream);
        cudaGetLastError();
    }
    return direct(stream);
}

extern "C" int moe_decode_step_chain_cache(int max_graphs) {
    if (max_graphs < 0 || max_graphs > 1024)
        return fail(MOE_EINVAL, "decode_step_chain_cache: %d graphs (0 .. 1024)", max_graphs);
    chain::clear_cache();
    chain::g_cache_max = max_graphs;
    return MOE_OK;
}
