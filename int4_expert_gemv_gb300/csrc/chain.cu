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
#include <cfloat>
#include <cstring>

#include "internal.h"

namespace moe {
namespace chain {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxR = 32;                 // LoRA rank bound
constexpr int kMaxK = 16;
constexpr uint64_t kCopyWaitNs = 1000000000ull;

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
    const float *topk_z;      // logits to rank in A (head N-1's), or null
    int topk_set, topk_tgt;   // where the route goes
    int32_t *err;
};

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ uint32_t saddr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;");
}

__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(saddr(dst)), "l"(src), "r"(bytes), "r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ void bar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void bar_expect(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)),
                 "r"(bytes) : "memory");
}

// Bounded wait for phase 0 of bar (this kernel's one use of it).
__device__ __forceinline__ bool bar_wait(uint64_t *bar, int32_t *err) {
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
        else if (now - t0 > kCopyWaitNs) {
            atomicExch(err, MOE_ETIMEOUT);
            return false;
        }
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
// conflicts).  Also the per-chunk sums.  Returns the sum of squares (every
// thread).
__device__ __forceinline__ float stage_vec(const float *src, int n, int vals, float *dst,
                                           float *sums, float *red) {
    float ss = 0.0f;
    for (int i = threadIdx.x; i < n / 4; i += blockDim.x) {      // n and vals: multiples of 4
        const float4 v = reinterpret_cast<const float4 *>(src)[i];
        const int c = (4 * i) / vals, j = 4 * i - c * vals;
        float *d = dst + c * (vals + 1) + j;
        d[0] = v.x;
        d[1] = v.y;
        d[2] = v.z;
        d[3] = v.w;
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
    __syncthreads();
    for (int c = threadIdx.x; c < n / vals; c += blockDim.x) {
        float a = 0.0f;
        for (int j = 0; j < vals; j++) a += dst[c * (vals + 1) + j];
        sums[c] = a;
    }
    return block_sum(ss, red);
}

__host__ __device__ inline size_t padded(int n, int vals) { return (size_t)(n / vals) * (vals + 1); }

__device__ __forceinline__ float half_at(const uint16_t *p, size_t i) { return half_f(p[i]); }

// Ranks E <= 1024 logits (value desc, index asc; NaN last) in one warp:
// route of layer tgt in set `set` (indices, softmax weights over the kept K,
// margin z_(K) - z_(K+1)).  Lane l holds logits l, l + 32, ...
__device__ void warp_route(const float *z, int E, int K, int32_t *ridx, float *rw, float *rmargin,
                           int set, int depth, int tgt) {
    const int lane = threadIdx.x & 31;
    float vals[32];
#pragma unroll
    for (int i = 0; i < 32; i++) {
        const int e = lane + 32 * i;
        const float v = e < E ? z[e] : -INFINITY;
        vals[i] = v == v ? v : -INFINITY;
    }
    float topv[kMaxK + 1];
    int topi[kMaxK + 1];
    const int rounds = K < E ? K + 1 : K;
    uint32_t taken = 0;
    for (int k = 0; k < rounds; k++) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < 32; i++) {
            const int e = lane + 32 * i;
            if (e < E && !(taken >> i & 1u) && (vals[i] > bv || (vals[i] == bv && e < bi))) {
                bv = vals[i];
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
        if (bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    if (lane == 0) {
        float sum = 0.0f;
        for (int k = 0; k < K; k++) sum += expf(topv[k] - topv[0]);
        for (int k = 0; k < K; k++) {
            ridx[((size_t)set * depth + tgt) * K + k] = topi[k];
            rw[((size_t)set * depth + tgt) * K + k] = expf(topv[k] - topv[0]) / sum;
        }
        rmargin[(size_t)set * depth + tgt] = K < E ? topv[K - 1] - topv[K] : INFINITY;
    }
}

// ---------------------------------------------------------------- A work split
// Units: the gate/up row pairs of every slot (slot-major, P bytes each), then
// (if the head runs) the fc1 rows and the l rows (R bytes each).  CTA c takes
// the units that start in its byte range [c T / n, (c + 1) T / n).
struct ASplit {
    long long gu_units, total, P, R;
    __host__ __device__ long long start(long long u) const {
        return u < gu_units ? u * P : gu_units * P + (u - gu_units) * R;
    }
    __host__ __device__ long long first_at(long long b) const {   // first unit starting at >= b
        if (b <= gu_units * P) return (b + P - 1) / P;
        return gu_units + (b - gu_units * P + R - 1) / R;
    }
    __host__ __device__ void range(int c, int n, long long &u0, long long &u1) const {
        u0 = first_at(total * c / n);
        u1 = first_at(total * (c + 1) / n);
    }
};

__host__ __device__ inline ASplit a_split(int S, int F, int H, int E, int head, uint32_t rec_d,
                                          uint32_t rec_dh) {
    ASplit s;
    s.gu_units = (long long)S * F;
    s.P = 2LL * rec_d;
    s.R = rec_dh;
    s.total = s.gu_units * s.P + (head ? (long long)(H + E) * s.R : 0);
    return s;
}

__device__ __forceinline__ const uint8_t *slot_blob(const CP &p, const int32_t *route, int s,
                                                    bool &bad) {
    if (s >= p.K) return p.L.shared;
    const int e = route[s];
    if ((unsigned)e >= (unsigned)p.E) {
        bad = true;
        return p.L.pool;
    }
    return p.L.pool + (size_t)e * p.stride;
}

// ---------------------------------------------------------------- kernel A
template <int BITS>
__global__ void __launch_bounds__(kThreads, 1) chain_a_kernel(const __grid_constant__ CP p) {
    constexpr int VALS = 128 / BITS;
    extern __shared__ __align__(128) uint8_t sm[];
    const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ASplit sp = a_split(p.S, p.F, p.H, p.E, p.head, p.rec_d, p.rec_dh);
    long long u0, u1;
    sp.range(c, p.n_cta, u0, u1);
    const uint32_t wbytes = (uint32_t)(sp.start(u1) - sp.start(u0));
    // shared memory: weights, x, chunk sums of x (4-bit chunks for the head),
    // table sums of the head rows, LoRA v, misc
    uint8_t *wts = sm;
    size_t off = (wbytes + 127) / 128 * 128;
    float *x = reinterpret_cast<float *>(sm + off);          // padded per BITS chunk
    off += padded(p.d, VALS) * 4;
    float *xs = reinterpret_cast<float *>(sm + off);          // BITS chunks
    off += (size_t)(p.d / VALS) * 4;
    float *x4 = BITS == 4 ? x : reinterpret_cast<float *>(sm + off);   // padded per 4-bit chunk (head)
    if (BITS != 4) off += padded(p.d, 32) * 4;
    float *xs4 = reinterpret_cast<float *>(sm + off);         // 4-bit chunks (head rows)
    off += (size_t)(p.d / 32) * 4;
    const long long h0 = u0 > sp.gu_units ? u0 : sp.gu_units;  // first head unit
    const int nh = u1 > h0 ? (int)(u1 - h0) : 0;
    float *tsum = reinterpret_cast<float *>(sm + off);
    off += (size_t)(nh + 1) * 4;
    float *tterm = reinterpret_cast<float *>(sm + off);       // [nh][2K + 1] table terms
    off += (size_t)(nh * (2 * p.K + 1) + 1) * 4;
    float *vx = reinterpret_cast<float *>(sm + off);          // gate/up LoRA A x
    off += 2 * kMaxR * 4;
    float *vwarp = reinterpret_cast<float *>(sm + off);       // per-warp sums of the partials
    off += kWarps * 32 * 4;
    float *red = reinterpret_cast<float *>(sm + off);
    off += 32 * 4;
    int32_t *route = reinterpret_cast<int32_t *>(sm + off);
    off += (kMaxK + 1) * 4;
    off = (off + 7) / 8 * 8;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + off);

    const int32_t *rcur = p.ridx + ((size_t)p.cur * p.depth + p.N) * p.K;
    const int32_t *rprv = p.ridx + ((size_t)p.prv * p.depth + p.N) * p.K;
    auto issue = [&]() {
        // the unit range's segments: per slot a run of pairs, fc1 rows, l rows
        if (threadIdx.x == 0) {
            bool bad = false;
            bar_expect(bar, wbytes);
            uint32_t at = 0;
            long long u = u0;
            while (u < u1) {
                const uint8_t *src;
                long long n;
                if (u < sp.gu_units) {
                    const int s = (int)(u / p.F), f = (int)(u % p.F);
                    n = (long long)min((long long)(p.F - f), u1 - u);
                    src = slot_blob(p, route, s, bad) + p.gu_off + (size_t)f * sp.P;
                    n *= sp.P;
                } else {
                    const long long r = u - sp.gu_units;
                    if (r < p.H) {
                        const long long m = min((long long)p.H - r, u1 - u);
                        src = p.L.fc1x + (size_t)r * sp.R;
                        n = m * sp.R;
                    } else {
                        const long long m = u1 - u;
                        src = p.L.lx + (size_t)(r - p.H) * sp.R;
                        n = m * sp.R;
                    }
                }
                bulk_copy(wts + at, src, (uint32_t)n, bar);
                at += (uint32_t)n;
                u = sp.first_at(sp.start(u) + n);
            }
            if (bad) atomicExch(p.err, MOE_EINVAL);
        }
    };
    if (threadIdx.x == 0) bar_init(bar);
    if (threadIdx.x < p.K && !p.route_late) route[threadIdx.x] = rcur[threadIdx.x];
    __syncthreads();
    if (!p.route_late) issue();
    // table sums of this CTA's head rows (the routes of layer N at t and t - 1)
    auto tables = [&]() {
        // item (row i, term j): j < K the current route's table row, then the
        // previous route's, then the bias -- one load each, in parallel; row
        // i's terms are then summed in that order
        const int nt = 2 * p.K + 1;
        for (int it = threadIdx.x; it < nh * nt; it += blockDim.x) {
            const int i = it / nt, j = it - i * nt;
            const long long r = h0 - sp.gu_units + i;
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
    grid_launch_dependents();
    grid_wait();
    if (p.route_late) {
        if (threadIdx.x < p.K) route[threadIdx.x] = rcur[threadIdx.x];
        __syncthreads();
        issue();
        tables();
    }
    // head N-1's route (the next token's route of layer N)
    if (c == 0 && warp == kWarps - 1 && p.topk_z)
        warp_route(p.topk_z, p.E, p.K, p.ridx, p.rw, p.rmargin, p.topk_set, p.depth, p.topk_tgt);
    // x and its chunk sums; 1/rms when x is an out
    const float ss = stage_vec(p.x_in, p.d, VALS, x, xs, red);
    if (BITS == 4) {
        for (int ch = threadIdx.x; ch < p.d / 32; ch += blockDim.x) xs4[ch] = xs[ch];
    } else {
        stage_vec(p.x_in, p.d, 32, x4, xs4, red);
    }
    const float inv = p.x_is_out ? 1.0f / sqrtf(ss / p.d + 1e-6f) : 1.0f;
    // the shared expert's gate/up LoRA: A x from the previous layer's partials
    const int gs = p.S - 1;
    const bool lora_here = p.gu_lora && u0 < (long long)(gs + 1) * p.F && u1 > (long long)gs * p.F;
    if (lora_here) {
        // warp w sums the partials of CTAs w, w + kWarps, ... (loads first,
        // then the sum in order), then warp 0 the warps' sums
        constexpr int kPer = 16;                    // up to 256 CTAs
        float v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; j++) {
            const int q = warp + j * kWarps;
            v[j] = q < p.n_cta ? p.vp[(size_t)q * 2 * kMaxR + lane] : 0.0f;
        }
        float a = 0.0f;
#pragma unroll
        for (int j = 0; j < kPer; j++) a += v[j];
        vwarp[warp * 32 + lane] = a;
    }
    __syncthreads();
    if (lora_here && warp == 0) {
        float a = 0.0f;
        for (int w = 0; w < kWarps; w++) a += vwarp[w * 32 + lane];
        vx[lane] = a * inv;
    }
    __syncthreads();
    if (!bar_wait(bar, p.err)) return;
    // units: warp w takes u0 + w, u0 + w + kWarps, ...
    for (long long u = u0 + warp; u < u1; u += kWarps) {
        const uint8_t *rec = wts + (sp.start(u) - sp.start(u0));
        if (u < sp.gu_units) {
            const int s = (int)(u / p.F), f = (int)(u % p.F);
            float gg = warp_sum(rec_dot<BITS>(rec, p.d, x, xs, lane), 32) * inv;
            float uu = warp_sum(rec_dot<BITS>(rec + p.rec_d, p.d, x, xs, lane), 32) * inv;
            if (s == gs && p.gu_lora) {
                const int rg = p.L.sr[0], ru = p.L.sr[1];
                float a = lane < rg ? half_at(p.L.sb[0], (size_t)f * rg + lane) * vx[lane] : 0.0f;
                float b = lane < ru ? half_at(p.L.sb[1], (size_t)f * ru + lane) * vx[rg + lane] : 0.0f;
                gg += p.L.ss[0] * warp_sum(a, 32);
                uu += p.L.ss[1] * warp_sum(b, 32);
            }
            if (lane == 0) p.h[(size_t)s * p.F + f] = silu_f(gg) * uu;
        } else {
            const long long r = u - sp.gu_units;
            const float a = warp_sum(rec_dot<4>(rec, p.d, x4, xs4, lane), 32) * inv + tsum[u - h0];
            if (lane == 0) {
                if (r < p.H) p.g[r] = gelu_erf_f(a);
                else if (p.H > 0) p.zl[r - p.H] = a;
                else p.z[r - p.H] = a;
            }
        }
    }
}

// ---------------------------------------------------------------- kernel B
// Output rows [o0, o1) and logit rows [e0, e1) of CTA c (even splits).
template <int BITS>
__global__ void __launch_bounds__(kThreads, 1) chain_b_kernel(const __grid_constant__ CP p) {
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
    float *hs = reinterpret_cast<float *>(sm + off);          // [S][F] padded per chunk
    off += padded(p.S * p.F, VALS) * 4;
    float *hsum = reinterpret_cast<float *>(sm + off);        // [S][F / VALS]
    off += (size_t)p.S * (p.F / VALS) * 4;
    float *gs = reinterpret_cast<float *>(sm + off);          // [H] padded per 4-bit chunk
    off += (p.H > 0 ? padded(p.H, 32) : 1) * 4;
    float *gsum = reinterpret_cast<float *>(sm + off);        // [H / 32]
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
    float *wk = reinterpret_cast<float *>(sm + off);          // combine weights
    off += (kMaxK + 1) * 4;
    int32_t *route = reinterpret_cast<int32_t *>(sm + off);
    off += (kMaxK + 1) * 4;
    float *red = reinterpret_cast<float *>(sm + off);
    off += 32 * 4;
    off = (off + 7) / 8 * 8;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + off);

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
    // the next layer's gate/up A columns of this CTA's rows (static data)
    const int r2n = p.vp_next ? p.nr[0] + p.nr[1] : 0;
    for (int it = threadIdx.x; it < r2n * no; it += blockDim.x) {
        const int k = it / no, i = it - k * no;
        const uint16_t *A = k < p.nr[0] ? p.nA[0] + (size_t)k * p.d : p.nA[1] + (size_t)(k - p.nr[0]) * p.d;
        anext[k * no + i] = half_at(A, o0 + i);
    }
    grid_launch_dependents();
    grid_wait();
    if (p.route_late) {
        if (threadIdx.x < p.K) {
            route[threadIdx.x] = rcur[threadIdx.x];
            wk[threadIdx.x] = wcur[threadIdx.x];
        }
        __syncthreads();
        issue();
    }
    // h of every slot with its chunk sums; g (head fc2 input) with 4-bit chunk sums
    stage_vec(p.h, p.S * p.F, VALS, hs, hsum, red);
    if (p.head && p.H > 0) stage_vec(p.g, p.H, 32, gs, gsum, red);
    __syncthreads();
    if (!bar_wait(bar, p.err)) return;
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
            for (int f = lane; f < p.F; f += 32) a = fmaf(half_f(A[f]), hrow[f + f / VALS], a);
            a = warp_sum(a, 32);
            if (lane == 0) vd[s * kMaxR + k] = (!shared && (unsigned)route[s] >= (unsigned)p.E) ? 0.0f : a;
        }
    }
    __syncthreads();
    // out rows: warp per row; lanes over the (slot, chunk) pairs
    const int cps = p.F / VALS, npair = p.S * cps;
    const size_t cb = code_bytes(p.F, BITS);
    for (int i = warp; i < no; i += kWarps) {
        const int o = o0 + i;
        float acc = 0.0f;
        for (int q = lane; q < npair; q += 32) {
            const int s = q / cps, ch = q - s * cps;
            const uint8_t *rec = wts + (size_t)s * dbytes + (size_t)i * p.rec_F;
            const uint4 w4 = *reinterpret_cast<const uint4 *>(rec + (size_t)kChunk * ch);
            const float2 sb = sb_f(*reinterpret_cast<const uint32_t *>(rec + cb + 4 * ((ch * VALS) / kGroup)));
            const float y = fmaf(sb.x, chunk_dot<BITS>(w4, hs + (size_t)(s * cps + ch) * (VALS + 1)),
                                 sb.y * hsum[s * cps + ch]);
            acc = fmaf(s < p.K ? wk[s] : 1.0f, y, acc);
        }
        // down LoRA: lane k < r of each adapter slot
        for (int s = 0; s < p.S; s++) {
            const bool shared = s >= p.K;
            const int r = shared ? p.L.sr[2] : p.L.r_d;
            if (r == 0 || lane >= r) continue;
            const int e = shared ? 0 : route[s];
            if (!shared && (unsigned)e >= (unsigned)p.E) continue;
            const uint16_t *B = shared ? p.L.sb[2] : p.L.lb_d + (size_t)e * p.L.lb_ds;
            const float sc = shared ? p.L.ss[2] : p.L.s_d;
            acc = fmaf((shared ? 1.0f : wk[s]) * sc, half_at(B, (size_t)o * r + lane) * vd[s * kMaxR + lane], acc);
        }
        acc = warp_sum(acc, 32);
        if (lane == 0) {
            const float v = p.x_in[o] + acc;
            outs[i] = v;
            p.out[o] = v;
        }
    }
    // head N's fc2 rows: z = fc2 g + b2 + l f
    for (int i = warp; i < ne; i += kWarps) {
        const int e = e0 + i;
        float a = 0.0f;
        if (p.H > 0) a = warp_sum(rec_dot<4>(wts + (size_t)p.S * dbytes + (size_t)i * p.rec_H, p.H, gs, gsum, lane), 32);
        if (lane == 0) p.z[e] = a + (p.L.b2 ? half_at(p.L.b2, e) : 0.0f) + p.zl[e];
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
    grid_wait();
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

// One warp: the route of layer tgt from logits z.
__global__ void __launch_bounds__(32) chain_topk_kernel(const __grid_constant__ CP p) {
    grid_wait();
    warp_route(p.topk_z, p.E, p.K, p.ridx, p.rw, p.rmargin, p.topk_set, p.depth, p.topk_tgt);
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
            long long u0, u1;
            sp.range(c, n_cta, u0, u1);
            const size_t wb = (size_t)(sp.start(u1) - sp.start(u0));
            const long long h0 = u0 > sp.gu_units ? u0 : sp.gu_units;
            const size_t nh = u1 > h0 ? (size_t)(u1 - h0) : 0;
            size_t need = (wb + 127) / 128 * 128 + padded(s.d, VALS) * 4 + (size_t)(s.d / VALS) * 4 +
                          (s.bits != 4 ? padded(s.d, 32) * 4 : 0) +
                          (size_t)(s.d / 32) * 4 + (nh + 1) * 4 + (nh * (2 * s.K + 1) + 1) * 4 +
                          2 * kMaxR * 4 + kWarps * 32 * 4 + 32 * 4 + (kMaxK + 1) * 4 + 16;
            if (need > a) a = need;
        }
    }
    const int no = (s.d + n_cta - 1) / n_cta, ne = (s.E + n_cta - 1) / n_cta;
    *sa = a;
    *sb = ((size_t)s.S * no * rec_F + (size_t)ne * rec_H + 127) / 128 * 128 + padded(s.S * s.F, VALS) * 4 +
          (size_t)s.S * (s.F / VALS) * 4 + (s.H > 0 ? padded(s.H, 32) : 1) * 4 +
          (size_t)(s.H > 0 ? s.H / 32 : 1) * 4 + (size_t)s.S * kMaxR * 4 +
          ((size_t)(s.K * s.rd_routed + s.rd_shared) * s.F * 2 + 15) / 16 * 16 +
          (size_t)2 * kMaxR * (no + 1) * 4 + (size_t)(no + 1) * 4 + 2 * (kMaxK + 1) * 4 + 32 * 4 + 16;
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

template <int BITS>
static int run(const moe_stack_desc *sd, const Shapes &s, const float *x0, float *out,
               int32_t *ridx, float *rw, float *rmargin, int t, uint8_t *ws, cudaStream_t st) {
    const int n_cta = sms_of_device();
    const Ws W = ws_layout(s.d, s.F, s.E, s.H, s.S, s.depth, n_cta);
    size_t sa, sb;
    smem_need(s, n_cta, &sa, &sb);
    int dev = 0, smem_max = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (sa > (size_t)smem_max || sb > (size_t)smem_max)
        return fail(MOE_EUNSUPPORTED, "decode_step_chain: %zu / %zu bytes of shared memory (at most %d)",
                    sa, sb, smem_max);
    const size_t sr = padded(s.d, 32) * 4 + (size_t)(s.d / 32) * 4 + 32 * 4 + 16;
    if (cudaFuncSetAttribute(chain_a_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sa) != cudaSuccess ||
        cudaFuncSetAttribute(chain_b_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sb) != cudaSuccess)
        return fail(MOE_ECUDA, "decode_step_chain: shared-memory attribute");
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
        // A ranks head N - 1's logits: the next token's route of layer N
        if (N >= 1 && head_runs(s, N - 1)) {
            p.topk_z = z + (size_t)(N - 1) * s.E;
            p.topk_set = nxt;
            p.topk_tgt = N;
        }
        if (int rc = launch(chain_a_kernel<BITS>, p, n_cta, kThreads, sa, !first, st, "A")) return rc;
        first = false;
        p.topk_z = nullptr;
        if (int rc = launch(chain_b_kernel<BITS>, p, n_cta, kThreads, sb, true, st, "B")) return rc;
    }
    // the last head (a single self-predicting layer: its own next route)
    if (head_runs(s, s.depth - 1)) {
        CP q = b;
        q.topk_z = z + (size_t)(s.depth - 1) * s.E;
        q.topk_set = nxt;
        q.topk_tgt = 0;
        if (int rc = launch(chain_topk_kernel, q, 1, 32, 0, true, st, "last head top-K")) return rc;
    }
    return MOE_OK;
}

}  // namespace chain
}  // namespace moe

using namespace moe;

extern "C" size_t moe_decode_step_chain_workspace_bytes(const moe_stack_desc *sd) {
    if (check_decode_stack(sd) != MOE_OK) return 0;
    const chain::Shapes s = chain::shapes_of(sd);
    const int sms = chain::sms_of_device();
    return chain::ws_layout(s.d, s.F, s.E, s.H, s.S, s.depth, sms > 0 ? sms : 256).total;
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
    uint8_t *w = static_cast<uint8_t *>(ws);
    return s.bits == 4 ? chain::run<4>(sd, s, x0, out, route_idx, route_w, route_margin, t, w, stream)
                       : chain::run<2>(sd, s, x0, out, route_idx, route_w, route_margin, t, w, stream);
}
