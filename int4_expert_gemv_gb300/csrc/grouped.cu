// grouped.cu -- batched / prefill expert FFN (T > 1 tokens, bf16 activations).
//
// The tokens' (token, slot) entries are sorted by expert (a stable counting
// sort: histogram, exclusive scan, scatter in token order), so each routed
// expert's weights are read once for all the tokens routed to it and the
// shared expert's once for all T tokens ("tokens sorted/grouped by expert":
// the batched configuration of xyznot.com/es/paper/2609.18063's workload
// list; the layer math is the decode layer's, per token).  Each expert's
// token group then runs as two GEMMs of the persistent tensor-core engine
// (gemm_pipe.cuh):
//
//   gate/up:  [2F records] x [d] . [d] x [n_e tokens]  -> h = silu(g) * u
//   down:     [d records]  x [F] . [F] x [n_e tokens]  -> y_slots
//
// with SwiGLU and the LoRA terms in the epilogues.  h is rounded to bf16
// before the down GEMM (the batched path's bf16 activations), as the oracle
// does.  Groups: g < E the routed experts, g = E the shared expert.
#include <cuda_bf16.h>

#include "gemm_pipe.cuh"
#include "gemm_umma.cuh"
#include "internal.h"

namespace moe {
namespace grouped {

using namespace pipe;

// ---------------------------------------------------------------- sort
// counts[e] = entries routed to expert e (e < E); counts[E] = entries with an
// index outside [0, E).  One warp per bucket.
// Whether entry value e falls in bucket b (b = E: outside [0, E)).
__device__ __forceinline__ bool in_bucket(int e, int b, int E) {
    return b < E ? e == b : (unsigned)e >= (unsigned)E;
}

constexpr int kSortU = 8;         // entries per lane loaded before they are ranked

__global__ void __launch_bounds__(256) sort_count_kernel(const int32_t *idx, int TK, int E,
                                                         int32_t *counts) {
    const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (b > E) return;
    int n = 0;
    for (int i0 = 0; i0 < TK; i0 += 32 * kSortU) {
        int e[kSortU];
#pragma unroll
        for (int u = 0; u < kSortU; u++) {
            const int i = i0 + 32 * u + lane;
            e[u] = i < TK ? idx[i] : -1;
        }
#pragma unroll
        for (int u = 0; u < kSortU; u++) {
            const bool m = i0 + 32 * u + lane < TK && in_bucket(e[u], b, E);
            n += __popc(__ballot_sync(0xffffffffu, m));
        }
    }
    if (lane == 0) counts[b] = n;
}

// offsets[b] = sum of counts[0..b); perm[offsets[b] + r] = r-th entry (t*K+k,
// in increasing order) of bucket b.  One warp per bucket.
__global__ void __launch_bounds__(256) sort_scatter_kernel(const int32_t *idx, int TK, int E,
                                                           const int32_t *counts,
                                                           int32_t *offsets, int32_t *perm) {
    const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (b > E) return;
    int off = 0;
    for (int j = lane; j < b; j += 32) off += counts[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
    if (lane == 0) {
        offsets[b] = off;
        if (b == E) offsets[E + 1] = off + counts[E];
    }
    int rank = 0;
    const uint32_t below = (1u << lane) - 1u;
    for (int i0 = 0; i0 < TK; i0 += 32 * kSortU) {
        int e[kSortU];
#pragma unroll
        for (int u = 0; u < kSortU; u++) {
            const int i = i0 + 32 * u + lane;
            e[u] = i < TK ? idx[i] : -1;
        }
#pragma unroll
        for (int u = 0; u < kSortU; u++) {
            const int i = i0 + 32 * u + lane;
            const bool m = i < TK && in_bucket(e[u], b, E);
            const uint32_t mask = __ballot_sync(0xffffffffu, m);
            if (m) perm[off + rank + __popc(mask & below)] = i;
            rank += __popc(mask);
        }
    }
}

// Slots whose expert index is outside [0, E) are never read: their outputs
// are NaN (as on the per-token path).  One warp per invalid entry.
__global__ void __launch_bounds__(256) invalid_fill_kernel(const int32_t *offsets, const int32_t *perm,
                                                           int E, int K, int S, int d, float *y) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int n = offsets[E + 1] - offsets[E];
    for (int i = w; i < n; i += (gridDim.x * blockDim.x) >> 5) {
        const int ent = perm[offsets[E] + i], t = ent / K, k = ent % K;
        float *row = y + ((size_t)t * S + k) * d;
        for (int o = lane; o < d; o += 32) row[o] = __int_as_float(0x7fc00000);
    }
}

// ---------------------------------------------------------------- work items
// A work item is (group g, row block rb, token tile): kRB records of group
// g's gate/up (or down) section against up to kTok of the group's tokens.
// Group g (g < E: routed expert g; g = E: the shared expert) owns items
// off[g] .. off[g+1]-1, row blocks fastest, so the CTAs running consecutive
// items read one token tile (from L2).  One CTA of 1024 threads, two groups
// per thread, a block-wide exclusive scan; both phases' lists in one launch.
__global__ void __launch_bounds__(1024) item_offsets_kernel(const int32_t *counts, int E, int T,
                                                            int G, int rb_gu, int rb_dn,
                                                            int32_t *off_gu, int32_t *off_dn) {
    __shared__ int wsum[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll 1
    for (int which = 0; which < 2; which++) {
        const int rb = which ? rb_dn : rb_gu;
        int32_t *off = which ? off_dn : off_gu;
        int n[2], v = 0;
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const int g = 2 * threadIdx.x + u;
            const int ng = g < G ? (g == E ? T : counts[g]) : 0;
            n[u] = rb * ((ng + kTok - 1) / kTok);
            v += n[u];
        }
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        if (warp == 0) {
            const int w = wsum[lane];
            int wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += y;
            }
            wsum[lane] = wi - w;
        }
        __syncthreads();
        const int ex = wsum[warp] + inc - v;
        const int g = 2 * threadIdx.x;
        if (g < G) off[g] = ex;
        if (g + 1 < G) off[g + 1] = ex + n[0];
        if (g + 1 == G || g + 2 == G) off[G] = ex + v;
        __syncthreads();
    }
}

__device__ __forceinline__ const LoraDev &slot_lora_g(const FfnParams &p, int s, int which) {
    return s < p.K ? p.lora[which] : p.shared_lora[which];
}

// Rows of x in sorted order: xg[pos] = x[token of entry perm[pos]] for the
// routed entries (pos < offsets[E]; invalid entries are never read) and
// xg[TK + t] = x[t] for the shared expert, with their per-group sums.  One
// warp per row; a group of 64 values is 8 lanes' 16-byte pieces.
__global__ void __launch_bounds__(256) gather_x_kernel(FfnParams p, int npos) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (w >= npos) return;
    const int TK = p.T * p.K;
    int t;
    if (w >= TK) t = w - TK;
    else if (w < p.offsets[p.E]) t = p.perm[w] / p.K;
    else return;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.xb + (size_t)t * p.d);
    uint4 *dst = reinterpret_cast<uint4 *>(p.xg + (size_t)w * p.d);
    const int ldg = gsum_ld(p.d), n16 = p.d / 8;
    for (int u0 = 0; u0 < n16; u0 += 32) {     // whole warp per pass (the shuffles)
        const int u = u0 + lane;
        float a = 0.0f;
        if (u < n16) {
            const uint4 v = src[u];
            dst[u] = v;
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
            for (int k = 0; k < 4; k++) a += __bfloat162float(h[k].x) + __bfloat162float(h[k].y);
        }
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        if ((lane & 7) == 0 && u < n16) p.xsum[(size_t)w * ldg + u / 8] = a;
    }
}

// One phase of the expert FFN as a job of the persistent engine: gate/up
// (2F records of d columns against the sorted x) or down (d records of F
// columns against h).  Both read their activations by sorted position: a
// routed group's entries are rows offsets[g] .., the shared expert's rows
// TK + t.  Shared scratch: the item offsets per group (G + 1), then the
// entry offsets (E + 1).
template <bool DOWN>
struct FfnJob {
    Maps maps;
    FfnParams p;
    const int32_t *off;
    int32_t *err;
    int G, RB, cols, nrows, TK;

    // Tensor maps and geometry; returns a moe_status.
    __host__ int make(const FfnParams &pp, const int32_t *item_off) {
        p = pp;
        off = item_off;
        err = p.err;
        G = p.E + (p.shared ? 1 : 0);
        TK = p.T * p.K;
        cols = DOWN ? p.F : p.d;
        nrows = DOWN ? p.d : 2 * p.F;
        RB = (nrows + kRB - 1) / kRB;
        const size_t rec = DOWN ? p.L.down_rec : p.L.gu_rec;
        const size_t sec = DOWN ? p.L.down_off : p.L.gu_off;
        if (int rc = weight_maps(maps, 0, p.pool + sec, rec, nrows, p.E, p.stride, p.bits)) return rc;
        const uint8_t *sh = p.shared ? p.shared + sec : p.pool + sec;
        if (int rc = weight_maps(maps, 1, sh, rec, nrows, 1, 0, p.bits)) return rc;
        const int npos = TK + (p.shared ? p.T : 0);
        return DOWN ? act_maps(maps, p.h16, p.hsum, npos, p.F)
                    : act_maps(maps, p.xg, p.xsum, npos, p.d);
    }

    __device__ void init(int32_t *sm) const {
        for (int g = threadIdx.x; g <= G; g += blockDim.x) sm[g] = off[g];
        for (int g = threadIdx.x; g <= p.E; g += blockDim.x) sm[G + 1 + g] = p.offsets[g];
    }
    __device__ int base(const int32_t *sm, int g) const { return g == p.E ? TK : sm[G + 1 + g]; }
    __device__ int n_items(const int32_t *sm) const { return sm[G]; }
    __device__ Item item(const int32_t *sm, int i) const {
        int lo = 0, hi = G;                     // sm[lo] <= i < sm[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (sm[mid] <= i) lo = mid;
            else hi = mid;
        }
        const int local = i - sm[lo];
        const int tile = local / RB;
        const int n = lo == p.E ? p.T : sm[G + 2 + lo] - sm[G + 1 + lo];
        Item it;
        it.g = lo;
        it.rb = local - tile * RB;
        it.t0 = tile * kTok;
        it.nt = min(kTok, n - it.t0);
        return it;
    }
    __device__ void weights(const Item &it, int &map, int &row, int &blob) const {
        map = it.g == p.E ? 1 : 0;
        row = it.rb * kRB;
        blob = it.g == p.E ? 0 : it.g;
    }
    __device__ int row0(const int32_t *sm, const Item &it) const { return base(sm, it.g) + it.t0; }
    // a routed entry's (token, slot) word: token * K + slot
    __device__ const int32_t *meta(const int32_t *sm, const Item &it) const {
        return it.g == p.E ? nullptr : p.perm + base(sm, it.g) + it.t0;
    }

    __device__ void epilogue(const int32_t *sm, const Item &it, const float *out,
                             const int32_t *ent, int tid, int nthr) const {
        const int nr = min(kRB, nrows - it.rb * kRB);
        const int pos0 = row0(sm, it);
        const bool shared = it.g == p.E;
        if (!DOWN) {
            // gate/up: records 2 fl (gate) and 2 fl + 1 (up) give h[f], f = rb * 64 + fl
            constexpr int kF = kRB / 2;
            for (int o = tid; o < it.nt * kF; o += nthr) {
                const int t = o / kF, fl = o - t * kF;
                if (2 * fl >= nr) continue;
                const int f = it.rb * kF + fl;
                float g = out[(2 * fl) * kOutLd + t], u = out[(2 * fl + 1) * kOutLd + t];
                const int e = shared ? 0 : ent[t];
                const int tok = shared ? it.t0 + t : e / p.K, sl = shared ? p.K : e - (e / p.K) * p.K;
                const LoraDev &lg = slot_lora_g(p, sl, 0), &lu = slot_lora_g(p, sl, 1);
                if (lg.r || lu.r) {
                    const size_t eo = shared ? 0 : (size_t)it.g;
                    const float *v = p.v + ((size_t)tok * p.slots + sl) * 3 * kMaxLoraRank;
                    if (lg.r) {
                        const uint16_t *B = lg.B + eo * lg.b_stride + (size_t)f * lg.r;
                        float a = 0.0f;
                        for (int k = 0; k < lg.r; k++) a = fmaf(half_f(B[k]), v[k], a);
                        g += lg.scale * a;
                    }
                    if (lu.r) {
                        const uint16_t *B = lu.B + eo * lu.b_stride + (size_t)f * lu.r;
                        float a = 0.0f;
                        for (int k = 0; k < lu.r; k++) a = fmaf(half_f(B[k]), v[kMaxLoraRank + k], a);
                        u += lu.scale * a;
                    }
                }
                p.h16[(size_t)(pos0 + t) * p.F + f] = __float2bfloat16_rn(silu_f(g) * u);
            }
        } else {
            // down: record ol gives y[o], o = rb * 128 + ol
            for (int o = tid; o < it.nt * kRB; o += nthr) {
                const int t = o / kRB, ol = o - t * kRB;
                if (ol >= nr) continue;
                const int oo = it.rb * kRB + ol;
                float y = out[ol * kOutLd + t];
                const int e = shared ? 0 : ent[t];
                const int tok = shared ? it.t0 + t : e / p.K, sl = shared ? p.K : e - (e / p.K) * p.K;
                const LoraDev &ld = slot_lora_g(p, sl, 2);
                if (ld.r) {
                    const size_t eo = shared ? 0 : (size_t)it.g;
                    const uint16_t *B = ld.B + eo * ld.b_stride + (size_t)oo * ld.r;
                    const float *vd = p.vd + (size_t)(pos0 + t) * kMaxLoraRank;
                    float a = 0.0f;
                    for (int k = 0; k < ld.r; k++) a = fmaf(half_f(B[k]), vd[k], a);
                    y += ld.scale * a;
                }
                p.y[((size_t)tok * p.slots + sl) * p.d + oo] = y;
            }
        }
    }
};

// vd[pos][i] = sum_f A_d[i][f] h[pos][f] for the sorted positions p0 ..
// npos - 1 whose slot has a down LoRA.  One warp per (position, i).
__global__ void __launch_bounds__(256) lora_down_ax_kernel(FfnParams p, int p0, int npos) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (w >= (npos - p0) * kMaxLoraRank) return;
    const int ps = p0 + w / kMaxLoraRank, i = w % kMaxLoraRank;
    const int TK = p.T * p.K;
    int t, sl;
    if (ps >= TK) {
        t = ps - TK;
        sl = p.K;
    } else {
        const int ent = p.perm[ps];
        t = ent / p.K;
        sl = ent % p.K;
    }
    const LoraDev &ld = slot_lora_g(p, sl, 2);
    if (i >= ld.r) return;
    const int ee = sl < p.K ? p.idx[(size_t)t * p.K + sl] : 0;
    if ((unsigned)ee >= (unsigned)p.E) return;
    const uint16_t *A = ld.A + (sl < p.K ? (size_t)ee * ld.a_stride : 0) + (size_t)i * p.F;
    const __nv_bfloat16 *h = p.h16 + (size_t)ps * p.F;
    float a = 0.0f;
    for (int f = lane; f < p.F; f += 32) a = fmaf(half_f(A[f]), __bfloat162float(h[f]), a);
    a = warp_sum(a, 32);
    if (lane == 0) p.vd[(size_t)ps * kMaxLoraRank + i] = a;
}

template <int BITS>
static int launch_bits(const FfnParams &p, cudaStream_t st) {
    const int TK = p.T * p.K;
    if (cudaMemsetAsync(p.err, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ECUDA;
    const int nb = (p.E + 1 + 7) / 8;           // one warp per bucket, 8 warps per CTA
    sort_count_kernel<<<nb, 256, 0, st>>>(p.idx, TK, p.E, p.counts);
    if (int rc = check_launch("sort_count_kernel")) return rc;
    sort_scatter_kernel<<<nb, 256, 0, st>>>(p.idx, TK, p.E, p.counts, p.offsets, p.perm);
    if (int rc = check_launch("sort_scatter_kernel")) return rc;
    invalid_fill_kernel<<<64, 256, 0, st>>>(p.offsets, p.perm, p.E, p.K, p.slots, p.d, p.y);
    if (int rc = check_launch("invalid_fill_kernel")) return rc;
    const int npos = TK + (p.shared ? p.T : 0);
    gather_x_kernel<<<(npos + 7) / 8, 256, 0, st>>>(p, npos);
    if (int rc = check_launch("gather_x_kernel")) return rc;
    if (p.any_gu_lora) {
        lora_ax_kernel_launch(p, st);
        if (int rc = check_launch("lora_ax_kernel")) return rc;
    }
    const int G = p.E + (p.shared ? 1 : 0);
    const int rb_gu = (2 * p.F + kRB - 1) / kRB, rb_dn = (p.d + kRB - 1) / kRB;
    item_offsets_kernel<<<1, 1024, 0, st>>>(p.counts, p.E, p.T, G, rb_gu, rb_dn, p.item_off,
                                            p.item_off + G + 1);
    if (int rc = check_launch("item_offsets_kernel")) return rc;
    const size_t scratch = (size_t)(G + 1 + p.E + 1) * sizeof(int32_t);
    const int sms = num_sms();
    FfnJob<false> gu;
    if (int rc = gu.make(p, p.item_off)) return rc;
    // mean tokens of a routed expert's group: the engine choice
    const double mean_tok = (double)p.T * p.K / p.E;
    if (int rc = umma::launch_batched_gemm<BITS>(gu, scratch, sms, st, "batched gemm (gate/up)", mean_tok))
        return rc;
    if (int rc = launch_group_sums(p.h16, npos, p.F, p.hsum, st)) return rc;
    if (p.lora[2].r || (p.shared && p.shared_lora[2].r)) {
        // positions [p0, npos): all of them, or the shared expert's alone
        const int p0 = p.lora[2].r ? 0 : TK;
        const int warps = (npos - p0) * kMaxLoraRank;
        lora_down_ax_kernel<<<(warps + 7) / 8, 256, 0, st>>>(p, p0, npos);
        if (int rc = check_launch("lora_down_ax_kernel")) return rc;
    }
    FfnJob<true> dn;
    if (int rc = dn.make(p, p.item_off + G + 1)) return rc;
    return umma::launch_batched_gemm<BITS>(dn, scratch, sms, st, "batched gemm (down)", mean_tok);
}

}  // namespace grouped

int launch_expert_ffn_grouped(const FfnParams &p, cudaStream_t st) {
    return p.bits == 4 ? grouped::launch_bits<4>(p, st) : grouped::launch_bits<2>(p, st);
}

}  // namespace moe

extern "C" int moe_debug_batched_trace(unsigned long long *buf) {
    moe::umma::trace_buf() = buf;
    return MOE_OK;
}

extern "C" int moe_debug_batched_engine(int mode) {
    if (mode < 0 || mode > 2) return moe::fail(MOE_EINVAL, "debug_batched_engine: mode %d", mode);
    moe::umma::engine_mode() = mode;
    return MOE_OK;
}

extern "C" int moe_debug_batched_waits(unsigned long long timeout_ns, int stall) {
    moe::pipe::wait_cfg() = moe::pipe::WaitCfg{timeout_ns, stall ? 1 : 0};
    return MOE_OK;
}
