// head_route.cu -- prerouter head, fused top-K/softmax router, fused combine.
//
// Head ("Arquitectura del cabezal Prerouter", xyznot.com/es/paper/2609.18063):
// features f = [x ; K-hot(cur) ; K-hot(prev)] of width d + 2E feed
//     head(f) = fc2(erf-gelu(fc1 f)) + l(f).
// The K-hot part of f is never materialised: the columns of fc1 and l that
// multiply it are stored transposed as row tables, and the 2K rows selected
// by the routes are gathered and added.
// Router: top-K of the head's logits; the prediction is the routing ("Ideas
// clave" of the same page).  Combine + residual (+ RMS normalisation) is the
// fused expert-combine kernel of "Arquitectura del Sistema" (kerneldigest.dev).
#include <cfloat>

#include "gemm_pipe.cuh"
#include "gemm_umma.cuh"
#include "internal.h"

namespace moe {

template <int BITS>
__device__ __forceinline__ float rec_dot(const uint8_t *rec, int cols, const float *xs,
                                         const float *xsum, int sub, int lpr) {
    constexpr int VALS = 128 / BITS;
    const int nch = cols / VALS;
    const size_t cb = code_bytes(cols, BITS);
    float acc = 0.0f;
    for (int c = sub; c < nch; c += lpr) {
        uint4 q = ld_stream16(rec + (size_t)kChunk * c);
        float2 sb = sb_f(ld_stream4(rec + cb + 4 * ((c * VALS) / kGroup)));
        acc += fmaf(sb.x, chunk_dot<BITS>(q, xs + c * VALS), sb.y * xsum[c]);
    }
    return acc;
}

__device__ __forceinline__ float f16_row_dot(const uint8_t *row, int cols, const float *xs,
                                             int sub, int lpr) {
    float acc = 0.0f;
    for (int c = sub; c < cols / 8; c += lpr)
        acc += chunk_dot_f16(ld_stream16(row + (size_t)kChunk * c), xs + 8 * c);
    return acc;
}

__device__ __forceinline__ float mat_row_dot(int prec, const uint8_t *m, int row, int cols,
                                             const float *xs, const float *xsum, int sub,
                                             int lpr) {
    if (prec == MOE_PREC_FP16)
        return f16_row_dot(m + (size_t)row * cols * 2, cols, xs, sub, lpr);
    return rec_dot<4>(m + (size_t)row * record_bytes(cols, 4), cols, xs, xsum, sub, lpr);
}

__device__ __forceinline__ int pow2_lanes(int n) {
    int l = 1;
    while (l * 2 <= n && l < 32) l *= 2;
    return l;
}

// Sum of the 2K gathered table rows: tab[cur[k]][col] and tab[E+prev[k]][col].
__device__ __forceinline__ float gather_rows(const uint16_t *tab, int width, int E,
                                             const int32_t *cur, const int32_t *prev, int K,
                                             int col) {
    float a = 0.0f;
    if (tab == nullptr) return a;
    // indices outside [0, E) contribute nothing (never read out of bounds)
    if (cur)
        for (int k = 0; k < K; k++)
            if ((unsigned)cur[k] < (unsigned)E) a += half_f(tab[(size_t)cur[k] * width + col]);
    if (prev)
        for (int k = 0; k < K; k++)
            if ((unsigned)prev[k] < (unsigned)E)
                a += half_f(tab[(size_t)(E + prev[k]) * width + col]);
    return a;
}

__device__ __forceinline__ float bias_f(const uint16_t *b, int i) {
    return b ? half_f(b[i]) : 0.0f;
}

// ---------------------------------------------------------------- fc1 + l
// Rows [0, H) are fc1 rows, rows [H, H+E) are l rows; all multiply x.
// grid (ceil((H+E)/rows_per_cta), T); block 256.
__global__ void __launch_bounds__(256) head_x_kernel(HeadParams p, int rows_per_cta) {
    extern __shared__ float sm[];
    const int t = blockIdx.y, d = p.d, H = p.H, E = p.E;
    float *xs = sm, *xsum = sm + d;
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        xs[i] = load_act(p.x, p.x_dtype, (size_t)t * d + i);
    __syncthreads();
    for (int c = threadIdx.x; c < d / 32; c += blockDim.x) {
        float a = 0.0f;
        for (int j = 0; j < 32; j++) a += xs[c * 32 + j];
        xsum[c] = a;
    }
    __syncthreads();
    const int32_t *cur = p.cur ? p.cur + (size_t)t * p.K : nullptr;
    const int32_t *prev = p.prev ? p.prev + (size_t)t * p.K : nullptr;
    const int nch = p.prec == MOE_PREC_FP16 ? d / 8 : d / 32;
    const int lpr = pow2_lanes(nch), rpw = 32 / lpr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int sub = lane % lpr, rsub = lane / lpr;
    const int r0 = blockIdx.x * rows_per_cta, r1 = min(H + E, r0 + rows_per_cta);
    for (int base = r0 + warp * rpw; base < r1; base += nw * rpw) {
        const int r = base + rsub;
        const bool ok = r < r1;
        float a = 0.0f;
        if (ok) {
            a = r < H ? mat_row_dot(p.prec, p.fc1x, r, d, xs, xsum, sub, lpr)
                      : mat_row_dot(p.prec, p.lx, r - H, d, xs, xsum, sub, lpr);
        }
        a = warp_sum(a, lpr);
        if (ok && sub == 0) {
            if (r < H) {
                a += gather_rows(p.fc1_tab, H, E, cur, prev, p.K, r) + bias_f(p.b1, r);
                p.g[(size_t)t * H + r] = gelu_erf_f(a);
            } else {
                const int e = r - H;
                a += gather_rows(p.l_tab, E, E, cur, prev, p.K, e) + bias_f(p.bl, e);
                if (H == 0) p.logits[(size_t)t * E + e] = a;
                else p.zl[(size_t)t * E + e] = a;
            }
        }
    }
}

// ---------------------------------------------------------------- fc2
// logits[t][e] = fc2[e] . g[t] + b2[e] + zl[t][e].  grid (ceil(E/rows), T).
__global__ void __launch_bounds__(256) head_fc2_kernel(HeadParams p, int rows_per_cta) {
    extern __shared__ float sm[];
    const int t = blockIdx.y, H = p.H, E = p.E;
    float *gs = sm, *gsum = sm + H;
    for (int i = threadIdx.x; i < H; i += blockDim.x) gs[i] = p.g[(size_t)t * H + i];
    __syncthreads();
    for (int c = threadIdx.x; c < H / 32; c += blockDim.x) {
        float a = 0.0f;
        for (int j = 0; j < 32; j++) a += gs[c * 32 + j];
        gsum[c] = a;
    }
    __syncthreads();
    const int nch = p.prec == MOE_PREC_FP16 ? H / 8 : H / 32;
    const int lpr = pow2_lanes(nch), rpw = 32 / lpr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int sub = lane % lpr, rsub = lane / lpr;
    const int r0 = blockIdx.x * rows_per_cta, r1 = min(E, r0 + rows_per_cta);
    for (int base = r0 + warp * rpw; base < r1; base += nw * rpw) {
        const int e = base + rsub;
        const bool ok = e < r1;
        float a = ok ? mat_row_dot(p.prec, p.fc2, e, H, gs, gsum, sub, lpr) : 0.0f;
        a = warp_sum(a, lpr);
        if (ok && sub == 0)
            p.logits[(size_t)t * E + e] = a + bias_f(p.b2, e) + p.zl[(size_t)t * E + e];
    }
}

// ---------------------------------------------------------------- batched
// The K-hot and bias terms of fc1 and l for every token: g[t][r] = the
// gathered fc1 table rows + b1, zl[t][e] (logits when H = 0) = the gathered
// l table rows + bl.  grid T, block 256; the batched head's GEMM epilogue
// adds the x part.
__global__ void __launch_bounds__(256) head_tab_kernel(HeadParams p) {
    __shared__ int32_t rc[32];
    const int t = blockIdx.x;
    const int nk = (p.cur || p.prev) ? p.K : 0;     // K <= 16 is checked when a route is given
    if (threadIdx.x < 2 * nk) {
        const int32_t *src = threadIdx.x < nk ? p.cur : p.prev;
        const int k = threadIdx.x < nk ? threadIdx.x : threadIdx.x - nk;
        rc[threadIdx.x] = src ? src[(size_t)t * nk + k] : -1;
    }
    __syncthreads();
    float *zl = p.H ? p.zl : p.logits;
    for (int r = threadIdx.x; r < p.H + p.E; r += blockDim.x) {
        const bool fc1 = r < p.H;
        const int col = fc1 ? r : r - p.H, width = fc1 ? p.H : p.E;
        const uint16_t *tab = fc1 ? p.fc1_tab : p.l_tab;
        float a = bias_f(fc1 ? p.b1 : p.bl, col);
        if (tab) {
            // indices outside [0, E) contribute nothing (never read out of bounds)
            for (int k = 0; k < 2 * nk; k++) {
                const int c = rc[k];
                if ((unsigned)c < (unsigned)p.E)
                    a += half_f(tab[(size_t)(k < nk ? c : p.E + c) * width + col]);
            }
        }
        if (fc1) p.g[(size_t)t * p.H + col] = a;
        else zl[(size_t)t * p.E + col] = a;
    }
}

// fc1 and l on x for T > 1 bf16 tokens (int4 head) as one job of the
// persistent tensor-core engine: rows [0, H) are fc1 rows, then E l rows,
// each against every token; the epilogue adds the x part to what
// head_tab_kernel wrote and applies gelu to the fc1 rows, as head_x_kernel
// does per token.
struct HeadXJob {
    pipe::Maps maps;
    HeadParams p;
    int32_t *err;
    int RB0, RB, cols;

    // Tensor maps (map 0: fc1x rows, map 1: l rows) and geometry.
    __host__ int make(const HeadParams &pp) {
        p = pp;
        err = p.err;
        RB0 = (p.H + pipe::kRB - 1) / pipe::kRB;
        RB = RB0 + (p.E + pipe::kRB - 1) / pipe::kRB;
        cols = p.d;
        const size_t rec = record_bytes(p.d, 4);
        if (int rc = pipe::weight_maps(maps, 1, p.lx, rec, p.E, 1, 0, 4)) return rc;
        if (int rc = p.H ? pipe::weight_maps(maps, 0, p.fc1x, rec, p.H, 1, 0, 4)
                         : pipe::weight_maps(maps, 0, p.lx, rec, p.E, 1, 0, 4))
            return rc;
        return pipe::act_maps(maps, p.x, p.xsum, p.T, p.d);
    }
    __device__ void init(int32_t *) const {}
    __device__ int n_items(const int32_t *) const {
        return RB * ((p.T + pipe::kTok - 1) / pipe::kTok);
    }
    __device__ pipe::Item item(const int32_t *, int i) const {
        const int tile = i / RB;
        pipe::Item it;
        it.g = 0;
        it.rb = i - tile * RB;
        it.t0 = tile * pipe::kTok;
        it.nt = min(pipe::kTok, p.T - it.t0);
        return it;
    }
    __device__ void weights(const pipe::Item &it, int &map, int &row, int &blob) const {
        map = it.rb < RB0 ? 0 : 1;
        row = (it.rb < RB0 ? it.rb : it.rb - RB0) * pipe::kRB;
        blob = 0;
    }
    __device__ int row0(const int32_t *, const pipe::Item &it) const { return it.t0; }
    __device__ const int32_t *meta(const int32_t *, const pipe::Item &) const { return nullptr; }
    __device__ void epilogue(const int32_t *, const pipe::Item &it, const float *out,
                             const int32_t *, int tid, int nthr) const {
        const bool fc1 = it.rb < RB0;
        const int base = (fc1 ? it.rb : it.rb - RB0) * pipe::kRB;
        const int nr = min(pipe::kRB, (fc1 ? p.H : p.E) - base);
        for (int o = tid; o < it.nt * pipe::kRB; o += nthr) {
            const int t = o / pipe::kRB, rl = o - t * pipe::kRB;
            if (rl >= nr) continue;
            const int tok = it.t0 + t, r = base + rl;
            const float a = out[rl * pipe::kOutLd + t];
            if (fc1) {
                // g = gelu(.), split as hi + lo (two bf16 rows) for the fc2 job
                const float gv = gelu_erf_f(a + p.g[(size_t)tok * p.H + r]);
                const __nv_bfloat16 hi = __float2bfloat16_rn(gv);
                p.gg[(size_t)(2 * tok) * p.H + r] = hi;
                p.gg[(size_t)(2 * tok + 1) * p.H + r] = __float2bfloat16_rn(gv - __bfloat162float(hi));
            } else {
                float *zp = (p.H ? p.zl : p.logits) + (size_t)tok * p.E + r;
                *zp = a + *zp;
            }
        }
    }
};

// fc2 on g for T > 1 bf16 tokens (int4 head): E records of H columns
// against the 2T rows of g split as bf16 hi + lo (g = hi + lo to about 16
// significant bits, so the logits keep fp32 accuracy); the epilogue adds a
// token's two rows, b2 and zl: logits[t][e].
struct Fc2Job {
    pipe::Maps maps;
    HeadParams p;
    int32_t *err;
    int RB, cols;

    __host__ int make(const HeadParams &pp) {
        p = pp;
        err = p.err;
        RB = (p.E + pipe::kRB - 1) / pipe::kRB;
        cols = p.H;
        const size_t rec = record_bytes(p.H, 4);
        if (int rc = pipe::weight_maps(maps, 0, p.fc2, rec, p.E, 1, 0, 4)) return rc;
        if (int rc = pipe::weight_maps(maps, 1, p.fc2, rec, p.E, 1, 0, 4)) return rc;
        return pipe::act_maps(maps, p.gg, p.ggsum, 2 * p.T, p.H);
    }
    __device__ void init(int32_t *) const {}
    __device__ int n_items(const int32_t *) const {
        return RB * ((2 * p.T + pipe::kTok - 1) / pipe::kTok);
    }
    __device__ pipe::Item item(const int32_t *, int i) const {
        const int tile = i / RB;
        pipe::Item it;
        it.g = 0;
        it.rb = i - tile * RB;
        it.t0 = tile * pipe::kTok;
        it.nt = min(pipe::kTok, 2 * p.T - it.t0);
        return it;
    }
    __device__ void weights(const pipe::Item &it, int &map, int &row, int &blob) const {
        map = 0;
        row = it.rb * pipe::kRB;
        blob = 0;
    }
    __device__ int row0(const int32_t *, const pipe::Item &it) const { return it.t0; }
    __device__ const int32_t *meta(const int32_t *, const pipe::Item &) const { return nullptr; }
    __device__ void epilogue(const int32_t *, const pipe::Item &it, const float *out,
                             const int32_t *, int tid, int nthr) const {
        const int base = it.rb * pipe::kRB;
        const int nr = min(pipe::kRB, p.E - base);
        for (int o = tid; o < (it.nt / 2) * pipe::kRB; o += nthr) {
            const int tl = o / pipe::kRB, rl = o - tl * pipe::kRB;
            if (rl >= nr) continue;
            const int tok = (it.t0 >> 1) + tl, e = base + rl;
            const float a = out[rl * pipe::kOutLd + 2 * tl] + out[rl * pipe::kOutLd + 2 * tl + 1];
            p.logits[(size_t)tok * p.E + e] = a + bias_f(p.b2, e) + p.zl[(size_t)tok * p.E + e];
        }
    }
};

int launch_prerouter_head(const HeadParams &p, cudaStream_t st) {
    const int threads = 256;
    if (p.T > 1 && p.x_dtype == MOE_DTYPE_BF16 && p.prec == MOE_PREC_AFFINE4) {
        const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(p.x);
        if (int rc = pipe::launch_group_sums(xb, p.T, p.d, p.xsum, st)) return rc;
        head_tab_kernel<<<p.T, threads, 0, st>>>(p);
        if (int rc = check_launch("head_tab_kernel")) return rc;
        if (cudaMemsetAsync(p.err, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ECUDA;
        HeadXJob job;
        if (int rc = job.make(p)) return rc;
        if (int rc = umma::launch_batched_gemm<4>(job, 0, num_sms(), st, "batched gemm (head fc1, l)", p.T))
            return rc;
        if (p.H > 0) {
            if (int rc = pipe::launch_group_sums(p.gg, 2 * p.T, p.H, p.ggsum, st)) return rc;
            Fc2Job f2;
            if (int rc = f2.make(p)) return rc;
            return umma::launch_batched_gemm<4>(f2, 0, num_sms(), st, "batched gemm (head fc2)", 2.0 * p.T);
        }
        return MOE_OK;
    } else {
        const int rows = 16;
        const size_t smem = (size_t)(p.d + p.d / 32) * sizeof(float);
        head_x_kernel<<<dim3((p.H + p.E + rows - 1) / rows, p.T), threads, smem, st>>>(p, rows);
        if (int rc = check_launch("head_x_kernel")) return rc;
    }
    if (p.H > 0) {
        const int rows = 16;
        const size_t smem = (size_t)(p.H + p.H / 32) * sizeof(float);
        head_fc2_kernel<<<dim3((p.E + rows - 1) / rows, p.T), threads, smem, st>>>(p, rows);
        if (int rc = check_launch("head_fc2_kernel")) return rc;
    }
    return MOE_OK;
}

// ---------------------------------------------------------------- top-K
// One warp per token.  Lane l holds logits l, l+32, ... (NV values).  K+1
// rounds of a warp-wide arg-max ordered by (value desc, index asc).
__device__ __forceinline__ bool better(float v, int i, float w, int j) {
    return v > w || (v == w && i < j);
}

template <int NV>
__global__ void __launch_bounds__(256) topk_kernel(const float *logits, int T, int E, int K,
                                                   int32_t *idx, float *wout, float *margin) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= T) return;                         // whole warp exits together
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = lane + 32 * i;
        const float z = e < E ? logits[(size_t)t * E + e] : -FLT_MAX;
        v[i] = z == z ? z : -INFINITY;          // a NaN logit ranks last
    }
    uint32_t taken = 0;
    float topv[17];
    int topi[17];
    const int rounds = K < E ? K + 1 : K;
    for (int k = 0; k < rounds; k++) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int e = lane + 32 * i;
            if (e < E && !(taken >> i & 1u) && better(v[i], e, bv, bi)) {
                bv = v[i];
                bi = e;
            }
        }
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        topv[k] = bv;
        topi[k] = bi;
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    if (lane == 0) {
        float sum = 0.0f;
        for (int k = 0; k < K; k++) sum += expf(topv[k] - topv[0]);
        for (int k = 0; k < K; k++) {
            idx[(size_t)t * K + k] = topi[k];
            wout[(size_t)t * K + k] = expf(topv[k] - topv[0]) / sum;
        }
        if (margin) margin[t] = K < E ? topv[K - 1] - topv[K] : INFINITY;
    }
}

int launch_topk(const float *logits, int T, int E, int K, int32_t *idx, float *w,
                float *margin, cudaStream_t st) {
    const int threads = 256, per = threads / 32;
    dim3 grid((T + per - 1) / per);
    const int nv = (E + 31) / 32;
    if (nv <= 1) topk_kernel<1><<<grid, threads, 0, st>>>(logits, T, E, K, idx, w, margin);
    else if (nv <= 2) topk_kernel<2><<<grid, threads, 0, st>>>(logits, T, E, K, idx, w, margin);
    else if (nv <= 4) topk_kernel<4><<<grid, threads, 0, st>>>(logits, T, E, K, idx, w, margin);
    else if (nv <= 8) topk_kernel<8><<<grid, threads, 0, st>>>(logits, T, E, K, idx, w, margin);
    else if (nv <= 16) topk_kernel<16><<<grid, threads, 0, st>>>(logits, T, E, K, idx, w, margin);
    else topk_kernel<32><<<grid, threads, 0, st>>>(logits, T, E, K, idx, w, margin);
    return check_launch("topk_kernel");
}

// ---------------------------------------------------------------- combine
// One CTA per token.  out = residual + sum_k w_k y_k (+ y_shared); optional
// x_next = out / sqrt(mean(out^2) + 1e-6).
__global__ void __launch_bounds__(256) combine_kernel(const float *y, const float *w, int K,
                                                      int has_shared, int d, const float *res,
                                                      float *out, float *xn) {
    __shared__ float red[32];
    const int t = blockIdx.x, slots = K + has_shared;
    const float *yt = y + (size_t)t * slots * d;
    const float *wt = w + (size_t)t * K;
    float ss = 0.0f;
    for (int i = threadIdx.x; i < d; i += blockDim.x) {
        float o = res[(size_t)t * d + i];
        for (int k = 0; k < K; k++) o = fmaf(wt[k], yt[(size_t)k * d + i], o);
        if (has_shared) o += yt[(size_t)K * d + i];
        out[(size_t)t * d + i] = o;
        ss = fmaf(o, o, ss);
    }
    if (xn == nullptr) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    ss = warp_sum(ss, 32);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.0f;
        for (int i = 0; i < nw; i++) a += red[i];
        red[0] = 1.0f / sqrtf(a / d + 1e-6f);
    }
    __syncthreads();
    const float inv = red[0];
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        xn[(size_t)t * d + i] = out[(size_t)t * d + i] * inv;
}

int launch_combine(const float *y, const float *w, int T, int K, int has_shared, int d,
                   const float *res, float *out, float *xn, cudaStream_t st) {
    combine_kernel<<<T, 256, 0, st>>>(y, w, K, has_shared, d, res, out, xn);
    return check_launch("combine_kernel");
}

}  // namespace moe
