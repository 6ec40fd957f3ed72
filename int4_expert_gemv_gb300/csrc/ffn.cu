// ffn.cu -- expert FFN kernels: gate/up GEMV + SwiGLU, down GEMV, LoRA deltas.
//
// Per selected expert (and the shared expert):
//   g = W_g x (+ s_g B_g A_g x),  u = W_u x (+ s_u B_u A_u x)
//   h = silu(g) * u                       fused SwiGLU ("Arquitectura del
//                                         Sistema", kerneldigest.dev page)
//   y = W_d h (+ s_d B_d A_d h)           unfused recovery LoRA ("Ejecucion
//                                         del adaptador no fusionado",
//                                         xyznot.com/es/paper/2609.18063)
// W are group-64 affine int4 / 2-bit weights read from packed records and
// dequantised in registers.  The pages' per-weight form
// fma(code, scale*x, bias*x) is applied per 16-byte chunk: the chunk's codes
// are dotted with x first, then fma(scale, sum code*x, bias*sum x) adds the
// affine terms, which is the same sum with two multiplies per chunk instead
// of two per weight.
#include "internal.h"

namespace moe {

// Partial dot product of one record (row) with x, over the chunks this lane
// owns (c = sub, sub + lpr, ...).  xs: x in shared memory; xsum: per-chunk
// sums of x.  The caller reduces the partials over the lpr lanes.
template <int BITS>
__device__ __forceinline__ float record_dot(const uint8_t *rec, int nch, size_t cb,
                                            const float *xs, const float *xsum, int sub,
                                            int lpr) {
    constexpr int VALS = 128 / BITS;
    float acc = 0.0f;
    for (int c = sub; c < nch; c += lpr) {
        uint4 q = ld_stream16(rec + (size_t)kChunk * c);
        float2 sb = sb_f(ld_stream4(rec + cb + 4 * ((c * VALS) / kGroup)));
        acc += fmaf(sb.x, chunk_dot<BITS>(q, xs + c * VALS), sb.y * xsum[c]);
    }
    return acc;
}

// Largest power of two <= min(32, n).
__device__ __forceinline__ int lanes_per_row(int n) {
    int l = 1;
    while (l * 2 <= n && l < 32) l *= 2;
    return l;
}

// Blob of slot s of token t; nullptr for an expert index outside [0, E)
// (such a slot is never read: its outputs are written as NaN).
__device__ __forceinline__ const uint8_t *slot_blob(const FfnParams &p, int t, int s) {
    if (s >= p.K) return p.shared;
    const int e = p.idx[(size_t)t * p.K + s];
    return (unsigned)e < (unsigned)p.E ? p.pool + (size_t)e * p.stride : nullptr;
}

__device__ __forceinline__ int slot_expert(const FfnParams &p, int t, int s) {
    const int e = s < p.K ? p.idx[(size_t)t * p.K + s] : 0;
    return (unsigned)e < (unsigned)p.E ? e : 0;
}

__device__ __forceinline__ const LoraDev &slot_lora(const FfnParams &p, int s, int which) {
    return s < p.K ? p.lora[which] : p.shared_lora[which];
}

// Loads x[t] (d values) into shared memory and the per-chunk sums of x.
template <int VALS>
__device__ __forceinline__ void stage_x(const void *x, int dtype, size_t base, int n,
                                        float *xs, float *xsum) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) xs[i] = load_act(x, dtype, base + i);
    __syncthreads();
    for (int c = threadIdx.x; c < n / VALS; c += blockDim.x) {
        float a = 0.0f;
        for (int j = 0; j < VALS; j++) a += xs[c * VALS + j];
        xsum[c] = a;
    }
    __syncthreads();
}

// ---------------------------------------------------------------- LoRA A x
// v[t*slots+s][which][i] = sum_k A[i][k] x[t][k] for the gate (which 0) and
// up (which 1) adapters of slot s = s0 + blockIdx.x.  grid (slots from s0,
// T), 256 threads.
__global__ void __launch_bounds__(256) lora_ax_kernel(FfnParams p, int s0) {
    extern __shared__ float sm[];
    const int s = s0 + blockIdx.x, t = blockIdx.y, d = p.d;
    float *xs = sm;
    for (int i = threadIdx.x; i < d; i += blockDim.x)
        xs[i] = load_act(p.x, p.x_dtype, (size_t)t * d + i);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int e = slot_expert(p, t, s);
    for (int which = 0; which < 2; which++) {
        const LoraDev &l = slot_lora(p, s, which);
        if (l.r == 0) continue;
        const uint16_t *A = l.A + (s < p.K ? (size_t)e * l.a_stride : 0);
        for (int i = warp; i < l.r; i += nw) {
            float a = 0.0f;
            for (int k = lane; k < d; k += 32) a = fmaf(half_f(A[(size_t)i * d + k]), xs[k], a);
            a = warp_sum(a, 32);
            if (lane == 0)
                p.v[(((size_t)t * p.slots + s) * 3 + which) * kMaxLoraRank + i] = a;
        }
    }
}

__device__ __forceinline__ float lora_b_row(const LoraDev &l, int s, int K, int e, int row,
                                            const float *v) {
    const uint16_t *B = l.B + (s < K ? (size_t)e * l.b_stride : 0) + (size_t)row * l.r;
    float a = 0.0f;
    for (int i = 0; i < l.r; i++) a = fmaf(half_f(B[i]), v[i], a);
    return l.scale * a;
}

// ---------------------------------------------------------------- gate/up
// grid (ceil(F / rows_per_cta), slots, T); block 256.  Each warp takes row
// pairs (gate row f, up row f: adjacent records) and writes h[t][s][f].
template <int BITS>
__global__ void __launch_bounds__(256) gateup_kernel(FfnParams p, int rows_per_cta) {
    extern __shared__ float sm[];
    constexpr int VALS = 128 / BITS;
    const int s = blockIdx.y, t = blockIdx.z, d = p.d, F = p.F;
    const int nch = d / VALS;
    float *xs = sm, *xsum = sm + d;
    stage_x<VALS>(p.x, p.x_dtype, (size_t)t * d, d, xs, xsum);

    const uint8_t *blob = slot_blob(p, t, s);
    if (blob == nullptr) {
        for (int f = blockIdx.x * rows_per_cta + threadIdx.x;
             f < min(F, (int)(blockIdx.x + 1) * rows_per_cta); f += blockDim.x)
            p.h[((size_t)t * p.slots + s) * F + f] = __int_as_float(0x7fc00000);
        return;
    }
    const uint8_t *gu = blob + p.L.gu_off;
    const int e = slot_expert(p, t, s);
    const size_t rec = p.L.gu_rec, cb = code_bytes(d, BITS);
    const int lpr = lanes_per_row(nch), rpw = 32 / lpr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int sub = lane % lpr, rsub = lane / lpr;
    const int f0 = blockIdx.x * rows_per_cta, f1 = min(F, f0 + rows_per_cta);
    const LoraDev &lg = slot_lora(p, s, 0), &lu = slot_lora(p, s, 1);
    const float *v = p.v + ((size_t)t * p.slots + s) * 3 * kMaxLoraRank;

    for (int base = f0 + warp * rpw; base < f1; base += nw * rpw) {
        const int f = base + rsub;
        const bool ok = f < f1;
        float ag = 0.0f, au = 0.0f;
        if (ok) {
            const uint8_t *rg = gu + (size_t)(2 * f) * rec;
            ag = record_dot<BITS>(rg, nch, cb, xs, xsum, sub, lpr);
            au = record_dot<BITS>(rg + rec, nch, cb, xs, xsum, sub, lpr);
        }
        ag = warp_sum(ag, lpr);
        au = warp_sum(au, lpr);
        if (ok && sub == 0) {
            if (lg.r) ag += lora_b_row(lg, s, p.K, e, f, v);
            if (lu.r) au += lora_b_row(lu, s, p.K, e, f, v + kMaxLoraRank);
            float h = silu_f(ag) * au;
            if (p.round_h_bf16) h = __bfloat162float(__float2bfloat16_rn(h));
            p.h[((size_t)t * p.slots + s) * F + f] = h;
        }
    }
}

// ---------------------------------------------------------------- down
// grid (ceil(d / rows_per_cta), slots, T); block 256.
template <int BITS>
__global__ void __launch_bounds__(256) down_kernel(FfnParams p, int rows_per_cta) {
    extern __shared__ float sm[];
    constexpr int VALS = 128 / BITS;
    const int s = blockIdx.y, t = blockIdx.z, d = p.d, F = p.F;
    const int nch = F / VALS;
    float *hs = sm, *hsum = sm + F, *vd = sm + F + nch;
    const size_t ts = (size_t)t * p.slots + s;
    stage_x<VALS>(p.h, MOE_DTYPE_F32, ts * F, F, hs, hsum);

    const int e = slot_expert(p, t, s);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const LoraDev &ld = slot_lora(p, s, 2);
    if (ld.r) {                                   // vd = A_d h
        const uint16_t *A = ld.A + (s < p.K ? (size_t)e * ld.a_stride : 0);
        for (int i = warp; i < ld.r; i += nw) {
            float a = 0.0f;
            for (int k = lane; k < F; k += 32) a = fmaf(half_f(A[(size_t)i * F + k]), hs[k], a);
            a = warp_sum(a, 32);
            if (lane == 0) vd[i] = a;
        }
        __syncthreads();
    }

    const uint8_t *blob = slot_blob(p, t, s);
    if (blob == nullptr) {
        for (int o = blockIdx.x * rows_per_cta + threadIdx.x;
             o < min(d, (int)(blockIdx.x + 1) * rows_per_cta); o += blockDim.x)
            p.y[ts * d + o] = __int_as_float(0x7fc00000);
        return;
    }
    const uint8_t *dn = blob + p.L.down_off;
    const size_t rec = p.L.down_rec, cb = code_bytes(F, BITS);
    const int lpr = lanes_per_row(nch), rpw = 32 / lpr;
    const int sub = lane % lpr, rsub = lane / lpr;
    const int o0 = blockIdx.x * rows_per_cta, o1 = min(d, o0 + rows_per_cta);
    for (int base = o0 + warp * rpw; base < o1; base += nw * rpw) {
        const int o = base + rsub;
        const bool ok = o < o1;
        float a = ok ? record_dot<BITS>(dn + (size_t)o * rec, nch, cb, hs, hsum, sub, lpr) : 0.0f;
        a = warp_sum(a, lpr);
        if (ok && sub == 0) {
            if (ld.r) a += lora_b_row(ld, s, p.K, e, o, vd);
            p.y[ts * d + o] = a;
        }
    }
}

// ---------------------------------------------------------------- launch
template <int BITS>
static int launch_bits(const FfnParams &p, cudaStream_t st) {
    constexpr int VALS = 128 / BITS;
    const int threads = 256;
    if (p.any_gu_lora) {
        lora_ax_kernel<<<dim3(p.slots, p.T), threads, p.d * sizeof(float), st>>>(p, 0);
        if (int rc = check_launch("lora_ax_kernel")) return rc;
    }
    {
        const int rows = 16;
        const size_t smem = (size_t)(p.d + p.d / VALS) * sizeof(float);
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(gateup_kernel<BITS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        gateup_kernel<BITS><<<dim3((p.F + rows - 1) / rows, p.slots, p.T), threads, smem, st>>>(
            p, rows);
        if (int rc = check_launch("gateup_kernel")) return rc;
    }
    {
        const int rows = 32;
        const size_t smem = (size_t)(p.F + p.F / VALS + kMaxLoraRank) * sizeof(float);
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(down_kernel<BITS>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        down_kernel<BITS><<<dim3((p.d + rows - 1) / rows, p.slots, p.T), threads, smem, st>>>(
            p, rows);
        if (int rc = check_launch("down_kernel")) return rc;
    }
    return MOE_OK;
}

// Only the slots that carry a gate or up adapter: all of them when the
// routed experts do, else the shared slot alone.
void lora_ax_kernel_launch(const FfnParams &p, cudaStream_t st) {
    const bool routed = p.lora[0].r || p.lora[1].r;
    lora_ax_kernel<<<dim3(routed ? p.slots : 1, p.T), 256, p.d * sizeof(float), st>>>(
        p, routed ? 0 : p.K);
}

int launch_expert_ffn(const FfnParams &p, cudaStream_t st) {
    return p.bits == 4 ? launch_bits<4>(p, st) : launch_bits<2>(p, st);
}

}  // namespace moe
