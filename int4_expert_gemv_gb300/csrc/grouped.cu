// grouped.cu -- batched / prefill expert FFN (T > 1 tokens, bf16 activations).
//
// The tokens' (token, slot) entries are sorted by expert (a stable counting
// sort: histogram, exclusive scan, scatter in token order), so each routed
// expert's weights are read once for all the tokens routed to it and the
// shared expert's once for all T tokens ("tokens sorted/grouped by expert":
// the batched configuration of xyznot.com/es/paper/2609.18063's workload
// list; the layer math is the decode layer's, per token).  Each expert's
// token group then runs as two GEMMs on the tensor cores (mma.sync
// m16n8k16, bf16 in, fp32 accumulate):
//
//   gate/up:  [2F records] x [d] . [d] x [n_e tokens]  -> h = silu(g) * u
//   down:     [d records]  x [F] . [F] x [n_e tokens]  -> y_slots
//
// The weight operand is the codes themselves, offset into one binade so that
// a bf16 holds them exactly and is formed by an OR: a 4-bit code q as 16 + q
// (bits 0x4180 | q << 3), a 2-bit one as 4 + q (bits 0x4080 | q << 5).  The
// MMA then computes sum((c + q) x) exactly per product and in fp32 per sum
// (c the offset), and the affine terms of the group (64 columns, scale s,
// bias b) are applied per group in fp32:
//   sum_k (q_k s + b) x_k = s * sum (c + q) x + (b - c s) * sum x,
// with sum x per token and group computed once.  The smallest such offset
// keeps the cancellation between the two terms small.  Dequantised weights
// are never rounded.  h is rounded to bf16 before the down GEMM (the batched
// path's bf16 activations), as the oracle does.
#include <cuda_bf16.h>

#include "internal.h"

namespace moe {
namespace grouped {

constexpr int kTok = 64;          // tokens per CTA tile (8 n-tiles of 8)
constexpr int kRows = 64;         // weight records per CTA tile (4 warps x m16)
constexpr int kKc = 256;          // columns per staged chunk (4 groups of 64)
constexpr int kThreads = 128;
constexpr int kXld = kKc + 8;     // padded row (bf16) of the staged activations
constexpr int kGpc = kKc / kGroup;

// ---------------------------------------------------------------- sort
// counts[e] = entries routed to expert e (e < E); counts[E] = entries with an
// index outside [0, E).  One warp per bucket.
__global__ void __launch_bounds__(256) sort_count_kernel(const int32_t *idx, int TK, int E,
                                                         int32_t *counts) {
    const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (b > E) return;
    int n = 0;
    for (int i0 = 0; i0 < TK; i0 += 32) {
        const int i = i0 + lane;
        const int e = i < TK ? idx[i] : 0;
        const bool m = i < TK && (b < E ? e == b : (unsigned)e >= (unsigned)E);
        n += __popc(__ballot_sync(0xffffffffu, m));
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
    for (int i0 = 0; i0 < TK; i0 += 32) {
        const int i = i0 + lane;
        const int e = i < TK ? idx[i] : 0;
        const bool m = i < TK && (b < E ? e == b : (unsigned)e >= (unsigned)E);
        const uint32_t mask = __ballot_sync(0xffffffffu, m);
        if (m) perm[off + rank + __popc(mask & below)] = i;
        rank += __popc(mask);
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

// sums[r][g] = sum of v[r][64 g .. 64 g + 63] (bf16 values, fp32 sum in a
// fixed order), rows r < rows.  One warp per (row, group).
__global__ void __launch_bounds__(256) group_sums_kernel(const __nv_bfloat16 *v, int rows,
                                                         int cols, float *sums) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int ng = cols / kGroup;
    if (w >= rows * ng) return;
    const int r = w / ng, g = w % ng;
    const __nv_bfloat162 p = reinterpret_cast<const __nv_bfloat162 *>(v + (size_t)r * cols + g * kGroup)[lane];
    float a = __bfloat162float(p.x) + __bfloat162float(p.y);
    a = warp_sum(a, 32);
    if (lane == 0) sums[(size_t)r * ng + g] = a;
}

// ---------------------------------------------------------------- tiles
// The tile's tokens: token index, sorted position (row of h), slot.
__device__ __forceinline__ void tile_tokens(const FfnParams &p, int e, int t0, int nt, int *tok,
                                            int *pos, int *slot) {
    const int TK = p.T * p.K;
    for (int i = threadIdx.x; i < kTok; i += blockDim.x) {
        int t = -1, ps = -1, sl = -1;
        if (i < nt) {
            if (e == p.E) {                 // the shared expert: every token in order
                t = t0 + i;
                ps = TK + t;
                sl = p.K;
            } else {
                ps = p.offsets[e] + t0 + i;
                const int ent = p.perm[ps];
                t = ent / p.K;
                sl = ent % p.K;
            }
        }
        tok[i] = t;
        pos[i] = ps;
        slot[i] = sl;
    }
}

// Offset c of the bf16 code values (c + q), and the bf16 bits of c.
template <int BITS> struct CodeOff;
template <> struct CodeOff<4> { static constexpr float c = 16.0f; static constexpr uint32_t bits = 0x4180u, shift = 3; };
template <> struct CodeOff<2> { static constexpr float c = 4.0f; static constexpr uint32_t bits = 0x4080u, shift = 5; };

// Two bf16 (c + q) of the codes at columns k, k+1 (k even) of a record.
template <int BITS>
__device__ __forceinline__ uint32_t code_pair(const uint8_t *codes, int k) {
    uint32_t q0, q1;
    if (BITS == 4) {
        const uint32_t b = codes[k >> 1];
        q0 = b & 15u;
        q1 = b >> 4;
    } else {
        const uint32_t b = codes[k >> 2], sh = (uint32_t)(k & 3) * 2u;
        q0 = (b >> sh) & 3u;
        q1 = (b >> (sh + 2u)) & 3u;
    }
    constexpr uint32_t sh = CodeOff<BITS>::shift;
    return (CodeOff<BITS>::bits * 0x10001u) | (q0 << sh) | (q1 << (16 + sh));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared-memory tile state of one CTA.
struct TileSmem {
    __nv_bfloat16 x[kTok * kXld];            // activations of the chunk, [token][k]
    uint8_t codes[kRows * (kKc / 2 + 16)];   // codes of the chunk, [record][kKc*BITS/8 + 16]
    uint32_t sb[kRows * kGpc];               // {scale, bias} per record and group
    float xs[kTok * kGpc];                   // sum of x per token and group
    int tok[kTok], pos[kTok], slot[kTok];
};

// acc/total: [n-tile][c fragment] of this warp's m16 records x 64 tokens.
// Runs the K loop over `cols` columns: per 256-column chunk the CTA stages
// the activations (rows act_row(i) of `act`, bf16), the codes and {s, b} of
// its kRows records (record r at rec0 + r * rec), and the per-group sums;
// per group of 64 columns the warp issues 4 x 8 MMAs into acc, then folds
// acc into total with the group's affine terms.
template <int BITS, typename ActRow>
__device__ __forceinline__ void gemm_tile(const uint8_t *rec0, size_t rec, int cols, int nrec,
                                          const __nv_bfloat16 *act, int act_ld, ActRow act_row,
                                          const float *gsum, int nt, TileSmem &s,
                                          float (&total)[8][4]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = warp * 16 + (lane >> 2), j = lane & 3;
    const int cbytes = cols * BITS / 8;
    const int ng = cols / kGroup;
    // code bytes of a record per chunk, padded by 16 so that the 8 records a
    // fragment reads fall in 8 different banks
    constexpr int CB = kKc * BITS / 8 + 16;
#pragma unroll
    for (int nti = 0; nti < 8; nti++)
#pragma unroll
        for (int q = 0; q < 4; q++) total[nti][q] = 0.0f;
#pragma unroll 1
    for (int k0 = 0; k0 < cols; k0 += kKc) {
        // the chunk: kc columns (cols is a multiple of 64, kc of the group)
        const int kc = min(kKc, cols - k0), gc = kc / kGroup;
        const int cb16 = kc * BITS / 8 / 16;
        // stage it: activations (16-byte pieces), codes, {s, b}, sums
        for (int i = threadIdx.x; i < kTok * (kc / 8); i += blockDim.x) {
            const int tkn = i / (kc / 8), c8 = i % (kc / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (tkn < nt) v = *reinterpret_cast<const uint4 *>(act + (size_t)act_row(tkn) * act_ld + k0 + c8 * 8);
            *reinterpret_cast<uint4 *>(&s.x[tkn * kXld + c8 * 8]) = v;
        }
        for (int i = threadIdx.x; i < kRows * cb16; i += blockDim.x) {
            const int r = i / cb16, c16 = i % cb16;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < nrec) v = ld_stream16(rec0 + (size_t)r * rec + (size_t)k0 * BITS / 8 + c16 * 16);
            *reinterpret_cast<uint4 *>(&s.codes[r * CB + c16 * 16]) = v;
        }
        for (int i = threadIdx.x; i < kRows * gc; i += blockDim.x) {
            const int r = i / gc, g = i % gc;
            s.sb[r * kGpc + g] = r < nrec ? ld_stream4(rec0 + (size_t)r * rec + cbytes + 4 * (k0 / kGroup + g)) : 0u;
        }
        for (int i = threadIdx.x; i < kTok * gc; i += blockDim.x) {
            const int tkn = i / gc, g = i % gc;
            s.xs[tkn * kGpc + g] = tkn < nt ? gsum[(size_t)act_row(tkn) * ng + k0 / kGroup + g] : 0.0f;
        }
        __syncthreads();
#pragma unroll 1
        for (int g = 0; g < gc; g++) {
            float acc[8][4];
#pragma unroll
            for (int nti = 0; nti < 8; nti++)
#pragma unroll
                for (int q = 0; q < 4; q++) acc[nti][q] = 0.0f;
#pragma unroll
            for (int ks = 0; ks < 4; ks++) {
                const int kb = g * kGroup + ks * 16;            // column within the chunk
                uint32_t a[4];
                a[0] = code_pair<BITS>(s.codes + r0 * CB, kb + 2 * j);
                a[1] = code_pair<BITS>(s.codes + (r0 + 8) * CB, kb + 2 * j);
                a[2] = code_pair<BITS>(s.codes + r0 * CB, kb + 8 + 2 * j);
                a[3] = code_pair<BITS>(s.codes + (r0 + 8) * CB, kb + 8 + 2 * j);
#pragma unroll
                for (int nti = 0; nti < 8; nti++) {
                    const __nv_bfloat16 *xb = &s.x[(nti * 8 + (lane >> 2)) * kXld + kb + 2 * j];
                    const uint32_t b0 = *reinterpret_cast<const uint32_t *>(xb);
                    const uint32_t b1 = *reinterpret_cast<const uint32_t *>(xb + 8);
                    mma_bf16(acc[nti], a, b0, b1);
                }
            }
            // affine terms of the group: s * acc + (b - c s) * sum x
            const float2 sb0 = sb_f(s.sb[r0 * kGpc + g]), sb1 = sb_f(s.sb[(r0 + 8) * kGpc + g]);
            constexpr float off = CodeOff<BITS>::c;
            const float c0 = fmaf(-off, sb0.x, sb0.y), c1 = fmaf(-off, sb1.x, sb1.y);
#pragma unroll
            for (int nti = 0; nti < 8; nti++) {
                const float x0 = s.xs[(nti * 8 + 2 * j) * kGpc + g];
                const float x1 = s.xs[(nti * 8 + 2 * j + 1) * kGpc + g];
                total[nti][0] = fmaf(sb0.x, acc[nti][0], fmaf(c0, x0, total[nti][0]));
                total[nti][1] = fmaf(sb0.x, acc[nti][1], fmaf(c0, x1, total[nti][1]));
                total[nti][2] = fmaf(sb1.x, acc[nti][2], fmaf(c1, x0, total[nti][2]));
                total[nti][3] = fmaf(sb1.x, acc[nti][3], fmaf(c1, x1, total[nti][3]));
            }
        }
        __syncthreads();
    }
}

__device__ __forceinline__ const LoraDev &slot_lora_g(const FfnParams &p, int s, int which) {
    return s < p.K ? p.lora[which] : p.shared_lora[which];
}

// ---------------------------------------------------------------- gate/up
// grid (F / 32, E + has_shared, token tiles); block 128.  CTA: gate/up rows
// f0 .. f0+31 (64 records) of expert blockIdx.y (E = the shared expert) for
// its tokens t0 .. t0+63.  Writes h (bf16) at the tokens' sorted positions.
template <int BITS>
__global__ void __launch_bounds__(kThreads) grouped_gateup_kernel(FfnParams p) {
    extern __shared__ __align__(16) uint8_t smraw[];
    TileSmem &s = *reinterpret_cast<TileSmem *>(smraw);
    const int e = blockIdx.y;
    const int n = e == p.E ? p.T : p.counts[e];
    const int f0 = blockIdx.x * (kRows / 2);
    const int nrec = min(kRows, 2 * (p.F - f0));
    const uint8_t *blob = e == p.E ? p.shared : p.pool + (size_t)e * p.stride;
    const uint8_t *rec0 = blob + p.L.gu_off + (size_t)(2 * f0) * p.L.gu_rec;
    // token tiles t0, t0 + gridDim.z * 64, ...: the grid covers T tokens per
    // expert; an index repeated within a token's K slots gives an expert more
    // than T entries, which the further passes take
#pragma unroll 1
    for (int t0 = blockIdx.z * kTok; t0 < n; t0 += gridDim.z * kTok) {
        const int nt = min(kTok, n - t0);
        __syncthreads();
        tile_tokens(p, e, t0, nt, s.tok, s.pos, s.slot);
        __syncthreads();
        float total[8][4];
        gemm_tile<BITS>(rec0, p.L.gu_rec, p.d, nrec, p.xb, p.d, [&](int i) { return s.tok[i]; },
                        p.xsum, nt, s, total);
        // epilogue: record 16 w + lane/4 (+8); even records are gate rows, odd
        // ones up rows (their values sit 4 lanes further)
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, j = lane & 3;
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const int rl = warp * 16 + (lane >> 2) + half * 8;      // record within the tile
            const int f = f0 + rl / 2;
            const bool gate = (rl & 1) == 0;
#pragma unroll
            for (int nti = 0; nti < 8; nti++)
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    const float gv = total[nti][half * 2 + c];
                    const float uv = __shfl_down_sync(0xffffffffu, gv, 4);
                    const int i = nti * 8 + 2 * j + c;
                    if (!gate || i >= nt || rl >= nrec) continue;
                    float g = gv, u = uv;
                    const int sl = s.slot[i], t = s.tok[i];
                    const LoraDev &lg = slot_lora_g(p, sl, 0), &lu = slot_lora_g(p, sl, 1);
                    if (lg.r || lu.r) {
                        const int ee = sl < p.K ? p.idx[(size_t)t * p.K + sl] : 0;
                        const float *v = p.v + ((size_t)t * p.slots + sl) * 3 * kMaxLoraRank;
                        if (lg.r) {
                            const uint16_t *B = lg.B + (sl < p.K ? (size_t)ee * lg.b_stride : 0) + (size_t)f * lg.r;
                            float a = 0.0f;
                            for (int k = 0; k < lg.r; k++) a = fmaf(half_f(B[k]), v[k], a);
                            g += lg.scale * a;
                        }
                        if (lu.r) {
                            const uint16_t *B = lu.B + (sl < p.K ? (size_t)ee * lu.b_stride : 0) + (size_t)f * lu.r;
                            float a = 0.0f;
                            for (int k = 0; k < lu.r; k++) a = fmaf(half_f(B[k]), v[kMaxLoraRank + k], a);
                            u += lu.scale * a;
                        }
                    }
                    const float h = silu_f(g) * u;
                    p.h16[(size_t)s.pos[i] * p.F + f] = __float2bfloat16_rn(h);
                }
        }
    }
}

// ---------------------------------------------------------------- down
// grid (d / 64, E + has_shared, token tiles); block 128.  CTA: down rows
// o0 .. o0+63 of expert blockIdx.y for its tokens; writes y_slots.
template <int BITS>
__global__ void __launch_bounds__(kThreads) grouped_down_kernel(FfnParams p) {
    extern __shared__ __align__(16) uint8_t smraw[];
    TileSmem &s = *reinterpret_cast<TileSmem *>(smraw);
    const int e = blockIdx.y;
    const int n = e == p.E ? p.T : p.counts[e];
    const int o0 = blockIdx.x * kRows;
    const int nrec = min(kRows, p.d - o0);
    const uint8_t *blob = e == p.E ? p.shared : p.pool + (size_t)e * p.stride;
    const uint8_t *rec0 = blob + p.L.down_off + (size_t)o0 * p.L.down_rec;
#pragma unroll 1
    for (int t0 = blockIdx.z * kTok; t0 < n; t0 += gridDim.z * kTok) {
        const int nt = min(kTok, n - t0);
        __syncthreads();
        tile_tokens(p, e, t0, nt, s.tok, s.pos, s.slot);
        __syncthreads();
        float total[8][4];
        gemm_tile<BITS>(rec0, p.L.down_rec, p.F, nrec, p.h16, p.F, [&](int i) { return s.pos[i]; },
                        p.hsum, nt, s, total);
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, j = lane & 3;
#pragma unroll
        for (int half = 0; half < 2; half++) {
            const int rl = warp * 16 + (lane >> 2) + half * 8;
            const int o = o0 + rl;
            if (rl >= nrec) continue;
#pragma unroll
            for (int nti = 0; nti < 8; nti++)
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    const int i = nti * 8 + 2 * j + c;
                    if (i >= nt) continue;
                    float y = total[nti][half * 2 + c];
                    const int sl = s.slot[i], t = s.tok[i];
                    const LoraDev &ld = slot_lora_g(p, sl, 2);
                    if (ld.r) {
                        const int ee = sl < p.K ? p.idx[(size_t)t * p.K + sl] : 0;
                        const uint16_t *B = ld.B + (sl < p.K ? (size_t)ee * ld.b_stride : 0) + (size_t)o * ld.r;
                        const float *vd = p.vd + (size_t)s.pos[i] * kMaxLoraRank;
                        float a = 0.0f;
                        for (int k = 0; k < ld.r; k++) a = fmaf(half_f(B[k]), vd[k], a);
                        y += ld.scale * a;
                    }
                    p.y[((size_t)t * p.slots + sl) * p.d + o] = y;
                }
        }
    }
}

// vd[pos][i] = sum_f A_d[i][f] h[pos][f] for every sorted position whose
// slot has a down LoRA.  One warp per (position, i).
__global__ void __launch_bounds__(256) lora_down_ax_kernel(FfnParams p, int npos) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (w >= npos * kMaxLoraRank) return;
    const int ps = w / kMaxLoraRank, i = w % kMaxLoraRank;
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
    const int nb = (p.E + 1 + 7) / 8;           // one warp per bucket, 8 warps per CTA
    sort_count_kernel<<<nb, 256, 0, st>>>(p.idx, TK, p.E, p.counts);
    if (int rc = check_launch("sort_count_kernel")) return rc;
    sort_scatter_kernel<<<nb, 256, 0, st>>>(p.idx, TK, p.E, p.counts, p.offsets, p.perm);
    if (int rc = check_launch("sort_scatter_kernel")) return rc;
    invalid_fill_kernel<<<64, 256, 0, st>>>(p.offsets, p.perm, p.E, p.K, p.slots, p.d, p.y);
    if (int rc = check_launch("invalid_fill_kernel")) return rc;
    {
        const int warps = p.T * (p.d / kGroup);
        group_sums_kernel<<<(warps + 7) / 8, 256, 0, st>>>(p.xb, p.T, p.d, p.xsum);
        if (int rc = check_launch("group_sums_kernel")) return rc;
    }
    if (p.any_gu_lora) {
        lora_ax_kernel_launch(p, st);
        if (int rc = check_launch("lora_ax_kernel")) return rc;
    }
    const int ntile = (p.T + kTok - 1) / kTok;  // the shared expert has T tokens, an expert at most T
    const int groups = p.E + (p.shared ? 1 : 0);
    const size_t smem = sizeof(TileSmem);
    cudaFuncSetAttribute(grouped_gateup_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(grouped_down_kernel<BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    grouped_gateup_kernel<BITS><<<dim3((p.F + kRows / 2 - 1) / (kRows / 2), groups, ntile), kThreads, smem, st>>>(p);
    if (int rc = check_launch("grouped_gateup_kernel")) return rc;
    const int npos = TK + (p.shared ? p.T : 0);
    {
        const int warps = npos * (p.F / kGroup);
        group_sums_kernel<<<(warps + 7) / 8, 256, 0, st>>>(p.h16, npos, p.F, p.hsum);
        if (int rc = check_launch("group_sums_kernel")) return rc;
    }
    if (p.lora[2].r || p.shared_lora[2].r) {
        const int warps = npos * kMaxLoraRank;
        lora_down_ax_kernel<<<(warps + 7) / 8, 256, 0, st>>>(p, npos);
        if (int rc = check_launch("lora_down_ax_kernel")) return rc;
    }
    grouped_down_kernel<BITS><<<dim3((p.d + kRows - 1) / kRows, groups, ntile), kThreads, smem, st>>>(p);
    return check_launch("grouped_down_kernel");
}

}  // namespace grouped

int launch_expert_ffn_grouped(const FfnParams &p, cudaStream_t st) {
    return p.bits == 4 ? grouped::launch_bits<4>(p, st) : grouped::launch_bits<2>(p, st);
}

}  // namespace moe
