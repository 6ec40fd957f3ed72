// step_common.cuh -- device primitives of the persistent decode-step kernel:
// mbarriers, bulk copies into shared memory, tagged (value, tag) words for
// dataflow between CTAs, bounded waits, and the paired-fp32 dequant dot.
#pragma once

#include "internal.h"

namespace moe {
namespace step {

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Tagged word: high 32 bits = tag, low 32 bits = fp32 value.  Written and read
// as single 64-bit accesses, so a reader sees either the old word or the new
// one whole; the tag doubles as the "ready" flag of the value.
__device__ __forceinline__ void put_tagged(uint64_t *p, uint32_t tag, float v) {
    const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ uint64_t get_word(const uint64_t *p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

__device__ __forceinline__ int ld_flag(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---------------------------------------------------------------- dequant dot
// x is kept pre-scaled and transposed in shared memory so that codes can be
// turned into floats without shifts: a code n at bit offset 4j (or 2j) of a
// word, OR-ed into the mantissa of 2^23, is the float 2^23 + n*16^j (4^j);
// subtracting 2^23 is exact, and multiplying by x*16^-j (4^-j) gives n*x with
// one rounding, the same as n*x.  Codes are handled in pairs with the paired
// fp32 instructions of sm_100+.
//
// Pre-scaled layout of one vector of n floats split in 16-byte chunks c of
// VALS = 128/BITS codes: float4 group q (0 .. VALS/4-1) of chunk c sits at
// float4 index q*nch + c (nch = n / VALS), so the lanes of a warp, each on its
// own chunk, read consecutive 16-byte words (no bank conflicts).
//   int4: word i (0..3), pair slot jj (0..1):  float4 q = 2i + jj holds
//         (x[8i+2jj]*16^-2jj, x[8i+2jj+4]*16^-2jj,
//          x[8i+2jj+1]*16^-(2jj+1), x[8i+2jj+5]*16^-(2jj+1)).
//   int2: word i (0..3), pair slot jj (0..3):  float4 q = 4i + jj holds
//         (x[16i+2jj]*4^-2jj, x[16i+2jj+8]*4^-2jj,
//          x[16i+2jj+1]*4^-(2jj+1), x[16i+2jj+9]*4^-(2jj+1)).

// float index of vector position `pos` in the pre-scaled layout
template <int BITS>
__device__ __forceinline__ int ps_index(int pos, int nch) {
    constexpr int VALS = 128 / BITS;
    const int c = pos / VALS, r = pos % VALS;
    if (BITS == 4) {
        const int i = r / 8, p = r % 8;          // word, position in word
        const int j = p & 3, hi = p >> 2;        // pair index j, second of pair
        const int q = 2 * i + (j >> 1);
        const int lane = (j & 1) * 2 + hi;       // (j even: x,y) (j odd: z,w)
        return (q * nch + c) * 4 + lane;
    } else {
        const int i = r / 16, p = r % 16;
        const int j = p & 7, hi = p >> 3;
        const int q = 4 * i + (j >> 1);
        const int lane = (j & 1) * 2 + hi;
        return (q * nch + c) * 4 + lane;
    }
}

template <int BITS>
__device__ __forceinline__ float ps_scale(int pos) {
    if (BITS == 4) return __uint_as_float((uint32_t)(127 - 4 * (pos % 8 & 3)) << 23);
    return __uint_as_float((uint32_t)(127 - 2 * (pos % 16 & 7)) << 23);
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
    return ((uint64_t)hi << 32) | lo;
}

__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ float f2_sum(uint64_t a) {
    return __uint_as_float((uint32_t)a) + __uint_as_float((uint32_t)(a >> 32));
}

constexpr uint32_t kMagic = 0x4B000000u;                       // 2^23
constexpr uint64_t kMagic2 = 0x4B0000004B000000ull;

// Accumulates the dot products of two code chunks (two rows) with one
// pre-scaled x chunk: acc0 += codes(q0) . x, acc1 += codes(q1) . x.
// xq: float4 pointer to group 0 of this chunk; groups are nch apart.
template <int BITS, int NR>
__device__ __forceinline__ void chunk_dot_ps(const uint4 *q, const float4 *xq, int nch,
                                             uint64_t *acc) {
    constexpr int PAIRS = BITS == 4 ? 4 : 8;           // pairs per word
    constexpr uint32_t M = (1u << BITS) - 1u;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        uint32_t w[NR], wh[NR];
#pragma unroll
        for (int r = 0; r < NR; r++) {
            const uint32_t *qq = reinterpret_cast<const uint32_t *>(&q[r]);
            w[r] = qq[i];
            wh[r] = qq[i] >> 16;
        }
#pragma unroll
        for (int jj = 0; jj < PAIRS / 2; jj++) {
            const float4 xv = xq[(size_t)(i * (PAIRS / 2) + jj) * nch];
            const uint64_t x0 = pack2(__float_as_uint(xv.x), __float_as_uint(xv.y));
            const uint64_t x1 = pack2(__float_as_uint(xv.z), __float_as_uint(xv.w));
            const int j0 = 2 * jj, j1 = 2 * jj + 1;
#pragma unroll
            for (int r = 0; r < NR; r++) {
                const uint64_t c0 = pack2((w[r] & (M << (BITS * j0))) | kMagic,
                                          (wh[r] & (M << (BITS * j0))) | kMagic);
                const uint64_t c1 = pack2((w[r] & (M << (BITS * j1))) | kMagic,
                                          (wh[r] & (M << (BITS * j1))) | kMagic);
                acc[r] = f2_fma(f2_sub(c0, kMagic2), x0, acc[r]);
                acc[r] = f2_fma(f2_sub(c1, kMagic2), x1, acc[r]);
            }
        }
    }
}

}  // namespace step
}  // namespace moe
