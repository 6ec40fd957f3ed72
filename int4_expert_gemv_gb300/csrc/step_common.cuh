// step_common.cuh -- device primitives of the persistent decode-step kernel:
// mbarriers, bulk copies into shared memory, tagged (value, tag) words for
// dataflow between CTAs, bounded waits, and the fixed-point dequant dot.
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

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may stay suspended up to `hint_ns` (it is
// woken as soon as the phase completes), so a waiting warp does not spin.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Orders this thread's generic-proxy view of global memory (e.g. what an
// acquire just made visible) before its later async-proxy (bulk copy) reads.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
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

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Publishes a ready flag after this thread's (and, through the fences the
// other warps executed before handing over, the CTA's) earlier global writes.
__device__ __forceinline__ void put_flag(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_flag(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// ---------------------------------------------------------------- dequant dot
// Integer dot products.  A vector x (x, h or gelu(a)) is staged per 16-byte
// code chunk c (VALS = 128/BITS values) as 16-bit fixed point with one
// power-of-two scale: xf = rint(x * 2^(15-e)), e the exponent of the chunk's
// largest |x| (2^(e-1) <= max < 2^e), clamped to [-32767, 32767]; xf is split
// into a signed high byte and an unsigned low byte (xf = 256 hi + lo).  A
// packed code word is cut into byte vectors of 4 codes with one mask (and a
// shift), and dp4a accumulates sum(code * hi) and sum(code * lo) exactly in
// int32.  The chunk's sum(code * xf) = 256 HI + LO is below 2^24, so its float
// and the product with 2^(e-15) are exact: the chunk dot is exactly
// codes . x^ with |x - x^| <= 2^(e-16) <= max|x| * 2^-15.
//
// Layout of one staged vector (nch chunks): the 4-code byte vectors of word i
// of a chunk are, for int4, A = positions 8i+{0,2,4,6} and B = 8i+{1,3,5,7};
// for int2, group g (0..3) = positions 16i + 4b + g (b = 0..3).  Their
// (hi, lo) words sit in uint4 slot k of chunk c at uint4 index k*nch + c
// (k = i for int4 as (A_hi, A_lo, B_hi, B_lo); k = 2i + g/2 for int2 as
// (G_hi, G_lo, G'_hi, G'_lo)), so lanes on consecutive chunks read consecutive
// 16-byte words.  Per chunk also: scale 2^(e-15) and xhat = sum(x^).

template <int BITS>
struct Fix {
    static constexpr int VALS = 128 / BITS;          // values per chunk
    static constexpr int SLOTS = BITS == 4 ? 4 : 8;  // uint4 per chunk
};

// uint4 slot and byte offset (within the uint4) of position pos of a chunk,
// for the high byte (the low byte is 4 bytes further).
template <int BITS>
__device__ __forceinline__ void fix_place(int pos, int &slot, int &byte) {
    if (BITS == 4) {
        const int i = pos >> 3, p = pos & 7;
        slot = i;
        byte = ((p & 1) ? 8 : 0) + (p >> 1);
    } else {
        const int i = pos >> 4, p = pos & 15, g = p & 3, b = p >> 2;
        slot = 2 * i + (g >> 1);
        byte = ((g & 1) ? 8 : 0) + b;
    }
}

// Stages one chunk whose values are spread over the 32 lanes of a warp
// (lane j holds positions j and, for int2, j + 32): writes the fixed-point
// bytes into xf (uint4 array, chunk c of nch), the scale and xhat.
template <int BITS>
__device__ __forceinline__ void stage_chunk(const float *v, int lane, uint8_t *xf, int c, int nch,
                                            float *scale, float *xhat) {
    constexpr int PER = Fix<BITS>::VALS / 32;
    // max |v| over the warp: the bit patterns of non-negative floats order
    // like the values
    uint32_t mb = 0;
#pragma unroll
    for (int k = 0; k < PER; k++) mb = max(mb, __float_as_uint(fabsf(v[k])));
    mb = __reduce_max_sync(0xffffffffu, mb);
    // e: 2^(e-1) <= m < 2^e; f = 2^(15-e) exactly; zero or subnormal m: all zero
    const bool nz = (mb >> 23) != 0;
    const int e = nz ? (int)((mb >> 23) & 0xff) - 126 : 0;
    const float f = nz ? __uint_as_float((uint32_t)(127 + 15 - e) << 23) : 0.0f;
    int sum = 0;
#pragma unroll
    for (int k = 0; k < PER; k++) {
        int q = (int)rintf(v[k] * f);
        q = max(-32767, min(32767, q));
        sum += q;
        const int pos = lane + 32 * k;
        int slot, byte;
        fix_place<BITS>(pos, slot, byte);
        uint8_t *w = xf + ((size_t)slot * nch + c) * 16;
        w[byte] = (uint8_t)((q >> 8) & 0xff);
        w[byte + 4] = (uint8_t)(q & 0xff);
    }
    sum = __reduce_add_sync(0xffffffffu, sum);
    if (lane == 0) {
        const float sc = nz ? __uint_as_float((uint32_t)(127 + e - 15) << 23) : 0.0f;
        scale[c] = sc;
        xhat[c] = (float)sum * sc;
    }
}

__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Exact codes . x^ of NR code chunks (NR rows) against one staged chunk:
// out[r] = (256 HI + LO) without the chunk scale.  xq: uint4 array of the
// staged vector, indexed slot*nch + c (this lane's chunk c).
template <int BITS, int NR>
__device__ __forceinline__ void chunk_dot_fix(const uint4 *q, const uint4 *xq, int nch, int c,
                                              int *out) {
    int hi[NR], lo[NR];
#pragma unroll
    for (int r = 0; r < NR; r++) hi[r] = lo[r] = 0;
    if (BITS == 4) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint4 xv = xq[i * nch + c];
#pragma unroll
            for (int r = 0; r < NR; r++) {
                const uint32_t w = (&q[r].x)[i];
                const uint32_t ca = w & 0x0F0F0F0Fu, cb = (w >> 4) & 0x0F0F0F0Fu;
                hi[r] = dp4a_us(ca, xv.x, hi[r]);
                lo[r] = dp4a_uu(ca, xv.y, lo[r]);
                hi[r] = dp4a_us(cb, xv.z, hi[r]);
                lo[r] = dp4a_uu(cb, xv.w, lo[r]);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; i++) {
#pragma unroll
            for (int h2 = 0; h2 < 2; h2++) {
                const uint4 xv = xq[(2 * i + h2) * nch + c];
#pragma unroll
                for (int r = 0; r < NR; r++) {
                    const uint32_t w = (&q[r].x)[i];
                    const uint32_t c0 = (w >> (4 * h2)) & 0x03030303u;
                    const uint32_t c1 = (w >> (4 * h2 + 2)) & 0x03030303u;
                    hi[r] = dp4a_us(c0, xv.x, hi[r]);
                    lo[r] = dp4a_uu(c0, xv.y, lo[r]);
                    hi[r] = dp4a_us(c1, xv.z, hi[r]);
                    lo[r] = dp4a_uu(c1, xv.w, lo[r]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; r++) out[r] = hi[r] * 256 + lo[r];
}

}  // namespace step
}  // namespace moe
