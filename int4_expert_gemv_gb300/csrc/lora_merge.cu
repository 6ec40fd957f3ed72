// lora_merge.cu -- merges a LoRA delta into packed records and requantises
// them in place or into a copy: W' = requantise(W + scale B A), group by group
// in the same affine form.  This is the merged alternative to the unfused
// adapter of "La otra mitad del muro de la memoria" (xyznot.com/es/paper/
// 2609.18063), section "Ejecucion del adaptador no fusionado", which keeps the
// adapter unfused because requantising the merged weights keeps little of its
// delta; the call exists to measure how little.
//
// The new codes are integers decided by floating point, so the arithmetic is
// fixed step by step in binary32 (every operation rounded to nearest even):
// for row o, group g, column k of the group
//     d_k = sum_{j<r} B[o][j] A[j][k]        (fmaf chain, j ascending, from 0)
//     w_k = fmaf(scale, d_k, fmaf(q_k, s, b))
//     s'  = f16((max w - min w) / (2^bits - 1)),  b' = f16(min w)
//     q'_k = s' == 0 ? 0 : clamp(rint((w_k - b') / s'), 0, 2^bits - 1)
#include "internal.h"

#include <cuda_fp16.h>

namespace moe {

namespace {

__device__ __forceinline__ float f16f(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ uint16_t f16bits(float v) { return __half_as_ushort(__float2half_rn(v)); }

// One warp per (row, group): lane l holds columns 2l and 2l + 1 of the group.
template <int BITS>
__global__ void __launch_bounds__(256) merge_lora_kernel(const uint8_t *src, size_t src_stride,
                                                         int rows, int cols, const uint16_t *A,
                                                         const uint16_t *B, int r, float scale,
                                                         uint8_t *dst, size_t dst_stride) {
    constexpr uint32_t kMax = (1u << BITS) - 1u;
    const int ng = cols / kGroup, lane = threadIdx.x & 31;
    const long long unit = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (unit >= (long long)rows * ng) return;                    // whole warp
    const int o = (int)(unit / ng), g = (int)(unit - (long long)o * ng);
    const uint8_t *rec = src + (size_t)o * src_stride;
    uint8_t *out = dst + (size_t)o * dst_stride;
    const size_t cb = code_bytes(cols, BITS);
    // codes of this lane's two columns (little-endian words: byte i of a group
    // holds 8 / BITS consecutive columns, the lowest in the low bits)
    uint32_t c0, c1;
    if (BITS == 4) {
        const uint32_t v = rec[(size_t)g * 32 + lane];
        c0 = v & 15u;
        c1 = v >> 4;
    } else {
        const uint32_t v = rec[(size_t)g * 16 + (lane >> 1)];
        const int sh = 4 * (lane & 1);
        c0 = (v >> sh) & 3u;
        c1 = (v >> (sh + 2)) & 3u;
    }
    const uint32_t sbw = *reinterpret_cast<const uint32_t *>(rec + cb + 4 * (size_t)g);
    const float s = f16f((uint16_t)(sbw & 0xffffu)), b = f16f((uint16_t)(sbw >> 16));
    const int k0 = g * kGroup + 2 * lane;
    // A columns k0, k0 + 1 as one 32-bit word per j; loads batched ahead of
    // the (ascending-j) fma chains
    const uint32_t *A2 = reinterpret_cast<const uint32_t *>(A) + k0 / 2;
    const uint16_t *Bo = B + (size_t)o * r;
    float d0 = 0.0f, d1 = 0.0f;
    int j = 0;
    for (; j + 8 <= r; j += 8) {
        uint32_t a[8];
        uint16_t bb[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            a[i] = A2[(size_t)(j + i) * (cols / 2)];
            bb[i] = Bo[j + i];
        }
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const float bj = f16f(bb[i]);
            d0 = fmaf(bj, f16f((uint16_t)(a[i] & 0xffffu)), d0);
            d1 = fmaf(bj, f16f((uint16_t)(a[i] >> 16)), d1);
        }
    }
    for (; j < r; j++) {
        const uint32_t a = A2[(size_t)j * (cols / 2)];
        const float bj = f16f(Bo[j]);
        d0 = fmaf(bj, f16f((uint16_t)(a & 0xffffu)), d0);
        d1 = fmaf(bj, f16f((uint16_t)(a >> 16)), d1);
    }
    const float w0 = fmaf(scale, d0, fmaf((float)c0, s, b));
    const float w1 = fmaf(scale, d1, fmaf((float)c1, s, b));
    float lo = fminf(w0, w1), hi = fmaxf(w0, w1);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, m));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, m));
    }
    const uint16_t s2 = f16bits(__fdiv_rn(__fsub_rn(hi, lo), (float)kMax));
    const uint16_t b2 = f16bits(lo);
    const float sf = f16f(s2), bf = f16f(b2);
    auto code = [&](float w) -> uint32_t {
        if (sf == 0.0f) return 0u;
        const float t = rintf(__fdiv_rn(__fsub_rn(w, bf), sf));
        return t <= 0.0f ? 0u : (t >= (float)kMax ? kMax : (uint32_t)t);
    };
    const uint32_t q0 = code(w0), q1 = code(w1);
    // every lane has read its group before any lane writes (in-place safe:
    // no other warp touches this group's bytes)
    __syncwarp();
    if (BITS == 4) {
        out[(size_t)g * 32 + lane] = (uint8_t)(q0 | (q1 << 4));
    } else {
        const uint32_t nib = q0 | (q1 << 2);
        const uint32_t hi_nib = __shfl_down_sync(0xffffffffu, nib, 1);
        if ((lane & 1) == 0) out[(size_t)g * 16 + (lane >> 1)] = (uint8_t)(nib | (hi_nib << 4));
    }
    if (lane == 0)
        *reinterpret_cast<uint32_t *>(out + cb + 4 * (size_t)g) = (uint32_t)s2 | ((uint32_t)b2 << 16);
    // the record's zero padding (a copy into a fresh buffer stays a valid record)
    if (g == 0) {
        const size_t used = cb + 4 * (size_t)ng, rec_b = record_bytes(cols, BITS);
        if (used + lane < rec_b) out[used + lane] = 0;
    }
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_merge_lora(const void *src, size_t src_stride, int rows, int cols, int bits,
                              const uint16_t *A, const uint16_t *B, int r, float scale, void *dst,
                              size_t dst_stride, cudaStream_t stream) {
    if (bits != 2 && bits != 4) return fail(MOE_EINVAL, "merge_lora: bits=%d (2 or 4)", bits);
    if (cols <= 0 || cols % kGroup) return fail(MOE_EINVAL, "merge_lora: cols=%d (a multiple of 64)", cols);
    if (rows < 0) return fail(MOE_EINVAL, "merge_lora: rows=%d", rows);
    if (r < 0 || r > 1024) return fail(MOE_EINVAL, "merge_lora: r=%d (0..1024)", r);
    if (r > 0 && (A == nullptr || B == nullptr || reinterpret_cast<uintptr_t>(A) % 4))
        return fail(MOE_EINVAL, "merge_lora: r > 0 with NULL (or not 4-byte aligned) A or B");
    if (rows == 0) return MOE_OK;
    if (src == nullptr || dst == nullptr) return fail(MOE_EINVAL, "merge_lora: NULL records");
    const size_t rec = record_bytes(cols, bits);
    if (src_stride < rec || dst_stride < rec || src_stride % 16 || dst_stride % 16 ||
        reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16)
        return fail(MOE_EINVAL, "merge_lora: strides %zu / %zu (>= %zu, multiples of 16) or "
                                "unaligned records", src_stride, dst_stride, rec);
    const long long units = (long long)rows * (cols / kGroup);
    const long long blocks = (units + 7) / 8;
    if (blocks > 0x7fffffffLL) return fail(MOE_EINVAL, "merge_lora: %lld groups", units);
    const uint8_t *s8 = static_cast<const uint8_t *>(src);
    uint8_t *d8 = static_cast<uint8_t *>(dst);
    if (bits == 4)
        merge_lora_kernel<4><<<(unsigned)blocks, 256, 0, stream>>>(s8, src_stride, rows, cols, A, B, r,
                                                                    scale, d8, dst_stride);
    else
        merge_lora_kernel<2><<<(unsigned)blocks, 256, 0, stream>>>(s8, src_stride, rows, cols, A, B, r,
                                                                    scale, d8, dst_stride);
    return check_launch("merge_lora_kernel");
}
