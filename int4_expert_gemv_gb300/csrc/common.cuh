// common.cuh -- layout, decode and load helpers shared by the sm_103a kernels.
//
// Packed weight records (one per matrix row): the row's codes (cols*bits/8
// bytes, little-endian uint32 words, element j of a word at bits
// [bits*j, bits*j+bits)), then one {fp16 scale, fp16 bias} pair per group of
// 64 columns, then zero padding to a multiple of 16 bytes.  The decoded weight
// is code*scale + bias: the affine dequantisation of the Metal fragment in
// "Inferencia de LLM MoE en MacBook Pro: Streaming de Expertos desde SSD con
// Metal" (kerneldigest.dev), "Arquitectura del Sistema".
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

constexpr int kGroup = 64;           // quantisation group along the input dim
constexpr int kChunk = 16;           // bytes per vector load
constexpr int kMaxSlots = 17;        // K <= 16 routed experts + 1 shared
constexpr int kMaxCacheSlots = 1024; // slots of one layer's expert cache
constexpr int kMaxLoraRank = 64;

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) {
    return (v + a - 1) / a * a;
}

// Bytes of the codes of one row.
__host__ __device__ constexpr size_t code_bytes(int cols, int bits) {
    return (size_t)cols * bits / 8;
}

__host__ __device__ constexpr size_t record_bytes(int cols, int bits) {
    return align_up(code_bytes(cols, bits) + (size_t)(cols / kGroup) * 4, kChunk);
}

// Layout of one expert blob: gate/up section (2F records of d columns, gate
// row f at record 2f, up row f at 2f+1) then the down section (d records of
// F columns); each section 256-byte aligned.
struct BlobLayout {
    size_t gu_rec, down_rec;     // record sizes
    size_t gu_off, down_off;     // section offsets
    size_t bytes;                // whole blob
};

__host__ __device__ inline BlobLayout blob_layout(int d, int F, int bits) {
    BlobLayout L;
    L.gu_rec = record_bytes(d, bits);
    L.down_rec = record_bytes(F, bits);
    L.gu_off = 0;
    L.down_off = align_up(2 * (size_t)F * L.gu_rec, 256);
    L.bytes = L.down_off + align_up((size_t)d * L.down_rec, 256);
    return L;
}

// ---------------------------------------------------------------- loads
// Streaming 16-byte load of weights: read once, keep out of L1.
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream4(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Exact float of a small unsigned code: the code placed in the mantissa of
// 2^23, minus 2^23.
__device__ __forceinline__ float code_f(uint32_t n) {
    return __uint_as_float(0x4B000000u | n) - 8388608.0f;
}

// {scale, bias} pair of a group, stored as two fp16 in one 32-bit word.
__device__ __forceinline__ float2 sb_f(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
}

// Dot product of one 16-byte chunk of codes with the matching x values
// (128/BITS consecutive floats in shared memory).
template <int BITS>
__device__ __forceinline__ float chunk_dot(uint4 q, const float *x) {
    constexpr int PER = 32 / BITS;
    constexpr uint32_t M = (1u << BITS) - 1u;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        a[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < PER; j++)
            a[i] = fmaf(code_f((w[i] >> (BITS * j)) & M), x[i * PER + j], a[i]);
    }
    return (a[0] + a[1]) + (a[2] + a[3]);
}

// Dot product of 8 fp16 weights (one 16-byte chunk) with 8 floats.
__device__ __forceinline__ float chunk_dot_f16(uint4 q, const float *x) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float a = 0.0f, b = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        a = fmaf(f.x, x[2 * i], a);
        b = fmaf(f.y, x[2 * i + 1], b);
    }
    return a + b;
}

__device__ __forceinline__ float warp_sum(float v, int width) {
    for (int o = width / 2; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float load_act(const void *x, int dtype, size_t i) {
    return dtype == MOE_DTYPE_F32 ? static_cast<const float *>(x)[i]
                                  : __bfloat162float(static_cast<const __nv_bfloat16 *>(x)[i]);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ float gelu_erf_f(float a) {
    return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f));
}

__device__ __forceinline__ float half_f(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// ---------------------------------------------------------------- errors
// Records a detail for moe_last_error() and returns `code`.
int fail(int code, const char *fmt, ...);
int check_launch(const char *what);

}  // namespace moe
