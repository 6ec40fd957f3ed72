// synth.cu -- GPU twin of the seeded synthetic-input generator (synth.py).
//
// Data only: it draws weights and activations and quantises them into the
// logical storage format; it holds none of the MoE layer's arithmetic and
// shares no code with the layer's kernels.  Every step is an exact integer
// operation or a single IEEE fp32 rounding, so the output equals the numpy
// twin bit for bit.
//
// Generator: SplitMix64 finaliser (Steele, Lea & Flood, OOPSLA 2014) over the
// counter key + (i+1)*0x9E3779B97F4A7C15; Gaussian values are Irwin-Hall sums
// of the four 16-bit fields of each word, centred and scaled once in fp32.
#include <cstdint>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__device__ __forceinline__ float gauss_at(uint64_t key, uint64_t i, float scale) {
    const uint64_t r = mix(key + (i + 1) * kGolden);
    const int s = (int)(r & 0xFFFF) + (int)((r >> 16) & 0xFFFF) + (int)((r >> 32) & 0xFFFF) +
                  (int)((r >> 48) & 0xFFFF) - 131070;
    return __fmul_rn((float)s, scale);
}

__global__ void gauss_f32_kernel(uint64_t key, uint64_t n, float scale, float *out) {
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
         i += (uint64_t)gridDim.x * blockDim.x)
        out[i] = gauss_at(key, i, scale);
}

__global__ void gauss_f16_kernel(uint64_t key, uint64_t n, float scale, __half *out) {
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
         i += (uint64_t)gridDim.x * blockDim.x)
        out[i] = __float2half_rn(gauss_at(key, i, scale));
}

// One thread per (row, group of 64): draw, min/max quantise, pack.
__global__ void affine_kernel(uint64_t key, int rows, int cols, int bits, float scale,
                              uint32_t *q, __half *s, __half *b) {
    const int groups = cols / 64;
    const uint64_t n = (uint64_t)rows * groups;
    const float levels = (float)((1 << bits) - 1);
    const int per = 32 / bits;
    for (uint64_t gi = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; gi < n;
         gi += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t row = gi / groups, g = gi % groups;
        const uint64_t first = row * cols + g * 64;
        float w[64];
        float mn = INFINITY, mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; j++) {
            w[j] = gauss_at(key, first + j, scale);
            mn = fminf(mn, w[j]);
            mx = fmaxf(mx, w[j]);
        }
        const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), levels));
        const __half b16 = __float2half_rn(mn);
        const float sf = __half2float(s16), bf = __half2float(b16);
        s[gi] = s16;
        b[gi] = b16;
        uint32_t *qw = q + (row * cols + g * 64) * bits / 32;
        for (int wi = 0; wi < 64 / per; wi++) {
            uint32_t word = 0;
            for (int j = 0; j < per; j++) {
                float c = 0.0f;
                if (sf > 0.0f)
                    c = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(w[wi * per + j], bf), sf)), 0.0f),
                              levels);
                word |= (uint32_t)c << (bits * j);
            }
            qw[wi] = word;
        }
    }
}

int grid_for(uint64_t n) {
    uint64_t b = (n + 255) / 256;
    return (int)(b < 65536 ? (b ? b : 1) : 65536);
}

}  // namespace

extern "C" {

// fp32 near-Gaussian values out[0..n) of stream `key` (scale = sigma/37837.227).
int synth_gauss_f32(uint64_t key, uint64_t n, float scale, float *out, cudaStream_t st) {
    gauss_f32_kernel<<<grid_for(n), 256, 0, st>>>(key, n, scale, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// The same values rounded to fp16 (round to nearest even).
int synth_gauss_f16(uint64_t key, uint64_t n, float scale, void *out, cudaStream_t st) {
    gauss_f16_kernel<<<grid_for(n), 256, 0, st>>>(key, n, scale, static_cast<__half *>(out));
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

// A [rows][cols] matrix drawn from stream `key` and min/max quantised per
// group of 64: q uint32 [rows][cols*bits/32], s and b fp16 [rows][cols/64].
int synth_affine(uint64_t key, int rows, int cols, int bits, float scale, uint32_t *q,
                 void *s, void *b, cudaStream_t st) {
    if (cols % 64 || (bits != 2 && bits != 4) || rows <= 0) return 1;
    affine_kernel<<<grid_for((uint64_t)rows * (cols / 64)), 256, 0, st>>>(
        key, rows, cols, bits, scale, q, static_cast<__half *>(s), static_cast<__half *>(b));
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

}  // extern "C"
