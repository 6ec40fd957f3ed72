// gather.cu -- copies the blobs of a layer's routed experts out of an expert
// pool that may live outside HBM (pinned host memory, which the GPU reads
// directly over NVLink-C2C on a Grace machine) into HBM slots, with the
// route rewritten to the slots.  The route comes from device memory, so the
// copy needs no host round trip and can run a whole token ahead: the routes of
// token t are predicted during token t-1 ("La otra mitad del muro de la
// memoria", xyznot.com/es/paper/2609.18063, "Ideas clave": the predicted route
// is the routing, which is what makes prefetching the experts possible).
#include "internal.h"

#include <algorithm>

namespace moe {

namespace {

// grid (n, parts): CTA (i, p) copies the p-th share of expert idx[i]'s blob
// in 16-byte words; CTA (i, 0) writes slot_idx[i].
__global__ void __launch_bounds__(256) gather_experts_kernel(const uint8_t *pool, size_t stride, int E,
                                                             const int32_t *idx, size_t blob_bytes,
                                                             uint8_t *slots, size_t slot_stride,
                                                             int n, int32_t *slot_idx) {
    const int i = blockIdx.x;
    const int e = idx[i];
    const bool ok = (unsigned)e < (unsigned)E;
    if (blockIdx.y == 0 && threadIdx.x == 0) slot_idx[i] = ok ? i : n;   // n: out of range -> NaN
    if (!ok) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(pool + (size_t)e * stride);
    uint4 *dst = reinterpret_cast<uint4 *>(slots + (size_t)i * slot_stride);
    const size_t words = blob_bytes / 16, step = (size_t)gridDim.y * blockDim.x;
    size_t w = (size_t)blockIdx.y * blockDim.x + threadIdx.x;
    // four independent loads in flight per thread
    for (; w + 3 * step < words; w += 4 * step) {
        const uint4 a = src[w], b = src[w + step], c = src[w + 2 * step], d = src[w + 3 * step];
        dst[w] = a;
        dst[w + step] = b;
        dst[w + 2 * step] = c;
        dst[w + 3 * step] = d;
    }
    for (; w < words; w += step) dst[w] = src[w];
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_gather_experts(const void *pool, size_t expert_stride, int E, const int32_t *idx,
                                  int n, size_t blob_bytes, void *slots, size_t slot_stride,
                                  int32_t *slot_idx, cudaStream_t stream) {
    if (n < 0 || n > kMaxSlots) return fail(MOE_EINVAL, "gather_experts: n=%d (0..%d)", n, kMaxSlots);
    if (n == 0) return MOE_OK;
    if (E <= 0) return fail(MOE_EINVAL, "gather_experts: E=%d", E);
    if (!pool || !idx || !slots || !slot_idx) return fail(MOE_EINVAL, "gather_experts: NULL pointer");
    if (blob_bytes == 0 || blob_bytes % 16 || expert_stride < blob_bytes || expert_stride % 16 ||
        slot_stride < blob_bytes || slot_stride % 16 || reinterpret_cast<uintptr_t>(pool) % 16 ||
        reinterpret_cast<uintptr_t>(slots) % 16)
        return fail(MOE_EINVAL, "gather_experts: blob %zu, strides %zu / %zu (16-byte multiples, "
                                ">= the blob) or unaligned pool / slots", blob_bytes, expert_stride,
                    slot_stride);
    // at most 16 CTAs per expert (4 x 16 B in flight per thread, 256 threads):
    // enough to keep the host link busy while leaving the SMs to the kernels
    // the gathers run beside
    const size_t words = blob_bytes / 16;
    const unsigned parts = (unsigned)std::max<size_t>(1, std::min<size_t>(16, words / (256 * 4)));
    gather_experts_kernel<<<dim3((unsigned)n, parts), 256, 0, stream>>>(
        static_cast<const uint8_t *>(pool), expert_stride, E, idx, blob_bytes,
        static_cast<uint8_t *>(slots), slot_stride, n, slot_idx);
    return check_launch("gather_experts_kernel");
}
