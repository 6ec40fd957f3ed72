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

// One warp: the cache decision for a route of n <= kMaxSlots experts over C
// slots.  Entry i: its expert's slot if a slot holds it (a hit), the slot an
// earlier entry of the same expert took, or else the least recently used
// slot this route does not use (empty slots first, then the oldest step,
// then the lowest index), whose tag becomes the expert (a miss: plan[i] =
// that slot, the copy kernel fills it).  Every slot the route uses gets age
// the call's step: the cache's device clock, advanced by one per call (so
// that calls replayed from a captured graph still age the slots).
// slot_idx[i] = the slot, or C for an index outside [0, E).
__global__ void __launch_bounds__(32) cache_plan_kernel(const int32_t *idx, int n, int E, int C,
                                                        int32_t *tags, int32_t *ages, int32_t *clock,
                                                        int32_t *slot_idx, int32_t *plan,
                                                        int32_t *stats) {
    __shared__ uint32_t pinned[(kMaxCacheSlots + 31) / 32];
    const int lane = threadIdx.x;
    int step = 0;
    if (lane == 0) step = ++*clock;
    step = __shfl_sync(0xffffffffu, step, 0);
    for (int w = lane; w < (C + 31) / 32; w += 32) pinned[w] = 0u;
    __syncwarp();
    int hits = 0, misses = 0;
    for (int i = 0; i < n; i++) {
        const int e = idx[i];
        int slot = C, copy = -1;
        if ((unsigned)e < (unsigned)E) {
            // a slot holding e (at most one does)
            int found = C;
            for (int j = lane; j < C; j += 32)
                if (tags[j] == e) found = j;
            for (int o = 16; o > 0; o >>= 1) found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
            if (found < C) {
                slot = found;
                // an earlier entry of this route may have just filled it
                bool earlier = false;
                for (int k = 0; k < i; k++) earlier |= idx[k] == e;
                if (!earlier) hits++;
            } else {
                // victim: among slots not pinned by this route, the smallest
                // (tag >= 0, age, index)
                unsigned long long best = ~0ull;
                for (int j = lane; j < C; j += 32) {
                    if (pinned[j >> 5] >> (j & 31) & 1u) continue;
                    const unsigned long long key =
                        ((unsigned long long)(tags[j] >= 0 ? 1u : 0u) << 63) |
                        ((unsigned long long)(uint32_t)(ages[j] + 0x40000000) << 31) | (unsigned)j;
                    best = key < best ? key : best;
                }
                for (int o = 16; o > 0; o >>= 1) {
                    const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
                    best = other < best ? other : best;
                }
                slot = (int)(best & 0x7fffffffu);
                copy = slot;
                misses++;
                if (lane == 0) tags[slot] = e;
                __syncwarp();
            }
            if (lane == 0) {
                pinned[slot >> 5] |= 1u << (slot & 31);
                ages[slot] = step;
            }
            __syncwarp();
        }
        if (lane == 0) {
            slot_idx[i] = slot;
            plan[i] = copy;
        }
    }
    if (lane == 0 && stats != nullptr) {
        atomicAdd(stats, hits);
        atomicAdd(stats + 1, misses);
    }
}

// grid (n, parts): CTA (i, p) copies the p-th share of expert idx[i]'s blob
// into slot plan[i] when the plan has one.
__global__ void __launch_bounds__(256) cache_fill_kernel(const uint8_t *pool, size_t stride,
                                                         const int32_t *idx, const int32_t *plan,
                                                         size_t blob_bytes, uint8_t *cache,
                                                         size_t slot_stride) {
    const int i = blockIdx.x;
    const int slot = plan[i];
    if (slot < 0) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(pool + (size_t)idx[i] * stride);
    uint4 *dst = reinterpret_cast<uint4 *>(cache + (size_t)slot * slot_stride);
    const size_t words = blob_bytes / 16, step = (size_t)gridDim.y * blockDim.x;
    size_t w = (size_t)blockIdx.y * blockDim.x + threadIdx.x;
    // eight independent loads in flight per thread (a read of host memory
    // over C2C waits microseconds)
    constexpr int kU = 8;
    for (; w + (kU - 1) * step < words; w += kU * step) {
        uint4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; u++) v[u] = src[w + u * step];
#pragma unroll
        for (int u = 0; u < kU; u++) dst[w + u * step] = v[u];
    }
    for (; w < words; w += step) dst[w] = src[w];
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" int moe_cache_experts(const void *pool, size_t expert_stride, int E, const int32_t *idx,
                                 int n, size_t blob_bytes, void *cache, size_t slot_stride, int C,
                                 int32_t *tags, int32_t *ages, int32_t *clock, int32_t *slot_idx,
                                 int32_t *plan, int32_t *stats, cudaStream_t stream) {
    if (n < 0 || n > kMaxSlots) return fail(MOE_EINVAL, "cache_experts: n=%d (0..%d)", n, kMaxSlots);
    if (n == 0) return MOE_OK;
    if (E <= 0 || C < n || C > kMaxCacheSlots)
        return fail(MOE_EINVAL, "cache_experts: E=%d C=%d (n <= C <= %d)", E, C, kMaxCacheSlots);
    if (!pool || !idx || !cache || !tags || !ages || !clock || !slot_idx || !plan)
        return fail(MOE_EINVAL, "cache_experts: NULL pointer");
    if (blob_bytes == 0 || blob_bytes % 16 || expert_stride < blob_bytes || expert_stride % 16 ||
        slot_stride < blob_bytes || slot_stride % 16 || reinterpret_cast<uintptr_t>(pool) % 16 ||
        reinterpret_cast<uintptr_t>(cache) % 16)
        return fail(MOE_EINVAL, "cache_experts: blob %zu, strides %zu / %zu (16-byte multiples, "
                                ">= the blob) or unaligned pool / cache", blob_bytes, expert_stride,
                    slot_stride);
    cache_plan_kernel<<<1, 32, 0, stream>>>(idx, n, E, C, tags, ages, clock, slot_idx, plan, stats);
    if (int rc = check_launch("cache_plan_kernel")) return rc;
    const size_t words = blob_bytes / 16;
    const unsigned parts = (unsigned)std::max<size_t>(1, std::min<size_t>(16, words / (256 * 8)));
    cache_fill_kernel<<<dim3((unsigned)n, parts), 256, 0, stream>>>(
        static_cast<const uint8_t *>(pool), expert_stride, idx, plan, blob_bytes,
        static_cast<uint8_t *>(cache), slot_stride);
    return check_launch("cache_fill_kernel");
}

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
