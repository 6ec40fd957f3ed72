// noalloc.cu -- moe_expert_ffn_int4_noalloc: the expert FFN call for callers
// that cannot provide a device workspace.
//
// The scratch lives in a file-scope __device__ array of fixed size, so the
// library needs no allocation at call time.  Every GPU that loads the library
// holds the array until the process exits.  Host code cannot use the array's
// name as a device address (on the host it names a stand-in object), so the
// device address is looked up with cudaGetSymbolAddress once per device, with
// that device current, on the first call made on it, and cached.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = MOE_FFN_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_ffn_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// The static array's device address on the current device (looked up once
// per device, with that device current, and cached).
int scratch_of_current_device(void **out, const char *who) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return moe::fail(MOE_ECUDA, "%s: cudaGetDevice: %s", who, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return moe::fail(MOE_EUNSUPPORTED, "%s: device %d >= %d", who, dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        e = cudaGetSymbolAddress(&g_scratch_addr[dev], g_ffn_scratch);
        if (e != cudaSuccess) {
            g_scratch_addr[dev] = nullptr;
            return moe::fail(MOE_ECUDA, "%s: cudaGetSymbolAddress: %s", who, cudaGetErrorString(e));
        }
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_expert_ffn_int4_noalloc(const moe_experts_desc *ed, const void *x,
                                           int x_dtype, const int32_t *idx, int T, int K,
                                           float *y_slots, cudaStream_t stream) {
    // Calls that need no scratch (an empty batch) or that the regular entry
    // point rejects on their arguments alone never touch the device: the
    // regular entry point validates them first, with no workspace, so both
    // entry points return the same status for bad arguments.
    if (int rc = moe_expert_ffn_int4(ed, x, x_dtype, idx, T <= 0 ? T : 0, K, y_slots, nullptr, 0,
                                     stream))
        return rc;
    if (T <= 0) return MOE_OK;
    const bool ptrs_ok = x && idx && y_slots && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(idx) % 4 == 0 &&
                         reinterpret_cast<uintptr_t>(y_slots) % 16 == 0;
    if (!ptrs_ok)      // the regular entry point's own MOE_EINVAL and message
        return moe_expert_ffn_int4(ed, x, x_dtype, idx, T, K, y_slots, nullptr, 0, stream);
    const size_t need = moe_expert_ffn_workspace_bytes(ed, T, K);
    if (need > kScratchBytes)
        return moe::fail(MOE_ENOSPACE,
                         "expert_ffn_noalloc: T=%d K=%d needs %zu bytes of scratch; the static "
                         "scratch holds %zu (MOE_FFN_STATIC_SCRATCH_BYTES)",
                         T, K, need, kScratchBytes);
    void *scratch = nullptr;
    if (int rc = scratch_of_current_device(&scratch, "expert_ffn_noalloc")) return rc;
    // Word 0 of the scratch is the call's status word (the batched path's
    // bounded waits record MOE_ETIMEOUT there); it starts every call at
    // MOE_OK, so moe_expert_ffn_noalloc_status reports this call alone.
    // Every kernel of the call writes the rest of the scratch it reads
    // before reading it, so nothing else has to be cleared between calls.
    const cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess)
        return moe::fail(MOE_ECUDA, "expert_ffn_noalloc: status reset: %s", cudaGetErrorString(e));
    return moe_expert_ffn_int4(ed, x, x_dtype, idx, T, K, y_slots, scratch, kScratchBytes,
                               stream);
}

extern "C" int moe_expert_ffn_noalloc_status(int *status, cudaStream_t stream) {
    if (status == nullptr) return moe::fail(MOE_EINVAL, "expert_ffn_noalloc_status: NULL status");
    void *scratch = nullptr;
    if (int rc = scratch_of_current_device(&scratch, "expert_ffn_noalloc_status")) return rc;
    int st = 0;
    cudaError_t e = cudaMemcpyAsync(&st, scratch, sizeof(int), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess)
        return moe::fail(MOE_ECUDA, "expert_ffn_noalloc_status: %s", cudaGetErrorString(e));
    *status = st;
    return MOE_OK;
}
