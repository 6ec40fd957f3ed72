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

}  // namespace

extern "C" int moe_expert_ffn_int4_noalloc(const moe_experts_desc *ed, const void *x,
                                           int x_dtype, const int32_t *idx, int T, int K,
                                           float *y_slots, cudaStream_t stream) {
    // Calls that need no scratch (an empty batch) or that the regular entry
    // point rejects on their arguments alone never touch the device.
    if (ed == nullptr || T <= 0)
        return moe_expert_ffn_int4(ed, x, x_dtype, idx, T, K, y_slots, nullptr, 0, stream);
    const size_t need = moe_expert_ffn_workspace_bytes(ed, T, K);
    if (need > kScratchBytes)
        return moe::fail(MOE_ENOSPACE,
                         "expert_ffn_noalloc: T=%d K=%d needs %zu bytes of scratch; the static "
                         "scratch holds %zu (MOE_FFN_STATIC_SCRATCH_BYTES)",
                         T, K, need, kScratchBytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return moe::fail(MOE_ECUDA, "expert_ffn_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return moe::fail(MOE_EUNSUPPORTED, "expert_ffn_noalloc: device %d >= %d", dev, kMaxDevices);
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_scratch_addr[dev] == nullptr) {
            e = cudaGetSymbolAddress(&g_scratch_addr[dev], g_ffn_scratch);
            if (e != cudaSuccess) {
                g_scratch_addr[dev] = nullptr;
                return moe::fail(MOE_ECUDA, "expert_ffn_noalloc: cudaGetSymbolAddress: %s",
                                 cudaGetErrorString(e));
            }
        }
        scratch = g_scratch_addr[dev];
    }
    // Every kernel of the call writes the scratch it reads before reading it,
    // so nothing has to be cleared between calls.
    return moe_expert_ffn_int4(ed, x, x_dtype, idx, T, K, y_slots, scratch, kScratchBytes,
                               stream);
}
