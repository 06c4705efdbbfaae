// moedc_layout for callers that cannot hand the library any device memory.
//
// The ordinary entry point asks the caller for a scratch buffer (the per-block
// expert and rank counts that the two layout kernels pass between them).  Some
// callers have no way to provide one: a plain-C host that has no device
// allocator of its own, a plugin running inside a framework whose memory pool
// owns all of the GPU and forbids outside cudaMalloc calls, or a serving loop
// that must not call cudaMalloc after start-up because the call can
// synchronise the device and fragment a memory budget fixed in advance.  For
// them this file keeps the scratch in a fixed-size array that lives in the
// library's own device image, so the call itself allocates nothing.
//
// Rules for users:
//  * The array holds MOEDC_STATIC_SCRATCH_BYTES per device and stays resident
//    on every GPU that loads the library until the process exits.  Shapes
//    that need more scratch than that on every path that uses scratch are
//    rejected with MOEDC_ERR_ARG before anything is launched.
//  * The first call on each device that uses scratch looks up the array's
//    device address (cudaGetSymbolAddress, with that device current) and
//    caches it; make that first call before any stream capture begins.
//    Shapes the sweep takes (no workspace asked for) look nothing up.
//  * Every call in the process shares the one array.  Calls whose kernels
//    overlap on the GPU (different streams, or different host threads without
//    ordering) race on it and give wrong slots; order them on one stream.
//  * The cached address is that of the device's primary context at the first
//    call.  cudaDeviceReset recreates the context and the array with it, so a
//    process must not reset a device after using this entry point on it.
//  * Nothing in the array needs to start at zero: the first layout kernel
//    writes every word the second one reads, so the leftovers of an earlier
//    call do no harm.
#include <mutex>

#include "common.cuh"

namespace {

// Scratch words for the layout's per-block counts; file scope, one copy per
// device.  Host code must never pass this symbol to a kernel: on the host it
// names a shadow, not device memory.  Only the address returned by
// cudaGetSymbolAddress is used.
static __device__ __align__(256) unsigned char g_layout_scratch[MOEDC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device, looked up once.
int scratch_address(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return MOEDC_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || p == nullptr)
            return MOEDC_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOEDC_OK;
}

}  // namespace

extern "C" int moedc_layout_static_scratch(const int32_t* topk_idx, int T, int K, int E, int R,
                                           int cap, int32_t* num_tokens_per_expert,
                                           int32_t* num_tokens_per_rank,
                                           uint8_t* is_token_in_rank, int32_t* slot,
                                           int32_t* dev_status, cudaStream_t stream)
{
    if (!moedc_host::layout_args_ok(T, K, E, R, cap)) return MOEDC_ERR_ARG;
    // the shape needs more scratch than the static array holds (on both paths
    // that use scratch: the single pass and the two-kernel layout)
    const size_t need = moedc_host::layout_geometry(T, K, E, R).ws;
    const size_t fast = moedc_host::layout_onepass_workspace_bytes(T, K, E, R);
    if (need > (size_t)MOEDC_STATIC_SCRATCH_BYTES &&
        (fast == 0 || fast > (size_t)MOEDC_STATIC_SCRATCH_BYTES))
        return MOEDC_ERR_ARG;
    if (need == 0 && fast == 0)   // the sweep: no scratch, so no address lookup either
        return moedc_layout(topk_idx, T, K, E, R, cap, num_tokens_per_expert,
                            num_tokens_per_rank, is_token_in_rank, slot, nullptr, 0, dev_status,
                            stream);
    void* scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != MOEDC_OK) return st;
    return moedc_layout(topk_idx, T, K, E, R, cap, num_tokens_per_expert, num_tokens_per_rank,
                        is_token_in_rank, slot, scratch, (size_t)MOEDC_STATIC_SCRATCH_BYTES,
                        dev_status, stream);
}
