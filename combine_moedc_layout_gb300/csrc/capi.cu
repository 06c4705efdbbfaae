// Entry points that launch nothing: version, status text, device queries,
// the test hook of the bounded waits.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace moedc_host {

int sm_count()
{
    // one cached value per device; reading it once per device keeps the
    // attribute query off the per-call path
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (dev < 0 || dev >= 64) return 152;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

int resident_blocks(const void* kernel, int threads, size_t smem)
{
    // blocks of `kernel` that fit on the whole device at once (occupancy x
    // SMs), cached per kernel, block size, shared-memory size and device;
    // grid-strided kernels launch at most this many so that no block waits
    // for a second wave.  The single-launch kernels' shared memory follows the
    // batch shape, so a serving loop meets many keys: the table keeps the most
    // recent ones (round-robin replacement once full).
    struct Entry {
        const void* kernel;
        int dev, threads;
        size_t smem;
        int blocks;
    };
    constexpr int kEntries = 256;
    static std::mutex mu;
    static Entry cache[kEntries];
    static int used = 0, next = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].kernel == kernel && cache[i].dev == dev && cache[i].threads == threads &&
            cache[i].smem == smem)
            return cache[i].blocks;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
            cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int blocks = per_sm * sm_count();
    cache[next] = Entry{kernel, dev, threads, smem, blocks};
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return blocks;
}

namespace {
// moedc_test_set_wait_extra: zero unless a test sets it
std::atomic<unsigned> g_test_wait_extra{0};
}  // namespace

unsigned test_wait_extra() { return g_test_wait_extra.load(std::memory_order_relaxed); }

}  // namespace moedc_host

extern "C" void moedc_test_set_wait_extra(unsigned extra_arrivals)
{
    moedc_host::g_test_wait_extra.store(extra_arrivals, std::memory_order_relaxed);
}

extern "C" int moedc_api_version(void) { return MOEDC_API_VERSION; }

extern "C" const char* moedc_strerror(int code)
{
    switch (code) {
    case MOEDC_OK: return "ok";
    case MOEDC_ERR_ARG: return "invalid argument (size, null or misaligned pointer, workspace)";
    case MOEDC_ERR_CAPACITY: return "an expert received more entries than cap; extra entries dropped";
    case MOEDC_ERR_EXPERT_RANGE: return "a top-k index lies outside [-1, E); entry treated as masked";
    case MOEDC_ERR_CUDA: return "a CUDA launch failed";
    case MOEDC_ERR_TIMEOUT: return "a bounded device wait gave up";
    case MOEDC_ERR_UNIMPLEMENTED: return "not implemented";
    default: return "unknown status code";
    }
}
