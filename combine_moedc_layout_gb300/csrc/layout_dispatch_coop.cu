// Layout + dispatch in one cooperative launch for large batches (more routing
// entries than the single-launch layout sweep takes).
//
// Sources: UCCL PR #749 "[EP] Low-latency mode batch tokens per destination"
// (code excerpt and discussion: per-expert routed-token counters, and a rank
// that must wait until the counts of all of its experts are known before it
// can send); MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on
// MI300X + CX7" (relay note: a grid barrier cost more than a 4-token copy -
// here the copy is hundreds of MB, so two barriers are small against it).
//
// Every block of a co-resident grid owns a contiguous chunk of tokens:
//   phase 1  rank the chunk's entries per expert in (t, k) order (one warp,
//            32-entry tiles, ballot match), count the chunk's entries per
//            expert and distinct tokens per rank, write its token-in-rank
//            rows, and publish the counts as column c of rows [E + R][B]
//   barrier
//   phase 2  block r scans row r in place (exclusive prefix over the chunks)
//            and writes the row total: an expert's or a rank's count
//   barrier
//   phase 3  slot = the chunk's prefix + its in-chunk rank; src_idx; then the
//            chunk's (token, 512-channel slice) copies, as the dispatch
//            kernel makes them.
// Each warp's first x slice is loaded before phase 1, so its DRAM latency
// overlaps the layout phases.
//
// The barriers are bounded waits on a 64-bit word whose high bits carry this
// launch's epoch and whose low bits count the arrivals; block 0 tags the
// words with the epoch at its start and the others arrive (one atomic add)
// only once they see the tag.  The epoch combines a per-call host counter
// (seeded from a clock) with a generation kept in the workspace and advanced
// by every launch, so neither an earlier launch, nor a replay of the same
// captured graph, nor uninitialised workspace contents can release a
// barrier.  A wait that runs out raises MOEDC_ERR_TIMEOUT and the block
// returns; the co-residency the waits rely on is guaranteed by the
// cooperative launch (it fails instead of running a grid that does not fit).
#include <atomic>
#include <chrono>
#include <climits>

#include "dispatch_item.cuh"

namespace moedc {

constexpr int kCoopThreads = 256;
constexpr int kCoopWarps = kCoopThreads / kWarp;
constexpr int kCoopMaxBlocks = 2048;          // columns of the count rows
constexpr int kCoopMaxEntries = 2048;         // routing entries of one chunk
constexpr int kCoopIdsPerThread = kCoopMaxEntries / kCoopThreads;
constexpr int kCoopScanPer = kCoopMaxBlocks / kCoopThreads;
constexpr size_t kCoopHeaderBytes = 256;      // barrier words before the count rows
constexpr int kArrivalBits = 20;
constexpr unsigned long long kArrivalMask = (1ull << kArrivalBits) - 1;
constexpr long long kCoopSpinLimit = 1ll << 21;   // x >= 64 ns sleeps: >= 0.13 s

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Header words of the workspace: the two barriers, the exit count, and the
// workspace's launch generation.
constexpr int kBar1 = 0, kBar2 = 1, kExit = 2, kGeneration = 3;
constexpr int kEpochBits = 64 - kArrivalBits;
constexpr unsigned long long kEpochMask = (1ull << kEpochBits) - 1;
constexpr unsigned long long kEpochStride = (1ull << 22) + 1;

// This launch's epoch: the host's per-call counter plus the workspace's
// generation times an odd stride.  Successful launches advance the
// generation by one at their end and a launch that gives up advances it
// further, so consecutive launches on one workspace - eager calls, replays of
// one captured graph (whose host counter is fixed), calls after a timeout -
// never share an epoch.
__device__ __forceinline__ unsigned long long launch_epoch(unsigned long long host_epoch,
                                                           unsigned long long generation)
{
    return (host_epoch + generation * kEpochStride) & kEpochMask;
}

// Wait (bounded) until the header word carries this launch's epoch: block 0
// tags the words at its start, and a block must not count itself on a word
// that still holds an earlier launch's value.
__device__ bool coop_tagged(const unsigned long long* w, unsigned long long epoch)
{
    for (long long it = 0; it < kCoopSpinLimit; ++it) {
        if ((ld_acquire_u64(w) >> kArrivalBits) == epoch) return true;
        __nanosleep(32);
    }
    return false;
}

// Grid barrier on header word `which`: true once `target` blocks of this
// epoch arrived; false when a wait runs out (the block then advances the
// generation so that the next launch on this workspace starts clean).
// Arrivals are single atomic adds: a compare-and-swap loop on one word
// serialises hundreds of blocks' retries (measured: ~0.6 ms per barrier).
__device__ bool coop_barrier(unsigned long long* bar, int which, unsigned long long epoch,
                             unsigned target, int* s_flag)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();   // this block's writes before its arrival
        bool ok = coop_tagged(bar + which, epoch);
        if (ok) {
            atomicAdd(bar + which, 1ull);
            ok = false;
            for (long long it = 0; it < kCoopSpinLimit; ++it) {
                const unsigned long long v = ld_acquire_u64(bar + which);
                if ((v >> kArrivalBits) == epoch && (v & kArrivalMask) >= target) {
                    ok = true;
                    break;
                }
                __nanosleep(64);
            }
        }
        __threadfence();
        if (!ok) atomicAdd(bar + kGeneration, 1ull);
        *s_flag = ok ? 1 : 0;
    }
    __syncthreads();
    return *s_flag != 0;
}

template <bool kFp8, bool kScaleCols>
__global__ void __launch_bounds__(kCoopThreads, 4)
layout_dispatch_coop_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_idx,
                            int T, int H, int K, int E, int R, int cap, int chunk,
                            int32_t* __restrict__ num_tokens_per_expert,
                            int32_t* __restrict__ num_tokens_per_rank,
                            uint8_t* __restrict__ is_token_in_rank, int32_t* __restrict__ slot,
                            void* __restrict__ recv, float* __restrict__ scales,
                            int32_t* __restrict__ src_idx, unsigned long long* __restrict__ bar,
                            int32_t* __restrict__ counts, unsigned long long host_epoch,
                            unsigned target, int32_t* __restrict__ status)
{
    pdl_enter();
    extern __shared__ int32_t smem[];
    __shared__ int s_flag;
    __shared__ int s_warp[kCoopWarps];
    __shared__ unsigned long long s_epoch;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int B = gridDim.x;
    const int c = blockIdx.x;
    const int epr = E / R;
    const int t0 = min(T, c * chunk);
    const int nt = min(T, t0 + chunk) - t0;
    const int n = nt * K;                        // <= kCoopMaxEntries
    int32_t* s_idx = smem;                       // [kCoopMaxEntries]
    int32_t* s_slot = s_idx + kCoopMaxEntries;   // [kCoopMaxEntries] in-chunk rank, then slot
    int32_t* s_h = s_slot + kCoopMaxEntries;     // [E]
    int32_t* s_hr = s_h + E;                     // [R]
    const int nslice = (H + kSlice - 1) / kSlice;
    const int items = nt * nslice;

    // the warp's first x slice does not depend on the layout: start it now
    SliceX xv{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (warp < items) {
        const int j = warp / nslice;
        xv = load_slice<kFp8>(x + (int64_t)(t0 + j) * H, H, warp - j * nslice, lane);
    }
    {
        int v[kCoopIdsPerThread];
#pragma unroll
        for (int j = 0; j < kCoopIdsPerThread; ++j) {
            const int i = threadIdx.x + j * kCoopThreads;
            v[j] = i < n ? __ldg(topk_idx + (int64_t)t0 * K + i) : 0;
        }
        for (int e = threadIdx.x; e < E; e += kCoopThreads) s_h[e] = 0;
        for (int r = threadIdx.x; r < R; r += kCoopThreads) s_hr[r] = 0;
        if (threadIdx.x == 0) {
            const unsigned long long ep = launch_epoch(host_epoch, ld_acquire_u64(bar + kGeneration));
            s_epoch = ep;
            if (blockIdx.x == 0) {   // tag this launch's barrier and exit words, counts zero
                volatile unsigned long long* vb = bar;
                vb[kBar1] = ep << kArrivalBits;
                vb[kBar2] = ep << kArrivalBits;
                vb[kExit] = ep << kArrivalBits;
                __threadfence();
            }
        }
#pragma unroll
        for (int j = 0; j < kCoopIdsPerThread; ++j) {
            const int i = threadIdx.x + j * kCoopThreads;
            if (i < n) s_idx[i] = v[j];
        }
    }
    __syncthreads();

    // ---- phase 1: in-chunk ranks and counts (warp 0), rank membership (the rest)
    if (warp == 0) {
        const unsigned lt = lanemask_lt();
        bool bad = false;
        for (int i0 = 0; i0 < n; i0 += kWarp) {
            const int i = i0 + lane;
            const int e = i < n ? s_idx[i] : -1;
            const bool v = e >= 0 && e < E;
            if (i < n && (e < -1 || e >= E)) bad = true;
            const unsigned peers = match_expert(e, v);
            int ls = -1;
            if (v) ls = s_h[e] + __popc(peers & lt);
            __syncwarp();
            if (v && (peers & lt) == 0) s_h[e] += __popc(peers);
            __syncwarp();
            if (i < n) s_slot[i] = ls;
        }
        if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
    } else {
        for (int b = threadIdx.x - kWarp; b < nt * R; b += kCoopThreads - kWarp) {
            const int j = b / R;
            const int r = b - j * R;
            const unsigned lo = (unsigned)(r * epr);
            uint8_t flag = 0;
            for (int k = 0; k < K; ++k)
                flag |= ((unsigned)s_idx[j * K + k] - lo < (unsigned)epr) ? 1 : 0;
            is_token_in_rank[(int64_t)(t0 + j) * R + r] = flag;
            if (flag) atomicAdd(&s_hr[r], 1);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kCoopThreads) counts[(int64_t)e * B + c] = s_h[e];
    for (int r = threadIdx.x; r < R; r += kCoopThreads)
        counts[(int64_t)(E + r) * B + c] = s_hr[r];
    const unsigned long long epoch = s_epoch;
    if (!coop_barrier(bar, kBar1, epoch, target, &s_flag)) {
        if (threadIdx.x == 0) raise_status(status, MOEDC_ERR_TIMEOUT);
        return;
    }

    // ---- phase 2: exclusive prefix over the chunks, one row per block
    for (int row = c; row < E + R; row += B) {
        int32_t* rp = counts + (int64_t)row * B;
        int v[kCoopScanPer];
        int mine = 0;
        const int base = threadIdx.x * kCoopScanPer;
#pragma unroll
        for (int j = 0; j < kCoopScanPer; ++j) {
            v[j] = base + j < B ? __ldcg(rp + base + j) : 0;
            mine += v[j];
        }
        int incl = mine;
#pragma unroll
        for (int d = 1; d < kWarp; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        if (lane == kWarp - 1) s_warp[warp] = incl;
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < kCoopWarps; ++w) {
            before += w < warp ? s_warp[w] : 0;
            total += s_warp[w];
        }
        int run = before + incl - mine;
#pragma unroll
        for (int j = 0; j < kCoopScanPer; ++j) {
            if (base + j < B) rp[base + j] = run;
            run += v[j];
        }
        if (threadIdx.x == 0) {
            if (row < E) {
                num_tokens_per_expert[row] = total;
                if (total > cap) raise_status(status, MOEDC_ERR_CAPACITY);
            } else {
                num_tokens_per_rank[row - E] = total;
            }
        }
        __syncthreads();   // s_warp is rewritten for the next row
    }
    if (!coop_barrier(bar, kBar2, epoch, target, &s_flag)) {
        if (threadIdx.x == 0) raise_status(status, MOEDC_ERR_TIMEOUT);
        return;
    }
    // every block is past the last barrier once all have counted themselves
    // out here; the last one advances the workspace's generation
    if (threadIdx.x == 0 &&
        ((atomicAdd(bar + kExit, 1ull) & kArrivalMask) + 1) == (unsigned long long)B)
        atomicAdd(bar + kGeneration, 1ull);

    // ---- phase 3: slots, src_idx, and the chunk's copies
    for (int i = threadIdx.x; i < n; i += kCoopThreads) {
        const int e = s_idx[i];
        int s = -1;
        if (e >= 0 && e < E) s = __ldcg(counts + (int64_t)e * B + c) + s_slot[i];
        s_slot[i] = s;
        slot[(int64_t)t0 * K + i] = s;
    }
    {
        const int64_t total = (int64_t)E * cap;
        const int64_t nthreads = (int64_t)B * kCoopThreads;
        for (int64_t i = (int64_t)c * kCoopThreads + threadIdx.x; i < total; i += nthreads) {
            const int e = (int)(i / cap);
            const int s = (int)(i - (int64_t)e * cap);
            if (s >= __ldcg(num_tokens_per_expert + e)) src_idx[i] = -1;
        }
    }
    __syncthreads();
    for (int item = warp; item < items;) {
        const int j = item / nslice;
        const int sl = item - j * nslice;
        const int next = item + kCoopWarps;
        SliceX nv{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (next < items) {
            const int j2 = next / nslice;
            nv = load_slice<kFp8>(x + (int64_t)(t0 + j2) * H, H, next - j2 * nslice, lane);
        }
        int my_row = -1;
        if (lane < K) {
            my_row = dest_row(s_idx[j * K + lane], s_slot[j * K + lane], E, cap);
            if (sl == 0 && my_row >= 0) src_idx[my_row] = t0 + j;
        }
        const int64_t sbase = kScaleCols ? colmajor_scale_base(my_row, cap, H / 128) : 0;
        store_slice<kFp8, kScaleCols>(xv, H, sl, lane, K, my_row, recv, scales, sbase, cap);
        xv = nv;
        item = next;
    }
}

}  // namespace moedc

namespace moedc_host {

namespace {

// Host part of the launch epochs: consecutive per process, starting from a
// clock-derived value, so that ordinary data left in a workspace (zeros, small
// integers, a uniform fill) does not carry a launch's epoch.
std::atomic<unsigned long long> g_epoch{
    (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() * 2654435761ull};

size_t coop_workspace_bytes(int E, int R)
{
    return moedc::kCoopHeaderBytes + (size_t)(E + R) * moedc::kCoopMaxBlocks * sizeof(int32_t);
}

}  // namespace

// The single launch is used where the layout alone would need two kernels
// (more entries than one sweep launch takes).  Below that, layout then
// dispatch is faster: measured at 4096 tokens, 61.9 us against 65.1 us - the
// two barriers cost ~3.5 us each and chunk-owned copies end less evenly than
// the dispatch kernel's grid-strided items - while at 40000 tokens (320000
// entries) the single launch takes 32.4 us against 64.5 us.
static bool layout_dispatch_coop_applies(int T, int K, int E, int R)
{
    return !layout_geometry(T, K, E, R).sweep;
}

size_t layout_dispatch_coop_workspace_bytes(int T, int K, int E, int R)
{
    return layout_dispatch_coop_applies(T, K, E, R) ? coop_workspace_bytes(E, R) : 0;
}

// MOEDC_ERR_UNIMPLEMENTED when the single launch does not apply (the caller
// then runs layout and dispatch as two launches); otherwise the launch status.
int launch_layout_dispatch_coop(const void* x, const int32_t* topk_idx, int T, int H, int K,
                                int E, int R, int cap, int out_dtype,
                                int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                uint8_t* is_token_in_rank, int32_t* slot, void* recv,
                                float* scales, int32_t* src_idx, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream)
{
    const int base = dtype_base(out_dtype);
    const bool cols = (out_dtype & MOEDC_SCALES_COL_MAJOR) != 0;
    if (out_dtype & MOEDC_SCALES_PER_TOKEN) return MOEDC_ERR_UNIMPLEMENTED;
    if (!layout_dispatch_coop_applies(T, K, E, R)) return MOEDC_ERR_UNIMPLEMENTED;
    if (!workspace || workspace_bytes < coop_workspace_bytes(E, R) || !aligned(workspace, 16))
        return MOEDC_ERR_UNIMPLEMENTED;
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) {
        clear_stale_error();
        return MOEDC_ERR_UNIMPLEMENTED;
    }
    const void* fn = base == MOEDC_BF16
                         ? (const void*)moedc::layout_dispatch_coop_kernel<false, false>
                     : cols ? (const void*)moedc::layout_dispatch_coop_kernel<true, true>
                            : (const void*)moedc::layout_dispatch_coop_kernel<true, false>;
    const size_t sm = (size_t)(2 * moedc::kCoopMaxEntries + E + R) * sizeof(int32_t);
    int64_t blocks = resident_blocks(fn, moedc::kCoopThreads, sm);
    if (blocks > moedc::kCoopMaxBlocks) blocks = moedc::kCoopMaxBlocks;
    if (blocks < 1) return MOEDC_ERR_UNIMPLEMENTED;
    const int64_t chunk = (T + blocks - 1) / blocks;
    if (chunk * K > moedc::kCoopMaxEntries) return MOEDC_ERR_UNIMPLEMENTED;

    // test hook: extra arrivals the barriers wait for, so that they run out
    const unsigned extra = test_wait_extra();
    const unsigned long long host_epoch = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    auto* bar = static_cast<unsigned long long*>(workspace);
    auto* counts = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) +
                                              moedc::kCoopHeaderBytes);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    const unsigned target = (unsigned)blocks + extra;
    const int ch = (int)chunk;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(moedc::kCoopThreads);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    clear_stale_error();
#define MOEDC_COOP_LAUNCH(F, C)                                                                  \
    cudaLaunchKernelEx(&cfg, moedc::layout_dispatch_coop_kernel<F, C>, xb, topk_idx, T, H,       \
                       K, E, R, cap, ch, num_tokens_per_expert, num_tokens_per_rank,           \
                       is_token_in_rank, slot, recv, scales, src_idx, bar, counts, host_epoch,  \
                       target, dev_status)
    const cudaError_t err = base == MOEDC_BF16 ? MOEDC_COOP_LAUNCH(false, false)
                            : cols             ? MOEDC_COOP_LAUNCH(true, true)
                                               : MOEDC_COOP_LAUNCH(true, false);
#undef MOEDC_COOP_LAUNCH
    if (err == cudaErrorCooperativeLaunchTooLarge) {
        // fewer SMs than the device reports (a partitioned GPU): two launches instead
        clear_stale_error();
        return MOEDC_ERR_UNIMPLEMENTED;
    }
    return err == cudaSuccess ? MOEDC_OK : MOEDC_ERR_CUDA;
}

}  // namespace moedc_host

extern "C" size_t moedc_layout_dispatch_workspace_bytes(int T, int K, int E, int R)
{
    if (!moedc_host::layout_args_ok(T, K, E, R, 1)) return 0;
    const size_t a = moedc_layout_workspace_bytes(T, K, E, R);
    const size_t b = moedc_host::layout_dispatch_coop_workspace_bytes(T, K, E, R);
    return a > b ? a : b;
}
