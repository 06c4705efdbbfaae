// Layout + dispatch in one launch for small batches (T * K <= 1024 entries).
//
// Sources: MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on MI300X
// + CX7".  At 4-16 tokens the pages find latency flat in tokens and hidden
// size (host enqueue and launches dominate, host view-cache note), that
// per-token work splits leave most warps idle (CombineSync and MultiWarpIter
// notes: split by (token, slice) with a 512-element floor), and that a grid
// barrier cost more than the copy it was meant to parallelise (relay note:
// block-local barriers only).  So every block recomputes the tiny layout in
// shared memory, block 0 alone publishes it, and all blocks copy slices.
#include <climits>

#include "dispatch_item.cuh"

namespace moedc {

constexpr int kFusedThreads = 128;
constexpr int kFusedWarps = kFusedThreads / kWarp;

template <bool kFp8, bool kScaleCols>
__global__ void __launch_bounds__(kFusedThreads)
fused_layout_dispatch_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_idx,
                             int T, int H, int K, int E, int R, int cap,
                             int32_t* __restrict__ num_tokens_per_expert,
                             int32_t* __restrict__ num_tokens_per_rank,
                             uint8_t* __restrict__ is_token_in_rank, int32_t* __restrict__ slot,
                             void* __restrict__ recv, float* __restrict__ scales,
                             int32_t* __restrict__ src_idx, int32_t* __restrict__ status)
{
    pdl_enter();
    extern __shared__ int32_t smem[];
    const int n = T * K;
    int32_t* s_idx = smem;                      // [n]
    int32_t* s_slot = s_idx + n;                // [n]
    int32_t* s_wcnt = s_slot + n;               // [kFusedWarps][E] per-warp counts, then offsets
    int32_t* s_cnt = s_wcnt + kFusedWarps * E;  // [E] totals, then block 0's [R] rank counts
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int epr = E / R;

    for (int i = threadIdx.x; i < kFusedWarps * E; i += blockDim.x) s_wcnt[i] = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_idx[i] = topk_idx[i];
    __syncthreads();

    // layout: each warp takes a contiguous run of 32-entry tiles in (t, k)
    // order, counts it per expert, the counts are scanned across warps, then
    // each warp ranks equal experts inside its tiles with __match_any_sync
    const int run = ((n + kFusedWarps * kWarp - 1) / (kFusedWarps * kWarp)) * kWarp;
    const int wbeg = min(n, warp * run);
    const int wend = min(n, wbeg + run);
    int32_t* my = s_wcnt + warp * E;
    const unsigned lt = lanemask_lt();
    for (int i0 = wbeg; i0 < wend; i0 += kWarp) {
        const int i = i0 + lane;
        const int e = i < wend ? s_idx[i] : -1;
        const bool v = e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, v ? e : -1);
        if (v && (peers & lt) == 0) my[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int acc = 0;
#pragma unroll
        for (int w = 0; w < kFusedWarps; ++w) {
            const int c = s_wcnt[w * E + e];
            s_wcnt[w * E + e] = acc;
            acc += c;
        }
        s_cnt[e] = acc;
    }
    __syncthreads();
    for (int i0 = wbeg; i0 < wend; i0 += kWarp) {
        const int i = i0 + lane;
        const int e = i < wend ? s_idx[i] : -1;
        const bool v = e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, v ? e : -1);
        int sv = -1;
        if (v) sv = my[e] + __popc(peers & lt);
        __syncwarp();
        if (v && (peers & lt) == 0) my[e] += __popc(peers);
        __syncwarp();
        if (i < wend) s_slot[i] = sv;
    }
    __syncthreads();

    if (blockIdx.x == 0) {
        // block 0 publishes the layout; rank membership is a range test per
        // (token, rank) pair, spread over all threads, counted in shared memory
        int32_t* s_rank = s_cnt + E;   // [R] (after the totals)
        for (int r = threadIdx.x; r < R; r += blockDim.x) s_rank[r] = 0;
        bool bad = false;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            slot[i] = s_slot[i];
            const int e = s_idx[i];
            if (e < -1 || e >= E) bad = true;
        }
        if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            num_tokens_per_expert[e] = s_cnt[e];
            if (s_cnt[e] > cap) raise_status(status, MOEDC_ERR_CAPACITY);
        }
        __syncthreads();   // s_rank zeroed
        for (int b = threadIdx.x; b < T * R; b += blockDim.x) {
            const int t = b / R;
            const int r = b - t * R;
            const unsigned lo = (unsigned)(r * epr);
            uint8_t flag = 0;
            for (int k = 0; k < K; ++k)
                flag |= ((unsigned)s_idx[t * K + k] - lo < (unsigned)epr) ? 1 : 0;
            is_token_in_rank[b] = flag;
            if (flag) atomicAdd(&s_rank[r], 1);
        }
        __syncthreads();
        for (int r = threadIdx.x; r < R; r += blockDim.x) num_tokens_per_rank[r] = s_rank[r];
    }

    // src_idx: -1 past each expert's count (grid-strided), t for filled slots
    {
        const int64_t total = (int64_t)E * cap;
        const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += nthreads) {
            const int e = (int)(i / cap);
            const int s = (int)(i - (int64_t)e * cap);
            if (s >= s_cnt[e]) src_idx[i] = -1;
        }
    }

    const int nslice = (H + kSlice - 1) / kSlice;
    const int items = T * nslice;
    const int nwarps = gridDim.x * kFusedWarps;
    for (int item = blockIdx.x * kFusedWarps + warp; item < items; item += nwarps) {
        const int t = item / nslice;
        const int sl = item - t * nslice;
        int my_row = -1;
        if (lane < K) {
            my_row = dest_row(s_idx[t * K + lane], s_slot[t * K + lane], E, cap);
            if (sl == 0 && my_row >= 0) src_idx[my_row] = t;
        }
        const SliceX v = load_slice<kFp8>(x + (int64_t)t * H, H, sl, lane);
        const int64_t sbase = kScaleCols ? colmajor_scale_base(my_row, cap, H / 128) : 0;
        store_slice<kFp8, kScaleCols>(v, H, sl, lane, K, my_row, recv, scales, sbase, cap);
    }
}

}  // namespace moedc

extern "C" int moedc_layout_dispatch(const void* x, const int32_t* topk_idx, int T, int H, int K,
                                     int E, int R, int cap, int out_dtype,
                                     int32_t* num_tokens_per_expert,
                                     int32_t* num_tokens_per_rank, uint8_t* is_token_in_rank,
                                     int32_t* slot, void* recv, float* scales, int32_t* src_idx,
                                     void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, cudaStream_t stream)
{
    using namespace moedc_host;
    if (!layout_args_ok(T, K, E, R, cap)) return MOEDC_ERR_ARG;
    if (!dtype_ok(out_dtype)) return MOEDC_ERR_ARG;
    const bool cols = (out_dtype & MOEDC_SCALES_COL_MAJOR) != 0;
    const int base = out_dtype & ~MOEDC_SCALES_COL_MAJOR;
    if (H < 8 || (base == MOEDC_BF16 && H % 8 != 0) || (base == MOEDC_FP8_E4M3 && H % 128 != 0))
        return MOEDC_ERR_ARG;
    if (base == MOEDC_FP8_E4M3 && (int64_t)E * cap * (H / 128) > INT32_MAX) return MOEDC_ERR_ARG;
    if (!num_tokens_per_expert || !num_tokens_per_rank || !dev_status || !recv || !src_idx)
        return MOEDC_ERR_ARG;
    if ((int64_t)E * cap > INT32_MAX || (int64_t)T * ((H + 511) / 512) > INT32_MAX / 2)
        return MOEDC_ERR_ARG;
    if (base == MOEDC_FP8_E4M3 && !scales) return MOEDC_ERR_ARG;
    if (T > 0 && (!x || !topk_idx || !is_token_in_rank || !slot)) return MOEDC_ERR_ARG;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(scales, 4) || !aligned(topk_idx, 4) ||
        !aligned(slot, 4) || !aligned(num_tokens_per_expert, 4) ||
        !aligned(num_tokens_per_rank, 4) || !aligned(src_idx, 4) || !aligned(dev_status, 4))
        return MOEDC_ERR_ARG;

    const int64_t n = (int64_t)T * K;
    if (n > MOEDC_FUSED_MAX_ENTRIES) {
        const LayoutGeom g = layout_geometry(T, K, E, R);
        if (g.ws > 0 && (!workspace || workspace_bytes < g.ws || !aligned(workspace, 16)))
            return MOEDC_ERR_ARG;
        int st = launch_layout(topk_idx, T, K, E, R, cap, num_tokens_per_expert,
                               num_tokens_per_rank, is_token_in_rank, slot, workspace,
                               dev_status, stream);
        if (st != MOEDC_OK) return st;
        return launch_dispatch(x, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap,
                               out_dtype, recv, scales, src_idx, dev_status, stream);
    }

    const int nslice = (H + moedc::kSlice - 1) / moedc::kSlice;
    const int64_t items = (int64_t)T * nslice;
    int64_t blocks = (items + moedc::kFusedWarps - 1) / moedc::kFusedWarps;
    const int64_t fill_blocks = ((int64_t)E * cap + moedc::kFusedThreads - 1) / moedc::kFusedThreads;
    if (blocks < fill_blocks) blocks = fill_blocks;
    const void* fn = base == MOEDC_BF16
                         ? (const void*)moedc::fused_layout_dispatch_kernel<false, false>
                     : cols ? (const void*)moedc::fused_layout_dispatch_kernel<true, true>
                            : (const void*)moedc::fused_layout_dispatch_kernel<true, false>;
    const size_t sm = (size_t)(2 * n + (moedc::kFusedWarps + 1) * E + R) * sizeof(int32_t);
    const int64_t resident = resident_blocks(fn, moedc::kFusedThreads, sm);
    if (blocks > resident) blocks = resident;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    clear_stale_error();
#define MOEDC_FUSED_LAUNCH(F, C)                                                                 \
    launch(moedc::fused_layout_dispatch_kernel<F, C>, (int)blocks, moedc::kFusedThreads, sm, stream, \
        xb, topk_idx, T, H, K, E, R, cap, num_tokens_per_expert, num_tokens_per_rank,          \
        is_token_in_rank, slot, recv, scales, src_idx, dev_status)
    if (base == MOEDC_BF16)
        MOEDC_FUSED_LAUNCH(false, false);
    else if (cols)
        MOEDC_FUSED_LAUNCH(true, true);
    else
        MOEDC_FUSED_LAUNCH(true, false);
#undef MOEDC_FUSED_LAUNCH
    return launch_status();
}
