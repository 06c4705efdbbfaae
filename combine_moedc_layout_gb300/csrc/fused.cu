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

template <bool kFp8>
__global__ void __launch_bounds__(kFusedThreads)
fused_layout_dispatch_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_idx,
                             int T, int H, int K, int E, int R, int cap,
                             int32_t* __restrict__ num_tokens_per_expert,
                             int32_t* __restrict__ num_tokens_per_rank,
                             uint8_t* __restrict__ is_token_in_rank, int32_t* __restrict__ slot,
                             void* __restrict__ recv, float* __restrict__ scales,
                             int32_t* __restrict__ src_idx, int32_t* __restrict__ status)
{
    extern __shared__ int32_t smem[];
    const int n = T * K;
    int32_t* s_idx = smem;          // [n]
    int32_t* s_slot = s_idx + n;    // [n]
    int32_t* s_cnt = s_slot + n;    // [E]
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int epr = E / R;

    for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = 0;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_idx[i] = topk_idx[i];
    __syncthreads();

    // layout, one warp, 32 entries at a time in (t, k) order
    if (warp == 0) {
        const unsigned lt = lanemask_lt();
        for (int i0 = 0; i0 < n; i0 += kWarp) {
            const int i = i0 + lane;
            const int e = i < n ? s_idx[i] : -1;
            const bool v = e >= 0 && e < E;
            const unsigned peers = __match_any_sync(0xffffffffu, v ? e : -1);
            int s = -1;
            if (v) s = s_cnt[e] + __popc(peers & lt);
            __syncwarp();
            if (v && (peers & lt) == 0) s_cnt[e] += __popc(peers);
            __syncwarp();
            if (i < n) s_slot[i] = s;
        }
    }
    __syncthreads();

    if (blockIdx.x == 0) {
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
        for (int b = threadIdx.x; b < T * R; b += blockDim.x) {
            const int t = b / R;
            const int r = b - t * R;
            uint8_t flag = 0;
            for (int k = 0; k < K; ++k) {
                const int e = s_idx[t * K + k];
                if (e >= 0 && e < E && e / epr == r) flag = 1;
            }
            is_token_in_rank[b] = flag;
        }
        for (int r = threadIdx.x; r < R; r += blockDim.x) {
            int c = 0;
            for (int t = 0; t < T; ++t) {
                bool in = false;
                for (int k = 0; k < K; ++k) {
                    const int e = s_idx[t * K + k];
                    if (e >= 0 && e < E && e / epr == r) in = true;
                }
                c += in ? 1 : 0;
            }
            num_tokens_per_rank[r] = c;
        }
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
        store_slice<kFp8>(v, H, sl, lane, K, my_row, recv, scales);
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
    if (H < 8 || (out_dtype == MOEDC_BF16 && H % 8 != 0) ||
        (out_dtype == MOEDC_FP8_E4M3 && H % 128 != 0) ||
        (out_dtype != MOEDC_BF16 && out_dtype != MOEDC_FP8_E4M3))
        return MOEDC_ERR_ARG;
    if (!num_tokens_per_expert || !num_tokens_per_rank || !dev_status || !recv || !src_idx)
        return MOEDC_ERR_ARG;
    if ((int64_t)E * cap > INT32_MAX || (int64_t)T * ((H + 511) / 512) > INT32_MAX / 2)
        return MOEDC_ERR_ARG;
    if (out_dtype == MOEDC_FP8_E4M3 && !scales) return MOEDC_ERR_ARG;
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
    const void* fn = out_dtype == MOEDC_FP8_E4M3
                         ? (const void*)moedc::fused_layout_dispatch_kernel<true>
                         : (const void*)moedc::fused_layout_dispatch_kernel<false>;
    const int64_t resident = resident_blocks(fn, moedc::kFusedThreads, (size_t)(2 * n + E) * 4);
    if (blocks > resident) blocks = resident;
    if (blocks < 1) blocks = 1;
    const size_t sm = (size_t)(2 * n + E) * sizeof(int32_t);
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    clear_stale_error();
    if (out_dtype == MOEDC_FP8_E4M3)
        moedc::fused_layout_dispatch_kernel<true><<<(int)blocks, moedc::kFusedThreads, sm, stream>>>(
            xb, topk_idx, T, H, K, E, R, cap, num_tokens_per_expert, num_tokens_per_rank,
            is_token_in_rank, slot, recv, scales, src_idx, dev_status);
    else
        moedc::fused_layout_dispatch_kernel<false><<<(int)blocks, moedc::kFusedThreads, sm, stream>>>(
            xb, topk_idx, T, H, K, E, R, cap, num_tokens_per_expert, num_tokens_per_rank,
            is_token_in_rank, slot, recv, scales, src_idx, dev_status);
    return launch_status();
}
