// Dispatch: scatter token rows into expert slots (bf16 copy or e4m3 + scales)
// and write the per-slot source-token index.
//
// Sources: DeepEP PR #693 "Pipeline direct NVLink dispatch with
// triple-buffered prefetch", Summary (hidden data, scale factors and routing
// of a token move together); MORI PR #614 "perf(ep): InterNodeV1LL low-token
// latency on MI300X + CX7" (flat stride over work items instead of per-block
// token ranges).  On one GPU the "remote store" is a plain HBM store, so the
// kernel is a write stream: each token row is read once and written K times.
#include <climits>

#include "dispatch_item.cuh"

namespace moedc {

#ifndef MOEDC_DISPATCH_MINB
#define MOEDC_DISPATCH_MINB 4
#endif

constexpr int kDispatchThreads = 256;

template <bool kFp8, bool kScaleCols>
__global__ void __launch_bounds__(kDispatchThreads, MOEDC_DISPATCH_MINB)
dispatch_kernel(const uint16_t* __restrict__ x, int T, int H,
                const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot,
                const int32_t* __restrict__ num_tokens_per_expert, int K, int E, int cap,
                void* __restrict__ recv, float* __restrict__ scales,
                int32_t* __restrict__ src_idx, int32_t* __restrict__ status)
{
    pdl_enter();
    const int lane = threadIdx.x % kWarp;
    const int nslice = (H + kSlice - 1) / kSlice;
    const int nwarps = gridDim.x * (blockDim.x / kWarp);
    const int dt = nwarps / nslice, dsl = nwarps - dt * nslice;
    bool bad = false;

    // a work item's inputs: the destination row of routing entry k == lane,
    // and the lane's x vectors
    auto load_item = [&](const ItemCursor& c, int& row, SliceX& v) {
        row = -1;
        v = SliceX{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (c.t >= T) return;
        if (lane < K) {
            const int e = __ldg(topk_idx + (int64_t)c.t * K + lane);
            const int s = __ldg(slot + (int64_t)c.t * K + lane);
            row = dest_row(e, s, E, cap);
            if (c.sl == 0 && (e < -1 || e >= E)) bad = true;
        }
        v = load_slice<kFp8>(x + (int64_t)c.t * H, H, c.sl, lane);
    };
    ItemCursor cur;
    cur.init(blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp, nslice);
    int my_row;
    SliceX xv;
    load_item(cur, my_row, xv);
    while (cur.t < T) {
        // the next item's routing and x travel while this one is stored
        ItemCursor nxt = cur;
        nxt.advance(dt, dsl, nslice);
        int nx_row;
        SliceX nx_v;
        load_item(nxt, nx_row, nx_v);
        if (cur.sl == 0 && lane < K && my_row >= 0) src_idx[my_row] = cur.t;
        const int64_t sbase = kScaleCols ? colmajor_scale_base(my_row, cap, H / 128) : 0;
        store_slice<kFp8, kScaleCols>(xv, H, cur.sl, lane, K, my_row, recv, scales, sbase, cap);
        cur = nxt;
        my_row = nx_row;
        xv = nx_v;
    }
    if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);

    // slots no entry reaches carry src_idx = -1
    const int64_t total = (int64_t)E * cap;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += nthreads) {
        const int e = (int)(i / cap);
        const int s = (int)(i - (int64_t)e * cap);
        if (s >= __ldg(num_tokens_per_expert + e)) src_idx[i] = -1;
    }
}

}  // namespace moedc

namespace moedc_host {

static bool dispatch_args_ok(const void* x, int T, int H, const int32_t* topk_idx,
                             const int32_t* slot, const int32_t* cnt, int K, int E, int cap,
                             int out_dtype, const void* recv, const float* scales,
                             const int32_t* src_idx, const int32_t* dev_status)
{
    if (T < 0 || H < 8 || K < 1 || K > MOEDC_MAX_K || E < 1 || E > MOEDC_MAX_E || cap < 1)
        return false;
    if (!dtype_ok(out_dtype)) return false;
    if ((out_dtype & MOEDC_SCALES_PER_TOKEN) && H > MOEDC_TOKEN_SCALE_MAX_H) return false;
    out_dtype = dtype_base(out_dtype);
    if (out_dtype == MOEDC_BF16 && H % 8 != 0) return false;
    if (out_dtype == MOEDC_FP8_E4M3 && H % 128 != 0) return false;
    if ((int64_t)E * cap > INT32_MAX) return false;
    if ((int64_t)T * ((H + 511) / 512) > INT32_MAX / 2) return false;
    if (!cnt || !recv || !src_idx || !dev_status) return false;
    if (out_dtype == MOEDC_FP8_E4M3 && !scales) return false;
    if (out_dtype == MOEDC_FP8_E4M3 && (int64_t)E * cap * (H / 128) > INT32_MAX) return false;
    if (T > 0 && (!x || !topk_idx || !slot)) return false;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(scales, 4) || !aligned(topk_idx, 4) ||
        !aligned(slot, 4) || !aligned(cnt, 4) || !aligned(src_idx, 4) || !aligned(dev_status, 4))
        return false;
    return true;
}

int launch_dispatch(const void* x, int T, int H, const int32_t* topk_idx, const int32_t* slot,
                    const int32_t* num_tokens_per_expert, int K, int E, int cap, int out_dtype,
                    void* recv, float* scales, int32_t* src_idx, int32_t* dev_status,
                    cudaStream_t stream)
{
    if (out_dtype & MOEDC_SCALES_PER_TOKEN)
        return launch_dispatch_token(x, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap,
                                     recv, scales, src_idx, dev_status, stream);
    const int warps_per_block = moedc::kDispatchThreads / moedc::kWarp;
    const int nslice = (H + moedc::kSlice - 1) / moedc::kSlice;
    const int64_t items = (int64_t)T * nslice;
    const int64_t fill = (int64_t)E * cap;
    int64_t blocks = (items + warps_per_block - 1) / warps_per_block;
    const int64_t fill_blocks = (fill + moedc::kDispatchThreads - 1) / moedc::kDispatchThreads;
    if (blocks < fill_blocks) blocks = fill_blocks;
    const bool cols = (out_dtype & MOEDC_SCALES_COL_MAJOR) != 0;
    const int base = out_dtype & ~MOEDC_SCALES_COL_MAJOR;
    const void* fn = base == MOEDC_BF16 ? (const void*)moedc::dispatch_kernel<false, false>
                     : cols             ? (const void*)moedc::dispatch_kernel<true, true>
                                        : (const void*)moedc::dispatch_kernel<true, false>;
    const int64_t resident = resident_blocks(fn, moedc::kDispatchThreads, 0);
    if (blocks > resident) blocks = resident;
    if (blocks < 1) blocks = 1;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    clear_stale_error();
    if (base == MOEDC_BF16)
        launch(moedc::dispatch_kernel<false, false>, (int)blocks, moedc::kDispatchThreads, 0, stream, xb, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, recv, scales, src_idx,
            dev_status);
    else if (cols)
        launch(moedc::dispatch_kernel<true, true>, (int)blocks, moedc::kDispatchThreads, 0, stream, xb, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, recv, scales, src_idx,
            dev_status);
    else
        launch(moedc::dispatch_kernel<true, false>, (int)blocks, moedc::kDispatchThreads, 0, stream, xb, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, recv, scales, src_idx,
            dev_status);
    return launch_status();
}

}  // namespace moedc_host

extern "C" int moedc_dispatch(const void* x, int T, int H, const int32_t* topk_idx,
                              const int32_t* slot, const int32_t* num_tokens_per_expert, int K,
                              int E, int cap, int out_dtype, void* recv, float* scales,
                              int32_t* src_idx, int32_t* dev_status, cudaStream_t stream)
{
    using namespace moedc_host;
    if (!dispatch_args_ok(x, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, out_dtype,
                          recv, scales, src_idx, dev_status))
        return MOEDC_ERR_ARG;
    return launch_dispatch(x, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, out_dtype,
                           recv, scales, src_idx, dev_status, stream);
}
