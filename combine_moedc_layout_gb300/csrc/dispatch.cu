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
#ifndef MOEDC_DISPATCH_BULK
#define MOEDC_DISPATCH_BULK 0   // 1: rows leave through shared-memory stages and bulk copies
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

// Bulk-copy staging: a warp writes its slice (e4m3 codes, or the bf16 row
// segment) into a shared-memory stage, and one lane sends the stage to each
// of the token's destination rows with one cp.async.bulk shared -> global
// copy per row, instead of every lane storing 16 bytes per row.  Two stages
// per warp: a stage is rewritten only after the copies issued from it two
// items earlier have finished reading it (bulk_group wait.read).  All copies
// are 1-D, to this GPU's own memory; rows and stages are 16-byte aligned and
// a slice is a multiple of 16 bytes (H % 128 == 0 for e4m3, H % 8 == 0 for
// bf16).
__device__ __forceinline__ void bulk_s2g(void* gdst, uint32_t ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gdst), "r"(ssrc), "r"(bytes) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

template <bool kFp8, bool kScaleCols>
__global__ void __launch_bounds__(kDispatchThreads, MOEDC_DISPATCH_MINB)
dispatch_bulk_kernel(const uint16_t* __restrict__ x, int T, int H,
                     const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot,
                     const int32_t* __restrict__ num_tokens_per_expert, int K, int E, int cap,
                     void* __restrict__ recv, float* __restrict__ scales,
                     int32_t* __restrict__ src_idx, int32_t* __restrict__ status)
{
    pdl_enter();
    constexpr int kStageBytes = 2 * kSlice;   // a bf16 slice; an e4m3 slice uses half
    __shared__ __align__(128) uint8_t s_stage[kDispatchThreads / kWarp][2][kStageBytes];
    const int lane = threadIdx.x % kWarp;
    const int wib = threadIdx.x / kWarp;
    const int nslice = (H + kSlice - 1) / kSlice;
    const int nwarps = gridDim.x * (blockDim.x / kWarp);
    const int dt = nwarps / nslice, dsl = nwarps - dt * nslice;
    const int G = H / 128;
    constexpr int esz = kFp8 ? 1 : 2;
    uint8_t* recv_b = static_cast<uint8_t*>(recv);
    const uint32_t stage0 = (uint32_t)__cvta_generic_to_shared(&s_stage[wib][0][0]);
    bool bad = false;

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
    int buf = 0;
    while (cur.t < T) {
        ItemCursor nxt = cur;
        nxt.advance(dt, dsl, nslice);
        int nx_row;
        SliceX nx_v;
        load_item(nxt, nx_row, nx_v);
        if (cur.sl == 0 && lane < K && my_row >= 0) src_idx[my_row] = cur.t;
        const int c0 = cur.sl * kSlice;
        const int nch = min(kSlice, H - c0);
        const uint32_t sb = stage0 + buf * kStageBytes;
        // the copies issued from this stage two items ago must have read it
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncwarp();
        float sc = 0.0f;
        if (kFp8) {
            const SliceQ sq = quant_slice_fp8(xv);
            sc = sq.sc;
            if (lane * 16 < nch) st_shared_v4(sb + lane * 16, sq.q);
        } else {
            if (lane * 8 < nch) st_shared_v4(sb + lane * 16, xv.a);
            if (256 + lane * 8 < nch) st_shared_v4(sb + 512 + lane * 16, xv.b);
        }
        // the stage's generic-proxy writes, visible to the bulk copies
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        const bool leader = kFp8 && (lane & 7) == 0 && lane * 16 < nch;
        const int g = (c0 + lane * 16) / 128;
        for (int k = 0; k < K; ++k) {
            const int row = __shfl_sync(0xffffffffu, my_row, k);
            if (row < 0) continue;
            if (lane == 0) bulk_s2g(recv_b + ((int64_t)row * H + c0) * esz, sb, (uint32_t)(nch * esz));
            if (leader) {
                const int64_t si = kScaleCols ? colmajor_scale_base(row, cap, G) + (int64_t)g * cap
                                              : (int64_t)row * G + g;
                st_global_cs_f32(scales + si, sc);
            }
        }
        if (lane == 0) asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        buf ^= 1;
        cur = nxt;
        my_row = nx_row;
        xv = nx_v;
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);

    // slots no entry reaches carry src_idx = -1
    const int64_t total = (int64_t)E * cap;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += nthreads) {
        const int e = (int)(i / cap);
        const int s2 = (int)(i - (int64_t)e * cap);
        if (s2 >= __ldg(num_tokens_per_expert + e)) src_idx[i] = -1;
    }
}

// Whole-row bulk copies (e4m3, row-major scales): a block owns a token; its
// warps quantise slices w, w + 8, ... into a shared-memory row stage (codes,
// then the row's scales), and one thread sends the codes and the scales to
// each destination row with two bulk copies.  Two stages; a stage is
// rewritten only after the copies of two tokens earlier have read it.
constexpr int kRowStageMax = 16384;   // codes + scales of one row, bytes

__global__ void __launch_bounds__(kDispatchThreads, 2)
dispatch_rowbulk_kernel(const uint16_t* __restrict__ x, int T, int H,
                        const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot,
                        const int32_t* __restrict__ num_tokens_per_expert, int K, int E, int cap,
                        uint8_t* __restrict__ recv, float* __restrict__ scales,
                        int32_t* __restrict__ src_idx, int32_t* __restrict__ status)
{
    pdl_enter();
    extern __shared__ __align__(128) uint8_t s_rows[];   // [2][row stage]
    __shared__ int s_dest[2][kWarp];
    const int lane = threadIdx.x % kWarp;
    const int wib = threadIdx.x / kWarp;
    constexpr int W = kDispatchThreads / kWarp;
    const int nslice = H / kSlice + (H % kSlice ? 1 : 0);
    const int G = H / 128;
    const int stage_bytes = (H + 4 * G + 127) / 128 * 128;
    const uint32_t stage0 = (uint32_t)__cvta_generic_to_shared(s_rows);
    bool bad = false;
    int buf = 0;
    // this warp's slices (at most 2 per warp while a row has <= 16 slices) of
    // the block's current token, loaded one token ahead
    SliceX xv[2];
    auto load_row = [&](int t) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int sl = wib + j * W;
            xv[j] = (t < T && sl < nslice) ? load_slice_fp8(x + (int64_t)t * H, H, sl, lane)
                                           : SliceX{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        }
    };
    load_row(blockIdx.x);
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (wib == 0) {
            int row = -1;
            if (lane < K) {
                const int e = __ldg(topk_idx + (int64_t)t * K + lane);
                const int s = __ldg(slot + (int64_t)t * K + lane);
                row = dest_row(e, s, E, cap);
                if (e < -1 || e >= E) bad = true;
                if (row >= 0) src_idx[row] = t;
            }
            s_dest[buf][lane] = row;
        }
        // the copies issued from this stage two tokens ago must have read it
        if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        uint8_t* stage = s_rows + buf * stage_bytes;
        const uint32_t sb = stage0 + buf * stage_bytes;
        float* s_sc = reinterpret_cast<float*>(stage + H);
        SliceQ sq[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) sq[j] = quant_slice_fp8(xv[j]);
        load_row(t + gridDim.x);   // the next token's slices travel while this one is staged
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c0 = (wib + j * W) * kSlice + lane * 16;
            if (c0 < H) {
                st_shared_v4(sb + c0, sq[j].q);
                if ((lane & 7) == 0) s_sc[c0 / 128] = sq[j].sc;
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int k = 0; k < K; ++k) {
                const int row = s_dest[buf][k];
                if (row < 0) continue;
                bulk_s2g(recv + (int64_t)row * H, sb, (uint32_t)H);
                bulk_s2g(scales + (int64_t)row * G, sb + H, (uint32_t)(4 * G));
            }
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        buf ^= 1;
    }
    if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
    const int64_t total = (int64_t)E * cap;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += nthreads) {
        const int e = (int)(i / cap);
        const int s2 = (int)(i - (int64_t)e * cap);
        if (s2 >= __ldg(num_tokens_per_expert + e)) src_idx[i] = -1;
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
#if MOEDC_DISPATCH_BULK == 2
    // e4m3 with row-major scales and 16-byte aligned scale rows: whole-row copies
    if (base == MOEDC_FP8_E4M3 && !cols && (H / 128) % 4 == 0 && aligned(scales, 16) &&
        H <= 2 * moedc::kSlice * (moedc::kDispatchThreads / moedc::kWarp) &&
        (size_t)((H + 4 * (H / 128) + 127) / 128 * 128) <= (size_t)moedc::kRowStageMax) {
        const size_t stage = (size_t)((H + 4 * (H / 128) + 127) / 128 * 128);
        const size_t sm = 2 * stage;
        static bool attr = cudaFuncSetAttribute((const void*)moedc::dispatch_rowbulk_kernel,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                2 * moedc::kRowStageMax) == cudaSuccess;
        if (attr) {
            int64_t rb = T;
            const int64_t fill_b = (fill + moedc::kDispatchThreads - 1) / moedc::kDispatchThreads;
            if (rb < fill_b) rb = fill_b;
            const int64_t res = resident_blocks((const void*)moedc::dispatch_rowbulk_kernel,
                                                moedc::kDispatchThreads, sm);
            if (rb > res) rb = res;
            if (rb < 1) rb = 1;
            clear_stale_error();
            launch(moedc::dispatch_rowbulk_kernel, (int)rb, moedc::kDispatchThreads, sm, stream,
                   static_cast<const uint16_t*>(x), T, H, topk_idx, slot, num_tokens_per_expert, K,
                   E, cap, static_cast<uint8_t*>(recv), scales, src_idx, dev_status);
            return launch_status();
        }
    }
#endif
#if MOEDC_DISPATCH_BULK == 1
    {
        const void* fn = base == MOEDC_BF16 ? (const void*)moedc::dispatch_bulk_kernel<false, false>
                         : cols             ? (const void*)moedc::dispatch_bulk_kernel<true, true>
                                            : (const void*)moedc::dispatch_bulk_kernel<true, false>;
        const int64_t resident = resident_blocks(fn, moedc::kDispatchThreads, 0);
        if (blocks > resident) blocks = resident;
        if (blocks < 1) blocks = 1;
        const uint16_t* xb = static_cast<const uint16_t*>(x);
        clear_stale_error();
        if (base == MOEDC_BF16)
            launch(moedc::dispatch_bulk_kernel<false, false>, (int)blocks, moedc::kDispatchThreads, 0,
                   stream, xb, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, recv, scales,
                   src_idx, dev_status);
        else if (cols)
            launch(moedc::dispatch_bulk_kernel<true, true>, (int)blocks, moedc::kDispatchThreads, 0,
                   stream, xb, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, recv, scales,
                   src_idx, dev_status);
        else
            launch(moedc::dispatch_bulk_kernel<true, false>, (int)blocks, moedc::kDispatchThreads, 0,
                   stream, xb, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap, recv, scales,
                   src_idx, dev_status);
        return launch_status();
    }
#endif
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
