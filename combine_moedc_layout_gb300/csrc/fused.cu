// Layout + dispatch in one launch for small batches (T * K <= 1024 entries).
//
// Sources: MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on MI300X
// + CX7".  At 4-16 tokens the pages find latency flat in tokens and hidden
// size (host enqueue and launches dominate, host view-cache note), that
// per-token work splits leave most warps idle (CombineSync and MultiWarpIter
// notes: split by (token, slice) with a 512-element floor), and that a grid
// barrier cost more than the copy it was meant to parallelise (relay note:
// block-local barriers only).  So every block recomputes the tiny layout in
// shared memory and copies slices; nothing waits on another block.
//
// The block's latency chain is what the launch costs, so each step is kept
// short: the first x slice and all routing ids are loaded up front (one DRAM
// round trip for both), per-warp expert counts come from shared-memory
// atomics, the in-tile ranking uses a bit-sliced ballot match (eleven
// independent ballots; the hardware match instruction was measured several
// times slower here), and the layout outputs are written by the warps that
// touch them (a token's slots by the warp copying its first slice, each
// rank's distinct-token count by one warp of the grid) instead of by one
// block after the others have finished their copies.
#include <climits>
#include <mutex>

#include "dispatch_item.cuh"

namespace moedc {

// Block width follows the entry count: every thread holds two routing ids,
// so 128-thread blocks take up to 256 entries and 512-thread blocks the rest.
// Narrow blocks keep more SMs copying when there are few tokens; wide blocks
// shorten each warp's share of the layout when there are many (measured: at 4
// tokens 128 threads beat 512 by 3 us, at 1024 entries 512 beat 128 by 2 us).
constexpr int kFusedIdsPerThread = 2;
constexpr int kFusedNarrow = 128;
constexpr int kFusedWide = MOEDC_FUSED_MAX_ENTRIES / kFusedIdsPerThread;
static_assert(kFusedWide == 512, "wide fused block");

// Shared memory (int32 words) of one block of `threads` for n entries, E experts.
__host__ __device__ constexpr size_t fused_smem_words(int threads, int n, int E)
{
    return 2 * (size_t)n + (size_t)(threads / kWarp + 1) * E;
}

// The layout of all n entries, rebuilt in this block's shared memory: each
// warp owns a contiguous run of 32-entry tiles in (t, k) order; the run is
// counted per expert, the counts are scanned across warps, then equal
// experts are ranked inside each tile in lane order.  On return s_idx holds
// the routing ids, s_slot the slots (-1 for masked / out-of-range entries) and
// s_cnt the per-expert counts.
template <int kThreads>
__device__ __forceinline__ void block_layout(const int32_t* __restrict__ topk_idx, int n, int E,
                                             int32_t* s_idx, int32_t* s_slot, int32_t* s_wcnt,
                                             int32_t* s_cnt)
{
    constexpr int kFusedWarps = kThreads / kWarp;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    {
        int v[kFusedIdsPerThread];
#pragma unroll
        for (int j = 0; j < kFusedIdsPerThread; ++j) {
            const int i = threadIdx.x + j * kThreads;
            v[j] = i < n ? topk_idx[i] : 0;
        }
        for (int i = threadIdx.x; i < kFusedWarps * E; i += kThreads) s_wcnt[i] = 0;
#pragma unroll
        for (int j = 0; j < kFusedIdsPerThread; ++j) {
            const int i = threadIdx.x + j * kThreads;
            if (i < n) s_idx[i] = v[j];
        }
    }
    __syncthreads();
    const int run = ((n + kFusedWarps * kWarp - 1) / (kFusedWarps * kWarp)) * kWarp;
    const int wbeg = min(n, warp * run);
    const int wend = min(n, wbeg + run);
    int32_t* my = s_wcnt + warp * E;
    for (int i = wbeg + lane; i < wend; i += kWarp) {
        const int e = s_idx[i];
        if (e >= 0 && e < E) atomicAdd(&my[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) {
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
    const unsigned lt = lanemask_lt();
    for (int i0 = wbeg; i0 < wend; i0 += kWarp) {
        const int i = i0 + lane;
        const int e = i < wend ? s_idx[i] : -1;
        const bool v = e >= 0 && e < E;
        const unsigned peers = match_expert(e, v);
        int sv = -1;
        if (v) sv = my[e] + __popc(peers & lt);
        __syncwarp();
        if (v && (peers & lt) == 0) my[e] += __popc(peers);
        __syncwarp();
        if (i < wend) s_slot[i] = sv;
    }
    __syncthreads();
}

// The layout outputs no single warp owns: the expert counts (block 0, with
// the capacity check), each rank's distinct-token count (one warp of the grid
// per rank), and src_idx = -1 past each expert's count (grid-strided).
template <int kThreads>
__device__ __forceinline__ void publish_counts(int T, int K, int E, int R, int cap,
                                               const int32_t* s_idx, const int32_t* s_cnt,
                                               int32_t* __restrict__ num_tokens_per_expert,
                                               int32_t* __restrict__ num_tokens_per_rank,
                                               int32_t* __restrict__ src_idx,
                                               int32_t* __restrict__ status)
{
    constexpr int kFusedWarps = kThreads / kWarp;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int epr = E / R;
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += kThreads) {
            num_tokens_per_expert[e] = s_cnt[e];
            if (s_cnt[e] > cap) raise_status(status, MOEDC_ERR_CAPACITY);
        }
    }
    const int nwarps = gridDim.x * kFusedWarps;
    for (int r = blockIdx.x * kFusedWarps + warp; r < R; r += nwarps) {
        const unsigned lo = (unsigned)(r * epr);
        int c = 0;
        for (int t = lane; t < T; t += kWarp) {
            bool f = false;
            for (int k = 0; k < K; ++k) f |= (unsigned)s_idx[t * K + k] - lo < (unsigned)epr;
            c += f;
        }
        c = __reduce_add_sync(0xffffffffu, c);
        if (lane == 0) num_tokens_per_rank[r] = c;
    }
    const int64_t total = (int64_t)E * cap;
    const int64_t nthreads = (int64_t)gridDim.x * kThreads;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < total; i += nthreads) {
        const int e = (int)(i / cap);
        const int s = (int)(i - (int64_t)e * cap);
        if (s >= s_cnt[e]) src_idx[i] = -1;
    }
}

// A token's entries, published by the one warp that handles the token's
// first slice: its slots, src_idx of its rows, the expert-range check, and
// its token-in-rank row.
__device__ __forceinline__ void publish_token(int t, int lane, int K, int E, int R, int cap,
                                              const int32_t* s_idx, const int32_t* s_slot,
                                              int32_t* __restrict__ slot,
                                              uint8_t* __restrict__ is_token_in_rank,
                                              int32_t* __restrict__ src_idx,
                                              int32_t* __restrict__ status)
{
    const int epr = E / R;
    if (lane < K) {
        const int e = s_idx[t * K + lane];
        const int sv = s_slot[t * K + lane];
        const int row = dest_row(e, sv, E, cap);
        slot[t * K + lane] = sv;
        if (e < -1 || e >= E) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
        if (row >= 0) src_idx[row] = t;
    }
    for (int r = lane; r < R; r += kWarp) {
        const unsigned lo = (unsigned)(r * epr);
        uint8_t flag = 0;
        for (int k = 0; k < K; ++k)
            flag |= ((unsigned)s_idx[t * K + k] - lo < (unsigned)epr) ? 1 : 0;
        is_token_in_rank[(int64_t)t * R + r] = flag;
    }
}

template <int kThreads, bool kFp8, bool kScaleCols>
__global__ void __launch_bounds__(kThreads)
fused_layout_dispatch_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ topk_idx,
                             int T, int H, int K, int E, int R, int cap,
                             int32_t* __restrict__ num_tokens_per_expert,
                             int32_t* __restrict__ num_tokens_per_rank,
                             uint8_t* __restrict__ is_token_in_rank, int32_t* __restrict__ slot,
                             void* __restrict__ recv, float* __restrict__ scales,
                             int32_t* __restrict__ src_idx, int32_t* __restrict__ status)
{
    constexpr int kFusedWarps = kThreads / kWarp;
    pdl_enter();
    extern __shared__ int32_t smem[];
    const int n = T * K;                        // <= kThreads * kFusedIdsPerThread
    int32_t* s_idx = smem;                      // [n]
    int32_t* s_slot = s_idx + n;                // [n]
    int32_t* s_wcnt = s_slot + n;               // [kFusedWarps][E] per-warp counts, then offsets
    int32_t* s_cnt = s_wcnt + kFusedWarps * E;  // [E] totals
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int nslice = (H + kSlice - 1) / kSlice;
    const int items = T * nslice;
    const int nwarps = gridDim.x * kFusedWarps;

    // the warp's first x slice does not depend on the layout: start it now
    int item = blockIdx.x * kFusedWarps + warp;
    SliceX xv{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (item < items) {
        const int t = item / nslice;
        xv = load_slice<kFp8>(x + (int64_t)t * H, H, item - t * nslice, lane);
    }
    block_layout<kThreads>(topk_idx, n, E, s_idx, s_slot, s_wcnt, s_cnt);
    publish_counts<kThreads>(T, K, E, R, cap, s_idx, s_cnt, num_tokens_per_expert,
                             num_tokens_per_rank, src_idx, status);

    for (; item < items; item += nwarps) {
        const int t = item / nslice;
        const int sl = item - t * nslice;
        int my_row = -1;
        if (lane < K) my_row = dest_row(s_idx[t * K + lane], s_slot[t * K + lane], E, cap);
        if (sl == 0)
            publish_token(t, lane, K, E, R, cap, s_idx, s_slot, slot, is_token_in_rank, src_idx,
                          status);
        const int64_t sbase = kScaleCols ? colmajor_scale_base(my_row, cap, H / 128) : 0;
        store_slice<kFp8, kScaleCols>(xv, H, sl, lane, K, my_row, recv, scales, sbase, cap);
        const int next = item + nwarps;
        if (next < items) {
            const int t2 = next / nslice;
            xv = load_slice<kFp8>(x + (int64_t)t2 * H, H, next - t2 * nslice, lane);
        }
    }
}

// The same with one e4m3 scale per token row: a block owns one token at a
// time (wide blocks: warp w holds slices w, w + 16, ... in registers), the
// warps' maxima meet in shared memory behind one barrier per token (double
// buffered), then every warp quantises its slices and stores the copies.
template <int kJ>
__global__ void __launch_bounds__(kFusedWide)
fused_layout_dispatch_token_kernel(const uint16_t* __restrict__ x,
                                   const int32_t* __restrict__ topk_idx, int T, int H, int K,
                                   int E, int R, int cap,
                                   int32_t* __restrict__ num_tokens_per_expert,
                                   int32_t* __restrict__ num_tokens_per_rank,
                                   uint8_t* __restrict__ is_token_in_rank,
                                   int32_t* __restrict__ slot, uint8_t* __restrict__ recv,
                                   float* __restrict__ scales, int32_t* __restrict__ src_idx,
                                   int32_t* __restrict__ status)
{
    constexpr int kFusedWarps = kFusedWide / kWarp;
    pdl_enter();
    extern __shared__ int32_t smem[];
    __shared__ float s_amax[2][kFusedWarps];
    const int n = T * K;
    int32_t* s_idx = smem;
    int32_t* s_slot = s_idx + n;
    int32_t* s_wcnt = s_slot + n;
    int32_t* s_cnt = s_wcnt + kFusedWarps * E;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int nslice = (H + kSlice - 1) / kSlice;

    // the block's first token's slices do not depend on the layout: start them now
    SliceX v[kJ];
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
        const int sl = warp + j * kFusedWarps;
        v[j] = SliceX{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if ((int)blockIdx.x < T && sl < nslice)
            v[j] = load_slice_fp8(x + (int64_t)blockIdx.x * H, H, sl, lane);
    }
    block_layout<kFusedWide>(topk_idx, n, E, s_idx, s_slot, s_wcnt, s_cnt);
    publish_counts<kFusedWide>(T, K, E, R, cap, s_idx, s_cnt, num_tokens_per_expert,
                               num_tokens_per_rank, src_idx, status);

    int buf = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, buf ^= 1) {
        if (t != (int)blockIdx.x) {
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                const int sl = warp + j * kFusedWarps;
                v[j] = SliceX{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
                if (sl < nslice) v[j] = load_slice_fp8(x + (int64_t)t * H, H, sl, lane);
            }
        }
        int my_row = -1;
        if (lane < K) my_row = dest_row(s_idx[t * K + lane], s_slot[t * K + lane], E, cap);
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const uint32_t w[8] = {v[j].a.x, v[j].a.y, v[j].a.z, v[j].a.w,
                                   v[j].b.x, v[j].b.y, v[j].b.z, v[j].b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
                amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
        }
#pragma unroll
        for (int d = kWarp / 2; d > 0; d >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        if (lane == 0) s_amax[buf][warp] = amax;
        __syncthreads();   // one per token; the other buffer is written next time
        float a = 0.0f;
        for (int w = 0; w < kFusedWarps; ++w) a = fmaxf(a, s_amax[buf][w]);
        a = fmaxf(a, 1e-4f);
        const float sc = __fdiv_rn(a, 448.0f);
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const int sl = warp + j * kFusedWarps;
            if (sl >= nslice) continue;   // uniform across the warp
            const int c0 = sl * kSlice + lane * 16;
            const uint32_t w[8] = {v[j].a.x, v[j].a.y, v[j].a.z, v[j].a.w,
                                   v[j].b.x, v[j].b.y, v[j].b.z, v[j].b.w};
            uint32_t p[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t lo = quant_pair(bf16_lo(w[2 * q]), bf16_hi(w[2 * q]), sc);
                const uint32_t hi = quant_pair(bf16_lo(w[2 * q + 1]), bf16_hi(w[2 * q + 1]), sc);
                p[q] = lo | (hi << 16);
            }
            const uint4 qv = make_uint4(p[0], p[1], p[2], p[3]);
            for (int k = 0; k < K; ++k) {
                const int row = __shfl_sync(0xffffffffu, my_row, k);
                if (row >= 0 && c0 < H)
                    st_global_recv(reinterpret_cast<uint4*>(recv + (int64_t)row * H + c0), qv);
            }
        }
        if (warp == 0) {
            publish_token(t, lane, K, E, R, cap, s_idx, s_slot, slot, is_token_in_rank, src_idx,
                          status);
            if (lane < K && my_row >= 0) st_global_recv_f32(scales + my_row, sc);
        }
    }
}

}  // namespace moedc

namespace {

// The wide block at its largest (1024 entries, MOEDC_MAX_E experts) needs
// more than the default 48 KB of dynamic shared memory: raise the limit of
// its instances once.  The attribute is per function and per device.
// (The narrow block needs at most 2 * 256 + 5 * MOEDC_MAX_E words, 22.5 KB.)
constexpr int kMaxDevices = 64;
std::mutex g_smem_mutex;
bool g_smem_set[kMaxDevices] = {};

bool fused_smem_ready()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_smem_mutex);
    if (g_smem_set[dev]) return true;
    constexpr int W = moedc::kFusedWide;
    const int bytes = (int)(moedc::fused_smem_words(W, MOEDC_FUSED_MAX_ENTRIES, MOEDC_MAX_E) *
                            sizeof(int32_t));
    if (cudaFuncSetAttribute(moedc::fused_layout_dispatch_kernel<W, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(moedc::fused_layout_dispatch_kernel<W, true, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(moedc::fused_layout_dispatch_kernel<W, true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(moedc::fused_layout_dispatch_token_kernel<1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(moedc::fused_layout_dispatch_token_kernel<2>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
        cudaFuncSetAttribute(moedc::fused_layout_dispatch_token_kernel<4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    g_smem_set[dev] = true;
    return true;
}

}  // namespace

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
    const bool per_token = (out_dtype & MOEDC_SCALES_PER_TOKEN) != 0;
    const int base = dtype_base(out_dtype);
    if (per_token && H > MOEDC_TOKEN_SCALE_MAX_H) return MOEDC_ERR_ARG;
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
    if (n > MOEDC_FUSED_MAX_ENTRIES && !per_token) {
        const int st = launch_layout_dispatch_coop(
            x, topk_idx, T, H, K, E, R, cap, out_dtype, num_tokens_per_expert,
            num_tokens_per_rank, is_token_in_rank, slot, recv, scales, src_idx, workspace,
            workspace_bytes, dev_status, stream);
        if (st != MOEDC_ERR_UNIMPLEMENTED) return st;
    }
    if (n > MOEDC_FUSED_MAX_ENTRIES) {
        const LayoutGeom g = layout_geometry(T, K, E, R);
        if (g.ws > 0 && (!workspace || workspace_bytes < g.ws || !aligned(workspace, 16)))
            return MOEDC_ERR_ARG;
        int st = launch_layout(topk_idx, T, K, E, R, cap, num_tokens_per_expert,
                               num_tokens_per_rank, is_token_in_rank, slot, workspace,
                               workspace_bytes, dev_status, stream);
        if (st != MOEDC_OK) return st;
        return launch_dispatch(x, T, H, topk_idx, slot, num_tokens_per_expert, K, E, cap,
                               out_dtype, recv, scales, src_idx, dev_status, stream);
    }

    const int nslice = (H + moedc::kSlice - 1) / moedc::kSlice;
    if (per_token) {   // a block owns whole tokens: a row's scale needs all its slices
        constexpr int W = moedc::kFusedWide;
        const int per_warp = (nslice + W / moedc::kWarp - 1) / (W / moedc::kWarp);   // 1 .. 4
        const void* fn = per_warp == 1   ? (const void*)moedc::fused_layout_dispatch_token_kernel<1>
                         : per_warp == 2 ? (const void*)moedc::fused_layout_dispatch_token_kernel<2>
                                         : (const void*)moedc::fused_layout_dispatch_token_kernel<4>;
        if (!fused_smem_ready()) return MOEDC_ERR_CUDA;
        const size_t sm = moedc::fused_smem_words(W, (int)n, E) * sizeof(int32_t);
        const int64_t fill_blocks = ((int64_t)E * cap + W - 1) / W;
        int64_t blocks = T > fill_blocks ? T : fill_blocks;
        const int64_t resident = resident_blocks(fn, W, sm);
        if (blocks > resident) blocks = resident;
        if (blocks < 1) blocks = 1;
        const uint16_t* xb = static_cast<const uint16_t*>(x);
        uint8_t* rb = static_cast<uint8_t*>(recv);
        clear_stale_error();
#define MOEDC_FUSED_TOKEN_LAUNCH(J)                                                               \
    launch(moedc::fused_layout_dispatch_token_kernel<J>, (int)blocks, W, sm, stream, xb, topk_idx, \
           T, H, K, E, R, cap, num_tokens_per_expert, num_tokens_per_rank, is_token_in_rank, slot, \
           rb, scales, src_idx, dev_status)
        if (per_warp == 1)
            MOEDC_FUSED_TOKEN_LAUNCH(1);
        else if (per_warp == 2)
            MOEDC_FUSED_TOKEN_LAUNCH(2);
        else
            MOEDC_FUSED_TOKEN_LAUNCH(4);
#undef MOEDC_FUSED_TOKEN_LAUNCH
        return launch_status();
    }
    const int64_t items = (int64_t)T * nslice;
    const bool wide = n > (int64_t)moedc::kFusedNarrow * moedc::kFusedIdsPerThread;
    const int threads = wide ? moedc::kFusedWide : moedc::kFusedNarrow;
    int64_t blocks = (items + threads / moedc::kWarp - 1) / (threads / moedc::kWarp);
    const int64_t fill_blocks = ((int64_t)E * cap + threads - 1) / threads;
    if (blocks < fill_blocks) blocks = fill_blocks;
    const void* fn;
    if (wide) {
        constexpr int W = moedc::kFusedWide;
        fn = base == MOEDC_BF16 ? (const void*)moedc::fused_layout_dispatch_kernel<W, false, false>
             : cols             ? (const void*)moedc::fused_layout_dispatch_kernel<W, true, true>
                                : (const void*)moedc::fused_layout_dispatch_kernel<W, true, false>;
        if (!fused_smem_ready()) return MOEDC_ERR_CUDA;
    } else {
        constexpr int N = moedc::kFusedNarrow;
        fn = base == MOEDC_BF16 ? (const void*)moedc::fused_layout_dispatch_kernel<N, false, false>
             : cols             ? (const void*)moedc::fused_layout_dispatch_kernel<N, true, true>
                                : (const void*)moedc::fused_layout_dispatch_kernel<N, true, false>;
    }
    const size_t sm = moedc::fused_smem_words(threads, (int)n, E) * sizeof(int32_t);
    const int64_t resident = resident_blocks(fn, threads, sm);
    if (blocks > resident) blocks = resident;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    clear_stale_error();
#define MOEDC_FUSED_LAUNCH(NT, F, C)                                                             \
    launch(moedc::fused_layout_dispatch_kernel<NT, F, C>, (int)blocks, NT, sm, stream, xb,       \
           topk_idx, T, H, K, E, R, cap, num_tokens_per_expert, num_tokens_per_rank,            \
           is_token_in_rank, slot, recv, scales, src_idx, dev_status)
#define MOEDC_FUSED_DTYPE(NT)                                                                    \
    do {                                                                                         \
        if (base == MOEDC_BF16)                                                                  \
            MOEDC_FUSED_LAUNCH(NT, false, false);                                                \
        else if (cols)                                                                           \
            MOEDC_FUSED_LAUNCH(NT, true, true);                                                  \
        else                                                                                     \
            MOEDC_FUSED_LAUNCH(NT, true, false);                                                 \
    } while (0)
    if (wide)
        MOEDC_FUSED_DTYPE(moedc::kFusedWide);
    else
        MOEDC_FUSED_DTYPE(moedc::kFusedNarrow);
#undef MOEDC_FUSED_DTYPE
#undef MOEDC_FUSED_LAUNCH
    return launch_status();
}
