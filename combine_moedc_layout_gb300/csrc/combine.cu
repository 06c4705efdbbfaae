// Combine: weighted gather-reduce of each token's K expert rows back into
// token order, binary32 accumulation in ascending k, bf16 output.
//
// Sources: MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on MI300X
// + CX7" — CombineSync note (split by (token, hidden slice), not by token, so
// a handful of tokens still spreads over the whole grid) and the zero-copy
// combine input note (the caller's expert outputs are read in place, never
// staged).  The kernel is an HBM read stream: K gathered rows per token.
#include <climits>

#include "common.cuh"

// Tuning knobs (compile-time): 16-byte vectors per lane per gathered row,
// rows whose loads are in flight together, and the minimum resident blocks
// per SM the register budget must allow.
#ifndef MOEDC_COMBINE_VEC
#define MOEDC_COMBINE_VEC 2
#endif
#ifndef MOEDC_COMBINE_BATCH
#define MOEDC_COMBINE_BATCH 8
#endif
#ifndef MOEDC_COMBINE_MINB
#define MOEDC_COMBINE_MINB 2
#endif

namespace moedc {

constexpr int kCombineThreads = 256;
constexpr int kCombineVec = MOEDC_COMBINE_VEC;
constexpr int kCombineSlice = 256 * kCombineVec;   // channels per warp item
constexpr int kCombineBatch = MOEDC_COMBINE_BATCH;

__global__ void __launch_bounds__(kCombineThreads, MOEDC_COMBINE_MINB)
combine_kernel(const uint16_t* __restrict__ expert_out, int E, int cap, int H,
               const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot,
               const float* __restrict__ topk_weights, int T, int K,
               uint16_t* __restrict__ y, int32_t* __restrict__ status, float neg_zero)
{
    pdl_enter();
    const int lane = threadIdx.x % kWarp;
    const int nslice = (H + kCombineSlice - 1) / kCombineSlice;
    const int64_t items = (int64_t)T * nslice;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / kWarp);
    bool bad = false;

    // routing entries of a work item: lane k < K holds entry k (expert, slot, weight)
    auto load_routing = [&](int64_t it, int& e, int& s, float& w) {
        e = -1; s = -1; w = 0.0f;
        if (it < items && lane < K) {
            const int64_t t = it / nslice;
            e = __ldg(topk_idx + t * K + lane);
            s = __ldg(slot + t * K + lane);
            w = __ldg(topk_weights + t * K + lane);
        }
    };
    int64_t item = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp;
    int my_e, my_s;
    float my_w;
    load_routing(item, my_e, my_s, my_w);
    for (; item < items; item += nwarps) {
        const int t = (int)(item / nslice);
        const int sl = (int)(item - (int64_t)t * nslice);
        if (sl == 0 && lane < K && (my_e < -1 || my_e >= E)) bad = true;
        // vector v of this lane covers channels c[v] .. c[v] + 8; each warp-wide
        // 16-byte access covers 512 contiguous bytes
        int c[kCombineVec];
        bool act[kCombineVec];
#pragma unroll
        for (int v = 0; v < kCombineVec; ++v) {
            c[v] = sl * kCombineSlice + v * 256 + lane * 8;
            act[v] = c[v] < H;
        }
        float2 acc[4 * kCombineVec];   // channel pairs
#pragma unroll
        for (int i = 0; i < 4 * kCombineVec; ++i) acc[i] = make_float2(0.0f, 0.0f);
        int nx_e, nx_s;
        float nx_w;

        for (int k0 = 0; k0 < K; k0 += kCombineBatch) {
            uint4 buf[kCombineBatch][kCombineVec];
            float wk[kCombineBatch];
            bool ok[kCombineBatch];
#pragma unroll
            for (int j = 0; j < kCombineBatch; ++j) {
                const int k = k0 + j;
                const int e = __shfl_sync(0xffffffffu, my_e, k & 31);
                const int s = __shfl_sync(0xffffffffu, my_s, k & 31);
                wk[j] = __shfl_sync(0xffffffffu, my_w, k & 31);
                ok[j] = k < K && e >= 0 && e < E && s >= 0 && s < cap;
                const uint16_t* row = ok[j] ? expert_out + ((int64_t)e * cap + s) * H : expert_out;
#pragma unroll
                for (int v = 0; v < kCombineVec; ++v) {
                    // unconditional: skipped entries read row 0 and are ignored below,
                    // so the batch is straight-line code with all its loads in flight
                    // (guarding each load measured 4-8% slower)
                    buf[j][v] = ld_global_nc(reinterpret_cast<const uint4*>(row + (act[v] ? c[v] : 0)));
                }
            }
            // the next item's routing travels while these rows are in flight
            if (k0 == 0) load_routing(item + nwarps, nx_e, nx_s, nx_w);
#pragma unroll
            for (int j = 0; j < kCombineBatch; ++j) {
                if (!ok[j]) continue;
                const float2 w2 = splat2(wk[j]);
#pragma unroll
                for (int v = 0; v < kCombineVec; ++v) {
                    const uint32_t u[4] = {buf[j][v].x, buf[j][v].y, buf[j][v].z, buf[j][v].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)   // acc + w * x, each rounded, never fused
                        acc[4 * v + i] = acc_prod2_rn(acc[4 * v + i], w2, bf16x2_to_f32x2(u[i]), neg_zero);
                }
            }
        }
        uint16_t* yrow = y + (int64_t)t * H;
#pragma unroll
        for (int v = 0; v < kCombineVec; ++v) {
            if (!act[v]) continue;
            const float2* a = acc + 4 * v;
            st_global_cs(reinterpret_cast<uint4*>(yrow + c[v]),
                         make_uint4(pack_bf16x2(a[0]), pack_bf16x2(a[1]), pack_bf16x2(a[2]),
                                    pack_bf16x2(a[3])));
        }
        my_e = nx_e;
        my_s = nx_s;
        my_w = nx_w;
    }
    if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
}

}  // namespace moedc

extern "C" int moedc_combine(const void* expert_out, int E, int cap, int H,
                             const int32_t* topk_idx, const int32_t* slot,
                             const float* topk_weights, int T, int K, void* y,
                             int32_t* dev_status, cudaStream_t stream)
{
    using namespace moedc_host;
    if (T < 0 || H < 8 || H % 8 != 0 || K < 1 || K > MOEDC_MAX_K || E < 1 || E > MOEDC_MAX_E ||
        cap < 1)
        return MOEDC_ERR_ARG;
    if (!expert_out || !dev_status) return MOEDC_ERR_ARG;
    if ((int64_t)E * cap > INT32_MAX) return MOEDC_ERR_ARG;
    if (T > 0 && (!topk_idx || !slot || !topk_weights || !y)) return MOEDC_ERR_ARG;
    if (!aligned(expert_out, 16) || !aligned(y, 16) || !aligned(topk_idx, 4) ||
        !aligned(slot, 4) || !aligned(topk_weights, 4) || !aligned(dev_status, 4))
        return MOEDC_ERR_ARG;
    if (T == 0) return MOEDC_OK;
    const int warps_per_block = moedc::kCombineThreads / moedc::kWarp;
    const int nslice = (H + moedc::kCombineSlice - 1) / moedc::kCombineSlice;
    const int64_t items = (int64_t)T * nslice;
    int64_t blocks = (items + warps_per_block - 1) / warps_per_block;
    const int64_t resident =
        resident_blocks((const void*)moedc::combine_kernel, moedc::kCombineThreads, 0);
    if (blocks > resident) blocks = resident;
    clear_stale_error();
    launch(moedc::combine_kernel, (int)blocks, moedc::kCombineThreads, 0, stream, static_cast<const uint16_t*>(expert_out), E, cap, H, topk_idx, slot, topk_weights, T, K,
        static_cast<uint16_t*>(y), dev_status, -0.0f);
    return launch_status();
}

namespace moedc {

constexpr int kCombine8Batch = 8;

// Combine from e4m3 expert outputs: lane covers 16 consecutive channels
// (one 16-byte load of codes per row, all in one 128-channel scale group).
__global__ void __launch_bounds__(kCombineThreads, 2)
combine_e4m3_kernel(const uint8_t* __restrict__ expert_out, const float* __restrict__ scales,
                    int scale_mode, int E, int cap, int H, const int32_t* __restrict__ topk_idx,
                    const int32_t* __restrict__ slot, const float* __restrict__ topk_weights,
                    int T, int K, uint16_t* __restrict__ y, int32_t* __restrict__ status, float neg_zero)
{
    pdl_enter();
    const int lane = threadIdx.x % kWarp;
    const int G = H / 128;
    const int nslice = (H + 511) / 512;
    const int nwarps = gridDim.x * (blockDim.x / kWarp);
    int gw = blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp;
    int t = gw / nslice, sl = gw - (gw / nslice) * nslice;
    const int dt = nwarps / nslice, dsl = nwarps - dt * nslice;
    bool bad = false;
    for (; t < T;) {
        int my_e = -1, my_s = -1;
        float my_w = 0.0f;
        if (lane < K) {
            my_e = __ldg(topk_idx + (int64_t)t * K + lane);
            my_s = __ldg(slot + (int64_t)t * K + lane);
            my_w = __ldg(topk_weights + (int64_t)t * K + lane);
            if (sl == 0 && (my_e < -1 || my_e >= E)) bad = true;
        }
        const int c0 = sl * 512 + lane * 16;
        const bool act = c0 < H;
        const int g = act ? c0 / 128 : 0;
        float2 acc[8];   // channel pairs
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = make_float2(0.0f, 0.0f);
        for (int k0 = 0; k0 < K; k0 += kCombine8Batch) {
            uint4 q[kCombine8Batch];
            float sc[kCombine8Batch], wk[kCombine8Batch];
            bool ok[kCombine8Batch];
            // unconditional loads (skipped entries read row 0), all in flight together
#pragma unroll
            for (int j = 0; j < kCombine8Batch; ++j) {
                const int k = k0 + j;
                const int e = __shfl_sync(0xffffffffu, my_e, k & 31);
                const int s = __shfl_sync(0xffffffffu, my_s, k & 31);
                wk[j] = __shfl_sync(0xffffffffu, my_w, k & 31);
                ok[j] = k < K && e >= 0 && e < E && s >= 0 && s < cap;
                const int64_t row = ok[j] ? (int64_t)e * cap + s : 0;
                const int64_t si = !ok[j]           ? 0
                                   : scale_mode == 2 ? row                              // per row
                                   : scale_mode == 1 ? ((int64_t)e * G + g) * cap + s   // [E][G][cap]
                                                     : row * G + g;                     // [E][cap][G]
                q[j] = ld_global_nc(reinterpret_cast<const uint4*>(expert_out + row * H +
                                                                     (act ? c0 : 0)));
                sc[j] = __ldg(scales + si);
            }
#pragma unroll
            for (int j = 0; j < kCombine8Batch; ++j) {
                if (!ok[j]) continue;
                const uint32_t u[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
                const float2 w2 = splat2(wk[j]), s2 = splat2(sc[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // acc + w * (q * s), each operation rounded, never fused
                    const float2 lo = mul2_rn(e4m3x2_to_f32x2(u[i] & 0xffffu), s2);
                    const float2 hi = mul2_rn(e4m3x2_to_f32x2(u[i] >> 16), s2);
                    acc[2 * i] = acc_prod2_rn(acc[2 * i], w2, lo, neg_zero);
                    acc[2 * i + 1] = acc_prod2_rn(acc[2 * i + 1], w2, hi, neg_zero);
                }
            }
        }
        if (act) {
            uint16_t* dst = y + (int64_t)t * H + c0;
            st_global_cs(reinterpret_cast<uint4*>(dst),
                         make_uint4(pack_bf16x2(acc[0]), pack_bf16x2(acc[1]), pack_bf16x2(acc[2]),
                                    pack_bf16x2(acc[3])));
            st_global_cs(reinterpret_cast<uint4*>(dst + 8),
                         make_uint4(pack_bf16x2(acc[4]), pack_bf16x2(acc[5]), pack_bf16x2(acc[6]),
                                    pack_bf16x2(acc[7])));
        }
        t += dt;
        sl += dsl;
        if (sl >= nslice) {
            sl -= nslice;
            t += 1;
        }
    }
    if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
}

// K <= 8: a warp owns half of a token's 512-channel slices; the routing of
// its rows (row index, weight, scale base) is derived once and kept in
// registers across those slices.  Each row's shuffles, address arithmetic
// and scale-index work were otherwise redone for every slice; hoisting them
// took the 4096-token workload from 75.8 to 59.4 us, packed binary32
// multiplies to 55.3 us, and 32-bit row indices with three blocks per SM
// (at two, ncu showed 24% of warps active and load waits as the first stall)
// to 53.5-54.0 us.
constexpr int kHalves = 2;   // measured: 1 part 63.5 us, 2 parts 59.4, 3 parts 60.4, 4 parts 68.6
__global__ void __launch_bounds__(kCombineThreads, 3)
combine_e4m3_rows_kernel(const uint8_t* __restrict__ expert_out, const float* __restrict__ scales,
                         int scale_mode, int E, int cap, int H,
                         const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot,
                         const float* __restrict__ topk_weights, int T, int K,
                         uint16_t* __restrict__ y, int32_t* __restrict__ status, float neg_zero)
{
    pdl_enter();
    const int lane = threadIdx.x % kWarp;
    const int G = H / 128;
    const int nslice = (H + 511) / 512;
    const int per_half = (nslice + kHalves - 1) / kHalves;
    const int items = T * kHalves;
    const int nwarps = gridDim.x * (blockDim.x / kWarp);
    bool bad = false;
    for (int item = blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp; item < items;
         item += nwarps) {
        const int t = item / kHalves;
        const int half = item - t * kHalves;
        int my_e = -1, my_s = -1;
        float my_w = 0.0f;
        if (lane < K) {
            my_e = __ldg(topk_idx + (int64_t)t * K + lane);
            my_s = __ldg(slot + (int64_t)t * K + lane);
            my_w = __ldg(topk_weights + (int64_t)t * K + lane);
            if (half == 0 && (my_e < -1 || my_e >= E)) bad = true;
        }
        // 32-bit row indices and scale bases (the host bounds E * cap * H / 128 by
        // INT32_MAX): fewer registers
        int rowi[kCombine8Batch];
        int sbase[kCombine8Batch];
        int sstep;   // scale index step per 128-channel group
        float wk[kCombine8Batch];
        unsigned okm = 0;
#pragma unroll
        for (int j = 0; j < kCombine8Batch; ++j) {
            const int e = __shfl_sync(0xffffffffu, my_e, j);
            const int sidx = __shfl_sync(0xffffffffu, my_s, j);
            wk[j] = __shfl_sync(0xffffffffu, my_w, j);
            const bool ok = j < K && e >= 0 && e < E && sidx >= 0 && sidx < cap;
            okm |= (ok ? 1u : 0u) << j;
            const int row = ok ? e * cap + sidx : 0;
            rowi[j] = row;
            sbase[j] = !ok ? 0 : scale_mode == 2 ? row
                         : scale_mode == 1 ? e * G * cap + sidx : row * G;
        }
        sstep = scale_mode == 2 ? 0 : scale_mode == 1 ? cap : 1;
        const int sl_end = min(nslice, (half + 1) * per_half);
        for (int sl = half * per_half; sl < sl_end; ++sl) {
            const int c0 = sl * 512 + lane * 16;
            const bool act = c0 < H;
            const int g = act ? c0 / 128 : 0;
            uint4 q[kCombine8Batch];
            float sc[kCombine8Batch];
#pragma unroll
            for (int j = 0; j < kCombine8Batch; ++j) {
                q[j] = ld_global_nc(reinterpret_cast<const uint4*>(
                    expert_out + (int64_t)rowi[j] * H + (act ? c0 : 0)));
                sc[j] = __ldg(scales + (((okm >> j) & 1u) ? sbase[j] + g * sstep : 0));
            }
            float2 acc[8];   // channel pairs
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < kCombine8Batch; ++j) {
                if (!((okm >> j) & 1u)) continue;
                const uint32_t u[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
                const float2 w2 = splat2(wk[j]), s2 = splat2(sc[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // acc + w * (q * s), each operation rounded, never fused
                    const float2 lo = mul2_rn(e4m3x2_to_f32x2(u[i] & 0xffffu), s2);
                    const float2 hi = mul2_rn(e4m3x2_to_f32x2(u[i] >> 16), s2);
                    acc[2 * i] = acc_prod2_rn(acc[2 * i], w2, lo, neg_zero);
                    acc[2 * i + 1] = acc_prod2_rn(acc[2 * i + 1], w2, hi, neg_zero);
                }
            }
            if (act) {
                uint16_t* dst = y + (int64_t)t * H + c0;
                st_global_cs(reinterpret_cast<uint4*>(dst),
                             make_uint4(pack_bf16x2(acc[0]), pack_bf16x2(acc[1]),
                                        pack_bf16x2(acc[2]), pack_bf16x2(acc[3])));
                st_global_cs(reinterpret_cast<uint4*>(dst + 8),
                             make_uint4(pack_bf16x2(acc[4]), pack_bf16x2(acc[5]),
                                        pack_bf16x2(acc[6]), pack_bf16x2(acc[7])));
            }
        }
    }
    if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
}

}  // namespace moedc

extern "C" int moedc_combine_e4m3(const void* expert_out, const float* expert_scales,
                                  int scale_layout, int E, int cap, int H,
                                  const int32_t* topk_idx, const int32_t* slot,
                                  const float* topk_weights, int T, int K, void* y,
                                  int32_t* dev_status, cudaStream_t stream)
{
    using namespace moedc_host;
    const int mode = scale_mode(scale_layout);
    if (mode < 0) return MOEDC_ERR_ARG;
    if (T < 0 || H < 128 || H % 128 != 0 || K < 1 || K > MOEDC_MAX_K || E < 1 ||
        E > MOEDC_MAX_E || cap < 1)
        return MOEDC_ERR_ARG;
    if ((int64_t)E * cap * (H / 128) > INT32_MAX || (int64_t)T * (H / 512 + 1) > INT32_MAX / 2)
        return MOEDC_ERR_ARG;
    if (!expert_out || !expert_scales || !dev_status) return MOEDC_ERR_ARG;
    if (T > 0 && (!topk_idx || !slot || !topk_weights || !y)) return MOEDC_ERR_ARG;
    if (!aligned(expert_out, 16) || !aligned(y, 16) || !aligned(expert_scales, 4) ||
        !aligned(topk_idx, 4) || !aligned(slot, 4) || !aligned(topk_weights, 4) ||
        !aligned(dev_status, 4))
        return MOEDC_ERR_ARG;
    if (T == 0) return MOEDC_OK;
    if (K <= moedc::kCombine8Batch) {
        const int64_t items = (int64_t)T * moedc::kHalves;
        int64_t blocks = (items + moedc::kCombineThreads / moedc::kWarp - 1) /
                         (moedc::kCombineThreads / moedc::kWarp);
        const int64_t resident = resident_blocks((const void*)moedc::combine_e4m3_rows_kernel,
                                                 moedc::kCombineThreads, 0);
        if (blocks > resident) blocks = resident;
        clear_stale_error();
        launch(moedc::combine_e4m3_rows_kernel, (int)blocks, moedc::kCombineThreads, 0, stream,
               static_cast<const uint8_t*>(expert_out), expert_scales, mode, E, cap, H, topk_idx,
               slot, topk_weights, T, K, static_cast<uint16_t*>(y), dev_status, -0.0f);
        return launch_status();
    }
    const int64_t items = (int64_t)T * ((H + 511) / 512);
    int64_t blocks = (items + moedc::kCombineThreads / moedc::kWarp - 1) /
                     (moedc::kCombineThreads / moedc::kWarp);
    const int64_t resident =
        resident_blocks((const void*)moedc::combine_e4m3_kernel, moedc::kCombineThreads, 0);
    if (blocks > resident) blocks = resident;
    clear_stale_error();
    launch(moedc::combine_e4m3_kernel, (int)blocks, moedc::kCombineThreads, 0, stream, static_cast<const uint8_t*>(expert_out), expert_scales, mode, E, cap, H,
        topk_idx, slot, topk_weights, T, K, static_cast<uint16_t*>(y), dev_status, -0.0f);
    return launch_status();
}
