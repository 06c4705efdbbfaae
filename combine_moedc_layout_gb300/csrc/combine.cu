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
               uint16_t* __restrict__ y, int32_t* __restrict__ status)
{
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
        float acc[8 * kCombineVec];
#pragma unroll
        for (int i = 0; i < 8 * kCombineVec; ++i) acc[i] = 0.0f;
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
#pragma unroll
                for (int v = 0; v < kCombineVec; ++v) {
                    const uint32_t u[4] = {buf[j][v].x, buf[j][v].y, buf[j][v].z, buf[j][v].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float* a = acc + 8 * v + 2 * i;
                        a[0] = __fadd_rn(a[0], __fmul_rn(wk[j], bf16_lo(u[i])));
                        a[1] = __fadd_rn(a[1], __fmul_rn(wk[j], bf16_hi(u[i])));
                    }
                }
            }
        }
        uint16_t* yrow = y + (int64_t)t * H;
#pragma unroll
        for (int v = 0; v < kCombineVec; ++v) {
            if (!act[v]) continue;
            const float* a = acc + 8 * v;
            st_global_cs(reinterpret_cast<uint4*>(yrow + c[v]),
                         make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                    pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7])));
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
    moedc::combine_kernel<<<(int)blocks, moedc::kCombineThreads, 0, stream>>>(
        static_cast<const uint16_t*>(expert_out), E, cap, H, topk_idx, slot, topk_weights, T, K,
        static_cast<uint16_t*>(y), dev_status);
    return launch_status();
}
