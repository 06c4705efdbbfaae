// Combine: weighted gather-reduce of each token's K expert rows back into
// token order, binary32 accumulation in ascending k, bf16 output.
//
// Sources: MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on MI300X
// + CX7" — CombineSync note (split by (token, hidden slice), not by token, so
// a handful of tokens still spreads over the whole grid) and the zero-copy
// combine input note (the caller's expert outputs are read in place, never
// staged).  The kernel is an HBM read stream: K gathered rows per token.
#include "common.cuh"

namespace moedc {

constexpr int kCombineThreads = 256;
constexpr int kCombineSlice = 512;   // channels per warp item
constexpr int kCombineBatch = 8;     // gathered rows in flight per lane

__global__ void __launch_bounds__(kCombineThreads)
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

    for (int64_t item = (int64_t)blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp;
         item < items; item += nwarps) {
        const int t = (int)(item / nslice);
        const int sl = (int)(item - (int64_t)t * nslice);
        int my_e = -1, my_s = -1;
        float my_w = 0.0f;
        if (lane < K) {
            my_e = topk_idx[(int64_t)t * K + lane];
            my_s = slot[(int64_t)t * K + lane];
            my_w = topk_weights[(int64_t)t * K + lane];
            if (sl == 0 && (my_e < -1 || my_e >= E)) bad = true;
        }
        // lane covers channels c0 .. c0+8 and c1 .. c1+8 (each warp access is 512 B)
        const int c0 = sl * kCombineSlice + lane * 8;
        const int c1 = c0 + 256;
        const bool a0 = c0 < H, a1 = c1 < H;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;

        for (int k0 = 0; k0 < K; k0 += kCombineBatch) {
            uint4 v0[kCombineBatch], v1[kCombineBatch];
            float wk[kCombineBatch];
            bool ok[kCombineBatch];
#pragma unroll
            for (int j = 0; j < kCombineBatch; ++j) {
                const int k = k0 + j;
                const int e = __shfl_sync(0xffffffffu, my_e, k & 31);
                const int s = __shfl_sync(0xffffffffu, my_s, k & 31);
                wk[j] = __shfl_sync(0xffffffffu, my_w, k & 31);
                ok[j] = k < K && e >= 0 && e < E && s >= 0 && s < cap;
                v0[j] = make_uint4(0, 0, 0, 0);
                v1[j] = make_uint4(0, 0, 0, 0);
                if (ok[j]) {
                    const uint16_t* row = expert_out + ((int64_t)e * cap + s) * H;
                    if (a0) v0[j] = ld_global_nc(reinterpret_cast<const uint4*>(row + c0));
                    if (a1) v1[j] = ld_global_nc(reinterpret_cast<const uint4*>(row + c1));
                }
            }
#pragma unroll
            for (int j = 0; j < kCombineBatch; ++j) {
                if (!ok[j]) continue;
                const uint32_t u[8] = {v0[j].x, v0[j].y, v0[j].z, v0[j].w,
                                       v1[j].x, v1[j].y, v1[j].z, v1[j].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(wk[j], bf16_lo(u[i])));
                    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(wk[j], bf16_hi(u[i])));
                }
            }
        }
        uint16_t* yrow = y + (int64_t)t * H;
        if (a0)
            st_global_cs(reinterpret_cast<uint4*>(yrow + c0),
                         make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                    pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
        if (a1)
            st_global_cs(reinterpret_cast<uint4*>(yrow + c1),
                         make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                                    pack_bf16x2(acc[12], acc[13]),
                                    pack_bf16x2(acc[14], acc[15])));
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
    if (T > 0 && (!topk_idx || !slot || !topk_weights || !y)) return MOEDC_ERR_ARG;
    if (!aligned(expert_out, 16) || !aligned(y, 16) || !aligned(topk_idx, 4) ||
        !aligned(slot, 4) || !aligned(topk_weights, 4) || !aligned(dev_status, 4))
        return MOEDC_ERR_ARG;
    if (T == 0) return MOEDC_OK;
    const int warps_per_block = moedc::kCombineThreads / moedc::kWarp;
    const int nslice = (H + moedc::kCombineSlice - 1) / moedc::kCombineSlice;
    const int64_t items = (int64_t)T * nslice;
    int64_t blocks = (items + warps_per_block - 1) / warps_per_block;
    const int64_t max_blocks = (int64_t)sm_count() * 8;
    if (blocks > max_blocks) blocks = max_blocks;
    moedc::combine_kernel<<<(int)blocks, moedc::kCombineThreads, 0, stream>>>(
        static_cast<const uint16_t*>(expert_out), E, cap, H, topk_idx, slot, topk_weights, T, K,
        static_cast<uint16_t*>(y), dev_status);
    return launch_status();
}
