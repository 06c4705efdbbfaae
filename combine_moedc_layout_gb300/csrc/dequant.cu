// e4m3 receive rows back to bf16: out = bf16(decode(q) * scale), with the
// scale of the element's 128-channel group or of its whole row.  This is the identity "expert" of a dispatch -> expert ->
// combine round (the dequantisation q * s that pairs with the e4m3 dispatch),
// and the bf16 view an expert without an FP8 path would read.  Only the
// filled rows (s < min(count, cap)) are converted.
#include <climits>

#include "common.cuh"

namespace moedc {

constexpr int kDequantThreads = 256;
constexpr int kDequantSlice = 512;   // channels per warp item (16 per lane)

// Work items are (filled row, 512-channel slice) pairs only: each block first
// turns min(count[e], cap) into an exclusive prefix over experts in shared
// memory, then a flat filled-row index f maps to its expert by binary search.
__global__ void __launch_bounds__(kDequantThreads)
dequant_e4m3_kernel(const uint8_t* __restrict__ recv, const float* __restrict__ scales,
                    int scale_mode, const int32_t* __restrict__ num_tokens_per_expert, int E,
                    int cap, int H, uint16_t* __restrict__ out)
{
    pdl_enter();
    __shared__ int s_pref[MOEDC_MAX_E + 1];
    __shared__ int s_part[kDequantThreads / kWarp];
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    // exclusive prefix of the filled rows per expert (E <= 1024 = 4 per thread)
    constexpr int kPer = (MOEDC_MAX_E + kDequantThreads - 1) / kDequantThreads;
    int v[kPer];
    int mine = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = threadIdx.x * kPer + j;
        v[j] = e < E ? min(__ldg(num_tokens_per_expert + e), cap) : 0;
        v[j] = max(v[j], 0);
        mine += v[j];
    }
    int incl = mine;
#pragma unroll
    for (int d = 1; d < kWarp; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == kWarp - 1) s_part[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_part[w];
    int run = before + incl - mine;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = threadIdx.x * kPer + j;
        if (e <= E) s_pref[e] = run;
        run += v[j];
    }
    if (threadIdx.x == 0) {   // the total (index E may lie past every thread's range)
        int tot = 0;
        for (int w = 0; w < kDequantThreads / kWarp; ++w) tot += s_part[w];
        s_pref[E] = tot;
    }
    __syncthreads();
    const int filled = s_pref[E];

    const int nslice = (H + kDequantSlice - 1) / kDequantSlice;
    const int G = H / 128;
    const int items = filled * nslice;
    const int nwarps = gridDim.x * (blockDim.x / kWarp);
    for (int item = blockIdx.x * (blockDim.x / kWarp) + warp; item < items; item += nwarps) {
        const int f = item / nslice;
        const int sl = item - f * nslice;
        int lo = 0, hi = E - 1;          // last expert whose prefix is <= f
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pref[mid] <= f) lo = mid; else hi = mid - 1;
        }
        const int sidx = f - s_pref[lo];
        const int64_t row = (int64_t)lo * cap + sidx;
        const int c0 = sl * kDequantSlice + lane * 16;
        if (c0 >= H) continue;
        const uint4 q = ld_global_nc(reinterpret_cast<const uint4*>(recv + row * H + c0));
        const int g = c0 / 128;
        const int64_t si = scale_mode == 2   ? row                                   // per row
                           : scale_mode == 1 ? ((int64_t)lo * G + g) * cap + sidx    // [E][G][cap]
                                             : row * G + g;                          // [E][cap][G]
        const float2 s2 = splat2(__ldg(scales + si));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // RN(q * s), then the bf16 nearest-even rounding
            o[2 * i] = pack_bf16x2(mul2_rn(e4m3x2_to_f32x2(w[i] & 0xffffu), s2));
            o[2 * i + 1] = pack_bf16x2(mul2_rn(e4m3x2_to_f32x2(w[i] >> 16), s2));
        }
        uint16_t* dst = out + row * H + c0;
        st_global_cs(reinterpret_cast<uint4*>(dst), make_uint4(o[0], o[1], o[2], o[3]));
        st_global_cs(reinterpret_cast<uint4*>(dst + 8), make_uint4(o[4], o[5], o[6], o[7]));
    }
}

}  // namespace moedc

extern "C" int moedc_dequant_e4m3(const void* recv, const float* scales, int scale_layout,
                                  const int32_t* num_tokens_per_expert, int E, int cap, int H,
                                  void* out_bf16, cudaStream_t stream)
{
    using namespace moedc_host;
    const int mode = scale_mode(scale_layout);
    if (mode < 0) return MOEDC_ERR_ARG;
    if (E < 1 || E > MOEDC_MAX_E || cap < 1 || H < 128 || H % 128 != 0) return MOEDC_ERR_ARG;
    if ((int64_t)E * cap * ((H + 511) / 512) > INT32_MAX) return MOEDC_ERR_ARG;
    if (!recv || !scales || !num_tokens_per_expert || !out_bf16) return MOEDC_ERR_ARG;
    if (!aligned(recv, 16) || !aligned(out_bf16, 16) || !aligned(scales, 4) ||
        !aligned(num_tokens_per_expert, 4))
        return MOEDC_ERR_ARG;
    // the filled-row count lives on the device: size the grid for the largest case
    const int64_t items = (int64_t)E * cap * ((H + moedc::kDequantSlice - 1) / moedc::kDequantSlice);
    int64_t blocks = (items + moedc::kDequantThreads / moedc::kWarp - 1) /
                     (moedc::kDequantThreads / moedc::kWarp);
    const int64_t resident =
        resident_blocks((const void*)moedc::dequant_e4m3_kernel, moedc::kDequantThreads, 0);
    if (blocks > resident) blocks = resident;
    clear_stale_error();
    launch(moedc::dequant_e4m3_kernel, (int)blocks, moedc::kDequantThreads, 0, stream, static_cast<const uint8_t*>(recv), scales, mode, num_tokens_per_expert, E,
        cap, H, static_cast<uint16_t*>(out_bf16));
    return launch_status();
}
