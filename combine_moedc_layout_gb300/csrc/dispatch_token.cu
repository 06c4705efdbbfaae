// e4m3 dispatch with one scale per token row.
//
// The scale rule is the per-128-channel one of the dispatch kernel with the
// group widened to the whole row: a = max |x[t][:]| clamped at 1e-4,
// s = a / 448, q = e4m3(x / s).  Sources: DeepEP PR #693 "Pipeline direct
// NVLink dispatch with triple-buffered prefetch", Summary (a token's scale
// factors travel with its hidden data); MORI PR #614 "perf(ep):
// InterNodeV1LL low-token latency on MI300X + CX7" (fp8 and bf16 dispatch
// tuned side by side at the serving shape).
//
// A row's scale needs all of its slices before any code can be written, so a
// thread block owns one token at a time: warp w holds slices w, w + W, ... in
// registers, the warps' maxima meet in shared memory behind one barrier, and
// every warp then quantises and stores its slices from registers.  x is read
// once; nothing is staged through global memory.
#include <climits>

#include "dispatch_item.cuh"

namespace moedc {

constexpr int kTokenMaxWarps = 16;

// |x| maximum of one lane's 16 channels of a slice
__device__ __forceinline__ float slice_amax(const SliceX& v)
{
    const uint32_t w[8] = {v.a.x, v.a.y, v.a.z, v.a.w, v.b.x, v.b.y, v.b.z, v.b.w};
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    return m;
}

// e4m3 codes of one lane's 16 channels (channel order = byte order)
__device__ __forceinline__ uint4 quant_slice(const SliceX& v, float sc)
{
    const uint32_t w[8] = {v.a.x, v.a.y, v.a.z, v.a.w, v.b.x, v.b.y, v.b.z, v.b.w};
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = quant_pair(bf16_lo(w[2 * j]), bf16_hi(w[2 * j]), sc);
        const uint32_t hi = quant_pair(bf16_lo(w[2 * j + 1]), bf16_hi(w[2 * j + 1]), sc);
        p[j] = lo | (hi << 16);
    }
    return make_uint4(p[0], p[1], p[2], p[3]);
}

// kJ: slices held per warp (W = blockDim.x / 32 warps cover kJ * W >= nslice)
template <int kJ>
__global__ void __launch_bounds__(kTokenMaxWarps * kWarp)
dispatch_token_kernel(const uint16_t* __restrict__ x, int T, int H,
                      const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ slot,
                      const int32_t* __restrict__ num_tokens_per_expert, int K, int E, int cap,
                      uint8_t* __restrict__ recv, float* __restrict__ scales,
                      int32_t* __restrict__ src_idx, int32_t* __restrict__ status)
{
    pdl_enter();
    __shared__ float s_amax[2][kTokenMaxWarps];
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int W = blockDim.x / kWarp;
    const int nslice = (H + kSlice - 1) / kSlice;
    bool bad = false;
    int buf = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, buf ^= 1) {
        int my_row = -1;
        if (lane < K) {
            const int e = __ldg(topk_idx + (int64_t)t * K + lane);
            const int s = __ldg(slot + (int64_t)t * K + lane);
            my_row = dest_row(e, s, E, cap);
            if (warp == 0 && (e < -1 || e >= E)) bad = true;
        }
        SliceX v[kJ];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const int sl = warp + j * W;
            v[j] = SliceX{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
            if (sl < nslice) v[j] = load_slice_fp8(x + (int64_t)t * H, H, sl, lane);
            amax = fmaxf(amax, slice_amax(v[j]));
        }
#pragma unroll
        for (int d = kWarp / 2; d > 0; d >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        if (lane == 0) s_amax[buf][warp] = amax;
        // one barrier per token: a warp writes the other buffer next time, and
        // cannot get there before every warp has passed the next barrier,
        // i.e. has finished reading this one
        __syncthreads();
        float a = 0.0f;
        for (int w = 0; w < W; ++w) a = fmaxf(a, s_amax[buf][w]);
        a = fmaxf(a, 1e-4f);
        const float sc = __fdiv_rn(a, 448.0f);
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
            const int sl = warp + j * W;
            if (sl >= nslice) continue;   // uniform across the warp
            const int c0 = sl * kSlice + lane * 16;
            const bool act = c0 < H;
            const uint4 q = quant_slice(v[j], sc);
            for (int k = 0; k < K; ++k) {
                const int row = __shfl_sync(0xffffffffu, my_row, k);
                if (row >= 0 && act)
                    st_global_recv(reinterpret_cast<uint4*>(recv + (int64_t)row * H + c0), q);
            }
        }
        if (warp == 0 && lane < K && my_row >= 0) {
            src_idx[my_row] = t;
            st_global_recv_f32(scales + my_row, sc);
        }
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

int launch_dispatch_token(const void* x, int T, int H, const int32_t* topk_idx,
                          const int32_t* slot, const int32_t* num_tokens_per_expert, int K,
                          int E, int cap, void* recv, float* scales, int32_t* src_idx,
                          int32_t* dev_status, cudaStream_t stream)
{
    if (H > MOEDC_TOKEN_SCALE_MAX_H) return MOEDC_ERR_ARG;
    const int nslice = (H + moedc::kSlice - 1) / moedc::kSlice;
    const int warps = nslice < moedc::kTokenMaxWarps ? nslice : moedc::kTokenMaxWarps;
    const int per_warp = (nslice + warps - 1) / warps;   // 1 .. 4
    const int threads = warps * moedc::kWarp;
    const void* fn = per_warp == 1   ? (const void*)moedc::dispatch_token_kernel<1>
                     : per_warp == 2 ? (const void*)moedc::dispatch_token_kernel<2>
                                     : (const void*)moedc::dispatch_token_kernel<4>;
    const int64_t fill_blocks = ((int64_t)E * cap + threads - 1) / threads;
    int64_t blocks = T > fill_blocks ? T : fill_blocks;
    const int64_t resident = resident_blocks(fn, threads, 0);
    if (blocks > resident) blocks = resident;
    if (blocks < 1) blocks = 1;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    uint8_t* rb = static_cast<uint8_t*>(recv);
    clear_stale_error();
    if (per_warp == 1)
        launch(moedc::dispatch_token_kernel<1>, (int)blocks, threads, 0, stream, xb, T, H,
               topk_idx, slot, num_tokens_per_expert, K, E, cap, rb, scales, src_idx, dev_status);
    else if (per_warp == 2)
        launch(moedc::dispatch_token_kernel<2>, (int)blocks, threads, 0, stream, xb, T, H,
               topk_idx, slot, num_tokens_per_expert, K, E, cap, rb, scales, src_idx, dev_status);
    else
        launch(moedc::dispatch_token_kernel<4>, (int)blocks, threads, 0, stream, xb, T, H,
               topk_idx, slot, num_tokens_per_expert, K, E, cap, rb, scales, src_idx, dev_status);
    return launch_status();
}

}  // namespace moedc_host
