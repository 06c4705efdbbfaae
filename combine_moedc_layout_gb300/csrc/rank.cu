// Rank-major packed receive: a token is copied once to each rank that hosts
// any of its experts, into that rank's contiguous buffer, instead of once per
// expert (UCCL PR #749 "[EP] Low-latency mode batch tokens per destination":
// tokens are batched per destination rank).  When several of a token's K
// experts share a rank this writes fewer rows than expert-major dispatch.
//
//   moedc_rank_layout    rank_slot[t][r]: position of token t in rank r's
//                        buffer (ascending t), from is_token_in_rank.
//   moedc_rank_dispatch  recv_rank[r][j] = x[t] (bf16 copy, or e4m3 codes with
//                        per-128 scales by the expert-dispatch rule).
//   moedc_rank_combine   y[t] = sum over ranks (ascending r) of the partial
//                        row each rank returns for the token.
#include <climits>

#include "dispatch_item.cuh"

namespace moedc {

constexpr int kRankLayoutThreads = 1024;
constexpr int kRankLayoutWarps = kRankLayoutThreads / kWarp;
constexpr int kRankV = 8;    // consecutive tokens per thread per round

// Block r owns rank r: an exclusive scan of column r of is_token_in_rank.
__global__ void __launch_bounds__(kRankLayoutThreads)
rank_layout_kernel(const uint8_t* __restrict__ is_token_in_rank, int T, int R, int cap_rank,
                   int32_t* __restrict__ rank_slot, int32_t* __restrict__ status)
{
    pdl_enter();
    __shared__ int s_warp[kRankLayoutWarps];
    __shared__ int s_total;
    const int r = blockIdx.x;
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    int running = 0;
    for (int base = 0; base < T; base += kRankLayoutThreads * kRankV) {
        const int t0 = base + threadIdx.x * kRankV;
        unsigned m = 0;
#pragma unroll
        for (int j = 0; j < kRankV; ++j)
            if (t0 + j < T && __ldg(is_token_in_rank + (int64_t)(t0 + j) * R + r)) m |= 1u << j;
        const int c = __popc(m);
        int incl = c;
#pragma unroll
        for (int d = 1; d < kWarp; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        if (lane == kWarp - 1) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int wv = s_warp[lane];
            int wi = wv;
#pragma unroll
            for (int d = 1; d < kWarp; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, wi, d);
                if (lane >= d) wi += y;
            }
            s_warp[lane] = wi - wv;
            if (lane == kWarp - 1) s_total = wi;
        }
        __syncthreads();
        int s = running + s_warp[warp] + incl - c;
#pragma unroll
        for (int j = 0; j < kRankV; ++j) {
            if (t0 + j >= T) break;
            const bool in = (m >> j) & 1u;
            rank_slot[(int64_t)(t0 + j) * R + r] = in ? s : -1;
            s += in ? 1 : 0;
        }
        running += s_total;
        __syncthreads();
    }
    if (threadIdx.x == 0 && running > cap_rank) raise_status(status, MOEDC_ERR_CAPACITY);
}

constexpr int kRankThreads = 256;

// Warp item (token, 512-channel slice); lane i holds the destination row of
// rank r0 + i for the ranks taken 32 at a time.
template <bool kFp8>
__global__ void __launch_bounds__(kRankThreads, 4)
rank_dispatch_kernel(const uint16_t* __restrict__ x, int T, int H,
                     const int32_t* __restrict__ rank_slot,
                     const int32_t* __restrict__ num_tokens_per_rank, int R, int cap_rank,
                     void* __restrict__ recv_rank, float* __restrict__ scales_rank,
                     int32_t* __restrict__ rank_src_idx)
{
    pdl_enter();
    const int lane = threadIdx.x % kWarp;
    const int nslice = (H + kSlice - 1) / kSlice;
    const int nwarps = gridDim.x * (blockDim.x / kWarp);
    const int dt = nwarps / nslice, dsl = nwarps - dt * nslice;
    ItemCursor cur;
    cur.init(blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp, nslice);
    for (; cur.t < T; cur.advance(dt, dsl, nslice)) {
        const SliceX v = load_slice<kFp8>(x + (int64_t)cur.t * H, H, cur.sl, lane);
        for (int r0 = 0; r0 < R; r0 += kWarp) {
            int row = -1;
            if (r0 + lane < R) {
                const int j = __ldg(rank_slot + (int64_t)cur.t * R + r0 + lane);
                if (j >= 0 && j < cap_rank) row = (r0 + lane) * cap_rank + j;
            }
            if (cur.sl == 0 && row >= 0) rank_src_idx[row] = cur.t;
            store_slice<kFp8>(v, H, cur.sl, lane, min(kWarp, R - r0), row, recv_rank,
                              scales_rank);
        }
    }
    // slots no token reaches carry rank_src_idx = -1
    const int64_t total = (int64_t)R * cap_rank;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += nthreads) {
        const int r = (int)(i / cap_rank);
        const int j = (int)(i - (int64_t)r * cap_rank);
        if (j >= __ldg(num_tokens_per_rank + r)) rank_src_idx[i] = -1;
    }
}

constexpr int kRankCombineBatch = 8;

// Warp item (token, 512-channel slice): each lane adds its 16 channels of the
// token's partial row from every rank, ascending r, in binary32.
__global__ void __launch_bounds__(kRankThreads, 2)
rank_combine_kernel(const uint16_t* __restrict__ rank_out, int R, int cap_rank, int H,
                    const int32_t* __restrict__ rank_slot, int T, uint16_t* __restrict__ y)
{
    pdl_enter();
    const int lane = threadIdx.x % kWarp;
    const int nslice = (H + 511) / 512;
    const int nwarps = gridDim.x * (blockDim.x / kWarp);
    const int dt = nwarps / nslice, dsl = nwarps - dt * nslice;
    ItemCursor cur;
    cur.init(blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp, nslice);
    for (; cur.t < T; cur.advance(dt, dsl, nslice)) {
        const int c0 = cur.sl * 512 + lane * 8;
        const int c1 = c0 + 256;
        const bool a0 = c0 < H, a1 = c1 < H;
        float2 acc[8];   // channel pairs
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = make_float2(0.0f, 0.0f);
        for (int r0 = 0; r0 < R; r0 += kWarp) {
            int my_row = -1;
            if (r0 + lane < R) {
                const int j = __ldg(rank_slot + (int64_t)cur.t * R + r0 + lane);
                if (j >= 0 && j < cap_rank) my_row = (r0 + lane) * cap_rank + j;
            }
            const int nr = min(kWarp, R - r0);
            for (int k0 = 0; k0 < nr; k0 += kRankCombineBatch) {
                uint4 b0[kRankCombineBatch], b1[kRankCombineBatch];
                bool ok[kRankCombineBatch];
                // every load is issued unconditionally (absent ranks read row 0 and
                // are skipped below), so the batch stays straight-line code and
                // all of its loads are in flight together
#pragma unroll
                for (int q = 0; q < kRankCombineBatch; ++q) {
                    const int k = k0 + q;
                    const int row = __shfl_sync(0xffffffffu, my_row, k & 31);
                    ok[q] = k < nr && row >= 0;
                    const uint16_t* src = rank_out + (int64_t)(ok[q] ? row : 0) * H;
                    b0[q] = ld_global_nc(reinterpret_cast<const uint4*>(src + (a0 ? c0 : 0)));
                    b1[q] = ld_global_nc(reinterpret_cast<const uint4*>(src + (a1 ? c1 : 0)));
                }
#pragma unroll
                for (int q = 0; q < kRankCombineBatch; ++q) {
                    if (!ok[q]) continue;
                    const uint32_t u[8] = {b0[q].x, b0[q].y, b0[q].z, b0[q].w,
                                           b1[q].x, b1[q].y, b1[q].z, b1[q].w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (i >= 4 && !a1) break;
                        acc[i] = add2_rn_unfed(acc[i], bf16x2_to_f32x2(u[i]));
                    }
                }
            }
        }
        uint16_t* yrow = y + (int64_t)cur.t * H;
        if (a0)
            st_global_cs(reinterpret_cast<uint4*>(yrow + c0),
                         make_uint4(pack_bf16x2(acc[0]), pack_bf16x2(acc[1]), pack_bf16x2(acc[2]),
                                    pack_bf16x2(acc[3])));
        if (a1)
            st_global_cs(reinterpret_cast<uint4*>(yrow + c1),
                         make_uint4(pack_bf16x2(acc[4]), pack_bf16x2(acc[5]), pack_bf16x2(acc[6]),
                                    pack_bf16x2(acc[7])));
    }
}

}  // namespace moedc

extern "C" int moedc_rank_layout(const uint8_t* is_token_in_rank, int T, int R, int cap_rank,
                                 int32_t* rank_slot, int32_t* dev_status, cudaStream_t stream)
{
    using namespace moedc_host;
    if (T < 0 || R < 1 || R > MOEDC_MAX_E || cap_rank < 1) return MOEDC_ERR_ARG;
    if ((int64_t)T * R > INT32_MAX) return MOEDC_ERR_ARG;
    if (!dev_status || (T > 0 && (!is_token_in_rank || !rank_slot))) return MOEDC_ERR_ARG;
    if (!aligned(rank_slot, 4) || !aligned(dev_status, 4)) return MOEDC_ERR_ARG;
    if (T == 0) return MOEDC_OK;
    clear_stale_error();
    launch(moedc::rank_layout_kernel, R, moedc::kRankLayoutThreads, 0, stream, is_token_in_rank, T, R, cap_rank, rank_slot, dev_status);
    return launch_status();
}

extern "C" int moedc_rank_dispatch(const void* x, int T, int H, const int32_t* rank_slot,
                                   const int32_t* num_tokens_per_rank, int R, int cap_rank,
                                   int out_dtype, void* recv_rank, float* scales_rank,
                                   int32_t* rank_src_idx, cudaStream_t stream)
{
    using namespace moedc_host;
    if (T < 0 || H < 8 || R < 1 || R > MOEDC_MAX_E || cap_rank < 1) return MOEDC_ERR_ARG;
    if (out_dtype != MOEDC_BF16 && out_dtype != MOEDC_FP8_E4M3) return MOEDC_ERR_ARG;
    if (out_dtype == MOEDC_BF16 && H % 8 != 0) return MOEDC_ERR_ARG;
    if (out_dtype == MOEDC_FP8_E4M3 && (H % 128 != 0 || !scales_rank)) return MOEDC_ERR_ARG;
    if ((int64_t)R * cap_rank > INT32_MAX || (int64_t)T * ((H + 511) / 512) > INT32_MAX / 2)
        return MOEDC_ERR_ARG;
    if (!num_tokens_per_rank || !recv_rank || !rank_src_idx) return MOEDC_ERR_ARG;
    if (T > 0 && (!x || !rank_slot)) return MOEDC_ERR_ARG;
    if (!aligned(x, 16) || !aligned(recv_rank, 16) || !aligned(scales_rank, 4) ||
        !aligned(rank_slot, 4) || !aligned(num_tokens_per_rank, 4) || !aligned(rank_src_idx, 4))
        return MOEDC_ERR_ARG;
    const int nslice = (H + moedc::kSlice - 1) / moedc::kSlice;
    const int64_t items = (int64_t)T * nslice;
    int64_t blocks = (items + moedc::kRankThreads / moedc::kWarp - 1) /
                     (moedc::kRankThreads / moedc::kWarp);
    const int64_t fill_blocks = ((int64_t)R * cap_rank + moedc::kRankThreads - 1) /
                                moedc::kRankThreads;
    if (blocks < fill_blocks) blocks = fill_blocks;
    const void* fn = out_dtype == MOEDC_FP8_E4M3 ? (const void*)moedc::rank_dispatch_kernel<true>
                                                 : (const void*)moedc::rank_dispatch_kernel<false>;
    const int64_t resident = resident_blocks(fn, moedc::kRankThreads, 0);
    if (blocks > resident) blocks = resident;
    if (blocks < 1) blocks = 1;
    const uint16_t* xb = static_cast<const uint16_t*>(x);
    clear_stale_error();
    if (out_dtype == MOEDC_FP8_E4M3)
        launch(moedc::rank_dispatch_kernel<true>, (int)blocks, moedc::kRankThreads, 0, stream, xb, T, H, rank_slot, num_tokens_per_rank, R, cap_rank, recv_rank, scales_rank,
            rank_src_idx);
    else
        launch(moedc::rank_dispatch_kernel<false>, (int)blocks, moedc::kRankThreads, 0, stream, xb, T, H, rank_slot, num_tokens_per_rank, R, cap_rank, recv_rank, scales_rank,
            rank_src_idx);
    return launch_status();
}

extern "C" int moedc_rank_combine(const void* rank_out, int R, int cap_rank, int H,
                                  const int32_t* rank_slot, int T, void* y, cudaStream_t stream)
{
    using namespace moedc_host;
    if (T < 0 || H < 8 || H % 8 != 0 || R < 1 || R > MOEDC_MAX_E || cap_rank < 1)
        return MOEDC_ERR_ARG;
    if ((int64_t)R * cap_rank > INT32_MAX || (int64_t)T * ((H + 511) / 512) > INT32_MAX / 2)
        return MOEDC_ERR_ARG;
    if (!rank_out || (T > 0 && (!rank_slot || !y))) return MOEDC_ERR_ARG;
    if (!aligned(rank_out, 16) || !aligned(y, 16) || !aligned(rank_slot, 4)) return MOEDC_ERR_ARG;
    if (T == 0) return MOEDC_OK;
    const int64_t items = (int64_t)T * ((H + 511) / 512);
    int64_t blocks = (items + moedc::kRankThreads / moedc::kWarp - 1) /
                     (moedc::kRankThreads / moedc::kWarp);
    const int64_t resident =
        resident_blocks((const void*)moedc::rank_combine_kernel, moedc::kRankThreads, 0);
    if (blocks > resident) blocks = resident;
    clear_stale_error();
    launch(moedc::rank_combine_kernel, (int)blocks, moedc::kRankThreads, 0, stream, static_cast<const uint16_t*>(rank_out), R, cap_rank, H, rank_slot, T,
        static_cast<uint16_t*>(y));
    return launch_status();
}
