// One dispatch work item: a 512-channel slice of one token row, copied (bf16)
// or quantised once and then stored to each of the token's K expert slots.
//
// The work is split by (token, hidden slice) rather than by token, following
// MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on MI300X + CX7"
// (DispatchIntraNode flat stride and CombineSync split notes; MultiWarpIter's
// measured floor of 512 elements per warp).  A token's K copies are identical,
// so the FP8 scale and codes of a slice are computed once and written K times.
#pragma once

#include "common.cuh"

namespace moedc {

constexpr int kSlice = 512;   // channels per warp item

// e4m3 codes (low byte = first) of RN(a / s) and RN(b / s): one correctly
// rounded binary32 division per element, then the satfinite nearest-even
// encode.  (Multiplying by a rounded reciprocal instead was measured to save
// no time here, so the division is kept as the definition states it.)
__device__ __forceinline__ uint32_t quant_pair(float a, float b, float s)
{
    return pack_e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
}

// Lane k < K of a warp holds entry k of the token (expert id and slot); the
// store loops broadcast them by k.
__device__ __forceinline__ bool dest_ok(int e, int s, int E, int cap)
{
    return e >= 0 && e < E && s >= 0 && s < cap;
}

// The x data one lane needs for a work item (two 16-byte vectors).
struct SliceX {
    uint4 a, b;
};

// bf16: lane covers channels {slice*512 + j*256 + lane*8 .. +8}, j = 0, 1, so
// each 16-byte access of the warp covers 512 contiguous bytes.
__device__ __forceinline__ SliceX load_slice_bf16(const uint16_t* __restrict__ xrow, int H,
                                                  int slice, int lane)
{
    const int c0 = slice * kSlice + lane * 8;
    const int c1 = c0 + 256;
    SliceX v{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (c0 < H) v.a = ld_global_nc(reinterpret_cast<const uint4*>(xrow + c0));
    if (c1 < H) v.b = ld_global_nc(reinterpret_cast<const uint4*>(xrow + c1));
    return v;
}

__device__ __forceinline__ void store_slice_bf16(const SliceX& v, int H, int slice, int lane,
                                                 int K, int my_row, uint16_t* __restrict__ recv)
{
    const int c0 = slice * kSlice + lane * 8;
    const int c1 = c0 + 256;
    const bool a0 = c0 < H, a1 = c1 < H;
    for (int k = 0; k < K; ++k) {
        const int row = __shfl_sync(0xffffffffu, my_row, k);
        if (row < 0) continue;
        uint16_t* dst = recv + (int64_t)row * H;
        if (a0) st_global_recv(reinterpret_cast<uint4*>(dst + c0), v.a);
        if (a1) st_global_recv(reinterpret_cast<uint4*>(dst + c1), v.b);
    }
}

// e4m3: lane covers 16 consecutive channels slice*512 + lane*16 .. +16, so
// each 128-channel scale group is held by 8 adjacent lanes and one 16-byte
// store per lane writes the lane's codes.
__device__ __forceinline__ SliceX load_slice_fp8(const uint16_t* __restrict__ xrow, int H,
                                                 int slice, int lane)
{
    const int c0 = slice * kSlice + lane * 16;
    SliceX v{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (c0 < H) {   // H % 128 == 0: a scale group is all in or all out
        v.a = ld_global_nc(reinterpret_cast<const uint4*>(xrow + c0));
        v.b = ld_global_nc(reinterpret_cast<const uint4*>(xrow + c0 + 8));
    }
    return v;
}

// kScaleCols: scales stored [E][G][cap] (group-major per expert) instead of
// [E][cap][G]; lane k then also holds my_sbase = e * G * cap + s for entry k.
// The lane's 16 codes and its group's scale: amax over the 8 lanes of the
// group (three xor shuffles), clamped, one division for the scale and one per
// element for the codes.
struct SliceQ {
    uint4 q;
    float sc;
};

__device__ __forceinline__ SliceQ quant_slice_fp8(const SliceX& v)
{
    const uint32_t w[8] = {v.a.x, v.a.y, v.a.z, v.a.w, v.b.x, v.b.y, v.b.z, v.b.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = bf16_lo(w[i]);
        f[2 * i + 1] = bf16_hi(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    // the 8 lanes of a group are aligned, so xor 1, 2, 4 stays inside it
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    amax = fmaxf(amax, 1e-4f);
    const float sc = __fdiv_rn(amax, 448.0f);
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = quant_pair(f[4 * j + 0], f[4 * j + 1], sc);
        const uint32_t hi = quant_pair(f[4 * j + 2], f[4 * j + 3], sc);
        p[j] = lo | (hi << 16);
    }
    return SliceQ{make_uint4(p[0], p[1], p[2], p[3]), sc};
}

template <bool kScaleCols>
__device__ __forceinline__ void store_slice_fp8(const SliceX& v, int H, int slice, int lane,
                                                int K, int my_row, int64_t my_sbase, int cap,
                                                uint8_t* __restrict__ recv,
                                                float* __restrict__ scales)
{
    const int G = H / 128;
    const int c0 = slice * kSlice + lane * 16;
    const bool act = c0 < H;
    const SliceQ sq = quant_slice_fp8(v);
    const uint4 q = sq.q;
    const float sc = sq.sc;
    const bool leader = (lane & 7) == 0;
    const int g = c0 / 128;
    for (int k = 0; k < K; ++k) {
        const int row = __shfl_sync(0xffffffffu, my_row, k);
        int64_t sbase = 0;
        if (kScaleCols) sbase = __shfl_sync(0xffffffffu, my_sbase, k);
        if (row < 0 || !act) continue;
        st_global_recv(reinterpret_cast<uint4*>(recv + (int64_t)row * H + c0), q);
        if (leader) {
            const int64_t si = kScaleCols ? sbase + (int64_t)g * cap : (int64_t)row * G + g;
            st_global_recv_f32(scales + si, sc);
        }
    }
}

template <bool kFp8>
__device__ __forceinline__ SliceX load_slice(const uint16_t* xrow, int H, int slice, int lane)
{
    return kFp8 ? load_slice_fp8(xrow, H, slice, lane) : load_slice_bf16(xrow, H, slice, lane);
}

template <bool kFp8, bool kScaleCols = false>
__device__ __forceinline__ void store_slice(const SliceX& v, int H, int slice, int lane, int K,
                                            int my_row, void* recv, float* scales,
                                            int64_t my_sbase = 0, int cap = 0)
{
    if (kFp8)
        store_slice_fp8<kScaleCols>(v, H, slice, lane, K, my_row, my_sbase, cap,
                                    static_cast<uint8_t*>(recv), scales);
    else
        store_slice_bf16(v, H, slice, lane, K, my_row, static_cast<uint16_t*>(recv));
}

// e * G * cap + s: where entry (e, s)'s group-0 scale sits in [E][G][cap] scales
__device__ __forceinline__ int64_t colmajor_scale_base(int row, int cap, int G)
{
    if (row < 0) return 0;
    const int e = row / cap;
    const int s = row - e * cap;
    return (int64_t)e * G * cap + s;
}

// Destination row index e * cap + s of a routing entry, or -1 when the entry
// is masked, out of range or dropped (the host checks E * cap fits in int).
__device__ __forceinline__ int dest_row(int e, int s, int E, int cap)
{
    return dest_ok(e, s, E, cap) ? e * cap + s : -1;
}

// Cursor over the flat (token, slice) item space of a grid-strided warp,
// advanced by a fixed stride without dividing.
struct ItemCursor {
    int t, sl;
    __device__ __forceinline__ void init(int item, int nslice)
    {
        t = item / nslice;
        sl = item - t * nslice;
    }
    __device__ __forceinline__ void advance(int dt, int dsl, int nslice)
    {
        t += dt;
        sl += dsl;
        if (sl >= nslice) {
            sl -= nslice;
            t += 1;
        }
    }
};

}  // namespace moedc
