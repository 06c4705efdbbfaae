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

// Lane `lane` of a warp holds entry k == lane of the token (k < K): its expert
// id and slot.  Broadcast helpers read them back by k.
struct Dest {
    int e;
    int s;
};

__device__ __forceinline__ bool dest_ok(int e, int s, int E, int cap)
{
    return e >= 0 && e < E && s >= 0 && s < cap;
}

// bf16: lane covers channels {slice*512 + j*256 + lane*8 .. +8}, j = 0, 1, so
// each 16-byte access of the warp covers 512 contiguous bytes.
__device__ __forceinline__ void dispatch_slice_bf16(const uint16_t* __restrict__ xrow, int H,
                                                    int slice, int lane, int K, int my_e,
                                                    int my_s, int E, int cap,
                                                    uint16_t* __restrict__ recv)
{
    const int c0 = slice * kSlice + lane * 8;
    const int c1 = c0 + 256;
    const bool a0 = c0 < H, a1 = c1 < H;
    uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
    if (a0) v0 = ld_global_nc(reinterpret_cast<const uint4*>(xrow + c0));
    if (a1) v1 = ld_global_nc(reinterpret_cast<const uint4*>(xrow + c1));
    for (int k = 0; k < K; ++k) {
        const int e = __shfl_sync(0xffffffffu, my_e, k);
        const int s = __shfl_sync(0xffffffffu, my_s, k);
        if (!dest_ok(e, s, E, cap)) continue;
        uint16_t* row = recv + ((int64_t)e * cap + s) * H;
        if (a0) st_global_cs(reinterpret_cast<uint4*>(row + c0), v0);
        if (a1) st_global_cs(reinterpret_cast<uint4*>(row + c1), v1);
    }
}

// e4m3: lane covers 16 consecutive channels slice*512 + lane*16 .. +16, so
// each 128-channel scale group is held by 8 adjacent lanes and one 16-byte
// store per lane writes the lane's codes.
__device__ __forceinline__ void dispatch_slice_fp8(const uint16_t* __restrict__ xrow, int H,
                                                   int slice, int lane, int K, int my_e,
                                                   int my_s, int E, int cap,
                                                   uint8_t* __restrict__ recv,
                                                   float* __restrict__ scales)
{
    const int G = H / 128;
    const int c0 = slice * kSlice + lane * 16;
    const bool act = c0 < H;   // H % 128 == 0: a scale group is all in or all out
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    if (act) {
        a = ld_global_nc(reinterpret_cast<const uint4*>(xrow + c0));
        b = ld_global_nc(reinterpret_cast<const uint4*>(xrow + c0 + 8));
    }
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
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
        const uint32_t lo = pack_e4m3x2(__fdiv_rn(f[4 * j + 0], sc), __fdiv_rn(f[4 * j + 1], sc));
        const uint32_t hi = pack_e4m3x2(__fdiv_rn(f[4 * j + 2], sc), __fdiv_rn(f[4 * j + 3], sc));
        p[j] = lo | (hi << 16);
    }
    const uint4 q = make_uint4(p[0], p[1], p[2], p[3]);
    const bool leader = (lane & 7) == 0;
    const int g = c0 / 128;
    for (int k = 0; k < K; ++k) {
        const int e = __shfl_sync(0xffffffffu, my_e, k);
        const int s = __shfl_sync(0xffffffffu, my_s, k);
        if (!dest_ok(e, s, E, cap) || !act) continue;
        const int64_t row = (int64_t)e * cap + s;
        st_global_cs(reinterpret_cast<uint4*>(recv + row * H + c0), q);
        if (leader) st_global_cs_f32(scales + row * G + g, sc);
    }
}

}  // namespace moedc
