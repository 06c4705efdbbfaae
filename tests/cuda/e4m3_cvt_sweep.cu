// Test-only kernel (not part of libmoedc): the library's binary32 -> e4m3fn
// conversion, moedc::pack_e4m3x2 (cvt.rn.satfinite.e4m3x2.f32), applied to a
// contiguous range of binary32 bit patterns, so a test can compare the
// hardware's rounding with the CPU oracle's encoder over all 2^32 patterns.
#include "common.cuh"

// out[i] = e4m3(bits (base + i)) for i < n; n is a multiple of 8.  Each thread
// converts 8 consecutive patterns and stores their 8 codes with one 8-byte
// store.
__global__ void e4m3_cvt_sweep_kernel(uint32_t base, uint32_t n, uint8_t* __restrict__ out)
{
    const uint32_t groups = n / 8;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < groups; i += stride) {
        const uint32_t p = base + 8u * i;
        uint32_t c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            c[j] = moedc::pack_e4m3x2(__uint_as_float(p + 2u * j), __uint_as_float(p + 2u * j + 1u));
        reinterpret_cast<uint2*>(out)[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    }
}

// Host launcher: 0 on success, the CUDA error code otherwise.  `out` is a
// device buffer of at least n bytes, 8-byte aligned.
extern "C" int e4m3_cvt_sweep(uint32_t base, uint32_t n, void* out, cudaStream_t stream)
{
    if (n % 8 != 0 || out == nullptr || (reinterpret_cast<uintptr_t>(out) % 8) != 0) return -1;
    if (n == 0) return 0;
    const uint32_t groups = n / 8;
    const int threads = 256;
    uint32_t blocks = (groups + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    e4m3_cvt_sweep_kernel<<<blocks, threads, 0, stream>>>(base, n, static_cast<uint8_t*>(out));
    return (int)cudaGetLastError();
}
