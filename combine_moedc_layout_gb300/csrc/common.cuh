// Shared device helpers for the libmoedc kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moedc.h"

namespace moedc {

constexpr int kWarp = 32;

// Raise the caller's status word to max(*status, code): the result does not
// depend on which thread reports first.
__device__ __forceinline__ void raise_status(int32_t* status, int code)
{
    atomicMax(status, code);
}

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Lanes of the warp holding the same expert as this lane (invalid lanes match
// each other): the intersection, over the bits of the key e + 1 (0 when
// invalid, at most MOEDC_MAX_E), of the lanes that agree on that bit.  Eleven
// independent ballots; in the shared-memory layout passes of the single-launch
// kernels the hardware match.any measured several times slower for 32 mostly
// distinct keys.
constexpr int kExpertKeyBits = 11;
static_assert(MOEDC_MAX_E < (1 << kExpertKeyBits), "expert match key width");
__device__ __forceinline__ unsigned match_expert(int e, bool valid)
{
    const int key = valid ? e + 1 : 0;
    unsigned peers = 0xffffffffu;
#pragma unroll
    for (int b = 0; b < kExpertKeyBits; ++b) {
        const bool bit = (key >> b) & 1;
        const unsigned m = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? m : ~m;
    }
    return peers;
}

// bf16 bit pattern -> binary32 (exact widening).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// binary32 -> bf16, round to nearest even (hardware cvt.rn.bf16x2.f32);
// `lo` lands in the low half of the result.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two binary32 values -> two e4m3fn codes, round to nearest even with
// saturation to +-448 (cvt.rn.satfinite.e4m3x2.f32); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi)
{
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3 codes (low byte first) -> two binary32 values.  Exact: every e4m3
// value is an f16 value, and f16 widens exactly.
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t two_codes, float& lo, float& hi)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two_codes));
    asm("cvt.f32.f16 %0, %1;" : "=f"(lo) : "h"((unsigned short)(h2 & 0xffffu)));
    asm("cvt.f32.f16 %0, %1;" : "=f"(hi) : "h"((unsigned short)(h2 >> 16)));
}

// Channel pairs in binary32.  The sm_100 family's packed binary32 multiply
// (mul.rn.f32x2) applies one IEEE round-to-nearest-even multiply to each of
// two lanes, so a pair of products costs one instruction where two scalar
// ones stood.  Sums stay scalar (__fadd_rn): with both the multiply and the
// add in packed form the compiler fused a packed product into the packed sum
// that consumes it, leaving the product unrounded - measured on this GPU,
// 83342 of the 4096-token e4m3 combine's outputs (and 1276 of the bf16
// combine's) came out one bf16 ulp away from the unfused result, while
// packed multiplies alone, and packed adds alone, were bit-exact against the
// scalar operations on 8 million random pairs and on every workload.  The
// method rounds every product before it is summed, so only one of the two
// may be packed; packed multiplies measured as fast as packed adds (e4m3
// combine 55.3 us for either, 59.4 us scalar).
// A product can instead come from a packed FMA whose addend is -0 held in a
// register (a kernel argument, so the compiler cannot see its value): x + -0
// is x for every x under round-to-nearest, so the result is the rounded
// product, and a sum that consumes an FMA's result cannot be contracted with
// it.  Then the sum may be packed as well.
// MOEDC_F32X2 selects the form for comparison builds: bit 0 packed
// multiplies, bit 1 packed adds (3 is the fusing form: not for use), bit 2
// weighted products as packed FMAs with a -0 addend and their sums packed.
#ifndef MOEDC_F32X2
#define MOEDC_F32X2 1
#endif

__device__ __forceinline__ unsigned long long f32x2_bits(float2 v)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(v.x), "f"(v.y));
    return r;
}

__device__ __forceinline__ float2 f32x2_from_bits(unsigned long long r)
{
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}

__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b)
{
#if MOEDC_F32X2 & 1
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f32x2_bits(a)), "l"(f32x2_bits(b)));
    return f32x2_from_bits(r);
#else
    return make_float2(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y));
#endif
}

__device__ __forceinline__ float2 add2_rn(float2 a, float2 b)
{
#if MOEDC_F32X2 & 2
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f32x2_bits(a)), "l"(f32x2_bits(b)));
    return f32x2_from_bits(r);
#else
    return make_float2(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y));
#endif
}

// Packed sum for operands that never come from a multiply (the rank
// combine's widened bf16 partials), where no product can be fused into it.
__device__ __forceinline__ float2 add2_rn_unfed(float2 a, float2 b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f32x2_bits(a)), "l"(f32x2_bits(b)));
    return f32x2_from_bits(r);
}

__device__ __forceinline__ float2 splat2(float s) { return make_float2(s, s); }

__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(f32x2_bits(a)), "l"(f32x2_bits(b)), "l"(f32x2_bits(c)));
    return f32x2_from_bits(r);
}

// acc + RN(w * x) lane by lane, the product rounded before the sum.
// `neg_zero` is -0.0f passed in at run time (bit 2 of MOEDC_F32X2).
__device__ __forceinline__ float2 acc_prod2_rn(float2 acc, float2 w, float2 x, float neg_zero)
{
#if MOEDC_F32X2 & 4
    return add2_rn_unfed(acc, fma2_rn(w, x, splat2(neg_zero)));
#else
    (void)neg_zero;
    return add2_rn(acc, mul2_rn(w, x));
#endif
}

// the two bf16 values of a 32-bit word (low half first), widened exactly
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w)
{
    return make_float2(bf16_lo(w), bf16_hi(w));
}

// two e4m3 codes (low byte first), widened exactly
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_codes)
{
    float lo, hi;
    e4m3x2_to_f32(two_codes, lo, hi);
    return make_float2(lo, hi);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float2 v) { return pack_bf16x2(v.x, v.y); }

// Plain 16-byte global accesses.  Streaming stores: written rows are not
// re-read by this kernel, so they should not displace reusable lines.
#ifndef MOEDC_LD_POLICY
#define MOEDC_LD_POLICY ".L1::no_allocate"
#endif

__device__ __forceinline__ uint4 ld_global_nc(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc" MOEDC_LD_POLICY ".v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

#ifndef MOEDC_ST_POLICY
#define MOEDC_ST_POLICY ".cs"
#endif

__device__ __forceinline__ void st_global_cs(uint4* p, uint4 v)
{
    asm volatile("st.global" MOEDC_ST_POLICY ".v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st_global_cs_f32(float* p, float v)
{
    asm volatile("st.global" MOEDC_ST_POLICY ".f32 [%0], %1;" :: "l"(p), "f"(v) : "memory");
}

// Stores of dispatched rows and their scales into the receive buffer: plain
// write-back stores, normal L2 priority.  The receive rows are what the next
// kernel reads (the experts), so marking them evict-first works against it.
// And in a layout -> dispatch -> combine step, evict-first receive rows left
// the step's time to where the buffers landed in memory: 143.5-151.5 us per
// 4096-token step from process to process, against 146.3-146.8 us in each of
// 13 processes with plain stores.
#ifndef MOEDC_RECV_ST_POLICY
#define MOEDC_RECV_ST_POLICY ""
#endif

__device__ __forceinline__ void st_global_recv(uint4* p, uint4 v)
{
    asm volatile("st.global" MOEDC_RECV_ST_POLICY ".v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st_global_recv_f32(float* p, float v)
{
    asm volatile("st.global" MOEDC_RECV_ST_POLICY ".f32 [%0], %1;" :: "l"(p), "f"(v) : "memory");
}

#ifndef MOEDC_PDL
#define MOEDC_PDL 1
#endif

// Programmatic dependent launch.  Every kernel of the library starts here: it
// waits (in hardware) until the previous kernel in the stream has completed
// and its memory is visible - a no-op when that launch carried no
// programmatic dependency - and then lets the next kernel in the stream start
// launching, so its blocks are scheduled while this one drains.  The next
// kernel can only launch once every block of this one has passed this point,
// so its waiting blocks never keep a block of this grid from being scheduled.
__device__ __forceinline__ void pdl_enter()
{
#if MOEDC_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

}  // namespace moedc

// Host-side helpers shared by the entry points.
namespace moedc_host {

// out_dtype: MOEDC_BF16, MOEDC_FP8_E4M3, or MOEDC_FP8_E4M3 | MOEDC_SCALES_COL_MAJOR
inline bool dtype_ok(int d)
{
    return d == MOEDC_BF16 || d == MOEDC_FP8_E4M3 ||
           d == (MOEDC_FP8_E4M3 | MOEDC_SCALES_COL_MAJOR) ||
           d == (MOEDC_FP8_E4M3 | MOEDC_SCALES_PER_TOKEN);
}
// the element type of an out_dtype, without its scale-layout flag
inline int dtype_base(int d) { return d & ~(MOEDC_SCALES_COL_MAJOR | MOEDC_SCALES_PER_TOKEN); }
// scale index mode of a scale_layout argument: 0 rows [E][cap][G], 1 columns
// [E][G][cap], 2 one per row [E][cap]; -1 for anything else
inline int scale_mode(int layout)
{
    return layout == 0                        ? 0
           : layout == MOEDC_SCALES_COL_MAJOR ? 1
           : layout == MOEDC_SCALES_PER_TOKEN ? 2
                                              : -1;
}
int sm_count();                 // multiprocessors of the current device
// blocks of `kernel` resident on the whole current device at once
int resident_blocks(const void* kernel, int threads, size_t smem);
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
// Launch checks read this library's own runtime error state (cudart is linked
// statically, so it is not shared with other runtimes in the process).
// clear_stale_error() drops a non-sticky error left by an earlier query so
// that launch_status() reports only the launch that follows it.
inline void clear_stale_error() { (void)cudaGetLastError(); }
inline int launch_status() { return cudaGetLastError() == cudaSuccess ? MOEDC_OK : MOEDC_ERR_CUDA; }

// Launch with the programmatic-stream-serialisation attribute (see
// pdl_enter); a failed launch is left in the runtime's last-error state for
// launch_status() to report.
template <typename... KArgs, typename... Args>
inline void launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = MOEDC_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    (void)cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Layout geometry: tokens per thread block of the layout kernels.
struct LayoutGeom {
    bool sweep;     // single-launch sweep path (no scratch)
    int tpc;        // blocked path: tokens per block
    int blocks;     // number of blocks (>= 1)
    size_t ws;      // scratch bytes (0 on the sweep path)
};
LayoutGeom layout_geometry(int T, int K, int E, int R);
bool layout_args_ok(int T, int K, int E, int R, int cap);

// Launches of the layout kernels (layout.cu); used by the fused entry point.
// Up to 65536 entries a workspace of layout_onepass_workspace_bytes selects
// the single-pass kernel (layout_onepass.cu), no workspace the sweep.
int launch_layout(const int32_t* topk_idx, int T, int K, int E, int R, int cap,
                  int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                  uint8_t* is_token_in_rank, int32_t* slot, void* workspace,
                  size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);
size_t layout_onepass_workspace_bytes(int T, int K, int E, int R);
// MOEDC_ERR_UNIMPLEMENTED when the shape or the workspace does not take it
int launch_layout_onepass(const int32_t* topk_idx, int T, int K, int E, int R, int cap,
                          int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                          uint8_t* is_token_in_rank, int32_t* slot, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);
// extra arrivals every bounded wait waits for (moedc_test_set_wait_extra)
unsigned test_wait_extra();
int launch_dispatch(const void* x, int T, int H, const int32_t* topk_idx, const int32_t* slot,
                    const int32_t* num_tokens_per_expert, int K, int E, int cap, int out_dtype,
                    void* recv, float* scales, int32_t* src_idx, int32_t* dev_status,
                    cudaStream_t stream);
// cooperative single-launch layout + dispatch (layout_dispatch_coop.cu);
// MOEDC_ERR_UNIMPLEMENTED when it does not apply
size_t layout_dispatch_coop_workspace_bytes(int T, int K, int E, int R);
int launch_layout_dispatch_coop(const void* x, const int32_t* topk_idx, int T, int H, int K,
                                int E, int R, int cap, int out_dtype,
                                int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                uint8_t* is_token_in_rank, int32_t* slot, void* recv,
                                float* scales, int32_t* src_idx, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream);
// e4m3 dispatch with one scale per token row (dispatch_token.cu)
int launch_dispatch_token(const void* x, int T, int H, const int32_t* topk_idx,
                          const int32_t* slot, const int32_t* num_tokens_per_expert, int K,
                          int E, int cap, void* recv, float* scales, int32_t* src_idx,
                          int32_t* dev_status, cudaStream_t stream);

}  // namespace moedc_host
