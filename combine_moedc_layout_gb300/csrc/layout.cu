// Routing layout: per-expert histogram, per-rank distinct-token counts,
// token-in-rank mask and the deterministic per-expert slot map.
//
// Sources: UCCL PR #749 "[EP] Low-latency mode batch tokens per destination"
// (code excerpt: the per-expert routed-token counter and the per-destination
// rank total built from the rank's local experts; its note that the send
// waits on the counts of all of a rank's experts is why the layout here is a
// complete pass that finishes before dispatch starts), and MORI PR #614
// "perf(ep): InterNodeV1LL low-token latency on MI300X + CX7" (routing-scan
// note: the topk loads are issued together and a negative sentinel expert is
// tested before any division).
//
// No atomics decide order.  Two paths, picked by the number of entries:
//
// Sweep (T*K <= kSweepMaxEntries, one launch, no scratch): block e < E owns
//   expert e and reads every entry (the whole top-k table is at most 256 KB
//   and stays in L2); a block-wide exclusive scan over per-thread match
//   counts gives each match its slot in (t, k) order.  Block E + r owns rank
//   r: it writes column r of is_token_in_rank and counts its tokens.  No
//   block waits on another.
//
// Blocked (larger T*K, two launches, caller scratch):
//   count:  block c histograms its contiguous run of tokens into scratch row
//           c, and counts the distinct tokens it sends to each rank.
//   assign: block c turns the rows of blocks < c into per-expert base
//           offsets, splits its own run over 8 warps (per-warp counts + a
//           scan across warps), then each warp walks its entries in order and
//           ranks equal experts inside a 32-entry tile with __match_any_sync.
//           The last block also writes the totals.
// Rank membership is a range test lo <= e < lo + E/R (no division).
#include "common.cuh"

namespace moedc {

constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / kWarp;
constexpr int kEntriesPerBlock = 1024;     // blocked path: (token, k) entries per block
constexpr int kMaxLayoutBlocks = 1024;
constexpr int kSweepThreads = 1024;
constexpr int kSweepWarps = kSweepThreads / kWarp;
constexpr int kSweepV = 16;                // consecutive entries per thread per round
constexpr int kSweepMaxEntries = 65536;    // sweep path up to here

__device__ __forceinline__ bool valid_expert(int e, int E) { return e >= 0 && e < E; }

// does token row `row` (K entries) send anything to the rank owning [lo, lo + epr)?
__device__ __forceinline__ bool token_in_rank(const int32_t* row, int K, int lo, int epr)
{
    for (int k = 0; k < K; ++k) {
        const unsigned d = (unsigned)row[k] - (unsigned)lo;
        if (d < (unsigned)epr) return true;
    }
    return false;
}

// is entry k the first of its token row that goes to the rank owning [lo, lo + epr)?
__device__ __forceinline__ bool first_in_rank(const int32_t* row, int k, int lo, int epr)
{
    for (int j = 0; j < k; ++j) {
        const unsigned d = (unsigned)row[j] - (unsigned)lo;
        if (d < (unsigned)epr) return false;
    }
    return true;
}

// Sweep layout: blocks [0, E) are experts, blocks [E, E + R) are ranks.
__global__ void __launch_bounds__(kSweepThreads)
layout_sweep_kernel(const int32_t* __restrict__ topk_idx, int T, int K, int E, int R, int cap,
                    bool vec_ok, int32_t* __restrict__ num_tokens_per_expert,
                    int32_t* __restrict__ num_tokens_per_rank,
                    uint8_t* __restrict__ is_token_in_rank, int32_t* __restrict__ slot,
                    int32_t* __restrict__ status)
{
    pdl_enter();
    __shared__ int32_t s_warp[kSweepWarps];
    __shared__ int32_t s_total;
    const int tid = threadIdx.x;
    const int lane = tid % kWarp;
    const int warp = tid / kWarp;
    const int n = T * K;

    if (blockIdx.x < E) {
        const int target = blockIdx.x;
        const bool sweeper = (blockIdx.x == 0);   // block 0 also marks invalid entries
        bool bad = false;
        int running = 0;
        for (int base = 0; base < n; base += kSweepThreads * kSweepV) {
            const int i0 = base + tid * kSweepV;
            int v[kSweepV];
            if (vec_ok && i0 + kSweepV <= n) {
                const int4* p = reinterpret_cast<const int4*>(topk_idx + i0);
#pragma unroll
                for (int q = 0; q < kSweepV / 4; ++q) {
                    const int4 w = __ldg(p + q);
                    v[4 * q] = w.x; v[4 * q + 1] = w.y; v[4 * q + 2] = w.z; v[4 * q + 3] = w.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < kSweepV; ++j)
                    v[j] = (i0 + j < n) ? __ldg(topk_idx + i0 + j) : -1;
            }
            unsigned m = 0;
#pragma unroll
            for (int j = 0; j < kSweepV; ++j) m |= (v[j] == target ? 1u : 0u) << j;
            if (sweeper) {
#pragma unroll
                for (int j = 0; j < kSweepV; ++j) {
                    if (i0 + j < n && !valid_expert(v[j], E)) {
                        slot[i0 + j] = -1;
                        if (v[j] != -1) bad = true;
                    }
                }
            }
            // block-wide exclusive scan of the per-thread match counts
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
            while (m) {
                const int j = __ffs(m) - 1;
                m &= m - 1;
                slot[i0 + j] = s++;
            }
            running += s_total;
            __syncthreads();   // s_warp / s_total are rewritten next round
        }
        if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
        if (tid == 0) {
            num_tokens_per_expert[target] = running;
            if (running > cap) raise_status(status, MOEDC_ERR_CAPACITY);
        }
        return;
    }

    // rank block: column r of is_token_in_rank and its token count
    const int r = blockIdx.x - E;
    const int epr = E / R;
    const int lo = r * epr;
    int c = 0;
    for (int t = tid; t < T; t += kSweepThreads) {
        const bool in = token_in_rank(topk_idx + (int64_t)t * K, K, lo, epr);
        is_token_in_rank[(int64_t)t * R + r] = in ? 1 : 0;
        c += in ? 1 : 0;
    }
#pragma unroll
    for (int d = kWarp / 2; d > 0; d >>= 1) c += __shfl_xor_sync(0xffffffffu, c, d);
    if (lane == 0) s_warp[warp] = c;
    __syncthreads();
    if (warp == 0) {
        int v = s_warp[lane];
#pragma unroll
        for (int d = kWarp / 2; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
        if (lane == 0) num_tokens_per_rank[r] = v;
    }
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_count_kernel(const int32_t* __restrict__ topk_idx, int T, int K, int E, int R, int tpc,
                    int32_t* __restrict__ ws_hist, int32_t* __restrict__ ws_rank,
                    int32_t* __restrict__ status)
{
    pdl_enter();
    extern __shared__ int32_t smem[];
    int32_t* s_idx = smem;                // [tpc * K]
    int32_t* s_hist = s_idx + tpc * K;    // [E]
    int32_t* s_rank = s_hist + E;         // [R]

    const int c = blockIdx.x;
    const int t0 = c * tpc;
    const int nt = min(tpc, T - t0);
    const int n = nt * K;
    const int epr = E / R;

    for (int i = threadIdx.x; i < E; i += blockDim.x) s_hist[i] = 0;
    for (int i = threadIdx.x; i < R; i += blockDim.x) s_rank[i] = 0;
    const int32_t* src = topk_idx + (int64_t)t0 * K;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_idx[i] = src[i];
    __syncthreads();

    bool bad = false;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int e = s_idx[i];
        if (e == -1) continue;
        if (!valid_expert(e, E)) { bad = true; continue; }
        atomicAdd(&s_hist[e], 1);
        const int k = i % K;
        const int r = e / epr;
        if (first_in_rank(s_idx + (i - k), k, r * epr, epr))
            atomicAdd(&s_rank[r], 1);
    }
    if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) ws_hist[(int64_t)c * E + i] = s_hist[i];
    for (int i = threadIdx.x; i < R; i += blockDim.x) ws_rank[(int64_t)c * R + i] = s_rank[i];
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_assign_kernel(const int32_t* __restrict__ topk_idx, int T, int K, int E, int R, int cap,
                     int tpc, const int32_t* __restrict__ ws_hist,
                     const int32_t* __restrict__ ws_rank,
                     int32_t* __restrict__ num_tokens_per_expert,
                     int32_t* __restrict__ num_tokens_per_rank,
                     uint8_t* __restrict__ is_token_in_rank, int32_t* __restrict__ slot,
                     int32_t* __restrict__ status)
{
    pdl_enter();
    extern __shared__ int32_t smem[];
    int32_t* s_idx = smem;                          // [tpc * K]
    int32_t* s_whist = s_idx + tpc * K;             // [kLayoutWarps][E]
    int32_t* s_base = s_whist + kLayoutWarps * E;   // [E]
    int32_t* s_rank = s_base + E;                   // [R]

    const int c = blockIdx.x;
    const bool last = (c == gridDim.x - 1);
    const int t0 = c * tpc;
    const int nt = max(0, min(tpc, T - t0));
    const int n = nt * K;
    const int epr = E / R;
    const int warp = threadIdx.x / kWarp;
    const int lane = threadIdx.x % kWarp;

    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) s_whist[i] = 0;
    for (int i = threadIdx.x; i < E; i += blockDim.x) s_base[i] = 0;
    for (int i = threadIdx.x; i < R; i += blockDim.x) s_rank[i] = 0;
    const int32_t* src = topk_idx + (int64_t)t0 * K;
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_idx[i] = src[i];
    __syncthreads();

    // base offsets: entries routed to each expert by the blocks before this one
    {
        const int m = c * E;
#pragma unroll 4
        for (int i = threadIdx.x; i < m; i += blockDim.x)
            atomicAdd(&s_base[i % E], ws_hist[i]);
    }
    if (last) {
        const int m = c * R;
        for (int i = threadIdx.x; i < m; i += blockDim.x)
            atomicAdd(&s_rank[i % R], ws_rank[i]);
        bool bad = false;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const int e = s_idx[i];
            if (e == -1) continue;
            if (!valid_expert(e, E)) { bad = true; continue; }
            const int k = i % K;
            const int r = e / epr;
            if (first_in_rank(s_idx + (i - k), k, r * epr, epr))
                atomicAdd(&s_rank[r], 1);
        }
        if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
    }

    // each warp owns a contiguous run of whole 32-entry tiles
    const int run = ((n + kLayoutWarps * kWarp - 1) / (kLayoutWarps * kWarp)) * kWarp;
    const int wbeg = min(n, warp * run);
    const int wend = min(n, wbeg + run);
    int32_t* my_hist = s_whist + warp * E;
    for (int i = wbeg + lane; i < wend; i += kWarp) {
        const int e = s_idx[i];
        if (valid_expert(e, E)) atomicAdd(&my_hist[e], 1);
    }
    __syncthreads();

    // exclusive scan across warps, on top of the block's base offset
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int acc = s_base[e];
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int v = s_whist[w * E + e];
            s_whist[w * E + e] = acc;
            acc += v;
        }
        if (last) {
            num_tokens_per_expert[e] = acc;
            if (acc > cap) raise_status(status, MOEDC_ERR_CAPACITY);
        }
    }
    if (last)
        for (int r = threadIdx.x; r < R; r += blockDim.x) num_tokens_per_rank[r] = s_rank[r];
    __syncthreads();

    // slots, tile by tile in entry order
    const unsigned lt = lanemask_lt();
    int32_t* dst = slot + (int64_t)t0 * K;
    for (int i0 = wbeg; i0 < wend; i0 += kWarp) {
        const int i = i0 + lane;
        const int e = (i < wend) ? s_idx[i] : -1;
        const bool v = valid_expert(e, E);
        const unsigned peers = __match_any_sync(0xffffffffu, v ? e : -1);
        int s = -1;
        if (v) s = my_hist[e] + __popc(peers & lt);
        __syncwarp();
        if (v && (peers & lt) == 0) my_hist[e] += __popc(peers);
        __syncwarp();
        if (i < wend) dst[i] = s;
    }

    // token-in-rank rows of this block's tokens
    uint8_t* rows = is_token_in_rank + (int64_t)t0 * R;
    for (int b = threadIdx.x; b < nt * R; b += blockDim.x) {
        const int t = b / R;
        const int r = b - t * R;
        rows[b] = token_in_rank(s_idx + t * K, K, r * epr, epr) ? 1 : 0;
    }
}

size_t count_smem(int tpc, int K, int E, int R) { return (size_t)(tpc * K + E + R) * 4; }
size_t assign_smem(int tpc, int K, int E, int R)
{
    return (size_t)(tpc * K + kLayoutWarps * E + E + R) * 4;
}

}  // namespace moedc

namespace moedc_host {

bool layout_args_ok(int T, int K, int E, int R, int cap)
{
    if (T < 0 || K < 1 || K > MOEDC_MAX_K || E < 1 || E > MOEDC_MAX_E || R < 1 || R > E ||
        E % R != 0 || cap < 1)
        return false;
    if ((int64_t)T * K > (int64_t)moedc::kMaxLayoutBlocks * 16384)
        return false;
    return true;
}

LayoutGeom layout_geometry(int T, int K, int E, int R)
{
    LayoutGeom g{};
    const int64_t n = (int64_t)T * K;
    if (n <= moedc::kSweepMaxEntries) {
        g.sweep = true;
        g.tpc = T;
        g.blocks = E + R;
        g.ws = 0;
        return g;
    }
    g.sweep = false;
    int tpc = (moedc::kEntriesPerBlock + K - 1) / K;
    const int min_tpc = (T + moedc::kMaxLayoutBlocks - 1) / moedc::kMaxLayoutBlocks;
    if (tpc < min_tpc) tpc = min_tpc;
    g.tpc = tpc;
    g.blocks = (T + tpc - 1) / tpc;
    g.ws = (size_t)g.blocks * (size_t)(E + R) * sizeof(int32_t);
    return g;
}

static int ensure_smem_attr(const void* fn, size_t bytes)
{
    if (bytes <= 48 * 1024) return MOEDC_OK;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
                   cudaSuccess
               ? MOEDC_OK
               : MOEDC_ERR_CUDA;
}

int launch_layout(const int32_t* topk_idx, int T, int K, int E, int R, int cap,
                  int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                  uint8_t* is_token_in_rank, int32_t* slot, void* workspace,
                  size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream)
{
    const LayoutGeom g = layout_geometry(T, K, E, R);
    // the single pass, wherever the shape and the workspace allow it
    const int st = launch_layout_onepass(topk_idx, T, K, E, R, cap, num_tokens_per_expert,
                                         num_tokens_per_rank, is_token_in_rank, slot, workspace,
                                         workspace_bytes, dev_status, stream);
    if (st != MOEDC_ERR_UNIMPLEMENTED) return st;
    if (g.sweep) {
        const bool vec_ok = aligned(topk_idx, 16);
        clear_stale_error();
        launch(moedc::layout_sweep_kernel, g.blocks, moedc::kSweepThreads, 0, stream, topk_idx, T, K, E, R, cap, vec_ok, num_tokens_per_expert, num_tokens_per_rank,
            is_token_in_rank, slot, dev_status);
        return launch_status();
    }
    // the two-kernel path (also the fallback of a refused single pass) needs its own scratch
    if (!workspace || workspace_bytes < g.ws || !aligned(workspace, 16)) return MOEDC_ERR_ARG;
    int32_t* ws_hist = static_cast<int32_t*>(workspace);
    int32_t* ws_rank = ws_hist + (size_t)g.blocks * E;
    if (g.blocks > 1) {
        const size_t sm = moedc::count_smem(g.tpc, K, E, R);
        if (ensure_smem_attr((const void*)moedc::layout_count_kernel, sm) != MOEDC_OK)
            return MOEDC_ERR_CUDA;
        clear_stale_error();
        launch(moedc::layout_count_kernel, g.blocks, moedc::kLayoutThreads, sm, stream, topk_idx, T, K, E, R, g.tpc, ws_hist, ws_rank, dev_status);
        if (launch_status() != MOEDC_OK) return MOEDC_ERR_CUDA;
    }
    const size_t sm = moedc::assign_smem(g.tpc, K, E, R);
    if (ensure_smem_attr((const void*)moedc::layout_assign_kernel, sm) != MOEDC_OK)
        return MOEDC_ERR_CUDA;
    clear_stale_error();
    launch(moedc::layout_assign_kernel, g.blocks, moedc::kLayoutThreads, sm, stream, topk_idx, T, K, E, R, cap, g.tpc, ws_hist, ws_rank, num_tokens_per_expert,
        num_tokens_per_rank, is_token_in_rank, slot, dev_status);
    return launch_status();
}

}  // namespace moedc_host

extern "C" size_t moedc_layout_workspace_bytes(int T, int K, int E, int R)
{
    if (!moedc_host::layout_args_ok(T, K, E, R, 1)) return 0;
    const size_t need = moedc_host::layout_geometry(T, K, E, R).ws;
    const size_t fast = moedc_host::layout_onepass_workspace_bytes(T, K, E, R);
    return need > fast ? need : fast;
}

extern "C" int moedc_layout(const int32_t* topk_idx, int T, int K, int E, int R, int cap,
                            int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                            uint8_t* is_token_in_rank, int32_t* slot, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream)
{
    using namespace moedc_host;
    if (!layout_args_ok(T, K, E, R, cap)) return MOEDC_ERR_ARG;
    if (!num_tokens_per_expert || !num_tokens_per_rank || !dev_status) return MOEDC_ERR_ARG;
    if (T > 0 && (!topk_idx || !is_token_in_rank || !slot)) return MOEDC_ERR_ARG;
    if (!aligned(topk_idx, 4) || !aligned(slot, 4) || !aligned(num_tokens_per_expert, 4) ||
        !aligned(num_tokens_per_rank, 4) || !aligned(dev_status, 4))
        return MOEDC_ERR_ARG;
    // beyond 65536 entries a workspace is required: one that holds either the
    // single-pass layout's rows or the two-kernel path's counts
    const LayoutGeom g = layout_geometry(T, K, E, R);
    const size_t fast = layout_onepass_workspace_bytes(T, K, E, R);
    const bool ws_ok = workspace && aligned(workspace, 16) &&
                       (workspace_bytes >= g.ws || (fast > 0 && workspace_bytes >= fast));
    if (g.ws > 0 && !ws_ok) return MOEDC_ERR_ARG;
    return launch_layout(topk_idx, T, K, E, R, cap, num_tokens_per_expert, num_tokens_per_rank,
                         is_token_in_rank, slot, workspace, workspace_bytes, dev_status, stream);
}
