// Routing layout in one pass over the routing table (from 4 chunks of 1024
// entries up to 144 chunks of 4096 entries, with a caller workspace).
//
// Sources: UCCL PR #749 "[EP] Low-latency mode batch tokens per destination"
// (code excerpt: per-expert routed-token counters published for the ranks
// that wait on them; its note that a rank's send waits on the counts of all
// of its experts), and MORI PR #614 "perf(ep): InterNodeV1LL low-token
// latency on MI300X + CX7" (routing-scan note: the top-k loads are issued
// together).  The layout's outputs are those of layout.cu; only the order of
// work differs.
//
// Block b owns chunk b: a run of whole tokens, at most 1024 * EPT (token, k)
// entries, EPT entries per thread (EPT = 1, 2 or 4: the smallest that keeps
// the chunks within one resident grid).
//   1. load the chunk's expert ids (one coalesced load);
//   2. rank each entry among the chunk's entries of the same expert in
//      (t, k) order: in-warp rank from the ballot match of each 32-entry tile
//      (with EPT > 1 plus the warp's running count of the expert), plus the
//      counts of the earlier warps (a scan over the 32 warp counts of each
//      expert), giving the chunk's per-expert totals; the chunk's
//      token-in-rank rows, and per rank the number of its tokens that reach
//      it;
//   3. publish those E + R counts as row b of the workspace, each count in a
//      64-bit word whose upper bits carry this launch's epoch, so that a word
//      is its own flag (no fence, no separate flag);
//   4. read rows 0 .. b-1, each word until it carries the epoch (a bounded
//      wait), and sum them into this chunk's base offsets;
//   5. slot = base + in-chunk rank; the last block writes the totals and the
//      capacity status.
// The table is read once in all (the sweep kernel reads it once per
// expert).  A block waits only on blocks with smaller indices; the launch
// is cooperative, so every block of the grid is resident and those waits
// end.  A wait that runs out raises MOEDC_ERR_TIMEOUT.
//
// Epochs: a launch's epoch is the per-call host counter plus a generation
// word of the workspace times an odd constant, cut to 51 bits (a count takes
// the low 13: a chunk never counts past 4096).  Every block reads the
// generation at its start; the last block advances it only after it has
// read every other block's row (so every block has read the generation),
// and a block that gives up advances it too.  Words left by earlier
// launches, by earlier replays of one captured graph (same host counter) or
// by uninitialised memory therefore do not carry the epoch (a random word
// matches with probability 2^-51): the workspace needs no initialisation.
#include <atomic>
#include <chrono>
#include <climits>
#include <mutex>

#include "common.cuh"

namespace moedc {

constexpr int kOpThreads = 1024;
constexpr int kOpWarps = kOpThreads / kWarp;
// At most this many chunks (blocks of 1024 threads, one per SM): the grid
// must be resident at once, and a device may report more SMs than a
// partition of it offers (the launch then falls back).
constexpr int kOpMaxChunks = 144;
// Fewer chunks than this take the sweep: one or two blocks rank everything
// serially, while the sweep spreads it over E + R blocks (measured at 1024
// entries: 9.8 us single pass, 8.2 us sweep).
constexpr int kOpMinChunks = 4;
constexpr size_t kOpHeaderBytes = 256;         // generation word, then padding
constexpr int kOpCountBits = 13;               // a chunk's counts are <= 4096
constexpr unsigned long long kOpCountMask = (1ull << kOpCountBits) - 1;
constexpr unsigned long long kOpTagMask = (1ull << (64 - kOpCountBits)) - 1;
constexpr long long kOpSpinLimit = 1ll << 21;   // polls, 64 ns sleeps after the first 64: >= 0.13 s
constexpr int kOpBatch = 16;                    // row words in flight per thread
constexpr unsigned long long kOpEpochStride = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ unsigned long long op_ld_relaxed(const unsigned long long* p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void op_st_relaxed(unsigned long long* p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ bool op_token_in_rank(const int32_t* row, int K, int lo, int epr)
{
    for (int k = 0; k < K; ++k)
        if ((unsigned)row[k] - (unsigned)lo < (unsigned)epr) return true;
    return false;
}

// A published word's count, once it carries `tag` (bounded wait); -1 if the
// wait ran out.  `w` is the word already loaded once.
__device__ int op_count_when_tagged(const unsigned long long* p, unsigned long long w,
                                    unsigned long long tag)
{
    for (long long it = 0; (w >> kOpCountBits) != tag; ++it) {
        if (it >= kOpSpinLimit) return -1;
        if (it >= 64) __nanosleep(64);   // spin first: the row is usually microseconds away
        w = op_ld_relaxed(p);
    }
    return (int)(w & kOpCountMask);
}

// Shared memory (dynamic, int32 words):
//   s_wc  [kOpWarps][E + 1]  per-warp expert counts, then their exclusive
//                            prefix over warps (rows padded against bank
//                            conflicts in the column scan)
//   s_cnt [E + R]            this chunk's counts (experts, then ranks)
//   s_pre [E + R]            entries / tokens of the chunks before this one
//   s_ids [1024 * EPT]       the chunk's expert ids; later the partial sums
//                            of step 4
// Warp w owns the chunk's entries [w * 32 * EPT, (w + 1) * 32 * EPT), EPT
// tiles of 32 in order; thread (w, lane) holds entry w * 32 * EPT + 32 u +
// lane of tile u.
template <int EPT>
__global__ void __launch_bounds__(kOpThreads, 1)
layout_onepass_kernel(const int32_t* __restrict__ topk_idx, int T, int K, int E, int R,
                      int cap, int tpc, int32_t* __restrict__ num_tokens_per_expert,
                      int32_t* __restrict__ num_tokens_per_rank,
                      uint8_t* __restrict__ is_token_in_rank, int32_t* __restrict__ slot,
                      unsigned long long* __restrict__ ws_generation,
                      unsigned long long* __restrict__ ws_rows, unsigned long long host_epoch,
                      unsigned wait_extra, int32_t* __restrict__ status)
{
    pdl_enter();
    extern __shared__ int32_t smem[];
    const int ER = E + R;
    const int wstride = E + 1;
    int32_t* s_wc = smem;
    int32_t* s_cnt = s_wc + kOpWarps * wstride;
    int32_t* s_pre = s_cnt + ER;
    int32_t* s_ids = s_pre + ER;
    __shared__ unsigned long long s_tag;

    const int tid = threadIdx.x;
    const int lane = tid % kWarp;
    const int warp = tid / kWarp;
    const int b = blockIdx.x;
    const int nb = gridDim.x;
    const int t0 = b * tpc;
    const int nt = max(0, min(tpc, T - t0));
    const int n = nt * K;
    const int epr = E / R;

    // 1. the chunk's ids (in flight while shared memory is cleared) and the epoch
    const int i0 = warp * kWarp * EPT + lane;   // entry of tile 0; tile u adds 32 u
    int e[EPT];
#pragma unroll
    for (int u = 0; u < EPT; ++u) {
        const int i = i0 + u * kWarp;
        e[u] = i < n ? __ldg(topk_idx + (int64_t)t0 * K + i) : -1;
    }
    if (tid == 0) {
        const unsigned long long gen = __ldcg(ws_generation);
        s_tag = ((host_epoch + gen * kOpEpochStride) | 1ull) & kOpTagMask;
    }
    for (int i = tid; i < kOpWarps * wstride; i += kOpThreads) s_wc[i] = 0;
    for (int i = tid; i < R; i += kOpThreads) s_cnt[E + i] = 0;
#pragma unroll
    for (int u = 0; u < EPT; ++u)
        if (i0 + u * kWarp < n) s_ids[i0 + u * kWarp] = e[u];
    __syncthreads();
    const unsigned long long tag = s_tag;

    // 2. in-chunk ranks and counts: tile by tile, an entry's rank in its warp
    //    is the warp's running count of its expert plus its rank in the tile
    bool bad = false;
    unsigned valid_bits = 0;
    int rank[EPT];
    int32_t* my_wc = s_wc + warp * wstride;
#pragma unroll
    for (int u = 0; u < EPT; ++u) {
        const bool in_chunk = i0 + u * kWarp < n;
        const bool valid = in_chunk && e[u] >= 0 && e[u] < E;
        bad = bad || (in_chunk && e[u] != -1 && !valid);
        valid_bits |= (valid ? 1u : 0u) << u;
        const unsigned peers = match_expert(e[u], valid);
        const unsigned before = peers & lanemask_lt();
        rank[u] = valid ? my_wc[e[u]] + __popc(before) : 0;
        __syncwarp();
        if (valid && before == 0) my_wc[e[u]] += __popc(peers);
        __syncwarp();
    }
    // token-in-rank rows of this chunk, and per rank its tokens that reach it.
    // With K a power of two up to 32, a 32-entry tile holds whole tokens, K
    // lanes each: the token's lanes OR their entries' rank bits by shuffles.
    // With R <= 32 as well, the ranks go in rounds of K: in round r0, lane k
    // of a token owns rank r0 + k: it writes that byte and sums the bit over
    // its tiles, and lanes of equal k sum across the warp's tokens before one
    // shared-memory add.
    if (K >= 2 && K <= kWarp && (K & (K - 1)) == 0 && R <= kWarp) {
        const int kl = lane & (K - 1);
        unsigned m[EPT];
#pragma unroll
        for (int u = 0; u < EPT; ++u) {
            m[u] = ((valid_bits >> u) & 1u) ? 1u << (e[u] / epr) : 0u;
            for (int d = 1; d < K; d <<= 1) m[u] |= __shfl_xor_sync(0xffffffffu, m[u], d);
        }
        for (int r0 = 0; r0 < R; r0 += K) {
            const int r = r0 + kl;
            int mine = 0;
#pragma unroll
            for (int u = 0; u < EPT; ++u) {
                const int i = i0 + u * kWarp;
                if (i < n && r < R) {
                    const int in = (int)((m[u] >> r) & 1u);
                    is_token_in_rank[((int64_t)t0 + i / K) * R + r] = (uint8_t)in;
                    mine += in;
                }
            }
            for (int d = K; d < kWarp; d <<= 1) mine += __shfl_xor_sync(0xffffffffu, mine, d);
            if (lane < K && r < R && mine) atomicAdd(&s_cnt[E + r], mine);
        }
    } else {
        // Otherwise each thread takes (token, rank) pairs and scans the token's ids
        // in shared memory.  When R divides the block, every pair a thread visits
        // has rank tid % R: the thread sums its own pairs and lanes of equal rank
        // combine by shuffles before one shared-memory add.
        uint8_t* inr = is_token_in_rank + (int64_t)t0 * R;
        const bool same_rank = (kOpThreads % R) == 0;
        int mine = 0;
        const int rshift = (R & (R - 1)) == 0 ? __ffs(R) - 1 : -1;   // R a power of two
        for (int p = tid; p < nt * R; p += kOpThreads) {
            const int tl = rshift >= 0 ? p >> rshift : p / R;
            const int rr = p - tl * R;
            const bool in = op_token_in_rank(s_ids + tl * K, K, rr * epr, epr);
            inr[p] = in ? 1 : 0;
            if (same_rank)
                mine += in ? 1 : 0;
            else if (in)
                atomicAdd(&s_cnt[E + rr], 1);
        }
        if (same_rank) {
            if (R < kWarp) {   // R divides 32: lanes l and l ^ d (d >= R) share a rank
                for (int d = kWarp / 2; d >= R; d >>= 1)
                    mine += __shfl_xor_sync(0xffffffffu, mine, d);
                if (lane < R && mine) atomicAdd(&s_cnt[E + lane], mine);
            } else if (mine) {
                atomicAdd(&s_cnt[E + tid % R], mine);
            }
        }
    }
    __syncthreads();
    // exclusive prefix over the 32 warps of each expert's count.  P adjacent
    // threads share an expert (P * E <= 1024, P a power of two up to 32);
    // each sums its run of 32 / P warp counts (independent shared-memory
    // loads), the P runs are scanned with log2(P) shuffles, and each thread
    // writes its run's prefixes.  With the padded rows a warp's loads fall in
    // distinct banks.
    {
        int P = 1;
        while (P < kWarp && 2 * P * E <= kOpThreads) P *= 2;
        const int per = kWarp / P;
        const int ex = tid / P;
        const int q = tid - ex * P;
        int32_t* col = s_wc + q * per * wstride + ex;
        int run = 0;
        if (ex < E)
            for (int i = 0; i < per; ++i) run += col[i * wstride];
        int incl = run;
        for (int d = 1; d < P; d <<= 1) {   // P divides 32: groups never straddle warps
            const int y = __shfl_up_sync(0xffffffffu, incl, d);
            if (q >= d) incl += y;
        }
        if (ex < E) {
            int acc = incl - run;
            for (int i = 0; i < per; ++i) {
                const int v = col[i * wstride];
                col[i * wstride] = acc;
                acc += v;
            }
            if (q == P - 1) s_cnt[ex] = incl;
        }
    }
    __syncthreads();

    // 3. publish this chunk's counts, each word tagged with the epoch
    unsigned long long* my_row = ws_rows + (int64_t)b * ER;
    for (int c = tid; c < ER; c += kOpThreads)
        op_st_relaxed(my_row + c, (tag << kOpCountBits) | (unsigned long long)s_cnt[c]);

    // 4. sum rows 0 .. b-1: G groups of threads split the rows, so that each
    //    thread has at most a few words to read, all in flight together.  The
    //    test hook makes the last block also wait for a word after the last
    //    row, which no block writes.
    const int G = ER <= kOpThreads ? kOpThreads / ER : 1;
    bool ok = true;
    for (int c0 = 0; c0 < ER; c0 += G > 1 ? ER : kOpThreads) {
        const int g = G > 1 ? tid / ER : 0;
        const int c = G > 1 ? tid - g * ER : c0 + tid;
        int acc = 0;
        if (g < G && c < ER) {
            for (int j0 = g; j0 < b && ok; j0 += G * kOpBatch) {
                // a batch of words, re-polled together until each carries the
                // epoch: the loads of one round are all in flight at once
                unsigned long long w[kOpBatch];
                unsigned pending = 0;
#pragma unroll
                for (int u = 0; u < kOpBatch; ++u) {
                    const int j = j0 + u * G;
                    w[u] = 0;
                    if (j < b) {
                        w[u] = op_ld_relaxed(ws_rows + (int64_t)j * ER + c);
                        pending |= 1u << u;
                    }
                }
                for (long long it = 0;; ++it) {
#pragma unroll
                    for (int u = 0; u < kOpBatch; ++u) {
                        if (((pending >> u) & 1u) && (w[u] >> kOpCountBits) == tag) {
                            acc += (int)(w[u] & kOpCountMask);
                            pending &= ~(1u << u);
                        }
                    }
                    if (pending == 0) break;
                    if (it >= kOpSpinLimit) {
                        ok = false;
                        break;
                    }
                    if (it >= 64) __nanosleep(64);   // spin first: rows are microseconds away
#pragma unroll
                    for (int u = 0; u < kOpBatch; ++u)
                        if ((pending >> u) & 1u)
                            w[u] = op_ld_relaxed(ws_rows + (int64_t)(j0 + u * G) * ER + c);
                }
            }
        }
        if (G > 1) {
            if (g < G && c < ER) s_ids[g * ER + c] = acc;   // the ids are no longer needed
        } else if (c < ER) {
            s_pre[c] = acc;
        }
    }
    if (wait_extra > 0 && b == nb - 1 && tid == 0) {
        const unsigned long long* spare = ws_rows + (int64_t)nb * ER;
        if (op_count_when_tagged(spare, op_ld_relaxed(spare), tag) < 0) ok = false;
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (tid == 0) {
            raise_status(status, MOEDC_ERR_TIMEOUT);
            atomicAdd(ws_generation, 1ull);   // the next launch starts from a fresh epoch
        }
        return;
    }
    if (G > 1) {
        for (int c = tid; c < ER; c += kOpThreads) {
            int acc = 0;
            for (int g = 0; g < G; ++g) acc += s_ids[g * ER + c];
            s_pre[c] = acc;
        }
        __syncthreads();
    }

    // 5. slots; totals from the last chunk
#pragma unroll
    for (int u = 0; u < EPT; ++u) {
        const int i = i0 + u * kWarp;
        if (i < n)
            __stcs(slot + (int64_t)t0 * K + i,
                   ((valid_bits >> u) & 1u) ? s_pre[e[u]] + my_wc[e[u]] + rank[u] : -1);
    }
    if (bad) raise_status(status, MOEDC_ERR_EXPERT_RANGE);
    if (b == nb - 1) {
        for (int c = tid; c < ER; c += kOpThreads) {
            const int total = s_pre[c] + s_cnt[c];
            if (c < E) {
                num_tokens_per_expert[c] = total;
                if (total > cap) raise_status(status, MOEDC_ERR_CAPACITY);
            } else {
                num_tokens_per_rank[c - E] = total;
            }
        }
        // every block has published (the last block read every row), so every
        // block has read the generation
        if (tid == 0) atomicAdd(ws_generation, 1ull);
    }
}

}  // namespace moedc

namespace moedc_host {

namespace {

// Host part of the epochs: consecutive per process from a clock-derived start.
std::atomic<unsigned long long> g_op_epoch{
    (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() *
    0xD1B54A32D192ED03ull};

// entries per thread, tokens per chunk and chunks of a shape, or false when
// the single pass does not take it (fewer than 4 chunks of 1024 entries: the
// sweep is faster; more than kOpMaxChunks even at 4 entries per thread)
struct OpPlan {
    int ept, tpc, chunks;
};

bool op_plan(int T, int K, OpPlan& p)
{
    if (T < 0 || K < 1) return false;
    for (int ept = 1; ept <= 4; ept *= 2) {
        const int tpc = moedc::kOpThreads * ept / K;
        const int64_t chunks = T > 0 ? ((int64_t)T + tpc - 1) / tpc : 1;
        if (ept == 1 && chunks < moedc::kOpMinChunks) return false;
        if (chunks <= moedc::kOpMaxChunks) {
            p = OpPlan{ept, tpc, (int)chunks};
            return true;
        }
    }
    return false;
}

size_t op_smem_bytes(int E, int R, int ept)
{
    return ((size_t)moedc::kOpWarps * (E + 1) + 2 * (size_t)(E + R) +
            (size_t)moedc::kOpThreads * ept) *
           sizeof(int32_t);
}

const void* op_kernel(int ept)
{
    return ept == 1   ? (const void*)moedc::layout_onepass_kernel<1>
           : ept == 2 ? (const void*)moedc::layout_onepass_kernel<2>
                      : (const void*)moedc::layout_onepass_kernel<4>;
}

constexpr int kOpMaxDevices = 64;
std::mutex g_op_smem_mutex;
bool g_op_smem_set[kOpMaxDevices] = {};

bool op_smem_ready()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kOpMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_op_smem_mutex);
    if (g_op_smem_set[dev]) return true;
    for (int ept = 1; ept <= 4; ept *= 2) {
        if (cudaFuncSetAttribute(op_kernel(ept), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)op_smem_bytes(MOEDC_MAX_E, MOEDC_MAX_E, ept)) !=
            cudaSuccess) {
            clear_stale_error();
            return false;
        }
    }
    g_op_smem_set[dev] = true;
    return true;
}

}  // namespace

// Workspace of the single-pass layout: the generation word (in a 256-byte
// header), then the chunks' rows of E + R tagged 64-bit counts, then one
// spare word (the test hook's wait target).  0 when the shape does not take
// this path.
size_t layout_onepass_workspace_bytes(int T, int K, int E, int R)
{
    OpPlan p;
    if (!op_plan(T, K, p)) return 0;
    return moedc::kOpHeaderBytes + ((size_t)p.chunks * (E + R) + 2) * sizeof(unsigned long long);
}

// MOEDC_ERR_UNIMPLEMENTED when the shape or the workspace does not take this path.
int launch_layout_onepass(const int32_t* topk_idx, int T, int K, int E, int R, int cap,
                          int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                          uint8_t* is_token_in_rank, int32_t* slot, void* workspace,
                          size_t workspace_bytes, int32_t* dev_status, cudaStream_t stream)
{
    const size_t need = layout_onepass_workspace_bytes(T, K, E, R);
    if (need == 0 || !workspace || workspace_bytes < need || !aligned(workspace, 16))
        return MOEDC_ERR_UNIMPLEMENTED;
    OpPlan plan;
    if (!op_plan(T, K, plan)) return MOEDC_ERR_UNIMPLEMENTED;
    const int tpc = plan.tpc;
    const int chunks = plan.chunks;
    const size_t sm = op_smem_bytes(E, R, plan.ept);
    // dynamic shared memory beyond the default 48 KB needs the kernel's limit
    // raised: once per device, to the largest size any shape needs
    if (sm > 48 * 1024 && !op_smem_ready()) return MOEDC_ERR_UNIMPLEMENTED;
    // the waits need every chunk's block resident at once
    if (chunks > resident_blocks(op_kernel(plan.ept), moedc::kOpThreads, sm))
        return MOEDC_ERR_UNIMPLEMENTED;

    char* ws = static_cast<char*>(workspace);
    auto* gen = reinterpret_cast<unsigned long long*>(ws);
    auto* rows = reinterpret_cast<unsigned long long*>(ws + moedc::kOpHeaderBytes);
    const unsigned long long host_epoch = g_op_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    const unsigned extra = test_wait_extra();

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)chunks);
    cfg.blockDim = dim3(moedc::kOpThreads);
    cfg.dynamicSmemBytes = sm;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = MOEDC_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    clear_stale_error();
#define MOEDC_OP_LAUNCH(P)                                                                      \
    cudaLaunchKernelEx(&cfg, moedc::layout_onepass_kernel<P>, topk_idx, T, K, E, R, cap, tpc,  \
                       num_tokens_per_expert, num_tokens_per_rank, is_token_in_rank, slot, gen, \
                       rows, host_epoch, extra, dev_status)
    const cudaError_t err = plan.ept == 1   ? MOEDC_OP_LAUNCH(1)
                            : plan.ept == 2 ? MOEDC_OP_LAUNCH(2)
                                            : MOEDC_OP_LAUNCH(4);
#undef MOEDC_OP_LAUNCH
    if (err == cudaErrorCooperativeLaunchTooLarge) {
        // fewer SMs than the device reports (a partitioned GPU): the sweep or the
        // two-kernel layout runs instead
        clear_stale_error();
        return MOEDC_ERR_UNIMPLEMENTED;
    }
    return err == cudaSuccess ? MOEDC_OK : MOEDC_ERR_CUDA;
}

}  // namespace moedc_host
