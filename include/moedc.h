/*
 * libmoedc — MoE expert-parallel token layout, dispatch and combine on one
 * GPU, with R "virtual ranks" that partition the expert dimension of a single
 * receive buffer (no inter-GPU transport).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  T tokens, H hidden channels, K routed experts per token, E experts,
 *  R virtual ranks (rank r owns experts [r*E/R, (r+1)*E/R); E % R == 0),
 *  cap slots per expert, G = H / 128 FP8 scale groups.
 *
 *  Every pointer is a DEVICE pointer owned by the caller.  The library never
 *  allocates, frees or synchronises.  Between calls it keeps only host-side
 *  caches (device attributes, occupancy) and a launch counter; the one
 *  environment variable it reads is a test hook of moedc_layout_dispatch.
 *  Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *  contain no host-side reads of device data.
 *
 *  Row-major layouts:
 *    x, y                 bf16   [T, H]
 *    topk_idx             int32  [T, K]   -1 = masked entry
 *    topk_weights         fp32   [T, K]
 *    slot                 int32  [T, K]   -1 = masked / dropped
 *    num_tokens_per_expert int32 [E]
 *    num_tokens_per_rank  int32  [R]
 *    is_token_in_rank     uint8  [T, R]   0 / 1
 *    recv, expert_out     bf16 or e4m3 [E, cap, H]   (expert-major)
 *    scales               fp32   [E, cap, G]  ([E, G, cap] or [E, cap] with
 *                                               the scale-layout flags below)
 *    src_idx              int32  [E, cap]
 *  x, y, recv and expert_out must be 16-byte aligned; the others 4-byte
 *  aligned (is_token_in_rank: any alignment).
 *
 * Errors
 * ------
 *  The return value reports argument errors found on the host (bad sizes,
 *  null or misaligned pointers, a workspace that is too small); nothing is
 *  launched when it is not MOEDC_OK.  MOEDC_ERR_CUDA means a launch failed.
 *  Errors that depend on the data are written to `dev_status`, a device int32
 *  the caller zeroes: each kernel raises it to max(*dev_status, code), so the
 *  word ends up holding the largest code met, independent of thread timing.
 *  A clean run leaves it untouched.
 *    MOEDC_ERR_EXPERT_RANGE  an index outside [-1, E); the entry is treated
 *                            as masked.
 *    MOEDC_ERR_CAPACITY      an expert received more than cap entries; the
 *                            slots still count on, and the entries whose slot
 *                            is >= cap are dropped by dispatch and combine.
 *    MOEDC_ERR_TIMEOUT       only from the cooperative single launch of
 *                            moedc_layout_dispatch: one of its two grid
 *                            barriers waited out its bound (>= 0.13 s, e.g.
 *                            when other work holds the SMs); its outputs are
 *                            then incomplete.  No other kernel waits on data
 *                            written by another block.
 *
 * Sources (page title, part of the page):
 *  [UCCL749]  UCCL PR #749 "[EP] Low-latency mode batch tokens per
 *             destination", code excerpt (per-expert routed-token counters,
 *             per-destination-rank token totals over the rank's experts).
 *  [DEEPEP693] DeepEP PR #693 "Pipeline direct NVLink dispatch with
 *             triple-buffered prefetch", Summary (token rows staged through
 *             shared memory; hidden data, scale factors and routing move
 *             together).
 *  [MORI614]  MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on
 *             MI300X + CX7": the notes on DispatchIntraNode's flat stride,
 *             CombineSync's (token, hidden slice) split, the MultiWarpIter
 *             512-element floor, block-local relay without grid barriers,
 *             the zero-copy combine input, the host view cache, and the
 *             negative sentinel expert.
 */
#ifndef MOEDC_H
#define MOEDC_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOEDC_API_VERSION 1

#if defined(__GNUC__)
#define MOEDC_EXPORT __attribute__((visibility("default")))
#else
#define MOEDC_EXPORT
#endif

typedef enum {
    MOEDC_OK = 0,
    MOEDC_ERR_ARG = 1,
    MOEDC_ERR_CAPACITY = 2,
    MOEDC_ERR_EXPERT_RANGE = 3,
    MOEDC_ERR_CUDA = 4,
    MOEDC_ERR_TIMEOUT = 5,
    MOEDC_ERR_UNIMPLEMENTED = 6
} moedc_status;

typedef enum { MOEDC_BF16 = 0, MOEDC_FP8_E4M3 = 1 } moedc_dtype;

/* OR-ed into the out_dtype of moedc_dispatch / moedc_layout_dispatch with
 * MOEDC_FP8_E4M3: the fp32 scales are stored [E][G][cap] (per expert, one
 * contiguous run of cap scales per 128-channel group, the order a grouped FP8
 * GEMM reads per K-block) instead of [E][cap][G].  Codes are unchanged. */
#define MOEDC_SCALES_COL_MAJOR 0x100

/* OR-ed into the out_dtype of moedc_dispatch / moedc_layout_dispatch with
 * MOEDC_FP8_E4M3 instead of MOEDC_SCALES_COL_MAJOR: one scale per token row
 * (the 128-channel rule with the group widened to all H channels), scales
 * [E][cap].  Also a scale_layout of moedc_dequant_e4m3 / moedc_combine_e4m3.
 * H <= MOEDC_TOKEN_SCALE_MAX_H with this flag. */
#define MOEDC_SCALES_PER_TOKEN 0x200
#define MOEDC_TOKEN_SCALE_MAX_H 32768

/* Limits checked on the host (MOEDC_ERR_ARG beyond them). */
#define MOEDC_MAX_K 32
#define MOEDC_MAX_E 1024

/* Version of this interface (MOEDC_API_VERSION of the build). */
MOEDC_EXPORT int moedc_api_version(void);

/* Static text for a status code; never NULL. */
MOEDC_EXPORT const char* moedc_strerror(int code);

/*
 * Bytes of device workspace for moedc_layout on this shape; also enough for
 * moedc_layout_dispatch to run as layout then dispatch.  The caller allocates
 * it (any 16-byte aligned device buffer of at least this size, no
 * initialisation needed) and may reuse it across calls that are ordered on
 * one stream; calls that can run at the same time need workspaces of their
 * own.  Up to T = 3 * floor(1024 / K) tokens (T * K = 3072 when K divides
 * 1024) the layout is one sweep launch that needs no workspace (the query
 * returns 0).  Beyond that it is a single pass over the routing table (one
 * cooperative launch) when it has a workspace of this size; up to 65536 entries the workspace is optional
 * (without it, NULL, the sweep runs), beyond 65536 it is required, and there
 * a smaller workspace that holds the two-kernel layout's counts is also
 * accepted (that layout then runs).  Results are identical on every path.
 * Returns 0 for arguments that the layout would reject.
 */
MOEDC_EXPORT size_t moedc_layout_workspace_bytes(int T, int K, int E, int R);

/*
 * Routing layout [UCCL749 code excerpt; MORI614 sentinel note].
 * Visiting entries (t, k) in ascending t, then k:
 *   slot[t][k]              = number of earlier entries routed to the same
 *                             expert (so each expert's slots run 0, 1, ... in
 *                             ascending source-token order); -1 if masked.
 *   num_tokens_per_expert[e] = entries routed to expert e.
 *   is_token_in_rank[t][r]  = 1 if any entry of token t goes to rank r.
 *   num_tokens_per_rank[r]  = number of distinct tokens with a 1 in column r.
 * Arguments: T >= 0, 1 <= K <= MOEDC_MAX_K, 1 <= E <= MOEDC_MAX_E,
 * 1 <= R <= E with E % R == 0, cap >= 1.  workspace may be NULL (or smaller
 * than moedc_layout_workspace_bytes()) when T * K <= 65536; beyond that it
 * must hold what one of the two layouts that use it needs (above).
 * Data errors (dev_status): MOEDC_ERR_EXPERT_RANGE, MOEDC_ERR_CAPACITY, and
 * MOEDC_ERR_TIMEOUT if a bounded wait of the single-pass layout gave up (its
 * outputs are then unspecified; the next call starts clean).
 */
MOEDC_EXPORT int moedc_layout(const int32_t* topk_idx, int T, int K, int E, int R, int cap,
                 int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                 uint8_t* is_token_in_rank, int32_t* slot,
                 void* workspace, size_t workspace_bytes,
                 int32_t* dev_status, cudaStream_t stream);

/*
 * moedc_layout for callers that cannot allocate device memory: no workspace
 * argument, the scratch lives in a fixed array inside the library.  The pages
 * have no counterpart to this entry point; it exists for hosts with no device
 * allocator of their own, plugins inside a framework whose memory pool owns
 * the GPU, and serving loops that may not call cudaMalloc after start-up.
 * Same arguments, results and data errors as moedc_layout, except:
 *  - shapes beyond 65536 entries whose scratch need exceeds
 *    MOEDC_STATIC_SCRATCH_BYTES on both layouts that use scratch return
 *    MOEDC_ERR_ARG and launch nothing (below that the sweep needs none);
 *  - the array (MOEDC_STATIC_SCRATCH_BYTES per device) stays resident on every
 *    GPU that loads the library until the process exits;
 *  - the first call on a device that uses the array (any shape for which
 *    moedc_layout_workspace_bytes is not 0) looks up its device address and
 *    caches it; make that first call before any stream capture begins;
 *  - all calls share the array, so calls that overlap on the GPU race and
 *    give wrong results: order them on one stream;
 *  - the cached address belongs to the device's current primary context: do
 *    not call cudaDeviceReset on a device after this entry point has run on
 *    it (the array is recreated at a new address and later calls would write
 *    through the stale one).
 * The call allocates nothing and calls no allocating routine.
 */
#define MOEDC_STATIC_SCRATCH_BYTES (1u << 20)
MOEDC_EXPORT int moedc_layout_static_scratch(const int32_t* topk_idx, int T, int K, int E,
                 int R, int cap, int32_t* num_tokens_per_expert,
                 int32_t* num_tokens_per_rank, uint8_t* is_token_in_rank, int32_t* slot,
                 int32_t* dev_status, cudaStream_t stream);

/*
 * Dispatch [DEEPEP693 Summary; MORI614 DispatchIntraNode note].
 * For every entry (t, k) with expert e in [0, E) and slot s in [0, cap):
 *   src_idx[e][s] = t
 *   MOEDC_BF16:     recv[e][s][:] = x[t][:]  (bit copy; recv is bf16)
 *   MOEDC_FP8_E4M3 (optionally | MOEDC_SCALES_COL_MAJOR, see above):
 *                   per group g of 128 channels, a = max |x[t][128g+i]|,
 *                   a = max(a, 1e-4f), sc = a / 448 (IEEE binary32 division),
 *                   recv[e][s][128g+i] = e4m3fn(x / sc) with one binary32
 *                   division and round-to-nearest-even, saturating to +-448;
 *                   scales[e][s][g] = sc.
 *   MOEDC_FP8_E4M3 | MOEDC_SCALES_PER_TOKEN: the same with a single group of
 *                   all H channels: a = max over the row, scales[e][s] = sc
 *                   ([E][cap]); H <= MOEDC_TOKEN_SCALE_MAX_H.
 * src_idx[e][s] = -1 for every s in [num_tokens_per_expert[e], cap).
 * Rows of recv / scales that no entry reaches are not written.
 * num_tokens_per_expert and slot are the outputs of moedc_layout for the same
 * topk_idx.  Arguments: T >= 0, H >= 8 with H % 8 == 0 (bf16) or
 * H % 128 == 0 (e4m3), K, E and cap as for moedc_layout; scales may be NULL
 * for MOEDC_BF16.
 * Data errors (dev_status): MOEDC_ERR_EXPERT_RANGE.
 */
MOEDC_EXPORT int moedc_dispatch(const void* x, int T, int H,
                   const int32_t* topk_idx, const int32_t* slot,
                   const int32_t* num_tokens_per_expert,
                   int K, int E, int cap, int out_dtype,
                   void* recv, float* scales, int32_t* src_idx,
                   int32_t* dev_status, cudaStream_t stream);

/*
 * Combine [MORI614 CombineSync and zero-copy combine input notes].
 *   y[t][h] = bf16_rne( sum over k = 0..K-1 ascending of
 *                       w[t][k] * float(expert_out[e][s][h]) )
 * with a binary32 accumulator that starts at +0, one rounded multiply and one
 * rounded add per term (never fused), skipping entries that are masked,
 * out of range, or have slot >= cap.  expert_out is read in place (bf16).
 * Arguments: T >= 0, H % 8 == 0, K, E and cap as for moedc_layout.
 * Data errors (dev_status): MOEDC_ERR_EXPERT_RANGE.
 */
MOEDC_EXPORT int moedc_combine(const void* expert_out, int E, int cap, int H,
                  const int32_t* topk_idx, const int32_t* slot,
                  const float* topk_weights, int T, int K,
                  void* y, int32_t* dev_status, cudaStream_t stream);

/*
 * e4m3 receive rows back to bf16 (the dequantisation q * s that pairs with
 * the e4m3 dispatch; used as the identity expert of a dispatch -> expert ->
 * combine round).  For every expert e, filled slot s < min(count[e], cap)
 * and channel h of group g = h / 128:
 *   out[e][s][h] = bf16_rne( float(recv[e][s][h]) * scales[e][s][g] )
 * with one binary32 multiply.  Rows past an expert's count are not written.
 * scale_layout: 0 for scales [E][cap][G], MOEDC_SCALES_COL_MAJOR for [E][G][cap],
 * MOEDC_SCALES_PER_TOKEN for one scale per row [E][cap] (every g uses it).
 * recv and out must be 16-byte aligned; H % 128 == 0.  No data errors.
 */
MOEDC_EXPORT int moedc_dequant_e4m3(const void* recv, const float* scales, int scale_layout,
                 const int32_t* num_tokens_per_expert, int E, int cap, int H,
                 void* out_bf16, cudaStream_t stream);

/*
 * Combine from e4m3 expert outputs with fp32 scales (the formats dispatch
 * produces; scale_layout as for moedc_dequant_e4m3, scale(e, s, g) being
 * scales[e][s] for every g with MOEDC_SCALES_PER_TOKEN):
 *   y[t][h] = bf16_rne( sum over k ascending of
 *                       w[t][k] * (float(expert_out[e][s][h]) * scale(e, s, h/128)) )
 * binary32 accumulator from +0, each product rounded, never fused; masked,
 * out-of-range and dropped entries skipped.  Reads 1 byte per element
 * instead of 2.  expert_out and y 16-byte aligned, H % 128 == 0.
 * Data errors (dev_status): MOEDC_ERR_EXPERT_RANGE.
 */
MOEDC_EXPORT int moedc_combine_e4m3(const void* expert_out, const float* expert_scales,
                 int scale_layout, int E, int cap, int H, const int32_t* topk_idx,
                 const int32_t* slot, const float* topk_weights, int T, int K, void* y,
                 int32_t* dev_status, cudaStream_t stream);

/*
 * Rank-major packed receive [UCCL749 title: tokens batched per destination].
 * A token goes to a rank once, however many of its experts live there, into
 * that rank's contiguous buffer of cap_rank rows.
 *
 * moedc_rank_layout: for each rank r, in ascending token order,
 *   rank_slot[t][r] = number of earlier tokens with is_token_in_rank[.][r] = 1,
 *                     when is_token_in_rank[t][r] = 1; -1 otherwise.
 *   Data error (dev_status): MOEDC_ERR_CAPACITY when a rank receives more than
 *   cap_rank tokens (slots keep counting; rows at slot >= cap_rank are dropped).
 *   is_token_in_rank and num_tokens_per_rank come from moedc_layout.
 *
 * moedc_rank_dispatch: for each (t, r) with j = rank_slot[t][r] in [0, cap_rank):
 *   rank_src_idx[r][j] = t; recv_rank[r][j][:] = x[t][:] (MOEDC_BF16), or the
 *   e4m3 codes and per-128 fp32 scales of x[t] by the moedc_dispatch rule
 *   (MOEDC_FP8_E4M3, scales_rank [R, cap_rank, H/128]; the scale-layout
 *   flags are not offered here: MOEDC_ERR_ARG).  rank_src_idx = -1
 *   for j in [num_tokens_per_rank[r], cap_rank); other rows are not written.
 *
 * moedc_rank_combine: each rank returns one bf16 partial row per received
 *   token (rank_out [R, cap_rank, H], the weighted sum over the token's
 *   experts on that rank, formed on the expert side), and
 *     y[t][h] = bf16_rne( sum over r ascending of float(rank_out[r][j][h]) )
 *   over the ranks with j = rank_slot[t][r] in [0, cap_rank), binary32
 *   accumulator from +0.  A token in no rank gives +0.
 * Arguments: T >= 0, 1 <= R <= MOEDC_MAX_E, cap_rank >= 1; H as for
 * moedc_dispatch / moedc_combine; x, recv_rank, rank_out, y 16-byte aligned.
 */
MOEDC_EXPORT int moedc_rank_layout(const uint8_t* is_token_in_rank, int T, int R, int cap_rank,
                 int32_t* rank_slot, int32_t* dev_status, cudaStream_t stream);
MOEDC_EXPORT int moedc_rank_dispatch(const void* x, int T, int H, const int32_t* rank_slot,
                 const int32_t* num_tokens_per_rank, int R, int cap_rank, int out_dtype,
                 void* recv_rank, float* scales_rank, int32_t* rank_src_idx,
                 cudaStream_t stream);
MOEDC_EXPORT int moedc_rank_combine(const void* rank_out, int R, int cap_rank, int H,
                 const int32_t* rank_slot, int T, void* y, cudaStream_t stream);

/*
 * Layout followed by dispatch, with the outputs of both calls
 * [MORI614 notes on low token counts: host enqueue and idle warps dominate].
 * For T * K <= MOEDC_FUSED_MAX_ENTRIES this is ONE kernel launch: every
 * thread block rebuilds the layout in shared memory (no inter-block
 * synchronisation), the blocks split the (token, 512-channel slice) copies,
 * and each layout output is written by the warp that owns it (a token's slots
 * and rank flags by the warp copying its first slice, a rank's count by one
 * warp, the expert counts by block 0).
 * With MOEDC_SCALES_PER_TOKEN (a row's scale needs all of its slices) the
 * single launch gives each block whole tokens instead.
 *
 * Beyond 65536 entries, with a workspace of at least
 * moedc_layout_dispatch_workspace_bytes(T, K, E, R) bytes, it is also ONE
 * launch, a cooperative one [UCCL749 per-expert counts a rank waits on]:
 * each block ranks and counts a contiguous chunk of tokens; a grid barrier;
 * one block per expert / rank scans the chunks' counts; a second barrier;
 * then each block assigns its chunk's slots and copies its chunk.  The
 * barriers are bounded waits (MOEDC_ERR_TIMEOUT when one runs out).  The
 * workspace needs no initialisation but must not be shared by calls that can
 * run at the same time.
 *
 * Everything else runs as moedc_layout then moedc_dispatch: 1024 < T * K <=
 * 65536 (where that is the faster form), a workspace smaller than
 * moedc_layout_dispatch_workspace_bytes (when T * K > 65536 it must still hold
 * the two-kernel layout's counts), a chunk that would exceed
 * 2048 entries, and MOEDC_SCALES_PER_TOKEN beyond 1024 entries.  Results are
 * identical on every path.
 *
 * The barriers' bounded waits are tested through moedc_test_set_wait_extra
 * (below), never through the environment.
 */
#define MOEDC_FUSED_MAX_ENTRIES 1024
MOEDC_EXPORT size_t moedc_layout_dispatch_workspace_bytes(int T, int K, int E, int R);
MOEDC_EXPORT int moedc_layout_dispatch(const void* x, const int32_t* topk_idx,
                          int T, int H, int K, int E, int R, int cap, int out_dtype,
                          int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                          uint8_t* is_token_in_rank, int32_t* slot,
                          void* recv, float* scales, int32_t* src_idx,
                          void* workspace, size_t workspace_bytes,
                          int32_t* dev_status, cudaStream_t stream);

/*
 * Test hook, not for production use.  With extra_arrivals = n > 0, every
 * later bounded wait of the library waits for something that never comes:
 * the cooperative launch of moedc_layout_dispatch makes its grid barriers
 * wait for n blocks more than the grid has, and the single-pass layout's
 * last block also waits for the flag of a chunk that does not exist.  Each
 * such wait runs out and the call reports MOEDC_ERR_TIMEOUT on its device
 * status; 0 (the initial value) restores normal waits.  Process-wide, read
 * once per call on the host (no environment lookup); it exists so that a
 * test can drive the timeout paths without a fault.
 */
MOEDC_EXPORT void moedc_test_set_wait_extra(unsigned extra_arrivals);

#ifdef __cplusplus
}
#endif

#endif /* MOEDC_H */
