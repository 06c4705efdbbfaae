/*
 * CPU oracle for MoE expert-parallel layout, dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * restatement of what the GPU library computes.  Only the test suite, the
 * package's smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (no fused multiply-add, IEEE single precision for every float operation).
 *
 * Sources (page title, part of the page):
 *  - UCCL PR #749 "[EP] Low-latency mode batch tokens per destination",
 *    code excerpt: a per-expert routed-token counter (atomic_counter_per_expert)
 *    and a per-destination-rank token total built from the counts of the
 *    rank's local experts (rank = expert / num_local_experts).
 *  - MORI PR #614 "perf(ep): InterNodeV1LL low-token latency on MI300X + CX7",
 *    routing-scan note: a negative (masked) expert id takes part in nothing.
 *  - DeepEP PR #693 "Pipeline direct NVLink dispatch with triple-buffered
 *    prefetch", Summary: FP8 dispatch carries per-token scale factors with the
 *    hidden payload.
 * The exact arithmetic (slot order, the FP8 scale rule, combine order) is the
 * method's stated definition; the pages print no formula for it.  Readings
 * where the pages are silent are listed in the design notes of the project.
 *
 * Parity pins: every function here is checked by CPU tests against brute
 * force, library routines (torch's bf16 / float8_e4m3fn casts) or closed forms.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* status codes of the library contract (restated here, not included) */
enum { ORACLE_OK = 0, ORACLE_ERR_CAPACITY = 2, ORACLE_ERR_EXPERT_RANGE = 3 };

static int raise_status(int cur, int code) { return code > cur ? code : cur; }

/* ------------------------------------------------------------------ bf16 */

/* bf16 is the upper half of an IEEE binary32 pattern. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even; NaN stays a quiet NaN. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)           /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xffffu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;                                /* carries into the exponent */
    return (uint16_t)upper;
}

/* --------------------------------------------------------------- e4m3fn */
/*
 * OCP 8-bit floating point, E4M3 flavour without infinities ("e4m3fn"):
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.  Exponent field 0
 * holds subnormals m * 2^-9; field 1..15 holds (8 + m) * 2^(field - 10); the
 * single pattern S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448.
 */
float oracle_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int ef = (c >> 3) & 0xf;
    int m = c & 7;
    double v;
    if (ef == 15 && m == 7)
        return sign ? -NAN : NAN;
    if (ef == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), ef - 10);
    return (float)(sign ? -v : v);
}

/* round a non-negative double that is an exact multiple of 1/2 or finer to
   the nearest integer, ties to even */
static double round_half_even(double q)
{
    double fl = floor(q);
    double d = q - fl;
    if (d > 0.5)
        return fl + 1.0;
    if (d < 0.5)
        return fl;
    return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

/*
 * Nearest e4m3fn value to v, ties to even, with saturation: any magnitude
 * beyond 448 becomes +-448 ("satfinite").  NaN -> 0x7f.  -0 -> 0x80.
 */
uint8_t oracle_e4m3_encode(float v)
{
    if (isnan(v))
        return 0x7f;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a > 448.0)
        return (uint8_t)(sign | 0x7e);
    if (a == 0.0)
        return sign;
    int ex;
    frexp(a, &ex);            /* a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1 */
    int e = ex - 1;
    if (e < -6) {
        /* subnormal range: quantum 2^-9, n in [0, 8]; n = 8 is the smallest normal */
        double n = round_half_even(ldexp(a, 9));
        return (uint8_t)(sign | (uint8_t)n);
    }
    /* normal: quantum 2^(e-3), n in [8, 16]; n = 16 carries into the next binade */
    double n = round_half_even(ldexp(a, 3 - e));
    int code = ((e + 7) << 3) + ((int)n - 8);
    return (uint8_t)(sign | code);
}

void oracle_e4m3_encode_n(const float* v, uint8_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e4m3_decode_n(const uint8_t* c, float* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

void oracle_f32_to_bf16_n(const float* v, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16(v[i]);
}

/* --------------------------------------------------------------- layout */
/*
 * Routing layout.  For entries (t, k) visited in ascending t, then k:
 *   e = topk_idx[t][k]; e == -1 is masked; e < -1 or e >= E is out of range
 *   (treated as masked, and the status reports it).
 *   slot[t][k] = number of earlier entries routed to e (ascending token order
 *                inside each expert), -1 for masked / out-of-range entries.
 *   num_tokens_per_expert[e] = number of entries routed to e.
 *   is_token_in_rank[t][r] = 1 when any of token t's entries goes to an
 *                expert of rank r = e / (E / R); rank r owns a contiguous run
 *                of E / R experts.
 *   num_tokens_per_rank[r] = number of distinct tokens with
 *                is_token_in_rank[t][r] = 1.
 * Returns the largest error code met: EXPERT_RANGE for a bad id, CAPACITY
 * when some expert receives more than `cap` entries (slots still count on).
 */
int oracle_layout(const int32_t* topk_idx, int T, int K, int E, int R, int cap,
                  int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                  uint8_t* is_token_in_rank, int32_t* slot)
{
    int status = ORACLE_OK;
    int epr = E / R;
    for (int e = 0; e < E; ++e)
        num_tokens_per_expert[e] = 0;
    for (int r = 0; r < R; ++r)
        num_tokens_per_rank[r] = 0;
    for (int64_t i = 0; i < (int64_t)T * R; ++i)
        is_token_in_rank[i] = 0;

    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[(int64_t)t * K + k];
            if (e == -1) {
                slot[(int64_t)t * K + k] = -1;
                continue;
            }
            if (e < -1 || e >= E) {
                slot[(int64_t)t * K + k] = -1;
                status = raise_status(status, ORACLE_ERR_EXPERT_RANGE);
                continue;
            }
            slot[(int64_t)t * K + k] = num_tokens_per_expert[e];
            num_tokens_per_expert[e] += 1;
            is_token_in_rank[(int64_t)t * R + e / epr] = 1;
        }
    }
    for (int t = 0; t < T; ++t)
        for (int r = 0; r < R; ++r)
            num_tokens_per_rank[r] += is_token_in_rank[(int64_t)t * R + r];
    for (int e = 0; e < E; ++e)
        if (num_tokens_per_expert[e] > cap)
            status = raise_status(status, ORACLE_ERR_CAPACITY);
    return status;
}

/* ------------------------------------------------------------- dispatch */

static int entry_valid(int e, int s, int E, int cap)
{
    return e >= 0 && e < E && s >= 0 && s < cap;
}

/*
 * Dispatch.  src_idx[E][cap] starts at -1 everywhere; for each valid entry
 * (t, k) with expert e and slot s < cap:
 *   src_idx[e][s] = t
 *   bf16 (fp8 == 0): recv[e][s][:] = x[t][:], a bit copy.
 *   e4m3 (fp8 != 0), per group g of 128 channels:
 *     a = max_i |x[t][128g + i]|           (exact)
 *     a = fmaxf(a, 1e-4f)
 *     s = a / 448.0f                         (one IEEE binary32 division)
 *     recv[e][s][128g + i] = e4m3(x / s)     (binary32 division, then the
 *                                              satfinite nearest-even encode)
 *     scales[e][s][g] = s
 * Rows of recv / scales with no entry are left untouched.
 * Returns EXPERT_RANGE if an entry names an expert outside [-1, E).
 */
int oracle_dispatch(const uint16_t* x, int T, int H, const int32_t* topk_idx,
                    const int32_t* slot, int K, int E, int cap, int fp8,
                    void* recv, float* scales, int32_t* src_idx)
{
    int status = ORACLE_OK;
    int G = H / 128;
    for (int64_t i = 0; i < (int64_t)E * cap; ++i)
        src_idx[i] = -1;
    for (int t = 0; t < T; ++t) {
        const uint16_t* xr = x + (int64_t)t * H;
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[(int64_t)t * K + k];
            int s = slot[(int64_t)t * K + k];
            if (e < -1 || e >= E)
                status = raise_status(status, ORACLE_ERR_EXPERT_RANGE);
            if (!entry_valid(e, s, E, cap))
                continue;
            int64_t row = (int64_t)e * cap + s;
            src_idx[row] = t;
            if (!fp8) {
                uint16_t* dst = (uint16_t*)recv + row * H;
                for (int h = 0; h < H; ++h)
                    dst[h] = xr[h];
                continue;
            }
            uint8_t* dst = (uint8_t*)recv + row * H;
            for (int g = 0; g < G; ++g) {
                float amax = 0.0f;
                for (int i = 0; i < 128; ++i) {
                    float v = fabsf(oracle_bf16_to_f32(xr[128 * g + i]));
                    if (v > amax)
                        amax = v;
                }
                amax = fmaxf(amax, 1e-4f);
                float scale = amax / 448.0f;
                for (int i = 0; i < 128; ++i) {
                    float q = oracle_bf16_to_f32(xr[128 * g + i]) / scale;
                    dst[128 * g + i] = oracle_e4m3_encode(q);
                }
                scales[row * G + g] = scale;
            }
        }
    }
    return status;
}

/*
 * Dispatch with one e4m3 scale per token row.  The rule is the per-128
 * rule above with the group widened to the whole row of H channels:
 *   a = max_h |x[t][h]|                      (exact)
 *   a = fmaxf(a, 1e-4f)
 *   s = a / 448.0f                             (one IEEE binary32 division)
 *   recv[e][s][h] = e4m3(x[t][h] / s)          (binary32 division, then the
 *                                               satfinite nearest-even encode)
 *   scales[e][s] = s                           (scales is [E][cap])
 * src_idx and the untouched rows as in oracle_dispatch.
 */
int oracle_dispatch_token_scale(const uint16_t* x, int T, int H, const int32_t* topk_idx,
                                const int32_t* slot, int K, int E, int cap,
                                uint8_t* recv, float* scales, int32_t* src_idx)
{
    int status = ORACLE_OK;
    for (int64_t i = 0; i < (int64_t)E * cap; ++i)
        src_idx[i] = -1;
    for (int t = 0; t < T; ++t) {
        const uint16_t* xr = x + (int64_t)t * H;
        float amax = 0.0f;
        for (int h = 0; h < H; ++h) {
            float v = fabsf(oracle_bf16_to_f32(xr[h]));
            if (v > amax)
                amax = v;
        }
        amax = fmaxf(amax, 1e-4f);
        float scale = amax / 448.0f;
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[(int64_t)t * K + k];
            int s = slot[(int64_t)t * K + k];
            if (e < -1 || e >= E)
                status = raise_status(status, ORACLE_ERR_EXPERT_RANGE);
            if (!entry_valid(e, s, E, cap))
                continue;
            int64_t row = (int64_t)e * cap + s;
            src_idx[row] = t;
            for (int h = 0; h < H; ++h)
                recv[row * H + h] = oracle_e4m3_encode(oracle_bf16_to_f32(xr[h]) / scale);
            scales[row] = scale;
        }
    }
    return status;
}

/* -------------------------------------------------------------- combine */
/*
 * Combine.  For every token t and channel h:
 *   acc = 0.0f
 *   for k = 0 .. K-1 (ascending), skipping masked / out-of-range entries and
 *   slots >= cap:
 *       p   = w[t][k] * float(expert_out[e][s][h])     (binary32 multiply)
 *       acc = acc + p                                   (binary32 add)
 *   y[t][h] = bf16(acc), nearest even.  A token with no valid entry gives +0.
 * Returns EXPERT_RANGE if an entry names an expert outside [-1, E).
 */
int oracle_combine(const uint16_t* expert_out, int E, int cap, int H,
                   const int32_t* topk_idx, const int32_t* slot, const float* topk_weights,
                   int T, int K, uint16_t* y)
{
    int status = ORACLE_OK;
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[(int64_t)t * K + k];
            if (e < -1 || e >= E)
                status = raise_status(status, ORACLE_ERR_EXPERT_RANGE);
        }
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int e = topk_idx[(int64_t)t * K + k];
                int s = slot[(int64_t)t * K + k];
                if (!entry_valid(e, s, E, cap))
                    continue;
                float v = oracle_bf16_to_f32(expert_out[((int64_t)e * cap + s) * H + h]);
                float p = topk_weights[(int64_t)t * K + k] * v;
                acc = acc + p;
            }
            y[(int64_t)t * H + h] = oracle_f32_to_bf16(acc);
        }
    }
    return status;
}

/* ------------------------------------------------------------- dequant */
/*
 * e4m3 receive rows back to bf16 (the "identity expert" of a dispatch ->
 * expert -> combine round): for every expert e and filled slot
 * s < min(num_tokens_per_expert[e], cap), channel h of group g = h / 128:
 *   p = decode(recv[e][s][h]) * scales[e][s][g]     (binary32 multiply)
 *   out[e][s][h] = bf16(p), nearest even.
 * Rows past an expert's count are left untouched.
 */
void oracle_dequant_e4m3(const uint8_t* recv, const float* scales,
                         const int32_t* num_tokens_per_expert, int E, int cap, int H,
                         uint16_t* out)
{
    int G = H / 128;
    for (int e = 0; e < E; ++e) {
        int filled = num_tokens_per_expert[e] < cap ? num_tokens_per_expert[e] : cap;
        for (int s = 0; s < filled; ++s) {
            int64_t row = (int64_t)e * cap + s;
            for (int h = 0; h < H; ++h) {
                float v = oracle_e4m3_decode(recv[row * H + h]);
                float p = v * scales[row * G + h / 128];
                out[row * H + h] = oracle_f32_to_bf16(p);
            }
        }
    }
}

/* the same with one scale per row (scales [E][cap]): p = decode(q) * scales[e][s] */
void oracle_dequant_e4m3_token(const uint8_t* recv, const float* scales,
                               const int32_t* num_tokens_per_expert, int E, int cap, int H,
                               uint16_t* out)
{
    for (int e = 0; e < E; ++e) {
        int filled = num_tokens_per_expert[e] < cap ? num_tokens_per_expert[e] : cap;
        for (int s = 0; s < filled; ++s) {
            int64_t row = (int64_t)e * cap + s;
            for (int h = 0; h < H; ++h) {
                float p = oracle_e4m3_decode(recv[row * H + h]) * scales[row];
                out[row * H + h] = oracle_f32_to_bf16(p);
            }
        }
    }
}

/* ------------------------------------------------ rank-major packed receive */
/*
 * Batching tokens per destination rank (UCCL PR #749, "[EP] Low-latency mode
 * batch tokens per destination"): a token goes to a rank once, however many
 * of its experts live there.
 *
 * Rank layout: for each rank r, visiting tokens in ascending t,
 *   rank_slot[t][r] = number of earlier tokens t' < t with
 *                     is_token_in_rank[t'][r] = 1, when is_token_in_rank[t][r]
 *                     is 1; -1 otherwise.
 * Returns CAPACITY when some rank receives more than cap_rank tokens (the
 * slots keep counting, rows at slot >= cap_rank are dropped downstream).
 */
int oracle_rank_layout(const uint8_t* is_token_in_rank, int T, int R, int cap_rank,
                       int32_t* rank_slot)
{
    int status = ORACLE_OK;
    for (int r = 0; r < R; ++r) {
        int count = 0;
        for (int t = 0; t < T; ++t) {
            if (is_token_in_rank[(int64_t)t * R + r]) {
                rank_slot[(int64_t)t * R + r] = count;
                count += 1;
            } else {
                rank_slot[(int64_t)t * R + r] = -1;
            }
        }
        if (count > cap_rank)
            status = raise_status(status, ORACLE_ERR_CAPACITY);
    }
    return status;
}

/*
 * Rank dispatch: rank_src_idx[R][cap_rank] starts at -1; for each (t, r) with
 * slot j = rank_slot[t][r] in [0, cap_rank):
 *   rank_src_idx[r][j] = t
 *   bf16: recv_rank[r][j][:] = x[t][:]
 *   e4m3: per group g of 128 channels the same rule as expert dispatch:
 *         a = max |x|, a = fmaxf(a, 1e-4f), s = a / 448.0f, codes = e4m3(x / s),
 *         scales_rank[r][j][g] = s.
 */
void oracle_rank_dispatch(const uint16_t* x, int T, int H, const int32_t* rank_slot, int R,
                          int cap_rank, int fp8, void* recv_rank, float* scales_rank,
                          int32_t* rank_src_idx)
{
    int G = H / 128;
    for (int64_t i = 0; i < (int64_t)R * cap_rank; ++i)
        rank_src_idx[i] = -1;
    for (int t = 0; t < T; ++t) {
        const uint16_t* xr = x + (int64_t)t * H;
        for (int r = 0; r < R; ++r) {
            int j = rank_slot[(int64_t)t * R + r];
            if (j < 0 || j >= cap_rank)
                continue;
            int64_t row = (int64_t)r * cap_rank + j;
            rank_src_idx[row] = t;
            if (!fp8) {
                uint16_t* dst = (uint16_t*)recv_rank + row * H;
                for (int h = 0; h < H; ++h)
                    dst[h] = xr[h];
                continue;
            }
            uint8_t* dst = (uint8_t*)recv_rank + row * H;
            for (int g = 0; g < G; ++g) {
                float amax = 0.0f;
                for (int i = 0; i < 128; ++i) {
                    float v = fabsf(oracle_bf16_to_f32(xr[128 * g + i]));
                    if (v > amax)
                        amax = v;
                }
                amax = fmaxf(amax, 1e-4f);
                float scale = amax / 448.0f;
                for (int i = 0; i < 128; ++i)
                    dst[128 * g + i] = oracle_e4m3_encode(oracle_bf16_to_f32(xr[128 * g + i]) / scale);
                scales_rank[row * G + g] = scale;
            }
        }
    }
}

/*
 * Rank combine: each rank returns one partial row per (token, rank) - the
 * weighted sum over the token's experts on that rank, formed on the expert
 * side - and
 *   y[t][h] = bf16( sum over r = 0..R-1 ascending of float(rank_out[r][j][h]) )
 * over the ranks with j = rank_slot[t][r] in [0, cap_rank), binary32
 * accumulator from +0, one rounded add per rank.  A token in no rank gives +0.
 */
void oracle_rank_combine(const uint16_t* rank_out, int R, int cap_rank, int H,
                         const int32_t* rank_slot, int T, uint16_t* y)
{
    for (int t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int r = 0; r < R; ++r) {
                int j = rank_slot[(int64_t)t * R + r];
                if (j < 0 || j >= cap_rank)
                    continue;
                acc = acc + oracle_bf16_to_f32(rank_out[((int64_t)r * cap_rank + j) * H + h]);
            }
            y[(int64_t)t * H + h] = oracle_f32_to_bf16(acc);
        }
    }
}

/* -------------------------------------------------------- e4m3 combine */
/*
 * Combine from e4m3 expert outputs with fp32 scales.  scale_mode 0: one scale
 * per 128 channels, row-major [E][cap][G]; 1: the same column-major
 * [E][G][cap]; 2: one scale per row, [E][cap].
 * For every token t and channel h, group g = h / 128:
 *   acc = 0.0f
 *   for k = 0 .. K-1 ascending, skipping masked / out-of-range / dropped entries:
 *       v   = decode(q[e][s][h]) * scale(e, s, g)    (binary32 multiply)
 *       p   = w[t][k] * v                            (binary32 multiply)
 *       acc = acc + p                                (binary32 add)
 *   y[t][h] = bf16(acc), nearest even.
 */
int oracle_combine_e4m3(const uint8_t* expert_out, const float* expert_scales, int scale_mode,
                        int E, int cap, int H, const int32_t* topk_idx, const int32_t* slot,
                        const float* topk_weights, int T, int K, uint16_t* y)
{
    int status = ORACLE_OK;
    int G = H / 128;
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int e = topk_idx[(int64_t)t * K + k];
            if (e < -1 || e >= E)
                status = raise_status(status, ORACLE_ERR_EXPERT_RANGE);
        }
        for (int h = 0; h < H; ++h) {
            float acc = 0.0f;
            int g = h / 128;
            for (int k = 0; k < K; ++k) {
                int e = topk_idx[(int64_t)t * K + k];
                int s = slot[(int64_t)t * K + k];
                if (!entry_valid(e, s, E, cap))
                    continue;
                int64_t row = (int64_t)e * cap + s;
                float sc = scale_mode == 2   ? expert_scales[row]
                           : scale_mode == 1 ? expert_scales[((int64_t)e * G + g) * cap + s]
                                             : expert_scales[row * G + g];
                float v = oracle_e4m3_decode(expert_out[row * H + h]) * sc;
                float p = topk_weights[(int64_t)t * K + k] * v;
                acc = acc + p;
            }
            y[(int64_t)t * H + h] = oracle_f32_to_bf16(acc);
        }
    }
    return status;
}
