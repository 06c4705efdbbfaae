/*
 * A plain C11 caller of libmoedc: no Python, no C++, no torch.  It allocates
 * device buffers with the CUDA runtime, runs layout -> bf16 dispatch ->
 * combine for one routing entry per token with weight 1 (so combine returns
 * x bit for bit) and then a top-4 e4m3 dispatch, and checks on the host:
 *   - the expert counts sum to the routed entries and each expert's slots are
 *     0, 1, ... in ascending token order;
 *   - src_idx inverts slot and is -1 past each expert's count;
 *   - y equals x exactly (K = 1, w = 1);
 *   - every e4m3 scale is positive and the status word stays clean.
 * Exit status 0 when all hold.  Build: gcc -std=c11 moe_round.c -lmoedc -lcudart
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moedc.h"

#define CHECK(cond, msg)                                              \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "moe_round: %s (line %d)\n", msg, __LINE__); \
            return 1;                                                 \
        }                                                             \
    } while (0)

static uint32_t lcg(uint32_t* s)
{
    *s = *s * 1664525u + 1013904223u;
    return *s >> 8;
}

static void* dev_alloc(size_t bytes)
{
    void* p = NULL;
    return cudaMalloc(&p, bytes) == cudaSuccess ? p : NULL;
}

int main(void)
{
    enum { T = 300, H = 256, E = 16, R = 4, K4 = 4 };
    uint32_t seed = 12345u;
    CHECK(moedc_api_version() == MOEDC_API_VERSION, "api version");

    /* inputs: bf16 bit patterns of small integers, one expert per token */
    uint16_t* hx = malloc((size_t)T * H * sizeof(uint16_t));
    int32_t hidx[T];
    float hw[T];
    int32_t count[E];
    memset(count, 0, sizeof(count));
    for (int i = 0; i < T * H; ++i) hx[i] = (uint16_t)(0x3f80u + (lcg(&seed) & 0x7fu));
    for (int t = 0; t < T; ++t) {
        hidx[t] = (int32_t)(lcg(&seed) % E);
        hw[t] = 1.0f;
        count[hidx[t]]++;
    }
    int cap = 0;
    for (int e = 0; e < E; ++e) cap = count[e] > cap ? count[e] : cap;

    void* x = dev_alloc((size_t)T * H * 2);
    int32_t* idx = dev_alloc(sizeof(hidx));
    float* w = dev_alloc(sizeof(hw));
    int32_t* cnt = dev_alloc(E * 4);
    int32_t* rk = dev_alloc(R * 4);
    uint8_t* inr = dev_alloc((size_t)T * R);
    int32_t* slot = dev_alloc(T * 4);
    void* recv = dev_alloc((size_t)E * cap * H * 2);
    int32_t* src = dev_alloc((size_t)E * cap * 4);
    void* y = dev_alloc((size_t)T * H * 2);
    int32_t* status = dev_alloc(4);
    CHECK(x && idx && w && cnt && rk && inr && slot && recv && src && y && status, "cudaMalloc");
    CHECK(cudaMemcpy(x, hx, (size_t)T * H * 2, cudaMemcpyHostToDevice) == cudaSuccess, "copy x");
    CHECK(cudaMemcpy(idx, hidx, sizeof(hidx), cudaMemcpyHostToDevice) == cudaSuccess, "copy idx");
    CHECK(cudaMemcpy(w, hw, sizeof(hw), cudaMemcpyHostToDevice) == cudaSuccess, "copy w");
    CHECK(cudaMemset(status, 0, 4) == cudaSuccess, "zero status");

    /* the layout's workspace, when the shape asks for one (not at this size) */
    const size_t wsb = moedc_layout_workspace_bytes(T, 1, E, R);
    void* ws = NULL;
    if (wsb > 0) {
        ws = dev_alloc(wsb);
        CHECK(ws != NULL, "cudaMalloc workspace");
    }
    CHECK(moedc_layout(idx, T, 1, E, R, cap, cnt, rk, inr, slot, ws, wsb, status, 0) == MOEDC_OK,
          "moedc_layout");
    CHECK(moedc_dispatch(x, T, H, idx, slot, cnt, 1, E, cap, MOEDC_BF16, recv, NULL, src, status,
                         0) == MOEDC_OK,
          "moedc_dispatch");
    CHECK(moedc_combine(recv, E, cap, H, idx, slot, w, T, 1, y, status, 0) == MOEDC_OK,
          "moedc_combine");
    /* a host-detectable argument error launches nothing */
    CHECK(moedc_combine(recv, E, cap, H + 1, idx, slot, w, T, 1, y, status, 0) == MOEDC_ERR_ARG,
          "argument check");
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "synchronise");

    int32_t hcnt[E], hslot[T], hst = -1;
    int32_t* hsrc = malloc((size_t)E * cap * 4);
    uint16_t* hy = malloc((size_t)T * H * 2);
    CHECK(cudaMemcpy(hcnt, cnt, sizeof(hcnt), cudaMemcpyDeviceToHost) == cudaSuccess, "cnt");
    CHECK(cudaMemcpy(hslot, slot, sizeof(hslot), cudaMemcpyDeviceToHost) == cudaSuccess, "slot");
    CHECK(cudaMemcpy(hsrc, src, (size_t)E * cap * 4, cudaMemcpyDeviceToHost) == cudaSuccess, "src");
    CHECK(cudaMemcpy(hy, y, (size_t)T * H * 2, cudaMemcpyDeviceToHost) == cudaSuccess, "y");
    CHECK(cudaMemcpy(&hst, status, 4, cudaMemcpyDeviceToHost) == cudaSuccess, "status");
    CHECK(hst == MOEDC_OK, "status word clean");
    int next[E];
    int total = 0;
    memset(next, 0, sizeof(next));
    for (int e = 0; e < E; ++e) {
        CHECK(hcnt[e] == count[e], "expert count");
        total += hcnt[e];
    }
    CHECK(total == T, "counts sum to the routed entries");
    for (int t = 0; t < T; ++t) {   /* ascending slots per expert, in token order */
        const int e = hidx[t];
        CHECK(hslot[t] == next[e], "slot order");
        CHECK(hsrc[e * cap + hslot[t]] == t, "src_idx inverts slot");
        next[e]++;
    }
    for (int e = 0; e < E; ++e)
        for (int s = hcnt[e]; s < cap; ++s) CHECK(hsrc[e * cap + s] == -1, "unfilled src_idx");
    CHECK(memcmp(hy, hx, (size_t)T * H * 2) == 0, "K = 1, w = 1 combine returns x exactly");

    /* top-4 of 16 with e4m3 codes and per-128 scales, through the one-call entry */
    int32_t* hidx4 = malloc((size_t)T * K4 * 4);
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K4; ++k) hidx4[t * K4 + k] = (int32_t)((t + 5 * k) % E);
    int32_t* idx4 = dev_alloc((size_t)T * K4 * 4);
    int32_t* slot4 = dev_alloc((size_t)T * K4 * 4);
    const int cap4 = T;   /* every expert receives at most T entries */
    void* recv4 = dev_alloc((size_t)E * cap4 * H);
    float* sc4 = dev_alloc((size_t)E * cap4 * (H / 128) * 4);
    int32_t* src4 = dev_alloc((size_t)E * cap4 * 4);
    CHECK(idx4 && slot4 && recv4 && sc4 && src4, "cudaMalloc (top-4)");
    CHECK(cudaMemcpy(idx4, hidx4, (size_t)T * K4 * 4, cudaMemcpyHostToDevice) == cudaSuccess,
          "copy idx4");
    CHECK(moedc_layout_dispatch(x, idx4, T, H, K4, E, R, cap4, MOEDC_FP8_E4M3, cnt, rk, inr, slot4,
                                recv4, sc4, src4, NULL, 0, status, 0) == MOEDC_OK,
          "moedc_layout_dispatch");
    CHECK(cudaDeviceSynchronize() == cudaSuccess, "synchronise (top-4)");
    float* hsc = malloc((size_t)E * cap4 * (H / 128) * 4);
    int32_t hcnt4[E];
    CHECK(cudaMemcpy(hcnt4, cnt, sizeof(hcnt4), cudaMemcpyDeviceToHost) == cudaSuccess, "cnt4");
    CHECK(cudaMemcpy(hsc, sc4, (size_t)E * cap4 * (H / 128) * 4, cudaMemcpyDeviceToHost) ==
              cudaSuccess,
          "scales");
    CHECK(cudaMemcpy(&hst, status, 4, cudaMemcpyDeviceToHost) == cudaSuccess, "status");
    CHECK(hst == MOEDC_OK, "status word clean (top-4)");
    total = 0;
    for (int e = 0; e < E; ++e) {
        total += hcnt4[e];
        for (int s = 0; s < hcnt4[e]; ++s)
            for (int g = 0; g < H / 128; ++g)
                CHECK(hsc[((size_t)e * cap4 + s) * (H / 128) + g] > 0.0f, "positive scale");
    }
    CHECK(total == T * K4, "top-4 counts");
    printf("moe_round: ok (%d tokens, bf16 round trip exact, e4m3 one-call layout+dispatch)\n", T);
    return 0;
}
