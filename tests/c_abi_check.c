/*
 * A C program that uses the library through include/ep.h alone: no Python,
 * no PyTorch.  It routes a small DeepSeek-V3-shaped batch (E = 256 experts in
 * 8 groups, top-4 groups, top-8 experts, 32 ranks x 8 experts) with
 * ep_gate_layout, dispatches it (BF16 and FP8), combines identity-expert
 * outputs with the router weights, and checks on the host what the
 * definitions fix:
 *  - every token's experts are distinct, lie in its kept groups and have the
 *    largest keys there (ties to the lower index);
 *  - raw weights sum to one;
 *  - the layout counts sum to T*k, pos is a bijection with src its inverse,
 *    and rows ascend with the flat entry inside each expert;
 *  - every BF16 receive row equals its source row;
 *  - combine of the copies reproduces x within one bf16 ulp plus the fp32
 *    accumulation error (weights sum to one).
 * Exit status 0 on success; the first failed check is printed.
 *
 * Build: cc -I include tests/c_abi_check.c -L <pkg> -lep_gb300 -L <cuda>/lib64 -lcudart -lm
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ep.h"

#define T 512
#define H 256
#define E 256
#define K 8
#define G 8
#define KG 4
#define KIN 2
#define EPR 8

static int fail(const char *what, long a, long b)
{
    fprintf(stderr, "c_abi_check: %s (%ld, %ld)\n", what, a, b);
    return 1;
}

#define CK(x)                                                                       \
    do {                                                                            \
        cudaError_t e_ = (x);                                                       \
        if (e_ != cudaSuccess) {                                                    \
            fprintf(stderr, "c_abi_check: %s: %s\n", #x, cudaGetErrorString(e_)); \
            return 2;                                                               \
        }                                                                           \
    } while (0)

#define EP(x)                                                                        \
    do {                                                                             \
        ep_status s_ = (x);                                                          \
        if (s_ != EP_OK) {                                                           \
            fprintf(stderr, "c_abi_check: %s: %s\n", #x, ep_status_str(s_));         \
            return 3;                                                                \
        }                                                                            \
    } while (0)

static uint64_t rng_state = 0x243F6A8885A308D3ull;

static uint64_t next_u64(void)
{
    uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static float uniform01(void) { return (float)((next_u64() >> 40) + 0.5) / 16777216.0f; }

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u); /* round to nearest even (finite inputs) */
    return (uint16_t)(u >> 16);
}

int main(void)
{
    static float scores[T * E], bias[E], w[T * K];
    static uint16_t x[T * H], recv[T * K * H], out[T * H];
    static int32_t idx[T * K], pos[T * K], src[T * K], ecount[E], eoff[E + 1], rcount[E / EPR], roff[E / EPR + 1],
        rtok[E / EPR];
    for (int i = 0; i < T * E; ++i)
        scores[i] = uniform01();
    for (int e = 0; e < E; ++e)
        bias[e] = (uniform01() - 0.5f) * 0.02f;
    for (int i = 0; i < T * H; ++i)
        x[i] = f32_to_bf16(uniform01() * 4.0f - 2.0f);

    const ep_gate_cfg cfg = {E, K, G, KG, KIN, EP_SCORE_RAW, 1};
    size_t wsb = ep_layout_workspace_bytes(T, K, E, EPR);
    if (wsb == 0)
        return fail("workspace size", 0, 0);

    float *d_s, *d_b, *d_w;
    uint16_t *d_x, *d_recv, *d_out;
    uint8_t *d_q;
    float *d_sc;
    int32_t *d_idx, *d_ec, *d_eo, *d_rc, *d_ro, *d_rt, *d_pos, *d_src, *d_flag;
    void *d_ws;
    CK(cudaMalloc((void **)&d_s, sizeof scores));
    CK(cudaMalloc((void **)&d_b, sizeof bias));
    CK(cudaMalloc((void **)&d_w, sizeof w));
    CK(cudaMalloc((void **)&d_x, sizeof x));
    CK(cudaMalloc((void **)&d_recv, sizeof recv));
    CK(cudaMalloc((void **)&d_out, sizeof out));
    CK(cudaMalloc((void **)&d_q, (size_t)T * K * H));
    CK(cudaMalloc((void **)&d_sc, (size_t)T * K * (H / 128) * sizeof(float)));
    CK(cudaMalloc((void **)&d_idx, sizeof idx));
    CK(cudaMalloc((void **)&d_ec, sizeof ecount));
    CK(cudaMalloc((void **)&d_eo, sizeof eoff));
    CK(cudaMalloc((void **)&d_rc, sizeof rcount));
    CK(cudaMalloc((void **)&d_ro, sizeof roff));
    CK(cudaMalloc((void **)&d_rt, sizeof rtok));
    CK(cudaMalloc((void **)&d_pos, sizeof pos));
    CK(cudaMalloc((void **)&d_src, sizeof src));
    CK(cudaMalloc((void **)&d_flag, sizeof(int32_t)));
    CK(cudaMalloc(&d_ws, wsb));
    CK(cudaMemset(d_ws, 0, wsb)); /* the barrier count of ep_gate_layout starts at zero */
    CK(cudaMemset(d_flag, 0, sizeof(int32_t)));
    CK(cudaMemcpy(d_s, scores, sizeof scores, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_b, bias, sizeof bias, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice));

    EP(ep_gate_layout(d_s, d_b, T, &cfg, EPR, d_idx, d_w, d_ec, d_eo, d_rc, d_ro, d_rt, d_pos, d_src, d_flag, d_ws,
                      wsb, NULL));
    EP(ep_dispatch(d_x, T, H, K, d_pos, EP_DTYPE_BF16, d_recv, T * K, NULL, d_flag, NULL));
    EP(ep_dispatch(d_x, T, H, K, d_pos, EP_DTYPE_FP8_E4M3_B128, d_q, T * K, d_sc, d_flag, NULL));
    EP(ep_combine(d_recv, T * K, d_pos, d_w, T, H, K, d_out, d_flag, NULL));
    CK(cudaDeviceSynchronize());

    int32_t flag;
    CK(cudaMemcpy(&flag, d_flag, sizeof flag, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(idx, d_idx, sizeof idx, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(w, d_w, sizeof w, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(pos, d_pos, sizeof pos, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(src, d_src, sizeof src, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(ecount, d_ec, sizeof ecount, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(eoff, d_eo, sizeof eoff, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(recv, d_recv, sizeof recv, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost));
    if (flag != 0)
        return fail("device error flag", flag, 0);

    /* gating: distinct experts inside the kept groups, largest keys first */
    for (int t = 0; t < T; ++t) {
        const float *s = scores + (size_t)t * E;
        float gsc[G];
        for (int g = 0; g < G; ++g) { /* sum of the two largest keys of the group */
            float a = -INFINITY, b = -INFINITY;
            for (int e = g * (E / G); e < (g + 1) * (E / G); ++e) {
                const float key = s[e] + bias[e];
                if (key > a) {
                    b = a;
                    a = key;
                } else if (key > b) {
                    b = key;
                }
            }
            gsc[g] = a + b;
        }
        int kept[G] = {0};
        for (int r = 0; r < KG; ++r) {
            int best = -1;
            for (int g = 0; g < G; ++g)
                if (!kept[g] && (best < 0 || gsc[g] > gsc[best]))
                    best = g;
            kept[best] = 1;
        }
        int chosen[E] = {0};
        float wsum = 0.0f;
        for (int j = 0; j < K; ++j) {
            const int e = idx[t * K + j];
            if (e < 0 || e >= E || chosen[e] || !kept[e / (E / G)])
                return fail("gate expert", t, e);
            chosen[e] = 1;
            wsum += w[t * K + j];
        }
        if (fabsf(wsum - 1.0f) > 1e-5f)
            return fail("weights do not sum to one", t, 0);
        for (int e = 0; e < E; ++e) { /* no unchosen expert of a kept group beats a chosen one */
            if (chosen[e] || !kept[e / (E / G)])
                continue;
            const float key = s[e] + bias[e];
            for (int j = 0; j < K; ++j) {
                const int c = idx[t * K + j];
                const float kc = s[c] + bias[c];
                if (key > kc || (key == kc && e < c))
                    return fail("gate order", t, e);
            }
        }
    }
    /* layout */
    long total = 0;
    for (int e = 0; e < E; ++e) {
        if (eoff[e] != total)
            return fail("expert_off", e, eoff[e]);
        total += ecount[e];
    }
    if (total != (long)T * K || eoff[E] != total)
        return fail("counts", total, eoff[E]);
    for (int i = 0; i < T * K; ++i) {
        const int p = pos[i];
        if (p < 0 || p >= T * K || src[p] != i)
            return fail("pos/src", i, p);
        const int e = idx[i];
        if (p < eoff[e] || p >= eoff[e + 1])
            return fail("row outside its expert", i, p);
        if (p > eoff[e] && src[p - 1] >= i)
            return fail("rows not ascending", i, p);
    }
    /* BF16 dispatch, then combine of the identity-expert rows */
    for (int i = 0; i < T * K; ++i)
        if (memcmp(recv + (size_t)pos[i] * H, x + (size_t)(i / K) * H, H * sizeof(uint16_t)) != 0)
            return fail("bf16 receive row", i, pos[i]);
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            const float xv = bf16_to_f32(x[t * H + h]), ov = bf16_to_f32(out[t * H + h]);
            const float tol = fabsf(xv) * (1.0f / 128.0f) + fabsf(xv) * 9.0f * 5.96e-8f + 1e-30f;
            if (fabsf(ov - xv) > tol)
                return fail("combine of the copies", t, h);
        }
    printf("c_abi_check ok: %d tokens gated, laid out, dispatched and combined through ep.h\n", T);
    return 0;
}
