/*
 * A C program that uses the library through include/ep.h alone: no Python,
 * no PyTorch.  It routes a small DeepSeek-V3-shaped batch (E = 256 experts in
 * 8 groups, top-4 groups, top-8 experts, 32 ranks x 8 experts) with
 * ep_gate_layout, dispatches it (BF16 and FP8), combines identity-expert
 * outputs with the router weights.  Its inputs come from the C generator
 * (synth/synth.c: the Python tests' DeepSeek-V3 workload, seed 1236, at
 * T = 512 and H = 256), and it checks the results against the CPU oracle
 * (oracle/oracle.c, linked as liboracle.so): gating indices, the whole
 * layout, BF16 rows and FP8 codes and scales bit for bit, weights within
 * (k+1) binary32 roundings, the combine within max(1 bf16 ulp, 1e-2
 * relative).  It also checks on the host what the definitions fix:
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
 * Build: cc -I include -I synth tests/c_abi_check.c synth/synth.c -L <pkg> -lep_gb300
 *        -L oracle -loracle -L <cuda>/lib64 -lcudart -lm
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ep.h"
#include "synth.h"

/* The CPU oracle (oracle/oracle.c), test infrastructure only. */
int orc_gate(const float *scores, const float *bias, int32_t T, int32_t E, int32_t k, int32_t n_groups,
             int32_t topk_group, int32_t topk_in_group, int32_t score_fn, int32_t normalize, int32_t *topk_idx,
             double *topk_w);
int orc_layout(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E, int32_t experts_per_rank,
               int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
               int32_t *rank_tokens, int32_t *pos, int32_t *src, int32_t *err_flag);
int orc_dispatch_bf16(const uint16_t *x, int32_t T, int32_t H, int32_t k, const int32_t *pos, uint16_t *recv);
int orc_dispatch_fp8(const uint16_t *x, int32_t T, int32_t H, int32_t k, const int32_t *pos, uint8_t *recv_q,
                     float *recv_s);
int orc_combine(const uint16_t *y, const int32_t *pos, const float *w, int32_t T, int32_t H, int32_t k,
                uint16_t *out);

#define T 512
#define H 256
#define E 256
#define K 8
#define G 8
#define KG 4
#define KIN 2
#define EPR 8
#define R (E / EPR)
#define SEED 1236 /* the DeepSeek-V3 workload's seed */

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

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}


int main(void)
{
    static float scores[T * E], bias[E], w[T * K];
    static uint16_t x[T * H], recv[T * K * H], out[T * H];
    static int32_t idx[T * K], pos[T * K], src[T * K], ecount[E], eoff[E + 1], rcount[R], roff[R + 1], rtok[R];
    static uint8_t q[T * K * H];
    static float qs[T * K * (H / 128)];
    /* the DeepSeek-V3 workload's arrays at this T and H: U(0,1) scores,
     * N(0, 0.01) bias, N(0,1) bf16 rows */
    synth_uniform_f32(SEED, SYNTH_S_SCORES, (size_t)T * E, scores);
    {
        double b64[E];
        synth_normal_f64(SEED, SYNTH_S_BIAS, E, b64);
        for (int e = 0; e < E; ++e)
            bias[e] = (float)(b64[e] * 0.01);
    }
    synth_normal_bf16(SEED, SYNTH_S_X, (size_t)T * H, 1.0, x);

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
    CK(cudaMemcpy(rcount, d_rc, sizeof rcount, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(roff, d_ro, sizeof roff, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(rtok, d_rt, sizeof rtok, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(recv, d_recv, sizeof recv, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(q, d_q, sizeof q, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(qs, d_sc, sizeof qs, cudaMemcpyDeviceToHost));
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

    /* parity with the CPU oracle on the same inputs */
    {
        static int32_t oidx[T * K], opos[T * K], osrc[T * K], oec[E], oeo[E + 1], orc[R], oro[R + 1], ort[R];
        static double ow[T * K];
        static uint16_t orecv[T * K * H], oout[T * H];
        static uint8_t oq[T * K * H];
        static float oqs[T * K * (H / 128)];
        int32_t oflag = 0;
        if (orc_gate(scores, bias, T, E, K, G, KG, KIN, EP_SCORE_RAW, 1, oidx, ow) != 0)
            return fail("oracle gate", 0, 0);
        for (int i = 0; i < T * K; ++i) {
            if (idx[i] != oidx[i])
                return fail("gate index vs oracle", i, oidx[i]);
            if (fabs((double)w[i] - ow[i]) > (K + 1) * 5.96e-8 * fabs(ow[i]))
                return fail("gate weight vs oracle", i, 0);
        }
        if (orc_layout(oidx, T, K, E, EPR, oec, oeo, orc, oro, ort, opos, osrc, &oflag) != 0 || oflag != 0)
            return fail("oracle layout", oflag, 0);
        if (memcmp(ecount, oec, sizeof oec) || memcmp(eoff, oeo, sizeof oeo) || memcmp(rcount, orc, sizeof orc) ||
            memcmp(roff, oro, sizeof oro) || memcmp(rtok, ort, sizeof ort) || memcmp(pos, opos, sizeof opos) ||
            memcmp(src, osrc, sizeof osrc))
            return fail("layout vs oracle", 0, 0);
        memset(orecv, 0, sizeof orecv);
        if (orc_dispatch_bf16(x, T, H, K, opos, orecv) != 0 || memcmp(recv, orecv, sizeof orecv))
            return fail("bf16 dispatch vs oracle", 0, 0);
        if (orc_dispatch_fp8(x, T, H, K, opos, oq, oqs) != 0 || memcmp(q, oq, sizeof oq) || memcmp(qs, oqs, sizeof oqs))
            return fail("fp8 dispatch vs oracle", 0, 0);
        if (orc_combine(orecv, opos, w, T, H, K, oout) != 0)
            return fail("oracle combine", 0, 0);
        for (int i = 0; i < T * H; ++i) {
            const float g = bf16_to_f32(out[i]), r = bf16_to_f32(oout[i]);
            const float ulp = fabsf(r) * (1.0f / 128.0f); /* one bf16 ulp is at most 2^-7 |r| */
            const float bar = fmaxf(ulp, 1e-2f * fabsf(r));
            if (fabsf(g - r) > bar + 1e-30f)
                return fail("combine vs oracle", i / H, i % H);
        }
    }
    printf("c_abi_check ok: %d tokens gated, laid out, dispatched and combined through ep.h; "
           "matches the oracle\n", T);
    return 0;
}
