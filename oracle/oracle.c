/*
 * oracle.c -- plain, single-threaded CPU statement of the MoE expert-parallel
 * hot path: group-limited top-k gating, dispatch layout, permute-scatter
 * (BF16 or FP8 e4m3 with 1x128 block scales), inverse gather and the
 * router-weighted combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * checked against.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library and includes nothing from it.
 *
 * Sources followed (the pages give the method in prose only):
 *  - "DeepEP de DeepSeek : la lib open source qui optimise la communication
 *    GPU pour les modeles MoE a l'echelle" (ai-master.dev), section
 *    "Group-limited gating algorithm": a token's choice is limited to a
 *    subgroup of the experts instead of the global top-N.
 *  - same page, section "Support FP8 et MXFP8": the dispatched payload may be
 *    FP8, halving the bytes against BF16.
 *  - "Expert Parallelism (Parallelisme d'experts)" (polydesk.ai glossary),
 *    sections "Le principe de base" (whole experts per GPU, 8 experts on
 *    4 GPUs -> 2 per GPU) and "Le pattern de communication all-to-all"
 *    (Phase 1 Dispatch: tokens go to the holders of their experts; Phase 2
 *    Combine: results come back and are combined weighted by the router
 *    scores).
 *  - hyper.ai story on NVIDIA Hybrid-EP (hyper.ai/fr/stories/b564891f...):
 *    each token activates only its top-k experts; buffers sized up front.
 *
 * Where the pages are silent the plain readings below are taken; each one is
 * also listed with its reason in the design notes of the repository:
 *  - group score = sum of the group's top `topk_in_group` selection keys,
 *    added in descending order in binary32; groups are contiguous blocks;
 *  - selection key = score + bias (binary32 add); the bias only selects,
 *    the weights come from the unbiased score;
 *  - ties (equal keys or equal group scores) go to the lower index; slots are
 *    filled in selection order (descending key, then lower index);
 *  - raw-score weights are normalised to sum to one when `normalize` is set;
 *    softmax weights are the full softmax renormalised over the chosen k;
 *  - FP8: per 128-column block, s = amax / 448 in binary32, q = e4m3(x / s)
 *    with a binary32 IEEE division and round-to-nearest-even saturating to
 *    +-448 (the decisions that produce integers are made in binary32, the
 *    precision the kernels use); a block with amax == 0 gets s = 0 and a
 *    signed zero code;
 *  - receive rows are grouped by expert (hence by logical rank, since a
 *    rank's experts are contiguous), ascending flat (token, slot) index
 *    within an expert;
 *  - topk_idx == -1 marks an empty slot (skipped, no error); any other
 *    out-of-range index sets bit 0 of *err_flag and is skipped.
 *
 * Everything that is not an integer decision is computed in binary64
 * (weights, the combine sum) and rounded once at the end.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fPIC -shared oracle.c -lm
 * (no fast-math, no contraction: every float operation is the one written).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_SCORE_RAW 0
#define ORC_SCORE_SOFTMAX 1

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* bfloat16 -> binary32: bf16 is the top half of a binary32. */
static float bf16_bits_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary64 -> bfloat16, round to nearest, ties to even, in one rounding.
 * bfloat16 keeps 8 significant bits and binary32's exponent range, so the
 * spacing at |v| in [2^e, 2^(e+1)) is 2^(e-7), and 2^-133 below 2^-126. */
uint16_t orc_bf16_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v))
        return 0x7FC0u;
    if (isinf(v))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e = ilogb(a);
    int qe = (e < -126 ? -126 : e) - 7;      /* exponent of one unit in the last place */
    double r = rint(ldexp(a, -qe));          /* default rounding mode: nearest-even */
    double mag = ldexp(r, qe);
    if (mag >= 0x1p128)
        return (uint16_t)(sign | 0x7F80u);   /* overflow rounds to infinity */
    float f = (float)mag;                    /* exact: mag has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite
 * magnitude 448 = 1.75 * 2^8; subnormals are m * 2^-9. */
double orc_e4m3_decode(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 0xF, m = c & 7;
    if (E == 15 && m == 7)
        return NAN;
    double mag = (E == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), E - 10);
    return s ? -mag : mag;
}

/* binary32 -> E4M3, round to nearest, ties to even, saturating: magnitudes
 * past the largest finite value (and infinities) become +-448. */
uint8_t orc_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    if (isnan(v))
        return (uint8_t)(sign | 0x7Fu);
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7Eu);
    if (a == 0.0)
        return sign;
    int e = ilogb(a);
    int qe = (e < -6 ? -6 : e) - 3;          /* normals: 2^(e-3); subnormals: 2^-9 */
    double r = rint(ldexp(a, -qe));
    double mag = ldexp(r, qe);               /* a < 448 so mag <= 448 */
    if (mag == 0.0)
        return sign;
    if (mag < 0x1p-6)                        /* subnormal: exponent field 0 */
        return (uint8_t)(sign | (uint8_t)ldexp(mag, 9));
    int me = ilogb(mag);
    int mant = (int)ldexp(mag, 3 - me) - 8;  /* 0..7 */
    return (uint8_t)(sign | ((me + 7) << 3) | mant);
}

void orc_e4m3_encode_array(const float *v, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(v[i]);
}

void orc_e4m3_decode_array(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_decode(c[i]);
}

void orc_bf16_from_double_array(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_from_double(v[i]);
}

/* ------------------------------------------------------------------------ */
/* Step 1: gating                                                            */
/* ------------------------------------------------------------------------ */

/* Router top-k with the group limit.  Returns 0, or -1 on bad arguments.
 *
 * scores   [T, E] binary32: raw affinities (score_fn RAW) or logits (SOFTMAX)
 * bias     [E] binary32 or NULL: added to the score for selection only
 * topk_idx [T, k] out: chosen experts, slot order = selection order
 * topk_w   [T, k] out: binary64 weights
 */
int orc_gate(const float *scores, const float *bias, int32_t T, int32_t E, int32_t k,
             int32_t n_groups, int32_t topk_group, int32_t topk_in_group,
             int32_t score_fn, int32_t normalize, int32_t *topk_idx, double *topk_w)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E || n_groups <= 0 || E % n_groups != 0)
        return -1;
    if (topk_group <= 0 || topk_group > n_groups)
        return -1;
    const int32_t gsize = E / n_groups;
    if (topk_in_group <= 0 || topk_in_group > gsize || (int64_t)topk_group * gsize < k)
        return -1;
    if (score_fn != ORC_SCORE_RAW && score_fn != ORC_SCORE_SOFTMAX)
        return -1;

    float *key = malloc(sizeof(float) * (size_t)E);
    float *gscore = malloc(sizeof(float) * (size_t)n_groups);
    float *top = malloc(sizeof(float) * (size_t)topk_in_group);
    char *kept = malloc((size_t)n_groups);
    char *chosen = malloc((size_t)E);
    double *prob = malloc(sizeof(double) * (size_t)E);
    if (!key || !gscore || !top || !kept || !chosen || !prob) {
        free(key); free(gscore); free(top); free(kept); free(chosen); free(prob);
        return -1;
    }

    for (int32_t t = 0; t < T; ++t) {
        const float *s = scores + (int64_t)t * E;
        for (int32_t e = 0; e < E; ++e)
            key[e] = bias ? s[e] + bias[e] : s[e];

        /* Group score: the group's largest topk_in_group keys, largest first. */
        for (int32_t g = 0; g < n_groups; ++g) {
            int32_t have = 0;
            for (int32_t e = g * gsize; e < (g + 1) * gsize; ++e) {
                /* insertion into a descending list of length topk_in_group */
                float v = key[e];
                int32_t at = have;
                while (at > 0 && top[at - 1] < v)
                    --at;
                if (at < topk_in_group) {
                    int32_t last = have < topk_in_group ? have : topk_in_group - 1;
                    for (int32_t q = last; q > at; --q)
                        top[q] = top[q - 1];
                    top[at] = v;
                    if (have < topk_in_group)
                        ++have;
                }
            }
            float sum = top[0];
            for (int32_t q = 1; q < topk_in_group; ++q)
                sum = sum + top[q];
            gscore[g] = sum;
        }

        /* Keep the topk_group best groups (ties: lower group index). */
        memset(kept, 0, (size_t)n_groups);
        for (int32_t r = 0; r < topk_group; ++r) {
            int32_t best = -1;
            for (int32_t g = 0; g < n_groups; ++g)
                if (!kept[g] && (best < 0 || gscore[g] > gscore[best]))
                    best = g;
            kept[best] = 1;
        }

        /* Top-k experts among the kept groups (ties: lower expert index). */
        memset(chosen, 0, (size_t)E);
        int32_t *idx = topk_idx + (int64_t)t * k;
        for (int32_t j = 0; j < k; ++j) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (kept[e / gsize] && !chosen[e] && (best < 0 || key[e] > key[best]))
                    best = e;
            chosen[best] = 1;
            idx[j] = best;
        }

        /* Weights, from the unbiased score. */
        double *w = topk_w + (int64_t)t * k;
        if (score_fn == ORC_SCORE_RAW) {
            double den = 0.0;
            for (int32_t j = 0; j < k; ++j)
                den += (double)s[idx[j]];
            for (int32_t j = 0; j < k; ++j)
                w[j] = normalize ? (double)s[idx[j]] / den : (double)s[idx[j]];
        } else {
            /* softmax over all E logits, then (if normalize) renormalised over
             * the chosen k */
            double mx = (double)s[0];
            for (int32_t e = 1; e < E; ++e)
                if ((double)s[e] > mx)
                    mx = (double)s[e];
            double z = 0.0;
            for (int32_t e = 0; e < E; ++e) {
                prob[e] = exp((double)s[e] - mx);
                z += prob[e];
            }
            for (int32_t e = 0; e < E; ++e)
                prob[e] /= z;
            double den = 0.0;
            for (int32_t j = 0; j < k; ++j)
                den += prob[idx[j]];
            for (int32_t j = 0; j < k; ++j)
                w[j] = normalize ? prob[idx[j]] / den : prob[idx[j]];
        }
    }
    free(key); free(gscore); free(top); free(kept); free(chosen); free(prob);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 2: dispatch layout                                                   */
/* ------------------------------------------------------------------------ */

/* Receive-buffer layout for logical ranks of `experts_per_rank` contiguous
 * experts each.  Returns 0, or -1 on bad arguments.
 *
 * expert_count[E]   entries routed to each expert
 * expert_off[E+1]   exclusive prefix sum of expert_count
 * rank_count[R]     entries routed to each rank (sum of its experts' counts)
 * rank_off[R+1]     exclusive prefix sum of rank_count
 * rank_tokens[R]    distinct tokens with at least one entry on the rank
 * pos[T*k]          receive row of entry i = t*k + j, or -1 if skipped
 * src[T*k]          inverse of pos (flat entry index of each receive row);
 *                   rows past expert_off[E] hold -1
 * err_flag          bit 0 set if an index is neither -1 nor in [0, E)
 */
int orc_layout(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E, int32_t experts_per_rank,
               int32_t *expert_count, int32_t *expert_off, int32_t *rank_count, int32_t *rank_off,
               int32_t *rank_tokens, int32_t *pos, int32_t *src, int32_t *err_flag)
{
    if (T < 0 || k <= 0 || E <= 0 || experts_per_rank <= 0 || E % experts_per_rank != 0)
        return -1;
    const int32_t R = E / experts_per_rank;
    const int64_t N = (int64_t)T * k;
    int32_t err = 0;

    memset(expert_count, 0, sizeof(int32_t) * (size_t)E);
    for (int64_t i = 0; i < N; ++i) {
        int32_t e = topk_idx[i];
        if (e >= 0 && e < E)
            expert_count[e] += 1;
        else if (e != -1)
            err |= 1;
    }
    expert_off[0] = 0;
    for (int32_t e = 0; e < E; ++e)
        expert_off[e + 1] = expert_off[e] + expert_count[e];

    rank_off[0] = 0;
    for (int32_t r = 0; r < R; ++r) {
        int32_t c = 0;
        for (int32_t e = r * experts_per_rank; e < (r + 1) * experts_per_rank; ++e)
            c += expert_count[e];
        rank_count[r] = c;
        rank_off[r + 1] = rank_off[r] + c;
    }

    char *touched = malloc((size_t)R);
    if (!touched)
        return -1;
    memset(rank_tokens, 0, sizeof(int32_t) * (size_t)R);
    for (int32_t t = 0; t < T; ++t) {
        memset(touched, 0, (size_t)R);
        for (int32_t j = 0; j < k; ++j) {
            int32_t e = topk_idx[(int64_t)t * k + j];
            if (e >= 0 && e < E)
                touched[e / experts_per_rank] = 1;
        }
        for (int32_t r = 0; r < R; ++r)
            rank_tokens[r] += touched[r];
    }
    free(touched);

    /* Stable order: walk the entries in flat order and hand out rows. */
    int32_t *next = malloc(sizeof(int32_t) * (size_t)E);
    if (!next)
        return -1;
    memcpy(next, expert_off, sizeof(int32_t) * (size_t)E);
    for (int64_t i = 0; i < N; ++i)
        src[i] = -1;
    for (int64_t i = 0; i < N; ++i) {
        int32_t e = topk_idx[i];
        if (e >= 0 && e < E) {
            pos[i] = next[e]++;
            src[pos[i]] = (int32_t)i;
        } else {
            pos[i] = -1;
        }
    }
    free(next);
    if (err_flag)
        *err_flag |= err;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Step 3: dispatch (permute-scatter)                                        */
/* ------------------------------------------------------------------------ */

/* BF16 mode: recv[pos[t*k+j], :] = x[t, :] for every entry with pos >= 0. */
int orc_dispatch_bf16(const uint16_t *x, int32_t T, int32_t H, int32_t k, const int32_t *pos,
                      uint16_t *recv)
{
    if (T < 0 || H <= 0 || k <= 0)
        return -1;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < k; ++j) {
            int32_t p = pos[(int64_t)t * k + j];
            if (p >= 0)
                memcpy(recv + (int64_t)p * H, x + (int64_t)t * H, sizeof(uint16_t) * (size_t)H);
        }
    return 0;
}

/* FP8 mode: per token, per block of 128 columns, s = amax/448 and
 * q = e4m3(x/s); every copy of the token gets the same codes and scales.
 * recv_q [T*k, H] bytes, recv_s [T*k, H/128] binary32.  H % 128 == 0. */
int orc_dispatch_fp8(const uint16_t *x, int32_t T, int32_t H, int32_t k, const int32_t *pos,
                     uint8_t *recv_q, float *recv_s)
{
    if (T < 0 || H <= 0 || H % 128 != 0 || k <= 0)
        return -1;
    const int32_t nb = H / 128;
    uint8_t *q = malloc((size_t)H);
    float *sc = malloc(sizeof(float) * (size_t)nb);
    if (!q || !sc) {
        free(q); free(sc);
        return -1;
    }
    for (int32_t t = 0; t < T; ++t) {
        const uint16_t *row = x + (int64_t)t * H;
        for (int32_t b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int32_t c = 0; c < 128; ++c) {
                float a = fabsf(bf16_bits_to_float(row[b * 128 + c]));
                if (a > amax)
                    amax = a;
            }
            float s = amax / 448.0f;
            sc[b] = s;
            for (int32_t c = 0; c < 128; ++c) {
                float v = bf16_bits_to_float(row[b * 128 + c]);
                if (amax == 0.0f)
                    q[b * 128 + c] = signbit(v) ? 0x80u : 0x00u;
                else
                    q[b * 128 + c] = orc_e4m3_encode(v / s);
            }
        }
        for (int32_t j = 0; j < k; ++j) {
            int32_t p = pos[(int64_t)t * k + j];
            if (p < 0)
                continue;
            memcpy(recv_q + (int64_t)p * H, q, (size_t)H);
            memcpy(recv_s + (int64_t)p * nb, sc, sizeof(float) * (size_t)nb);
        }
    }
    free(q);
    free(sc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Steps 4 and 5: inverse gather and weighted combine                        */
/* ------------------------------------------------------------------------ */

/* out[t, h] = bf16( sum_j w[t, j] * y[pos[t*k+j], h] ), the sum taken over the
 * entries with pos >= 0 in binary64 and rounded once to bfloat16. */
int orc_combine(const uint16_t *y, const int32_t *pos, const float *w, int32_t T, int32_t H,
                int32_t k, uint16_t *out)
{
    if (T < 0 || H <= 0 || k <= 0)
        return -1;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int32_t j = 0; j < k; ++j) {
                int32_t p = pos[(int64_t)t * k + j];
                if (p >= 0)
                    acc += (double)w[(int64_t)t * k + j] * (double)bf16_bits_to_float(y[(int64_t)p * H + h]);
            }
            out[(int64_t)t * H + h] = orc_bf16_from_double(acc);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Next rows: MXFP8, FP8-input combine, capacity, backward                   */
/* ------------------------------------------------------------------------ */

/* MXFP8 (OCP Microscaling Formats v1.0, MXFP8 with E4M3 elements): blocks of
 * 32 columns share one power-of-two scale X = 2^e with
 * e = floor(log2(amax)) - 8 (8 = exponent of E4M3's largest normal, 448 =
 * 1.75 * 2^8), clamped to [-127, 127] and stored as the E8M0 byte e + 127.
 * Elements are e4m3(x / X), nearest-even, saturating; x / X is exact (a
 * power-of-two scaling).  A block with amax = 0 gets e = -127 (byte 0) and
 * signed-zero codes.  The pages name MXFP8 ("DeepEP de DeepSeek ...",
 * section "Support FP8 et MXFP8") without defining it; the definition is the
 * OCP one.  recv_q [T*k, H] bytes, recv_e [T*k, H/32] E8M0 bytes.
 * H % 32 == 0. */
int orc_dispatch_mxfp8(const uint16_t *x, int32_t T, int32_t H, int32_t k, const int32_t *pos,
                       uint8_t *recv_q, uint8_t *recv_e)
{
    if (T < 0 || H <= 0 || H % 32 != 0 || k <= 0)
        return -1;
    const int32_t nb = H / 32;
    uint8_t *q = malloc((size_t)H);
    uint8_t *eb = malloc((size_t)nb);
    if (!q || !eb) {
        free(q); free(eb);
        return -1;
    }
    for (int32_t t = 0; t < T; ++t) {
        const uint16_t *row = x + (int64_t)t * H;
        for (int32_t b = 0; b < nb; ++b) {
            double amax = 0.0;
            for (int32_t c = 0; c < 32; ++c) {
                double a = fabs((double)bf16_bits_to_float(row[b * 32 + c]));
                if (a > amax)
                    amax = a;
            }
            int e = (amax == 0.0) ? -127 : ilogb(amax) - 8;
            if (e < -127)
                e = -127;
            if (e > 127)
                e = 127;
            eb[b] = (uint8_t)(e + 127);
            for (int32_t c = 0; c < 32; ++c) {
                double v = (double)bf16_bits_to_float(row[b * 32 + c]);
                double scaled = ldexp(v, -e);               /* exact */
                if (amax == 0.0)
                    q[b * 32 + c] = signbit(v) ? 0x80u : 0x00u;
                else  /* (float) is exact, or flushes a far-below-2^-10 value to a signed zero */
                    q[b * 32 + c] = orc_e4m3_encode((float)scaled);
            }
        }
        for (int32_t j = 0; j < k; ++j) {
            int32_t p = pos[(int64_t)t * k + j];
            if (p < 0)
                continue;
            memcpy(recv_q + (int64_t)p * H, q, (size_t)H);
            memcpy(recv_e + (int64_t)p * nb, eb, (size_t)nb);
        }
    }
    free(q);
    free(eb);
    return 0;
}

/* Combine of FP8 expert outputs: the dequantised value of a code is its E4M3
 * value times its block's scale -- fp32 scales per 128 columns
 * (scale_kind 0) or E8M0 powers of two per 32 columns (scale_kind 1).
 * out[t, h] = bf16( sum_j w[t, j] * dequant(yq[pos[t, j], h]) ) in binary64. */
int orc_combine_fp8(const uint8_t *yq, const void *yscale, int32_t scale_kind, const int32_t *pos, const float *w,
                    int32_t T, int32_t H, int32_t k, uint16_t *out)
{
    if (T < 0 || H <= 0 || k <= 0 || (scale_kind != 0 && scale_kind != 1))
        return -1;
    const int32_t bs = scale_kind == 0 ? 128 : 32;
    if (H % bs != 0)
        return -1;
    const int32_t nb = H / bs;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int32_t j = 0; j < k; ++j) {
                int32_t p = pos[(int64_t)t * k + j];
                if (p < 0)
                    continue;
                double s = scale_kind == 0 ? (double)((const float *)yscale)[(int64_t)p * nb + h / bs]
                                           : ldexp(1.0, (int)((const uint8_t *)yscale)[(int64_t)p * nb + h / bs] - 127);
                acc += (double)w[(int64_t)t * k + j] * (orc_e4m3_decode(yq[(int64_t)p * H + h]) * s);
            }
            out[(int64_t)t * H + h] = orc_bf16_from_double(acc);
        }
    return 0;
}

/* Capacity-limited layout: expert e owns the fixed receive rows
 * [e * capacity, (e + 1) * capacity).  Entries are taken in flat (token,
 * slot) order; an expert's first `capacity` entries get its rows in that
 * order, later ones are dropped (pos = -1) -- the capacity factor / token
 * dropping lever of "Expert Parallelism (Parallelisme d'experts)", section
 * "Defis et optimisations" (Load balancing).  Outputs as orc_layout, with:
 * expert_count[E] = kept entries, expert_off[e] = e * capacity,
 * rank_count[R] = kept entries of the rank, rank_off[r] = r * epr * capacity,
 * rank_tokens[R] = distinct tokens with a kept entry on the rank,
 * expert_dropped[E] = entries past capacity, src[E * capacity] = flat entry
 * of each row or -1 for an empty row. */
int orc_layout_capacity(const int32_t *topk_idx, int32_t T, int32_t k, int32_t E, int32_t experts_per_rank,
                        int32_t capacity, int32_t *expert_count, int32_t *expert_off, int32_t *rank_count,
                        int32_t *rank_off, int32_t *rank_tokens, int32_t *expert_dropped, int32_t *pos,
                        int32_t *src, int32_t *err_flag)
{
    if (T < 0 || k <= 0 || E <= 0 || experts_per_rank <= 0 || E % experts_per_rank != 0 || capacity < 0)
        return -1;
    const int32_t R = E / experts_per_rank;
    const int64_t N = (int64_t)T * k;
    int32_t err = 0;
    memset(expert_count, 0, sizeof(int32_t) * (size_t)E);
    memset(expert_dropped, 0, sizeof(int32_t) * (size_t)E);
    for (int64_t i = 0; i < (int64_t)E * capacity; ++i)
        src[i] = -1;
    for (int64_t i = 0; i < N; ++i) {
        int32_t e = topk_idx[i];
        pos[i] = -1;
        if (e < 0 || e >= E) {
            if (e != -1)
                err |= 1;
            continue;
        }
        if (expert_count[e] < capacity) {
            pos[i] = e * capacity + expert_count[e];
            src[pos[i]] = (int32_t)i;
            expert_count[e] += 1;
        } else {
            expert_dropped[e] += 1;
        }
    }
    for (int32_t e = 0; e <= E; ++e)
        expert_off[e] = e * capacity;
    for (int32_t r = 0; r <= R; ++r)
        rank_off[r] = r * experts_per_rank * capacity;
    char *touched = malloc((size_t)R);
    if (!touched)
        return -1;
    for (int32_t r = 0; r < R; ++r) {
        int32_t c = 0;
        for (int32_t e = r * experts_per_rank; e < (r + 1) * experts_per_rank; ++e)
            c += expert_count[e];
        rank_count[r] = c;
        rank_tokens[r] = 0;
    }
    for (int32_t t = 0; t < T; ++t) {
        memset(touched, 0, (size_t)R);
        for (int32_t j = 0; j < k; ++j)
            if (pos[(int64_t)t * k + j] >= 0)
                touched[topk_idx[(int64_t)t * k + j] / experts_per_rank] = 1;
        for (int32_t r = 0; r < R; ++r)
            rank_tokens[r] += touched[r];
    }
    free(touched);
    if (err_flag)
        *err_flag |= err;
    return 0;
}

/* Backward of the BF16 dispatch (a copy): each source row's gradient is the
 * sum of its copies' gradients, grad_x[t] = bf16( sum_j grad_recv[pos[t,j]] )
 * in binary64; a token with no copy gets zeros. */
int orc_dispatch_backward(const uint16_t *grad_recv, const int32_t *pos, int32_t T, int32_t H, int32_t k,
                          uint16_t *grad_x)
{
    if (T < 0 || H <= 0 || k <= 0)
        return -1;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int32_t j = 0; j < k; ++j) {
                int32_t p = pos[(int64_t)t * k + j];
                if (p >= 0)
                    acc += (double)bf16_bits_to_float(grad_recv[(int64_t)p * H + h]);
            }
            grad_x[(int64_t)t * H + h] = orc_bf16_from_double(acc);
        }
    return 0;
}

/* Backward of the weighted combine out[t] = sum_j w[t,j] * y[pos[t,j]]:
 * grad_y[pos[t,j], h] = bf16( w[t,j] * grad_out[t,h] ) (exact product, one
 * rounding) and grad_w[t,j] = sum_h grad_out[t,h] * y[pos[t,j], h]
 * (binary64; 0 for an empty slot).  Rows of grad_y no entry names are left
 * untouched. */
int orc_combine_backward(const uint16_t *grad_out, const uint16_t *y, const int32_t *pos, const float *w,
                         int32_t T, int32_t H, int32_t k, uint16_t *grad_y, double *grad_w)
{
    if (T < 0 || H <= 0 || k <= 0)
        return -1;
    for (int32_t t = 0; t < T; ++t)
        for (int32_t j = 0; j < k; ++j) {
            int32_t p = pos[(int64_t)t * k + j];
            double dot = 0.0;
            if (p >= 0) {
                double wj = (double)w[(int64_t)t * k + j];
                for (int32_t h = 0; h < H; ++h) {
                    double g = (double)bf16_bits_to_float(grad_out[(int64_t)t * H + h]);
                    grad_y[(int64_t)p * H + h] = orc_bf16_from_double(wj * g);
                    dot += g * (double)bf16_bits_to_float(y[(int64_t)p * H + h]);
                }
            }
            grad_w[(int64_t)t * k + j] = dot;
        }
    return 0;
}
