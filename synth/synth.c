/* Seeded synthetic inputs in C (see synth.h for the definitions). */
#include "synth.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ull
#define SYNTH_PAIR_BLOCK ((size_t)1 << 22)

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) { return mix64((seed << 32) + stream); }

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t i)
{
    return mix64(stream_key(seed, stream) + (i + 1) * SYNTH_GOLDEN);
}

void synth_uniform_f32(uint64_t seed, uint64_t stream, size_t n, float *out)
{
    const uint64_t key = stream_key(seed, stream);
    for (size_t i = 0; i < n; ++i) {
        const uint64_t u = mix64(key + (uint64_t)(i + 1) * SYNTH_GOLDEN) >> 41; /* 23 random bits */
        out[i] = (float)(((double)u * 2.0 + 1.0) * 0x1p-24);
    }
}

void synth_normal_f64(uint64_t seed, uint64_t stream, size_t n, double *out)
{
    const uint64_t ka = stream_key(seed, stream), kb = stream_key(seed, stream + 0x10000);
    const size_t pairs = (n + 1) / 2;
    for (size_t p = 0; p < pairs; ++p) {
        /* pair p of block c0 draws counter 2*c0 + (p - c0) of both streams */
        const size_t c0 = (p / SYNTH_PAIR_BLOCK) * SYNTH_PAIR_BLOCK;
        const uint64_t ctr = (uint64_t)(2 * c0 + (p - c0)) + 1;
        const uint64_t a = mix64(ka + ctr * SYNTH_GOLDEN), b = mix64(kb + ctr * SYNTH_GOLDEN);
        const double u1 = ((double)(a >> 11) + 1.0) * 0x1p-53; /* (0, 1] */
        const double u2 = (double)(b >> 11) * 0x1p-53;         /* [0, 1) */
        const double r = sqrt(-2.0 * log(u1));
        const double th = 2.0 * M_PI * u2;
        out[2 * p] = r * cos(th);
        if (2 * p + 1 < n)
            out[2 * p + 1] = r * sin(th);
    }
}

uint16_t synth_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u); /* nearest, ties to even (finite inputs) */
    return (uint16_t)(u >> 16);
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, size_t n, double sigma, uint16_t *out)
{
    if (n == 0)
        return;
    double *z = malloc(n * sizeof(double));
    if (!z)
        abort();
    synth_normal_f64(seed, stream, n, z);
    for (size_t i = 0; i < n; ++i)
        out[i] = synth_f32_to_bf16((float)(z[i] * sigma));
    free(z);
}
