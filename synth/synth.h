/*
 * Seeded synthetic inputs in C: the same generator as the Python module
 * synth/__init__.py, so that C programs (tests/c_abi_check.c) draw the very
 * arrays the Python tests draw.  Random numbers only: none of the method's
 * arithmetic lives here.
 *
 * Value i (0-based) of stream (seed, s) is
 *   mix64(mix64(seed * 2^32 + s) + (i + 1) * 0x9E3779B97F4A7C15)
 * with the splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  Uniforms are odd multiples
 * of 2^-24 in (0, 1); normals come from the Box-Muller transform in binary64
 * on pairs of draws from streams s and s + 0x10000, in blocks of 2^22 pairs
 * (the block layout of the Python generator); hidden rows are bfloat16,
 * nearest-even from binary32.  The normals go through libm (log, sqrt,
 * cos, sin), so a rare last bit may differ from numpy's; uniforms and
 * everything integer are exact.
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Streams of one workload (as in the Python module). */
enum { SYNTH_S_SCORES = 1, SYNTH_S_BIAS = 2, SYNTH_S_X = 3, SYNTH_S_PERM = 4, SYNTH_S_Y = 5, SYNTH_S_W = 6 };

uint64_t synth_u64(uint64_t seed, uint64_t stream, uint64_t i);
void synth_uniform_f32(uint64_t seed, uint64_t stream, size_t n, float *out);
void synth_normal_f64(uint64_t seed, uint64_t stream, size_t n, double *out);
uint16_t synth_f32_to_bf16(float f);
/* N(0, sigma^2) rounded to binary32, then to bfloat16 bits. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, size_t n, double sigma, uint16_t *out);

#ifdef __cplusplus
}
#endif

#endif
