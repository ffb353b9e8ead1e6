/*
 * Seeded synthetic inputs for attention: iid normal samples, counter-based.
 *
 * This module is shared by the fp64 oracle and the GPU path as their common
 * source of inputs. It holds none of the attention arithmetic: it only draws
 * numbers and rounds them to the storage type the kernels read.
 *
 * Generator (all published definitions, written here from them):
 *   - SplitMix64 (Steele, Lea, Flood, "Fast Splittable Pseudorandom Number
 *     Generators", OOPSLA 2014): the 64-bit finaliser mix64 below, applied to a
 *     Weyl sequence  key + (i + 1) * GAMMA.  Element i of a stream depends only on
 *     (seed, stream, i), so any slice can be generated independently and in
 *     parallel, with identical values on every machine.
 *   - Uniform in (0,1):  u = ((x >> 11) + 0.5) * 2^-53.
 *   - Box-Muller transform (Box and Muller, 1958): for pair p the uniforms
 *     u1 = U(2p), u2 = U(2p+1) give z0 = r cos(2 pi u2), z1 = r sin(2 pi u2) with
 *     r = sqrt(-2 ln u1); element 2p is z0 and element 2p+1 is z1.
 *   - Storage rounding: x * sigma (fp64) -> fp32 by the C cast (round to nearest
 *     even) -> bf16 by round-to-nearest-even on the fp32 bit pattern.
 *
 * Built with -ffp-contract=off so that no FMA contraction changes the values
 * between compilers or architectures.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed + GAMMA) ^ (stream * 0xD1B54A32D192ED03ULL));
}

static double uniform_open(uint64_t key, uint64_t i) {
  uint64_t x = mix64(key + (i + 1ULL) * GAMMA);
  return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

static double normal_at(uint64_t key, int64_t idx) {
  const double two_pi = 6.283185307179586476925286766559;
  uint64_t p = (uint64_t)idx >> 1;
  double u1 = uniform_open(key, 2 * p);
  double u2 = uniform_open(key, 2 * p + 1);
  double r = sqrt(-2.0 * log(u1));
  return (idx & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  /* inputs are finite normals: no NaN handling needed, but keep NaN a NaN */
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* Element idx of the stream, for idx in [offset, offset + n). */
void seeded_normal_f64(uint64_t seed, uint64_t stream, int64_t offset, int64_t n,
                       double sigma, double* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) out[t] = normal_at(key, offset + t) * sigma;
}

void seeded_normal_f32(uint64_t seed, uint64_t stream, int64_t offset, int64_t n,
                       double sigma, float* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) out[t] = (float)(normal_at(key, offset + t) * sigma);
}

void seeded_normal_bf16(uint64_t seed, uint64_t stream, int64_t offset, int64_t n,
                        double sigma, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t)
    out[t] = f32_to_bf16_rne((float)(normal_at(key, offset + t) * sigma));
}

/* Plain conversion helpers so callers need no second rounding routine. */
void seeded_f64_to_bf16(const double* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n; ++t) out[t] = f32_to_bf16_rne((float)in[t]);
}
