/*
 * Seeded synthetic input generator shared by the tests, the bench and the
 * oracle's callers.  It holds none of the MoE layer's arithmetic: it only
 * turns (seed, tensor tag, element index) into a stored fp32 or bf16 value.
 *
 * Definition (counter based, so any element can be produced independently):
 *   key      = sm64_mix(seed * 2^32 + tag)
 *   u64(c)   = sm64_mix(key + (c + 1) * 0x9E3779B97F4A7C15)
 *              i.e. the c-th output of a SplitMix64 generator seeded with key
 *              (S. Vigna's SplitMix64: golden-gamma increment, then the
 *              variant-13 finaliser with shifts 30/27/31).
 *   unif(c)  = (u64(c) >> 11) * 2^-53                      in [0, 1)
 *   Box-Muller on the pair i (counters 2i, 2i+1), in fp64:
 *              u1 = 1 - unif(2i) in (0, 1],  u2 = unif(2i+1)
 *              r  = sqrt(-2 ln u1)
 *              z[2i] = r cos(2 pi u2),  z[2i+1] = r sin(2 pi u2)
 *   value    = mean + std * z, rounded to fp32 (round to nearest even),
 *              and for bf16 the fp32 bits rounded to nearest even to 16 bits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tag) {
  return sm64_mix((seed << 32) + tag);
}

static inline double unif53(uint64_t key, uint64_t c) {
  uint64_t u = sm64_mix(key + (c + 1ULL) * 0x9E3779B97F4A7C15ULL);
  return (double)(u >> 11) * (1.0 / 9007199254740992.0);
}

static inline double normal_at(uint64_t key, uint64_t i) {
  uint64_t pair = i >> 1;
  double u1 = 1.0 - unif53(key, 2 * pair);
  double u2 = unif53(key, 2 * pair + 1);
  double r = sqrt(-2.0 * log(u1));
  double a = 6.283185307179586476925286766559 * u2;
  return (i & 1) ? r * sin(a) : r * cos(a);
}

/* fp32 -> bf16 bits, round to nearest even; NaN stays NaN (quiet). */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

uint64_t seeded_u64(uint64_t seed, uint64_t tag, uint64_t c) {
  return sm64_mix(stream_key(seed, tag) + (c + 1ULL) * 0x9E3779B97F4A7C15ULL);
}

double seeded_normal_f64(uint64_t seed, uint64_t tag, uint64_t i) {
  return normal_at(stream_key(seed, tag), i);
}

/* out[i] = fp32(mean + std * z(offset + i)), i < n */
void seeded_normal_f32(uint64_t seed, uint64_t tag, double mean, double std, uint64_t offset,
                       int64_t n, float* out) {
  uint64_t key = stream_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(mean + std * normal_at(key, offset + (uint64_t)i));
}

/* out[i] = bf16(fp32(mean + std * z(offset + i))) as raw bits, i < n */
void seeded_normal_bf16(uint64_t seed, uint64_t tag, double mean, double std, uint64_t offset,
                        int64_t n, uint16_t* out) {
  uint64_t key = stream_key(seed, tag);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i)
    out[i] = f32_to_bf16_rne((float)(mean + std * normal_at(key, offset + (uint64_t)i)));
}

/* bf16 bits -> fp32 values (exact widening). */
void seeded_bf16_to_f32(const uint16_t* in, int64_t n, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint32_t u = (uint32_t)in[i] << 16;
    memcpy(&out[i], &u, 4);
  }
}

/* fp32 -> bf16 bits, round to nearest even. */
void seeded_f32_to_bf16(const float* in, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/* The c-th output of a SplitMix64 generator whose state starts at `state`
 * (exposed so that tests can check the generator against published values). */
uint64_t seeded_splitmix_raw(uint64_t state, uint64_t c) {
  return sm64_mix(state + (c + 1ULL) * 0x9E3779B97F4A7C15ULL);
}
