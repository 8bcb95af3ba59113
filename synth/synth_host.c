/*
 * Seeded synthetic inputs, host side.
 *
 * This file holds no arithmetic of the MoE decode step.  It only turns a
 * (seed, tag, element index) triple into a pseudo-random value, so that the
 * CPU oracle and the GPU path can be fed bit-identical inputs.  The device
 * side (synth_dev.cu) implements the same two published definitions on its
 * own; neither file includes the other.
 *
 *  - Philox4x32-10: the counter-based generator of Salmon, Moraes, Dror and
 *    Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4,
 *    with its round multipliers 0xD2511F53 / 0xCD9E8D57 and Weyl key
 *    increments 0x9E3779B9 / 0xBB67AE85.
 *  - An approximately normal deviate: the Irwin-Hall sum of eight uniform
 *    16-bit halves of one Philox block, centred and scaled to unit variance
 *    (Irwin 1927, Hall 1927).  It uses integer arithmetic and one fp32
 *    multiply only, so it is bit-identical on any IEEE machine.
 *
 * Keying: key = (seed, tag), counter = (index low 32 bits, index high 32 bits,
 * 0, 0).  One Philox block per element.
 */
#include <stdint.h>
#include <stddef.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

/* sqrt(12 / 8) rounded to fp32: the Irwin-Hall sum of 8 unit uniforms has
 * variance 8/12. */
#define SYNTH_IH8_SCALE 1.2247449f

void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                         uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Unit-variance Irwin-Hall(8) deviate for element `index` of stream (seed, tag). */
float synth_unit_normal(uint32_t seed, uint32_t tag, uint64_t index) {
  uint32_t ctr[4] = {(uint32_t)index, (uint32_t)(index >> 32), 0u, 0u};
  uint32_t key[2] = {seed, tag};
  uint32_t r[4];
  synth_philox4x32_10(ctr, key, r);
  int32_t s = 0;
  for (int i = 0; i < 4; ++i) s += (int32_t)(r[i] & 0xFFFFu) + (int32_t)(r[i] >> 16);
  /* sum of (u + 1/2)/65536 minus 4, times 65536: an exact integer */
  int32_t n = s - 262140;
  float z = (float)n * (1.0f / 65536.0f); /* exact: |n| < 2^24, power-of-two scale */
  return z * SYNTH_IH8_SCALE;
}

float synth_normal(uint32_t seed, uint32_t tag, uint64_t index, float mu, float sigma) {
  float z = synth_unit_normal(seed, tag, index);
  float t = sigma * z; /* two separate fp32 roundings: built with -ffp-contract=off */
  return mu + t;
}

/* Round-to-nearest-even fp32 -> bf16 bit pattern (finite inputs). */
uint16_t synth_f32_to_bf16(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)((u + bias) >> 16);
}

void synth_normal_f32(float* out, uint64_t n, uint32_t seed, uint32_t tag, float mu,
                      float sigma) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = synth_normal(seed, tag, (uint64_t)i, mu, sigma);
}

void synth_normal_bf16(uint16_t* out, uint64_t n, uint32_t seed, uint32_t tag, float mu,
                       float sigma) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = synth_f32_to_bf16(synth_normal(seed, tag, (uint64_t)i, mu, sigma));
}

/* Raw Philox words, for tests and for seeded permutations. */
void synth_philox_words(uint32_t* out, uint64_t n_blocks, uint32_t seed, uint32_t tag) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n_blocks; ++i) {
    uint32_t ctr[4] = {(uint32_t)i, (uint32_t)((uint64_t)i >> 32), 0u, 0u};
    uint32_t key[2] = {seed, tag};
    synth_philox4x32_10(ctr, key, out + 4 * i);
  }
}
