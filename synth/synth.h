/*
 * Seeded, counter-based synthetic input generator.
 *
 * This header is the single definition of the test and benchmark inputs
 * (per-rank bf16 gradients and the gathered bf16 buffer).  It is compiled
 * twice: by gcc into the host generator (synth_host.c) and by nvcc into the
 * device fill kernel (synth_fill.cu), so both sides see the same bits for the
 * same (key, index).  It holds none of the reduce-scatter or placement
 * arithmetic: only hashing, a normal-ish draw and a bf16 rounding of that draw.
 *
 * Definitions used:
 *  - splitmix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom
 *    number generators", OOPSLA 2014): the 64-bit mixing function with the
 *    constants 0xBF58476D1CE4E5B9 / 0x94D049BB133111EB and shifts 30/27/31,
 *    applied to key + (ctr + 1) * 0x9E3779B97F4A7C15 (the golden gamma).
 *  - Irwin-Hall approximation of a normal: the sum of four independent
 *    uniform 16-bit integers taken from one 64-bit hash, centred.  The sum
 *    s in [0, 262140] has variance 4 * (2^32 - 1) / 12, so 2s - 262140 has a
 *    standard deviation of almost exactly 131072 / sqrt(3); multiplying by
 *    amp = sigma * sqrt(3) / 131072 gives standard deviation sigma.
 *  - bf16 round-to-nearest-even of a finite fp32 value by integer bit
 *    arithmetic on its top 16 bits.
 */
#ifndef TIDE_SYNTH_H
#define TIDE_SYNTH_H

#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SYNTH_FN __host__ __device__ static inline
#else
#define SYNTH_FN static inline
#endif

/* Stream tags: independent hash streams per kind of input. */
#define SYNTH_STREAM_GRAD 1u     /* per-rank gradient of one parameter     */
#define SYNTH_STREAM_GATHER 2u   /* full parameter value behind the AG buffer */
#define SYNTH_STREAM_ZERO 3u     /* per (rank, expert) unrouted decision     */
#define SYNTH_STREAM_SWEEP 4u    /* rank-sweep shape draws                   */
#define SYNTH_STREAM_SHARD 5u    /* fp32 shard values (pack inputs)          */
#define SYNTH_OUTLIER_SALT 0xD1B54A32D192ED03ull

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Counter-based draw: the ctr-th output of a splitmix64 sequence seeded at key. */
SYNTH_FN uint64_t synth_hash(uint64_t key, uint64_t ctr) {
  return synth_mix64(key + (ctr + 1ull) * 0x9E3779B97F4A7C15ull);
}

/* Key of one input tensor: (seed, stream, a, b), e.g. (seed, GRAD, rank, param). */
SYNTH_FN uint64_t synth_key(uint64_t seed, uint32_t stream, uint64_t a, uint64_t b) {
  return synth_hash(synth_hash(synth_hash(seed, stream), a), b);
}

SYNTH_FN uint32_t synth_f32_bits(float f) {
#if defined(__CUDA_ARCH__)
  return __float_as_uint(f);
#else
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
#endif
}

SYNTH_FN float synth_mul(float a, float b) {
#if defined(__CUDA_ARCH__)
  return __fmul_rn(a, b);
#else
  return a * b;
#endif
}

/* bf16 bits of a finite fp32 value, IEEE 754-2008 roundTiesToEven on the
 * 16 dropped bits (adding 0x7FFF plus the lowest kept bit carries exactly
 * when the dropped part is above half an ulp, or equal with an odd kept part). */
SYNTH_FN uint16_t synth_bf16_rne(float f) {
  uint32_t u = synth_f32_bits(f);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/*
 * Element idx of the tensor with key `key`:
 *   v = (2 * (u0 + u1 + u2 + u3) - 262140) * amp         (fp32, one rounding)
 *   v = v * outlier_mult   if outlier_every != 0 and a second hash of idx
 *                          is divisible by outlier_every  (fp32, one rounding)
 *   return bf16_rne(v)
 */
SYNTH_FN uint16_t synth_bf16(uint64_t key, uint64_t idx, float amp,
                             uint32_t outlier_every, float outlier_mult) {
  uint64_t h = synth_hash(key, idx);
  int32_t s = (int32_t)(h & 0xFFFFu) + (int32_t)((h >> 16) & 0xFFFFu) +
              (int32_t)((h >> 32) & 0xFFFFu) + (int32_t)(h >> 48);
  float v = synth_mul((float)(2 * s - 262140), amp);
  if (outlier_every != 0u &&
      synth_hash(key ^ SYNTH_OUTLIER_SALT, idx) % (uint64_t)outlier_every == 0ull)
    v = synth_mul(v, outlier_mult);
  return synth_bf16_rne(v);
}

/* fp32 element idx of the tensor with key `key`: the same Irwin-Hall draw
 * without the bf16 rounding, so all 24 mantissa bits vary (inputs of the
 * fp32 -> bf16 pack). */
SYNTH_FN float synth_f32(uint64_t key, uint64_t idx, float amp) {
  uint64_t h = synth_hash(key, idx);
  int32_t s = (int32_t)(h & 0xFFFFu) + (int32_t)((h >> 16) & 0xFFFFu) +
              (int32_t)((h >> 32) & 0xFFFFu) + (int32_t)(h >> 48);
  return synth_mul((float)(2 * s - 262140), amp);
}

#endif /* TIDE_SYNTH_H */
