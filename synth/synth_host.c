/*
 * Host side of the synthetic input generator (see synth.h).  Built by gcc
 * into libsynth_host.so; the test and benchmark harness call it through
 * ctypes to materialise inputs in host memory and to regenerate single
 * elements for sampled checks of full-size device runs.
 */
#include <math.h>
#include <stdint.h>

#include "synth.h"

uint64_t synth_hash_host(uint64_t key, uint64_t ctr) { return synth_hash(key, ctr); }

uint64_t synth_key_host(uint64_t seed, uint32_t stream, uint64_t a, uint64_t b) {
  return synth_key(seed, stream, a, b);
}

/* amp for a standard deviation sigma, rounded once to fp32. */
float synth_amp_host(double sigma) { return (float)(sigma * sqrt(3.0) / 131072.0); }

/* out[i] = synth_bf16(key, first + i, ...) for i in [0, n). */
void synth_fill_bf16_host(uint16_t* out, int64_t n, uint64_t key, uint64_t first,
                          float amp, uint32_t outlier_every, float outlier_mult) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = synth_bf16(key, first + (uint64_t)i, amp, outlier_every, outlier_mult);
}

/* Gather variant: out[i] = synth_bf16(key, idx[i], ...). */
void synth_gather_bf16_host(uint16_t* out, const int64_t* idx, int64_t n, uint64_t key,
                            float amp, uint32_t outlier_every, float outlier_mult) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = synth_bf16(key, (uint64_t)idx[i], amp, outlier_every, outlier_mult);
}

/* out[i] = synth_f32(key, first + i, amp) for i in [0, n). */
void synth_fill_f32_host(float* out, int64_t n, uint64_t key, uint64_t first, float amp) {
  for (int64_t i = 0; i < n; ++i) out[i] = synth_f32(key, first + (uint64_t)i, amp);
}
