/*
 * Seeded, counter-based input generator shared by the test harness, the bench
 * and the smoke run. It holds no arithmetic of the MoE step itself: it only
 * turns (seed, stream, index) into numbers.
 *
 * Every value is a pure function of (seed, stream, index), so any slice of any
 * tensor can be regenerated on the host or on the device, in any order, with
 * bit-identical results. Only integer operations and one IEEE
 * round-to-nearest-even fp32 multiply are used, so the host build (gcc) and the
 * device build (nvcc) agree bit for bit.
 *
 * Bits: the SplitMix64 output function (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; the finaliser constants are
 * the published "Mix13" variant by D. Stafford) evaluated at state
 * key + n * 0x9E3779B97F4A7C15, i.e. the n-th output of a SplitMix64 sequence
 * started at `key`, which is what makes it counter-based.
 *
 * Normals: the Irwin-Hall sum of twelve 16-bit uniforms, centred:
 *     z = (sum_{j<12} (c_j + 1/2) / 65536) - 6 = (S - 393210) / 65536,
 * S = sum of the twelve 16-bit integers c_j. z has mean 0, variance 1
 * (up to 2^-32), support [-6, 6] and a 2^-16 grid; it is computed exactly in
 * integers and the final scale by sigma is a single fp32 multiply.
 */
#ifndef SYNTH_RNG_H
#define SYNTH_RNG_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_FN __host__ __device__ static inline
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ull

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Key of one independent stream (one tensor, one redraw round, ...). */
SYNTH_FN uint64_t synth_stream_key(uint64_t seed, uint64_t stream) {
  return synth_mix64(synth_mix64(seed ^ 0x5851F42D4C957F2Dull) + stream * SYNTH_GAMMA);
}

/* n-th 64-bit output of the stream. */
SYNTH_FN uint64_t synth_u64(uint64_t key, uint64_t n) {
  return synth_mix64(key + (n + 1) * SYNTH_GAMMA);
}

/* Irwin-Hall(12) standard deviate for element `idx`, exactly representable in fp32. */
SYNTH_FN float synth_std_normal(uint64_t key, uint64_t idx) {
  int64_t s = 0;
  for (int j = 0; j < 3; ++j) {
    uint64_t w = synth_u64(key, 3 * idx + (uint64_t)j);
    s += (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) +
         (int64_t)((w >> 32) & 0xFFFF) + (int64_t)(w >> 48);
  }
  /* |s - 393210| <= 393210 < 2^24: exact in fp32, and so is the 2^-16 scale. */
  return (float)(s - 393210) * (1.0f / 65536.0f);
}

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite). */
SYNTH_FN uint16_t synth_f32_to_bf16_bits(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t lsb = (v.u >> 16) & 1u;
  return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

#endif
