/*
 * synth_rng.h -- counter-based generator for the seeded synthetic inputs.
 *
 * This header is the input generator shared by the CPU oracle and by the GPU
 * test/bench harness.  It holds none of the decode step's arithmetic: it only
 * turns (seed, tensor id, element index) into a number, identically on the
 * host and on the device.
 *
 * Definition (the same on every platform, bit for bit):
 *   mix64(z)      : the SplitMix64 output function (Steele, Lea & Flood,
 *                   "Fast splittable pseudorandom number generators",
 *                   OOPSLA 2014; constants as published by Vigna):
 *                     z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *                     z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *   key(seed,tid) = mix64(mix64(seed + GAMMA) ^ tid)
 *   word(key, c)  = mix64(key + (c + 1) * GAMMA),  GAMMA = 0x9E3779B97F4A7C15
 *
 *   normal(seed, tid, i): the Irwin-Hall approximation of N(0,1): the sum of
 *   the twelve 32-bit halves of word(key, 6i) .. word(key, 6i+5), minus
 *   6*2^32, divided by 2^32.  Every step up to that quotient is exact in
 *   integer or double arithmetic, so host and device agree bit for bit.  The
 *   result has mean 0, variance 1 and support [-6, 6].
 *   normal_bf16(seed, tid, i, sigma) = bf16_rne((float)(normal * sigma)).
 *
 *   uniform_int(seed, tid, i, n) = (hi32(word(key, i)) * n) >> 32, in [0, n).
 *
 * No floating-point operation here may be contracted into an FMA: the only
 * floating-point operations are one int->double conversion, one subtraction
 * and one multiplication by a power of two (all exact) and one
 * multiplication by sigma.
 */
#ifndef SYNTH_RNG_H
#define SYNTH_RNG_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_HD __host__ __device__ __forceinline__
#else
#define SYN_HD static inline
#endif

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

SYN_HD uint64_t syn_mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

SYN_HD uint64_t syn_key(uint64_t seed, uint64_t tid) {
  return syn_mix64(syn_mix64(seed + SYN_GAMMA) ^ tid);
}

SYN_HD uint64_t syn_word(uint64_t key, uint64_t c) {
  return syn_mix64(key + (c + 1ULL) * SYN_GAMMA);
}

/* Irwin-Hall(12) standard normal approximation, exact in double. */
SYN_HD double syn_normal(uint64_t key, uint64_t i) {
  uint64_t s = 0;
  for (int j = 0; j < 6; ++j) {
    uint64_t w = syn_word(key, 6ULL * i + (uint64_t)j);
    s += (w & 0xFFFFFFFFULL) + (w >> 32);
  }
  /* s < 12 * 2^32 < 2^36: the conversion and the subtraction are exact. */
  double z = (double)(int64_t)s - 25769803776.0; /* 6 * 2^32 */
  return z * (1.0 / 4294967296.0);              /* exact: power of two */
}

/* Round-to-nearest-even float -> bf16 bits (NaN is never produced here). */
SYN_HD uint16_t syn_f32_to_bf16(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

SYN_HD uint16_t syn_normal_bf16(uint64_t key, uint64_t i, double sigma) {
  double x = syn_normal(key, i) * sigma;
  return syn_f32_to_bf16((float)x);
}

SYN_HD uint32_t syn_uniform_int(uint64_t key, uint64_t i, uint32_t n) {
  uint64_t w = syn_word(key, i);
  return (uint32_t)(((w >> 32) * (uint64_t)n) >> 32);
}

/* Uniform double in [0, 1) with 53 random bits. */
SYN_HD double syn_uniform01(uint64_t key, uint64_t i) {
  uint64_t w = syn_word(key, i);
  return (double)(w >> 11) * (1.0 / 9007199254740992.0);
}

#endif /* SYNTH_RNG_H */
