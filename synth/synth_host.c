/*
 * synth_host.c -- host side of the seeded input generator (see synth_rng.h).
 *
 * Fills host buffers with the generator's values.  Used by the CPU oracle
 * (which may regenerate any input on the fly from the same definition) and
 * by the Python harness for small configurations.  OpenMP splits the index
 * range; every element depends only on its own index, so the thread count
 * never changes a value.
 */
#include <stddef.h>
#include <stdint.h>
#include "synth_rng.h"

uint64_t syn_host_key(uint64_t seed, uint64_t tid) { return syn_key(seed, tid); }

/* out[j] = normal_bf16(seed, tid, offset + j, sigma), j < n. */
void syn_host_fill_normal_bf16(uint64_t seed, uint64_t tid, double sigma,
                               uint16_t *out, int64_t n, int64_t offset) {
  const uint64_t key = syn_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j)
    out[j] = syn_normal_bf16(key, (uint64_t)(offset + j), sigma);
}

/* out[j] = normal(seed, tid, offset + j) as double (for distribution tests). */
void syn_host_fill_normal_f64(uint64_t seed, uint64_t tid, double *out,
                              int64_t n, int64_t offset) {
  const uint64_t key = syn_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; ++j) out[j] = syn_normal(key, (uint64_t)(offset + j));
}

/* out[j] = uniform_int(seed, tid, offset + j, m). */
void syn_host_fill_uniform_int(uint64_t seed, uint64_t tid, uint32_t m,
                               int32_t *out, int64_t n, int64_t offset) {
  const uint64_t key = syn_key(seed, tid);
  for (int64_t j = 0; j < n; ++j)
    out[j] = (int32_t)syn_uniform_int(key, (uint64_t)(offset + j), m);
}

/* Seeded Fisher-Yates permutation of 0..n-1 (draw i picks from [0, i]). */
void syn_host_permutation(uint64_t seed, uint64_t tid, int32_t *out, int64_t n) {
  const uint64_t key = syn_key(seed, tid);
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  for (int64_t i = n - 1; i > 0; --i) {
    int64_t j = (int64_t)syn_uniform_int(key, (uint64_t)i, (uint32_t)(i + 1));
    int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}
