/*
 * synth_dev.cu -- device side of the seeded input generator (see synth_rng.h).
 *
 * Writes the generator's values straight into device buffers, so that the
 * 61 GB of full-scale synthetic weights never cross the host link.  Every
 * value is bit-identical to what synth_host.c produces for the same
 * (seed, tensor id, index); a GPU test checks that on samples.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth_rng.h"

namespace {

__global__ void fill_normal_bf16_kernel(uint64_t key, double sigma, uint16_t *out,
                                        int64_t n, int64_t offset) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    out[j] = syn_normal_bf16(key, (uint64_t)(offset + j), sigma);
}

__global__ void fill_const_bf16_kernel(uint16_t bits, uint16_t *out, int64_t n) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride)
    out[j] = bits;
}

int grid_for(int64_t n) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace

extern "C" {

/* out[j] = normal_bf16(seed, tid, offset + j, sigma) for j < n (device ptr). */
int syn_dev_fill_normal_bf16(uint64_t seed, uint64_t tid, double sigma, void *out,
                             int64_t n, int64_t offset, void *stream) {
  if (n <= 0) return 0;
  fill_normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(
      syn_key(seed, tid), sigma, (uint16_t *)out, n, offset);
  return (int)cudaGetLastError();
}

/* out[j] = bits for j < n (device ptr); used for all-ones norm gains. */
int syn_dev_fill_const_bf16(uint16_t bits, void *out, int64_t n, void *stream) {
  if (n <= 0) return 0;
  fill_const_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(
      bits, (uint16_t *)out, n);
  return (int)cudaGetLastError();
}

}  // extern "C"
