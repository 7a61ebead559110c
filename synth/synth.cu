// Host and device front ends of the counter-based generator in synth_rng.h.
// Both loops evaluate the same inline functions, so a tensor generated on the
// GPU equals, bit for bit, the same tensor generated on the host.
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth_rng.h"

namespace {

__global__ void normal_f32_kernel(uint64_t key, uint64_t offset, uint64_t n, float sigma, float* out) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = __fmul_rn(synth_std_normal(key, offset + i), sigma);
}

__global__ void normal_bf16_kernel(uint64_t key, uint64_t offset, uint64_t n, float sigma, uint16_t* out) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = synth_f32_to_bf16_bits(__fmul_rn(synth_std_normal(key, offset + i), sigma));
}

int grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ull * 16) g = 152ull * 16;
  return g == 0 ? 1 : (int)g;
}

}  // namespace

extern "C" {

// out[i] = sigma * z(seed, stream, offset + i), i < n  (host memory)
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float sigma, float* out) {
  uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = synth_std_normal(key, offset + (uint64_t)i) * sigma;
}

// Same values rounded to bf16 (bit patterns), host memory.
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float sigma, uint16_t* out) {
  uint64_t key = synth_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (int64_t)n; ++i)
    out[i] = synth_f32_to_bf16_bits(synth_std_normal(key, offset + (uint64_t)i) * sigma);
}

// n raw 64-bit outputs of a stream (host memory).
void synth_u64_fill(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, uint64_t* out) {
  uint64_t key = synth_stream_key(seed, stream);
  for (uint64_t i = 0; i < n; ++i) out[i] = synth_u64(key, offset + i);
}

// Device versions: `out` is device memory, the fill is enqueued on `stream_handle`
// (a cudaStream_t). Returns the cudaError_t of the launch.
int synth_normal_f32_device(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float sigma,
                            float* out, void* stream_handle) {
  if (n == 0) return 0;
  normal_f32_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream_handle>>>(
      synth_stream_key(seed, stream), offset, n, sigma, out);
  return (int)cudaGetLastError();
}

int synth_normal_bf16_device(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n, float sigma,
                             uint16_t* out, void* stream_handle) {
  if (n == 0) return 0;
  normal_bf16_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream_handle>>>(
      synth_stream_key(seed, stream), offset, n, sigma, out);
  return (int)cudaGetLastError();
}

}  // extern "C"
