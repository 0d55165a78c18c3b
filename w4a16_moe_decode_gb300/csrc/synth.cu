// Seeded synthetic inputs on the device (SplitMix64 streams, Irwin-Hall
// normals); the definition is in flint_synth.h and is shared, as a definition
// only, with the CPU generator used by the tests.
#include <cuda_bf16.h>

#include "flint_synth.h"

namespace {

constexpr uint64_t GOLDEN = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void k_synth(uint64_t key, uint64_t start, size_t n, float sigma, int out_bf16, void* out) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const uint64_t idx = start + i;
    int64_t acc = 0;
#pragma unroll
    for (int w = 0; w < 3; ++w) {
      const uint64_t u = mix64(key + (3 * idx + w + 1) * GOLDEN);
#pragma unroll
      for (int f = 0; f < 4; ++f) acc += 2 * (int64_t)((u >> (16 * f)) & 0xFFFF) + 1;
    }
    acc -= 12 * 65536;
    const float z = (float)acc * 0x1p-17f;  // exact: |acc| < 2^20
    const float v = z * sigma;
    if (out_bf16) {
      const __nv_bfloat16 b = __float2bfloat16_rn(v);
      static_cast<uint16_t*>(out)[i] = *reinterpret_cast<const uint16_t*>(&b);
    } else {
      static_cast<float*>(out)[i] = v;
    }
  }
}

}  // namespace

extern "C" uint64_t flint_synth_stream_key(uint64_t seed, uint32_t layer, uint32_t tensor, uint32_t expert) {
  const uint64_t packed = ((uint64_t)(layer & 0xFFFF) << 48) | ((uint64_t)(tensor & 0xFFFF) << 32) | expert;
  return mix64(seed ^ mix64(packed));
}

extern "C" int flint_synth_normal(uint64_t key, uint64_t start, size_t n, float sigma, int32_t out_bf16, void* out,
                                  cudaStream_t stream) {
  if (!out) return 1;
  if (n == 0) return 0;
  size_t blocks = (n + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  k_synth<<<(unsigned)blocks, 256, 0, stream>>>(key, start, n, sigma, out_bf16, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
