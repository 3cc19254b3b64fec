/* Device build of the generator in synth.h: the same values as synth_cpu.c. */
#include <cuda_runtime.h>
#include "synth.h"

__global__ void synth_normal_kernel(uint64_t key, uint64_t start, uint64_t n, float scale,
                                    const float* __restrict__ table, float* __restrict__ out) {
  uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) {
    float v = table[synth_index16(key, start + i)];
    out[i] = __fmul_rn(v, scale);
  }
}

/* Returns 0 on success, else the cudaError_t of the launch. */
extern "C" int synth_normal_f32_cuda(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t n,
                                     float scale, const float* table_dev, float* out_dev,
                                     cudaStream_t stream) {
  if (n == 0) return 0;
  const uint64_t key = synth_key(seed, tensor_id);
  uint64_t blocks = (n + 255) / 256;
  if (blocks > 152ull * 64ull) blocks = 152ull * 64ull;
  synth_normal_kernel<<<(unsigned)blocks, 256, 0, stream>>>(key, start, n, scale, table_dev, out_dev);
  return (int)cudaGetLastError();
}
