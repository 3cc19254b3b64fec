// Test helper: occupy one SM for a bounded time.  One CTA with a large
// dynamic shared-memory request, so no other large-smem CTA fits on its SM,
// spins on %globaltimer for `ns` nanoseconds and exits.  Always terminates.
#include <cstdint>
#include <cuda_runtime.h>

__global__ void occupy_sm(unsigned long long ns, int* started) {
  extern __shared__ volatile uint8_t pad[];
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  if (threadIdx.x == 0) { pad[0] = 1; atomicExch(started, 1); }
  do {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
}

extern "C" int occupy_one_sm(unsigned long long ns, int smem_bytes, int* started, cudaStream_t stream) {
  if (cudaFuncSetAttribute(occupy_sm, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
    return (int)cudaGetLastError();
  occupy_sm<<<1, 32, smem_bytes, stream>>>(ns, started);
  return (int)cudaGetLastError();
}
