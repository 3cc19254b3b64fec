// Block quantiser: fp32 [rows, cols] -> E4M3 or E2M1 codes + one UE8M0 scale
// per 32 consecutive elements of a row.  It is the quantisation that precedes
// the fused call (the "pre-dispatch" step of sglang PR #36657, section Fix;
// recipe (1, 1, 32) of the fp8_fp4_mega_moe call quoted on the digest page of
// the same PR, 关键源码片段).  One thread per 32-element block.
#include "common.cuh"
#include "numerics.cuh"

namespace mm {

template <bool kE4M3>
__global__ void __launch_bounds__(256) quantize_kernel(const float* __restrict__ src, long long nblocks,
                                                       uint8_t* __restrict__ dst, uint8_t* __restrict__ sf) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < nblocks; b += stride) {
    const float4* s4 = reinterpret_cast<const float4*>(src + b * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 t = __ldg(s4 + i);
      v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int s = block_scale_exp<kE4M3>(amax);
    const float inv = exp2_neg(s);
    if (kE4M3) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        w[i] = e4m3_code(v[4 * i] * inv) | (e4m3_code(v[4 * i + 1] * inv) << 8) |
               (e4m3_code(v[4 * i + 2] * inv) << 16) | (e4m3_code(v[4 * i + 3] * inv) << 24);
      }
      uint4* d4 = reinterpret_cast<uint4*>(dst + b * 32);
      d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
      d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t x = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) x |= e2m1_code(v[8 * i + j] * inv) << (4 * j);
        w[i] = x;
      }
      *reinterpret_cast<uint4*>(dst + b * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    sf[b] = (uint8_t)(s + 127);
  }
}

// Host launcher (kept in this translation unit: template kernels are launched
// where they are defined).
cudaError_t launch_quantize(const float* src, long long nblocks, bool e4m3, uint8_t* dst, uint8_t* sf,
                            int grid, cudaStream_t stream) {
  if (e4m3) quantize_kernel<true><<<grid, 256, 0, stream>>>(src, nblocks, dst, sf);
  else      quantize_kernel<false><<<grid, 256, 0, stream>>>(src, nblocks, dst, sf);
  return cudaGetLastError();
}

}  // namespace mm
