// Block quantiser: fp32 [rows, cols] -> E4M3 or E2M1 codes + one UE8M0 scale
// per 32 consecutive elements of a row.  It is the quantisation that precedes
// the fused call (the "pre-dispatch" step of sglang PR #36657, section Fix;
// recipe (1, 1, 32) of the fp8_fp4_mega_moe call quoted on the digest page of
// the same PR, 关键源码片段).  One thread per 32-element block.
#include <algorithm>

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

// The (1, 128, 128) recipe's quantiser (DeepGEMM SM90 MegaMoE dev log, Phase 1
// entry: the SM90 wrapper's recipe with float scale factors): fp32
// [rows, cols] -> E4M3 codes and one fp32 scale per block of block_rows x 128
// (block_rows 1 for activations, 128 for weights).  Scale s = a / 448 for a
// block with largest magnitude a (1 for a zero block); code = RNE E4M3 of the
// IEEE fp32 quotient v / s, saturating.
__device__ __forceinline__ float f8b_scale(float amax) {
  return amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// Blocks of 1 x 128: one warp per block, four values per lane.
__global__ void __launch_bounds__(256) quantize_f8b_rows_kernel(const float* __restrict__ src, long long nblocks,
                                                                uint8_t* __restrict__ dst, float* __restrict__ sf) {
  const int lane = threadIdx.x & 31;
  const long long stride = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long b = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblocks; b += stride) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(src + b * 128) + lane);
    float amax = fmaxf(fmaxf(fabsf(t.x), fabsf(t.y)), fmaxf(fabsf(t.z), fabsf(t.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = f8b_scale(amax);
    const uint32_t w = e4m3_code(__fdiv_rn(t.x, sc)) | (e4m3_code(__fdiv_rn(t.y, sc)) << 8) |
                       (e4m3_code(__fdiv_rn(t.z, sc)) << 16) | (e4m3_code(__fdiv_rn(t.w, sc)) << 24);
    reinterpret_cast<uint32_t*>(dst + b * 128)[lane] = w;
    if (lane == 0) sf[b] = sc;
  }
}

// Blocks of 128 x 128: one CTA of 256 threads per block; thread t holds four
// consecutive columns of rows t / 32 + 8i (i < 16).
__global__ void __launch_bounds__(256) quantize_f8b_tiles_kernel(const float* __restrict__ src, int rows, int cols,
                                                                 uint8_t* __restrict__ dst, float* __restrict__ sf) {
  __shared__ float s_max[8];
  const int nbc = cols / 128;
  const long long nblocks = (long long)(rows / 128) * nbc;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (long long b = blockIdx.x; b < nblocks; b += gridDim.x) {
    const int br = (int)(b / nbc), bc = (int)(b % nbc);
    const float* base = src + (size_t)br * 128 * cols + (size_t)bc * 128 + 4 * lane;
    float4 v[16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[i] = __ldg(reinterpret_cast<const float4*>(base + (size_t)(warp + 8 * i) * cols));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) s_max[warp] = amax;
    __syncthreads();
    amax = s_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, s_max[i]);
    const float sc = f8b_scale(amax);
    uint8_t* dbase = dst + (size_t)br * 128 * cols + (size_t)bc * 128 + 4 * lane;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w = e4m3_code(__fdiv_rn(v[i].x, sc)) | (e4m3_code(__fdiv_rn(v[i].y, sc)) << 8) |
                         (e4m3_code(__fdiv_rn(v[i].z, sc)) << 16) | (e4m3_code(__fdiv_rn(v[i].w, sc)) << 24);
      *reinterpret_cast<uint32_t*>(dbase + (size_t)(warp + 8 * i) * cols) = w;
    }
    if (t == 0) sf[b] = sc;
    __syncthreads();                     // s_max is reused by the next block
  }
}

cudaError_t launch_quantize_f8b(const float* src, long long rows, long long cols, int block_rows, uint8_t* dst,
                                float* sf, int max_ctas, cudaStream_t stream) {
  if (block_rows == 1) {
    const long long nblocks = rows * (cols / 128);
    const long long ctas = std::min<long long>((nblocks + 7) / 8, max_ctas);
    quantize_f8b_rows_kernel<<<(int)std::max(1ll, ctas), 256, 0, stream>>>(src, nblocks, dst, sf);
  } else {
    const long long nblocks = (rows / 128) * (cols / 128);
    const long long ctas = std::min<long long>(nblocks, max_ctas);
    quantize_f8b_tiles_kernel<<<(int)std::max(1ll, ctas), 256, 0, stream>>>(src, (int)rows, (int)cols, dst, sf);
  }
  return cudaGetLastError();
}

// Weight scales -> scale atoms: a UE8M0 matrix [rows, kb] (kb = K / 32 blocks
// per row) becomes [rows / 128][kb / 4] atoms of 512 bytes, atom (rb, s) lane
// l holding the 4 bytes of stage s (blocks 4s .. 4s + 3) of rows 128 rb + l,
// + 32 + l, + 64 + l and + 96 + l.  One thread per 16-byte lane of an atom.
__global__ void __launch_bounds__(256) prepare_weight_scales_kernel(const uint8_t* __restrict__ sf, long long rows,
                                                                    int kb, uint8_t* __restrict__ out) {
  const int stages = kb / 4;
  const long long nlanes = rows / 128 * stages * 32;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nlanes; i += stride) {
    const int l = (int)(i & 31);
    const long long atom = i >> 5;                     // rb * stages + s
    const long long rb = atom / stages;
    const int s = (int)(atom - rb * stages);
    const uint8_t* src = sf + (size_t)(rb * 128 + l) * kb + 4 * s;
    uint32_t w[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) w[c] = __ldg(reinterpret_cast<const uint32_t*>(src + (size_t)c * 32 * kb));
    reinterpret_cast<uint4*>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

cudaError_t launch_prepare_weight_scales(const uint8_t* sf, long long rows, int kb, uint8_t* out, int max_ctas,
                                         cudaStream_t stream) {
  const long long nlanes = rows / 128 * (kb / 4) * 32;
  const long long ctas = std::min<long long>((nlanes + 255) / 256, max_ctas);
  prepare_weight_scales_kernel<<<(int)std::max(1ll, ctas), 256, 0, stream>>>(sf, rows, kb, out);
  return cudaGetLastError();
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
