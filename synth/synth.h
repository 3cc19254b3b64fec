/*
 * Seeded, counter-based synthetic input generator (shared definition).
 *
 * This header is the whole generator: it is compiled once as host C (the
 * CPU side used by the tests and the oracle's inputs) and once as CUDA
 * device code (the GPU side used by the benchmark and the GPU tests), so
 * both produce the same fp32 values bit for bit.  It holds none of the
 * MoE layer's arithmetic: no quantisation, no routing, no matmul.
 *
 * Definition.
 *   - SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): the n-th output of a stream whose state
 *     starts at `key` is mix64(key + (n + 1) * GOLDEN).
 *   - A tensor is a stream keyed by key = mix64(seed * GOLDEN + tensor_id *
 *     STREAM_MULT + 1).  Element i of the tensor takes the 16-bit field
 *     (i mod 4) of output n = i / 4, so one 64-bit output feeds four
 *     consecutive elements.
 *   - The 16-bit field j indexes a 65536-entry fp32 table of standard-normal
 *     quantiles, table[j] = Phi^-1((j + 0.5) / 65536), supplied by the
 *     caller (it is computed once per process and handed to both sides).
 *   - value = table[j] * scale, one IEEE fp32 multiply.
 */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>

#ifdef __CUDACC__
#define SYNTH_FN static __host__ __device__ __forceinline__
#else
#define SYNTH_FN static inline
#endif

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL
#define SYNTH_STREAM_MULT 0xD1B54A32D192ED03ULL

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYNTH_FN uint64_t synth_key(uint64_t seed, uint64_t tensor_id) {
  return synth_mix64(seed * SYNTH_GOLDEN + tensor_id * SYNTH_STREAM_MULT + 1ULL);
}

/* 16-bit table index of element i of the stream `key`. */
SYNTH_FN uint32_t synth_index16(uint64_t key, uint64_t i) {
  uint64_t w = synth_mix64(key + ((i >> 2) + 1ULL) * SYNTH_GOLDEN);
  return (uint32_t)((w >> (16u * (uint32_t)(i & 3u))) & 0xFFFFu);
}

#endif
