/* Host build of the generator in synth.h (OpenMP over elements). */
#include "synth.h"
#include <stddef.h>

/* out[i] = table[index16(key(seed, tensor_id), start + i)] * scale, i < n. */
void synth_normal_f32(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t n,
                      float scale, const float* table, float* out) {
  const uint64_t key = synth_key(seed, tensor_id);
  long long nn = (long long)n;
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < nn; ++i) {
    float v = table[synth_index16(key, start + (uint64_t)i)];
    out[i] = v * scale;
  }
}

/* Raw 64-bit stream outputs (used for permutations and for pinning). */
void synth_u64(uint64_t seed, uint64_t tensor_id, uint64_t start, uint64_t n, uint64_t* out) {
  const uint64_t key = synth_key(seed, tensor_id);
  for (uint64_t i = 0; i < n; ++i) out[i] = synth_mix64(key + (start + i + 1ULL) * SYNTH_GOLDEN);
}
