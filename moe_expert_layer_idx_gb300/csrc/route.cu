// Routing kernel: per-launch reset, expert histogram, prefix scan, stable
// permutation and the per-expert N-block table of the persistent kernel.
//
// The pages' kernel does this as its dispatch prologue ("workspace clean ->
// expert count -> source token-topk index write", DeepGEMM SM90 MegaMoE dev
// log, Phase 2 entry) and resets its readiness flags on every launch (DeepGEMM
// PR #451, "Reset MegaMoE combine readiness for CUDA graph replay").  Here one
// CTA of 1024 threads does it in three passes over topk_idx:
//   1. each warp owns a contiguous segment of the flat (t*k + j) array and
//      counts it into its own row of a [32][E] shared-memory histogram
//      (__match_any_sync groups equal experts; one leader lane adds the group);
//   2. a column scan over the 32 warp rows plus a block-wide scan over experts
//      give counts, offsets and, per warp, the first slot of each expert;
//   3. each warp re-walks its segment in order and scatters: slot = base +
//      rank among equal experts of lower lane, so within an expert the flat
//      order is kept (a stable counting sort).
#include "common.cuh"

#include <climits>

namespace mm {

__device__ __forceinline__ int block_exclusive_scan_1024(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int res = (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(1024, 1) route_kernel(const RouteParams p) {
  extern __shared__ int32_t hist[];   // [32][E]
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_bad;

  const int E = p.E, A = p.A;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(p.ws + p.L.ctrl);
  int32_t* counts = reinterpret_cast<int32_t*>(p.ws + p.L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(p.ws + p.L.offsets);
  int32_t* items = reinterpret_cast<int32_t*>(p.ws + p.L.items);
  uint32_t* arrival = reinterpret_cast<uint32_t*>(p.ws + p.L.arrival);
  uint32_t* l1_done = reinterpret_cast<uint32_t*>(p.ws + p.L.l1_done);
  int32_t* perm = reinterpret_cast<int32_t*>(p.ws + p.L.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(p.ws + p.L.inv);

  // -- reset: status, abort flag, tile counter, readiness counters
  for (int i = tid; i < kCtrlWords; i += blockDim.x) ctrl[i] = 0u;
  for (int i = tid; i < E; i += blockDim.x) { arrival[i] = 0u; l1_done[i] = 0u; }
  for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] = 0;
  if (tid == 0) s_bad = INT_MAX;
  __syncthreads();

  const int seg = (A + 31) / 32;
  const int beg = min(warp * seg, A);
  const int end = min(beg + seg, A);
  int32_t* myhist = hist + warp * E;

  // -- pass 1: per-warp histograms
  for (int base = beg; base < end; base += 32) {
    const int f = base + lane;
    const bool in = f < end;
    const int e = in ? p.topk_idx[f] : -1;
    const bool ok = in && e >= 0 && e < E;
    if (in && !ok && e != -1) atomicMin(&s_bad, f);
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
    if (ok && lane == __ffs(peers) - 1) myhist[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  if (s_bad != INT_MAX) {
    if (tid == 0) {
      ctrl[kStatus] = (uint32_t)MM_ERR_BAD_INDEX;
      ctrl[kErrInfo] = (uint32_t)s_bad;
      ctrl[kAbort] = 1u;
    }
    return;
  }

  // -- pass 2: counts, offsets, per-warp bases, N-block table
  int cnt = 0;
  if (tid < E) {
    for (int w = 0; w < 32; ++w) {
      const int c = hist[w * E + tid];
      hist[w * E + tid] = cnt;
      cnt += c;
    }
  }
  const int off = block_exclusive_scan_1024(cnt, s_warp);
  const int nb = n_blocks(cnt, p.max_n);
  const int nb_off = block_exclusive_scan_1024(nb, s_warp);
  if (tid < E) {
    counts[tid] = cnt;
    offsets[tid] = off;
    items[tid] = nb_off;
    for (int w = 0; w < 32; ++w) hist[w * E + tid] += off;
    if (tid == E - 1) {
      offsets[E] = off + cnt;
      items[E] = nb_off + nb;
    }
  }
  __syncthreads();

  // -- pass 3: stable scatter
  for (int base = beg; base < end; base += 32) {
    const int f = base + lane;
    const bool in = f < end;
    const int e = in ? p.topk_idx[f] : -1;
    const bool ok = in && e >= 0;
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (ok) {
      const int slot = myhist[e] + rank;
      perm[slot] = f;
      inv[f] = slot;
    } else if (in) {
      inv[f] = -1;
    }
    __syncwarp();
    if (ok && lane == __ffs(peers) - 1) myhist[e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace mm
