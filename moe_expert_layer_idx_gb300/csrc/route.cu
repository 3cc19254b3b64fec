// Routing: per-launch reset, expert histogram, prefix scan, stable
// permutation, and the token-block tables of the persistent kernel (each
// expert's first block, and one record per block).
//
// The pages' kernel does this as the first part of its dispatch: it clears
// its workspace, counts the assignments of each expert and records, for every
// slot, which (token, k) pair it came from (DeepGEMM SM90 MegaMoE dev log,
// Phase 2 entry); and it resets its readiness flags on every launch (DeepGEMM
// PR #451, "Reset MegaMoE combine readiness for CUDA graph replay").
//
// The flat (t*k + j) array is cut into contiguous pieces, each walked in
// order by one warp, 32 entries at a time:
//   1. count: the warp adds its piece into its own row of a [32][E]
//      shared-memory histogram (__match_any_sync groups equal experts; one
//      leader lane adds the group);
//   2. scan: counts, offsets and, for every piece, the first slot of each
//      expert (all earlier pieces' counts of that expert come before it);
//   3. scatter: the warp re-walks its piece in order; slot = the piece's base
//      + rank among equal experts of lower lane, so within an expert the flat
//      order is kept (a stable counting sort).
// Up to 2048 assignments, one 1024-thread CTA does all three passes
// (route_kernel).  Larger batches are split into chunks of about 1024
// assignments, one CTA each: route_count_kernel writes each chunk's expert
// counts, route_scan_kernel (one CTA) scans them over chunks and experts, and
// route_scatter_kernel recounts its chunk per warp and scatters.  One SM walks
// about 0.5 assignments per cycle, so a single CTA takes ~130 us for a batch
// of 65,536; split, the passes take a few microseconds.
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

// Both walks go 32 entries at a time, in order; the entries of kAhead such
// steps are loaded together first.
constexpr int kAhead = 8;

// Pass 1 over the flat entries [beg, end): adds each expert's count into
// myhist (this warp's row).  The smallest flat index holding a value outside
// [-1, E) goes to *s_bad (shared, atomicMin).
__device__ __forceinline__ void count_piece(const int32_t* topk_idx, int beg, int end, int E, int32_t* myhist,
                                            int* s_bad, int lane) {
  for (int base = beg; base < end; base += 32 * kAhead) {
    int ev[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int f = base + 32 * u + lane;
      ev[u] = f < end ? __ldg(topk_idx + f) : -1;
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int f = base + 32 * u + lane;
      const bool in = f < end;
      const int e = ev[u];
      const bool ok = in && e >= 0 && e < E;
      if (in && !ok && e != -1) atomicMin(s_bad, f);
      const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
      if (ok && lane == __ffs(peers) - 1) myhist[e] += __popc(peers);
      __syncwarp();
    }
  }
}

// Pass 3 over [beg, end): myhist[e] holds the next slot of expert e for this
// piece; writes perm and inv (-1 for an empty slot).
__device__ __forceinline__ void scatter_piece(const int32_t* topk_idx, int beg, int end, int32_t* myhist,
                                              int32_t* perm, int32_t* inv, int lane) {
  for (int base = beg; base < end; base += 32 * kAhead) {
    int ev[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int f = base + 32 * u + lane;
      ev[u] = f < end ? __ldg(topk_idx + f) : -1;
    }
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int f = base + 32 * u + lane;
      const bool in = f < end;
      const int e = ev[u];
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
}

// Status, abort flag, tile counter and readiness counters of the launch.
__device__ __forceinline__ void reset_control(const RouteParams& p) {
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(p.ws + p.L.ctrl);
  uint32_t* arrival = reinterpret_cast<uint32_t*>(p.ws + p.L.arrival);
  uint32_t* l1_done = reinterpret_cast<uint32_t*>(p.ws + p.L.l1_done);
  for (int i = threadIdx.x; i < kCtrlWords; i += blockDim.x) ctrl[i] = 0u;
  for (int i = threadIdx.x; i < p.E; i += blockDim.x) { arrival[i] = 0u; l1_done[i] = 0u; }
}

__device__ __forceinline__ void report_bad_index(const RouteParams& p, int first_bad) {
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(p.ws + p.L.ctrl);
  ctrl[kStatus] = (uint32_t)MM_ERR_BAD_INDEX;
  ctrl[kErrInfo] = (uint32_t)first_bad;
  ctrl[kAbort] = 1u;
}

// Counts, offsets and the token-block tables from the per-expert totals
// (thread e < E holds expert e's count): items[e] = the first token block of
// expert e, and blocks[b] = {e, items[e], offsets[e], counts[e]} for every
// block b of expert e, so that the layer kernel decodes a tile with one
// 16-byte load.  Returns expert tid's offset.
__device__ __forceinline__ int write_tables(const RouteParams& p, int cnt, int* s_warp) {
  int32_t* counts = reinterpret_cast<int32_t*>(p.ws + p.L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(p.ws + p.L.offsets);
  int32_t* items = reinterpret_cast<int32_t*>(p.ws + p.L.items);
  int4* blocks = reinterpret_cast<int4*>(p.ws + p.L.blocks);
  const int tid = threadIdx.x, E = p.E;
  const int off = block_exclusive_scan_1024(cnt, s_warp);
  const int nb = n_blocks(cnt, p.max_n);
  const int nb_off = block_exclusive_scan_1024(nb, s_warp);
  if (tid < E) {
    counts[tid] = cnt;
    offsets[tid] = off;
    items[tid] = nb_off;
    for (int b = 0; b < nb; ++b) blocks[nb_off + b] = make_int4(tid, nb_off, off, cnt);
    if (tid == E - 1) {
      offsets[E] = off + cnt;
      items[E] = nb_off + nb;
    }
  }
  return off;
}

// ---------------------------------------------------------------- one CTA
__global__ void __launch_bounds__(1024, 1) route_kernel(const RouteParams p) {
  extern __shared__ int32_t hist[];   // [32][E]
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_bad;

  const int E = p.E, A = p.A;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* perm = reinterpret_cast<int32_t*>(p.ws + p.L.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(p.ws + p.L.inv);

  reset_control(p);
  for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] = 0;
  if (tid == 0) s_bad = INT_MAX;
  __syncthreads();

  const int seg = (A + 31) / 32;
  const int beg = min(warp * seg, A);
  const int end = min(beg + seg, A);
  int32_t* myhist = hist + warp * E;

  count_piece(p.topk_idx, beg, end, E, myhist, &s_bad, lane);
  __syncthreads();
  if (s_bad != INT_MAX) {
    if (tid == 0) report_bad_index(p, s_bad);
    return;
  }

  // per-warp bases: expert e's slots of warp w follow those of warps < w
  int cnt = 0;
  if (tid < E) {
    for (int w = 0; w < 32; ++w) {
      const int c = hist[w * E + tid];
      hist[w * E + tid] = cnt;
      cnt += c;
    }
  }
  const int off = write_tables(p, cnt, s_warp);
  if (tid < E)
    for (int w = 0; w < 32; ++w) hist[w * E + tid] += off;
  __syncthreads();

  scatter_piece(p.topk_idx, beg, end, myhist, perm, inv, lane);
}

// ---------------------------------------------------------------- chunks
// The rhist region holds cnt[E][C] (expert-major: the count kernel writes
// each chunk's totals, the scan kernel replaces them by the chunk's first
// slot of the expert relative to the expert's offset), then bad[C].

__global__ void __launch_bounds__(1024, 1) route_count_kernel(const RouteParams p) {
  extern __shared__ int32_t hist[];   // [32][E]
  __shared__ int32_t s_bad;
  const int E = p.E, C = p.C, c = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* rh = reinterpret_cast<int32_t*>(p.ws + p.L.rhist);
  int32_t* bad = rh + (size_t)E * C;

  for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] = 0;
  if (tid == 0) s_bad = INT_MAX;
  __syncthreads();
  const int cbeg = min(c * p.chunk, p.A), cend = min(cbeg + p.chunk, p.A);
  const int seg = (cend - cbeg + 31) / 32;
  const int beg = min(cbeg + warp * seg, cend), end = min(beg + seg, cend);
  count_piece(p.topk_idx, beg, end, E, hist + warp * E, &s_bad, lane);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int tot = 0;
    for (int w = 0; w < 32; ++w) tot += hist[w * E + e];
    rh[(size_t)e * C + c] = tot;
  }
  if (tid == 0) bad[c] = s_bad;
}

__global__ void __launch_bounds__(1024, 1) route_scan_kernel(const RouteParams p) {
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_cnt[1024];
  __shared__ int32_t s_bad;
  const int E = p.E, C = p.C;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* rh = reinterpret_cast<int32_t*>(p.ws + p.L.rhist);
  const int32_t* bad = rh + (size_t)E * C;

  reset_control(p);
  if (tid == 0) s_bad = INT_MAX;
  __syncthreads();
  if (tid < C) atomicMin(&s_bad, bad[tid]);
  __syncthreads();
  if (s_bad != INT_MAX) {
    if (tid == 0) report_bad_index(p, s_bad);
    return;
  }

  // each expert's counts over the chunks (C <= 128: four 32-lane steps),
  // replaced by their exclusive prefix; the total is the expert's count
  for (int e = warp; e < E; e += 32) {
    int32_t* row = rh + (size_t)e * C;
    int v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = j * 32 + lane < C ? row[j * 32 + lane] : 0;
    int carry = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int x = v[j];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (j * 32 + lane < C) row[j * 32 + lane] = carry + x - v[j];
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_cnt[e] = carry;
  }
  __syncthreads();
  write_tables(p, tid < E ? s_cnt[tid] : 0, s_warp);
}

__global__ void __launch_bounds__(1024, 1) route_scatter_kernel(const RouteParams p) {
  extern __shared__ int32_t hist[];   // [32][E]
  __shared__ int32_t s_unused;
  const int E = p.E, C = p.C, c = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t* ctrl = reinterpret_cast<const uint32_t*>(p.ws + p.L.ctrl);
  if (ld_volatile(&ctrl[kStatus]) != 0u) return;      // a bad index was reported
  const int32_t* rh = reinterpret_cast<const int32_t*>(p.ws + p.L.rhist);
  const int32_t* offsets = reinterpret_cast<const int32_t*>(p.ws + p.L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(p.ws + p.L.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(p.ws + p.L.inv);

  for (int i = tid; i < 32 * E; i += blockDim.x) hist[i] = 0;
  if (tid == 0) s_unused = INT_MAX;
  __syncthreads();
  const int cbeg = min(c * p.chunk, p.A), cend = min(cbeg + p.chunk, p.A);
  const int seg = (cend - cbeg + 31) / 32;
  const int beg = min(cbeg + warp * seg, cend), end = min(beg + seg, cend);
  int32_t* myhist = hist + warp * E;
  count_piece(p.topk_idx, beg, end, E, myhist, &s_unused, lane);
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) {
    int run = offsets[e] + rh[(size_t)e * C + c];
    for (int w = 0; w < 32; ++w) {
      const int h = hist[w * E + e];
      hist[w * E + e] = run;
      run += h;
    }
  }
  __syncthreads();
  scatter_piece(p.topk_idx, beg, end, myhist, perm, inv, lane);
}

}  // namespace mm
