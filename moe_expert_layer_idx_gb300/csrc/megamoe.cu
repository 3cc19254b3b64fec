// The persistent fused MoE expert layer kernel for GB300 (sm_103a).
//
// One CTA per SM (grid sized by the host from the SM count minus a reserve,
// rounded down to even -- sglang PR #36657 "[Blackwell] Reserve SMs for
// DeepGEMM MegaMoE grid barriers", sections Root cause and Fix).  The
// dispatch below is a static grid-stride loop, so the layer is only sure to
// progress when every CTA is resident at once; the reserve keeps that true
// while another stream holds a few SMs.  Phases:
//
//  0. dispatch: every warp copies expert-sorted token rows into the workspace,
//     writes their UE8M0 scales into the token block's scale atoms, and bumps
//     that expert's arrival counter with a release.  The pages' dispatch pulls each token's row and scales from
//     whichever rank holds it and then releases a per-expert arrival count
//     (DeepGEMM SM90 MegaMoE dev log, Phase 2 entry); here every row is local.
//  1. tiles, warp-specialised, dynamically scheduled (see TileFeed):
//       warps 0 and 3, lane 0  TMA producers; they split each stage's boxes
//                              (in the thin tiles also its scale atoms, by bulk
//                              copies onto the same barrier);
//       warp 1, lane 0         MMA issuer: scale atoms -> TMEM (tcgen05.cp),
//                              then 4 x tcgen05.mma kind::mxf8f6f4 block_scale
//                              (K = 32 each) per 128-wide K stage;
//       warp 2                 scale loader of the 128-token tiles: copies each
//                              stage's ready-made scale atoms (token rows, both
//                              weight halves) with coalesced 16-byte loads;
//       warps 4-11             epilogue: warp w reads TMEM lanes 32(w%4)..+31,
//                              the two warps of a lane quarter split the columns.
//     The MMA puts up to 128 tokens of one expert on M (E4M3, operand A) and
//     256 weight rows on N (E2M1, operand B, 128-byte swizzled, packed FP4
//     widened to 8-bit containers by the 16U4_ALIGN16B tensor map).  Each MMA
//     instruction consumes 4 KB of FP4 weights, which keeps the tensor pipe's
//     per-instruction cost under the weight stream at decode batch sizes.
//     L1 tile (expert e, 128 intermediate features, a token block): B rows
//     [0,128) are the gate rows and [128,256) the up rows of those features, so
//     TMEM lane m holds both halves of token m; its epilogue thread applies the
//     clamp and SwiGLU, requantises each 32 features to E4M3 + UE8M0 in
//     registers, writes its l1_acts row, and the tile releases the expert's
//     L1-done count.  L2 tile (expert e, 256 hidden rows -- 128 for a tail --,
//     a token block) waits for that count, multiplies by the token's top-k
//     weight and writes fp32 rows indexed by the flat assignment (fp32, not
//     bf16: when a token's k contributions cancel, a bf16 rounding of each one
//     is large next to their sum).
// The combine, y[t] = bf16(sum_j of the weighted rows t*k + j, in ascending
// j), is a second, non-persistent kernel on the same stream (combine_kernel):
// the kernel boundary orders every L2 row before it, so the layer kernel has
// no whole-grid barrier, and the combine runs on every SM at HBM rate.  (The
// pages' kernel synchronises its grid after the epilogue and combines in the
// same kernel.)
//
// Every wait is bounded (global timer + abort flag): a wait that runs out
// records MM_ERR_TIMEOUT with the SM and the wait site, raises the abort flag,
// and the CTA drains its own in-flight copies and MMAs, frees its TMEM and
// returns -- the pages' kernel likewise reports a grid-sync timeout with the
// SM, the thread and the barrier's index (digest of PR #36657, 功能与动机)
// instead of hanging.
// All counters are reset by the routing kernel of the same launch, never
// keyed on %gridid (DeepGEMM PR #451).
#include "common.cuh"
#include "numerics.cuh"

namespace mm {

struct Tile {
  int layer;   // 1 or 2
  int e;       // expert
  int nb;      // weight block: 128 intermediate features (L1) or 256 hidden rows (L2)
  int r0;      // first slot of the token block
  int rows;    // tokens in the block (<= 128)
  int m16;     // rows rounded up to 16: token rows loaded
  int n;       // MMA N: 256, or 128 for a hidden tail
  int ks;      // K stages
  int tag;     // tile index (reported with a wait that gives up)
  int blk;     // global index of the token block (its scale atoms)
};

// Tiles are numbered L1 first, then L2; within a layer expert-major, then the
// weight block, then the token block, so the token blocks that share a weight
// tile run close together and find it in L2.
// An expert's tiles are [items[e] * NB, items[e + 1] * NB), so tt / NB is one
// of its token blocks, whose record names the expert and its tables.
__device__ __forceinline__ int4 tile_record(int t, int nL1, const ForwardParams& p) {
  const bool l1 = t < nL1;
  const int tt = l1 ? t : t - nL1;
  return __ldg(reinterpret_cast<const int4*>(p.ws + p.L.blocks) + tt / (l1 ? p.mt1 : p.mt2));
}
__device__ __forceinline__ void decode_tile(int t, int nL1, const ForwardParams& p, const int4 rec, Tile& ti) {
  const bool l1 = t < nL1;
  const int tt = l1 ? t : t - nL1;
  const int NB = l1 ? p.mt1 : p.mt2;
  const int e = rec.x, i0 = rec.y, cnt = rec.w;
  const int mbk = n_blocks(cnt, p.max_rows);    // token blocks of this expert
  const int local = tt - i0 * NB;
  const int nb = local / mbk;
  const int mb = local - nb * mbk;
  const int rpb = (cnt + mbk - 1) / mbk;
  const int start = mb * rpb;
  ti.layer = l1 ? 1 : 2;
  ti.e = e;
  ti.nb = nb;
  ti.r0 = rec.z + start;
  ti.rows = min(rpb, cnt - start);
  ti.m16 = (ti.rows + 15) & ~15;
  ti.n = l1 ? kTileN : min(kTileN, p.H - nb * kTileN);
  ti.ks = l1 ? p.ks1 : p.ks2;
  ti.tag = t & 0xFFFFFF;
  ti.blk = i0 + mb;
}

// Where slot s's row sits among a layer's token-scale atoms (slot s belongs to
// expert e; token blocks as the routing kernels made them: n_blocks(count,
// max_rows) balanced blocks per expert, `halves` 128-row halves each), packed
// as (block half << 9) | byte position within the atom; the byte offset of
// stage j is then atom_offset(packed, S) + j * kAtomBytes (S stages per row).
__device__ __forceinline__ uint32_t token_atom_slot(const ForwardParams& p, const int32_t* items,
                                                    const int32_t* counts, const int32_t* offsets, int e, int s,
                                                    int halves) {
  const int cnt = __ldg(counts + e);
  const int mbk = n_blocks(cnt, p.max_rows);
  const int rpb = (cnt + mbk - 1) / mbk;
  const int i = s - __ldg(offsets + e);
  const int mb = i / rpb, row = i - mb * rpb;
  const int b = __ldg(items + e) + mb;
  return ((uint32_t)(b * halves + (row >> 7)) << 9) | (uint32_t)atom_pos(row & 127);
}
__device__ __forceinline__ size_t atom_offset(uint32_t packed, int S) {
  return (size_t)(packed >> 9) * S * kAtomBytes + (packed & 511u);
}

// Dynamic tile schedule.  Producer 0 claims the next tile index from a global
// counter (reset by the routing kernel of the same launch), decodes it and
// publishes the decoded tile in a small shared-memory ring; every other role
// takes the tiles from the ring in the same order.  layer == 0 ends the
// stream.  The atomic for the next tile is issued as soon as the current one
// is published, so its round trip overlaps the current tile's loads.
// Tiles are claimed in increasing index order (all L1 tiles before any L2
// tile, expert-major) and L1 tiles wait only for the dispatch, so the oldest
// unfinished L1 tile is always either running or held (claimed ahead) by a CTA
// whose running tile is an L1 tile or an L2 tile of a larger index: no cycle of
// waits can form.
// In a pair, the even CTA's producer 0 claims for both: it also writes each
// tile into the odd CTA's ring and arrives on that ring's barrier; the odd
// CTA's readers take tiles from their own ring (acquiring at cluster scope)
// and free the slot on the even CTA's barrier, which counts both CTAs' readers.
struct TileFeed {
  Tile* ring;
  uint64_t* full;
  uint64_t* empty;
  uint32_t i = 0;
  int ahead = -1;              // producer 0: index claimed for the next publication
  int4 ahead_rec;              // and its token-block record, once loaded ahead (rec_ready)
  bool rec_ready = false;
  bool peer = false;           // a reader of the odd CTA of a pair
  uint32_t empty_cl = 0;       // odd CTA: cluster address of the even CTA's empty[0]
  uint32_t peer_ring_cl = 0;   // even CTA's producer 0: the odd CTA's ring[0] and full[0]
  uint32_t peer_full_cl = 0;
  __device__ TileFeed(Tile* r, uint64_t* f, uint64_t* e) : ring(r), full(f), empty(e) {}
  // The pair's wiring: rank 0 publishes to rank 1; rank 1 frees rank 0's slots.
  __device__ void pair(uint32_t rank) {
    if (rank == 0) {
      peer_ring_cl = cluster_addr(smem_u32(ring), 1);
      peer_full_cl = cluster_addr(smem_u32(full), 1);
    } else {
      peer = true;
      empty_cl = cluster_addr(smem_u32(empty), 0);
    }
  }
  __device__ bool wait_full(uint32_t slot, uint32_t ph, uint32_t* ctrl, unsigned long long to) {
    return peer ? mbar_wait<true>(smem_u32(&full[slot]), ph, ctrl, to, kSiteTileRing << 24)
                : mbar_wait(smem_u32(&full[slot]), ph, ctrl, to, kSiteTileRing << 24);
  }
  __device__ void release(uint32_t slot) {
    if (peer) mbar_arrive_cluster(empty_cl + 8u * slot);
    else mbar_arrive(smem_u32(&empty[slot]));
  }

  // Producer 0: claim, decode, publish.  Returns false at the end of the stream or on abort (ok = false).
  __device__ bool claim(uint32_t* counter, int total, int nL1, const ForwardParams& p, uint32_t* ctrl,
                        unsigned long long to, bool& ok, Tile& ti) {
    const uint32_t slot = i % kTileRing, ph = (i / kTileRing) & 1u;
    ++i;
    if (!mbar_wait<true>(smem_u32(&empty[slot]), ph ^ 1u, ctrl, to, kSiteTileRing << 24)) { ok = false; return false; }
    const int t = ahead >= 0 ? ahead : (int)atomicAdd(counter, 1u);
    if (t < total) decode_tile(t, nL1, p, rec_ready ? ahead_rec : tile_record(t, nL1, p), ti);
    else ti.layer = 0;
    rec_ready = false;
    ring[slot] = ti;
    if (peer_ring_cl != 0) {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(&ti);
#pragma unroll
      for (int q = 0; q < (int)(sizeof(Tile) / 4); ++q) st_cluster_u32(peer_ring_cl + slot * sizeof(Tile) + 4 * q, w[q]);
      mbar_arrive_cluster(peer_full_cl + 8u * slot);   // release: the remote writes come first
    }
    mbar_arrive(smem_u32(&full[slot]));          // release: the tile is visible to the readers
    ahead = t < total ? (int)atomicAdd(counter, 1u) : -1;   // consumed at the next claim
    return ti.layer != 0;
  }
  // Producer 0, part-way through the current tile's loads (the atomic for the
  // next index has returned by then): the next tile's record is loaded now, so
  // the next claim decodes it without a memory round trip.
  __device__ void prefetch(int total, int nL1, const ForwardParams& p) {
    if (!rec_ready && ahead >= 0 && ahead < total) {
      ahead_rec = tile_record(ahead, nL1, p);
      rec_ready = true;
    }
  }
  // One reading thread.
  __device__ bool take(uint32_t* ctrl, unsigned long long to, bool& ok, Tile& ti) {
    const uint32_t slot = i % kTileRing, ph = (i / kTileRing) & 1u;
    ++i;
    if (!wait_full(slot, ph, ctrl, to)) { ok = false; return false; }
    ti = ring[slot];
    release(slot);
    return ti.layer != 0;
  }
  // A whole warp: lane 0 waits, every lane then observes the completed phase
  // itself (it stays complete until this warp's arrival frees the slot) and
  // reads the tile; lane 0 frees the slot after the warp has read it.
  __device__ bool take_warp(int lane, uint32_t* ctrl, unsigned long long to, bool& ok, Tile& ti) {
    const uint32_t slot = i % kTileRing, ph = (i / kTileRing) & 1u;
    ++i;
    bool w = true;
    if (lane == 0) w = wait_full(slot, ph, ctrl, to);
    w = __shfl_sync(0xffffffffu, w, 0);
    if (!w) { ok = false; return false; }
    if (peer) (void)mbar_try_wait<true>(smem_u32(&full[slot]), ph);
    else (void)mbar_try_wait(smem_u32(&full[slot]), ph);
    ti = ring[slot];
    __syncwarp();
    if (lane == 0) release(slot);
    return ti.layer != 0;
  }
};

__device__ __forceinline__ uint32_t l1_tiles_of(const int32_t* items, int e, int mt1) {
  return (uint32_t)((__ldg(items + e + 1) - __ldg(items + e)) * mt1);
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}


template <class V>
__global__ void __launch_bounds__(kThreads, 1)
megamoe_kernel(const __grid_constant__ CUtensorMap tm_w1, const __grid_constant__ CUtensorMap tm_w2,
               const __grid_constant__ CUtensorMap tm_xs16, const __grid_constant__ CUtensorMap tm_xs128,
               const __grid_constant__ CUtensorMap tm_l1a16, const __grid_constant__ CUtensorMap tm_l1a128,
               const __grid_constant__ ForwardParams p) {
  constexpr int kStages = V::kStages;     // ring slots
  constexpr int kSub = V::kSub;           // sub-stages per slot; sub-stage buffers are indexed slot * kSub + u
  constexpr int kABytes = V::kABytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kSubs = kStages * kSub;
  uint8_t* sA = sm;                                   // [kSubs] token rows
  uint8_t* sB = sA + kSubs * kABytes;                 // [kSubs] weight rows
  uint8_t* sSFA = sB + kSubs * V::kBStageBytes;       // [kSubs] token scale atom
  uint8_t* sSFB = sSFA + kSubs * kSFABytes;           // [kSubs] two weight scale atoms
  float* sX = reinterpret_cast<float*>(sSFB + kSubs * kSFBBytes);   // [kEpiWarps] transpose buffers
  float* sAmax = reinterpret_cast<float*>(sSFB + kSubs * kSFBBytes + V::kXposeBytes);   // kF8B: [4][2][32]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sSFB + kSubs * kSFBBytes + V::kXposeBytes + V::kAmaxBytes);
  uint64_t* full = bars;                     // [kStages] both producers' TMA bytes + the scale loader's atoms
  uint64_t* empty = bars + kStages;          // [kStages] MMAs reading the stage are done
  uint64_t* tfull = bars + 2 * kStages;      // accumulator ready
  uint64_t* tempty = tfull + 1;              // accumulator drained (every epilogue warp)
  uint64_t* drain = tempty + 1;              // final MMA drain
  uint64_t* tile_full = drain + 1;           // [kTileRing] tile index published
  uint64_t* tile_empty = tile_full + kTileRing;   // [kTileRing] read by every consumer role
  uint64_t* pfull = tile_empty + kTileRing;       // kF8B: [2] partial accumulator written
  uint64_t* pempty = pfull + 2;                   // kF8B: [2] partial accumulator taken by every epilogue warp
  // tmem base, stages consumed (MMA), stages issued (producer 0), status read at the start, stages
  // armed (scale loader), stages issued (producer 1)
  uint32_t* s_misc = reinterpret_cast<uint32_t*>(pempty + 2);
  int32_t* s_vote = reinterpret_cast<int32_t*>(s_misc + 8);    // epilogue votes [2][kEpiWarps]
  Tile* s_tiles = reinterpret_cast<Tile*>(s_vote + 2 * kEpiWarps);   // [kTileRing] claimed tiles

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int G = V::kCtas;                     // CTA group of every tcgen05 instruction
  const uint32_t crank = V::kPair ? cluster_rank() : 0u;
  const bool leader = crank == 0;                 // the CTA that issues the MMAs
  uint32_t* ctrl = reinterpret_cast<uint32_t*>(p.ws + p.L.ctrl);
  // A nonzero status (the routing rejected the input) ends the launch.  The
  // two CTAs of a pair must take the same decision, because each blocks in the
  // collective TMEM allocation and the cluster barriers until the other comes:
  // they both go through the prologue and follow the even CTA's reading.
  const uint32_t status0 = ld_volatile(&ctrl[kStatus]);
  if constexpr (!V::kPair) {
    if (status0 != 0u) return;
  }

  const int32_t* counts = reinterpret_cast<const int32_t*>(p.ws + p.L.counts);
  const int32_t* offsets = reinterpret_cast<const int32_t*>(p.ws + p.L.offsets);
  const int32_t* items = reinterpret_cast<const int32_t*>(p.ws + p.L.items);
  uint32_t* arrival = reinterpret_cast<uint32_t*>(p.ws + p.L.arrival);
  uint32_t* l1_done = reinterpret_cast<uint32_t*>(p.ws + p.L.l1_done);
  const int32_t* perm = reinterpret_cast<const int32_t*>(p.ws + p.L.perm);
  uint8_t* xs = p.ws + p.L.xs;
  uint8_t* xs_sf = p.ws + p.L.xs_sf;
  uint8_t* l1a = p.ws + p.L.l1a;
  uint8_t* l1a_sf = p.ws + p.L.l1a_sf;
  float* stage_out = reinterpret_cast<float*>(p.ws + p.L.stage);
  const unsigned long long to = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // producers (+ the scale loader), of both CTAs of a pair
      mbar_init(&full[s], (V::kSLWarp ? 2 + 1 : 2) * G);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiWarps * G);
    mbar_init(drain, 1);
    for (int i = 0; i < kTileRing; ++i) {
      mbar_init(&tile_full[i], 1);
      mbar_init(&tile_empty[i], kTileReaders * G);   // a pair's odd CTA has as many readers as the even one
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], kEpiWarps);
    }
    for (int i = 1; i < 8; ++i) s_misc[i] = 0;
    s_misc[3] = status0;                        // read by the odd CTA of a pair
    fence_mbar_init();
    prefetch_tensormap(&tm_w1);
    prefetch_tensormap(&tm_w2);
    prefetch_tensormap(&tm_xs16);
    prefetch_tensormap(&tm_xs128);
    prefetch_tensormap(&tm_l1a16);
    prefetch_tensormap(&tm_l1a128);
  }
  if (warp == 1) {
    tc_alloc<G>(smem_u32(&s_misc[0]), kTmemCols);   // a pair allocates in both CTAs together
    tc_relinquish<G>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (V::kPair) cluster_sync();          // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = s_misc[0];
  bool skip = false;                               // (outside a pair the status was checked above)
  if constexpr (V::kPair) skip = ld_cluster_u32(cluster_addr(smem_u32(&s_misc[3]), 0)) != 0u;
  if (!skip) {

  // ------------------------------------------------------------ 0. dispatch
  if (!V::kBf16 && p.x_bf16 != nullptr) {
    // bf16 activations of the FP8 x FP4 layer: one warp per token reads its row once; lane b quantises
    // 32-element blocks b, b + 32, ... (E4M3 + UE8M0 by the scale rule of the
    // L1 epilogue) and writes each block to every slot of the token, then each
    // slot's expert arrival count is released.
    const int32_t* inv = reinterpret_cast<const int32_t*>(p.ws + p.L.inv);
    const int H = p.H, k = p.k, nblk = H / 32;
    for (int t = blockIdx.x * (kThreads / 32) + warp; t < p.T; t += gridDim.x * (kThreads / 32)) {
      int my_e = -1, my_slot = -1;                   // lane j < k: slot j of the token
      uint32_t my_atom = 0;                          // and its row's place among the scale atoms
      if (lane < k) {
        my_e = __ldg(p.topk_idx + (size_t)t * k + lane);
        if (my_e >= 0) {
          my_slot = __ldg(inv + (size_t)t * k + lane);
          my_atom = token_atom_slot(p, items, counts, offsets, my_e, my_slot, V::kCtas);
        }
      }
      const uint4* src = reinterpret_cast<const uint4*>(p.x_bf16 + (size_t)t * H);
      // every lane runs the same iterations, so slot j's row and atom place can be
      // fetched from lane j by a shuffle at the point of use
      for (int b0 = 0; b0 < nblk; b0 += 32) {
        const int b = b0 + lane;
        const bool act = b < nblk;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        int sc = 0;
        if (act) {
          float v[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 q = __ldg(src + 4 * b + c);
            const uint32_t u4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[8 * c + 2 * i] = __uint_as_float(u4[i] << 16);             // bf16 -> fp32 is exact
              v[8 * c + 2 * i + 1] = __uint_as_float(u4[i] & 0xFFFF0000u);
            }
          }
          float a = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
          sc = block_scale_exp<true>(a);
          const float inv_s = exp2_neg(sc);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            w[i] = e4m3_code(v[4 * i] * inv_s) | (e4m3_code(v[4 * i + 1] * inv_s) << 8) |
                   (e4m3_code(v[4 * i + 2] * inv_s) << 16) | (e4m3_code(v[4 * i + 3] * inv_s) << 24);
        }
        for (int j = 0; j < k; ++j) {
          const int slot = __shfl_sync(0xffffffffu, my_slot, j);
          const uint32_t at = __shfl_sync(0xffffffffu, my_atom, j);
          if (act && slot >= 0) {
            uint4* d4 = reinterpret_cast<uint4*>(xs + (size_t)slot * H + 32 * b);
            d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
            d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            xs_sf[atom_offset(at, H / 128) + (size_t)(b >> 2) * kAtomBytes + (b & 3)] = (uint8_t)(sc + 127);
          }
        }
      }
      fence_proxy_async_global();
      __threadfence();
      __syncwarp();
      if (my_e >= 0) red_release_add(&arrival[my_e], 1u);
    }
  } else {
    const int nvalid = __ldg(offsets + p.E);
    const int H = p.H;
    constexpr int esz = V::kBf16 ? 2 : 1;          // bytes per activation element
    const int nvec = H * esz / 16, nsf = H / 128;
    // A warp copies its slots s0, s0 + G, ... in batches of kBatch: the batch's
    // perm and expert entries are loaded together, each row with up to 16
    // loads in flight per lane, and one fence covers the whole batch before
    // its arrival counts are released.
    constexpr int kBatch = 4;
    const int G = gridDim.x * (kThreads / 32);
    for (int s0 = blockIdx.x * (kThreads / 32) + warp; s0 < nvalid; s0 += kBatch * G) {
      int fs[kBatch], es[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) fs[u] = s0 + u * G < nvalid ? __ldg(perm + s0 + u * G) : -1;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) es[u] = fs[u] >= 0 ? __ldg(p.topk_idx + fs[u]) : -1;
      // the rows go two at a time: both rows' loads (up to 8 per lane each) in flight together
#pragma unroll
      for (int u0 = 0; u0 < kBatch; u0 += 2) {
        const bool h0 = fs[u0] >= 0, h1 = fs[u0 + 1] >= 0;   // warp-uniform
        const uint4* src0 = reinterpret_cast<const uint4*>(p.x + (size_t)(h0 ? fs[u0] / p.k : 0) * H * esz);
        const uint4* src1 = reinterpret_cast<const uint4*>(p.x + (size_t)(h1 ? fs[u0 + 1] / p.k : 0) * H * esz);
        uint4* dst0 = reinterpret_cast<uint4*>(xs + (size_t)(s0 + u0 * G) * H * esz);
        uint4* dst1 = reinterpret_cast<uint4*>(xs + (size_t)(s0 + (u0 + 1) * G) * H * esz);
        for (int c0 = lane; c0 < nvec; c0 += 32 * 8) {
          uint4 v0[8], v1[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (h0 && c0 + 32 * i < nvec) v0[i] = __ldg(src0 + c0 + 32 * i);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (h1 && c0 + 32 * i < nvec) v1[i] = __ldg(src1 + c0 + 32 * i);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (h0 && c0 + 32 * i < nvec) dst0[c0 + 32 * i] = v0[i];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (h1 && c0 + 32 * i < nvec) dst1[c0 + 32 * i] = v1[i];
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (fs[u] < 0) continue;                      // warp-uniform
        const int s = s0 + u * G;
        const int t = fs[u] / p.k;
        if constexpr (V::kF8B) {
          // fp32 scale per 128 elements: rows of H / 32 bytes, in slot order
          const uint32_t* ssf = reinterpret_cast<const uint32_t*>(p.x_sf + (size_t)t * (H / 32));
          uint32_t* dsf = reinterpret_cast<uint32_t*>(xs_sf + (size_t)s * (H / 32));
          for (int c = lane; c < nsf; c += 32) dsf[c] = __ldg(ssf + c);
        } else if constexpr (!V::kBf16) {
          // the 4 UE8M0 bytes of stage c go to the row's place in the block's stage-c atom
          const uint32_t* ssf = reinterpret_cast<const uint32_t*>(p.x_sf + (size_t)t * (H / 32));
          uint8_t* da = xs_sf + atom_offset(token_atom_slot(p, items, counts, offsets, es[u], s, V::kCtas), nsf);
          for (int c = lane; c < nsf; c += 32) *reinterpret_cast<uint32_t*>(da + (size_t)c * kAtomBytes) = __ldg(ssf + c);
        }
      }
      fence_proxy_async_global();
      __threadfence();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (es[u] >= 0) red_release_add(&arrival[es[u]], 1u);
      }
    }
  }

  const int nItems = __ldg(items + p.E);
  const int nL1 = nItems * p.mt1;
  const int total = nL1 + nItems * p.mt2;

  // ------------------------------------------------------------ 1. tiles
  if (warp == 0 || warp == 3) {
    if (lane == 0) {
      // ---------------- TMA producers
      // One thread issues TMA at a limited rate, so two threads share each
      // stage: producer `pid` loads weight rows [128*pid, 128*pid + 128) of the
      // tile (L1: the gate rows, then the up rows) and the 16-row token boxes j
      // with j % 2 == pid (a single 128-row token box goes to producer 0), and
      // arms the stage's barrier with its own bytes.
      // In a pair, CTA r loads token rows [128r, 128r + 128) of the block and
      // weight rows [128r, 128r + 128) of the tile (one box, producer 0; a
      // single 128-row token box goes to producer 1), and every load of both
      // CTAs completes on the even CTA's barrier.
      const int pid = warp == 0 ? 0 : 1;
      uint32_t stage = 0, phase = 0, issued = 0;
      int ready_key = -1;            // (layer, expert) whose dependency was last seen satisfied
      bool ok = true;
      TileFeed feed(s_tiles, tile_full, tile_empty);
      if constexpr (V::kPair) feed.pair(crank);
      const bool claimer = pid == 0 && leader;
      while (ok) {
        Tile ti;
        const bool more = claimer ? feed.claim(&ctrl[kNextTile], total, nL1, p, ctrl, to, ok, ti)
                                  : feed.take(ctrl, to, ok, ti);
        if (!more) break;
        const uint32_t tag = (uint32_t)ti.tag;
        const int key = ti.e * 2 + ti.layer - 1;
        if (key != ready_key) {
          if (ti.layer == 1)
            ok = counter_wait(&arrival[ti.e], (uint32_t)__ldg(counts + ti.e), ctrl, to, (kSiteArrival << 24) | tag);
          else
            ok = counter_wait(&l1_done[ti.e], G * l1_tiles_of(items, ti.e, p.mt1), ctrl, to,
                              (kSiteL1Done << 24) | tag);
          if (!ok) break;
          fence_proxy_async_global();
          ready_key = key;
        }
        const int tr = (int)crank * kTileM;                       // this CTA's first row of the block
        const int rows = max(0, min(ti.rows - tr, kTileM));
        const int m16 = (rows + 15) & ~15;
        const int r0 = ti.r0 + tr;
        const bool full_box = V::kARows == kTileM && p.a_box128 && m16 == kTileM;
        const int box_pid = V::kPair ? 1 : 0;                    // producer of a single 128-row token box
        const int nbox = m16 / 16;
        const int my_a_bytes = full_box ? (pid == box_pid ? kABytes : 0) : ((nbox + 1 - pid) / 2) * 16 * kBlockK;
        const bool my_b = V::kPair ? pid == 0 : (pid == 0 || ti.n > 128);
        // scale atoms by bulk copy: each producer its weight half's atoms, producer 1 the token atoms
        // (producer 0 issues the single 128-row token box)
        constexpr bool kAtoms = !V::kNoSF && !V::kSLWarp;
        const int sf_bytes = kAtoms ? (my_b ? kAtomBytes : 0) + (pid == 1 ? kAtomBytes : 0) : 0;
        const uint32_t bytes = (uint32_t)((my_b ? V::kWeightBoxTx : 0) + my_a_bytes + sf_bytes);   // per K stage
        const CUtensorMap* tm_b = ti.layer == 1 ? &tm_w1 : &tm_w2;
        const CUtensorMap* tm_a = ti.layer == 1 ? (full_box ? &tm_xs128 : &tm_xs16)
                                                : (full_box ? &tm_l1a128 : &tm_l1a16);
        const int bsel = V::kPair ? (int)crank : pid;             // which 128-row half of the weight tile
        const int b_row = ti.layer == 1 ? ti.e * 2 * p.I + ti.nb * kL1Feat + bsel * p.I
                                        : ti.e * p.H + ti.nb * kTileN + bsel * 128;
        // stage 0 of this tile's weight-half atoms ([row / 128][K / 128]) and token atoms ([block][K / 128])
        const uint8_t* w_atoms = (ti.layer == 1 ? p.w1_sf : p.w2_sf) + (size_t)(b_row / 128) * ti.ks * kAtomBytes;
        const uint8_t* t_atoms = (ti.layer == 1 ? xs_sf : l1a_sf) + (size_t)ti.blk * ti.ks * kAtomBytes;
        for (int kk0 = 0; kk0 < ti.ks; kk0 += kSub) {
          const int nsub = min(kSub, ti.ks - kk0);
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, ctrl, to, (kSiteEmpty << 24) | tag)) { ok = false; break; }
          const uint32_t fb = smem_u32(&full[stage]);
          const uint32_t fbar = V::kPair ? cluster_addr(fb, 0) : fb;
          if constexpr (V::kPair) mbar_arrive_expect_tx_cluster(fbar, bytes * (uint32_t)nsub);
          else mbar_arrive_expect_tx(fbar, bytes * (uint32_t)nsub);
          if constexpr (kAtoms) {
            // the slot's nsub stages of an atom sequence are contiguous on both sides
            const uint32_t nb_sf = (uint32_t)(nsub * kAtomBytes);
            if (my_b)
              bulk_load(smem_u32(sSFB + stage * kSub * kSFBBytes + bsel * kSub * kAtomBytes),
                        w_atoms + (size_t)kk0 * kAtomBytes, nb_sf, fbar);
            if (pid == 1)
              bulk_load(smem_u32(sSFA + stage * kSub * kSFABytes), t_atoms + (size_t)kk0 * kAtomBytes, nb_sf, fbar);
          }
          for (int u = 0; u < nsub; ++u) {
            const int gs = stage * kSub + u;
            const uint32_t a_dst = smem_u32(sA + gs * kABytes);
            const uint32_t b_dst = smem_u32(sB + gs * V::kBStageBytes) + (uint32_t)(V::kPair ? 0 : pid * 128 * kBlockK);
            const int kx = (kk0 + u) * V::kKStage;
            auto load = [&](uint32_t dst, const CUtensorMap* m, int y) {
              if constexpr (V::kPair) tma_load_2d_pair(dst, m, fbar, kx, y);
              else tma_load_2d(dst, m, fbar, kx, y);
            };
            if (my_b) load(b_dst, tm_b, b_row);
            if (full_box) {
              if (pid == box_pid) load(a_dst, tm_a, r0);
            } else {
              for (int j = pid; j < nbox; j += 2) load(a_dst + j * 16 * kBlockK, tm_a, r0 + 16 * j);
            }
          }
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
          if (claimer && kk0 == 2 * kSub) feed.prefetch(total, nL1, p);
        }
      }
      s_misc[2 + 3 * pid] = issued;     // s_misc[2] (producer 0), s_misc[5] (producer 1)
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (in a pair: the even CTA's, for both)
      // Stage s's descriptors are stage 0's plus s * (stage bytes / 16) in the
      // start-address field (shared addresses stay below 256 KB: no carry).
      const uint64_t a_desc0 = desc_sw128(smem_u32(sA));
      const uint64_t b_desc0 = desc_sw128(smem_u32(sB));
      const uint64_t sfa_desc0 = desc_sf(smem_u32(sSFA));
      const uint64_t sfb_desc0 = desc_sf(smem_u32(sSFB));
      const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
      // a pair commits to the odd CTA's barriers as well (same offsets there)
      const uint32_t empty0_peer = V::kPair ? cluster_addr(empty0, 1) : 0u;
      const uint32_t tfull_peer = V::kPair ? cluster_addr(smem_u32(tfull), 1) : 0u;
      uint32_t stage = 0, phase = 0, aphase = 0, consumed = 0;
      uint32_t pc = 0;                               // kF8B: partial accumulators written
      bool ok = true;
      TileFeed feed(s_tiles, tile_full, tile_empty);
      while (ok) {
        Tile ti;
        if (!feed.take(ctrl, to, ok, ti)) break;
        const uint32_t tag = (uint32_t)ti.tag;
        if constexpr (!V::kF8B) {
          if (!mbar_wait<V::kPair>(smem_u32(tempty), aphase ^ 1u, ctrl, to, (kSiteTmemEmpty << 24) | tag)) break;
          tc_fence_after();
        }
        const uint32_t id0 = idesc_mx((uint32_t)ti.n, 0u, (uint32_t)(kTileM * G));
        const uint32_t id1 = id0 | (1u << 4) | (1u << 29);
        const uint32_t id2 = id0 | (2u << 4) | (2u << 29);
        const uint32_t id3 = id0 | (3u << 4) | (3u << 29);
        const bool two_sfb = ti.n > 128;
        const uint32_t idb = idesc_bf16((uint32_t)ti.n);
        const uint32_t idf8 = idesc_f8((uint32_t)ti.n);
        for (int kk0 = 0; kk0 < ti.ks; kk0 += kSub) {
          const int nsub = min(kSub, ti.ks - kk0);
          if (!mbar_wait<V::kPair>(full0 + stage * 8u, phase, ctrl, to, (kSiteFull << 24) | tag)) { ok = false; break; }
          for (int u = 0; u < nsub; ++u) {
            const uint32_t so = (uint32_t)(stage * kSub + u);
            const uint32_t acc0 = (kk0 + u) != 0 ? 1u : 0u;
            const uint64_t ad = a_desc0 + (uint64_t)(so * (uint32_t)(kABytes >> 4));
            const uint64_t bd = b_desc0 + (uint64_t)(so * (uint32_t)(V::kBStageBytes >> 4));
            if constexpr (V::kF8B) {
              // each 128-K stage into its own partial accumulator (alternating halves of TMEM),
              // once the epilogue has taken that half's previous partial
              const uint32_t pb = pc & 1u, pph = (pc >> 1) & 1u;
              if (!mbar_wait(smem_u32(&pempty[pb]), pph ^ 1u, ctrl, to, (kSiteTmemEmpty << 24) | tag)) { ok = false; break; }
              tc_fence_after();
              const uint32_t d = tmem + 256u * pb;
              tc_mma_f8(d, ad, bd, idf8, 0u);                            // K = 32 each: +32 bytes
              tc_mma_f8(d, ad + 2, bd + 2, idf8, 1u);
              tc_mma_f8(d, ad + 4, bd + 4, idf8, 1u);
              tc_mma_f8(d, ad + 6, bd + 6, idf8, 1u);
              tc_commit<G>(smem_u32(&pfull[pb]));
              ++pc;
            } else if constexpr (V::kBf16) {
              tc_mma_f16(tmem, ad, bd, idb, acc0);                       // K = 16 each: +32 bytes
              tc_mma_f16(tmem, ad + 2, bd + 2, idb, 1u);
              tc_mma_f16(tmem, ad + 4, bd + 4, idb, 1u);
              tc_mma_f16(tmem, ad + 6, bd + 6, idb, 1u);
            } else {
              // a slot's weight atoms: [128-row half][sub-stage]
              const uint64_t sfb_d = sfb_desc0 + (uint64_t)((stage * kSub * kSFBBytes + u * kAtomBytes) >> 4);
              const uint32_t sfa_t = tmem + kSFCol0 + so * kSFSetCols, sfb_t = sfa_t + 4;
              tc_cp_sf<G>(sfa_t, sfa_desc0 + (uint64_t)(so * (uint32_t)(kSFABytes >> 4)));
              tc_cp_sf<G>(sfb_t, sfb_d);
              if (two_sfb) tc_cp_sf<G>(sfb_t + 4, sfb_d + (uint64_t)((kSub * kAtomBytes) >> 4));
              tc_mma_mx<G>(tmem, ad, bd, id0, sfa_t, sfb_t, acc0);
              tc_mma_mx_acc<G>(tmem, ad + 2, bd + 2, id1, sfa_t, sfb_t);   // K = 32 each: +32 bytes
              tc_mma_mx_acc<G>(tmem, ad + 4, bd + 4, id2, sfa_t, sfb_t);
              tc_mma_mx_acc<G>(tmem, ad + 6, bd + 6, id3, sfa_t, sfb_t);
            }
          }
          tc_commit<G>(empty0 + stage * 8u);
          if constexpr (V::kPair) tc_commit<G>(empty0_peer + stage * 8u);
          ++consumed;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if constexpr (!V::kF8B) {
          tc_commit<G>(smem_u32(tfull));
          if constexpr (V::kPair) tc_commit<G>(tfull_peer);
        }
        aphase ^= 1u;
      }
      s_misc[1] = consumed;
      tc_commit<G>(smem_u32(drain));
      if (!mbar_wait_drain(smem_u32(drain), 0, to)) set_error(ctrl, MM_ERR_TIMEOUT, kSiteDrain << 24);
    }
  } else if (warp == 2 && !V::kSLWarp) {
    // ---------------- scale atoms come with the TMA loads (or there are none): only follow the tile feed
    TileFeed feed(s_tiles, tile_full, tile_empty);
    bool fed = true;
    Tile ti;
    while (feed.take_warp(lane, ctrl, to, fed, ti)) {}
  } else if (warp == 2) {
   if constexpr (V::kSLWarp) {
    // ---------------- scale loader (32 lanes)
    // Copies, stage by stage, the token atom of this CTA's 128 rows of the
    // block and the weight atoms of both 128-row halves of the tile into
    // shared memory (in a pair each CTA holds all 256 rows' weight scales: the
    // MMA reads them from each CTA's TMEM); lane l moves bytes [16l, 16l + 16)
    // of each atom, the loads of 4 stages in flight at a time.  Every lane
    // fences its stores (the tensor core reads through the async proxy) and
    // lane 0 arrives on the full barrier (in a pair, the even CTA's).
    uint32_t stage = 0, phase = 0, armed = 0;
    int ready_key = -1;
    TileFeed feed(s_tiles, tile_full, tile_empty);
    if constexpr (V::kPair) feed.pair(crank);
    const uint32_t full0 = V::kPair ? cluster_addr(smem_u32(&full[0]), 0) : smem_u32(&full[0]);
    for (;;) {
      bool fed = true;
      Tile ti;
      if (!feed.take_warp(lane, ctrl, to, fed, ti)) break;
      const uint32_t tag = (uint32_t)ti.tag;
      bool ok = true;
      const int key = ti.e * 2 + ti.layer - 1;
      if (key != ready_key) {
        if (lane == 0) {
          ok = (ti.layer == 1)
                   ? counter_wait(&arrival[ti.e], (uint32_t)__ldg(counts + ti.e), ctrl, to, (kSiteArrival << 24) | tag)
                   : counter_wait(&l1_done[ti.e], G * l1_tiles_of(items, ti.e, p.mt1), ctrl, to,
                                  (kSiteL1Done << 24) | tag);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        __syncwarp();
        // every lane acquires the writers' atoms before reading them
        if (ti.layer == 1) (void)ld_acquire(&arrival[ti.e]); else (void)ld_acquire(&l1_done[ti.e]);
        ready_key = key;
      }
      const int S = ti.ks;
      const int b_row0 = ti.layer == 1 ? ti.e * 2 * p.I + ti.nb * kL1Feat : ti.e * p.H + ti.nb * kTileN;
      const int b_row1 = ti.layer == 1 ? b_row0 + p.I : b_row0 + 128;
      const uint8_t* wsf = ti.layer == 1 ? p.w1_sf : p.w2_sf;
      const uint8_t* ta = (ti.layer == 1 ? xs_sf : l1a_sf) + ((size_t)(ti.blk * V::kCtas + (int)crank) * S) * kAtomBytes +
                          lane * 16;
      const uint8_t* tb0 = wsf + (size_t)(b_row0 / 128) * S * kAtomBytes + lane * 16;
      const uint8_t* tb1 = wsf + (size_t)((ti.n > 128 ? b_row1 : b_row0) / 128) * S * kAtomBytes + lane * 16;
      for (int g0 = 0; g0 < S && ok; g0 += 4) {
        const int ng = min(4, S - g0);
        uint4 a[4], b0[4], b1[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q < ng) {
            const size_t o = (size_t)(g0 + q) * kAtomBytes;
            a[q] = __ldcg(reinterpret_cast<const uint4*>(ta + o));
            b0[q] = __ldg(reinterpret_cast<const uint4*>(tb0 + o));
            b1[q] = __ldg(reinterpret_cast<const uint4*>(tb1 + o));
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q >= ng) break;
          bool w = true;
          if (lane == 0) w = mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, ctrl, to, (kSiteEmpty << 24) | tag);
          w = __shfl_sync(0xffffffffu, w, 0);
          if (!w) { ok = false; break; }
          reinterpret_cast<uint4*>(sSFA + stage * kSFABytes)[lane] = a[q];
          reinterpret_cast<uint4*>(sSFB + stage * kSFBBytes)[lane] = b0[q];
          reinterpret_cast<uint4*>(sSFB + stage * kSFBBytes + kAtomBytes)[lane] = b1[q];
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            if constexpr (V::kPair) mbar_arrive_cluster(full0 + stage * 8u);
            else mbar_arrive(full0 + stage * 8u);
          }
          ++armed;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) break;
    }
    if (lane == 0) s_misc[4] = armed;
   }
  } else {
    // ---------------- epilogue: warp w reads TMEM lanes 32q..32q+31 (token rows), q = w % 4;
    // the warps w < 8 and w >= 8 of a quarter take the first and second half of the columns
    const int ew = warp - 4;
    const int q = warp & 3;
    const int hh = ew >> 2;
    uint32_t aphase = 0;
    int vote_buf = 0;
    TileFeed feed(s_tiles, tile_full, tile_empty);
    if constexpr (V::kPair) feed.pair(crank);
    // the accumulator is freed on the MMA-issuing CTA's barrier
    const uint32_t tempty_bar = V::kPair ? cluster_addr(smem_u32(tempty), 0) : smem_u32(tempty);
    uint32_t pc = 0;                 // kF8B: partial accumulators taken
    bool failed = false;             // kF8B: a wait inside the last tile gave up
    for (;;) {
      bool ok = true;
      Tile ti;
      if (feed.take_warp(lane, ctrl, to, ok, ti)) {
        if constexpr (!V::kF8B) {
          if (lane == 0)
            ok = mbar_wait<V::kPair>(smem_u32(tfull), aphase, ctrl, to, (kSiteTmemFull << 24) | (uint32_t)ti.tag);
          ok = __shfl_sync(0xffffffffu, ok, 0);
        }
      } else {
        ok = false;      // end of the feed (or abort): leave together
      }
      ok = ok && !failed;
      // the epilogue warps decide together, so none waits alone on a named barrier
      if (lane == 0) s_vote[vote_buf * kEpiWarps + ew] = ok ? 1 : 0;
      named_bar_sync(3, 32 * kEpiWarps);
      bool all_ok = true;
#pragma unroll
      for (int i = 0; i < kEpiWarps; ++i) all_ok &= s_vote[vote_buf * kEpiWarps + i] != 0;
      vote_buf ^= 1;
      if (!all_ok) break;
      tc_fence_after();
      // Each thread takes its whole share of the accumulator into registers (one
      // token row; 64 gate + 64 up columns for L1, up to 128 output columns for
      // L2), frees the accumulator for the next tile's MMAs, and only then does
      // the arithmetic and the stores.
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
      const int tr = (int)crank * kTileM;                  // this CTA's first row of the block
      const int rows = max(0, min(ti.rows - tr, kTileM));  // this CTA's rows (all of them outside a pair)
      const int row = q * 32 + lane;                       // token row of this CTA's share
      const bool valid = row < rows;
      const size_t slot = (size_t)ti.r0 + tr + row;
      const bool live_warp = q * 32 < rows;                // warp-uniform: some row of this quarter is live
      float v[128];
      const int nh = ti.layer == 1 ? kL1Feat / 2 : ti.n >> 1;   // this warp's columns (per operand for L1)
      if constexpr (V::kF8B) {
        // ---- the (1, 128, 128) recipe: v += partial(kk) x (token scale x weight-block scale), stage by stage
#pragma unroll
        for (int i = 0; i < 128; ++i) v[i] = 0.f;
        // the token scales were written by other CTAs (dispatch, or the L1 epilogue): acquire their release
        if (ti.layer == 1) (void)ld_acquire(&arrival[ti.e]); else (void)ld_acquire(&l1_done[ti.e]);
        const int kb = ti.ks;                                        // 128-wide K blocks per row
        const float* tok_s = reinterpret_cast<const float*>(ti.layer == 1 ? xs_sf : l1a_sf) +
                             (size_t)min((int)slot, p.A - 1) * kb;
        const float* w_s = reinterpret_cast<const float*>(ti.layer == 1 ? p.w1_sf : p.w2_sf);
        // weight-scale rows: L1 the gate block nb and the up block I/128 + nb of expert e; L2 the
        // 128-row block that holds this warp's output columns
        const size_t wr0 = ti.layer == 1 ? ((size_t)ti.e * (2 * p.I / 128) + ti.nb) * kb
                                         : ((size_t)ti.e * (p.H / 128) + (ti.nb * kTileN + hh * nh) / 128) * kb;
        const size_t wr1 = ti.layer == 1 ? wr0 + (size_t)(p.I / 128) * kb : wr0;
        // The three scales of stage kk + 1 are loaded while stage kk's partial is added.  The token
        // scales are read only after the first partial has landed: its MMAs waited (through the
        // producers) for the token rows, and so for their scales, to be complete.
        float sx_n = 0.f, w0_n = 0.f, w1_n = 0.f;
        for (int kk = 0; kk < kb; ++kk) {
          const uint32_t pb = pc & 1u, pph = (pc >> 1) & 1u;
          ++pc;
          bool got = true;
          if (lane == 0) got = mbar_wait(smem_u32(&pfull[pb]), pph, ctrl, to, (kSiteTmemFull << 24) | (uint32_t)ti.tag);
          got = __shfl_sync(0xffffffffu, got, 0);
          if (got) {
            tc_fence_after();
            if (kk == 0) {
              sx_n = valid ? __ldcg(tok_s) : 0.f;
              w0_n = __ldg(w_s + wr0);
              w1_n = __ldg(w_s + wr1);
            }
            const float sx = sx_n, w0 = w0_n, w1 = w1_n;
            if (kk + 1 < kb) {
              sx_n = valid ? __ldcg(tok_s + kk + 1) : 0.f;
              w0_n = __ldg(w_s + wr0 + kk + 1);
              w1_n = __ldg(w_s + wr1 + kk + 1);
            }
            if (live_warp) {
              const float c0 = sx * w0, c1 = sx * w1;
              const uint32_t pbase = tbase + 256u * pb;
              // four 16-column loads per TMEM round trip (64 contiguous columns: one operand's
              // half in L1, this warp's first or second 64 outputs in L2)
#pragma unroll
              for (int j = 0; j < 8; j += 4) {
                const bool l1 = ti.layer == 1;
                if (!l1 && j * 16 >= nh) break;
                const uint32_t col0 = l1 ? (uint32_t)((j < 4 ? 0 : kL1Feat) + hh * 64)
                                         : (uint32_t)(hh * nh + j * 16);
                float t[4][16];
#pragma unroll
                for (int x = 0; x < 4; ++x) tc_ld16(pbase + col0 + 16 * x, t[x]);
                tc_wait_ld();
                const float c = (l1 && j >= 4) ? c1 : c0;
#pragma unroll
                for (int x = 0; x < 4; ++x)
#pragma unroll
                  for (int i = 0; i < 16; ++i) v[(j + x) * 16 + i] = fmaf(t[x][i], c, v[(j + x) * 16 + i]);
              }
            }
          } else {
            failed = true;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&pempty[pb]));
        }
      } else if (live_warp) {
        if (ti.layer == 1) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_ld16(tbase + (uint32_t)(hh * 64 + j * 16), *reinterpret_cast<float(*)[16]>(&v[j * 16]));
            tc_ld16(tbase + (uint32_t)(kL1Feat + hh * 64 + j * 16), *reinterpret_cast<float(*)[16]>(&v[64 + j * 16]));
          }
        } else {
          const int c_beg = hh * nh;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j * 16 < nh) tc_ld16(tbase + (uint32_t)(c_beg + j * 16), *reinterpret_cast<float(*)[16]>(&v[j * 16]));
        }
        tc_wait_ld();
      }
      if constexpr (!V::kF8B) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (V::kPair) mbar_arrive_cluster(tempty_bar);
          else mbar_arrive(tempty_bar);
        }
      }
      if (V::kF8B && ti.layer == 1) {
        // ---- L1 of the (1, 128, 128) recipe (every epilogue warp: the block max is exchanged
        // through shared memory with the partner warp that holds the other 64 features of the
        // token's 128): clamp + SwiGLU in fp32, one fp32 scale per 128 features, E4M3 codes
        const float L = p.clamp;
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float gg = v[i], uu = v[64 + i];
          if (p.use_clamp) {
            gg = fminf(gg, L);
            uu = fminf(fmaxf(uu, -L), L);
          }
          v[i] = gg * __fdividef(1.0f, 1.0f + __expf(-gg)) * uu;   // fast-math SiLU
          a = fmaxf(a, fabsf(v[i]));
        }
        sAmax[(q * 2 + hh) * 32 + lane] = a;
        named_bar_sync(4, 32 * kEpiWarps);
        a = fmaxf(a, sAmax[(q * 2 + (hh ^ 1)) * 32 + lane]);
        const float sc = a == 0.f ? 1.0f : __fdiv_rn(a, 448.0f);
        if (valid) {
          uint4* d4 = reinterpret_cast<uint4*>(l1a + slot * p.I + ti.nb * kL1Feat + hh * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const float* hv = &v[16 * i + 4 * b];
              w[b] = e4m3_code(__fdiv_rn(hv[0], sc)) | (e4m3_code(__fdiv_rn(hv[1], sc)) << 8) |
                     (e4m3_code(__fdiv_rn(hv[2], sc)) << 16) | (e4m3_code(__fdiv_rn(hv[3], sc)) << 24);
            }
            d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (hh == 0) reinterpret_cast<float*>(l1a_sf)[slot * (p.I / 128) + ti.nb] = sc;
        }
      } else if (live_warp) {
        if (V::kBf16 && ti.layer == 1) {
          // ---- L1 of the bf16 layer: features [64hh, 64hh + 64): clamp + SwiGLU, rounded to bf16
          const float L = p.clamp;
          // bf16 pair i/2 goes in place into v[i/2], a gate value already consumed
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            float hv[2];
#pragma unroll
            for (int d = 0; d < 2; ++d) {
              float gg = v[i + d], uu = v[64 + i + d];
              if (p.use_clamp) {
                gg = fminf(gg, L);
                uu = fminf(fmaxf(uu, -L), L);
              }
              hv[d] = gg * __fdividef(1.0f, 1.0f + __expf(-gg)) * uu;   // fast-math SiLU
            }
            v[i / 2] = __uint_as_float((uint32_t)bf16_bits_rn(hv[0]) | ((uint32_t)bf16_bits_rn(hv[1]) << 16));
          }
          if (valid) {
            uint4* d4 = reinterpret_cast<uint4*>(l1a + (slot * p.I + ti.nb * kL1Feat + hh * 64) * 2);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              d4[i] = make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]), __float_as_uint(v[4 * i + 2]),
                                 __float_as_uint(v[4 * i + 3]));
          }
        } else if (ti.layer == 1) {
          // ---- L1: features [64hh, 64hh + 64) of the row: clamp + SwiGLU, then E4M3 + UE8M0 per 32
          const float L = p.clamp;
          uint8_t* dst = l1a + slot * p.I + ti.nb * kL1Feat + hh * 64;
          uint32_t sfw = 0;
#pragma unroll
          for (int bi = 0; bi < 2; ++bi) {
            float* h = &v[bi * 32];                          // SwiGLU result overwrites the gate values
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float gg = v[bi * 32 + i], uu = v[64 + bi * 32 + i];
              if (p.use_clamp) {
                gg = fminf(gg, L);
                uu = fminf(fmaxf(uu, -L), L);
              }
              h[i] = gg * __fdividef(1.0f, 1.0f + __expf(-gg)) * uu;   // fast-math SiLU
            }
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(h[i]));
            const int s = block_scale_exp<true>(a);
            const float inv = exp2_neg(s);
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              w[i] = e4m3_code(h[4 * i] * inv) | (e4m3_code(h[4 * i + 1] * inv) << 8) |
                     (e4m3_code(h[4 * i + 2] * inv) << 16) | (e4m3_code(h[4 * i + 3] * inv) << 24);
            if (valid) {
              uint4* d4 = reinterpret_cast<uint4*>(dst + bi * 32);
              d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
              d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
            sfw |= (uint32_t)(s + 127) << (8 * bi);
          }
          if (valid)   // bytes 2hh, 2hh + 1 of the row in the block's atom of L2 stage nb
            *reinterpret_cast<uint16_t*>(l1a_sf + ((size_t)(ti.blk * V::kCtas + (int)crank) * (p.I / 128) + ti.nb) * kAtomBytes +
                                         atom_pos(row) + 2 * hh) = (uint16_t)sfw;
        } else {
          // ---- L2: this warp's nh output columns x top-k weight -> fp32 row of the flat assignment
          int f = 0;
          float wt = 0.f;
          if (valid) {
            f = __ldg(perm + slot);
            wt = __ldg(p.topk_w + f);
          }
          const int c_beg = hh * nh;
          if constexpr (V::kXpose) {
            // 16 columns at a time pass through this warp's transpose buffer (32 rows x four
            // 16-byte chunks; chunk c of row r sits at position c ^ ((r >> 1) & 3), which keeps
            // both the row-wise writes and the column-wise reads free of bank conflicts); lane l
            // then stores chunk l % 4 of rows l / 4 + 8i, whole 64-byte row segments.
            float4* xb = reinterpret_cast<float4*>(sX + ew * (32 * 16));
            const int rr = lane >> 2, cc = lane & 3;
            int fr[4];
            uint32_t live = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = rr + 8 * i;
              fr[i] = __shfl_sync(0xffffffffu, f, r);
              live |= (q * 32 + r < rows ? 1u : 0u) << i;
            }
            float* const col0 = stage_out + ti.nb * kTileN + c_beg + 4 * cc;
            const int wsw = (lane >> 1) & 3;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (j * 16 < nh) {
#pragma unroll
                for (int t = 0; t < 4; ++t)
                  xb[lane * 4 + (t ^ wsw)] = make_float4(v[j * 16 + 4 * t] * wt, v[j * 16 + 4 * t + 1] * wt,
                                                         v[j * 16 + 4 * t + 2] * wt, v[j * 16 + 4 * t + 3] * wt);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int r = rr + 8 * i;
                  const float4 val = xb[r * 4 + (cc ^ ((r >> 1) & 3))];
                  if ((live >> i) & 1u) *reinterpret_cast<float4*>(col0 + (size_t)fr[i] * p.H + j * 16) = val;
                }
                __syncwarp();
              }
            }
          } else {
            // few rows per tile: each thread stores its own row directly
            float4* d4 = reinterpret_cast<float4*>(stage_out + (size_t)f * p.H + ti.nb * kTileN + c_beg);
            if (valid) {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (j * 4 < nh) d4[j] = make_float4(v[4 * j] * wt, v[4 * j + 1] * wt, v[4 * j + 2] * wt, v[4 * j + 3] * wt);
            }
          }
        }
      }
      if (ti.layer == 1) {
        fence_proxy_async_global();
        __threadfence();
        named_bar_sync(3, 32 * kEpiWarps);
        if (ew == 0 && lane == 0) red_release_add(&l1_done[ti.e], 1u);
      }
      aphase ^= 1u;
    }
    __threadfence();
  }

  }  // !skip

  // ------------------------------------------------------------ teardown
  __syncthreads();
  // A pair: both CTAs' roles have stopped and recorded their counts before the
  // even CTA drains, and it finishes draining before either CTA frees its TMEM
  // or exits (loads of both CTAs complete on the even CTA's barriers, and its
  // MMAs read the odd CTA's shared memory).
  if constexpr (V::kPair) cluster_sync();
  if (threadIdx.x == 0 && leader) {
    // After an abort, TMA loads may still be landing.  Each issued but
    // unconsumed stage's barrier completes once its bytes land, provided every
    // role's arrival was made; make the missing ones here (a role that stopped
    // early: its arrival, no bytes; the scale loader has already waited for its
    // own copies).  Roles: each CTA's two producers and scale loader.
    uint32_t cnt[3 * G];
    cnt[0] = s_misc[2];
    cnt[1] = s_misc[5];
    cnt[2] = V::kSLWarp ? s_misc[4] : 0xFFFFFFFFu;
    if constexpr (V::kPair) {
      const uint32_t misc_peer = cluster_addr(smem_u32(s_misc), 1);
      cnt[3] = ld_cluster_u32(misc_peer + 4 * 2);
      cnt[4] = ld_cluster_u32(misc_peer + 4 * 5);
      cnt[5] = ld_cluster_u32(misc_peer + 4 * 4);
    }
    const uint32_t consumed = s_misc[1];
    uint32_t issued = 0;
#pragma unroll
    for (int c = 0; c < G; ++c) issued = max(issued, max(cnt[3 * c], cnt[3 * c + 1]));
    for (uint32_t s = consumed; s < issued; ++s) {
      const uint32_t bar = smem_u32(&full[s % kStages]);
#pragma unroll
      for (int r = 0; r < 3 * G; ++r)
        if (s >= cnt[r]) mbar_arrive(bar);
      if (!mbar_wait_drain(bar, (s / kStages) & 1u, to)) set_error(ctrl, MM_ERR_TIMEOUT, kSiteDrain << 24);
    }
  }
  if constexpr (V::kPair) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc<G>(tmem, kTmemCols);
  }
}

// The top-k weighted combine, one warp per (token, 256 outputs): 32 uint4
// chunks of 8 bf16, one per lane, whose k rows' loads all go out together (a
// small batch is one round trip per warp, not four).  y[t, c] = bf16_RNE(sum over the token's
// valid slots j, ascending, of stage[t*k + j, c]), summed in fp32 from zero; a
// token routed nowhere gets a zero row.  Nothing is combined after an error.
constexpr int kCombineChunks = 32;   // 8-element chunks per warp item
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ ForwardParams p) {
  const uint32_t* ctrl = reinterpret_cast<const uint32_t*>(p.ws + p.L.ctrl);
  if (ld_volatile(&ctrl[kStatus]) != 0u) return;
  const float* stage_out = reinterpret_cast<const float*>(p.ws + p.L.stage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, k = p.k;
  const int nchunk = H / 8;
  const int per_item = kCombineChunks;
  const int items_per_token = (nchunk + per_item - 1) / per_item;
  const int nitems = p.T * items_per_token;
  const int wpb = blockDim.x >> 5;
  for (int it = blockIdx.x * wpb + warp; it < nitems; it += gridDim.x * wpb) {
    const int t = it / items_per_token;
    const int c_beg = (it - t * items_per_token) * per_item;
    const int c_end = min(c_beg + per_item, nchunk);
    const int idx = lane < k ? __ldg(p.topk_idx + (size_t)t * k + lane) : -1;
    const unsigned valid = __ballot_sync(0xffffffffu, idx >= 0);
    const float4* rows = reinterpret_cast<const float4*>(stage_out + (size_t)t * k * H);
    uint4* yrow = reinterpret_cast<uint4*>(p.y + (size_t)t * H);
    for (int c = c_beg + lane; c < c_end; c += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      // the k rows' loads go out together (8 at a time), then the sum runs in ascending j
      for (int j0 = 0; j0 < k; j0 += 8) {
        float4 a[8], b[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (j0 + jj < k && ((valid >> (j0 + jj)) & 1u)) {
            a[jj] = __ldcs(rows + (size_t)(j0 + jj) * (H / 4) + 2 * c);
            b[jj] = __ldcs(rows + (size_t)(j0 + jj) * (H / 4) + 2 * c + 1);
          }
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (j0 + jj < k && ((valid >> (j0 + jj)) & 1u)) {
            acc[0] += a[jj].x; acc[1] += a[jj].y; acc[2] += a[jj].z; acc[3] += a[jj].w;
            acc[4] += b[jj].x; acc[5] += b[jj].y; acc[6] += b[jj].z; acc[7] += b[jj].w;
          }
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        o[i] = (uint32_t)bf16_bits_rn(acc[2 * i]) | ((uint32_t)bf16_bits_rn(acc[2 * i + 1]) << 16);
      yrow[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// ---------------------------------------------------------------- host side
// Template kernels are configured and launched in the translation unit that
// defines them.
int layer_max_rows(int variant) {
  switch (variant) {
    case kVariantThin: return ThinVariant::kBlockRows;
    case kVariantBf16Thin: return Bf16ThinVariant::kBlockRows;
    case kVariantPair: return PairVariant::kBlockRows;
    case kVariantF8B: return F8BVariant::kBlockRows;
    default: return WideVariant::kBlockRows;
  }
}

template <class V>
static cudaLaunchConfig_t launch_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = V::kSmemBytes;
  cfg.stream = stream;
  attr->id = cudaLaunchAttributeClusterDimension;
  attr->val.clusterDim.x = V::kCtas;
  attr->val.clusterDim.y = 1;
  attr->val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// CTAs of the layer kernel that can be resident at once on the whole device
// (for a pair: twice the clusters that fit).
template <class V>
static cudaError_t prepare_one(int* resident, int sms) {
  cudaError_t e = cudaFuncSetAttribute(megamoe_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, V::kSmemBytes);
  if (e != cudaSuccess) return e;
  if constexpr (V::kPair) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = launch_config<V>(2 * (sms / 2), nullptr, &attr);
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, megamoe_kernel<V>, &cfg);
    *resident = 2 * clusters;
    return e;
  } else {
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, megamoe_kernel<V>, kThreads, V::kSmemBytes);
    *resident = per_sm * sms;
    return e;
  }
}

cudaError_t layer_prepare(int variant, int sms, int* resident) {
  switch (variant) {
    case kVariantThin: return prepare_one<ThinVariant>(resident, sms);
    case kVariantBf16Wide: return prepare_one<Bf16WideVariant>(resident, sms);
    case kVariantBf16Thin: return prepare_one<Bf16ThinVariant>(resident, sms);
    case kVariantPair: return prepare_one<PairVariant>(resident, sms);
    case kVariantF8B: return prepare_one<F8BVariant>(resident, sms);
    default: return prepare_one<WideVariant>(resident, sms);
  }
}

template <class V>
static cudaError_t launch_one(int grid, cudaStream_t stream, const CUtensorMap* maps, const ForwardParams& p) {
  if constexpr (V::kPair) {
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = launch_config<V>(grid, stream, &attr);
    return cudaLaunchKernelEx(&cfg, megamoe_kernel<V>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
  } else {
    megamoe_kernel<V><<<grid, kThreads, V::kSmemBytes, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
    return cudaGetLastError();
  }
}

// maps: W1, W2, dispatched tokens (16- and 128-row boxes), L1 activations (16- and 128-row boxes)
// The layer kernel, then the combine kernel on the same stream (8 CTAs of 256
// threads per layer CTA: a full SM's worth of warps on each of those SMs).
cudaError_t layer_launch(int variant, int grid, cudaStream_t stream, const CUtensorMap* maps, const ForwardParams& p) {
  cudaError_t e;
  switch (variant) {
    case kVariantThin: e = launch_one<ThinVariant>(grid, stream, maps, p); break;
    case kVariantBf16Wide: e = launch_one<Bf16WideVariant>(grid, stream, maps, p); break;
    case kVariantBf16Thin: e = launch_one<Bf16ThinVariant>(grid, stream, maps, p); break;
    case kVariantPair: e = launch_one<PairVariant>(grid, stream, maps, p); break;
    case kVariantF8B: e = launch_one<F8BVariant>(grid, stream, maps, p); break;
    default: e = launch_one<WideVariant>(grid, stream, maps, p); break;
  }
  if (e != cudaSuccess) return e;
  const long long items = (long long)p.T * ((p.H / 8 + kCombineChunks - 1) / kCombineChunks);
  const long long want = (items + 7) / 8;
  const int blocks = (int)std::max(1ll, std::min(want, 8ll * grid));
  combine_kernel<<<blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mm
