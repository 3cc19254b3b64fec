// Shared definitions of the GB300 fused MoE expert layer: workspace layout,
// tile geometry and thin inline-PTX wrappers (mbarrier, TMA, tcgen05).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/megamoe.h"

namespace mm {

// ----------------------------------------------------------------- geometry
// One MMA tile: up to 128 tokens of one expert on M (E4M3, operand A) times
// 256 weight rows on N (E2M1, operand B), K staged 128 at a time.  Putting the
// weights on N makes every tcgen05.mma consume 4 KB of FP4 weights, so the
// tensor pipe's per-instruction cost stays below the weight stream even when
// an expert holds only a few tokens (decode batches).
constexpr int kBlockK = 128;        // K per pipeline stage: 4 UE8M0 scale blocks of 32
constexpr int kTileM = 128;         // MMA M: tokens per tile
constexpr int kTileN = 256;         // MMA N: weight rows per tile
constexpr int kL1Feat = 128;        // intermediate features per L1 tile (128 gate + 128 up rows)
constexpr int kEpiWarps = 8;        // epilogue warps: two per 32-lane TMEM quarter
constexpr int kThreads = 32 * (4 + kEpiWarps);   // producer, MMA, scale loader, producer, epilogue

constexpr int kBBytes = kTileN * kBlockK;           // 32 KB: 256 weight rows x 128 padded FP4 bytes
// A packed-FP4 TMA box counts its global (packed) bytes toward the barrier's
// transaction count, not its padded shared-memory footprint.
constexpr int kBHalfTxBytes = 128 * kBlockK / 2;    // 8 KB: one 128-row weight box
constexpr int kSFABytes = 512;                      // one 128-row scale atom (tokens)
constexpr int kSFBBytes = 1024;                     // two 128-row scale atoms (weights)
constexpr int kBarBytes = 512;                      // mbarriers + small shared state

// ----------------------------------------------------------------- scale atoms
// The UE8M0 scales of 128 rows for one 128-wide K stage (4 blocks of 32), in
// the order tcgen05.cp (32x128b, warpx4) copies them into TMEM: 32 lanes of 16
// bytes, lane l holding the 4 scale bytes of rows l, 32 + l, 64 + l and 96 + l.
// Byte (row r, block k) of an atom sits at atom_pos(r) + k.  Both operands'
// scales reach shared memory as whole atoms:
// * weights: prepared once (mm_prepare_weight_scales) as [row / 128][K / 128]
//   atoms of a [rows, K/32] scale matrix;
// * tokens: written by the kernel itself (dispatch, L1 epilogue) as
//   [token block][128-row half][K / 128] atoms in the workspace.
constexpr int kAtomBytes = 512;
__host__ __device__ inline int atom_pos(int r) { return (r & 31) * 16 + (r >> 5) * 4; }
// Token-scale atoms of a layer with K-dimension K: room for every token block
// of any layer kernel (at most 2E + A/32 block halves: blocks of >= 32 rows,
// one half per 128 rows of a block).
__host__ __device__ inline size_t token_atom_bytes(size_t A, int E, int K) {
  return (2 * (size_t)E + (A + 31) / 32) * (size_t)(K / 128) * kAtomBytes;
}

// Tile ring of the dynamic schedule: depth, and the number of roles that read
// each entry (producer 1, scale loader, MMA issuer, the epilogue warps).
constexpr int kTileRing = 4;
constexpr int kTileReaders = 1 + 1 + 1 + kEpiWarps;

// TMEM columns: one 256-column fp32 accumulator, then one set of scale-factor
// columns per ring stage (4 token + 8 weight columns each), so that a stage's
// scale copy never targets columns an earlier stage's MMAs may still read.
// (Two 256-column accumulators plus any scale columns would exceed the 512.)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSFCol0 = 256;                   // first scale-factor set
constexpr uint32_t kSFSetCols = 12;                 // SFA: +0..3, SFB: +4..11

// A kernel variant: the token rows a shared-memory stage holds and the ring
// depth.  The MMA always reads 128 token rows from a stage's A address; the
// thin variant keeps only 32 rows per stage, so rows 32..127 of its MMA read
// whatever follows in shared memory and land in accumulator lanes that no
// epilogue thread reads.  Its ring is half again as deep, which is what a
// decode batch (a few tokens per expert, weight streaming) needs.  The wide
// variant adds the epilogue's transpose buffers (see kXposeBytes).
//
// kBf16 selects the bf16 x bf16 layer: bf16 activations and weights, no scale
// factors, tcgen05.mma kind::f16, bf16 L1 activations.  Its K stage is 64
// elements, so rows stay 128 bytes and every shared-memory footprint and box
// byte count of a stage is that of the FP8 x FP4 layer.
//
// kSub: K sub-stages (128 wide each, or 64 for bf16) per ring slot.  A slot is
// one full/empty barrier round trip; two sub-stages per slot halve the round
// trips, waits and commits per weight byte at the same bytes in flight.
//
// kPair: a cluster of two CTAs on neighbouring SMs computes each tile with
// one MMA of M = 256 (tcgen05 cta_group::2): up to 256 tokens of one expert,
// 128 per CTA, times the tile's 256 weight rows, of which each CTA loads and
// holds 128.  A CTA's stage then carries half the weight bytes, so the ring
// can be half again as deep, and each weight row is read once per 256 tokens
// instead of once per 128.  The even CTA of the pair issues every MMA; the
// odd one loads its share, writes its scale atoms and runs the epilogue of
// its 128 accumulator rows.
//
// kF8B: the (1, 128, 128) recipe: E4M3 activations and weights with fp32
// scales per 1 x 128 and 128 x 128 blocks.  The MMA (kind::f8f6f4, no block
// scales) writes each 128-wide K stage into one of two partial accumulators
// in TMEM; the epilogue warps add partial x (token scale x weight-block scale)
// into fp32 registers, stage by stage, and requantise the L1 activations with
// one fp32 scale per token and 128 features.
template <int kARows_, int kStages_, bool kXpose_, bool kBf16_, int kSub_ = 1, bool kPair_ = false,
          bool kF8B_ = false>
struct Variant {
  static constexpr int kARows = kARows_;
  static constexpr int kStages = kStages_;            // ring slots
  static constexpr int kSub = kSub_;                   // sub-stages per slot
  static_assert(kSub == 1 || kSub == 2, "sub-stages per slot");
  static constexpr bool kXpose = kXpose_;
  static constexpr bool kBf16 = kBf16_;
  static constexpr bool kPair = kPair_;
  static_assert(!kPair || (!kBf16 && kARows == kTileM && kSub == 1), "the pair variant is the wide FP8 x FP4 one");
  static constexpr bool kF8B = kF8B_;
  static_assert(!kF8B || (!kBf16 && !kPair && kARows == kTileM && kSub == 1), "the per-128 recipe runs wide tiles");
  static constexpr bool kNoSF = kBf16 || kF8B;         // no block-scale atoms for the MMA
  // Who moves a stage's scale atoms into shared memory: in the 128-token
  // tiles (one CTA or a pair) the scale-loader warp, with coalesced loads, so
  // that the producers issue only the TMA boxes (their issue time per stage is
  // what limits those tiles; a pair's CTAs also need the weight atoms of both
  // halves); in the thin tiles the producers, by bulk copies beside the boxes.
  static constexpr bool kSLWarp = !kNoSF && kSub == 1 && kARows == 128;
  static constexpr int kCtas = kPair ? 2 : 1;          // CTAs that share one MMA tile
  static constexpr int kBlockRows = kARows * kCtas;    // largest token block of a tile
  static constexpr int kKStage = kBf16 ? kBlockK / 2 : kBlockK;     // K elements per stage
  static constexpr int kWeightBoxTx = kNoSF ? 128 * 128 : kBHalfTxBytes;   // one 128-row weight box (bytes)
  static constexpr int kABytes = kARows * kBlockK;
  static constexpr int kBStageBytes = kPair ? kBBytes / 2 : kBBytes;       // weight rows this CTA holds
  static constexpr int kStageBytes = kABytes + kBStageBytes + kSFABytes + kSFBBytes;
  // Epilogue transpose buffer per warp: 32 token rows x 16 fp32 columns, so the
  // L2 epilogue stores whole 64-byte row segments instead of 16-byte pieces of
  // 32 different rows.
  static constexpr int kXposeBytes = kXpose ? kEpiWarps * 32 * 16 * 4 : 0;
  // kF8B: per-row block maxima exchanged by the two warps of a lane quarter
  static constexpr int kAmaxBytes = kF8B ? kEpiWarps * 32 * 4 : 0;
  static constexpr int kSmemBytes = kStages * kSub * kStageBytes + kXposeBytes + kAmaxBytes + kBarBytes + 1024 /*align*/;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kABytes % 1024 == 0 && kBStageBytes % 1024 == 0, "SW128 tiles need 1 KB alignment");
  static_assert(kARows % 16 == 0 && kARows <= kTileM, "token rows per stage");
  // barriers (2 per stage, 3 accumulator/drain, 2 per tile-ring slot, 4 partial-accumulator),
  // misc words, votes, tile ring
  static_assert((2 * kStages + 3 + 2 * kTileRing + 4) * 8 + 8 * 4 + 2 * kEpiWarps * 4 + kTileRing * 10 * 4 <= kBarBytes,
                "barrier region");
  static_assert(kSFCol0 + kStages * kSub * kSFSetCols <= kTmemCols, "scale-factor sets fit TMEM");
  // the MMA's 128-row A window of the last sub-stage stays inside the allocation
  static_assert((kStages * kSub - 1) * kABytes + kTileM * kBlockK <= kStages * kSub * kStageBytes, "A window");
};
using WideVariant = Variant<128, 4, true, false>;
using ThinVariant = Variant<32, 3, false, false, 2>;
using Bf16WideVariant = Variant<128, 4, true, true>;
using Bf16ThinVariant = Variant<32, 6, false, true>;
using PairVariant = Variant<128, 6, true, false, 1, true>;
using F8BVariant = Variant<128, 4, true, false, 1, false, true>;
enum VariantId : int {
  kVariantWide = 0, kVariantThin = 1, kVariantBf16Wide = 2, kVariantBf16Thin = 3, kVariantPair = 4, kVariantF8B = 5,
  kNumVariants = 6
};


// ----------------------------------------------------------------- control block
// 32-bit words at the head of the workspace (words 4 and 7..63 are unused).
enum CtrlWord : int {
  kStatus = 0, kErrSm = 1, kErrInfo = 2, kAbort = 3, kSiteMask = 5, kNextTile = 6, kCtrlWords = 64
};


// Wait sites recorded in the error info word (site << 24 | tile & 0xFFFFFF);
// the numbers are part of the reported value, so a retired site keeps its gap.
enum WaitSite : uint32_t {
  kSiteFull = 1, kSiteEmpty = 2, kSiteTmemFull = 3, kSiteTmemEmpty = 4,
  kSiteArrival = 5, kSiteL1Done = 6, kSiteDrain = 8, kSiteTileRing = 10   // 7 and 9: retired
};

// ----------------------------------------------------------------- workspace
struct Layout {
  size_t ctrl, counts, offsets, items, arrival, l1_done, perm, inv;
  size_t xs, xs_sf, l1a, l1a_sf, stage, rhist, blocks, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Routing CTAs: one 1024-thread CTA handles up to 2048 assignments alone;
// larger batches are split into contiguous chunks of about 1024 assignments
// (at most 128 chunks), counted, scanned and scattered by three kernels.
constexpr int kRouteChunk = 1024;
constexpr int kMaxRouteCtas = 128;     // the scan kernel takes an expert's chunk counts in 4 steps of 32
static_assert(kMaxRouteCtas <= 128, "route_scan_kernel scans at most 128 chunks");
__host__ __device__ inline int route_ctas(long long A) {
  if (A <= 2 * kRouteChunk) return 1;
  const long long c = (A + kRouteChunk - 1) / kRouteChunk;
  return c < kMaxRouteCtas ? (int)c : kMaxRouteCtas;
}

// esz: bytes per activation element (1: E4M3 codes with UE8M0 scales; 2: bf16,
// whose scale regions stay unused).
__host__ __device__ inline Layout make_layout(long long T, int E, int k, int H, int I, int esz = 1) {
  Layout L;
  const size_t A = (size_t)T * (size_t)k;
  size_t o = 0;
  L.ctrl = o;     o = align256(o + 4 * kCtrlWords);
  L.counts = o;   o = align256(o + 4 * (size_t)E);
  L.offsets = o;  o = align256(o + 4 * (size_t)(E + 1));
  L.items = o;    o = align256(o + 4 * (size_t)(E + 1));
  L.arrival = o;  o = align256(o + 4 * (size_t)E);
  L.l1_done = o;  o = align256(o + 4 * (size_t)E);
  L.perm = o;     o = align256(o + 4 * A);
  L.inv = o;      o = align256(o + 4 * A);
  L.xs = o;       o = align256(o + A * (size_t)H * esz);
  // (E4M3 x E2M1: scale atoms; the (1, 128, 128) recipe: fp32 scales per slot row, which fit too)
  L.xs_sf = o;    o = align256(o + token_atom_bytes(A, E, H));
  L.l1a = o;      o = align256(o + A * (size_t)I * esz);
  L.l1a_sf = o;   o = align256(o + token_atom_bytes(A, E, I));
  L.stage = o;    o = align256(o + A * (size_t)H * 4);
  // per-chunk expert counts, then base slots, [E][C] int32, and one bad-index word per chunk
  const size_t C = (size_t)route_ctas((long long)A);
  L.rhist = o;    o = align256(o + 4 * (size_t)E * C + 4 * C);
  // one record per token block, in block order (at most one block per assignment):
  // int32 {expert, expert's first block, expert's first slot, expert's count}
  L.blocks = o;   o = align256(o + 16 * A);
  L.total = o;
  return L;
}

// Number of token blocks an expert with `count` assignments splits into;
// blocks are balanced, each at most `max_n` rows.
__host__ __device__ inline int n_blocks(int count, int max_n) { return (count + max_n - 1) / max_n; }

// ----------------------------------------------------------------- parameters
struct ForwardParams {
  int T, E, k, H, I;
  int A;                       // T * k
  int mt1, mt2;                // weight blocks per expert: I/128 (L1), ceil(H/256) (L2)
  int ks1, ks2;                // K stages of L1 / L2: H/128, I/128
  int use_clamp;
  float clamp;
  int a_box128;                // token count allows one 128-row TMA box per stage
  int max_rows;                // rows per token block at most (the routing's block size)
  unsigned long long timeout_ns;
  const uint8_t* x;            // E4M3 activations and scales, or
  const uint8_t* x_sf;
  const uint16_t* x_bf16;      // bf16 activations, quantised in the dispatch (then x, x_sf are null)
  const int32_t* topk_idx;
  const float* topk_w;
  const uint8_t* w1_sf;
  const uint8_t* w2_sf;
  uint16_t* y;                 // bf16 bits
  uint8_t* ws;
  Layout L;
};

struct RouteParams {
  int T, E, k;
  int A;
  int C, chunk;                // routing CTAs and the assignments each one owns
  int max_n;                   // largest token block of the layer kernel
  const int32_t* topk_idx;
  uint8_t* ws;
  Layout L;
};

// ----------------------------------------------------------------- device helpers
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smid() {
  uint32_t s;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
  return s;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile(const uint32_t* p) {
  return *reinterpret_cast<const volatile uint32_t*>(p);
}

// Generic-proxy global writes <-> async-proxy (TMA) global reads.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Record the first device-side error of a launch and raise the abort flag.
__device__ __forceinline__ void set_error(uint32_t* ctrl, int code, uint32_t info) {
  atomicOr(&ctrl[kSiteMask], 1u << ((info >> 24) & 31u));   // every wait site that gave up
  if (atomicCAS(&ctrl[kStatus], 0u, (uint32_t)code) == 0u) {
    ctrl[kErrSm] = smid();
    ctrl[kErrInfo] = info;
  }
  __threadfence();
  atomicExch(&ctrl[kAbort], 1u);
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// kCluster: acquire at cluster scope, for a phase completed by arrivals from
// the other CTA of a pair (its shared-memory writes become visible).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if constexpr (kCluster)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

// Bounded wait on an mbarrier phase: polls the abort flag and the global timer.
// Returns false if the time limit passed or another thread raised the abort flag.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* ctrl,
                                          unsigned long long timeout_ns, uint32_t site) {
  if (mbar_try_wait<kCluster>(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t it = 0;
  while (!mbar_try_wait<kCluster>(bar, parity)) {
    if ((++it & 63u) == 0u) {
      if (ld_volatile(&ctrl[kAbort]) != 0u) return false;
      if (globaltimer() - t0 > timeout_ns) {
        set_error(ctrl, MM_ERR_TIMEOUT, site);
        return false;
      }
    }
  }
  return true;
}

// Bounded wait used while tearing down after an abort: it ignores the abort
// flag (the copies and MMAs in flight must land before the CTA exits) and
// stops only at the time limit.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t it = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++it & 63u) == 0u && globaltimer() - t0 > timeout_ns) return false;
  }
  return true;
}

// ---- clusters of two CTAs (the pair variant)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address in the cluster's shared window of the variable at `saddr` (this
// CTA's shared address) in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}
// Every thread of both CTAs: orders each CTA's earlier memory operations
// (including remote ones) before the other's later ones.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of either CTA (cluster address); release at cluster
// scope orders this thread's earlier shared-memory writes before it.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cl) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(bar_cl) : "memory");
}
// Arrive with an expected transaction count; relaxed (it announces TMA bytes
// only, it publishes no data of its own).
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar_cl, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;"
               :: "r"(bar_cl), "r"(bytes) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr_cl, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr_cl), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr_cl) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr_cl) : "memory");
  return v;
}

// Bounded wait until a global counter reaches `target` (acquire).
__device__ __forceinline__ bool counter_wait(const uint32_t* p, uint32_t target, uint32_t* ctrl,
                                             unsigned long long timeout_ns, uint32_t site) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = globaltimer();
  uint32_t it = 0;
  while (ld_acquire(p) < target) {
    __nanosleep(64);
    if ((++it & 15u) == 0u) {
      if (ld_volatile(&ctrl[kAbort]) != 0u) return false;
      if (globaltimer() - t0 > timeout_ns) {
        set_error(ctrl, MM_ERR_TIMEOUT, site);
        return false;
      }
    }
  }
  return true;
}

// ---- TMA (2-D tiled load into this CTA's shared memory)
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Contiguous bytes global -> this CTA's shared memory (bulk copy, async proxy),
// completing on one of this CTA's barriers; addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
// TMA into this CTA's shared memory, completing on a barrier of either CTA of
// a pair (cluster address): the pair's loads all land on the leader's barrier.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cl,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cl)
      : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05.  G = 1: one CTA; G = 2: a pair of CTAs (cluster of two) that
// allocate TMEM together and whose MMAs the even CTA issues for both: operand
// A rows 0-127 and B rows 0..N/2-1 from the even CTA's shared memory, the
// rest from the odd CTA's at the same offsets; each CTA's TMEM receives its
// own 128 accumulator rows; scale copies fill both CTAs' TMEM from their own
// shared memory, and the B scales must cover all N in both.
template <int G = 1>
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (G == 2)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst_smem), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst_smem), "r"(ncols) : "memory");
}
template <int G = 1>
__device__ __forceinline__ void tc_relinquish() {
  if constexpr (G == 2) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <int G = 1>
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (G == 2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Arrive on `bar` (a shared address of this CTA, or a cluster address of
// either CTA of a pair) once this thread's earlier MMAs and copies are done.
template <int G = 1>
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  if constexpr (G == 2)
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}
// Copy a 32-row x 16-byte scale atom from shared memory to 4 TMEM columns,
// replicated to the four 32-lane quarters.
template <int G = 1>
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t src_desc) {
  if constexpr (G == 2)
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(src_desc) : "memory");
  else
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" :: "r"(taddr), "l"(src_desc) : "memory");
}
// D (+)= (A * 2^sfa) . (B * 2^sfb)^T, block-scaled, one scale per 32 K.
template <int G = 1>
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (G == 2)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// Same, always accumulating into D.
template <int G = 1>
__device__ __forceinline__ void tc_mma_mx_acc(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem) {
  if constexpr (G == 2)
    asm volatile(
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], 1;"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  else
    asm volatile(
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], 1;"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}
// 32 lanes x 16 columns of 32-bit accumulators into registers.
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr) : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor, K-major operand tile with 128-byte swizzle:
// rows of 128 bytes, 8-row groups 1024 bytes apart (tile base 1 KB aligned).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address (16-byte units)
  d |= (uint64_t)1 << 16;                           // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                           // descriptor version
  d |= (uint64_t)2 << 61;                           // 128-byte swizzle
  return d;
}
// Descriptor of a dense 32-row x 16-byte scale atom (no swizzle; 8-row groups 128 B apart).
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}
// Instruction descriptor of kind::mxf8f6f4 with UE8M0 scales: A = E4M3 tokens
// (M = 128, or 256 over a pair), B = E2M1 weights (N), both K-major; sf_id
// selects the scale byte (the 32-element K block within the 128-element stage).
__device__ __forceinline__ uint32_t idesc_mx(uint32_t n, uint32_t sf_id, uint32_t m = 128) {
  uint32_t d = 0;
  d |= sf_id << 4;                 // B scale-factor id
  d |= 0u << 7;                    // A format: E4M3
  d |= 5u << 10;                   // B format: E2M1
  d |= (n >> 3) << 17;             // N / 8
  d |= 1u << 23;                   // scale format: UE8M0
  d |= (m >> 4) << 24;             // M / 16
  d |= sf_id << 29;                // A scale-factor id
  return d;
}

// Instruction descriptor of kind::f16: A = bf16 tokens (M = 128), B = bf16
// weights (N), fp32 accumulator, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(uint32_t n) {
  uint32_t d = 0;
  d |= 1u << 4;                    // accumulator format: F32
  d |= 1u << 7;                    // A format: BF16
  d |= 1u << 10;                   // B format: BF16
  d |= (n >> 3) << 17;             // N / 8
  d |= (128u >> 4) << 24;          // M / 16
  return d;
}
// Instruction descriptor of kind::f8f6f4 without block scales: A = E4M3 tokens
// (M = 128), B = E4M3 weights (N), fp32 accumulator, both K-major.
__device__ __forceinline__ uint32_t idesc_f8(uint32_t n) {
  uint32_t d = 0;
  d |= 1u << 4;                    // accumulator format: F32
  d |= 0u << 7;                    // A format: E4M3
  d |= 0u << 10;                   // B format: E4M3
  d |= (n >> 3) << 17;             // N / 8
  d |= (128u >> 4) << 24;          // M / 16
  return d;
}
// D (+)= A . B^T, E4M3 operands (K = 32 per instruction), no scales.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (+)= A . B^T, bf16 operands (K = 16 per instruction).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

#endif  // __CUDACC__

}  // namespace mm
