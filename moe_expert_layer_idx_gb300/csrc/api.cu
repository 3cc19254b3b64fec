// Host side of the C ABI declared in include/megamoe.h: argument checks,
// workspace layout, launch sizing with the SM reserve, TMA descriptors and
// the two launches of mm_forward.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace mm {
__global__ void route_kernel(const RouteParams p);
__global__ void route_count_kernel(const RouteParams p);
__global__ void route_scan_kernel(const RouteParams p);
__global__ void route_scatter_kernel(const RouteParams p);
int layer_max_rows(int variant);
cudaError_t layer_prepare(int variant, int sms, int* resident);
cudaError_t layer_launch(int variant, int grid, cudaStream_t stream, const CUtensorMap* maps, const ForwardParams& p);
cudaError_t launch_quantize(const float* src, long long nblocks, bool e4m3, uint8_t* dst, uint8_t* sf,
                            int grid, cudaStream_t stream);
cudaError_t launch_prepare_weight_scales(const uint8_t* sf, long long rows, int kb, uint8_t* out, int max_ctas,
                                         cudaStream_t stream);
cudaError_t launch_quantize_f8b(const float* src, long long rows, long long cols, int block_rows, uint8_t* dst,
                                float* sf, int max_ctas, cudaStream_t stream);
}  // namespace mm

using namespace mm;

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;
constexpr int kDefaultReserve = 2;   // sglang PR #36657, Summary: two SMs by default
constexpr int kDefaultPair = 0;      // two-CTA tiles measured slower than one-CTA tiles: off unless switched on

std::atomic<int> g_reserved{-1};
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
std::atomic<int> g_pair{-1};       // two-CTA MMA tiles for wide batches: -1 = not yet read from the environment

int reserved_now() {
  int r = g_reserved.load();
  if (r >= 0) return r;
  int v = kDefaultReserve;
  if (const char* env = std::getenv("MM_RESERVED_SMS")) {
    char* end = nullptr;
    long x = std::strtol(env, &end, 10);
    if (end != env) v = x < 0 ? 0 : (x > 1 << 20 ? 1 << 20 : (int)x);
  }
  int expected = -1;
  g_reserved.compare_exchange_strong(expected, v);
  return g_reserved.load();
}

int pair_now() {
  int v = g_pair.load();
  if (v >= 0) return v;
  v = kDefaultPair;
  if (const char* env = std::getenv("MM_PAIR_MMA")) {
    char* end = nullptr;
    long x = std::strtol(env, &end, 10);
    if (end != env) v = x != 0 ? 1 : 0;
  }
  int expected = -1;
  g_pair.compare_exchange_strong(expected, v);
  return g_pair.load();
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(long long T, int E, int k, int H, int I) {
  if (T < 0 || E < 1 || k < 1 || H < 1 || I < 1) return MM_ERR_INVALID_ARG;
  if (E > 1024 || k > 16) return MM_ERR_UNSUPPORTED_SHAPE;
  if (H % 128 != 0 || H > 32768) return MM_ERR_UNSUPPORTED_SHAPE;
  if (I % 128 != 0 || I > 16384) return MM_ERR_UNSUPPORTED_SHAPE;
  if (T * (long long)k > (1ll << 24)) return MM_ERR_UNSUPPORTED_SHAPE;
  // weight rows addressed by a 32-bit TMA coordinate
  if ((long long)E * 2 * I >= (1ll << 31) || (long long)E * H >= (1ll << 31)) return MM_ERR_UNSUPPORTED_SHAPE;
  return MM_OK;
}

// ---- per-device state
struct DevState {
  bool ready = false;
  int sms = 0;
  int max_resident[kNumVariants] = {};   // layer kernel CTAs resident at once, per variant
};

// Kernel variant for a batch: with at most 16 assignments per expert on
// average (decode), the thin variant's deeper weight ring; otherwise 128-token
// tiles, or 256-token tiles on a pair of CTAs (FP8 x FP4 layer, hidden size a
// multiple of 256 so that every L2 weight block splits into two 128-row
// halves, and the pair switch on).
int pick_variant(long long assignments, int experts, int hidden, bool bf16_layer) {
  const bool thin = assignments <= 16ll * experts;
  if (bf16_layer) return thin ? kVariantBf16Thin : kVariantBf16Wide;
  if (thin) return kVariantThin;
  return (hidden % 256 == 0 && pair_now()) ? kVariantPair : kVariantWide;
}
std::mutex g_mu;
DevState g_dev[128];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int device_state(int* dev_out, DevState** st_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return MM_ERR_NO_DEVICE; }
  if (dev < 0 || dev >= 128) return MM_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& st = g_dev[dev];
  if (!st.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) { cudaGetLastError(); return MM_ERR_NO_DEVICE; }
    if (prop.major != 10 || prop.minor != 3) return MM_ERR_NO_DEVICE;   // built for sm_103a only
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return MM_ERR_CUDA;
      }
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 32 * 1024 * 4) != cudaSuccess ||
        cudaFuncSetAttribute(route_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 32 * 1024 * 4) !=
            cudaSuccess ||
        cudaFuncSetAttribute(route_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 32 * 1024 * 4) !=
            cudaSuccess) {
      cudaGetLastError();
      return MM_ERR_CUDA;
    }
    for (int v = 0; v < kNumVariants; ++v) {
      int resident = 0;
      if (layer_prepare(v, prop.multiProcessorCount, &resident) != cudaSuccess) {
        cudaGetLastError();
        return MM_ERR_CUDA;
      }
      st.max_resident[v] = resident;
    }
    st.sms = prop.multiProcessorCount;
    st.ready = true;
  }
  *dev_out = dev;
  *st_out = &st;
  return MM_OK;
}

int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1,
              uint64_t row_bytes, uint32_t b0, uint32_t b1) {
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {b0, b1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MM_OK : MM_ERR_CUDA;
}

// `variant`: the layer kernel that consumes the routing (its largest token block).
int launch_route(int T, int E, int k, int variant, const int32_t* topk_idx, uint8_t* ws, const Layout& L,
                 cudaStream_t st) {
  RouteParams rp;
  rp.T = T; rp.E = E; rp.k = k; rp.A = T * k;
  rp.C = route_ctas(rp.A);
  rp.chunk = (rp.A + rp.C - 1) / rp.C;
  rp.max_n = layer_max_rows(variant);   // the same token blocks for both layers
  rp.topk_idx = topk_idx;
  rp.ws = ws;
  rp.L = L;
  const size_t smem = (size_t)32 * E * 4;
  if (rp.C == 1) {
    route_kernel<<<1, 1024, smem, st>>>(rp);
  } else {
    route_count_kernel<<<rp.C, 1024, smem, st>>>(rp);
    route_scan_kernel<<<1, 1024, 0, st>>>(rp);
    route_scatter_kernel<<<rp.C, 1024, smem, st>>>(rp);
  }
  if (cudaGetLastError() != cudaSuccess) return MM_ERR_CUDA;
  return MM_OK;
}

int common_checks(int T, int E, int k, int H, int I, const void* workspace, size_t workspace_bytes, Layout* L,
                  int esz = 1) {
  int rc = check_shape(T, E, k, H, I);
  if (rc != MM_OK) return rc;
  if (!workspace || !aligned(workspace, 256)) return MM_ERR_INVALID_ARG;
  *L = make_layout(T, E, k, H, I, esz);
  if (workspace_bytes < L->total) return MM_ERR_WORKSPACE_TOO_SMALL;
  return MM_OK;
}

}  // namespace

extern "C" {

size_t mm_workspace_size(int max_tokens, int experts, int topk, int hidden, int inter) {
  if (check_shape(max_tokens, experts, topk, hidden, inter) != MM_OK) return 0;
  return make_layout(max_tokens, experts, topk, hidden, inter).total;
}

int mm_set_reserved_sms(int n) {
  const int prev = reserved_now();
  g_reserved.store(n < 0 ? 0 : n);
  return prev;
}

int mm_get_reserved_sms(void) { return reserved_now(); }

int mm_set_pair_mma(int enable) {
  const int prev = pair_now();
  g_pair.store(enable != 0 ? 1 : 0);
  return prev;
}

int mm_get_pair_mma(void) { return pair_now(); }

int mm_layer_variant(int num_tokens, int experts, int topk, int hidden, int bf16_layer) {
  if (num_tokens < 0 || experts < 1 || topk < 1) return MM_ERR_INVALID_ARG;
  return pick_variant((long long)num_tokens * topk, experts, hidden, bf16_layer != 0);
}

int mm_grid_size(int device_sms, int reserved_sms, int num_sms, int max_resident) {
  if (device_sms < 2) return MM_ERR_INVALID_ARG;
  const int res = reserved_sms < 0 ? 0 : reserved_sms;
  const int cap = std::max(2, device_sms - res);
  const int want = num_sms > 0 ? std::min(num_sms, device_sms) : device_sms;
  int g = std::min(cap, want);
  g -= g % 2;
  g = std::max(g, 2);
  if (max_resident > 0 && g > max_resident) {
    g = max_resident - max_resident % 2;
    if (g < 1) g = max_resident;
  }
  return g;
}

void mm_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns.store(ns ? ns : kDefaultTimeoutNs); }
unsigned long long mm_get_wait_timeout_ns(void) { return g_timeout_ns.load(); }

// The fused layer.  recipe kMx (FP8 x FP4, UE8M0 per 32): E4M3 activations
// (x, x_sf) when x_bf16 is null, else bf16 activations quantised in the
// dispatch.  kBf16 (bf16 x bf16): bf16 activations in x and bf16 weights, no
// scale factors.  kF8B (the (1, 128, 128) recipe): E4M3 activations and
// weights, fp32 scales per 1 x 128 (x_sf) and 128 x 128 (l1_sf, l2_sf) blocks.
// A missing input is MM_ERR_INVALID_ARG (after the shape checks and the T = 0
// early return).
enum Recipe : int { kMx = 0, kBf16 = 1, kF8B = 2 };
static int forward_impl(int recipe, int num_tokens, int experts, int topk, int hidden, int inter,
                        const void* x, const void* x_sf, const void* x_bf16, const int32_t* topk_idx,
                        const float* topk_w, const void* l1_w, const void* l1_sf, const void* l2_w,
                        const void* l2_sf, void* y, float clamp, int num_sms,
                        void* workspace, size_t workspace_bytes, mm_stream_t stream) {
  const int T = num_tokens, E = experts, k = topk, H = hidden, I = inter;
  int rc = check_shape(T, E, k, H, I);
  if (rc != MM_OK) return rc;
  if (T == 0) return MM_OK;
  const bool bf16_layer = recipe == kBf16, f8b = recipe == kF8B;
  const bool fp8_in = !bf16_layer && x_bf16 == nullptr;
  const bool scales = !bf16_layer;
  if ((bf16_layer && !x) || (fp8_in && (!x || !x_sf)) || !topk_idx || !topk_w || !l1_w || !l2_w || !y ||
      (scales && (!l1_sf || !l2_sf)))
    return MM_ERR_INVALID_ARG;
  if ((bf16_layer && !aligned(x, 16)) || (fp8_in && (!aligned(x, 16) || !aligned(x_sf, 4))) ||
      (!bf16_layer && !fp8_in && !aligned(x_bf16, 16)) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
      !aligned(l1_w, 32) || !aligned(l2_w, 32) ||
      (scales && (!aligned(l1_sf, f8b ? 4 : 16) || !aligned(l2_sf, f8b ? 4 : 16))) ||   // scale atoms: bulk copies
      !aligned(y, 16))
    return MM_ERR_INVALID_ARG;
  if (std::isnan(clamp)) return MM_ERR_INVALID_ARG;
  Layout L;
  rc = common_checks(T, E, k, H, I, workspace, workspace_bytes, &L, bf16_layer ? 2 : 1);
  if (rc != MM_OK) return rc;

  int dev;
  DevState* st;
  rc = device_state(&dev, &st);
  if (rc != MM_OK) return rc;
  const int variant = f8b ? (int)kVariantF8B : pick_variant((long long)T * k, E, H, bf16_layer);
  const int grid = mm_grid_size(st->sms, reserved_now(), num_sms, st->max_resident[variant]);
  const int A = T * k;
  uint8_t* ws = static_cast<uint8_t*>(workspace);

  // W1 / W2 as [rows][K] packed FP4, 128 x 128 boxes (widened to 8-bit containers
  // in shared memory); dispatched tokens and L1 activations as [A][K] bytes,
  // 16-row and 128-row boxes.
  alignas(64) CUtensorMap maps[6];
  // bf16 layer: every operand bf16, [rows][K] with 64-element (128-byte) boxes
  const int kk = bf16_layer ? kBlockK / 2 : kBlockK;
  if (bf16_layer) {
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (encode_2d(&maps[0], bf, l1_w, (uint64_t)H, (uint64_t)E * 2 * I, (uint64_t)H * 2, kk, 128) != MM_OK ||
        encode_2d(&maps[1], bf, l2_w, (uint64_t)I, (uint64_t)E * H, (uint64_t)I * 2, kk, 128) != MM_OK ||
        encode_2d(&maps[2], bf, ws + L.xs, (uint64_t)H, (uint64_t)A, (uint64_t)H * 2, kk, 16) != MM_OK ||
        encode_2d(&maps[3], bf, ws + L.xs, (uint64_t)H, (uint64_t)A, (uint64_t)H * 2, kk, kTileM) != MM_OK ||
        encode_2d(&maps[4], bf, ws + L.l1a, (uint64_t)I, (uint64_t)A, (uint64_t)I * 2, kk, 16) != MM_OK ||
        encode_2d(&maps[5], bf, ws + L.l1a, (uint64_t)I, (uint64_t)A, (uint64_t)I * 2, kk, kTileM) != MM_OK)
      return MM_ERR_CUDA;
  } else if (f8b) {
    // E4M3 weights [rows][K], one byte per element, 128 x 128 boxes
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (encode_2d(&maps[0], u8, l1_w, (uint64_t)H, (uint64_t)E * 2 * I, H, kBlockK, 128) != MM_OK ||
        encode_2d(&maps[1], u8, l2_w, (uint64_t)I, (uint64_t)E * H, I, kBlockK, 128) != MM_OK ||
        encode_2d(&maps[2], u8, ws + L.xs, (uint64_t)H, (uint64_t)A, H, kBlockK, 16) != MM_OK ||
        encode_2d(&maps[3], u8, ws + L.xs, (uint64_t)H, (uint64_t)A, H, kBlockK, kTileM) != MM_OK ||
        encode_2d(&maps[4], u8, ws + L.l1a, (uint64_t)I, (uint64_t)A, I, kBlockK, 16) != MM_OK ||
        encode_2d(&maps[5], u8, ws + L.l1a, (uint64_t)I, (uint64_t)A, I, kBlockK, kTileM) != MM_OK)
      return MM_ERR_CUDA;
  } else if (encode_2d(&maps[0], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, l1_w, (uint64_t)H, (uint64_t)E * 2 * I, H / 2,
                kBlockK, 128) != MM_OK ||
      encode_2d(&maps[1], CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, l2_w, (uint64_t)I, (uint64_t)E * H, I / 2,
                kBlockK, 128) != MM_OK ||
      encode_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT8, ws + L.xs, (uint64_t)H, (uint64_t)A, H, kBlockK, 16) != MM_OK ||
      encode_2d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_UINT8, ws + L.xs, (uint64_t)H, (uint64_t)A, H, kBlockK,
                kTileM) != MM_OK ||
      encode_2d(&maps[4], CU_TENSOR_MAP_DATA_TYPE_UINT8, ws + L.l1a, (uint64_t)I, (uint64_t)A, I, kBlockK, 16) != MM_OK ||
      encode_2d(&maps[5], CU_TENSOR_MAP_DATA_TYPE_UINT8, ws + L.l1a, (uint64_t)I, (uint64_t)A, I, kBlockK,
                kTileM) != MM_OK)
    return MM_ERR_CUDA;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = launch_route(T, E, k, variant, topk_idx, ws, L, s);
  if (rc != MM_OK) return rc;

  ForwardParams fp;
  fp.T = T; fp.E = E; fp.k = k; fp.H = H; fp.I = I; fp.A = A;
  fp.mt1 = I / kL1Feat; fp.mt2 = (H + kTileN - 1) / kTileN;
  fp.ks1 = H / kk; fp.ks2 = I / kk;
  fp.use_clamp = (std::isfinite(clamp) && clamp > 0.f) ? 1 : 0;
  fp.clamp = fp.use_clamp ? clamp : 0.f;
  fp.a_box128 = A >= kTileM ? 1 : 0;
  fp.max_rows = layer_max_rows(variant);
  fp.timeout_ns = g_timeout_ns.load();
  fp.x = (fp8_in || bf16_layer) ? static_cast<const uint8_t*>(x) : nullptr;
  fp.x_sf = fp8_in ? static_cast<const uint8_t*>(x_sf) : nullptr;
  fp.x_bf16 = (fp8_in || bf16_layer) ? nullptr : static_cast<const uint16_t*>(x_bf16);
  fp.topk_idx = topk_idx;
  fp.topk_w = topk_w;
  fp.w1_sf = static_cast<const uint8_t*>(l1_sf);
  fp.w2_sf = static_cast<const uint8_t*>(l2_sf);
  fp.y = static_cast<uint16_t*>(y);
  fp.ws = ws;
  fp.L = L;
  if (layer_launch(variant, grid, s, maps, fp) != cudaSuccess) return MM_ERR_CUDA;
  return MM_OK;
}

int mm_forward(int num_tokens, int experts, int topk, int hidden, int inter,
               const void* x, const void* x_sf, const int32_t* topk_idx, const float* topk_w,
               const void* l1_w, const void* l1_sf, const void* l2_w, const void* l2_sf,
               void* y, float clamp, int num_sms,
               void* workspace, size_t workspace_bytes, mm_stream_t stream) {
  return forward_impl(kMx, num_tokens, experts, topk, hidden, inter, x, x_sf, nullptr, topk_idx, topk_w, l1_w,
                      l1_sf, l2_w, l2_sf, y, clamp, num_sms, workspace, workspace_bytes, stream);
}

int mm_f8b_forward(int num_tokens, int experts, int topk, int hidden, int inter,
                   const void* x, const float* x_sf, const int32_t* topk_idx, const float* topk_w,
                   const void* l1_w, const float* l1_sf, const void* l2_w, const float* l2_sf,
                   void* y, float clamp, int num_sms,
                   void* workspace, size_t workspace_bytes, mm_stream_t stream) {
  if ((l1_w && !aligned(l1_w, 16)) || (l2_w && !aligned(l2_w, 16))) return MM_ERR_INVALID_ARG;
  return forward_impl(kF8B, num_tokens, experts, topk, hidden, inter, x, x_sf, nullptr, topk_idx, topk_w, l1_w,
                      l1_sf, l2_w, l2_sf, y, clamp, num_sms, workspace, workspace_bytes, stream);
}

int mm_forward_bf16(int num_tokens, int experts, int topk, int hidden, int inter,
                    const void* x_bf16, const int32_t* topk_idx, const float* topk_w,
                    const void* l1_w, const void* l1_sf, const void* l2_w, const void* l2_sf,
                    void* y, float clamp, int num_sms,
                    void* workspace, size_t workspace_bytes, mm_stream_t stream) {
  return forward_impl(kMx, num_tokens, experts, topk, hidden, inter, nullptr, nullptr, x_bf16, topk_idx, topk_w,
                      l1_w, l1_sf, l2_w, l2_sf, y, clamp, num_sms, workspace, workspace_bytes, stream);
}

size_t mm_bf16_workspace_size(int max_tokens, int experts, int topk, int hidden, int inter) {
  if (check_shape(max_tokens, experts, topk, hidden, inter) != MM_OK) return 0;
  return make_layout(max_tokens, experts, topk, hidden, inter, 2).total;
}

int mm_bf16_forward(int num_tokens, int experts, int topk, int hidden, int inter,
                    const void* x, const int32_t* topk_idx, const float* topk_w,
                    const void* l1_w, const void* l2_w, void* y, float clamp, int num_sms,
                    void* workspace, size_t workspace_bytes, mm_stream_t stream) {
  return forward_impl(kBf16, num_tokens, experts, topk, hidden, inter, x, nullptr, nullptr, topk_idx, topk_w, l1_w,
                      nullptr, l2_w, nullptr, y, clamp, num_sms, workspace, workspace_bytes, stream);
}

int mm_route(int num_tokens, int experts, int topk, int hidden, int inter, const int32_t* topk_idx,
             void* workspace, size_t workspace_bytes, mm_stream_t stream) {
  Layout L;
  int rc = common_checks(num_tokens, experts, topk, hidden, inter, workspace, workspace_bytes, &L);
  if (rc != MM_OK) return rc;
  if (num_tokens == 0) return MM_OK;
  if (!topk_idx || !aligned(topk_idx, 4)) return MM_ERR_INVALID_ARG;
  int dev;
  DevState* st;
  rc = device_state(&dev, &st);
  if (rc != MM_OK) return rc;
  return launch_route(num_tokens, experts, topk, pick_variant((long long)num_tokens * topk, experts, hidden, false),
                      topk_idx, static_cast<uint8_t*>(workspace), L, reinterpret_cast<cudaStream_t>(stream));
}

int mm_read_routing(int num_tokens, int experts, int topk, int hidden, int inter, const void* workspace,
                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv) {
  int rc = check_shape(num_tokens, experts, topk, hidden, inter);
  if (rc != MM_OK) return rc;
  if (!workspace) return MM_ERR_INVALID_ARG;
  const Layout L = make_layout(num_tokens, experts, topk, hidden, inter);
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const size_t A = (size_t)num_tokens * topk;
  if (cudaDeviceSynchronize() != cudaSuccess) { cudaGetLastError(); return MM_ERR_CUDA; }
  if (counts && cudaMemcpy(counts, ws + L.counts, 4 * (size_t)experts, cudaMemcpyDeviceToHost) != cudaSuccess) return MM_ERR_CUDA;
  if (offsets && cudaMemcpy(offsets, ws + L.offsets, 4 * (size_t)(experts + 1), cudaMemcpyDeviceToHost) != cudaSuccess) return MM_ERR_CUDA;
  if (A && perm && cudaMemcpy(perm, ws + L.perm, 4 * A, cudaMemcpyDeviceToHost) != cudaSuccess) return MM_ERR_CUDA;
  if (A && inv && cudaMemcpy(inv, ws + L.inv, 4 * A, cudaMemcpyDeviceToHost) != cudaSuccess) return MM_ERR_CUDA;
  return MM_OK;
}

int mm_get_status(const void* workspace, mm_stream_t stream, int* sm, int* info) {
  if (!workspace) return MM_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) { cudaGetLastError(); return MM_ERR_CUDA; }
  uint32_t w[6] = {0, 0, 0, 0, 0, 0};
  if (cudaMemcpy(w, workspace, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) { cudaGetLastError(); return MM_ERR_CUDA; }
  if (sm) *sm = (int)w[kErrSm];
  if (info) *info = (int)w[kErrInfo];
  return (int)w[kStatus];
}

int mm_workspace_region(int which, int num_tokens, int experts, int topk, int hidden, int inter,
                        size_t* offset, size_t* bytes) {
  if (check_shape(num_tokens, experts, topk, hidden, inter) != MM_OK) return MM_ERR_INVALID_ARG;
  const Layout L = make_layout(num_tokens, experts, topk, hidden, inter);
  const size_t starts[15] = {L.ctrl, L.counts, L.offsets, L.items, L.arrival, L.l1_done, L.perm, L.inv,
                             L.xs, L.xs_sf, L.l1a, L.l1a_sf, L.stage, L.rhist, L.blocks};
  if (which < 0 || which > 14) return MM_ERR_INVALID_ARG;
  const size_t A = (size_t)num_tokens * topk;
  const size_t C = (size_t)route_ctas((long long)A);
  const size_t exact[15] = {4 * (size_t)kCtrlWords, 4 * (size_t)experts, 4 * (size_t)(experts + 1),
                            4 * (size_t)(experts + 1), 4 * (size_t)experts, 4 * (size_t)experts, 4 * A, 4 * A,
                            A * hidden, token_atom_bytes(A, experts, hidden), A * inter,
                            token_atom_bytes(A, experts, inter), A * hidden * 4,
                            4 * (size_t)experts * C + 4 * C, 16 * A};
  if (offset) *offset = starts[which];
  if (bytes) *bytes = exact[which];
  return MM_OK;
}

int mm_quantize_mx(const float* src, long long rows, long long cols, int fmt, void* dst, void* dst_sf,
                   mm_stream_t stream) {
  if (rows < 0 || cols < 0 || cols % 32 != 0) return MM_ERR_INVALID_ARG;
  if (fmt != MM_FMT_E4M3 && fmt != MM_FMT_E2M1) return MM_ERR_INVALID_ARG;
  const long long nblocks = rows * (cols / 32);
  if (nblocks == 0) return MM_OK;
  if (!src || !dst || !dst_sf || !aligned(src, 16) || !aligned(dst, 16)) return MM_ERR_INVALID_ARG;
  int dev;
  DevState* st;
  int rc = device_state(&dev, &st);
  if (rc != MM_OK) return rc;
  long long blocks = (nblocks + 255) / 256;
  const long long cap = (long long)st->sms * 16;
  if (blocks > cap) blocks = cap;
  if (launch_quantize(src, nblocks, fmt == MM_FMT_E4M3, static_cast<uint8_t*>(dst), static_cast<uint8_t*>(dst_sf),
                      (int)blocks, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MM_ERR_CUDA;
  return MM_OK;
}

int mm_prepare_weight_scales(const void* sf, long long rows, long long k, void* out, mm_stream_t stream) {
  if (rows < 0 || k < 0 || rows % 128 != 0 || k % 128 != 0 || k / 32 > (1ll << 30)) return MM_ERR_INVALID_ARG;
  if (rows * k == 0) return MM_OK;
  if (!sf || !out || !aligned(sf, 4) || !aligned(out, 16)) return MM_ERR_INVALID_ARG;
  int dev;
  DevState* st;
  int rc = device_state(&dev, &st);
  if (rc != MM_OK) return rc;
  if (launch_prepare_weight_scales(static_cast<const uint8_t*>(sf), rows, (int)(k / 32), static_cast<uint8_t*>(out),
                                   st->sms * 16, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MM_ERR_CUDA;
  return MM_OK;
}

}  // extern "C"

extern "C" int mm_quantize_f8b(const float* src, long long rows, long long cols, int block_rows, void* dst,
                               float* dst_sf, mm_stream_t stream) {
  if (rows < 0 || cols < 0 || cols % 128 != 0) return MM_ERR_INVALID_ARG;
  if (block_rows != 1 && block_rows != 128) return MM_ERR_INVALID_ARG;
  if (rows % block_rows != 0) return MM_ERR_INVALID_ARG;
  if (block_rows == 128 && (rows > (1ll << 31) - 1 || cols > (1ll << 31) - 1)) return MM_ERR_INVALID_ARG;
  if (rows * cols == 0) return MM_OK;
  if (!src || !dst || !dst_sf || !aligned(src, 16) || !aligned(dst, 4) || !aligned(dst_sf, 4)) return MM_ERR_INVALID_ARG;
  int dev;
  DevState* st;
  int rc = device_state(&dev, &st);
  if (rc != MM_OK) return rc;
  if (launch_quantize_f8b(src, rows, cols, block_rows, static_cast<uint8_t*>(dst), dst_sf, st->sms * 16,
                          reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MM_ERR_CUDA;
  return MM_OK;
}
