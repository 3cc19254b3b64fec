// mm_forward_noalloc: the fused layer with its workspace in a fixed device
// array that the library owns, for callers that cannot allocate device
// memory themselves (see include/megamoe.h for who they are and why), and
// mm_noalloc_get_status, which reads the status word of that array.
//
// The scratch array below is a file-scope __device__ variable: it exists on
// every GPU where this library's kernels are loaded and stays there until the
// process exits.  In host code its name is only a host-side stand-in, never a
// device address, so the device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and passed to the kernels
// as an ordinary workspace pointer.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;   // 64 MiB

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[128] = {};   // device address of the array, per device ordinal

// Device address of the array on device `dev` (current), looked up once per
// device; MM_OK or MM_ERR_CUDA.
int scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MM_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MM_OK;
}

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) { cudaGetLastError(); return MM_ERR_NO_DEVICE; }
  if (*dev < 0 || *dev >= 128) return MM_ERR_NO_DEVICE;
  return MM_OK;
}

}  // namespace

extern "C" int mm_forward_noalloc(int num_tokens, int experts, int topk, int hidden, int inter,
                                  const void* x, const void* x_sf, const int32_t* topk_idx, const float* topk_w,
                                  const void* l1_w, const void* l1_sf, const void* l2_w, const void* l2_sf,
                                  void* y, float clamp, int num_sms, mm_stream_t stream) {
  const size_t need = mm_workspace_size(num_tokens, experts, topk, hidden, inter);
  if (need == 0) {
    // unsupported dimensions: let mm_forward report the precise reason
    return mm_forward(num_tokens, experts, topk, hidden, inter, x, x_sf, topk_idx, topk_w, l1_w, l1_sf, l2_w,
                      l2_sf, y, clamp, num_sms, nullptr, 0, stream);
  }
  if (need > kNoAllocScratchBytes) return MM_ERR_WORKSPACE_TOO_SMALL;   // beyond the fixed scratch
  if (num_tokens == 0) return MM_OK;

  int dev = 0;
  int rc = current_device(&dev);
  if (rc != MM_OK) return rc;
  void* ws = nullptr;
  rc = scratch_address(dev, &ws);
  if (rc != MM_OK) return rc;
  return mm_forward(num_tokens, experts, topk, hidden, inter, x, x_sf, topk_idx, topk_w, l1_w, l1_sf, l2_w, l2_sf,
                    y, clamp, num_sms, ws, kNoAllocScratchBytes, stream);
}

// The status word lives at the head of the array, as at the head of any
// workspace, so mm_get_status reads it once the array's address is known.
extern "C" int mm_noalloc_get_status(mm_stream_t stream, int* sm, int* info) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc != MM_OK) return rc;
  void* ws = nullptr;
  rc = scratch_address(dev, &ws);
  if (rc != MM_OK) return rc;
  return mm_get_status(ws, stream, sm, info);
}
