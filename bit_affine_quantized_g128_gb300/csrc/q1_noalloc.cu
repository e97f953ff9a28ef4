// q1_ffn_fused_noalloc: the fused FFN with its intermediate h [M][F] (bf16) in
// a fixed device array of this library instead of a caller workspace, for
// callers that must not allocate at all.  The call adds nothing to the
// arithmetic: it runs q1_ffn_fused with that array as the workspace.
//
// The array is a file-scope __device__ variable (one per device), so the
// call makes no allocation; its address comes from cudaGetSymbolAddress the
// first time the call runs on a device and is cached per device.
#include <atomic>

#include "q1_internal.h"

namespace {

constexpr size_t kFfnStaticBytes = Q1_FFN_NOALLOC_BYTES;  // h: M * F * 2 bytes at most
__device__ __align__(256) unsigned char g_ffn_static[kFfnStaticBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_ffn_static_addr[kMaxDevices];

// Device address of g_ffn_static on the current device (nullptr on error).
void *ffn_static_addr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < kMaxDevices) {
    void *p = g_ffn_static_addr[dev].load(std::memory_order_acquire);
    if (p) return p;
  }
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_ffn_static) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (dev >= 0 && dev < kMaxDevices) g_ffn_static_addr[dev].store(p, std::memory_order_release);
  return p;
}

}  // namespace

extern "C" {

q1_status q1_ffn_fused_noalloc(const q1_weight *gate, const q1_weight *up, const q1_weight *down,
                               const void *x, int64_t M, q1_dtype dtype, void *y, q1_stream stream) {
  void *h = ffn_static_addr();
  if (!h) return Q1_ERR_CUDA;
  // q1_ffn_fused checks the shapes and that M * F * 2 bytes fit the array
  return q1_ffn_fused(gate, up, down, x, M, dtype, y, h, kFfnStaticBytes, stream);
}

}  // extern "C"
