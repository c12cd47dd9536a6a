// m2scan_bwd_noalloc: the backward for callers that cannot allocate device
// memory themselves (see include/m2scan.h). The weight-gradient slots live in
// a fixed-size array that this library places in every GPU's global memory;
// the call then runs exactly the kernels of m2scan_bwd on that array.
#include <cuda_runtime.h>

#include <mutex>

#include "m2scan.h"

namespace {

// Weight-gradient scratch shared by every m2scan_bwd_noalloc call on a device.
// Every GPU that loads this library holds these bytes until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[M2SCAN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device. The name
// g_noalloc_scratch in host code is only a host-side stand-in, so the address
// is looked up once per device, with that device current.
m2scan_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return M2SCAN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return M2SCAN_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return M2SCAN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return M2SCAN_OK;
}

}  // namespace

extern "C" m2scan_status m2scan_bwd_noalloc(
    const float* h_history, const float* h_s2, const float* W_A, const float* W_B,
    const float* W_C, const float* W_O, float tw, const float* d_h_enriched, int64_t B, int32_t K,
    int32_t SH2, int32_t D, float* d_h_history, float* d_h_s2, float* dW_A, float* dW_B,
    float* dW_C, float* dW_O, m2scan_stream_t stream) {
  const size_t need = m2scan_bwd_workspace_bytes(B, K, SH2, D);
  if (need == 0)  // invalid shape (reported by m2scan_bwd) or B == 0: no scratch is used
    return m2scan_bwd(h_history, h_s2, W_A, W_B, W_C, W_O, tw, d_h_enriched, B, K, SH2, D,
                      d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O, nullptr, 0, stream);
  if (need > M2SCAN_NOALLOC_SCRATCH_BYTES) return M2SCAN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const m2scan_status st = scratch_address(&scratch);
  if (st != M2SCAN_OK) return st;
  return m2scan_bwd(h_history, h_s2, W_A, W_B, W_C, W_O, tw, d_h_enriched, B, K, SH2, D,
                    d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O, scratch,
                    M2SCAN_NOALLOC_SCRATCH_BYTES, stream);
}
