// Host side of the m2scan C ABI: argument checks, kernel-path choice, TMA
// descriptor encoding and launches. Nothing here synchronises the device
// except m2scan_read_device_flags, which says so.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/m2scan.h"
#include "m2scan_internal.h"

namespace m2scan {
cudaError_t prepare_generic_kernels(int max_smem);
cudaError_t prepare_fwd_tc_kernels(int max_smem);
cudaError_t prepare_bwd_tc_kernels(int max_smem);
cudaError_t prepare_fwd_tc16_kernels(int max_smem);
}  // namespace m2scan

using namespace m2scan;

// Device error word: bit kErrWaitTimeout is set by a kernel whose bounded
// wait on a copy gave up.
__device__ unsigned g_m2scan_err_word;

namespace {

thread_local int t_last_cuda_error = 0;
thread_local int t_last_launches = 0;
std::atomic<int> g_force_generic{0};

constexpr int kMaxDevices = 64;
std::mutex g_prep_mutex;
bool g_prepared[kMaxDevices] = {};
unsigned* g_err_ptr[kMaxDevices] = {};
int g_max_smem[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

m2scan_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return M2SCAN_ERR_CUDA;
}

// Per-device one-time set-up: shared-memory limits of the kernels, the device
// address of the error word and the TMA descriptor encoder.
m2scan_status prepare_device(int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return M2SCAN_ERR_DEVICE;
  // A host thread that has made no runtime call yet has no current context,
  // and the tensor-map encoder (a driver entry point) needs one: make the
  // device's primary context current on this thread.
  if ((e = cudaSetDevice(dev)) != cudaSuccess) return cuda_fail(e);
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_prep_mutex);
  if (g_prepared[dev]) return M2SCAN_OK;
  int major = 0, minor = 0, smem = 0;
  if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
    return cuda_fail(e);
  if (major != 10 || minor != 3) return M2SCAN_ERR_DEVICE;  // built for sm_103a only
  if ((e = prepare_generic_kernels(smem)) != cudaSuccess) return cuda_fail(e);
  if ((e = prepare_fwd_tc_kernels(smem)) != cudaSuccess) return cuda_fail(e);
  if ((e = prepare_bwd_tc_kernels(smem)) != cudaSuccess) return cuda_fail(e);
  if ((e = prepare_fwd_tc16_kernels(smem)) != cudaSuccess) return cuda_fail(e);
  if ((e = prepare_fwd_bf16_kernels(smem)) != cudaSuccess) return cuda_fail(e);
  if ((e = prepare_wide_kernels()) != cudaSuccess) return cuda_fail(e);
  if ((e = prepare_bwd_bf16_kernels()) != cudaSuccess) return cuda_fail(e);
  void* p = nullptr;
  if ((e = cudaGetSymbolAddress(&p, g_m2scan_err_word)) != cudaSuccess) return cuda_fail(e);
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (q != cudaDriverEntryPointSuccess || !fn) return M2SCAN_ERR_DEVICE;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  g_err_ptr[dev] = static_cast<unsigned*>(p);
  g_max_smem[dev] = smem;
  g_prepared[dev] = true;
  return M2SCAN_OK;
}

// Debug timeline of the fused kernels (builds with M2SCAN_TRACE): the address
// of a device buffer given by M2SCAN_TRACE_PTR, else none.
unsigned long long* trace_buffer() {
#ifdef M2SCAN_TRACE
  static unsigned long long* p = [] {
    const char* s = getenv("M2SCAN_TRACE_PTR");
    return s ? reinterpret_cast<unsigned long long*>(strtoull(s, nullptr, 0)) : nullptr;
  }();
  return p;
#else
  return nullptr;
#endif
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  uintptr_t lo, hi;  // [lo, hi)
};

Span span(const void* p, uint64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Span{lo, lo + static_cast<uintptr_t>(bytes)};
}

bool overlaps(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

// Shape checks shared by every entry point. Element counts must stay below 2^40.
m2scan_status check_shape(int64_t B, int32_t K, int32_t SH2, int32_t D) {
  if (B < 0 || K < 1 || SH2 < 4 || SH2 % 4 != 0 || D < 1) return M2SCAN_ERR_SHAPE;
  const uint64_t lim = 1ull << 40;
  if (static_cast<uint64_t>(K) * static_cast<uint64_t>(SH2) > lim) return M2SCAN_ERR_SHAPE;
  if (B > 0 && static_cast<uint64_t>(B) > lim / (static_cast<uint64_t>(K) * SH2))
    return M2SCAN_ERR_SHAPE;
  if (static_cast<uint64_t>(SH2) * static_cast<uint64_t>(D) > (1ull << 28)) return M2SCAN_ERR_SHAPE;
  return M2SCAN_OK;
}

int slots_for(int64_t B) { return B < kMaxSlots ? static_cast<int>(B) : kMaxSlots; }

// 1 = fused tensor-core kernels (plan->tc says which forward), 2 = generic,
// 3 = wide-state tensor-core kernels, 0 = unsupported.
int choose_path(int64_t B, int32_t K, int32_t SH2, int32_t D, bool bwd, int max_smem,
                FastArgs* plan) {
  if (!g_force_generic.load() && B <= 0x7fffffffll) {
    if (!bwd && fwd_tc16_plan(K, SH2, D, plan) && plan->smem_bytes <= max_smem) return 1;
    if (!bwd && fwd_tc_plan(K, SH2, D, plan) && plan->smem_bytes <= max_smem) return 1;
    if (bwd && bwd_tc_plan(K, SH2, D, plan) && plan->smem_bytes <= max_smem) return 1;
    // (the wide-state kernels address rows with 32-bit TMA coordinates)
    if (wide_path_ok(K, SH2, D) && B * K < (1ll << 31)) return 3;
  }
  if (generic_smem_bytes(bwd, K, SH2, D) <= static_cast<size_t>(max_smem)) return 2;
  return 0;
}

CUresult encode_map(CUtensorMap* m, const float* ptr, int rank, const cuuint64_t* dims,
                    const cuuint64_t* strides, const cuuint32_t* box,
                    CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_FLOAT32) {
  const cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, type, rank, const_cast<float*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

CUresult m2scan::encode_tensor_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
                                   const cuuint64_t* strides, const cuuint32_t* box,
                                   CUtensorMapSwizzle swizzle, CUtensorMapDataType type) {
  const cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, type, rank, const_cast<void*>(ptr), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

namespace {

// bf16 h_history [SH2, K, B] (box [64, K, S_max]) and h_s2 [SH2, B] (box
// [64, S_max]): 64 bf16 = one 128-byte swizzled row per box row.
bool encode_bf16_maps(FastArgs* a, const void* h_history, const void* h_s2, int64_t B) {
  const cuuint64_t SH2 = static_cast<cuuint64_t>(a->SH2), K = static_cast<cuuint64_t>(a->K);
  const cuuint64_t d3[3] = {SH2, K, static_cast<cuuint64_t>(B)};
  const cuuint64_t s3[2] = {SH2 * 2, SH2 * K * 2};
  const cuuint32_t b3[3] = {64u, static_cast<cuuint32_t>(K), static_cast<cuuint32_t>(a->S_max)};
  if (encode_map(&a->tm_h, static_cast<const float*>(h_history), 3, d3, s3, b3,
                 CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != CUDA_SUCCESS)
    return false;
  const cuuint64_t d2[2] = {SH2, static_cast<cuuint64_t>(B)};
  const cuuint64_t s2[1] = {SH2 * 2};
  const cuuint32_t b2[2] = {64u, static_cast<cuuint32_t>(a->S_max)};
  if (encode_map(&a->tm_hs, static_cast<const float*>(h_s2), 2, d2, s2, b2,
                 CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) != CUDA_SUCCESS)
    return false;
  std::memcpy(&a->tm_g, &a->tm_hs, sizeof(CUtensorMap));
  return true;
}

// Tensor maps of the fused tensor-core kernels: h_history as [SH2, K, B] with box
// [32, K, S_max]; h_s2 and (backward) d_h_enriched as [SH2, B] with box [32, S_max].
bool encode_fast_maps(FastArgs* a, const float* h_history, const float* h_s2, const float* g,
                      int64_t B) {
  const cuuint64_t SH2 = static_cast<cuuint64_t>(a->SH2), K = static_cast<cuuint64_t>(a->K);
  const cuuint64_t d3[3] = {SH2, K, static_cast<cuuint64_t>(B)};
  const cuuint64_t s3[2] = {SH2 * 4, SH2 * K * 4};
  const cuuint32_t b3[3] = {static_cast<cuuint32_t>(kChunk), static_cast<cuuint32_t>(K),
                            static_cast<cuuint32_t>(a->S_max)};
  if (encode_map(&a->tm_h, h_history, 3, d3, s3, b3) != CUDA_SUCCESS) return false;
  const cuuint64_t d2[2] = {SH2, static_cast<cuuint64_t>(B)};
  const cuuint64_t s2[1] = {SH2 * 4};
  const cuuint32_t b2[2] = {static_cast<cuuint32_t>(kChunk), static_cast<cuuint32_t>(a->S_max)};
  if (encode_map(&a->tm_hs, h_s2, 2, d2, s2, b2) != CUDA_SUCCESS) return false;
  if (g) {
    if (encode_map(&a->tm_g, g, 2, d2, s2, b2) != CUDA_SUCCESS) return false;
  } else {
    std::memcpy(&a->tm_g, &a->tm_hs, sizeof(CUtensorMap));
  }
  return true;
}

}  // namespace

extern "C" {

const char* m2scan_status_str(m2scan_status s) {
  switch (s) {
    case M2SCAN_OK: return "ok";
    case M2SCAN_ERR_NULL: return "a required pointer is NULL";
    case M2SCAN_ERR_SHAPE: return "invalid shape (need B>=0, K>=1, SH2>=4, SH2%4==0, D>=1)";
    case M2SCAN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case M2SCAN_ERR_ALIAS: return "an output overlaps an input or another output";
    case M2SCAN_ERR_WORKSPACE: return "workspace missing or smaller than m2scan_bwd_workspace_bytes";
    case M2SCAN_ERR_UNSUPPORTED: return "shape not supported by any kernel instance";
    case M2SCAN_ERR_CUDA: return "a CUDA runtime call failed (see m2scan_last_cuda_error)";
    case M2SCAN_ERR_DEVICE: return "no usable sm_103 device is current";
  }
  return "unknown status";
}

int m2scan_last_cuda_error(void) { return t_last_cuda_error; }

int m2scan_last_launch_count(void) { return t_last_launches; }

int m2scan_set_force_generic(int force) { return g_force_generic.exchange(force ? 1 : 0); }

int m2scan_path_for(int32_t K, int32_t SH2, int32_t D) {
  if (check_shape(1, K, SH2, D) != M2SCAN_OK) return 0;
  FastArgs plan;
  const int max_smem = 227 * 1024;
  return choose_path(1, K, SH2, D, true, max_smem, &plan);
}

int m2scan_fwd_path_for(int32_t K, int32_t SH2, int32_t D) {
  if (check_shape(1, K, SH2, D) != M2SCAN_OK) return 0;
  FastArgs plan;
  const int max_smem = 227 * 1024;
  return choose_path(1, K, SH2, D, false, max_smem, &plan);
}

size_t m2scan_bwd_workspace_bytes(int64_t B, int32_t K, int32_t SH2, int32_t D) {
  if (check_shape(B, K, SH2, D) != M2SCAN_OK || B == 0) return 0;
  const size_t slots = static_cast<size_t>(slots_for(B)) * 4 * static_cast<size_t>(SH2) * D * sizeof(float);
  if (!wide_path_ok(K, SH2, D)) return slots;
  // the wide-state kernels also keep dA|dB and [dC | ctx] there; the generic
  // kernels (forced for tests) use the slots alone
  const size_t wide = wide_bwd_workspace_bytes(B, K, SH2);
  return wide > slots ? wide : slots;
}

m2scan_status m2scan_selftest_wait_timeout(uint64_t limit_ns, uint64_t* out,
                                           m2scan_stream_t stream) {
  if (!out) return M2SCAN_ERR_NULL;
  if (!aligned16(out)) return M2SCAN_ERR_ALIGN;
  if (limit_ns < 1000ull || limit_ns > 100000000ull) return M2SCAN_ERR_SHAPE;
  int dev = 0;
  m2scan_status st = prepare_device(&dev);
  if (st != M2SCAN_OK) return st;
  const cudaError_t e = launch_wait_timeout_selftest(
      g_err_ptr[dev], limit_ns, reinterpret_cast<unsigned long long*>(out), stream);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 1;
  return M2SCAN_OK;
}

m2scan_status m2scan_read_device_flags(uint32_t* flags) {
  if (!flags) return M2SCAN_ERR_NULL;
  int dev = 0;
  m2scan_status st = prepare_device(&dev);
  if (st != M2SCAN_OK) return st;
  unsigned v = 0, zero = 0;
  cudaError_t e = cudaMemcpy(&v, g_err_ptr[dev], sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(g_err_ptr[dev], &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = v;
  return M2SCAN_OK;
}

m2scan_status m2scan_fwd_ex(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw,
                            const float* gate_scale, int64_t B, int32_t K, int32_t SH2,
                            int32_t D, float* h_enriched, m2scan_stream_t stream) {
  t_last_launches = 0;
  m2scan_status st = check_shape(B, K, SH2, D);
  if (st != M2SCAN_OK) return st;
  if (!W_A || !W_B || !W_C || !W_O) return M2SCAN_ERR_NULL;
  if (B > 0 && (!h_history || !h_s2 || !h_enriched)) return M2SCAN_ERR_NULL;
  const void* ptrs[] = {h_history, h_s2, W_A, W_B, W_C, W_O, h_enriched};
  for (const void* p : ptrs)
    if (!aligned16(p)) return M2SCAN_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(gate_scale) & 3u) != 0) return M2SCAN_ERR_ALIGN;
  const uint64_t nw = static_cast<uint64_t>(SH2) * D * 4;
  const uint64_t nb = static_cast<uint64_t>(B) * SH2 * 4;
  const Span out = span(h_enriched, nb);
  const Span ins[] = {span(h_history, nb * K), span(h_s2, nb), span(W_A, nw), span(W_B, nw),
                      span(W_C, nw), span(W_O, nw), span(gate_scale, gate_scale ? 4 : 0)};
  for (const Span& s : ins)
    if (overlaps(out, s)) return M2SCAN_ERR_ALIAS;
  if (B == 0) return M2SCAN_OK;
  int dev = 0;
  if ((st = prepare_device(&dev)) != M2SCAN_OK) return st;
  FastArgs fa;
  const int path = choose_path(B, K, SH2, D, false, g_max_smem[dev], &fa);
  if (path == 0) return M2SCAN_ERR_UNSUPPORTED;
  const int grid = slots_for(B);
  cudaError_t e;
  if (path == 1) {
    fa.h_history = h_history; fa.h_s2 = h_s2; fa.g = nullptr;
    fa.W_A = W_A; fa.W_B = W_B; fa.W_C = W_C; fa.W_O = W_O;
    fa.out0 = h_enriched; fa.out1 = nullptr; fa.ws = nullptr; fa.gate_scale = gate_scale;
    fa.err = g_err_ptr[dev]; fa.B = B; fa.tw = tw; fa.trace = trace_buffer();
    if (!encode_fast_maps(&fa, h_history, h_s2, nullptr, B)) return M2SCAN_ERR_UNSUPPORTED;
    e = fa.tc == 2 ? launch_fwd_tc16(fa, grid, stream) : launch_fwd_tc(D, fa, grid, stream);
  } else if (path == 3) {
    e = launch_wide_fwd(h_history, h_s2, W_A, W_B, W_C, W_O, tw, B, K, SH2, h_enriched,
                        gate_scale, g_err_ptr[dev], stream);
  } else {
    GenericArgs ga{h_history, h_s2, nullptr, W_A, W_B, W_C, W_O, h_enriched, nullptr, nullptr,
                   B, K, SH2, D, tw, gate_scale};
    e = launch_generic(false, ga, grid, g_max_smem[dev], stream);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 1;
  return M2SCAN_OK;
}

m2scan_status m2scan_fwd_bf16(const void* h_history, const void* h_s2, const float* W_A,
                              const float* W_B, const float* W_C, const float* W_O, float tw,
                              const float* gate_scale, int64_t B, int32_t K, int32_t SH2,
                              int32_t D, void* h_enriched, m2scan_stream_t stream) {
  t_last_launches = 0;
  m2scan_status st = check_shape(B, K, SH2, D);
  if (st != M2SCAN_OK) return st;
  FastArgs fa;
  if (!fwd_bf16_plan(K, SH2, D, &fa) || B > 0x7fffffffll) return M2SCAN_ERR_UNSUPPORTED;
  if (!W_A || !W_B || !W_C || !W_O) return M2SCAN_ERR_NULL;
  if (B > 0 && (!h_history || !h_s2 || !h_enriched)) return M2SCAN_ERR_NULL;
  const void* ptrs[] = {h_history, h_s2, W_A, W_B, W_C, W_O, h_enriched};
  for (const void* p : ptrs)
    if (!aligned16(p)) return M2SCAN_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(gate_scale) & 3u) != 0) return M2SCAN_ERR_ALIGN;
  const uint64_t nw = static_cast<uint64_t>(SH2) * D * 4;
  const uint64_t nb = static_cast<uint64_t>(B) * SH2 * 2;  // bf16 rows
  const Span out = span(h_enriched, nb);
  const Span ins[] = {span(h_history, nb * K), span(h_s2, nb), span(W_A, nw), span(W_B, nw),
                      span(W_C, nw), span(W_O, nw), span(gate_scale, gate_scale ? 4 : 0)};
  for (const Span& s : ins)
    if (overlaps(out, s)) return M2SCAN_ERR_ALIAS;
  if (B == 0) return M2SCAN_OK;
  int dev = 0;
  if ((st = prepare_device(&dev)) != M2SCAN_OK) return st;
  if (fa.smem_bytes > g_max_smem[dev]) return M2SCAN_ERR_UNSUPPORTED;
  fa.h_history = static_cast<const float*>(h_history);
  fa.h_s2 = static_cast<const float*>(h_s2);
  fa.g = nullptr;
  fa.W_A = W_A; fa.W_B = W_B; fa.W_C = W_C; fa.W_O = W_O;
  fa.out0 = static_cast<float*>(h_enriched); fa.out1 = nullptr; fa.ws = nullptr;
  fa.gate_scale = gate_scale;
  fa.err = g_err_ptr[dev]; fa.B = B; fa.tw = tw; fa.trace = trace_buffer();
  if (!encode_bf16_maps(&fa, h_history, h_s2, B)) return M2SCAN_ERR_UNSUPPORTED;
  const cudaError_t e = launch_fwd_bf16(fa, slots_for(B), stream);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 1;
  return M2SCAN_OK;
}

m2scan_status m2scan_fwd(const float* h_history, const float* h_s2, const float* W_A,
                         const float* W_B, const float* W_C, const float* W_O, float tw,
                         int64_t B, int32_t K, int32_t SH2, int32_t D, float* h_enriched,
                         m2scan_stream_t stream) {
  return m2scan_fwd_ex(h_history, h_s2, W_A, W_B, W_C, W_O, tw, nullptr, B, K, SH2, D,
                       h_enriched, stream);
}

size_t m2scan_blend_fwd_workspace_bytes(int32_t SH2, int32_t D) {
  if (SH2 < 4 || SH2 % 4 != 0 || D < 1) return 0;
  return static_cast<size_t>(SH2) * D * sizeof(float);
}

size_t m2scan_blend_bwd_workspace_bytes(int64_t B, int32_t K, int32_t SH2, int32_t D) {
  if (check_shape(B, K, SH2, D) != M2SCAN_OK) return 0;
  return m2scan_bwd_workspace_bytes(B, K, SH2, D) + 2 * m2scan_blend_fwd_workspace_bytes(SH2, D);
}

m2scan_status m2scan_fwd_blend(const float* h_history, const float* h_s2, const float* W_A,
                               const float* W_B, const float* W_C, const float* temporal_weight,
                               const float* gate_scale, int64_t B, int32_t K, int32_t SH2,
                               int32_t D, float* h_enriched, void* workspace,
                               size_t workspace_bytes, m2scan_stream_t stream) {
  t_last_launches = 0;
  m2scan_status st = check_shape(B, K, SH2, D);
  if (st != M2SCAN_OK) return st;
  const size_t need = m2scan_blend_fwd_workspace_bytes(SH2, D);
  if (!workspace || workspace_bytes < need) return M2SCAN_ERR_WORKSPACE;
  if (!aligned16(workspace) || !aligned16(temporal_weight)) return M2SCAN_ERR_ALIGN;
  const uint64_t nb = static_cast<uint64_t>(B) * SH2 * 4, nw = static_cast<uint64_t>(SH2) * D * 4;
  const Span ws = span(workspace, need);
  const Span others[] = {span(h_history, nb * K), span(h_s2, nb), span(W_A, nw), span(W_B, nw),
                         span(W_C, nw), span(h_enriched, nb),
                         span(temporal_weight, temporal_weight ? SH2 * 4ull : 0),
                         span(gate_scale, gate_scale ? 4 : 0)};
  for (const Span& o : others)
    if (overlaps(ws, o)) return M2SCAN_ERR_ALIAS;
  if (overlaps(span(h_enriched, nb), span(temporal_weight, temporal_weight ? SH2 * 4ull : 0)))
    return M2SCAN_ERR_ALIAS;
  if (B == 0) return M2SCAN_OK;
  int dev = 0;
  if ((st = prepare_device(&dev)) != M2SCAN_OK) return st;
  float* W_O = static_cast<float*>(workspace);
  cudaError_t e = launch_blend_expand(temporal_weight, SH2, D, W_O, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  st = m2scan_fwd_ex(h_history, h_s2, W_A, W_B, W_C, W_O, 1.0f, gate_scale, B, K, SH2, D,
                     h_enriched, stream);
  if (st == M2SCAN_OK) t_last_launches += 1;
  return st;
}

m2scan_status m2scan_bwd_blend(const float* h_history, const float* h_s2, const float* W_A,
                               const float* W_B, const float* W_C, const float* temporal_weight,
                               const float* gate_scale, const float* d_h_enriched, int64_t B,
                               int32_t K, int32_t SH2, int32_t D, float* d_h_history,
                               float* d_h_s2, float* dW_A, float* dW_B, float* dW_C,
                               float* d_temporal_weight, void* workspace, size_t workspace_bytes,
                               m2scan_stream_t stream) {
  t_last_launches = 0;
  m2scan_status st = check_shape(B, K, SH2, D);
  if (st != M2SCAN_OK) return st;
  const size_t need = m2scan_blend_bwd_workspace_bytes(B, K, SH2, D);
  if (!workspace || workspace_bytes < need) return M2SCAN_ERR_WORKSPACE;
  if (!aligned16(workspace) || !aligned16(temporal_weight) || !aligned16(d_temporal_weight))
    return M2SCAN_ERR_ALIGN;
  const size_t base = m2scan_bwd_workspace_bytes(B, K, SH2, D);
  const size_t nwo = m2scan_blend_fwd_workspace_bytes(SH2, D);
  unsigned char* w8 = static_cast<unsigned char*>(workspace);
  float* W_O = reinterpret_cast<float*>(w8 + base);
  float* dW_O = reinterpret_cast<float*>(w8 + base + nwo);
  const Span ws = span(workspace, need);
  const Span tw_in = span(temporal_weight, temporal_weight ? SH2 * 4ull : 0);
  const Span tw_out = span(d_temporal_weight, d_temporal_weight ? SH2 * 4ull : 0);
  if (overlaps(ws, tw_in) || overlaps(ws, tw_out) || overlaps(tw_in, tw_out))
    return M2SCAN_ERR_ALIAS;
  const uint64_t nb = static_cast<uint64_t>(B) * SH2 * 4, nw = static_cast<uint64_t>(SH2) * D * 4;
  const Span layer[] = {span(h_history, nb * K), span(h_s2, nb), span(W_A, nw), span(W_B, nw),
                        span(W_C, nw), span(d_h_enriched, nb), span(d_h_history, nb * K),
                        span(d_h_s2, nb), span(dW_A, nw), span(dW_B, nw), span(dW_C, nw),
                        span(gate_scale, gate_scale ? 4 : 0)};
  for (const Span& o : layer)
    if (overlaps(ws, o) || overlaps(tw_out, o)) return M2SCAN_ERR_ALIAS;
  if (B > 0) {
    int dev = 0;
    if ((st = prepare_device(&dev)) != M2SCAN_OK) return st;
  }
  int n = 0;
  if (B > 0) {
    const cudaError_t e = launch_blend_expand(temporal_weight, SH2, D, W_O, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    ++n;
  }
  st = m2scan_bwd_ex(h_history, h_s2, W_A, W_B, W_C, W_O, 1.0f, gate_scale, d_h_enriched, B, K,
                     SH2, D, d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace, base, stream);
  if (st != M2SCAN_OK) return st;
  n += t_last_launches;
  if (d_temporal_weight) {
    if (B == 0) {
      const cudaError_t e = cudaMemsetAsync(d_temporal_weight, 0, SH2 * 4ull, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    } else {
      const cudaError_t e = launch_blend_dw(dW_O, SH2, D, d_temporal_weight, stream);
      if (e != cudaSuccess) return cuda_fail(e);
      ++n;
    }
  }
  t_last_launches = n;
  return M2SCAN_OK;
}

size_t m2scan_bias_grad_workspace_bytes(int64_t N, int32_t C) {
  if (N < 0 || C < 1 || static_cast<uint64_t>(N) * static_cast<uint64_t>(C) > (1ull << 40)) return 0;
  if (N == 0) return 0;
  return static_cast<size_t>(colsum_partials(N)) * static_cast<size_t>(C) * sizeof(float);
}

m2scan_status m2scan_bias_grad(const float* dy, int64_t N, int32_t C, float* db,
                               int32_t accumulate, void* workspace, size_t workspace_bytes,
                               m2scan_stream_t stream) {
  t_last_launches = 0;
  if (N < 0 || C < 1 || static_cast<uint64_t>(N) * static_cast<uint64_t>(C) > (1ull << 40))
    return M2SCAN_ERR_SHAPE;
  if (!db || (N > 0 && !dy)) return M2SCAN_ERR_NULL;
  if (!aligned16(dy) || !aligned16(db)) return M2SCAN_ERR_ALIGN;
  const size_t need = m2scan_bias_grad_workspace_bytes(N, C);
  if (N > 0 && (!workspace || workspace_bytes < need)) return M2SCAN_ERR_WORKSPACE;
  if (N > 0 && !aligned16(workspace)) return M2SCAN_ERR_ALIGN;
  const Span out = span(db, static_cast<uint64_t>(C) * 4);
  const Span in = span(dy, static_cast<uint64_t>(N) * C * 4);
  const Span ws = span(workspace, N > 0 ? need : 0);
  if (overlaps(out, in) || overlaps(out, ws) || overlaps(in, ws)) return M2SCAN_ERR_ALIAS;
  int dev = 0;
  m2scan_status st = prepare_device(&dev);
  if (st != M2SCAN_OK) return st;
  if (N == 0) {
    if (accumulate) return M2SCAN_OK;  // adding an empty sum
    const cudaError_t e = cudaMemsetAsync(db, 0, static_cast<size_t>(C) * 4, stream);
    return e == cudaSuccess ? M2SCAN_OK : cuda_fail(e);
  }
  int n = 0;
  const cudaError_t e = launch_colsum(dy, N, C, db, accumulate ? 1 : 0,
                                      static_cast<float*>(workspace), stream, &n);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = n;
  return M2SCAN_OK;
}

m2scan_status m2scan_bwd_ex(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw,
                            const float* gate_scale, const float* d_h_enriched, int64_t B,
                            int32_t K, int32_t SH2, int32_t D, float* d_h_history,
                            float* d_h_s2, float* dW_A, float* dW_B, float* dW_C, float* dW_O,
                            void* workspace, size_t workspace_bytes, m2scan_stream_t stream) {
  t_last_launches = 0;
  m2scan_status st = check_shape(B, K, SH2, D);
  if (st != M2SCAN_OK) return st;
  if (!W_A || !W_B || !W_C || !W_O || !dW_A || !dW_B || !dW_C || !dW_O) return M2SCAN_ERR_NULL;
  if (B > 0 && (!h_history || !h_s2 || !d_h_enriched || !d_h_history || !d_h_s2))
    return M2SCAN_ERR_NULL;
  const void* ptrs[] = {h_history, h_s2, W_A, W_B, W_C, W_O, d_h_enriched, d_h_history,
                        d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return M2SCAN_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(gate_scale) & 3u) != 0) return M2SCAN_ERR_ALIGN;
  const size_t need = m2scan_bwd_workspace_bytes(B, K, SH2, D);
  if (need > 0 && (!workspace || workspace_bytes < need)) return M2SCAN_ERR_WORKSPACE;
  const uint64_t nw = static_cast<uint64_t>(SH2) * D * 4;
  const uint64_t nb = static_cast<uint64_t>(B) * SH2 * 4;
  const Span outs[] = {span(d_h_history, nb * K), span(d_h_s2, nb), span(dW_A, nw),
                       span(dW_B, nw), span(dW_C, nw), span(dW_O, nw), span(workspace, need)};
  const Span ins[] = {span(h_history, nb * K), span(h_s2, nb), span(W_A, nw), span(W_B, nw),
                      span(W_C, nw), span(W_O, nw), span(d_h_enriched, nb),
                      span(gate_scale, gate_scale ? 4 : 0)};
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
    for (const Span& s : ins)
      if (overlaps(outs[i], s)) return M2SCAN_ERR_ALIAS;
    for (size_t k = i + 1; k < sizeof(outs) / sizeof(outs[0]); ++k)
      if (overlaps(outs[i], outs[k])) return M2SCAN_ERR_ALIAS;
  }
  if (B == 0) {
    float* dws[] = {dW_A, dW_B, dW_C, dW_O};
    for (float* p : dws) {
      cudaError_t e = cudaMemsetAsync(p, 0, nw, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return M2SCAN_OK;
  }
  int dev = 0;
  if ((st = prepare_device(&dev)) != M2SCAN_OK) return st;
  FastArgs fa;
  const int path = choose_path(B, K, SH2, D, true, g_max_smem[dev], &fa);
  if (path == 0) return M2SCAN_ERR_UNSUPPORTED;
  const int grid = slots_for(B);
  float* ws = static_cast<float*>(workspace);
  cudaError_t e;
  if (path == 1) {
    fa.h_history = h_history; fa.h_s2 = h_s2; fa.g = d_h_enriched;
    fa.W_A = W_A; fa.W_B = W_B; fa.W_C = W_C; fa.W_O = W_O;
    fa.out0 = d_h_history; fa.out1 = d_h_s2; fa.ws = ws; fa.gate_scale = gate_scale;
    fa.err = g_err_ptr[dev]; fa.B = B; fa.tw = tw; fa.trace = trace_buffer();
    if (!encode_fast_maps(&fa, h_history, h_s2, d_h_enriched, B)) return M2SCAN_ERR_UNSUPPORTED;
    e = launch_bwd_tc(fa, grid, stream);
  } else if (path == 3) {
    int n = 0;
    e = launch_wide_bwd(h_history, h_s2, W_A, W_B, W_C, W_O, tw, d_h_enriched, B, K, SH2, d_h_history,
                        d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace, gate_scale, g_err_ptr[dev], stream,
                        &n);
    t_last_launches = n;
    if (e != cudaSuccess) return cuda_fail(e);
    return M2SCAN_OK;
  } else {
    GenericArgs ga{h_history, h_s2, d_h_enriched, W_A, W_B, W_C, W_O, d_h_history, d_h_s2, ws,
                   B, K, SH2, D, tw, gate_scale};
    e = launch_generic(true, ga, grid, g_max_smem[dev], stream);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_reduce(ws, grid, SH2 * D, dW_A, dW_B, dW_C, dW_O, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 2;
  return M2SCAN_OK;
}

m2scan_status m2scan_bwd_bf16(const void* h_history, const void* h_s2, const float* W_A,
                              const float* W_B, const float* W_C, const float* W_O, float tw,
                              const float* gate_scale, const void* d_h_enriched, int64_t B,
                              int32_t K, int32_t SH2, int32_t D, void* d_h_history, void* d_h_s2,
                              float* dW_A, float* dW_B, float* dW_C, float* dW_O, void* workspace,
                              size_t workspace_bytes, m2scan_stream_t stream) {
  t_last_launches = 0;
  m2scan_status st = check_shape(B, K, SH2, D);
  if (st != M2SCAN_OK) return st;
  if (!W_A || !W_B || !W_C || !W_O || !dW_A || !dW_B || !dW_C || !dW_O) return M2SCAN_ERR_NULL;
  if (B > 0 && (!h_history || !h_s2 || !d_h_enriched || !d_h_history || !d_h_s2))
    return M2SCAN_ERR_NULL;
  const void* ptrs[] = {h_history, h_s2, W_A, W_B, W_C, W_O, d_h_enriched, d_h_history,
                        d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return M2SCAN_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(gate_scale) & 3u) != 0) return M2SCAN_ERR_ALIGN;
  const size_t need = m2scan_bwd_workspace_bytes(B, K, SH2, D);
  if (need > 0 && (!workspace || workspace_bytes < need)) return M2SCAN_ERR_WORKSPACE;
  const uint64_t nw = static_cast<uint64_t>(SH2) * D * 4;
  const uint64_t nb = static_cast<uint64_t>(B) * SH2 * 2;  // bf16 rows
  const Span outs[] = {span(d_h_history, nb * K), span(d_h_s2, nb), span(dW_A, nw),
                       span(dW_B, nw), span(dW_C, nw), span(dW_O, nw), span(workspace, need)};
  const Span ins[] = {span(h_history, nb * K), span(h_s2, nb), span(W_A, nw), span(W_B, nw),
                      span(W_C, nw), span(W_O, nw), span(d_h_enriched, nb),
                      span(gate_scale, gate_scale ? 4 : 0)};
  for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
    for (const Span& s : ins)
      if (overlaps(outs[i], s)) return M2SCAN_ERR_ALIAS;
    for (size_t k = i + 1; k < sizeof(outs) / sizeof(outs[0]); ++k)
      if (overlaps(outs[i], outs[k])) return M2SCAN_ERR_ALIAS;
  }
  if (B == 0) {
    float* dws[] = {dW_A, dW_B, dW_C, dW_O};
    for (float* p : dws) {
      cudaError_t e = cudaMemsetAsync(p, 0, nw, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return M2SCAN_OK;
  }
  int dev = 0;
  if ((st = prepare_device(&dev)) != M2SCAN_OK) return st;
  const int grid = slots_for(B);
  float* ws = static_cast<float*>(workspace);
  FastArgs fa{};
  if (!g_force_generic.load() && bwd_bf16_tc_plan(B, K, SH2, D, &fa) &&
      fa.smem_bytes <= g_max_smem[dev]) {
    // the tensor-core kernel: 2-D bf16 tensor maps, 128-byte swizzle
    const cuuint64_t sh = static_cast<cuuint64_t>(SH2);
    const cuuint64_t dh[2] = {sh, static_cast<cuuint64_t>(B) * K}, ds[2] = {sh, static_cast<cuuint64_t>(B)};
    const cuuint64_t str[1] = {sh * 2};
    const cuuint32_t bh[2] = {64, 128}, bs[2] = {64, static_cast<cuuint32_t>(fa.S_max)};
    const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (encode_tensor_map(&fa.tm_h, h_history, 2, dh, str, bh, sw, bf) != CUDA_SUCCESS ||
        encode_tensor_map(&fa.tm_hs, h_s2, 2, ds, str, bs, sw, bf) != CUDA_SUCCESS ||
        encode_tensor_map(&fa.tm_g, d_h_enriched, 2, ds, str, bs, sw, bf) != CUDA_SUCCESS)
      return M2SCAN_ERR_UNSUPPORTED;
    fa.W_A = W_A; fa.W_B = W_B; fa.W_C = W_C; fa.W_O = W_O;
    fa.out0 = static_cast<float*>(d_h_history); fa.out1 = static_cast<float*>(d_h_s2);
    fa.ws = ws; fa.gate_scale = gate_scale; fa.err = g_err_ptr[dev]; fa.B = B; fa.tw = tw;
    cudaError_t e = launch_bwd_bf16_tc(fa, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_reduce(ws, grid, SH2 * D, dW_A, dW_B, dW_C, dW_O, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    t_last_launches = 2;
    return M2SCAN_OK;
  }
  const size_t smem = generic_smem_bytes(true, K, SH2, D);
  if (smem > static_cast<size_t>(g_max_smem[dev])) return M2SCAN_ERR_UNSUPPORTED;
  GenericArgs ga{static_cast<const float*>(h_history), static_cast<const float*>(h_s2),
                 static_cast<const float*>(d_h_enriched), W_A, W_B, W_C, W_O,
                 static_cast<float*>(d_h_history), static_cast<float*>(d_h_s2), ws,
                 B, K, SH2, D, tw, gate_scale};
  cudaError_t e = launch_generic(true, ga, grid, g_max_smem[dev], stream, true);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_reduce(ws, grid, SH2 * D, dW_A, dW_B, dW_C, dW_O, stream);
  if (e != cudaSuccess) return cuda_fail(e);
  t_last_launches = 2;
  return M2SCAN_OK;
}

m2scan_status m2scan_bwd(const float* h_history, const float* h_s2, const float* W_A,
                         const float* W_B, const float* W_C, const float* W_O, float tw,
                         const float* d_h_enriched, int64_t B, int32_t K, int32_t SH2,
                         int32_t D, float* d_h_history, float* d_h_s2, float* dW_A,
                         float* dW_B, float* dW_C, float* dW_O, void* workspace,
                         size_t workspace_bytes, m2scan_stream_t stream) {
  return m2scan_bwd_ex(h_history, h_s2, W_A, W_B, W_C, W_O, tw, nullptr, d_h_enriched, B, K,
                       SH2, D, d_h_history, d_h_s2, dW_A, dW_B, dW_C, dW_O, workspace,
                       workspace_bytes, stream);
}

}  // extern "C"
