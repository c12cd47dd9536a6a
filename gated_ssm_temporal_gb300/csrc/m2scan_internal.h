// Internal declarations shared by the m2scan host API and its kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace m2scan {

constexpr int kThreads = 256;     // threads per CTA of the generic and small kernels
constexpr int kMaxStages = 6;     // copy-ring depth of the fused kernels, at most
constexpr int kMaxSlots = 152;    // CTAs (= weight-gradient slots) per call, at most
constexpr int kTileRows = 128;    // rows (samples x K) per pass-1 tile, at most
constexpr int kChunk = 32;        // SH2 columns per pass-1 chunk (128 bytes)

// Arguments of the fused kernels. The three tensor maps describe h_history as
// a 3-D tensor [SH2, K, B] (box [32, K, S_max]) and h_s2 / d_h_enriched as 2-D
// tensors [SH2, B] (box [32, S_max]), all with 128-byte swizzle. Offsets are
// bytes from the 1024-aligned start of dynamic shared memory.
struct alignas(128) FastArgs {
  CUtensorMap tm_h;
  CUtensorMap tm_hs;
  CUtensorMap tm_g;
  const float* h_history;
  const float* h_s2;
  const float* g;
  const float* W_A;
  const float* W_B;
  const float* W_C;
  const float* W_O;
  float* out0;  // forward: h_enriched; backward: d_h_history
  float* out1;  // backward: d_h_s2
  float* ws;    // backward: weight-gradient slots [P][4][SH2*D]
  const float* gate_scale;  // one float multiplying every gate, or null (1)
  unsigned* err;
  unsigned long long* trace;  // debug timeline buffer (builds with M2SCAN_TRACE), else null
  long long B;
  int K;
  int SH2;
  int S_max;    // samples per tile, at most (also the TMA box depth)
  int SG;       // samples per pass-2 sample item
  int stage_bytes;
  int hc_bytes;  // bytes of the h_history box (S_max*K rows of 128 bytes)
  int sc_bytes;  // bytes of one h_s2 / d_h_enriched box (S_max rows)
  int off_S;     // offset of the h_s2 box inside a chunk stage
  int off_G;     // offset of the d_h_enriched box inside a chunk stage
  int off_wab, off_wct, off_wo, off_p, off_cs, off_ctx, off_dctx, off_dc, off_bar;
  int off_hlo;    // tensor-core path: two [128 x 32] buffers of h - tf32(h)
  int off_wt;     // tensor-core path: W_A|W_B transposed, K-major tiles (tf32 part)
  int n_stages;   // depth of the copy ring
  int tc;         // 1: tensor-core kernel (fwd_tc / bwd_tc), 2: tensor-core forward for D = 4, 16
  int tmem_cols;  // TMEM columns allocated by each CTA (power of two)
  int smem_bytes;
  int Dr;       // tensor-core kernels for D = 16: the layer's D (4, 8 or 16); states
                // Dr .. 15 are zero-padded inside the kernel
  float tw;
};

struct GenericArgs {
  const float* h_history;
  const float* h_s2;
  const float* g;
  const float* W_A;
  const float* W_B;
  const float* W_C;
  const float* W_O;
  float* out0;
  float* out1;
  float* ws;
  long long B;
  int K;
  int SH2;
  int D;
  float tw;
  const float* gate_scale;  // one float multiplying every gate, or null (1)
  int staged = 0;           // set by launch_generic: weights, h rows and slot in shared memory
};

// Shapes of the fused tensor-core kernels (the fast path of m2scan.h).
inline bool fast_path_ok(int K, int SH2, int D) {
  return (D == 4 || D == 8 || D == 16) && SH2 >= kChunk && SH2 % kChunk == 0 && SH2 <= 256 &&
         SH2 * D <= 4096 && K >= 1 && K <= kTileRows;
}
size_t generic_smem_bytes(bool bwd, int K, int SH2, int D);

// Tensor-core kernels for wide states (D = 64, SH2 % 128 == 0, K <= 128).
bool wide_path_ok(int K, int SH2, int D);
int wide_ranges(int64_t B);
size_t wide_bwd_workspace_bytes(int64_t B, int32_t K, int32_t SH2);
cudaError_t launch_wide_fwd(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw, int64_t B,
                            int K, int SH2, float* h_enriched, const float* gate_scale, unsigned* err,
                            cudaStream_t stream);
cudaError_t launch_wide_bwd(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw,
                            const float* g, int64_t B, int K, int SH2, float* d_h_history,
                            float* d_h_s2, float* dW_A, float* dW_B, float* dW_C, float* dW_O,
                            void* workspace, const float* gate_scale, unsigned* err,
                            cudaStream_t stream, int* n_launches);
cudaError_t prepare_wide_kernels();
// Warp-specialised tensor-core forward (D in {8, 16}).
bool fwd_tc_plan(int K, int SH2, int D, FastArgs* a);
cudaError_t launch_fwd_tc(int D, const FastArgs& a, int grid, cudaStream_t stream);
// Warp-specialised tensor-core forward for D = 16 (8 compute warps, two TMEM
// accumulator sets; plan->tc = 2).
bool fwd_tc16_plan(int K, int SH2, int D, FastArgs* a);
cudaError_t launch_fwd_tc16(const FastArgs& a, int grid, cudaStream_t stream);
// Tensor-core forward with bf16 activations (D = 16, SH2 % 64 == 0, SH2 <= 256,
// K <= 128; plan->tc = 3). tm_h / tm_hs must describe bf16 tensors.
bool fwd_bf16_plan(int K, int SH2, int D, FastArgs* a);
cudaError_t launch_fwd_bf16(const FastArgs& a, int grid, cudaStream_t stream);
cudaError_t prepare_fwd_bf16_kernels(int max_smem);
// Warp-specialised tensor-core backward (D = 4, 8, 16; plan->Dr = D).
bool bwd_tc_plan(int K, int SH2, int D, FastArgs* a);
cudaError_t launch_bwd_tc(const FastArgs& a, int grid, cudaStream_t stream);
// bf16: the activations (h_history, h_s2, g, out0, out1) are bfloat16. The
// staged form is used when generic_staged_smem_bytes fits max_smem; the plain
// form needs generic_smem_bytes <= max_smem (the caller checks that).
cudaError_t launch_generic(bool bwd, GenericArgs a, int grid, int max_smem, cudaStream_t stream,
                           bool bf16 = false);
cudaError_t launch_reduce(const float* ws, int slots, int n, float* dW_A, float* dW_B,
                          float* dW_C, float* dW_O, cudaStream_t stream);
// Bias-gradient column sum (two launches): partial sums of P = colsum_partials(N)
// row ranges into part [P][C], then their fixed-order sum into db.
int colsum_partials(long long N);
// The pages' per-feature blend as the layer's output step: W_O[s, j] = w[j] / D
// (w may be null: ones), and dw[j] = sum_s dW_O[s, j] / D.
cudaError_t launch_blend_expand(const float* w, int SH2, int D, float* W_O, cudaStream_t stream);
cudaError_t launch_blend_dw(const float* dW_O, int SH2, int D, float* dw, cudaStream_t stream);
cudaError_t launch_colsum(const float* dy, long long N, int C, float* db, int accumulate,
                          float* part, cudaStream_t stream, int* n_launches);

unsigned* device_error_word();  // device address of the error word (current device)

// TMA descriptor of a 2-D or 3-D fp32 tensor with the given swizzle (driver
// entry point looked up at set-up; L2 promotion 256 B, zero fill out of bounds).
CUresult encode_tensor_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
                           const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle,
                           CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_FLOAT32);

// Tensor-core backward with bf16 activations (D = 16, SH2 % 64 == 0,
// SH2 <= 256, K <= 128, B * K < 2^31). tm_h = h_history as [B*K rows][SH2]
// bf16 (box 64 x 128 rows), tm_hs / tm_g = h_s2 / d_h_enriched [B][SH2] bf16
// (box 64 x S_max), all 128-byte swizzle; ws = the weight-gradient slots.
bool bwd_bf16_tc_plan(int64_t B, int K, int SH2, int D, FastArgs* a);
cudaError_t launch_bwd_bf16_tc(const FastArgs& a, int grid, cudaStream_t stream);
cudaError_t prepare_bwd_bf16_kernels();

// Self-test of the bounded barrier wait (one CTA; see m2scan_selftest.cu).
cudaError_t launch_wait_timeout_selftest(unsigned* err, unsigned long long limit_ns,
                                         unsigned long long* out, cudaStream_t stream);

}  // namespace m2scan
