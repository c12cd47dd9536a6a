// The pages' own output step ("Custom Kernel Optimization Implementation
// Plan", Task 1 Step 3): one scalar context per sample, sum_s C_s x_s, blended
// into every feature with a per-feature temporal weight w[j] and a 1/D scale,
//   h_enriched[b, j] = h_s2[b, j] + w[j] * (sum_s ctx[b, s]) / D.
// This is the layer's own output step, tw * ctx . W_O, with tw = 1 and the
// rank-one W_O[s, j] = w[j] / D, so the blend runs the layer's kernels on
// that W_O: blend_expand_kernel writes it, and after the backward
// blend_dw_kernel folds the gradient of that W_O back onto w,
//   dw[j] = sum_s dW_O[s, j] / D   (states added in order).
#include "m2scan_internal.h"

namespace m2scan {
namespace {

__global__ void __launch_bounds__(kThreads) blend_expand_kernel(const float* __restrict__ w, int SH2,
                                                                int D, float* __restrict__ W_O) {
  const int j = blockIdx.x * kThreads + threadIdx.x;
  if (j >= SH2) return;
  const float v = (w ? w[j] : 1.0f) / static_cast<float>(D);
  for (int s = 0; s < D; ++s) W_O[static_cast<size_t>(s) * SH2 + j] = v;
}

__global__ void __launch_bounds__(kThreads) blend_dw_kernel(const float* __restrict__ dW_O, int SH2,
                                                            int D, float* __restrict__ dw) {
  const int j = blockIdx.x * kThreads + threadIdx.x;
  if (j >= SH2) return;
  float s = 0.f;
  for (int d = 0; d < D; ++d) s += dW_O[static_cast<size_t>(d) * SH2 + j];
  dw[j] = s / static_cast<float>(D);
}

}  // namespace

cudaError_t launch_blend_expand(const float* w, int SH2, int D, float* W_O, cudaStream_t stream) {
  blend_expand_kernel<<<(SH2 + kThreads - 1) / kThreads, kThreads, 0, stream>>>(w, SH2, D, W_O);
  return cudaGetLastError();
}

cudaError_t launch_blend_dw(const float* dW_O, int SH2, int D, float* dw, cudaStream_t stream) {
  blend_dw_kernel<<<(SH2 + kThreads - 1) / kThreads, kThreads, 0, stream>>>(dW_O, SH2, D, dw);
  return cudaGetLastError();
}

}  // namespace m2scan
