// Bias gradient of a fully connected layer: db[c] (+)= sum over rows r of
// dy[r, c] for a row-major [N, C] fp32 matrix ("Phase 3 Kernel Optimization
// Implementation Plan", Task 2: the two-phase reduction over the batch, block
// partials then a second pass over the partials in a fixed order).
//
// Phase 1 (colsum_partial_kernel): CTA p owns rows [p*N/P, (p+1)*N/P) and
// walks the columns in blocks of up to 256. For a block of Cb columns thread
// t takes column t % Cb and row phase t / Cb, so a warp always reads 32
// consecutive floats of the matrix (a block narrower than 256 columns spans
// several rows per pass). Each thread adds its rows in order; the row phases
// of a column are then added in phase order through shared memory and the
// CTA writes one partial per column to the workspace [P][C].
// Phase 2 (colsum_final_kernel): eight lanes per column add partials
// g, g + 8, ... in order, the eight sums are combined in lane order through
// shuffles, and lane 0 writes (or adds into) db.
// The row split depends on N only, so results are bit-identical run to run
// and across GPUs; nothing uses floating-point atomics.
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kColThreads = 256;
constexpr int kColUnroll = 8;

__global__ void __launch_bounds__(kColThreads) colsum_partial_kernel(const float* __restrict__ dy,
                                                                    long long N, int C, int P,
                                                                    float* __restrict__ part) {
  __shared__ float red[kColThreads];
  const int t = threadIdx.x, p = blockIdx.x;
  const long long r0 = N * p / P, r1 = N * (p + 1) / P;
  for (int c0 = 0; c0 < C; c0 += kColThreads) {
    const int cb = min(kColThreads, C - c0);
    const int ry = t / cb, RY = kColThreads / cb;
    const int c = c0 + t - ry * cb;
    float acc = 0.f;
    if (ry < RY) {
      const float* src = dy + (r0 + ry) * static_cast<long long>(C) + c;
      const long long step = static_cast<long long>(RY) * C;
      long long r = r0 + ry;
      // kColUnroll loads in flight, added in row order
      for (; r + static_cast<long long>(kColUnroll - 1) * RY < r1; r += static_cast<long long>(kColUnroll) * RY) {
        float v[kColUnroll];
#pragma unroll
        for (int u = 0; u < kColUnroll; ++u) v[u] = __ldcs(src + u * step);
#pragma unroll
        for (int u = 0; u < kColUnroll; ++u) acc += v[u];
        src += kColUnroll * step;
      }
      for (; r < r1; r += RY) {
        acc += __ldcs(src);
        src += step;
      }
    }
    red[t] = acc;
    __syncthreads();
    if (t < cb) {
      float s = red[t];
      for (int k = 1; k < RY; ++k) s += red[k * cb + t];
      part[static_cast<long long>(p) * C + c0 + t] = s;
    }
    __syncthreads();
  }
}

constexpr int kFinThreads = 256;  // 32 columns per CTA, eight lanes each

__global__ void __launch_bounds__(kFinThreads) colsum_final_kernel(const float* __restrict__ part,
                                                                  int P, int C, float* db,
                                                                  int accumulate) {
  const int lane = threadIdx.x & 31, g = lane & 7;
  const int c = blockIdx.x * (kFinThreads / 8) + (threadIdx.x >> 3);
  float s = 0.f;
  if (c < C) {
    // partials g, g + 8, ... (at most 19 of them: P <= 152), all requested
    // before the first add
    float v[(kMaxSlots + 7) / 8];
#pragma unroll
    for (int i = 0; i < (kMaxSlots + 7) / 8; ++i) {
      const int p = g + 8 * i;
      v[i] = p < P ? part[static_cast<long long>(p) * C + c] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < (kMaxSlots + 7) / 8; ++i) s += v[i];
  }
  float r = s;
#pragma unroll
  for (int k = 1; k < 8; ++k) r += __shfl_sync(0xffffffffu, s, (lane & ~7) + k);
  if (g == 0 && c < C) db[c] = accumulate ? db[c] + r : r;
}

}  // namespace

int colsum_partials(long long N) {
  // about 64 rows per CTA, at most one CTA per SM
  const long long p = (N + 63) / 64;
  return static_cast<int>(p < 1 ? 1 : (p > kMaxSlots ? kMaxSlots : p));
}

cudaError_t launch_colsum(const float* dy, long long N, int C, float* db, int accumulate,
                          float* part, cudaStream_t stream, int* n_launches) {
  const int P = colsum_partials(N);
  colsum_partial_kernel<<<P, kColThreads, 0, stream>>>(dy, N, C, P, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int per_cta = kFinThreads / 8;
  colsum_final_kernel<<<(C + per_cta - 1) / per_cta, kFinThreads, 0, stream>>>(part, P, C, db,
                                                                             accumulate);
  *n_launches = 2;
  return cudaGetLastError();
}

}  // namespace m2scan
