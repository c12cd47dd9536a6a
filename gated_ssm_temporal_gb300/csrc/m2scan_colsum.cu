// Bias gradient of a fully connected layer: db[c] (+)= sum over rows r of
// dy[r, c] for a row-major [N, C] fp32 matrix ("Phase 3 Kernel Optimization
// Implementation Plan", Task 2: the two-phase reduction over the batch, block
// partials then a second pass over the partials in a fixed order).
//
// Phase 1 (colsum_partial_kernel): CTA p owns rows [p*N/P, (p+1)*N/P) and
// walks the columns in blocks of up to 256 lanes (a lane is a float4 of
// columns when C % 4 == 0, else one column). For a block of Cb lanes thread
// t takes lane t % Cb and row phase t / Cb, so a warp always reads 32
// consecutive lanes of the matrix (a block narrower than 256 lanes spans
// several rows per pass). Each thread requests 16 of its rows at a time and
// adds them in row order; the row phases of a lane are then combined by a
// fixed pairwise tree in shared memory and the CTA writes one partial per
// column to the workspace [P][C].
// Phase 2 (colsum_final_kernel): eight lanes per column add partials
// g, g + 8, ... in order, the eight sums are combined in lane order through
// shuffles, and lane 0 writes (or adds into) db. It is launched as a
// programmatic dependent of phase 1, so its CTAs are resident before phase 1
// ends and only wait for the partials.
// The row split depends on N only, so results are bit-identical run to run
// and across GPUs; nothing uses floating-point atomics.
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kColThreads = 256;
constexpr int kColBatch = 16;  // rows requested at once per thread

__device__ __forceinline__ void add_to(float& a, float b) { a += b; }
__device__ __forceinline__ void add_to(float4& a, float4 b) {
  a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
}
template <typename V> __device__ __forceinline__ V zero_of();
template <> __device__ __forceinline__ float zero_of<float>() { return 0.f; }
template <> __device__ __forceinline__ float4 zero_of<float4>() { return make_float4(0.f, 0.f, 0.f, 0.f); }

// V = float4: C % 4 == 0 and lanes are column quads; V = float: one column per lane.
template <typename V>
__global__ void __launch_bounds__(kColThreads) colsum_partial_kernel(const float* __restrict__ dy,
                                                                    long long N, int C, int P,
                                                                    float* __restrict__ part) {
  // the final sum may be scheduled now; it waits for this grid's partials
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ V red[kColThreads];
  constexpr int kW = sizeof(V) / sizeof(float);
  const int t = threadIdx.x, p = blockIdx.x;
  const long long r0 = N * p / P, r1 = N * (p + 1) / P;
  const int L = C / kW;  // lanes per row
  const V* rows = reinterpret_cast<const V*>(dy);
  for (int l0 = 0; l0 < L; l0 += kColThreads) {
    const int cb = min(kColThreads, L - l0);
    const int ry = t / cb, RY = kColThreads / cb;
    const int l = l0 + t - ry * cb;
    V acc = zero_of<V>();
    if (ry < RY) {
      for (long long r = r0 + ry; r < r1; r += static_cast<long long>(kColBatch) * RY) {
        V v[kColBatch];
#pragma unroll
        for (int u = 0; u < kColBatch; ++u) {
          const long long rr = r + static_cast<long long>(u) * RY;
          v[u] = rr < r1 ? __ldcs(rows + rr * L + l) : zero_of<V>();
        }
        // rows in order; a missing row adds an exact zero
#pragma unroll
        for (int u = 0; u < kColBatch; ++u) add_to(acc, v[u]);
      }
    }
    red[t] = acc;
    __syncthreads();
    // row phases 0 .. RY-1 of each lane: fixed pairwise tree, phase k + h into k
    for (int R = RY; R > 1;) {
      const int h = (R + 1) >> 1;
      if (ry < R - h) add_to(red[t], red[t + h * cb]);
      R = h;
      __syncthreads();
    }
    if (t < cb) {
      const V s = red[t];
      float* dst = part + static_cast<long long>(p) * C + static_cast<long long>(l0 + t) * kW;
      if constexpr (kW == 4) {
        *reinterpret_cast<float4*>(dst) = s;
      } else {
        *dst = s;
      }
    }
    __syncthreads();
  }
}

constexpr int kFinThreads = 256;  // 32 columns per CTA, eight lanes each

__global__ void __launch_bounds__(kFinThreads) colsum_final_kernel(const float* __restrict__ part,
                                                                  int P, int C, float* db,
                                                                  int accumulate) {
  // the partials are written by the preceding kernel in the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
  // about 16 rows per CTA, at most one CTA per SM
  const long long p = (N + 15) / 16;
  return static_cast<int>(p < 1 ? 1 : (p > kMaxSlots ? kMaxSlots : p));
}

cudaError_t launch_colsum(const float* dy, long long N, int C, float* db, int accumulate,
                          float* part, cudaStream_t stream, int* n_launches) {
  const int P = colsum_partials(N);
  if (C % 4 == 0)
    colsum_partial_kernel<float4><<<P, kColThreads, 0, stream>>>(dy, N, C, P, part);
  else
    colsum_partial_kernel<float><<<P, kColThreads, 0, stream>>>(dy, N, C, P, part);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int per_cta = kFinThreads / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((C + per_cta - 1) / per_cta));
  cfg.blockDim = dim3(kFinThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, colsum_final_kernel, static_cast<const float*>(part), P, C, db,
                         accumulate);
  *n_launches = 2;
  return e;
}

}  // namespace m2scan
