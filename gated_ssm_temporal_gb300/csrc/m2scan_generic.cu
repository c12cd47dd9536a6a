// Generic kernels of the gated temporal scan layer, for shapes that neither
// the fused tensor-core kernels nor the wide-state kernels take (e.g. D = 24,
// or SH2 = 36), and the slot reduction that every backward family ends with.
//
// The generic kernels keep one sample at a time in shared memory: each CTA
// owns the samples [c*B/P, (c+1)*B/P) and the weight-gradient slot c. Every
// slot entry is owned by one fixed thread (entry e by thread e % 256), so the
// partial sums are formed in a fixed order without atomics.
//
// Staged form (GenericArgs::staged, chosen by the launcher when it fits the
// device's shared memory): the four weight matrices, the sample's h_history
// rows (as fp32) and the CTA's slot live in shared memory, and the slot is
// written to global memory once, after the last sample. Every sum is formed
// in the same order as in the unstaged form, so both give identical bits.
//
// T is the type of the activations (h_history, h_s2, dY in; the layer's
// output or the input gradients out): float, or bfloat16 for the pages'
// "bf16 inputs/outputs with fp32 accumulation" variant. Weights, weight
// gradients and every product and sum are fp32 either way; a bf16 output is
// the fp32 result rounded to nearest even.
#include <cuda_bf16.h>

#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void store_as(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_as(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <bool BWD, typename T>
__global__ void __launch_bounds__(kThreads) generic_kernel(const GenericArgs a) {
  const T* h_history = reinterpret_cast<const T*>(a.h_history);
  const T* h_s2 = reinterpret_cast<const T*>(a.h_s2);
  const T* g_in = reinterpret_cast<const T*>(a.g);
  T* out0 = reinterpret_cast<T*>(a.out0);
  T* out1 = reinterpret_cast<T*>(a.out1);
  extern __shared__ float4 smem_f4[];
  float* sm = reinterpret_cast<float*>(smem_f4);
  const int K = a.K, SH2 = a.SH2, D = a.D, TD = 2 * D;
  float* sAB = sm;            // [K][2D]: A|B, then A|x, then dA|dB
  float* sHs = sAB + K * TD;  // [SH2]
  float* sG = sHs + SH2;      // [SH2]
  float* sC = sG + SH2;       // [D]
  float* sCtx = sC + D;
  float* sDctx = sCtx + D;
  float* sDC = sDctx + D;
  const int tid = threadIdx.x;
  const int P = gridDim.x, cta = blockIdx.x;
  const long long b0 = a.B * cta / P, b1 = a.B * (cta + 1) / P;
  const int n = SH2 * D;
  const bool staged = a.staged != 0;
  // staged only: h rows [K][SH2]; W_A, W_B, W_C [SH2][D] in rows of ldw = D + 1
  // and W_O [D][SH2] in rows of ldo = SH2 + 1 (the padding keeps the loops
  // that walk j across a warp free of bank conflicts); slot [4][n]
  const int ldw = staged ? D + 1 : D, ldo = staged ? SH2 + 1 : SH2;
  float* sH = sDC + D;
  float* sWA = sH + static_cast<size_t>(K) * SH2;
  const size_t nw = static_cast<size_t>(SH2) * (D + 1);  // D * (SH2 + 1) is the same less SH2 - D
  float* sWB = sWA + nw;
  float* sWC = sWB + nw;
  float* sWO = sWC + nw;
  float* sSlot = sWO + static_cast<size_t>(D) * (SH2 + 1);
  const float* W_A = staged ? sWA : a.W_A;
  const float* W_B = staged ? sWB : a.W_B;
  const float* W_C = staged ? sWC : a.W_C;
  const float* W_O = staged ? sWO : a.W_O;
  float* gslot = BWD ? a.ws + static_cast<size_t>(cta) * 4 * n : nullptr;
  float* slot = (BWD && staged) ? sSlot : gslot;
  if (staged) {
    for (int e = tid; e < n; e += kThreads) {
      const int j = e / D, d = e - (e / D) * D;
      sWA[j * ldw + d] = a.W_A[e];
      sWB[j * ldw + d] = a.W_B[e];
      sWC[j * ldw + d] = a.W_C[e];
      const int dd = e / SH2, jj = e - (e / SH2) * SH2;
      sWO[dd * ldo + jj] = a.W_O[e];
    }
  }
  if (BWD)
    for (int e = tid; e < 4 * n; e += kThreads) slot[e] = 0.f;
  __syncthreads();

  for (long long b = b0; b < b1; ++b) {
    const T* h = h_history + b * K * SH2;
    for (int j = tid; j < SH2; j += kThreads) {
      sHs[j] = to_f32(h_s2[b * SH2 + j]);
      if (BWD) sG[j] = to_f32(g_in[b * SH2 + j]);
    }
    if (staged)
      for (int e = tid; e < K * SH2; e += kThreads) sH[e] = to_f32(h[e]);
    __syncthreads();
    // projections A|B (one output per thread and step), C and d_ctx
    for (int e = tid; e < K * TD; e += kThreads) {
      const int t = e / TD, k = e - (e / TD) * TD;
      const float* W = k < D ? W_A : W_B;
      const int col = k < D ? k : k - D;
      float s = 0.f;
      if (staged) {
        const float* hr = sH + static_cast<size_t>(t) * SH2;
        for (int j = 0; j < SH2; ++j) s = fmaf(hr[j], W[j * ldw + col], s);
      } else {
        const T* hr = h + static_cast<size_t>(t) * SH2;
        for (int j = 0; j < SH2; ++j) s = fmaf(to_f32(hr[j]), W[j * ldw + col], s);
      }
      sAB[e] = s;
    }
    for (int d = tid; d < D; d += kThreads) {
      float c = 0.f;
      for (int j = 0; j < SH2; ++j) c = fmaf(sHs[j], W_C[j * ldw + d], c);
      sC[d] = c;
      if (BWD) {
        float o = 0.f;
        for (int j = 0; j < SH2; ++j) o = fmaf(sG[j], W_O[static_cast<size_t>(d) * ldo + j], o);
        sDctx[d] = a.tw * o;
      }
    }
    __syncthreads();
    // scan (and reverse scan)
    const float gsc = load_gate_scale(a.gate_scale);
    for (int d = tid; d < D; d += kThreads) {
      float x = 0.f;
      for (int t = 0; t < K; ++t) {
        float* pr = sAB + t * TD;
        x = fmaf(gsc * sigmoidf_(pr[d]), x, pr[D + d]);
        if (BWD) pr[D + d] = x;  // A stays in place, B_t is replaced by x_t
      }
      sCtx[d] = sC[d] * x;
      if (BWD) {
        sDC[d] = sDctx[d] * x;
        float dx = sDctx[d] * sC[d];
        for (int t = K - 1; t >= 0; --t) {
          float* pr = sAB + t * TD;
          const float at = pr[d];
          const float sg0 = sigmoidf_(at);
          const float dsg = gsc * (sg0 * sigmoidf_(-at));  // sigmoid' without cancellation near 1
          const float sg = gsc * sg0;
          const float xprev = t > 0 ? pr[D + d - TD] : 0.f;
          pr[D + d] = dx;
          pr[d] = dx * xprev * dsg;
          dx *= sg;
        }
      }
    }
    __syncthreads();
    if (!BWD) {
      for (int j = tid; j < SH2; j += kThreads) {
        float o = 0.f;
        for (int d = 0; d < D; ++d) o = fmaf(sCtx[d], W_O[static_cast<size_t>(d) * ldo + j], o);
        store_as(out0 + b * SH2 + j, fmaf(a.tw, o, sHs[j]));
      }
    } else {
      for (int e = tid; e < K * SH2; e += kThreads) {
        const int t = e / SH2, j = e - (e / SH2) * SH2;
        const float* pr = sAB + t * TD;
        float s = 0.f;
        for (int d = 0; d < D; ++d) {
          s = fmaf(pr[d], W_A[j * ldw + d], s);
          s = fmaf(pr[D + d], W_B[j * ldw + d], s);
        }
        store_as(out0 + (b * K + t) * SH2 + j, s);
      }
      for (int j = tid; j < SH2; j += kThreads) {
        float s = sG[j];
        for (int d = 0; d < D; ++d) s = fmaf(sDC[d], W_C[j * ldw + d], s);
        store_as(out1 + b * SH2 + j, s);
      }
      for (int e = tid; e < n; e += kThreads) {
        const int j = e / D, d = e - (e / D) * D;
        float sa = 0.f, sb = 0.f;
        for (int t = 0; t < K; ++t) {
          const float hv = staged ? sH[static_cast<size_t>(t) * SH2 + j]
                                  : to_f32(h[static_cast<size_t>(t) * SH2 + j]);
          sa = fmaf(hv, sAB[t * TD + d], sa);
          sb = fmaf(hv, sAB[t * TD + D + d], sb);
        }
        slot[e] += sa;
        slot[n + e] += sb;
        slot[2 * n + e] += sHs[j] * sDC[d];
      }
      for (int e = tid; e < n; e += kThreads) {
        const int d = e / SH2, j = e - (e / SH2) * SH2;
        slot[3 * n + e] += a.tw * sCtx[d] * sG[j];
      }
    }
    __syncthreads();
  }
  if (BWD && staged)
    for (int e = tid; e < 4 * n; e += kThreads) gslot[e] = sSlot[e];
  if (BWD) {
    __syncthreads();
    if (tid == 0) signal_dependent_launch();
  }
}

// dW[e] = sum over slots p = 0..P-1 of ws[p][e], added in a fixed order:
// eight interleaved partial sums per element (slots g, g+8, ...), then the
// eight partials in order. Each CTA covers 128 consecutive elements.
__global__ void __launch_bounds__(kThreads) reduce_kernel(const float* __restrict__ ws, int P,
                                                          int n, float* dW_A, float* dW_B,
                                                          float* dW_C, float* dW_O) {
  __shared__ float4 red[8][32];
  // launched as a programmatic dependent of the kernel that wrote the slots:
  // nothing is read before that grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const long long total = 4ll * n;
  const long long e0 = static_cast<long long>(blockIdx.x) * 128 + 4 * lane;
  // all loads of a thread are issued before the first add (P <= 152 = 8 x 19)
  constexpr int kPerGroup = (kMaxSlots + 7) / 8;
  float4 v[kPerGroup];
#pragma unroll
  for (int i = 0; i < kPerGroup; ++i) {
    const int p = grp + 8 * i;
    v[i] = (p < P && e0 < total)
               ? *reinterpret_cast<const float4*>(ws + static_cast<size_t>(p) * total + e0)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float4 s = v[0];
#pragma unroll
  for (int i = 1; i < kPerGroup; ++i) {
    s.x += v[i].x; s.y += v[i].y; s.z += v[i].z; s.w += v[i].w;
  }
  red[grp][lane] = s;
  __syncthreads();
  if (grp == 0 && e0 < total) {
    float4 r = red[0][lane];
    for (int g = 1; g < 8; ++g) {
      const float4 v = red[g][lane];
      r.x += v.x; r.y += v.y; r.z += v.z; r.w += v.w;
    }
    const int which = static_cast<int>(e0 / n);
    const int i = static_cast<int>(e0 - static_cast<long long>(which) * n);
    float* out = which == 0 ? dW_A : (which == 1 ? dW_B : (which == 2 ? dW_C : dW_O));
    *reinterpret_cast<float4*>(out + i) = r;
  }
}

}  // namespace

size_t generic_smem_bytes(bool bwd, int K, int SH2, int D) {
  (void)bwd;
  return sizeof(float) * (static_cast<size_t>(K) * 2 * D + 2 * static_cast<size_t>(SH2) + 4 * D);
}

size_t generic_staged_smem_bytes(bool bwd, int K, int SH2, int D) {
  const size_t sh = static_cast<size_t>(SH2), d = static_cast<size_t>(D);
  return generic_smem_bytes(bwd, K, SH2, D) +
         sizeof(float) * (static_cast<size_t>(K) * sh + 3 * sh * (d + 1) + d * (sh + 1) +
                          (bwd ? 4 * sh * d : 0));
}

cudaError_t launch_generic(bool bwd, GenericArgs a, int grid, int max_smem, cudaStream_t stream,
                           bool bf16) {
  const size_t staged = generic_staged_smem_bytes(bwd, a.K, a.SH2, a.D);
  a.staged = staged <= static_cast<size_t>(max_smem) ? 1 : 0;
  const size_t smem = a.staged ? staged : generic_smem_bytes(bwd, a.K, a.SH2, a.D);
  if (bf16) {
    if (bwd)
      generic_kernel<true, __nv_bfloat16><<<grid, kThreads, smem, stream>>>(a);
    else
      generic_kernel<false, __nv_bfloat16><<<grid, kThreads, smem, stream>>>(a);
  } else {
    if (bwd)
      generic_kernel<true, float><<<grid, kThreads, smem, stream>>>(a);
    else
      generic_kernel<false, float><<<grid, kThreads, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce(const float* ws, int slots, int n, float* dW_A, float* dW_B,
                          float* dW_C, float* dW_O, cudaStream_t stream) {
  const long long total = 4ll * n;
  const int grid = static_cast<int>((total + 127) / 128);
  // A programmatic dependent of the slot-writing kernel: its launch is
  // prepared while that kernel's last CTAs finish (they signal after their
  // final barrier), and its griddepcontrol.wait keeps every read behind the
  // completion of that kernel. Backward call at B = 8192, K = 8, SH2 = 256:
  // 81.9 -> 77.8 us against a plain launch.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, reduce_kernel, ws, slots, n, dW_A, dW_B, dW_C, dW_O);
}

cudaError_t prepare_generic_kernels(int max_smem) {
  const void* kernels[] = {reinterpret_cast<const void*>(generic_kernel<false, float>),
                           reinterpret_cast<const void*>(generic_kernel<true, float>),
                           reinterpret_cast<const void*>(generic_kernel<false, __nv_bfloat16>),
                           reinterpret_cast<const void*>(generic_kernel<true, __nv_bfloat16>)};
  for (const void* k : kernels) {
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace m2scan
