// Wide-state kernels of the gated temporal scan layer (D = 64, SH2 % 128 == 0,
// K <= 128) on the FP32 FMA pipe.
//
// With D = 64 the projection weights [W_A|W_B] are 2·SH2·D floats (256 KB at
// SH2 = 512), too large to stay in shared memory, so every product is a
// tiled matrix product: a 128 x 128 output block per CTA, 8 x 8 outputs per
// thread, the reduction dimension streamed through shared memory in chunks
// of 32 (both operands staged, the next chunk prefetched into registers
// while the current one is multiplied).
//
//   wide_fwd_kernel   per 128-row tile (S = 128 / K samples, S <= 16):
//                     A|B = h_history . [W_A|W_B], C = h_s2 . W_C, the scan
//                     x_t = sigmoid(A_t) x_{t-1} + B_t, ctx = C x_{K-1} and
//                     h_enriched = h_s2 + tw ctx . W_O.
//   wide_bwd_kernel   per tile: the same projections and d_ctx = tw dY . W_O^T,
//                     the replay and reverse scan (dB_t = dx, dA_t = dx x_{t-1}
//                     sigmoid'(A_t), dx <- dx sigmoid(A_t)), d_h_s2 = dY +
//                     dC . W_C^T, d_h_history = dA|dB . [W_A|W_B]^T; dA|dB and
//                     [dC | ctx] go to the workspace.
//   wide_dw_kernel    the weight gradients as products over the batch:
//                     dW_A|dW_B = h^T . dA|dB over all rows, dW_C = h_s2^T . dC
//                     and dW_O = tw ctx^T . dY over all samples. CTA (job, p)
//                     sums the samples of range p into slot p; the slot
//                     reduction then adds the slots in a fixed order, so dW is
//                     bit-identical run to run.
#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kWT = 256;       // threads per CTA
constexpr int kWD = 64;        // state size D
constexpr int kWN = 128;       // output block columns (A|B = 2D)
constexpr int kWM = 128;       // output block rows
constexpr int kWKc = 32;       // reduction chunk
constexpr int kLd = 132;       // leading dimension (floats) of staged chunks and blocks
constexpr int kWSmax = 16;     // samples per tile, at most
constexpr int kWRanges = 38;   // sample ranges (weight-gradient slots) of the dW products

struct WideArgs {
  const float* h_history;
  const float* h_s2;
  const float* g;  // d_h_enriched (backward)
  const float* W_A;
  const float* W_B;
  const float* W_C;
  const float* W_O;
  float* out0;  // forward: h_enriched; backward: d_h_history
  float* out1;  // backward: d_h_s2
  float* dab;   // backward: dA|dB [B*K][128]
  float* cc;    // backward: [dC | ctx] [B][128]
  float* slots; // backward: weight-gradient slots [P][4][SH2*D]
  const float* gate_scale;  // one float multiplying every gate, or null (1)
  long long B;
  int K;
  int SH2;
  int S_max;
  int P;  // dW ranges
  float tw;
};

// Thread (ty, tx) of the 16 x 16 grid owns rows blk_row(ty, i) = 4 ty + i and 64 + 4 ty + i
// (i < 4) and columns 4 tx + j and 64 + 4 tx + j of a 128 x 128 block.
__device__ __forceinline__ int blk_row(int ty, int i) { return i < 4 ? 4 * ty + i : 60 + 4 * ty + i; }

// acc += At^T . Bs over one chunk: At[k][m] (k < 32, m < 128), Bs[k][n].
__device__ __forceinline__ void chunk_mma(const float* At, const float* Bs, int ty, int tx,
                                          float (&acc)[8][8]) {
#pragma unroll 8
  for (int k = 0; k < kWKc; ++k) {
    const float4 a0 = lds4(At + k * kLd + 4 * ty), a1 = lds4(At + k * kLd + 64 + 4 * ty);
    const float4 b0 = lds4(Bs + k * kLd + 4 * tx), b1 = lds4(Bs + k * kLd + 64 + 4 * tx);
    const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
}

__device__ __forceinline__ void zero_acc(float (&acc)[8][8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
}

__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// Shared memory of the per-tile kernels (floats). The partial sums of C and
// d_ctx are read before the backward writes dA|dB, so they share its buffer.
struct TileSmem {
  float* At;    // [32][kLd] A chunk, transposed
  float* Bs;    // [32][kLd] B chunk
  float* AB;    // [128][kLd] A|B of the tile's rows
  float* DABt;  // [128][kLd] dA|dB transposed (backward)
  float* SvT;   // [32][kWSmax] h_s2 chunk, transposed
  float* GvT;   // [32][kWSmax] dY chunk, transposed (backward)
  float* WCc;   // [32][64] W_C chunk
  float* WOt;   // [32][64] W_O^T chunk (backward)
  float* C;     // [kWSmax][64]
  float* Dctx;  // [kWSmax][64]
  float* CtxT;  // [64][kWSmax] ctx (forward) or dC (backward), transposed
  float* red;   // [4][kWSmax][64] partial sums of C over the k quarters
  float* red2;  // [4][kWSmax][64] partial sums of d_ctx (backward)
};

__device__ __forceinline__ TileSmem carve(float* s, bool bwd) {
  TileSmem m;
  m.At = s;    s += kWKc * kLd;
  m.Bs = s;    s += kWKc * kLd;
  m.AB = s;    s += kWM * kLd;
  m.SvT = s;   s += kWKc * kWSmax;
  m.GvT = s;   s += kWKc * kWSmax;
  m.WCc = s;   s += kWKc * kWD;
  m.WOt = s;   s += kWKc * kWD;
  m.C = s;     s += kWSmax * kWD;
  m.Dctx = s;  s += kWSmax * kWD;
  m.CtxT = s;  s += kWD * kWSmax;
  if (bwd) {
    m.DABt = s;
    m.red = s;
    m.red2 = s + 4 * kWSmax * kWD;
  } else {
    m.DABt = nullptr;
    m.red = s;
    m.red2 = nullptr;
  }
  return m;
}

size_t tile_smem_floats(bool bwd) {
  const size_t fixed = 2 * kWKc * kLd + kWM * kLd + 2 * kWKc * kWSmax + 2 * kWKc * kWD +
                       2 * kWSmax * kWD + kWD * kWSmax;
  return fixed + (bwd ? kWN * kLd : 4 * kWSmax * kWD);
}

// Projections of one tile: acc = h rows [row0, row0 + R_t) . [W_A|W_B] (rows
// past R_t are zero), red[kq] = partial C (and d_ctx) over the k quarter kq.
template <bool BWD>
__device__ void tile_projections(const WideArgs& a, const TileSmem& m, long long b0, int S_t,
                                 float (&acc)[8][8]) {
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int SH2 = a.SH2, K = a.K, R_t = S_t * K;
  const long long row0 = b0 * K;
  const int nq = SH2 / kWKc;
  // C / d_ctx: thread = (k quarter kq, sample quad sq, state quad dq)
  const int kq = tid >> 6, sq = (tid >> 4) & 3, dq = tid & 15;
  float cacc[4][4], gacc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) cacc[i][j] = gacc[i][j] = 0.f;
  zero_acc(acc);
  float4 ra[4], rb[4], rs, rg, rc[2], ro[2];
  auto load = [&](int q) {
    const int k0 = q * kWKc;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = tid + kWT * u;
      const int r = f & 127, c4 = f >> 7;
      ra[u] = r < R_t ? ldg4(a.h_history + (row0 + r) * SH2 + k0 + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      const int k = f >> 5, b4 = f & 31;
      rb[u] = ldg4((b4 < 16 ? a.W_A : a.W_B) + static_cast<size_t>(k0 + k) * kWD + 4 * (b4 & 15));
    }
    {
      const int s = tid >> 3, c4 = tid & 7;  // tid < 128: sample s < 16
      const bool ok = tid < kWSmax * 8 && s < S_t;
      rs = ok ? ldg4(a.h_s2 + (b0 + s) * SH2 + k0 + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (BWD) rg = ok ? ldg4(a.g + (b0 + s) * SH2 + k0 + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int f = tid + kWT * u;  // 512 float4 of [32][64]
      rc[u] = ldg4(a.W_C + static_cast<size_t>(k0 + (f >> 4)) * kWD + 4 * (f & 15));
      if (BWD) ro[u] = ldg4(a.W_O + static_cast<size_t>(f >> 3) * SH2 + k0 + 4 * (f & 7));  // W_O[d][k0 + k]
    }
  };
  auto store = [&]() {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = tid + kWT * u;
      const int r = f & 127, c4 = f >> 7;
      m.At[(4 * c4 + 0) * kLd + r] = ra[u].x;
      m.At[(4 * c4 + 1) * kLd + r] = ra[u].y;
      m.At[(4 * c4 + 2) * kLd + r] = ra[u].z;
      m.At[(4 * c4 + 3) * kLd + r] = ra[u].w;
      sts4(m.Bs + (f >> 5) * kLd + 4 * (f & 31), rb[u]);
    }
    if (tid < kWSmax * 8) {
      const int s = tid >> 3, c4 = tid & 7;
      m.SvT[(4 * c4 + 0) * kWSmax + s] = rs.x;
      m.SvT[(4 * c4 + 1) * kWSmax + s] = rs.y;
      m.SvT[(4 * c4 + 2) * kWSmax + s] = rs.z;
      m.SvT[(4 * c4 + 3) * kWSmax + s] = rs.w;
      if (BWD) {
        m.GvT[(4 * c4 + 0) * kWSmax + s] = rg.x;
        m.GvT[(4 * c4 + 1) * kWSmax + s] = rg.y;
        m.GvT[(4 * c4 + 2) * kWSmax + s] = rg.z;
        m.GvT[(4 * c4 + 3) * kWSmax + s] = rg.w;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int f = tid + kWT * u;
      sts4(m.WCc + (f >> 4) * kWD + 4 * (f & 15), rc[u]);
      if (BWD) {
        const int d = f >> 3, c4 = f & 7;
        m.WOt[(4 * c4 + 0) * kWD + d] = ro[u].x;
        m.WOt[(4 * c4 + 1) * kWD + d] = ro[u].y;
        m.WOt[(4 * c4 + 2) * kWD + d] = ro[u].z;
        m.WOt[(4 * c4 + 3) * kWD + d] = ro[u].w;
      }
    }
  };
  load(0);
  __syncthreads();  // the previous tile's readers of the staging buffers are done
  store();
  __syncthreads();
  for (int q = 0; q < nq; ++q) {
    if (q + 1 < nq) load(q + 1);
    chunk_mma(m.At, m.Bs, ty, tx, acc);
#pragma unroll
    for (int k = 8 * kq; k < 8 * kq + 8; ++k) {
      const float4 sv = lds4(m.SvT + k * kWSmax + 4 * sq), wc = lds4(m.WCc + k * kWD + 4 * dq);
      const float s4[4] = {sv.x, sv.y, sv.z, sv.w}, w4[4] = {wc.x, wc.y, wc.z, wc.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) cacc[i][j] = fmaf(s4[i], w4[j], cacc[i][j]);
      if (BWD) {
        const float4 gv = lds4(m.GvT + k * kWSmax + 4 * sq), wo = lds4(m.WOt + k * kWD + 4 * dq);
        const float g4[4] = {gv.x, gv.y, gv.z, gv.w}, o4[4] = {wo.x, wo.y, wo.z, wo.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) gacc[i][j] = fmaf(g4[i], o4[j], gacc[i][j]);
      }
    }
    __syncthreads();
    if (q + 1 < nq) store();
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    sts4(m.red + (kq * kWSmax + 4 * sq + i) * kWD + 4 * dq,
         make_float4(cacc[i][0], cacc[i][1], cacc[i][2], cacc[i][3]));
    if (BWD)
      sts4(m.red2 + (kq * kWSmax + 4 * sq + i) * kWD + 4 * dq,
           make_float4(gacc[i][0], gacc[i][1], gacc[i][2], gacc[i][3]));
  }
}

// A|B block (registers) into AB, C (and d_ctx) summed over the four k
// quarters in order.
template <bool BWD>
__device__ void tile_readout(const WideArgs& a, const TileSmem& m, const float (&acc)[8][8]) {
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = blk_row(ty, i);
    sts4(m.AB + r * kLd + 4 * tx, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
    sts4(m.AB + r * kLd + 64 + 4 * tx, make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]));
  }
  __syncthreads();  // red complete
  for (int e = tid; e < kWSmax * kWD; e += kWT) {
    float c = m.red[e];
    for (int q = 1; q < 4; ++q) c += m.red[q * kWSmax * kWD + e];
    m.C[e] = c;
    if (BWD) {
      float o = m.red2[e];
      for (int q = 1; q < 4; ++q) o += m.red2[q * kWSmax * kWD + e];
      m.Dctx[e] = a.tw * o;
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kWT, 1) wide_fwd_kernel(const WideArgs a) {
  extern __shared__ float4 smem_w4[];
  const TileSmem m = carve(reinterpret_cast<float*>(smem_w4), false);
  const int tid = threadIdx.x;
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max;
  const long long n_tiles = (a.B + S_max - 1) / S_max;
  for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const long long b0 = t * S_max;
    const int S_t = static_cast<int>(min(static_cast<long long>(S_max), a.B - b0));
    float acc[8][8];
    tile_projections<false>(a, m, b0, S_t, acc);
    tile_readout<false>(a, m, acc);
    // scan: one (sample, state) pair per thread and step
    const float gsc = load_gate_scale(a.gate_scale);
    for (int p = tid; p < S_t * kWD; p += kWT) {
      const int s = p >> 6, d = p & 63;
      float x = 0.f;
      for (int u = 0; u < K; ++u) {
        const float* pr = m.AB + (s * K + u) * kLd;
        x = fmaf(gsc * sigmoid_fast(pr[d]), x, pr[kWD + d]);
      }
      m.CtxT[d * kWSmax + s] = m.C[s * kWD + d] * x;
    }
    __syncthreads();
    // output: thread = 4 samples x 4 columns per column quad; each W_O
    // element serves the 4 samples
    {
      const int sq = tid >> 6, jq = tid & 63;
      if (4 * sq < S_t) {
        for (int j4 = jq; 4 * j4 < SH2; j4 += 64) {
          float o[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[i][j] = 0.f;
#pragma unroll 4
          for (int d = 0; d < kWD; ++d) {
            const float4 cv = lds4(m.CtxT + d * kWSmax + 4 * sq);
            const float4 wv = ldg4(a.W_O + static_cast<size_t>(d) * SH2 + 4 * j4);
            const float c4[4] = {cv.x, cv.y, cv.z, cv.w}, w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int j = 0; j < 4; ++j) o[i][j] = fmaf(c4[i], w4[j], o[i][j]);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int s = 4 * sq + i;
            if (s < S_t) {
              const float4 hv = ldg4(a.h_s2 + (b0 + s) * SH2 + 4 * j4);
              *reinterpret_cast<float4*>(a.out0 + (b0 + s) * SH2 + 4 * j4) =
                  make_float4(fmaf(a.tw, o[i][0], hv.x), fmaf(a.tw, o[i][1], hv.y),
                              fmaf(a.tw, o[i][2], hv.z), fmaf(a.tw, o[i][3], hv.w));
            }
          }
        }
      }
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kWT, 1) wide_bwd_kernel(const WideArgs a) {
  extern __shared__ float4 smem_w4[];
  const TileSmem m = carve(reinterpret_cast<float*>(smem_w4), true);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max;
  const long long n_tiles = (a.B + S_max - 1) / S_max;
  for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const long long b0 = t * S_max;
    const int S_t = static_cast<int>(min(static_cast<long long>(S_max), a.B - b0));
    const int R_t = S_t * K;
    const long long row0 = b0 * K;
    float acc[8][8];
    tile_projections<true>(a, m, b0, S_t, acc);
    tile_readout<true>(a, m, acc);
    // replay and reverse scan per (sample, state); dA|dB transposed into DABt
    // (zero past the tile) and to the workspace, [dC | ctx] to the workspace
    for (int e = tid; e < kWN * kWM; e += kWT) {
      const int c = e >> 7, r = e & 127;
      if (r >= R_t) m.DABt[c * kLd + r] = 0.f;
    }
    const float gsc = load_gate_scale(a.gate_scale);
    for (int p = tid; p < S_t * kWD; p += kWT) {
      const int s = p >> 6, d = p & 63;
      float x = 0.f;
      for (int u = 0; u < K; ++u) {  // B_t is replaced by x_t
        float* pr = m.AB + (s * K + u) * kLd;
        x = fmaf(gsc * sigmoid_fast(pr[d]), x, pr[kWD + d]);
        pr[kWD + d] = x;
      }
      const float Cv = m.C[s * kWD + d], dctx = m.Dctx[s * kWD + d];
      const float dC = dctx * x;
      m.CtxT[d * kWSmax + s] = dC;
      a.cc[(b0 + s) * kWN + d] = dC;
      a.cc[(b0 + s) * kWN + kWD + d] = Cv * x;
      float dx = dctx * Cv;
      for (int u = K - 1; u >= 0; --u) {
        const int r = s * K + u;
        const float* pr = m.AB + r * kLd;
        float sg, dsg;
        sigmoid_and_slope(pr[d], sg, dsg);
        sg *= gsc;
        dsg *= gsc;
        const float xprev = u > 0 ? pr[kWD + d - kLd] : 0.f;
        const float dA = dx * xprev * dsg, dB = dx;
        dx *= sg;
        m.DABt[d * kLd + r] = dA;
        m.DABt[(kWD + d) * kLd + r] = dB;
        a.dab[(row0 + r) * kWN + d] = dA;
        a.dab[(row0 + r) * kWN + kWD + d] = dB;
      }
    }
    __syncthreads();
    // d_h_s2 = dY + dC . W_C^T: thread = column j (its W_C row in
    // registers) x every sample of the tile
    for (int j = tid; j < SH2; j += kWT) {
      float4 w[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) w[q] = ldg4(a.W_C + static_cast<size_t>(j) * kWD + 4 * q);
      for (int s = 0; s < S_t; ++s) {
        float o = __ldg(a.g + (b0 + s) * SH2 + j);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          o = fmaf(m.CtxT[(4 * q + 0) * kWSmax + s], w[q].x, o);
          o = fmaf(m.CtxT[(4 * q + 1) * kWSmax + s], w[q].y, o);
          o = fmaf(m.CtxT[(4 * q + 2) * kWSmax + s], w[q].z, o);
          o = fmaf(m.CtxT[(4 * q + 3) * kWSmax + s], w[q].w, o);
        }
        a.out1[(b0 + s) * SH2 + j] = o;
      }
    }
    // d_h_history = dA|dB . [W_A|W_B]^T, per 128-column block of SH2
    for (int jb = 0; jb < SH2 / kWN; ++jb) {
      zero_acc(acc);
      float4 rb[4];
      auto loadB = [&](int kc) {  // B[c][n] = W_x[128 jb + n][c], c in [32 kc, 32 kc + 32)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int f = tid + kWT * u;
          const int n = f & 127, c4 = f >> 7;
          const int c = kWKc * kc + 4 * c4;
          rb[u] = ldg4((c < kWD ? a.W_A : a.W_B) + static_cast<size_t>(kWN * jb + n) * kWD + (c & 63));
        }
      };
      auto storeB = [&]() {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int f = tid + kWT * u;
          const int n = f & 127, c4 = f >> 7;
          m.Bs[(4 * c4 + 0) * kLd + n] = rb[u].x;
          m.Bs[(4 * c4 + 1) * kLd + n] = rb[u].y;
          m.Bs[(4 * c4 + 2) * kLd + n] = rb[u].z;
          m.Bs[(4 * c4 + 3) * kLd + n] = rb[u].w;
        }
      };
      loadB(0);
      __syncthreads();
      storeB();
      __syncthreads();
      for (int kc = 0; kc < kWN / kWKc; ++kc) {
        if (kc + 1 < kWN / kWKc) loadB(kc + 1);
        chunk_mma(m.DABt + kWKc * kc * kLd, m.Bs, ty, tx, acc);
        __syncthreads();
        if (kc + 1 < kWN / kWKc) storeB();
        __syncthreads();
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = blk_row(ty, i);
        if (r < R_t) {
          float* dst = a.out0 + (row0 + r) * SH2 + kWN * jb;
          *reinterpret_cast<float4*>(dst + 4 * tx) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
          *reinterpret_cast<float4*>(dst + 64 + 4 * tx) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        }
      }
    }
    __syncthreads();
  }
}

// Weight gradients. CTA = (job, range p): jobs [0, nb) are dW_A|dW_B blocks
// (128 rows j of SH2 x 128 columns of dA|dB, reduced over the rows of the
// range), [nb, 2 nb) dW_C blocks (h_s2^T . [dC | ctx], the dC half kept) and
// [2 nb, 3 nb) dW_O blocks (dY^T . [dC | ctx], the ctx half kept, times tw),
// reduced over the samples of the range; nb = SH2 / 128.
__global__ void __launch_bounds__(kWT, 1) wide_dw_kernel(const WideArgs a) {
  extern __shared__ float4 smem_w4[];
  float* At = reinterpret_cast<float*>(smem_w4);
  float* Bs = At + kWKc * kLd;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int SH2 = a.SH2, K = a.K, P = a.P, nb = SH2 / kWN;
  const int job = blockIdx.x / P, p = blockIdx.x - (blockIdx.x / P) * P;
  const int kind = job / nb, jb = job - kind * nb;
  const long long s_lo = a.B * p / P, s_hi = a.B * (p + 1) / P;
  const long long k_lo = kind == 0 ? s_lo * K : s_lo, k_hi = kind == 0 ? s_hi * K : s_hi;
  const float* Asrc = kind == 0 ? a.h_history : (kind == 1 ? a.h_s2 : a.g);
  const float* Bsrc = kind == 0 ? a.dab : a.cc;
  float acc[8][8];
  zero_acc(acc);
  float4 ra[4], rb[4];
  auto load = [&](long long k0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = tid + kWT * u;
      const int k = f >> 5, c4 = f & 31;
      const bool ok = k0 + k < k_hi;
      ra[u] = ok ? ldg4(Asrc + (k0 + k) * SH2 + kWN * jb + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
      rb[u] = ok ? ldg4(Bsrc + (k0 + k) * kWN + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto store = [&]() {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int f = tid + kWT * u;
      const int k = f >> 5, c4 = f & 31;
      sts4(At + k * kLd + 4 * c4, ra[u]);
      sts4(Bs + k * kLd + 4 * c4, rb[u]);
    }
  };
  if (k_lo < k_hi) {
    load(k_lo);
    store();
    __syncthreads();
    for (long long k0 = k_lo; k0 < k_hi; k0 += kWKc) {
      if (k0 + kWKc < k_hi) load(k0 + kWKc);
      chunk_mma(At, Bs, ty, tx, acc);
      __syncthreads();
      if (k0 + kWKc < k_hi) store();
      __syncthreads();
    }
  }
  const int n = SH2 * kWD;
  float* slot = a.slots + static_cast<size_t>(p) * 4 * n;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int j = kWN * jb + blk_row(ty, i);
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // columns 4 tx + 64 h .. + 3
      const float4 v = make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
      const int c = 64 * h + 4 * tx;
      if (kind == 0) {
        *reinterpret_cast<float4*>(slot + h * n + static_cast<size_t>(j) * kWD + 4 * tx) = v;
      } else if (kind == 1 && h == 0) {
        *reinterpret_cast<float4*>(slot + 2 * n + static_cast<size_t>(j) * kWD + c) = v;
      } else if (kind == 2 && h == 1) {
        const int d = c - kWD;
        slot[3 * n + static_cast<size_t>(d) * SH2 + j] = a.tw * v.x;
        slot[3 * n + static_cast<size_t>(d + 1) * SH2 + j] = a.tw * v.y;
        slot[3 * n + static_cast<size_t>(d + 2) * SH2 + j] = a.tw * v.z;
        slot[3 * n + static_cast<size_t>(d + 3) * SH2 + j] = a.tw * v.w;
      }
    }
  }
}

}  // namespace

bool wide_path_ok(int K, int SH2, int D) {
  return D == kWD && SH2 >= kWN && SH2 % kWN == 0 && K >= 1 && K <= kWM &&
         tile_smem_floats(true) * sizeof(float) <= 227 * 1024;
}

int wide_ranges(int64_t B) { return B < kWRanges ? static_cast<int>(B) : kWRanges; }

size_t wide_bwd_workspace_bytes(int64_t B, int32_t K, int32_t SH2) {
  const size_t slots = static_cast<size_t>(wide_ranges(B)) * 4 * static_cast<size_t>(SH2) * kWD;
  const size_t dab = static_cast<size_t>(B) * K * kWN;
  const size_t cc = static_cast<size_t>(B) * kWN;
  return (slots + dab + cc) * sizeof(float);
}

static WideArgs wide_args(const float* h_history, const float* h_s2, const float* g, const float* W_A,
                          const float* W_B, const float* W_C, const float* W_O, float tw, int64_t B,
                          int K, int SH2) {
  WideArgs w{};
  w.h_history = h_history; w.h_s2 = h_s2; w.g = g;
  w.W_A = W_A; w.W_B = W_B; w.W_C = W_C; w.W_O = W_O;
  w.B = B; w.K = K; w.SH2 = SH2; w.tw = tw;
  int S_max = kWM / K;
  w.S_max = S_max < kWSmax ? S_max : kWSmax;
  return w;
}

static int wide_grid(const WideArgs& w) {
  const long long n_tiles = (w.B + w.S_max - 1) / w.S_max;
  return static_cast<int>(n_tiles < kMaxSlots ? n_tiles : kMaxSlots);
}

cudaError_t launch_wide_fwd(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw, int64_t B,
                            int K, int SH2, float* h_enriched, const float* gate_scale,
                            cudaStream_t stream) {
  WideArgs w = wide_args(h_history, h_s2, nullptr, W_A, W_B, W_C, W_O, tw, B, K, SH2);
  w.out0 = h_enriched;
  w.gate_scale = gate_scale;
  wide_fwd_kernel<<<wide_grid(w), kWT, tile_smem_floats(false) * sizeof(float), stream>>>(w);
  return cudaGetLastError();
}

// Three launches and the slot reduction: returns the number of launches in *n.
cudaError_t launch_wide_bwd(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw,
                            const float* g, int64_t B, int K, int SH2, float* d_h_history,
                            float* d_h_s2, float* dW_A, float* dW_B, float* dW_C, float* dW_O,
                            void* workspace, const float* gate_scale, cudaStream_t stream, int* n) {
  WideArgs w = wide_args(h_history, h_s2, g, W_A, W_B, W_C, W_O, tw, B, K, SH2);
  w.gate_scale = gate_scale;
  w.out0 = d_h_history;
  w.out1 = d_h_s2;
  w.P = wide_ranges(B);
  float* ws = static_cast<float*>(workspace);
  w.slots = ws;
  w.dab = ws + static_cast<size_t>(w.P) * 4 * static_cast<size_t>(SH2) * kWD;
  w.cc = w.dab + static_cast<size_t>(B) * K * kWN;
  *n = 0;
  wide_bwd_kernel<<<wide_grid(w), kWT, tile_smem_floats(true) * sizeof(float), stream>>>(w);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*n;
  const int jobs = 3 * (SH2 / kWN);
  wide_dw_kernel<<<jobs * w.P, kWT, 2 * kWKc * kLd * sizeof(float), stream>>>(w);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n;
  e = launch_reduce(w.slots, w.P, SH2 * kWD, dW_A, dW_B, dW_C, dW_O, stream);
  if (e == cudaSuccess) ++*n;
  return e;
}

cudaError_t prepare_wide_kernels() {
  cudaError_t e = cudaFuncSetAttribute(wide_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(tile_smem_floats(false) * sizeof(float)));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wide_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tile_smem_floats(true) * sizeof(float)));
  return e;
}

}  // namespace m2scan
