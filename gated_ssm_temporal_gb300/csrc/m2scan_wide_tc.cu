// Wide-state kernels of the gated temporal scan layer (D = 64, SH2 % 128 == 0,
// K <= 128) with their large contractions on the tensor cores.
//
// With D = 64 the projection weights [W_A|W_B] are 2·SH2·D floats (256 KB at
// SH2 = 512), too large to keep in shared memory: every CTA streams them from
// L2 chunk by chunk next to the activations. Every product is 3 x TF32 on
// tcgen05 (x = hi + lo with hi = x rounded to tf32 and lo the exact fp32
// remainder; hi.hi + hi.lo + lo.hi into one fp32 TMEM accumulator,
// issued by one thread in a fixed order, so results do not depend on timing).
// The remainders are formed by the compute warps in shared memory at the
// position of the value they belong to, so no operand is ever transposed by a
// thread: the weights enter the projections as MN-major operands (128-byte
// swizzle with 32-byte atoms, as TMA lays them out) and the weight-gradient
// products read h_history, h_s2, dY, dA|dB and [dC | ctx] MN-major too.
//
//   wide_tc_kernel<false, KPP>  forward, per 128-row tile (S = 128 / K samples,
//       S <= 16): A|B = h_history . [W_A|W_B] on the tensor cores (32-column
//       chunks of SH2 through a ring of four stages); C = h_s2 . W_C on the FMA
//       pipe during the chunks; the scan x_t = sigmoid(A_t) x_{t-1} + B_t,
//       ctx = C x_{K-1} and h_enriched = h_s2 + tw ctx . W_O.
//   wide_tc_kernel<true, KPP>   backward, per tile: the same projections and
//       d_ctx = tw dY . W_O^T; replay and reverse scan (dB_t = dx, dA_t =
//       dx x_{t-1} sigmoid'(A_t), dx <- dx sigmoid(A_t)); dA|dB split into tf32
//       part and remainder in TMEM (A operand) for d_h_history =
//       dA|dB . [W_A|W_B]^T on the tensor cores (four 128-column blocks, two
//       accumulators in turn). dA|dB and [dC | ctx] go to the workspace.
//   wide_dhs2_kernel       d_h_s2 = dY + dC . W_C^T over the whole batch on
//       the FMA pipe, from the dC the tile kernel left in the workspace.
//   wide_tc_dw_kernel      the weight gradients as products over the batch:
//       dW_A|dW_B = h^T . dA|dB over all rows, dW_C = h_s2^T . dC and
//       dW_O^T = dY^T . ctx (times tw) over all samples. CTA (job, p) sums the
//       rows of sample range p into slot p; the slot reduction adds the slots
//       in a fixed order, so the weight gradients are bit-identical run to run.
//
// The steps are those of "Custom Kernel Optimization Implementation Plan",
// Tasks 1-2 (projections, scan, reverse scan, weight gradients), with the
// output step h_s2 + tw ctx . W_O of the layer.
#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kWD = 64;           // state size D
constexpr int kWN = 128;          // A|B columns (2D)
constexpr int kWRows = 128;       // rows per tile
constexpr int kWSmax = 16;        // samples per tile, at most
// Sample ranges (weight-gradient slots) of the dW products: as many as the
// other kernel families use, so that no tensor-core accumulation chain gets
// long (a range's rows / 16 steps per accumulator at most).
constexpr int kWRanges = kMaxSlots;
constexpr int kCW = 8;            // compute warps of the tile kernels
constexpr int kCT = kCW * 32;     // compute threads
constexpr int kTileThreads = kCT + 64;  // + producer warp + MMA warp
constexpr int kProdWarp = kCW, kMmaWarp = kCW + 1;
constexpr int kNst = 4;           // copy ring depth of the tile kernels
constexpr uint32_t kBox = 16384;  // a [128 x 128 B] operand box
constexpr uint32_t kStage = 2 * kBox + 4096;  // h and W (or two W boxes) + the h_s2 / dY boxes
constexpr uint32_t kABBytes = kWRows * kWN * 4;

// Tile kernels: shared memory (bytes from the 1024-aligned base). The two
// remainder buffers (h lo and W lo of one stage each, 32 KB) share the A|B
// buffer: they are only in use while chunks stream, A|B only after.
constexpr uint32_t kOffAB = kNst * kStage;         // A|B, then dA|dB: [128][128] floats, swizzled
constexpr uint32_t kOffC = kOffAB + kABBytes;      // C [16][64]
constexpr uint32_t kOffDctx = kOffC + 4096;        // d_ctx [16][64]
constexpr uint32_t kOffX = kOffDctx + 4096;        // ctx (forward) or dC (backward), [64][16]
constexpr uint32_t kOffBar = kOffX + 4096;
constexpr uint32_t kTileSmem = kOffBar + 256 + 1024;

// dW kernel: three stages of A, A lo, B, B lo.
constexpr int kDwNst = 3;
constexpr int kDwCW = 4;          // compute warps (remainders; read-back)
constexpr int kDwThreads = kDwCW * 32 + 64;
constexpr uint32_t kDwStage = 4 * kBox;
constexpr uint32_t kDwOffBar = kDwNst * kDwStage;
constexpr uint32_t kDwSmem = kDwOffBar + 128 + 1024;

// Arguments of the tile kernels. Tensor maps: tm_h = h_history as [B*K rows][SH2]
// (box 32 x 128 rows, 128-byte swizzle: the K-major A operand of the
// projections); tm_wa / tm_wb = W_A / W_B [SH2][64] (box 32 x 32, 128-byte
// swizzle with 32-byte atoms: MN-major B operand of the projections); tm_wak /
// tm_wbk = the same weights as K-major B operand of d_h_history (box 32
// columns x 128 rows, 128-byte swizzle); tm_hs / tm_g = h_s2 / d_h_enriched
// [B][SH2] (box 32 x S_max, 128-byte swizzle) for the C / d_ctx dots.
struct alignas(128) WideTcArgs {
  CUtensorMap tm_h, tm_wa, tm_wb, tm_wak, tm_wbk, tm_hs, tm_g;
  CUtensorMap tm_wal, tm_wbl;  // backward: remainders of the split weights
  const float* h_s2;
  const float* W_C;
  const float* W_O;
  float* out0;     // forward: h_enriched; backward: d_h_history
  float* dab;      // backward: dA|dB [B*K][128]
  float* cc;       // backward: [dC | ctx] [B][128]
  const float* gate_scale;
  unsigned* err;
  long long B;
  int K, SH2, S_max;
  float tw;
};

// Arguments of the weight-gradient products: tm_a = h_history [B*K][SH2],
// h_s2 [B][SH2], d_h_enriched [B][SH2]; tm_b = dA|dB [B*K][128], [dC | ctx]
// [B][128]; all box 32 x 32 rows, 128-byte swizzle with 32-byte atoms
// (MN-major operands).
struct alignas(128) WideDwArgs {
  CUtensorMap tm_a[3];
  CUtensorMap tm_b[2];
  float* slots;  // [P][4][SH2 * 64]
  unsigned* err;
  long long B;
  int K, SH2, P;
  float tw;
};

struct TileBars {
  uint64_t full[kNst];    // producer -> all: stage loaded
  uint64_t empty[kNst];   // MMA commit -> producer: stage consumed
  uint64_t split[kNst];   // compute (one arrival per warp) -> MMA: remainders written
  uint64_t acc_full;      // MMA -> compute: the tile's projections done
  uint64_t acc_free;      // compute -> MMA: projections read back (forward)
  uint64_t dab_ready;     // compute -> MMA: dA|dB in TMEM (backward)
  uint64_t dh_full[2];    // MMA -> compute: a d_h block done
  uint64_t dh_free[2];    // compute -> MMA: that block read back
  uint64_t wlo_full[2];   // W remainder loader -> MMA: a chunk's W_lo in remainder buffer p (backward)
  uint64_t tile_done;     // MMA -> W remainder loader: every product of a tile done (backward)
  uint32_t tslot;
};

struct DwBars {
  uint64_t full[kDwNst];
  uint64_t empty[kDwNst];
  uint64_t split[kDwNst];
  uint64_t done;
  uint32_t tslot;
};

// Element (r, c) of the [128][128] float A|B buffer: float4 slots XOR-ed with
// the row, so that a warp's 32 rows at one column and 32 columns of one row
// both spread over the banks.
__device__ __forceinline__ int ab_idx(int r, int c) {
  return r * kWN + ((((c >> 2) ^ (r & 31))) << 2) + (c & 3);
}

__device__ __forceinline__ float4 ldg4w(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// Remainders of `n4` float4 of a stage buffer, in place: with `round_hi`,
// hi[i] becomes tf32_rn(x) and lo[i] = x - tf32_rn(x), exact and at most half
// a tf32 ulp, so that hi.hi + hi.lo + lo.hi misses only lo.lo and the
// truncation of lo when the tensor core reads it (about 2^-21 of the product,
// four times less than with a truncated hi); else hi[i] keeps x (the tensor
// core reads its truncated tf32 part) and lo[i] = x - trunc_tf32(x).
__device__ __forceinline__ void split_buf(float* hi, float* lo, int n4, int t, int nt, bool round_hi) {
  for (int i = t; i < n4; i += nt) {
    float4 v = reinterpret_cast<float4*>(hi)[i];
    float4 l;
    if (round_hi) {
      const float4 h = make_float4(tf32_rn(v.x), tf32_rn(v.y), tf32_rn(v.z), tf32_rn(v.w));
      l = make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w);
      reinterpret_cast<float4*>(hi)[i] = h;
    } else {
      l = make_float4(v.x - tf32_trunc(v.x), v.y - tf32_trunc(v.y), v.z - tf32_trunc(v.z),
                      v.w - tf32_trunc(v.w));
    }
    reinterpret_cast<float4*>(lo)[i] = l;
  }
}

// The same for two [128 x 128 B] boxes at once (h and the weights of a
// stage) with a compile-time share per thread: every load is issued before
// the first store, so a thread has all eight 16-byte pieces in flight.
template <int kThr>
__device__ __forceinline__ void split_two_boxes(float* hi0, float* lo0, float* hi1, float* lo1, int t) {
  constexpr int kPer = static_cast<int>(kBox / 16) / kThr;  // float4 pieces of one box per thread
  static_assert(kPer * kThr == static_cast<int>(kBox / 16), "box not divisible by the thread count");
  float4 v[2 * kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    v[u] = reinterpret_cast<const float4*>(hi0)[t + u * kThr];
    v[kPer + u] = reinterpret_cast<const float4*>(hi1)[t + u * kThr];
  }
#pragma unroll
  for (int u = 0; u < 2 * kPer; ++u) {
    const float4 x = v[u];
    const float4 h = make_float4(tf32_rn(x.x), tf32_rn(x.y), tf32_rn(x.z), tf32_rn(x.w));
    float* hi = u < kPer ? hi0 : hi1;
    float* lo = u < kPer ? lo0 : lo1;
    const int i = t + (u % kPer) * kThr;
    reinterpret_cast<float4*>(hi)[i] = h;
    reinterpret_cast<float4*>(lo)[i] = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
  }
}

// The same for one [128 x 128 B] box.
template <int kThr>
__device__ __forceinline__ void split_one_box(float* hi0, float* lo0, int t) {
  constexpr int kPer = static_cast<int>(kBox / 16) / kThr;
  static_assert(kPer * kThr == static_cast<int>(kBox / 16), "box not divisible by the thread count");
  float4 v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) v[u] = reinterpret_cast<const float4*>(hi0)[t + u * kThr];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const float4 x = v[u];
    const float4 h = make_float4(tf32_rn(x.x), tf32_rn(x.y), tf32_rn(x.z), tf32_rn(x.w));
    reinterpret_cast<float4*>(hi0)[t + u * kThr] = h;
    reinterpret_cast<float4*>(lo0)[t + u * kThr] = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
  }
}

// The weights' split for the backward, written once per call: out holds
// [W_A hi | W_A lo | W_B hi | W_B lo], n = SH2 x D floats each, hi = tf32_rn(w)
// and lo = w - hi as the tile kernels' own split forms them.
__global__ void __launch_bounds__(256) wide_wsplit_kernel(const float* __restrict__ W_A,
                                                          const float* __restrict__ W_B,
                                                          float* __restrict__ out, int n) {
  const int n4 = n / 4;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 2 * n4; i += gridDim.x * blockDim.x) {
    const int m = i < n4 ? 0 : 1, k = i - m * n4;
    const float4 x = __ldg(reinterpret_cast<const float4*>(m == 0 ? W_A : W_B) + k);
    const float4 h = make_float4(tf32_rn(x.x), tf32_rn(x.y), tf32_rn(x.z), tf32_rn(x.w));
    float4* o = reinterpret_cast<float4*>(out + static_cast<size_t>(2 * m) * n);
    o[k] = h;
    o[n4 + k] = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
  }
}

// Position in a ring of n barriers: index and the parity of its current use.
struct Ring {
  int i = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

// KPP: chunk columns per thread in the C / d_ctx dots, fixed by the samples
// per tile (S_max > 8: 8; S_max > 4: 4; else 2), so that the per-thread
// weight arrays are exactly as large as they are used.
template <bool BWD, int KPP>
__global__ void __launch_bounds__(kTileThreads, 1) wide_tc_kernel(const __grid_constant__ WideTcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  float* sAB = reinterpret_cast<float*>(base + kOffAB);
  float* sC = reinterpret_cast<float*>(base + kOffC);
  float* sDctx = reinterpret_cast<float*>(base + kOffDctx);
  float* sX = reinterpret_cast<float*>(base + kOffX);  // [64][16]: ctx (forward) or dC (backward)
  TileBars* bb = reinterpret_cast<TileBars*>(base + kOffBar);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max;
  const int NQ = SH2 / 32;
  const long long n_tiles = (a.B + S_max - 1) / S_max;
  constexpr uint32_t kCols = 512u;

  if (tid == kProdWarp * 32) {
    for (int s = 0; s < kNst; ++s) {
      mbar_init(&bb->full[s], 1);
      mbar_init(&bb->empty[s], 1);
      mbar_init(&bb->split[s], kCW);
    }
    mbar_init(&bb->acc_full, 1);
    mbar_init(&bb->acc_free, kCW);
    mbar_init(&bb->dab_ready, kCW);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bb->dh_full[s], 1);
      mbar_init(&bb->dh_free[s], kCW);
      mbar_init(&bb->wlo_full[s], 1);
    }
    mbar_init(&bb->tile_done, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&bb->tslot, kCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bb->tslot;

  if (warp == kProdWarp) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      Ring r;
      int n = 0;
      auto take = [&]() -> unsigned char* {
        if (n >= kNst) bounded_wait(&bb->empty[r.i], r.ph ^ 1u, a.err);
        return base + r.i * kStage;
      };
      for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const long long b0 = t * S_max;
        const int row0 = static_cast<int>(b0 * K);
        for (int q = 0; q < NQ; ++q) {
          unsigned char* sp = take();
          uint64_t* bar = &bb->full[r.i];
          mbar_arrive_expect_tx(bar, 2 * kBox + (BWD ? 2u : 1u) * static_cast<uint32_t>(S_max) * 128u);
          tma_load_2d(sp, &a.tm_h, 32 * q, row0, bar);
          tma_load_2d(sp + kBox, &a.tm_wa, 0, 32 * q, bar);
          tma_load_2d(sp + kBox + 4096, &a.tm_wa, 32, 32 * q, bar);
          tma_load_2d(sp + kBox + 8192, &a.tm_wb, 0, 32 * q, bar);
          tma_load_2d(sp + kBox + 12288, &a.tm_wb, 32, 32 * q, bar);
          tma_load_2d(sp + 2 * kBox, &a.tm_hs, 32 * q, static_cast<int>(b0), bar);
          if (BWD) tma_load_2d(sp + 2 * kBox + 2048, &a.tm_g, 32 * q, static_cast<int>(b0), bar);
          r.next(kNst);
          ++n;
        }
        if (BWD) {
          // d_h B operands: per 128-row block of [W_A|W_B] two stages of two
          // 32-column K atoms (W_A columns 0-31, 32-63, then W_B's), K-major
          for (int nb = 0; nb < SH2 / kWN; ++nb)
            for (int half = 0; half < 2; ++half) {
              unsigned char* sp = take();
              uint64_t* bar = &bb->full[r.i];
              mbar_arrive_expect_tx(bar, 2 * kBox);
              const CUtensorMap* m = half == 0 ? &a.tm_wak : &a.tm_wbk;
              tma_load_2d(sp, m, 0, kWN * nb, bar);
              tma_load_2d(sp + kBox, m, 32, kWN * nb, bar);
              r.next(kNst);
              ++n;
            }
        }
      }
    } else if (BWD && lane == 1) {
      // W remainder loader: the backward's weights come split (tf32 part and
      // remainder) from the workspace; the tf32 parts travel in the stages,
      // the remainders go straight into remainder buffer cq & 1 once the
      // products of stage use cq - 2, which read it, are done. The first two
      // chunks of a tile follow the previous tile's d_h stages, whose end the
      // MMA thread signals once (tile_done); the others wait for chunk cq - 2
      // of the same tile. So every wait starts at most one phase ahead of its
      // barrier, and the MMA thread, which needs these copies, cannot get two
      // phases ahead of the loader.
      int cq = 0, lt = 0;
      const int n_dh = 2 * (SH2 / kWN);
      for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
        if (lt > 0) bounded_wait(&bb->tile_done, (lt - 1) & 1, a.err);
        for (int q = 0; q < NQ; ++q, ++cq) {
          if (q >= 2) bounded_wait(&bb->empty[(cq - 2) % kNst], ((cq - 2) / kNst) & 1, a.err);
          unsigned char* lo = base + kOffAB + 2 * kBox * (cq & 1) + kBox;
          uint64_t* bar = &bb->wlo_full[cq & 1];
          mbar_arrive_expect_tx(bar, kBox);
          tma_load_2d(lo, &a.tm_wal, 0, 32 * q, bar);
          tma_load_2d(lo + 4096, &a.tm_wal, 32, 32 * q, bar);
          tma_load_2d(lo + 8192, &a.tm_wbl, 0, 32 * q, bar);
          tma_load_2d(lo + 12288, &a.tm_wbl, 32, 32 * q, bar);
        }
        cq += n_dh;  // the d_h stages: their remainders come from the compute warps
      }
    }
  } else if (warp == kMmaWarp) {
    // --------------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_p = idesc_tf32_mn(128, kWN, 0, 1);  // A K-major, B MN-major
      constexpr uint32_t idesc_d = idesc_tf32_mn(128, kWN, 0, 0);  // A in TMEM, B K-major
      Ring r;
      int lt = 0, cq = 0;    // cq: stages consumed (the remainder buffer is cq & 1)
      int uses[2] = {0, 0};  // d_h blocks issued into each accumulator so far
      int wlo[2] = {0, 0};   // backward: W remainders taken from each buffer so far
      for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
        // TMEM is free again: the previous tile's projections (forward) or
        // its last d_h blocks (backward, which also means that its products
        // reading dA|dB are done) have been read back
        if (BWD) {
          for (int b = 0; b < 2; ++b)
            if (uses[b] > 0) bounded_wait(&bb->dh_free[b], (uses[b] - 1) & 1, a.err);
        } else if (lt > 0) {
          bounded_wait(&bb->acc_free, (lt - 1) & 1, a.err);
        }
        for (int q = 0; q < NQ; ++q) {
          bounded_wait(&bb->full[r.i], r.ph, a.err);
          bounded_wait(&bb->split[r.i], r.ph, a.err);
          if (BWD) bounded_wait(&bb->wlo_full[cq & 1], wlo[cq & 1]++ & 1, a.err);
          tc_fence_after();
          const uint32_t st = smem_addr(base + r.i * kStage);
          const uint32_t lo = smem_addr(base + kOffAB + 2 * kBox * (cq & 1));
          const uint64_t ah = umma_desc_sw128(st), al = umma_desc_sw128(lo);
          const uint64_t bh = desc_mn32(st + kBox, 4096u), bl = desc_mn32(lo + kBox, 4096u);
          // chunk q into accumulator q mod 4 (four short accumulation chains)
          const uint32_t acc = tmem + kWN * (q & 3);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            umma_tf32(acc, ah + 2u * ks, bh + 64u * ks, idesc_p, (q >= 4 || ks > 0) ? 1u : 0u);
            umma_tf32(acc, ah + 2u * ks, bl + 64u * ks, idesc_p, 1u);
            umma_tf32(acc, al + 2u * ks, bh + 64u * ks, idesc_p, 1u);
          }
          umma_commit(&bb->empty[r.i]);
          r.next(kNst);
          ++cq;
        }
        umma_commit(&bb->acc_full);
        if (BWD) {
          bounded_wait(&bb->dab_ready, lt & 1, a.err);
          tc_fence_after();
          for (int nb = 0; nb < SH2 / kWN; ++nb) {
            const int buf = nb & 1;
            const uint32_t d = tmem + kWN * buf;
            if (uses[buf] > 0) bounded_wait(&bb->dh_free[buf], (uses[buf] - 1) & 1, a.err);
            ++uses[buf];
            for (int half = 0; half < 2; ++half) {
              bounded_wait(&bb->full[r.i], r.ph, a.err);
              bounded_wait(&bb->split[r.i], r.ph, a.err);
              tc_fence_after();
              const uint32_t st = smem_addr(base + r.i * kStage);
              const uint32_t lo = smem_addr(base + kOffAB + 2 * kBox * (cq & 1));
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                const int ka = 2 * half + kk;  // K columns [32 ka, 32 ka + 32) of dA|dB
                const uint64_t bh = umma_desc_sw128(st + kBox * kk);
                const uint64_t bl = umma_desc_sw128(lo + kBox * kk);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                  const uint32_t ahi = tmem + 256u + 32u * ka + 8u * ks, alo = ahi + 128u;
                  umma_tf32_ta(d, ahi, bh + 2u * ks, idesc_d, (half > 0 || kk > 0 || ks > 0) ? 1u : 0u);
                  umma_tf32_ta(d, ahi, bl + 2u * ks, idesc_d, 1u);
                  umma_tf32_ta(d, alo, bh + 2u * ks, idesc_d, 1u);
                }
              }
              umma_commit(&bb->empty[r.i]);
              r.next(kNst);
              ++cq;
            }
            umma_commit(&bb->dh_full[buf]);
          }
          // lands once every product of the tile is done: the remainder
          // loader may then fill both remainder buffers for the next tile
          // (none after the last tile, where nobody would wait for it)
          if (t + gridDim.x < n_tiles) umma_commit(&bb->tile_done);
        }
      }
    }
  } else {
    // ----------------------------------------------------------------- compute
    const int q4 = warp & 3, hsel = warp >> 2;  // TMEM lane quadrant; column half
    const int row = 32 * q4 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const float gsc = load_gate_scale(a.gate_scale);
    // C / d_ctx partial dots: thread = (state quad dq, sample quad sq, k part kp)
    constexpr int NKP = 32 / KPP, NSQ = 16 / NKP;
    const int dq = tid & 15, sq = (tid >> 4) % NSQ, kp = (tid >> 4) / NSQ;
    Ring r;
    int lt = 0, cq = 0;     // cq: stages consumed (the remainder buffer is cq & 1)
    int reads[2] = {0, 0};  // d_h blocks read back from each accumulator so far
    // a remainder buffer is written again once the products of the stage
    // before last, which read it, are done (that stage's commit)
    auto lo_buffer = [&]() -> float* {
      if (cq >= 2) bounded_wait(&bb->empty[(cq - 2) % kNst], ((cq - 2) / kNst) & 1, a.err);
      return reinterpret_cast<float*>(base + kOffAB + 2 * kBox * (cq & 1));
    };
    for (long long t = blockIdx.x; t < n_tiles; t += gridDim.x, ++lt) {
      const long long b0 = t * S_max;
      const int S_t = static_cast<int>(min(static_cast<long long>(S_max), a.B - b0));
      const int R_t = S_t * K;
      const long long row0 = b0 * K;
      float cacc[4][4], gacc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) cacc[i][j] = gacc[i][j] = 0.f;
      // ============================================ projection chunks
      // W_C (and W_O) values of chunk q for this thread's dots; those of
      // chunk q + 1 are loaded as soon as chunk q's dots have used them, so
      // their latency runs under the next chunk's wait and remainder work
      float4 wcr[KPP], wor[KPP];
      auto load_chunk_weights = [&](int q) {
        const int k0 = 32 * q;
#pragma unroll
        for (int kk = 0; kk < KPP; ++kk) {
          const int k = kp * KPP + kk;
          wcr[kk] = ldg4w(a.W_C + static_cast<size_t>(k0 + k) * kWD + 4 * dq);
        }
        if (BWD) {
          // W_O rows 4 dq .. 4 dq + 3 over this thread's KPP consecutive
          // columns: 16-byte loads along each row (8-byte when KPP = 2), then
          // regrouped by column
          float ow[4][KPP];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* rowp = a.W_O + static_cast<size_t>(4 * dq + i) * SH2 + k0 + kp * KPP;
            if constexpr (KPP >= 4) {
#pragma unroll
              for (int c = 0; c < KPP; c += 4) {
                const float4 v = ldg4w(rowp + c);
                ow[i][c] = v.x; ow[i][c + 1] = v.y; ow[i][c + 2] = v.z; ow[i][c + 3] = v.w;
              }
            } else {
              const float2 v = __ldg(reinterpret_cast<const float2*>(rowp));
              ow[i][0] = v.x;
              ow[i][1] = v.y;
            }
          }
#pragma unroll
          for (int kk = 0; kk < KPP; ++kk) wor[kk] = make_float4(ow[0][kk], ow[1][kk], ow[2][kk], ow[3][kk]);
        }
      };
      load_chunk_weights(0);
      for (int q = 0; q < NQ; ++q) {
        bounded_wait(&bb->full[r.i], r.ph, a.err);
        float* sp = reinterpret_cast<float*>(base + r.i * kStage);
        float* lo = lo_buffer();
        if (BWD)
          split_one_box<kCT>(sp, lo, tid);  // h (the weights arrive split)
        else
          split_two_boxes<kCT>(sp, lo, sp + kBox / 4, lo + kBox / 4, tid);  // h, W_A|W_B
        {
          const float* hs = sp + 2 * kBox / 4;
          const float* gv = hs + 512;
#pragma unroll
          for (int kk = 0; kk < KPP; ++kk) {
            const int k = kp * KPP + kk;
            const float w4[4] = {wcr[kk].x, wcr[kk].y, wcr[kk].z, wcr[kk].w};
            const float o4[4] = {wor[kk].x, wor[kk].y, wor[kk].z, wor[kk].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int s = 4 * sq + i;
              const float hv = hs[sw128_idx(s, k)];
#pragma unroll
              for (int j = 0; j < 4; ++j) cacc[i][j] = fmaf(hv, w4[j], cacc[i][j]);
              if (BWD) {
                const float g = gv[sw128_idx(s, k)];
#pragma unroll
                for (int j = 0; j < 4; ++j) gacc[i][j] = fmaf(g, o4[j], gacc[i][j]);
              }
            }
          }
        }
        if (q + 1 < NQ) load_chunk_weights(q + 1);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb->split[r.i]);
        r.next(kNst);
        ++cq;
      }
      // the tile's projections are done: the remainder buffers (which share
      // the A|B buffer) have been read
      bounded_wait(&bb->acc_full, lt & 1, a.err);
      tc_fence_after();
      // ===================== C and d_ctx: partial sums of the k parts, in order
      {
        float* red = sAB;  // free until the read-back below
        float* red2 = sAB + 4096;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int s = 4 * sq + i;
          sts4(red + (kp * 4 * NSQ + s) * kWD + 4 * dq,
               make_float4(cacc[i][0], cacc[i][1], cacc[i][2], cacc[i][3]));
          if (BWD)
            sts4(red2 + (kp * 4 * NSQ + s) * kWD + 4 * dq,
                 make_float4(gacc[i][0], gacc[i][1], gacc[i][2], gacc[i][3]));
        }
        named_sync(1, kCT);
        for (int e = tid; e < S_t * kWD; e += kCT) {
          const int s = e >> 6, d = e & 63;
          float c = 0.f, o = 0.f;
          for (int p = 0; p < NKP; ++p) {
            c += red[(p * 4 * NSQ + s) * kWD + d];
            if (BWD) o += red2[(p * 4 * NSQ + s) * kWD + d];
          }
          sC[e] = c;
          if (BWD) sDctx[e] = a.tw * o;
        }
        named_sync(1, kCT);
      }
      // ============================== projections: TMEM -> shared memory
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 16) {
        float v[16];
        {
          uint32_t r0[16], r1[16], r2[16], r3[16];
          const uint32_t ta = lane_base + 64u * hsel + c0;
          tmem_ld16_nowait(ta, r0);
          tmem_ld16_nowait(ta + kWN, r1);
          tmem_ld16_nowait(ta + 2 * kWN, r2);
          tmem_ld16_nowait(ta + 3 * kWN, r3);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            v[i] = (__uint_as_float(r0[i]) + __uint_as_float(r1[i])) +
                   (__uint_as_float(r2[i]) + __uint_as_float(r3[i]));
        }
        const int c = 64 * hsel + c0;
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          sts4(sAB + ab_idx(row, c + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
      }
      tc_fence_before();
      if (!BWD) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb->acc_free);
      }
      named_sync(1, kCT);
      // ===================================================== scan per (s, d)
      // two (sample, state) pairs per thread side by side (p0 and p0 + kCT):
      // each pair's arithmetic is unchanged, the two chains overlap
      for (int p0 = tid; p0 < S_t * kWD; p0 += 2 * kCT) {
        const bool two = p0 + kCT < S_t * kWD;
        int ss[2], dd[2], rbb[2];
        float xx[2] = {0.f, 0.f};
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int p = p0 + jj * kCT;
          ss[jj] = p >> 6;
          dd[jj] = p & 63;
          rbb[jj] = ss[jj] * K;
        }
        for (int u = 0; u < K; ++u) {  // backward: B_t is replaced by x_t
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            if (jj == 1 && !two) break;
            float* pb = sAB + ab_idx(rbb[jj] + u, kWD + dd[jj]);
            xx[jj] = fmaf(gsc * sigmoid_fast(sAB[ab_idx(rbb[jj] + u, dd[jj])]), xx[jj], *pb);
            if (BWD) *pb = xx[jj];
          }
        }
        float dxx[2] = {0.f, 0.f};
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          if (jj == 1 && !two) break;
          const int s = ss[jj], d = dd[jj];
          const float Cv = sC[s * kWD + d];
          if (!BWD) {
            sX[d * kWSmax + s] = Cv * xx[jj];
          } else {
            const float dctx = sDctx[s * kWD + d];
            const float dC = dctx * xx[jj];
            sX[d * kWSmax + s] = dC;
            a.cc[(b0 + s) * kWN + d] = dC;
            a.cc[(b0 + s) * kWN + kWD + d] = Cv * xx[jj];
            dxx[jj] = dctx * Cv;
          }
        }
        if (BWD) {
          for (int u = K - 1; u >= 0; --u) {
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              if (jj == 1 && !two) break;
              const int rr = rbb[jj] + u, d = dd[jj];
              float sg, dsg;
              sigmoid_and_slope(sAB[ab_idx(rr, d)], sg, dsg);
              sg *= gsc;
              dsg *= gsc;
              const float xprev = u > 0 ? sAB[ab_idx(rr - 1, kWD + d)] : 0.f;
              sAB[ab_idx(rr, d)] = dxx[jj] * xprev * dsg;
              sAB[ab_idx(rr, kWD + d)] = dxx[jj];
              dxx[jj] *= sg;
            }
          }
        }
      }
      named_sync(1, kCT);
      if (!BWD) {
        // ============ output h_enriched = h_s2 + tw ctx . W_O: thread = column
        // j, its 64 W_O values loaded at once, every sample of the tile
        for (int j = tid; j < SH2; j += kCT) {
          float w[kWD];
#pragma unroll
          for (int d = 0; d < kWD; ++d) w[d] = __ldg(a.W_O + static_cast<size_t>(d) * SH2 + j);
          // four samples per step: s is a multiple of 4, their sX values in
          // one 16-byte read per state (entries past S_t read, not stored)
          for (int s = 0; s < S_t; s += 4) {
            const int ns = min(4, S_t - s);
            float hs[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) hs[u] = u < ns ? __ldg(a.h_s2 + (b0 + s + u) * SH2 + j) : 0.f;
            float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int d = 0; d < kWD; ++d) {
              const float4 x = *reinterpret_cast<const float4*>(sX + d * kWSmax + s);
              o[0] = fmaf(x.x, w[d], o[0]);
              o[1] = fmaf(x.y, w[d], o[1]);
              o[2] = fmaf(x.z, w[d], o[2]);
              o[3] = fmaf(x.w, w[d], o[3]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (u < ns) a.out0[(b0 + s + u) * SH2 + j] = fmaf(a.tw, o[u], hs[u]);
          }
        }
      } else {
        // ======= dA|dB rows into TMEM (tf32 part at 256, remainder at 384) and
        // to the workspace; the previous tile's d_h products are complete (its
        // last block was read back below)
        {
          const bool ok = row < R_t;
          float* dst = a.dab + (row0 + row) * kWN + 64 * hsel;
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 16) {
            float hi[16], lo[16];
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
              const float4 v = lds4(sAB + ab_idx(row, 64 * hsel + c0 + i));
              if (ok) *reinterpret_cast<float4*>(dst + c0 + i) = v;
              const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                hi[i + e] = tf32_rn(vv[e]);
                lo[i + e] = vv[e] - hi[i + e];
              }
            }
            tmem_st16(lane_base + 256u + 64u * hsel + c0, hi);
            tmem_st16(lane_base + 384u + 64u * hsel + c0, lo);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bb->dab_ready);
        }
        named_sync(1, kCT);  // dA|dB read: the remainder buffers may overwrite it
        // ====== d_h_history per 128-column block: remainders of the weight
        // tiles, then the previous block read back from TMEM to global memory
        const int NB = SH2 / kWN;
        auto readback = [&](int nb) {
          const int buf = nb & 1;
          bounded_wait(&bb->dh_full[buf], reads[buf] & 1, a.err);
          ++reads[buf];
          tc_fence_after();
          const bool ok = row < R_t;
          float* dst = a.out0 + (row0 + row) * SH2 + kWN * nb + 64 * hsel;
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 16) {
            float v[16];
            tmem_ld<16>(lane_base + kWN * buf + 64u * hsel + c0, v);
            if (ok) {
#pragma unroll
              for (int i = 0; i < 16; i += 4)
                *reinterpret_cast<float4*>(dst + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bb->dh_free[buf]);
        };
        for (int nb = 0; nb < NB; ++nb) {
          for (int half = 0; half < 2; ++half) {
            bounded_wait(&bb->full[r.i], r.ph, a.err);
            float* sp = reinterpret_cast<float*>(base + r.i * kStage);
            float* lo = lo_buffer();
            split_two_boxes<kCT>(sp, lo, sp + kBox / 4, lo + kBox / 4, tid);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bb->split[r.i]);
            r.next(kNst);
            ++cq;
          }
          if (nb >= 1) readback(nb - 1);
        }
        readback(NB - 1);
      }
      named_sync(1, kCT);  // sC, sDctx, sX and sAB are reused by the next tile
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kCols);
}

// Weight gradients on the tensor cores. CTA = (job, range p): jobs [0, nb)
// are dW_A|dW_B blocks (128 rows j of SH2 x the 128 columns of dA|dB, reduced
// over the rows of the range), [nb, 2 nb) dW_C blocks (h_s2^T . dC) and
// [2 nb, 3 nb) dW_O^T blocks (dY^T . ctx, times tw), reduced over the samples
// of the range; nb = SH2 / 128. Both operands are MN-major TMA tiles of 32
// rows; rows past the range are zeroed before the products. A range has
// thousands of rows, and a long chain of tensor-core accumulations drifts, so
// the sums are kept short: per 8 rows one product A . [B_hi | B_lo] (N = 2 x
// NOUT) puts hi.hi into the main half of an accumulator and hi.lo into its
// correction half, a second product adds lo.hi into the correction half only,
// and even and odd 32-row chunks use separate accumulators; the four parts are
// added in fp32 at the end.
__global__ void __launch_bounds__(kDwThreads, 1) wide_tc_dw_kernel(const __grid_constant__ WideDwArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  DwBars* bb = reinterpret_cast<DwBars*>(base + kDwOffBar);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int SH2 = a.SH2, P = a.P, nb = SH2 / kWN;
  const int job = blockIdx.x / P, p = blockIdx.x - job * P;
  const int kind = job / nb, jb = job - kind * nb;
  const long long s_lo = a.B * p / P, s_hi = a.B * (p + 1) / P;
  const long long r_lo = kind == 0 ? s_lo * a.K : s_lo, r_hi = kind == 0 ? s_hi * a.K : s_hi;
  const int NC = static_cast<int>((r_hi - r_lo + 31) / 32);
  const int NA = kind == 0 ? 4 : 2;  // 32-column atoms of B
  const CUtensorMap* ma = &a.tm_a[kind];
  const CUtensorMap* mb = &a.tm_b[kind == 0 ? 0 : 1];
  const int b_col0 = kind == 2 ? 64 : 0;
  const int prod_warp = kDwCW, mma_warp = kDwCW + 1;

  if (tid == prod_warp * 32) {
    for (int s = 0; s < kDwNst; ++s) {
      mbar_init(&bb->full[s], 1);
      mbar_init(&bb->empty[s], 1);
      mbar_init(&bb->split[s], kDwCW);
    }
    mbar_init(&bb->done, 1);
    fence_barrier_init();
  }
  if (warp == mma_warp) tmem_alloc(&bb->tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bb->tslot;

  if (warp == prod_warp) {
    if (lane == 0) {
      Ring r;
      for (int c = 0; c < NC; ++c) {
        if (c >= kDwNst) bounded_wait(&bb->empty[r.i], r.ph ^ 1u, a.err);
        unsigned char* sp = base + r.i * kDwStage;
        uint64_t* bar = &bb->full[r.i];
        const int rr = static_cast<int>(r_lo) + 32 * c;
        mbar_arrive_expect_tx(bar, 4096u * (4 + NA));
        for (int m = 0; m < 4; ++m) tma_load_2d(sp + 4096 * m, ma, kWN * jb + 32 * m, rr, bar);
        for (int n = 0; n < NA; ++n) tma_load_2d(sp + 2 * kBox + 4096 * n, mb, b_col0 + 32 * n, rr, bar);
        r.next(kDwNst);
      }
    }
  } else if (warp == mma_warp) {
    if (lane == 0) {
      // B_hi atoms and then B_lo atoms (4096 bytes apart) form one MN-major
      // operand [B_hi | B_lo] of 2 NOUT columns
      const uint32_t nout = 32u * NA;
      const uint32_t idesc2 = idesc_tf32_mn(128, 2 * nout, 1, 1), idesc1 = idesc_tf32_mn(128, nout, 1, 1);
      Ring r;
      for (int c = 0; c < NC; ++c) {
        bounded_wait(&bb->full[r.i], r.ph, a.err);
        bounded_wait(&bb->split[r.i], r.ph, a.err);
        tc_fence_after();
        const uint32_t st = smem_addr(base + r.i * kDwStage);
        const uint64_t ah = desc_mn32(st, 4096u), al = desc_mn32(st + kBox, 4096u);
        const uint64_t bh = desc_mn32(st + 2 * kBox, 4096u);
        const uint32_t acc = tmem + 2u * nout * (c & 1);  // main half, then correction half
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          umma_tf32(acc, ah + 64u * ks, bh + 64u * ks, idesc2, (c >= 2 || ks > 0) ? 1u : 0u);
          umma_tf32(acc + nout, al + 64u * ks, bh + 64u * ks, idesc1, 1u);
        }
        umma_commit(&bb->empty[r.i]);
        r.next(kDwNst);
      }
      umma_commit(&bb->done);
    }
  } else {
    // remainders of both operands; rows past the range zeroed (TMA fetched
    // the next range's rows there, or zeros past the end of the tensor)
    const int ct = tid;  // 0 .. 127
    Ring r;
    for (int c = 0; c < NC; ++c) {
      bounded_wait(&bb->full[r.i], r.ph, a.err);
      float* sp = reinterpret_cast<float*>(base + r.i * kDwStage);
      const int valid = static_cast<int>(min(static_cast<long long>(32), r_hi - r_lo - 32ll * c));
      if (valid < 32) {
        // an atom holds 32 rows of 128 bytes (the 32-byte swizzle only moves
        // data within a row), so row k of every atom is bytes [128 k, 128 k + 128)
        for (int i = ct; i < 8 * 32 * 8; i += kDwCW * 32) {  // 8 atoms x 32 rows x 8 float4
          const int atom = i >> 8, k = (i >> 3) & 31, c4 = i & 7;
          if (k >= valid && (atom < 4 || atom - 4 < NA)) {
            float* buf = sp + (atom < 4 ? 0 : 2 * kBox / 4) + 1024 * (atom & 3);
            reinterpret_cast<float4*>(buf)[k * 8 + c4] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        named_sync(1, kDwCW * 32);
      }
      if (NA == 4) {
        // both operands are full [128 x 128 B] boxes: every load of a thread
        // is issued before its first store
        split_two_boxes<kDwCW * 32>(sp, sp + kBox / 4, sp + 2 * kBox / 4, sp + 3 * kBox / 4, ct);
      } else {
        split_buf(sp, sp + kBox / 4, kBox / 16, ct, kDwCW * 32, true);
        split_buf(sp + 2 * kBox / 4, sp + 2 * kBox / 4 + 1024 * NA, NA * 256, ct, kDwCW * 32, true);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bb->split[r.i]);
      r.next(kDwNst);
    }
    // read-back: thread = row j of the block (TMEM lane), columns = states
    bounded_wait(&bb->done, 0, a.err);
    tc_fence_after();
    const int j = kWN * jb + 32 * warp + lane;
    const uint32_t lb = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    const int n = SH2 * kWD;
    const uint32_t nout = 32u * NA;
    float* slot = a.slots + static_cast<size_t>(p) * 4 * n;
    for (int c0 = 0; c0 < static_cast<int>(nout); c0 += 16) {
      float v[16];
      {
        // (main even + main odd) + (correction even + correction odd); the odd
        // set exists when the range has a second chunk
        uint32_t m0[16], c0r[16], m1[16], c1r[16];
        tmem_ld16_nowait(lb + c0, m0);
        tmem_ld16_nowait(lb + nout + c0, c0r);
        if (NC > 1) {
          tmem_ld16_nowait(lb + 2 * nout + c0, m1);
          tmem_ld16_nowait(lb + 3 * nout + c0, c1r);
        }
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float mm = NC > 1 ? __uint_as_float(m0[i]) + __uint_as_float(m1[i]) : __uint_as_float(m0[i]);
          const float cc = NC > 1 ? __uint_as_float(c0r[i]) + __uint_as_float(c1r[i]) : __uint_as_float(c0r[i]);
          v[i] = mm + cc;
        }
      }
      if (kind == 0) {
        float* dst = slot + (c0 < 64 ? 0 : n) + static_cast<size_t>(j) * kWD + (c0 & 63);
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      } else if (kind == 1) {
        float* dst = slot + 2 * n + static_cast<size_t>(j) * kWD + c0;
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) slot[3 * n + static_cast<size_t>(c0 + i) * SH2 + j] = a.tw * v[i];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) signal_dependent_launch();
  if (warp == mma_warp) tmem_dealloc(tmem, 512);
}

// d_h_s2 = dY + dC . W_C^T ("Custom Kernel Optimization Implementation Plan",
// Task 2: the input gradient of the C projection) over the whole batch. CTA =
// 128 samples x 128 columns, thread = 8 samples x 8 columns (4 in each
// 64-column half, so that a warp's W_C reads are contiguous); dC (columns 0..63
// of the workspace's [dC | ctx] rows) and the CTA's 128 rows of W_C are staged
// transposed in shared memory (68 KB), so that for each state d a thread reads
// its 8 dC values and 8 W_C values as two 16-byte pieces each and does 64
// multiply-adds with them. Every output starts from dY and adds its 64
// products in state order with fused multiply-adds.
constexpr int kHsS = 128, kHsJ = 128, kHsThreads = 256;
constexpr int kHsPadS = kHsS + 4, kHsPadJ = kHsJ + 4;  // row strides, 16-byte multiples
constexpr uint32_t kHsSmem = (kWD * kHsPadS + kWD * kHsPadJ) * 4;

__global__ void __launch_bounds__(kHsThreads) wide_dhs2_kernel(const float* __restrict__ g,
                                                                const float* __restrict__ cc,
                                                                const float* __restrict__ W_C,
                                                                float* __restrict__ out, long long B,
                                                                int SH2) {
  extern __shared__ __align__(16) float hs_smem[];
  float* sdc = hs_smem;                  // dC^T [d][s]
  float* swc = hs_smem + kWD * kHsPadS;  // W_C^T [d][j]
  const int tid = threadIdx.x;
  const long long s0 = static_cast<long long>(blockIdx.x) * kHsS;
  const int j0 = blockIdx.y * kHsJ;
  const int ns = static_cast<int>(min(static_cast<long long>(kHsS), B - s0));
  // this thread's outputs start from dY: samples 8 sg .. 8 sg + 7, columns
  // 4 cg .. 4 cg + 3 and 64 + 4 cg .. 64 + 4 cg + 3 (a warp reads two 256-byte
  // row pieces of two samples); requested first, their latency runs under
  // the staging below
  const int cg = tid & 15, sg = tid >> 4;
  float o[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int sl = 8 * sg + i;
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    if (sl < ns) {
      const float* gp = g + (s0 + sl) * SH2 + j0 + 4 * cg;
      a0 = ldg4w(gp);
      a1 = ldg4w(gp + kHsJ / 2);
    }
    o[i][0] = a0.x; o[i][1] = a0.y; o[i][2] = a0.z; o[i][3] = a0.w;
    o[i][4] = a1.x; o[i][5] = a1.y; o[i][6] = a1.z; o[i][7] = a1.w;
  }
  // staging: consecutive threads take consecutive samples (or columns), so
  // the transposed stores fall in distinct banks; each pass issues all its
  // loads before its first store
  constexpr int kPer = kHsS * (kWD / 4) / kHsThreads;  // float4 per thread and matrix
  static_assert(kHsS == kHsJ && kPer * kHsThreads == kHsS * (kWD / 4), "staging split");
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    float4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = tid + u * kHsThreads, r = i % kHsS, d4 = i / kHsS;
      if (m == 0)
        v[u] = r < ns ? ldg4w(cc + (s0 + r) * kWN + 4 * d4) : make_float4(0.f, 0.f, 0.f, 0.f);
      else
        v[u] = ldg4w(W_C + static_cast<size_t>(j0 + r) * kWD + 4 * d4);
    }
    float* dst = m == 0 ? sdc : swc;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = tid + u * kHsThreads, r = i % kHsS, d4 = i / kHsS;
      dst[(4 * d4 + 0) * kHsPadS + r] = v[u].x;
      dst[(4 * d4 + 1) * kHsPadS + r] = v[u].y;
      dst[(4 * d4 + 2) * kHsPadS + r] = v[u].z;
      dst[(4 * d4 + 3) * kHsPadS + r] = v[u].w;
    }
  }
  __syncthreads();
#pragma unroll 2
  for (int d = 0; d < kWD; ++d) {
    const float4 x0 = *reinterpret_cast<const float4*>(sdc + d * kHsPadS + 8 * sg);
    const float4 x1 = *reinterpret_cast<const float4*>(sdc + d * kHsPadS + 8 * sg + 4);
    const float4 w0 = *reinterpret_cast<const float4*>(swc + d * kHsPadJ + 4 * cg);
    const float4 w1 = *reinterpret_cast<const float4*>(swc + d * kHsPadJ + kHsJ / 2 + 4 * cg);
    const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    const float ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int c = 0; c < 8; ++c) o[i][c] = fmaf(xs[i], ws[c], o[i][c]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int sl = 8 * sg + i;
    if (sl < ns) {
      float* op = out + (s0 + sl) * SH2 + j0 + 4 * cg;
      *reinterpret_cast<float4*>(op) = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
      *reinterpret_cast<float4*>(op + kHsJ / 2) = make_float4(o[i][4], o[i][5], o[i][6], o[i][7]);
    }
  }
}

}  // namespace

bool wide_path_ok(int K, int SH2, int D) {
  return D == kWD && SH2 >= kWN && SH2 % kWN == 0 && K >= 1 && K <= kWRows &&
         kTileSmem <= 227u * 1024u;
}

int wide_ranges(int64_t B) { return B < kWRanges ? static_cast<int>(B) : kWRanges; }

size_t wide_bwd_workspace_bytes(int64_t B, int32_t K, int32_t SH2) {
  const size_t slots = static_cast<size_t>(wide_ranges(B)) * 4 * static_cast<size_t>(SH2) * kWD;
  const size_t dab = static_cast<size_t>(B) * K * kWN;
  const size_t cc = static_cast<size_t>(B) * kWN;
  const size_t wsplit = 4 * static_cast<size_t>(SH2) * kWD;  // the weights' tf32 parts and remainders
  return (slots + dab + cc + wsplit) * sizeof(float);
}

static int wide_s_max(int K) {
  const int s = kWRows / K;
  return s < kWSmax ? s : kWSmax;
}

// Tensor maps of the tile kernels (see WideTcArgs).
static bool wide_tile_maps(WideTcArgs* w, const float* h_history, const float* h_s2, const float* g,
                           const float* W_A, const float* W_B, int64_t B, int K, int SH2) {
  const cuuint64_t rows = static_cast<cuuint64_t>(B) * K, sh = static_cast<cuuint64_t>(SH2);
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B, sw32 = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
  {
    const cuuint64_t d[2] = {sh, rows}, s[1] = {sh * 4};
    const cuuint32_t b[2] = {32, kWRows};
    if (encode_tensor_map(&w->tm_h, h_history, 2, d, s, b, sw) != CUDA_SUCCESS) return false;
  }
  {
    const cuuint64_t d[2] = {static_cast<cuuint64_t>(kWD), sh}, s[1] = {kWD * 4};
    const cuuint32_t bm[2] = {32, 32}, bk[2] = {32, kWN};
    if (encode_tensor_map(&w->tm_wa, W_A, 2, d, s, bm, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&w->tm_wb, W_B, 2, d, s, bm, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&w->tm_wak, W_A, 2, d, s, bk, sw) != CUDA_SUCCESS ||
        encode_tensor_map(&w->tm_wbk, W_B, 2, d, s, bk, sw) != CUDA_SUCCESS)
      return false;
  }
  {
    const cuuint64_t d[2] = {sh, static_cast<cuuint64_t>(B)}, s[1] = {sh * 4};
    const cuuint32_t b[2] = {32, static_cast<cuuint32_t>(w->S_max)};
    if (encode_tensor_map(&w->tm_hs, h_s2, 2, d, s, b, sw) != CUDA_SUCCESS) return false;
    if (encode_tensor_map(&w->tm_g, g ? g : h_s2, 2, d, s, b, sw) != CUDA_SUCCESS) return false;
  }
  return true;
}

// Chunk columns per thread of the C / d_ctx dots for S_max samples per tile.
static int wide_kpp(int S_max) { return S_max > 8 ? 8 : (S_max > 4 ? 4 : 2); }

template <bool BWD>
static void launch_wide_tile(const WideTcArgs& w, int grid, cudaStream_t stream) {
  switch (wide_kpp(w.S_max)) {
    case 8: wide_tc_kernel<BWD, 8><<<grid, kTileThreads, kTileSmem, stream>>>(w); break;
    case 4: wide_tc_kernel<BWD, 4><<<grid, kTileThreads, kTileSmem, stream>>>(w); break;
    default: wide_tc_kernel<BWD, 2><<<grid, kTileThreads, kTileSmem, stream>>>(w); break;
  }
}

static int wide_grid(int64_t B, int S_max) {
  const long long n_tiles = (B + S_max - 1) / S_max;
  return static_cast<int>(n_tiles < kMaxSlots ? n_tiles : kMaxSlots);
}

cudaError_t launch_wide_fwd(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw, int64_t B,
                            int K, int SH2, float* h_enriched, const float* gate_scale, unsigned* err,
                            cudaStream_t stream) {
  WideTcArgs w{};
  w.S_max = wide_s_max(K);
  if (!wide_tile_maps(&w, h_history, h_s2, nullptr, W_A, W_B, B, K, SH2)) return cudaErrorInvalidValue;
  w.h_s2 = h_s2; w.W_C = W_C; w.W_O = W_O; w.out0 = h_enriched;
  w.gate_scale = gate_scale; w.err = err; w.B = B; w.K = K; w.SH2 = SH2; w.tw = tw;
  launch_wide_tile<false>(w, wide_grid(B, w.S_max), stream);
  return cudaGetLastError();
}

// The weights' split, the tile kernel, d_h_s2, the weight-gradient products
// and the slot reduction: the number of launches goes to *n.
cudaError_t launch_wide_bwd(const float* h_history, const float* h_s2, const float* W_A,
                            const float* W_B, const float* W_C, const float* W_O, float tw,
                            const float* g, int64_t B, int K, int SH2, float* d_h_history,
                            float* d_h_s2, float* dW_A, float* dW_B, float* dW_C, float* dW_O,
                            void* workspace, const float* gate_scale, unsigned* err,
                            cudaStream_t stream, int* n) {
  *n = 0;
  WideTcArgs w{};
  w.S_max = wide_s_max(K);
  if (!wide_tile_maps(&w, h_history, h_s2, g, W_A, W_B, B, K, SH2)) return cudaErrorInvalidValue;
  const int P = wide_ranges(B);
  float* ws = static_cast<float*>(workspace);
  float* slots = ws;
  float* dab = ws + static_cast<size_t>(P) * 4 * static_cast<size_t>(SH2) * kWD;
  float* cc = dab + static_cast<size_t>(B) * K * kWN;
  // the weights split once for every CTA: [W_A hi | W_A lo | W_B hi | W_B lo];
  // the projections' B operands (MN-major) then come from these arrays
  float* wsplit = cc + static_cast<size_t>(B) * kWN;
  const int nw = SH2 * kWD;
  {
    const CUtensorMapSwizzle sw32 = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
    const cuuint64_t d[2] = {static_cast<cuuint64_t>(kWD), static_cast<cuuint64_t>(SH2)}, s[1] = {kWD * 4};
    const cuuint32_t bm[2] = {32, 32};
    if (encode_tensor_map(&w.tm_wa, wsplit, 2, d, s, bm, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&w.tm_wal, wsplit + nw, 2, d, s, bm, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&w.tm_wb, wsplit + 2 * nw, 2, d, s, bm, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&w.tm_wbl, wsplit + 3 * nw, 2, d, s, bm, sw32) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  w.h_s2 = h_s2; w.W_C = W_C; w.W_O = W_O; w.out0 = d_h_history;
  w.dab = dab; w.cc = cc; w.gate_scale = gate_scale; w.err = err;
  w.B = B; w.K = K; w.SH2 = SH2; w.tw = tw;
  wide_wsplit_kernel<<<(2 * (nw / 4) + 255) / 256, 256, 0, stream>>>(W_A, W_B, wsplit, nw);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*n;
  launch_wide_tile<true>(w, wide_grid(B, w.S_max), stream);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n;
  const dim3 hs_grid(static_cast<unsigned>((B + kHsS - 1) / kHsS), static_cast<unsigned>(SH2 / kHsJ));
  wide_dhs2_kernel<<<hs_grid, kHsThreads, kHsSmem, stream>>>(g, cc, W_C, d_h_s2, B, SH2);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n;
  WideDwArgs dw{};
  {
    const CUtensorMapSwizzle sw32 = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
    const cuuint64_t sh = static_cast<cuuint64_t>(SH2), rows = static_cast<cuuint64_t>(B) * K,
                     bb = static_cast<cuuint64_t>(B), wn = kWN;
    const cuuint32_t box[2] = {32, 32};
    const cuuint64_t dh[2] = {sh, rows}, ds[2] = {sh, bb}, sa[1] = {sh * 4};
    const cuuint64_t dd[2] = {wn, rows}, dc[2] = {wn, bb}, sb[1] = {wn * 4};
    if (encode_tensor_map(&dw.tm_a[0], h_history, 2, dh, sa, box, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&dw.tm_a[1], h_s2, 2, ds, sa, box, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&dw.tm_a[2], g, 2, ds, sa, box, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&dw.tm_b[0], dab, 2, dd, sb, box, sw32) != CUDA_SUCCESS ||
        encode_tensor_map(&dw.tm_b[1], cc, 2, dc, sb, box, sw32) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  dw.slots = slots; dw.err = err; dw.B = B; dw.K = K; dw.SH2 = SH2; dw.P = P; dw.tw = tw;
  const int jobs = 3 * (SH2 / kWN);
  wide_tc_dw_kernel<<<jobs * P, kDwThreads, kDwSmem, stream>>>(dw);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ++*n;
  e = launch_reduce(slots, P, SH2 * kWD, dW_A, dW_B, dW_C, dW_O, stream);
  if (e == cudaSuccess) ++*n;
  return e;
}

cudaError_t prepare_wide_kernels() {
  const void* tiles[] = {
      reinterpret_cast<const void*>(wide_tc_kernel<false, 2>), reinterpret_cast<const void*>(wide_tc_kernel<false, 4>),
      reinterpret_cast<const void*>(wide_tc_kernel<false, 8>), reinterpret_cast<const void*>(wide_tc_kernel<true, 2>),
      reinterpret_cast<const void*>(wide_tc_kernel<true, 4>), reinterpret_cast<const void*>(wide_tc_kernel<true, 8>)};
  cudaError_t e = cudaSuccess;
  for (const void* k : tiles)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kTileSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wide_tc_dw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kDwSmem));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(wide_dhs2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kHsSmem));
  return e;
}

}  // namespace m2scan
