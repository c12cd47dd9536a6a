// Backward of the gated temporal scan layer with bf16 activations on the tensor
// cores (D = 16, SH2 % 64 == 0, SH2 <= 256, K <= 128): h_history, h_s2 and
// d_h_enriched are bfloat16 inputs, d_h_history and d_h_s2 bfloat16 outputs,
// weights and weight gradients fp32, every sum fp32.
//
// One persistent CTA per weight-gradient slot walks its samples in tiles of at
// most 128 rows (S samples x K). A bf16 activation is exact as a tensor-core
// operand, so no remainder of it is ever formed; the fp32 factors are split
// into bf16 parts (x = x0 + x1 + x2, 24 significant bits). And a 64-column
// block of h_history as TMA writes it (128-byte rows, 128-byte swizzle) is
// both a K-major operand (rows x columns) and an MN-major one (columns x
// rows), so no operand is ever transposed by a thread. Per tile:
//   pass 1   blocks of h_history stream through a ring of three stages with the
//            matching 64 columns of h_s2 and d_h_enriched. One MMA thread
//            forms A|B = h . [W0 | W1 | W2] (kind::f16, N = 96, the three parts
//            of [W_A|W_B] resident in shared memory); the compute warps form
//            C = h_s2 . W_C and d_ctx = tw dY . W_O^T on the FMA pipe.
//   scan     replay of the forward scan and the reverse scan of the
//            implementation plan's Task 2 ("Custom Kernel Optimization
//            Implementation Plan"): dB_t = dx, dA_t = dx x_{t-1} sigmoid'(A_t),
//            dx <- dx sigmoid(A_t), one thread per (sample, state). dA|dB go,
//            split into bf16 parts, into one buffer T of 128 rows of 128 tile
//            rows: rows [a0 | a0 | a1 | a2] (32 each: dA then dB).
//   d_h      d_h_history = dA|dB . [W_A|W_B]^T as a0 W0 + a0 W1 + a1 W0: T read
//            MN-major (tile rows x parts) against [W0 | W1] rows of the
//            weights, resident in shared memory; read back, rounded to bf16.
//   dW, items  the producer streams the tile's h_history blocks again (with
//            h_s2 and dY); the MMA thread accumulates
//            dW_A|dW_B^T += T . h (T read K-major, h MN-major) in tensor memory
//            over every tile of the CTA, while the compute warps accumulate dW_C
//            and dW_O in registers and write d_h_s2 = dY + dC . W_C^T.
// Each CTA writes its partial sums once to its slot; the slot reduction adds
// the slots in a fixed order, so the weight gradients are bit-identical run
// to run.
#include <cuda_bf16.h>

#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kD = 16;
constexpr int kTD = 32;            // columns of A|B (2D)
constexpr int kCW = 8;             // compute warps
constexpr int kCT = kCW * 32;
constexpr int kThreadsB = kCT + 64;  // + producer warp + MMA warp
constexpr int kProd = kCW, kMma = kCW + 1;
constexpr int kNst = 3;            // copy ring depth
constexpr int kBlk = 64;           // SH2 columns (bf16) per block: one 128-byte row
constexpr int kMaxNB = 4;          // blocks per row, at most (SH2 <= 256)
constexpr uint32_t kHBox = 16384;  // [128 rows x 128 B]
constexpr uint32_t kStageB = kHBox + 4096;  // h block + h_s2 / dY boxes (S_max x 128 B each)
constexpr int kPadW = 4;           // padding (floats) of the fp32 weight rows

// shared memory (bytes from the 1024-aligned base)
constexpr uint32_t kOffWp = 0;                                // [NB][96 x 128 B] pass-1 weights
constexpr uint32_t kOffWr = kOffWp + kMaxNB * 96 * 128;       // [SH2 x 128 B] d_h weights
constexpr uint32_t kOffT = kOffWr + 256 * 128;                // [2][128 x 128 B] dA|dB parts
constexpr uint32_t kOffRing = kOffT + 2 * kHBox;
constexpr uint32_t kOffAB = kOffRing + kNst * kStageB;        // A|B fp32 [128][32], swizzled
constexpr uint32_t kOffWct = kOffAB + 128 * kTD * 4;          // W_C^T fp32 [16][SH2 + 4]
constexpr uint32_t kOffWo = kOffWct + kD * (256 + kPadW) * 4; // W_O fp32 [16][SH2 + 4]
constexpr uint32_t kOffSm = kOffWo + kD * (256 + kPadW) * 4;  // dC, ctx [16][16] each
constexpr uint32_t kOffBarB = kOffSm + 2 * 16 * kD * 4;
constexpr uint32_t kSmemB = kOffBarB + 256 + 1024;

struct Bars {
  uint64_t full[kNst];   // producer -> all: stage loaded
  uint64_t empty[kNst];  // stage read: MMA commit + one arrival per compute warp
  uint64_t acc_full;     // MMA -> compute: the tile's projections done
  uint64_t t_ready;      // compute -> MMA: T written (one arrival per warp)
  uint64_t dh_full;      // MMA -> compute: d_h done
  uint64_t dh_free;      // compute -> MMA: d_h read back (one arrival per warp)
  uint64_t dw_done;      // MMA -> compute: every weight-gradient product done
  uint32_t tslot;
};

// TMEM columns: [0, 256) the projections (96 columns), then d_h (SH2 columns)
// of the same tile; [256, 256 + SH2) dW_A|dW_B^T: lane = part row of T, column
// = feature j.
constexpr uint32_t kColDW = 256;

__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 128-byte-swizzled shared-memory descriptor with explicit byte offsets:
// LBO = between 64-element blocks along M/N (MN-major operands), SBO = between
// 8-row groups.
__device__ __forceinline__ uint64_t desc_sw128x(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Byte offset of element (row, c) in a region of 128-byte rows of 64 bf16,
// 128-byte swizzle (16-byte chunk index XOR-ed with row mod 8).
__device__ __forceinline__ uint32_t bf_off(int row, int c) {
  return static_cast<uint32_t>(row) * 128u + ((((c >> 3) ^ (row & 7))) << 4) + (c & 7) * 2u;
}

__device__ __forceinline__ float bfv(const unsigned char* base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + off));
}

__device__ __forceinline__ void put_bf(unsigned char* base, uint32_t off, float v) {
  *reinterpret_cast<__nv_bfloat16*>(base + off) = __float2bfloat16_rn(v);
}

// v = p0 + p1 + p2 with each part a bf16 (round to nearest), 24 significant bits.
__device__ __forceinline__ void bf_parts(float v, float& p0, float& p1, float& p2) {
  p0 = __bfloat162float(__float2bfloat16_rn(v));
  const float r1 = v - p0;
  p1 = __bfloat162float(__float2bfloat16_rn(r1));
  p2 = __bfloat162float(__float2bfloat16_rn(r1 - p1));
}

struct Ring {
  int i = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++i == kNst) {
      i = 0;
      ph ^= 1u;
    }
  }
};

__global__ void __launch_bounds__(kThreadsB, 1) bwd_bf16_tc_kernel(const __grid_constant__ FastArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* sWp = base + kOffWp;
  unsigned char* sWr = base + kOffWr;
  unsigned char* sT = base + kOffT;
  float* sAB = reinterpret_cast<float*>(base + kOffAB);
  float* sWct = reinterpret_cast<float*>(base + kOffWct);
  float* sWo = reinterpret_cast<float*>(base + kOffWo);
  float* sDC = reinterpret_cast<float*>(base + kOffSm);  // [16][16]
  float* sCtx = sDC + 16 * kD;                           // [16][16]
  Bars* bb = reinterpret_cast<Bars*>(base + kOffBarB);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max, NB = SH2 / kBlk;
  const int SH2P = SH2 + kPadW;
  const long long B = a.B;
  const int P = gridDim.x, cta = blockIdx.x;
  const long long cb0 = B * cta / P;
  const int n_c = static_cast<int>(B * (cta + 1) / P - cb0);
  const int T = (n_c + S_max - 1) / S_max;
  const int t_base = n_c / T, t_extra = n_c - (n_c / T) * T;
  auto tile_start = [&](int i) -> long long {
    return cb0 + static_cast<long long>(i) * t_base + (i < t_extra ? i : t_extra);
  };

  if (tid == kProd * 32) {
    for (int s = 0; s < kNst; ++s) {
      mbar_init(&bb->full[s], 1);
      mbar_init(&bb->empty[s], 1 + kCW);
    }
    mbar_init(&bb->acc_full, 1);
    mbar_init(&bb->t_ready, kCW);
    mbar_init(&bb->dh_full, 1);
    mbar_init(&bb->dh_free, kCW);
    mbar_init(&bb->dw_done, 1);
    fence_barrier_init();
  }
  if (warp == kMma) tmem_alloc(&bb->tslot, 512);
  // the producer requests the first stages (they need no weights) before the
  // weights are staged, so that both latencies overlap
  Ring pr;
  int pn = 0, ptile = 0, ppass = 0, pq = 0;  // producer: stages issued; position of the next
  auto produce_one = [&]() {
    const long long tb0 = tile_start(ptile);
    const int row0 = static_cast<int>(tb0 * K);
    if (pn >= kNst) bounded_wait(&bb->empty[pr.i], pr.ph ^ 1u, a.err);
    unsigned char* sp = base + kOffRing + pr.i * kStageB;
    uint64_t* bar = &bb->full[pr.i];
    mbar_arrive_expect_tx(bar, kHBox + 2u * static_cast<uint32_t>(S_max) * 128u);
    tma_load_2d(sp, &a.tm_h, kBlk * pq, row0, bar);
    tma_load_2d(sp + kHBox, &a.tm_hs, kBlk * pq, static_cast<int>(tb0), bar);
    tma_load_2d(sp + kHBox + 2048, &a.tm_g, kBlk * pq, static_cast<int>(tb0), bar);
    pr.next();
    ++pn;
    if (++pq == NB) {
      pq = 0;
      if (++ppass == 2) {
        ppass = 0;
        ++ptile;
      }
    }
  };
  if (tid == kProd * 32)
    for (int i = 0; i < kNst && ptile < T; ++i) produce_one();
  // ---- weights, thread = feature j: the three bf16 parts of [W_A|W_B] row j
  // (pass 1: rows p * 32 + c of block j / 64), [W0 | W1] row j (d_h), and W_C^T,
  // W_O as fp32 rows for the FMA pipe. Every global load is issued first.
  if (warp < kCW) {
    const int j = tid;
    if (j < SH2) {
      float4 wr[8], wcr[4];
      float wor[kD];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wr[i] = __ldg(reinterpret_cast<const float4*>(a.W_A + j * kD) + i);
        wr[4 + i] = __ldg(reinterpret_cast<const float4*>(a.W_B + j * kD) + i);
        wcr[i] = __ldg(reinterpret_cast<const float4*>(a.W_C + j * kD) + i);
      }
#pragma unroll
      for (int c = 0; c < kD; ++c) wor[c] = __ldg(a.W_O + c * SH2 + j);
      const int q = j / kBlk, jj = j % kBlk;
      unsigned char* wp = sWp + q * 96 * 128;
#pragma unroll
      for (int c = 0; c < kTD; ++c) {
        const float4 v4 = wr[c >> 2];
        const float w = (c & 3) == 0 ? v4.x : (c & 3) == 1 ? v4.y : (c & 3) == 2 ? v4.z : v4.w;
        float p0, p1, p2;
        bf_parts(w, p0, p1, p2);
        put_bf(wp, bf_off(c, jj), p0);
        put_bf(wp, bf_off(kTD + c, jj), p1);
        put_bf(wp, bf_off(2 * kTD + c, jj), p2);
        put_bf(sWr, bf_off(j, c), p0);
        put_bf(sWr, bf_off(j, kTD + c), p1);
      }
#pragma unroll
      for (int c = 0; c < kD; ++c) {
        const float4 v4 = wcr[c >> 2];
        sWct[c * SH2P + j] = (c & 3) == 0 ? v4.x : (c & 3) == 1 ? v4.y : (c & 3) == 2 ? v4.z : v4.w;
        sWo[c * SH2P + j] = wor[c];
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bb->tslot;

  if (warp == kProd) {
    // ---------------------------------------------------------------- producer
    if (lane == 0)
      while (ptile < T) produce_one();
  } else if (warp == kMma) {
    // --------------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_p = idesc_f16(128, 96, 0, 0);
      const uint32_t idesc_h = idesc_f16(128, SH2, 1, 0);
      constexpr uint32_t idesc_w = idesc_f16(128, kBlk, 0, 1);
      const uint32_t ring = smem_addr(base + kOffRing), wp = smem_addr(sWp), wr = smem_addr(sWr),
                     tt = smem_addr(sT);
      Ring r;
      for (int t = 0; t < T; ++t) {
        if (t > 0) bounded_wait(&bb->dh_free, (t - 1) & 1, a.err);  // columns [0, 256) free
        // pass 1: A|B = h . [W0 | W1 | W2]
        for (int q = 0; q < NB; ++q) {
          bounded_wait(&bb->full[r.i], r.ph, a.err);
          tc_fence_after();
          const uint64_t ad = umma_desc_sw128(ring + r.i * kStageB);
          const uint64_t bd = umma_desc_sw128(wp + q * 96 * 128);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_f16(tmem, ad + 2u * ks, bd + 2u * ks, idesc_p, (q > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bb->empty[r.i]);
          r.next();
        }
        umma_commit(&bb->acc_full);
        bounded_wait(&bb->t_ready, t & 1, a.err);
        tc_fence_after();
        // d_h = [a0 | a0] . [W0 | W1] + a1 . W0: T MN-major (tile rows in two
        // 64-row blocks 16 KB apart), 16 part rows per step (2048 bytes)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          umma_f16(tmem, desc_sw128x(tt + 2048u * ks, kHBox, 1024u),
                   desc_sw128x(wr + 32u * ks, 16u, 1024u), idesc_h, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
          umma_f16(tmem, desc_sw128x(tt + 2048u * (4 + ks), kHBox, 1024u),
                   desc_sw128x(wr + 32u * ks, 16u, 1024u), idesc_h, 1u);
        umma_commit(&bb->dh_full);
        // dW_A|dW_B^T[part row, j] += T . h: T K-major (16 tile rows per step,
        // 32 bytes; the second 64 tile rows 16 KB on), h block MN-major
        for (int q = 0; q < NB; ++q) {
          bounded_wait(&bb->full[r.i], r.ph, a.err);
          tc_fence_after();
          const uint32_t hb = ring + r.i * kStageB;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_f16(tmem + kColDW + kBlk * q,
                     desc_sw128x(tt + kHBox * (ks >> 2) + 32u * (ks & 3), 16u, 1024u),
                     desc_sw128x(hb + 2048u * ks, kHBox, 1024u), idesc_w,
                     (t > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bb->empty[r.i]);
          r.next();
        }
      }
      umma_commit(&bb->dw_done);
    }
  } else {
    // ----------------------------------------------------------------- compute
    const int q4 = warp & 3, hsel = warp >> 2;  // TMEM lane quadrant, column half
    const int row = 32 * q4 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q4) << 16);
    const float gsc = load_gate_scale(a.gate_scale);
    const int ss = tid >> 4, sd = tid & 15;  // (sample, state) of the scan
    const int jp = (tid >> 4) & 3, sq = tid >> 6;  // dots: 16-column part, sample quad
    const int jj = tid & 63, cq = tid >> 6;  // column in a block, state / sample quad of the items
    float wcacc[kMaxNB][4], woacc[kMaxNB][4];  // dW_C[j][4cq + e], dW_O[4cq + e][j] partial sums
#pragma unroll
    for (int q = 0; q < kMaxNB; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) wcacc[q][e] = woacc[q][e] = 0.f;
    Ring r;
    for (int t = 0; t < T; ++t) {
      const long long tb0 = tile_start(t);
      const int S_t = static_cast<int>(tile_start(t + 1) - tb0);
      const int R_t = S_t * K;
      const long long row0 = tb0 * K;
      // ===== pass 1: C and d_ctx; thread = (state sd, samples 4 sq .. 4 sq + 3,
      // columns 16 jp .. 16 jp + 15 of each block): a weight row serves 4 samples
      float cacc[4] = {0.f, 0.f, 0.f, 0.f}, gacc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < NB; ++q) {
        bounded_wait(&bb->full[r.i], r.ph, a.err);
        const unsigned char* sp = base + kOffRing + r.i * kStageB;
        const unsigned char* hs = sp + kHBox;
        const unsigned char* gs = hs + 2048;
        const float* wc = sWct + sd * SH2P + kBlk * q;
        const float* wo = sWo + sd * SH2P + kBlk * q;
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          const int c8 = 2 * jp + h8;
          const float4 w0 = lds4(wc + 8 * c8), w1 = lds4(wc + 8 * c8 + 4);
          const float4 o0 = lds4(wo + 8 * c8), o1 = lds4(wo + 8 * c8 + 4);
          const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          const float ov[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint4 hv = *reinterpret_cast<const uint4*>(hs + bf_off(4 * sq + i, 8 * c8));
            const uint4 g4 = *reinterpret_cast<const uint4*>(gs + bf_off(4 * sq + i, 8 * c8));
            const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w}, gw[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              cacc[i] = fmaf(__uint_as_float(hw[e] << 16), wv[2 * e], cacc[i]);
              cacc[i] = fmaf(__uint_as_float(hw[e] & 0xFFFF0000u), wv[2 * e + 1], cacc[i]);
              gacc[i] = fmaf(__uint_as_float(gw[e] << 16), ov[2 * e], gacc[i]);
              gacc[i] = fmaf(__uint_as_float(gw[e] & 0xFFFF0000u), ov[2 * e + 1], gacc[i]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb->empty[r.i]);
        r.next();
      }
      // the four column parts added in order (A|B's buffer is free until the
      // read-back below)
      float cv, gv;
      {
        float* red = sAB;  // [4 jp][16 s][16 d], C then d_ctx
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          red[(jp * 16 + 4 * sq + i) * kD + sd] = cacc[i];
          red[1024 + (jp * 16 + 4 * sq + i) * kD + sd] = gacc[i];
        }
        named_sync(1, kCT);
        cv = (red[ss * kD + sd] + red[(16 + ss) * kD + sd]) +
             (red[(32 + ss) * kD + sd] + red[(48 + ss) * kD + sd]);
        gv = (red[1024 + ss * kD + sd] + red[1024 + (16 + ss) * kD + sd]) +
             (red[1024 + (32 + ss) * kD + sd] + red[1024 + (48 + ss) * kD + sd]);
        named_sync(1, kCT);
      }
      const float dctx = a.tw * gv;
      // =========================== projections: TMEM -> A|B (three parts added)
      bounded_wait(&bb->acc_full, t & 1, a.err);
      tc_fence_after();
      {
        float v[3][16];
        tmem_ld<16>(lane_base + 16u * hsel, v[0]);
        tmem_ld<16>(lane_base + kTD + 16u * hsel, v[1]);
        tmem_ld<16>(lane_base + 2 * kTD + 16u * hsel, v[2]);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const int c4 = (4 * hsel + i / 4) ^ (row & 7);
          sts4(sAB + row * kTD + 4 * c4,
               make_float4((v[0][i] + v[1][i]) + v[2][i], (v[0][i + 1] + v[1][i + 1]) + v[2][i + 1],
                           (v[0][i + 2] + v[1][i + 2]) + v[2][i + 2],
                           (v[0][i + 3] + v[1][i + 3]) + v[2][i + 3]));
        }
      }
      tc_fence_before();
      named_sync(1, kCT);
      // ======== scan and reverse scan of (sample ss, state sd); dA|dB parts -> T
      auto ab = [&](int rr, int c) -> float& {
        return sAB[rr * kTD + ((((c >> 2) ^ (rr & 7))) << 2) + (c & 3)];
      };
      auto put_t = [&](int prow, int rr, float v) {
        put_bf(sT + kHBox * (rr >> 6), bf_off(prow, rr & 63), v);
      };
      if (ss < S_t) {
        const int rb = ss * K;
        float x = 0.f;
        for (int u = 0; u < K; ++u) {  // B_t is replaced by x_t
          x = fmaf(gsc * sigmoid_fast(ab(rb + u, sd)), x, ab(rb + u, kD + sd));
          ab(rb + u, kD + sd) = x;
        }
        sDC[ss * kD + sd] = dctx * x;
        sCtx[ss * kD + sd] = cv * x;
        float dx = dctx * cv;
        if ((K & 7) == 0) {
          // K a multiple of 8: a group of 8 steps is 8 consecutive tile rows
          // (16 bytes of a part row), written at once per part row
          const int prow[8] = {sd, kTD + sd, 2 * kTD + sd, 3 * kTD + sd,
                               kD + sd, kTD + kD + sd, 2 * kTD + kD + sd, 3 * kTD + kD + sd};
          for (int g = K / 8 - 1; g >= 0; --g) {
            uint32_t pk[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) pk[i][0] = pk[i][1] = pk[i][2] = pk[i][3] = 0u;
#pragma unroll
            for (int uu = 7; uu >= 0; --uu) {
              const int rr = rb + 8 * g + uu;
              float sg, dsg;
              sigmoid_and_slope(ab(rr, sd), sg, dsg);
              sg *= gsc;
              dsg *= gsc;
              const float xprev = (8 * g + uu) > 0 ? ab(rr - 1, kD + sd) : 0.f;
              const float dA = dx * xprev * dsg, dB = dx;
              dx *= sg;
              float v[8];
              bf_parts(dA, v[0], v[2], v[3]);
              bf_parts(dB, v[4], v[6], v[7]);
              v[1] = v[0];
              v[5] = v[4];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
                pk[i][uu >> 1] |= (uu & 1) ? b << 16 : b;
              }
            }
            const int r0 = rb + 8 * g;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(sT + kHBox * (r0 >> 6) + bf_off(prow[i], r0 & 63)) =
                  make_uint4(pk[i][0], pk[i][1], pk[i][2], pk[i][3]);
          }
        } else {
          for (int u = K - 1; u >= 0; --u) {
            const int rr = rb + u;
            float sg, dsg;
            sigmoid_and_slope(ab(rr, sd), sg, dsg);
            sg *= gsc;
            dsg *= gsc;
            const float xprev = u > 0 ? ab(rr - 1, kD + sd) : 0.f;
            const float dA = dx * xprev * dsg, dB = dx;
            dx *= sg;
            float p0, p1, p2;
            bf_parts(dA, p0, p1, p2);
            put_t(sd, rr, p0);
            put_t(kTD + sd, rr, p0);
            put_t(2 * kTD + sd, rr, p1);
            put_t(3 * kTD + sd, rr, p2);
            bf_parts(dB, p0, p1, p2);
            put_t(kD + sd, rr, p0);
            put_t(kTD + kD + sd, rr, p0);
            put_t(2 * kTD + kD + sd, rr, p1);
            put_t(3 * kTD + kD + sd, rr, p2);
          }
        }
      }
      if (R_t < 128) {  // rows past the tile: zero (the dW products read them)
        for (int e = tid; e < 128 * (128 - R_t); e += kCT) {
          const int prow = e & 127, rr = R_t + (e >> 7);
          put_t(prow, rr, 0.f);
        }
      }
      fence_proxy_async_smem();
      named_sync(1, kCT);
      if (lane == 0) mbar_arrive(&bb->t_ready);
      // ===== items per block: dW_C, dW_O partial sums and d_h_s2 (thread =
      // column jj of the block x state quad / sample quad cq)
#pragma unroll
      for (int q = 0; q < kMaxNB; ++q) {
        if (q >= NB) break;
        bounded_wait(&bb->full[r.i], r.ph, a.err);
        const unsigned char* sp = base + kOffRing + r.i * kStageB;
        const unsigned char* hs = sp + kHBox;
        const unsigned char* gs = hs + 2048;
        const int j = kBlk * q + jj;
#pragma unroll 4
        for (int s = 0; s < S_t; ++s) {
          const float hv = bfv(hs, bf_off(s, jj)), g = bfv(gs, bf_off(s, jj));
          const float4 dc = lds4(sDC + s * kD + 4 * cq), cx = lds4(sCtx + s * kD + 4 * cq);
          wcacc[q][0] = fmaf(hv, dc.x, wcacc[q][0]);
          wcacc[q][1] = fmaf(hv, dc.y, wcacc[q][1]);
          wcacc[q][2] = fmaf(hv, dc.z, wcacc[q][2]);
          wcacc[q][3] = fmaf(hv, dc.w, wcacc[q][3]);
          woacc[q][0] = fmaf(g, cx.x, woacc[q][0]);
          woacc[q][1] = fmaf(g, cx.y, woacc[q][1]);
          woacc[q][2] = fmaf(g, cx.z, woacc[q][2]);
          woacc[q][3] = fmaf(g, cx.w, woacc[q][3]);
        }
        {
          float wcj[kD];
#pragma unroll
          for (int c = 0; c < kD; ++c) wcj[c] = sWct[c * SH2P + j];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int s = 4 * cq + i;
            if (s < S_t) {
              float o = bfv(gs, bf_off(s, jj));
#pragma unroll
              for (int c4 = 0; c4 < kD / 4; ++c4) {
                const float4 dc = lds4(sDC + s * kD + 4 * c4);
                o = fmaf(dc.x, wcj[4 * c4], o);
                o = fmaf(dc.y, wcj[4 * c4 + 1], o);
                o = fmaf(dc.z, wcj[4 * c4 + 2], o);
                o = fmaf(dc.w, wcj[4 * c4 + 3], o);
              }
              reinterpret_cast<__nv_bfloat16*>(a.out1)[(tb0 + s) * SH2 + j] = __float2bfloat16_rn(o);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb->empty[r.i]);
        r.next();
      }
      // ============== d_h_history rows: TMEM -> bf16 -> global memory
      bounded_wait(&bb->dh_full, t & 1, a.err);
      tc_fence_after();
      {
        const int half = SH2 / 2;
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.out0) + (row0 + row) * SH2 + half * hsel;
        for (int c0 = 0; c0 < half; c0 += 16) {
          float v[16];
          tmem_ld<16>(lane_base + half * hsel + c0, v);
          if (row < R_t) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
              w[i] = *reinterpret_cast<const uint32_t*>(&p);
            }
            *reinterpret_cast<uint4*>(dst + c0) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(dst + c0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bb->dh_free);
      named_sync(1, kCT);  // sAB, sDC, sCtx are reused by the next tile
    }
    // ================================ partial sums into the CTA's slot
    float* slot = a.ws + static_cast<size_t>(cta) * 4 * SH2 * kD;
    const int n = SH2 * kD;
#pragma unroll
    for (int q = 0; q < kMaxNB; ++q) {
      if (q >= NB) break;
      const int j = kBlk * q + jj;
      *reinterpret_cast<float4*>(slot + 2 * n + j * kD + 4 * cq) =
          make_float4(wcacc[q][0], wcacc[q][1], wcacc[q][2], wcacc[q][3]);
#pragma unroll
      for (int e = 0; e < 4; ++e) slot[3 * n + (4 * cq + e) * SH2 + j] = a.tw * woacc[q][e];
    }
    // dW_A|dW_B: part rows a0 (lanes 0-31), a1 (64-95) and a2 (96-127) added
    // per 64-column block, through the (now idle) copy ring
    bounded_wait(&bb->dw_done, 0, a.err);
    tc_fence_after();
    float* red = reinterpret_cast<float*>(base + kOffRing);  // [3][32][64]
    for (int q = 0; q < NB; ++q) {
      if (hsel == 0 && q4 != 1) {
        const int pi = q4 == 0 ? 0 : q4 - 1;
#pragma unroll
        for (int c0 = 0; c0 < kBlk; c0 += 16) {
          float v[16];
          tmem_ld<16>(lane_base + kColDW + kBlk * q + c0, v);
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            sts4(red + (pi * 32 + lane) * kBlk + c0 + i, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
        }
      }
      named_sync(1, kCT);
      for (int e = tid; e < kTD * kBlk; e += kCT) {
        const int c = e / kBlk, jb = e % kBlk, j = kBlk * q + jb;
        const float v = (red[c * kBlk + jb] + red[(32 + c) * kBlk + jb]) + red[(64 + c) * kBlk + jb];
        slot[(c < kD ? 0 : n) + j * kD + (c & (kD - 1))] = v;
      }
      named_sync(1, kCT);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) signal_dependent_launch();
  if (warp == kMma) tmem_dealloc(tmem, 512);
}

}  // namespace

bool bwd_bf16_tc_plan(int64_t B, int K, int SH2, int D, FastArgs* a) {
  if (D != kD || SH2 < kBlk || SH2 % kBlk != 0 || SH2 > kMaxNB * kBlk || K < 1 || K > 128) return false;
  if (B * K >= (1ll << 31)) return false;
  int S_max = 128 / K;
  if (S_max > 16) S_max = 16;
  a->S_max = S_max;
  a->K = K;
  a->SH2 = SH2;
  a->smem_bytes = static_cast<int>(kSmemB);
  return kSmemB <= 227u * 1024u;
}

cudaError_t launch_bwd_bf16_tc(const FastArgs& a, int grid, cudaStream_t stream) {
  bwd_bf16_tc_kernel<<<grid, kThreadsB, kSmemB, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t prepare_bwd_bf16_kernels() {
  return cudaFuncSetAttribute(bwd_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kSmemB));
}

}  // namespace m2scan
