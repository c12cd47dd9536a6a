// Backward of the gated temporal scan layer with its three large contractions
// on the tensor cores, warp-specialised (D = 16, SH2 % 32 == 0, SH2 <= 256,
// K <= 128; D = 4 and 8 run with their states zero-padded to 16).
//
// One persistent CTA per weight-gradient slot walks its samples in tiles of at
// most 128 rows (S samples x K). Per tile:
//   pass 1   the producer warp streams 32-column chunks of h_history, h_s2 and
//            d_h_enriched (TMA boxes, 128-byte swizzle). The MMA warp
//            recomputes A|B = h . [W_A|W_B] with the chunk as the A operand
//            straight from shared memory (the tensor core reads the top 19 bits
//            of each fp32, i.e. trunc(h)); meanwhile the compute warps write
//            h - trunc(h) into tensor memory and a second MMA thread adds that
//            remainder's product. Each thread commits once per chunk (a commit
//            stalls only the issuing thread's MMA stream, so the two overlap):
//            the main commit and the remainder thread's arrival free the
//            chunk's stage, the remainder commit its TMEM buffer. The compute
//            warps also form C = h_s2 . W_C and d_ctx = tw dY . W_O^T on the
//            FMA pipe.
//   scan     replay of the forward scan and the reverse scan of the
//            implementation plan's Task 2 ("Custom Kernel Optimization
//            Implementation Plan"): dB_t = dx, dA_t = dx x_{t-1} sigmoid'(A_t),
//            dx <- dx sigmoid(A_t). dA|dB is stored split into a tf32 part
//            and the remainder, row-major (B operand of d_h); each 16-row
//            item copies its rows transposed (B operand of dW_A|dW_B).
//   d_h      d_h_history^T[j, row] = [W_A|W_B][j, :] . dA|dB[row, :] per
//            64-row half of the tile, 3 x tf32, the weights (split the same
//            way) held in tensor memory as the A operand.
//   per row  the producer streams the tile's h_history rows again, 16 at a
//            time; the compute warps write them transposed into tensor memory
//            (h and h - trunc(h)) and the MMA warp accumulates
//            dW_A|dW_B^T += h^T . dA|dB over every tile of the CTA. The same
//            stage then carries the 16 rows of d_h_history out: the producer
//            warp issues that bulk copy before it reuses the stage, so the
//            output stream is spread over the tile and the compute warps
//            never wait for it.
//   per sample dW_C, dW_O partial sums and d_h_s2 = dY + dC . W_C^T (FMA pipe).
// The weight-gradient partial sums are written once to the CTA's workspace
// slot; the slot reduction adds the slots in a fixed order.
#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kBwdThreads = kComputeThreads + 96;
constexpr int kProducerWarp = kComputeWarps;
constexpr int kMmaWarp = kComputeWarps + 1;   // projections trunc(h) . [W_hi | W_lo], d_h, dW
constexpr int kCorrWarp = kComputeWarps + 2;  // projection remainders (h - trunc h) . W_hi
constexpr int kRowItem = 16;       // h_history rows per dW item
constexpr int kBwdSampleItem = 8;  // samples per dW_C/dW_O/d_h_s2 item
constexpr int kChunkRing = 6;      // chunk hand-off barriers (>= the copy ring's depth)
// A chunk's stage is free once its main products are done and the compute
// warps have read it (cempty); a sample or row item's stage once the compute
// warps arrive on empty.
constexpr int kLoBufs = 3;  // TMEM buffers of h - trunc(h) for the projections

struct BwdBars {
  uint64_t full[kMaxStages];          // producer -> all: stage loaded
  uint64_t empty[kMaxStages];         // compute -> producer: sample / row item in stage s released (one arrival per warp)
  uint64_t cempty[kMaxStages];        // chunk in stage s released: main products done (commit) + compute read (arrive)
  uint64_t loready[kChunkRing];       // compute -> remainder MMA thread: chunk c read, h - trunc(h) in TMEM
  uint64_t lofree[kLoBufs];           // remainder MMA thread -> all: remainder buffer's products done
  uint64_t mdone;              // main MMA thread -> compute: the tile's main projection products done
  uint64_t bready;             // compute -> MMA: dA|dB operands written
  uint64_t dhready[2];         // MMA -> compute: d_h of a 64-row half done
  uint64_t dhfree[2];          // compute -> MMA: that d_h read back
  uint64_t htready[2];         // compute -> MMA: transposed rows in TMEM
  uint64_t htfree[2];          // MMA -> compute: transposed rows consumed
  uint64_t dwdone;             // MMA -> compute: every dW MMA done
  uint32_t tslot;
  uint32_t pad;
};

// TMEM columns (128 lanes each):
//   [0, 128)    projection accumulators trunc(h) . [W_hi | W_lo] of the even
//               and of the odd chunks (64 columns each); later d_h^T of one
//               64-row half: j-half h at 64 h (N = 64 rows)
//   [128, 224)  during the projections: three buffers of h - trunc(h) for a
//               chunk (A operand, 32 columns each)
//   [224, 256)  during the projections: (h - trunc h) . W_hi, a sum of its own
//               so that no accumulation order depends on timing
//   [128, 256)  during the row items: transposed h rows, two buffers p of
//               [j-half 0 | j-half 1], each 16 columns of h then 16 of
//               h - trunc(h)
//   [256, 384)  dW_A|dW_B^T accumulators: j-half h at 256 + 64 h,
//               [h . dAB_hi (32) | h . dAB_lo + (h - trunc h) . dAB_hi (32)]
//   [384, 512)  [W_A|W_B] rows as the d_h A operand: j-half h at 384 + 64 h,
//               32 columns tf32 part, 32 columns remainder
constexpr uint32_t kColCorr = 224;
constexpr uint32_t kColLo = 128;
constexpr uint32_t kColHT = 128;
constexpr uint32_t kColDW = 256;
constexpr uint32_t kColW = 384;

// Position in a ring of n barriers: index and the parity of its current use.
struct RingPos {
  int i = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

// Order of a tile's items after its NC chunks: sample item 0, row items 0-3,
// the other sample items, then row items 4 on. While the compute warps work
// on a sample item the MMA warp computes the next half of d_h.
// kind 1: sample item idx, kind 2: row item idx.
__device__ __forceinline__ void post_item(int p, int NSI, int NRI, int& kind, int& idx) {
  if (NSI > 0) {
    if (p == 0) {
      kind = 1;
      idx = 0;
      return;
    }
    --p;
  }
  const int r1 = NRI < 4 ? NRI : 4;
  if (p < r1) {
    kind = 2;
    idx = p;
    return;
  }
  p -= r1;
  const int s1 = NSI > 0 ? NSI - 1 : 0;
  if (p < s1) {
    kind = 1;
    idx = 1 + p;
    return;
  }
  kind = 2;
  idx = 4 + (p - s1);
}

// DR: the layer's states (4, 8 or 16; a compile-time constant, so that the
// D = 16 kernel is exactly the unpadded one).
template <int DR>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_tc_kernel(const __grid_constant__ FastArgs a) {
  constexpr int D = 16, TD = 32, FD = 64;  // states inside the kernel
  constexpr int Dr = DR;  // the layer's states; the others have zero weights
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  float* sW = reinterpret_cast<float*>(base + a.off_wt);       // NC tiles [FD][32], swizzled
  float* sW_Ct = reinterpret_cast<float*>(base + a.off_wct);   // W_C transposed [D][SH2]
  float* sPh = reinterpret_cast<float*>(base + a.off_p);       // A|B, then dA|dB tf32 part [128][32] swizzled
  float* sPl = reinterpret_cast<float*>(base + a.off_hlo);     // dA|dB remainder, same layout
  float* sDT = reinterpret_cast<float*>(base + a.off_wab);     // dA|dB^T [hi 32 | lo 32][2 x 16 rows], swizzled
  float* sC = reinterpret_cast<float*>(base + a.off_cs);       // C [S_max][D]
  float* sCtx = reinterpret_cast<float*>(base + a.off_ctx);    // ctx [S_max][D]
  float* sDctx = reinterpret_cast<float*>(base + a.off_dctx);  // d_ctx [S_max][D]
  float* sDC = reinterpret_cast<float*>(base + a.off_dc);      // dC [S_max][D]
  BwdBars* bb = reinterpret_cast<BwdBars*>(base + a.off_bar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int trace_n = 0;
  (void)trace_n;
  if (tid == 0) TRACE_AT(0, 1);
  if (tid == 0) TRACE_CTA(0);
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max, NST = a.n_stages;
  const uint32_t stage_bytes = static_cast<uint32_t>(a.stage_bytes);
  const int NC = SH2 / kChunk;
  const long long B = a.B;
  const int P = gridDim.x, cta = blockIdx.x;
  const long long cb0 = B * cta / P;
  const int n_c = static_cast<int>(B * (cta + 1) / P - cb0);
  const int T = (n_c + S_max - 1) / S_max;
  const int t_base = n_c / T, t_extra = n_c - (n_c / T) * T;
  auto tile_start = [&](int i) -> long long {
    return cb0 + static_cast<long long>(i) * t_base + (i < t_extra ? i : t_extra);
  };
  auto n_sample_items = [&](int S_t) { return (S_t + kBwdSampleItem - 1) / kBwdSampleItem; };
  auto n_row_items = [&](int S_t) { return (S_t * K + kRowItem - 1) / kRowItem; };
  auto stage_ptr = [&](int st) { return base + static_cast<uint32_t>(st) * stage_bytes; };

  if (tid == kProducerWarp * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_hs)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_g)) : "memory");
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bb->full[s], 1);
      mbar_init(&bb->empty[s], kComputeWarps);
      mbar_init(&bb->cempty[s], 2);
    }
    for (int s = 0; s < kChunkRing; ++s) mbar_init(&bb->loready[s], kComputeWarps);
    for (int s = 0; s < kLoBufs; ++s) mbar_init(&bb->lofree[s], 1);
    mbar_init(&bb->mdone, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bb->dhready[s], 1);
      mbar_init(&bb->dhfree[s], kComputeWarps);
      mbar_init(&bb->htready[s], kComputeWarps);
      mbar_init(&bb->htfree[s], 1);
    }
    mbar_init(&bb->bready, 1);
    mbar_init(&bb->dwdone, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&bb->tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bb->tslot;
  if (tid == 0) TRACE_AT(0, 3);

  // ---- producer: per tile NC chunks, then the other items (post_item order).
  // A stage that held a sample or row item holds that item's output once the
  // compute warps release it: the producer stores it before reusing the stage.
  RingPos lp, rp;                  // next stage to load, oldest stage not yet released
  uint32_t eph = 0;                // bit s: parity of the next empty[s] phase
  uint32_t cph = 0;                // bit s: parity of the next cempty[s] phase
  int pn = 0, ptile = 0, pit = 0;  // items loaded; tile and item of the next load
  int rn = 0, rtile = 0, rit = 0;  // items released; tile and item of the next release
  auto release_one = [&]() {
    if (rit < NC) {
      bounded_wait(&bb->cempty[rp.i], (cph >> rp.i) & 1u, a.err);
      cph ^= 1u << rp.i;
    } else {
      bounded_wait(&bb->empty[rp.i], (eph >> rp.i) & 1u, a.err);
      eph ^= 1u << rp.i;
    }
    const long long tb0 = tile_start(rtile);
    const int S_t = static_cast<int>(tile_start(rtile + 1) - tb0);
    const int NSI = n_sample_items(S_t), NRI = n_row_items(S_t);
    if (rit >= NC) {
      const unsigned char* sp = stage_ptr(rp.i);
      int kind, idx;
      post_item(rit - NC, NSI, NRI, kind, idx);
      if (kind == 1) {
        const int s0 = idx * kBwdSampleItem;
        const int ns = min(kBwdSampleItem, S_t - s0);
        bulk_store(a.out1 + (tb0 + s0) * SH2, sp, static_cast<uint32_t>(ns) * SH2 * 4u);
      } else {
        const int r0 = idx * kRowItem;
        const int nr = min(kRowItem, S_t * K - r0);
        bulk_store(a.out0 + (tb0 * K + r0) * SH2, sp, static_cast<uint32_t>(nr) * SH2 * 4u);
      }
      bulk_commit();
      bulk_wait_read_all();
    }
    rp.next(NST);
    ++rn;
    if (++rit == NC + NSI + NRI) {
      rit = 0;
      ++rtile;
    }
  };
  auto produce_one = [&]() {
    const long long tb0 = tile_start(ptile);
    const int S_t = static_cast<int>(tile_start(ptile + 1) - tb0);
    const int NSI = n_sample_items(S_t), NRI = n_row_items(S_t);
    if (pn >= NST) release_one();
    unsigned char* sp = stage_ptr(lp.i);
    uint64_t* bar = &bb->full[lp.i];
    int kind = 0, idx = pit;
    if (pit >= NC) post_item(pit - NC, NSI, NRI, kind, idx);
    if (kind == 0) {
      mbar_arrive_expect_tx(bar, a.hc_bytes + 2 * a.sc_bytes);
      tma_load_3d(sp, &a.tm_h, pit * kChunk, 0, static_cast<int>(tb0), bar);
      tma_load_2d(sp + a.off_S, &a.tm_hs, pit * kChunk, static_cast<int>(tb0), bar);
      tma_load_2d(sp + a.off_G, &a.tm_g, pit * kChunk, static_cast<int>(tb0), bar);
    } else if (kind == 1) {
      const int s0 = idx * kBwdSampleItem;
      const int ns = min(kBwdSampleItem, S_t - s0);
      const uint32_t rb = static_cast<uint32_t>(ns) * SH2 * 4u;
      mbar_arrive_expect_tx(bar, 2u * rb);
      bulk_load(sp, a.h_s2 + (tb0 + s0) * SH2, rb, bar);
      bulk_load(sp + static_cast<size_t>(kBwdSampleItem) * SH2 * 4, a.g + (tb0 + s0) * SH2, rb, bar);
    } else {
      const int r0 = idx * kRowItem;
      const int nr = min(kRowItem, S_t * K - r0);
      const uint32_t rb = static_cast<uint32_t>(nr) * SH2 * 4u;
      mbar_arrive_expect_tx(bar, rb);
      bulk_load(sp, a.h_history + (tb0 * K + r0) * SH2, rb, bar);
    }
    lp.next(NST);
    ++pn;
    if (++pit == NC + NSI + NRI) {
      pit = 0;
      ++ptile;
    }
  };

  // ---- weights: compute thread = row j of W_A, W_B, W_C (j < SH2 <= 256):
  // [W_A|W_B] row j into TMEM, the projection B tiles and W_C^T into shared
  // memory; the 32 threads of a warp hold 32 consecutive rows, so every
  // transposed or swizzled store of a warp lands in one 128-byte row (no bank
  // conflicts). Every global load is issued before the first store.
  {
    const int wh = warp >> 2;  // j-half of this compute warp's TMEM rows
    const int wj = 128 * wh + 32 * (warp & 3) + lane;
    const bool wok = warp < kComputeWarps && wj < SH2;
    float4 wr[8], wcr[4];
    if (warp < kComputeWarps) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float* src = (q < 4 ? a.W_A : a.W_B) + wj * Dr + 4 * (q & 3);
        wr[q] = wok && 4 * (q & 3) < Dr ? __ldg(reinterpret_cast<const float4*>(src)) : z;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        wcr[q] = wok && 4 * q < Dr ? __ldg(reinterpret_cast<const float4*>(a.W_C + wj * Dr + 4 * q)) : z;
    }
    // the first stages are requested after the weights, so that the weight
    // loads are not queued behind them
    if (warp == kProducerWarp && lane == 0)
      for (int i = 0; i < NST && ptile < T; ++i) produce_one();
    if (warp < kComputeWarps) {
      // thread = TMEM lane = row j of [W_A|W_B] within its j-half
      float hi[32], lo[32];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float v4[4] = {wr[q].x, wr[q].y, wr[q].z, wr[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hi[4 * q + e] = tf32_rn(v4[e]);
          lo[4 * q + e] = v4[e] - hi[4 * q + e];
        }
      }
      const uint32_t tw0 = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + kColW + 64u * wh;
      tmem_st16(tw0, hi);
      tmem_st16(tw0 + 16u, hi + 16);
      tmem_st16(tw0 + 32u, lo);
      tmem_st16(tw0 + 48u, lo + 16);
      if (wok) {
        float* tile = sW + (wj >> 5) * FD * 32;
        const int jj = wj & 31;
#pragma unroll
        for (int d = 0; d < D; ++d) {
          tile[sw128_idx(d, jj)] = hi[d];
          tile[sw128_idx(D + d, jj)] = hi[D + d];
          tile[sw128_idx(TD + d, jj)] = lo[d];
          tile[sw128_idx(TD + D + d, jj)] = lo[D + d];
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          sW_Ct[(4 * q) * SH2 + wj] = wcr[q].x;
          sW_Ct[(4 * q + 1) * SH2 + wj] = wcr[q].y;
          sW_Ct[(4 * q + 2) * SH2 + wj] = wcr[q].z;
          sW_Ct[(4 * q + 3) * SH2 + wj] = wcr[q].w;
        }
      }
      tmem_st_wait();
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) TRACE_AT(0, 2);
  if (tid == 0) TRACE_CTA(1);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      while (ptile < T) {
        TRACE_AT(1, 100 + pit);
        produce_one();
      }
      while (rn < pn) release_one();
      bulk_wait_all();
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc64 = umma_idesc_tf32(128, 64);
      constexpr uint32_t idesc32 = umma_idesc_tf32(128, 32);
      const uint32_t ph = smem_addr(sPh), pl = smem_addr(sPl), dt = smem_addr(sDT);
      const uint32_t ring = smem_addr(base);
      const uint32_t w0 = smem_addr(sW);
      // descriptor + 2 u advances its start address by 32 u bytes (one K step)
      auto issue_dh = [&](int rh) {
        // d_h^T[j, 64 rh + n] for both j-halves; cross terms first
        for (int h = 0; 128 * h < SH2; ++h) {
          const uint32_t dd = tmem + 64u * h, wh = tmem + kColW + 64u * h, wl = wh + 32u;
          const uint64_t bh0 = umma_desc_sw128(ph + 8192u * rh), bl0 = umma_desc_sw128(pl + 8192u * rh);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            umma_tf32_ta(dd, wh + 8u * ks, bl0 + 2u * ks, idesc64, ks != 0);
            umma_tf32_ta(dd, wl + 8u * ks, bh0 + 2u * ks, idesc64, 1u);
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) umma_tf32_ta(dd, wh + 8u * ks, bh0 + 2u * ks, idesc64, 1u);
        }
      };
      RingPos tp;  // stage of the tile's first item
      int ri = 0;
      bool dw_first = true;
      for (int t = 0; t < T; ++t) {
        const long long tb0 = tile_start(t);
        const int S_t = static_cast<int>(tile_start(t + 1) - tb0);
        const int NSI = n_sample_items(S_t), NRI = n_row_items(S_t);
        TRACE_AT(2, 290);
        // the previous tile's d_h has been read back (its dW MMAs, which read
        // the columns of the remainder products, were issued by this thread)
        if (t > 0) bounded_wait(&bb->dhfree[1], (t - 1) & 1, a.err);
        // pass 1: the main products of each chunk as it lands, in chunk order
        // into the even- or odd-chunk accumulator; a commit per chunk frees
        // the stage (with the remainder thread's arrival), one per tile hands
        // the main products to the compute warps
        {
          RingPos pm = tp;
          for (int qm = 0; qm < NC; ++qm) {
            bounded_wait(&bb->full[pm.i], pm.ph, a.err);
            tc_fence_after();
            const uint64_t ad = umma_desc_sw128(ring + static_cast<uint32_t>(pm.i) * stage_bytes);
            const uint64_t bd = umma_desc_sw128(w0 + static_cast<uint32_t>(qm * FD * 128));
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_tf32(tmem + 64u * (qm & 1), ad + 2u * ks, bd + 2u * ks, idesc64, (qm >= 2 || ks > 0) ? 1u : 0u);
            umma_commit(&bb->cempty[pm.i]);
            pm.next(NST);
          }
          umma_commit(&bb->mdone);
        }
        for (int i = 0; i < NC + NSI + NRI; ++i) tp.next(NST);
        TRACE_AT(2, 500);
        // d_h of rows [0, 64), then per 16 rows the dW MMAs; rows [64, 128)
        // once the first half has been read back
        bounded_wait(&bb->bready, t & 1, a.err);
        TRACE_AT(2, 600);
        tc_fence_after();
        issue_dh(0);
        umma_commit(&bb->dhready[0]);
        for (int k = 0; k < NRI; ++k, ++ri) {
          if (k == 4) {
            bounded_wait(&bb->dhfree[0], t & 1, a.err);
            tc_fence_after();
            issue_dh(1);
            umma_commit(&bb->dhready[1]);
          }
          bounded_wait(&bb->htready[ri & 1], (ri >> 1) & 1, a.err);
          tc_fence_after();
          const uint64_t bt = umma_desc_sw128(dt + 64u * (ri & 1));
          for (int h = 0; 128 * h < SH2; ++h) {
            const uint32_t araw = tmem + kColHT + 64u * (ri & 1) + 32u * h, alo = araw + 16u;
            const uint32_t dw = tmem + kColDW + 64u * h;
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              umma_tf32_ta(dw, araw + 8u * ks, bt + 2u * ks, idesc64, (dw_first && ks == 0) ? 0u : 1u);
              umma_tf32_ta(dw + TD, alo + 8u * ks, bt + 2u * ks, idesc32, 1u);
            }
          }
          dw_first = false;
          umma_commit(&bb->htfree[ri & 1]);
        }
        if (NRI <= 4) {
          bounded_wait(&bb->dhfree[0], t & 1, a.err);
          tc_fence_after();
          issue_dh(1);
          umma_commit(&bb->dhready[1]);
        }
        TRACE_AT(2, 601);
      }
      umma_commit(&bb->dwdone);
    }
  } else if (warp == kCorrWarp) {
    // ------------------------------------- MMA: projection remainders
    // (h - trunc h) . W_hi of each chunk once the compute warps have written
    // its remainder, into a sum of its own; a commit per chunk frees the
    // remainder buffer. These columns hold the previous tile's transposed
    // rows until its dW MMAs are done; the compute warps wait for that
    // before they hand over the tile's first remainder.
    if (lane == 0) {
      constexpr uint32_t idesc32 = umma_idesc_tf32(128, 32);
      const uint32_t w0 = smem_addr(sW);
      RingPos tp, lr, lf;
      for (int t = 0; t < T; ++t) {
        const int S_t = static_cast<int>(tile_start(t + 1) - tile_start(t));
        RingPos pc = tp;
        for (int qc = 0; qc < NC; ++qc) {
          bounded_wait(&bb->loready[lr.i], lr.ph, a.err);
          tc_fence_after();
          TRACE_AT(3, 400 + qc);
          mbar_arrive(&bb->cempty[pc.i]);  // the compute warps are done with the stage
          const uint32_t al = tmem + kColLo + 32u * lf.i;
          const uint64_t bd = umma_desc_sw128(w0 + static_cast<uint32_t>(qc * FD * 128));
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_tf32_ta(tmem + kColCorr, al + 8u * ks, bd + 2u * ks, idesc32, (qc > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bb->lofree[lf.i]);
          lr.next(kChunkRing);
          lf.next(kLoBufs);
          pc.next(NST);
        }
        for (int i = 0; i < NC + n_sample_items(S_t) + n_row_items(S_t); ++i) tp.next(NST);
      }
    }
  } else {
    // ------------------------------------------------------------- compute
    // 8 warps, two per TMEM lane quadrant: sub = 0 / 1 selects the half of a
    // row's columns (projections) or the j-half (transposed rows, d_h, dW).
    const int qd = warp & 3, sub = warp >> 2;
    const int row = 32 * qd + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    const float gsc = load_gate_scale(a.gate_scale);
    // C / d_ctx partial dots: thread = (role, state, column quad), all 16
    // samples of a tile; role 0 sums h_s2 . W_C, role 1 dY . W_O^T
    const int sd_jq = tid & 7, sd_d = (tid >> 3) & 15, sd_role = tid >> 7;
    const int sd_box = sd_role == 0 ? a.off_S : a.off_G;  // bytes from the stage
    // (a padded state's W_O row is zero: it is not read)
    const bool sd_wok = sd_role == 0 || sd_d < Dr;
    const float* sd_w = sd_role == 0 ? sW_Ct + sd_d * SH2 + 4 * sd_jq : a.W_O + (sd_wok ? sd_d : 0) * SH2 + 4 * sd_jq;
    // h of this thread in a chunk: its row, columns 16 sub .. 16 sub + 15
    int lo_off[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) lo_off[v] = row * 32 + (((4 * sub + v) ^ (row & 7)) << 2);
    // dW_C (role 0: h_s2 x dC) or dW_O (role 1: dY x ctx): rows 4 jq .. 4 jq + 3
    // x states 8 dh .. 8 dh + 7
    const int cw_role = tid >> 7, cw_jq = tid & 63, cw_dh = (tid >> 6) & 1;
    const bool cw_own = 4 * cw_jq < SH2;
    float cacc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) cacc[i][e] = 0.f;
    // transposed rows and d_h: thread = row j of SH2 (TMEM lane), 16 rows
    const int jrow = 128 * sub + row;
    const bool jok = jrow < SH2;
    RingPos ip;  // stage of the next item
    RingPos lr;  // loready position of the next chunk
    RingPos lf;  // remainder buffer of the next chunk
    int c = 0, ri = 0;
    for (int t = 0; t < T; ++t) {
      const long long tb0 = tile_start(t);
      const int S_t = static_cast<int>(tile_start(t + 1) - tb0);
      const int R_t = S_t * K;
      const int NSI = n_sample_items(S_t), NRI = n_row_items(S_t);
      float sacc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) sacc[i] = 0.f;
      // the remainder buffers share TMEM with the previous tile's transposed
      // rows: wait until the dW MMAs of its last two row items are done
      if (ri >= 1) bounded_wait(&bb->htfree[(ri - 1) & 1], ((ri - 1) >> 1) & 1, a.err);
      if (ri >= 2) bounded_wait(&bb->htfree[ri & 1], ((ri - 2) >> 1) & 1, a.err);
      // ====================================================== pass 1 chunks
      // Per chunk: h - trunc(h) into its TMEM buffer; the C / d_ctx dots run
      // while that store lands, and the chunk is handed to the remainder MMA
      // thread at the top of the next iteration (or after the last one).
      RingPos lr_prev = lr;
      for (int q = 0; q < NC; ++q, ++c) {
        const float4 w = sd_role == 0 ? lds4(sd_w + q * kChunk)
                         : sd_wok   ? __ldg(reinterpret_cast<const float4*>(sd_w + q * kChunk))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        if (tid == 0) TRACE_AT(0, 10);
        bounded_wait(&bb->full[ip.i], ip.ph, a.err);
        if (tid == 0) TRACE_AT(0, 11);
        const unsigned char* sp = stage_ptr(ip.i);
        const float* Hc = reinterpret_cast<const float*>(sp);
        float lo[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 x = lds4(Hc + lo_off[v]);
          lo[4 * v] = x.x - tf32_trunc(x.x);
          lo[4 * v + 1] = x.y - tf32_trunc(x.y);
          lo[4 * v + 2] = x.z - tf32_trunc(x.z);
          lo[4 * v + 3] = x.w - tf32_trunc(x.w);
        }
        if (q > 0) {  // the previous chunk's remainder has landed: hand it over
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bb->loready[lr_prev.i]);
          lr_prev = lr;
        }
        // the buffer's previous chunk c - 3 is done
        if (c >= kLoBufs) bounded_wait(&bb->lofree[lf.i], lf.ph ^ 1u, a.err);
        tc_fence_after();
        tmem_st16(lane_base + kColLo + 32u * lf.i + 16u * sub, lo);
        lr.next(kChunkRing);
        lf.next(kLoBufs);
        {
          // all 16 rows of the box even past S_max: the reads stay inside
          // shared memory and the sums of missing samples are never stored
          const float* bp = reinterpret_cast<const float*>(sp + sd_box);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 v = lds4(bp + i * 32 + ((sd_jq ^ (i & 7)) << 2));
            float x = sacc[i];
            x = fmaf(v.x, w.x, x); x = fmaf(v.y, w.y, x); x = fmaf(v.z, w.z, x); x = fmaf(v.w, w.w, x);
            sacc[i] = x;
          }
        }
        ip.next(NST);
        if (tid == 0) TRACE_AT(0, 13);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bb->loready[lr_prev.i]);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) sacc[i] += __shfl_xor_sync(0xffffffffu, sacc[i], m);
      }
      if (sd_jq == 0) {
        float* dst = sd_role == 0 ? sC : sDctx;
        const float scale = sd_role == 0 ? 1.f : a.tw;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < S_t) dst[i * D + sd_d] = scale * sacc[i];
      }
      // ==================================== projections: TMEM -> shared memory
      if (tid == 0) TRACE_AT(0, 20);
      // the tile's main products and the remainder products of its last chunk
      bounded_wait(&bb->mdone, t & 1, a.err);
      bounded_wait(&bb->lofree[(c - 1) % kLoBufs], ((c - 1) / kLoBufs) & 1, a.err);
      if (tid == 0) TRACE_AT(0, 21);
      tc_fence_after();
      {
        const int c0 = 16 * sub;  // columns c0 .. c0 + 15 of A|B
        uint32_t r0[16], r1[16], r2[16], r3[16], r4[16];
        tmem_ld16_nowait(lane_base + c0, r0);
        tmem_ld16_nowait(lane_base + TD + c0, r1);
        tmem_ld16_nowait(lane_base + 64u + c0, r2);
        tmem_ld16_nowait(lane_base + 64u + TD + c0, r3);
        tmem_ld16_nowait(lane_base + kColCorr + c0, r4);
        tmem_ld_wait();
        const bool odd = NC > 1;  // the odd-chunk sum exists
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float m1 = odd ? __uint_as_float(r2[i]) : 0.f;
          const float c1 = odd ? __uint_as_float(r3[i]) : 0.f;
          v[i] = (__uint_as_float(r0[i]) + m1) + ((__uint_as_float(r1[i]) + c1) + __uint_as_float(r4[i]));
        }
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          sts4(sPh + sw128_idx(row, c0 + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
      }
      tc_fence_before();
      named_sync(1, kComputeThreads);
      if (tid == 0) TRACE_AT(0, 22);
      // ================================ scan and reverse scan per (sample, state)
      if (tid < S_t * D && (K & 7) == 0) {
        // K a multiple of 8: every group of 8 rows starts at a swizzle phase
        // of 0, so the offsets of this thread's two columns within a group
        // are the same for every group
        const int s = tid >> 4, d = tid & 15, rb = s * K;
        int oa[8], ob[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          oa[u] = u * 32 + ((((d >> 2)) ^ u) << 2) + (d & 3);
          ob[u] = u * 32 + (((4 + (d >> 2)) ^ u) << 2) + (d & 3);
        }
        float x = 0.f;
        for (int g = 0; g < K; g += 8) {  // replay: B_t is replaced by x_t
          float* pg = sPh + (rb + g) * 32;
          float av[8], bv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            av[u] = pg[oa[u]];
            bv[u] = pg[ob[u]];
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) av[u] = gsc * sigmoid_fast(av[u]);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            x = fmaf(av[u], x, bv[u]);
            pg[ob[u]] = x;
          }
        }
        const float Cv = sC[s * D + d], dctx = sDctx[s * D + d];
        sCtx[s * D + d] = Cv * x;
        sDC[s * D + d] = dctx * x;
        float dx = dctx * Cv;
        for (int g = K - 8; g >= 0; g -= 8) {
          float* pg = sPh + (rb + g) * 32;
          float* lg = sPl + (rb + g) * 32;
          float av[8], xp[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) av[u] = pg[oa[u]];
          xp[0] = g > 0 ? pg[ob[7] - 256] : 0.f;  // x of the last row of the previous group
#pragma unroll
          for (int u = 1; u < 8; ++u) xp[u] = pg[ob[u - 1]];
#pragma unroll
          for (int u = 7; u >= 0; --u) {
            float sg, dsg;
            sigmoid_and_slope(av[u], sg, dsg);
            sg *= gsc;
            dsg *= gsc;
            const float dB = dx, dA = dx * xp[u] * dsg;
            dx *= sg;
            const float ah = tf32_rn(dA), bh = tf32_rn(dB);
            pg[oa[u]] = ah;
            pg[ob[u]] = bh;
            lg[oa[u]] = dA - ah;
            lg[ob[u]] = dB - bh;
          }
        }
      } else if (tid < S_t * D) {
          const int s = tid >> 4, d = tid & 15, rb = s * K;
          float x = 0.f;
          for (int k0 = 0; k0 < K; k0 += 8) {  // replay: B_t is replaced by x_t
            const int n = min(8, K - k0);
            float av[8], bv[8];
  #pragma unroll
            for (int u = 0; u < 8; ++u)
              if (u < n) {
                av[u] = sPh[sw128_idx(rb + k0 + u, d)];
                bv[u] = sPh[sw128_idx(rb + k0 + u, D + d)];
              }
  #pragma unroll
            for (int u = 0; u < 8; ++u)
              if (u < n) av[u] = gsc * sigmoid_fast(av[u]);
  #pragma unroll
            for (int u = 0; u < 8; ++u)
              if (u < n) {
                x = fmaf(av[u], x, bv[u]);
                sPh[sw128_idx(rb + k0 + u, D + d)] = x;
              }
          }
          const float Cv = sC[s * D + d], dctx = sDctx[s * D + d];
          sCtx[s * D + d] = Cv * x;
          sDC[s * D + d] = dctx * x;
          float dx = dctx * Cv;
          for (int k1 = K; k1 > 0; k1 -= 8) {
            const int k0 = k1 > 8 ? k1 - 8 : 0, n = k1 - k0;
            float av[8], xp[8];
  #pragma unroll
            for (int u = 0; u < 8; ++u)
              if (u < n) {
                const int r = rb + k0 + u;
                av[u] = sPh[sw128_idx(r, d)];
                xp[u] = (k0 + u > 0) ? sPh[sw128_idx(r - 1, D + d)] : 0.f;
              }
  #pragma unroll
            for (int u = 7; u >= 0; --u)
              if (u < n) {
                const int r = rb + k0 + u;
                float sg, dsg;
                sigmoid_and_slope(av[u], sg, dsg);
                sg *= gsc;
                dsg *= gsc;
                const float dB = dx, dA = dx * xp[u] * dsg;
                dx *= sg;
                const float ah = tf32_rn(dA), bh = tf32_rn(dB);
                const float al = dA - ah, bl = dB - bh;
                sPh[sw128_idx(r, d)] = ah;
                sPh[sw128_idx(r, D + d)] = bh;
                sPl[sw128_idx(r, d)] = al;
                sPl[sw128_idx(r, D + d)] = bl;
              }
          }
      }
      fence_proxy_async_smem();
      named_sync(1, kComputeThreads);
      if (tid == 0) mbar_arrive(&bb->bready);
      if (tid == 0) TRACE_AT(0, 24);
      // ======= sample items (dW_C, dW_O partial sums, d_h_s2) and 16-row items
      // (h^T into TMEM for dW, d_h_history rows out), in post_item order
      for (int pi = 0; pi < NSI + NRI; ++pi) {
        int kind, k;
        post_item(pi, NSI, NRI, kind, k);
        bounded_wait(&bb->full[ip.i], ip.ph, a.err);
        float* stg = reinterpret_cast<float*>(stage_ptr(ip.i));
        const int st = ip.i;
        ip.next(NST);
        if (kind == 1) {
          if (tid == 0) TRACE_AT(0, 31);
          float* hsb = stg;
          const float* gb = hsb + static_cast<size_t>(kBwdSampleItem) * SH2;
          const int s0 = k * kBwdSampleItem, ns = min(kBwdSampleItem, S_t - s0);
          if (cw_own) {
            const float* rowp = (cw_role == 0 ? hsb : gb) + 4 * cw_jq;
            const float* vecp = (cw_role == 0 ? sDC : sCtx) + s0 * D + 8 * cw_dh;
            auto accumulate = [&](int s) {
              const float4 hv = lds4(rowp + s * SH2);
              const float4 v0 = lds4(vecp + s * D), v1 = lds4(vecp + s * D + 4);
              const float hvv[4] = {hv.x, hv.y, hv.z, hv.w};
              const float vvv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
              for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) cacc[i][e] = fmaf(hvv[i], vvv[e], cacc[i][e]);
            };
            if (ns == kBwdSampleItem) {
              // a full item: no per-sample condition, so the loads of later
              // samples can be issued ahead of the products of earlier ones
#pragma unroll
              for (int s = 0; s < kBwdSampleItem; ++s) accumulate(s);
            } else {
              for (int s = 0; s < ns; ++s) accumulate(s);
            }
          }
          named_sync(1, kComputeThreads);  // h_s2 rows no longer needed: d_h_s2 goes there
          {
            // two samples sq, sq + 4 per thread: each W_C^T element serves both
            const int jq = tid & 63, sq = tid >> 6;
            if (sq < ns && 4 * jq < SH2) {
              const bool two = sq + 4 < ns;
              float4 o0 = lds4(gb + sq * SH2 + 4 * jq);
              float4 o1 = two ? lds4(gb + (sq + 4) * SH2 + 4 * jq) : make_float4(0.f, 0.f, 0.f, 0.f);
              const float* dc0 = sDC + (s0 + sq) * D;
              const float* dc1 = sDC + (s0 + (two ? sq + 4 : sq)) * D;
#pragma unroll
              for (int dq = 0; dq < 4; ++dq) {
                const float4 a0 = lds4(dc0 + 4 * dq), a1 = lds4(dc1 + 4 * dq);
                const float d0[4] = {a0.x, a0.y, a0.z, a0.w}, d1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float4 wv = lds4(sW_Ct + (4 * dq + e) * SH2 + 4 * jq);
                  o0.x = fmaf(d0[e], wv.x, o0.x); o0.y = fmaf(d0[e], wv.y, o0.y);
                  o0.z = fmaf(d0[e], wv.z, o0.z); o0.w = fmaf(d0[e], wv.w, o0.w);
                  o1.x = fmaf(d1[e], wv.x, o1.x); o1.y = fmaf(d1[e], wv.y, o1.y);
                  o1.z = fmaf(d1[e], wv.z, o1.z); o1.w = fmaf(d1[e], wv.w, o1.w);
                }
              }
              sts4(hsb + sq * SH2 + 4 * jq, o0);
              if (two) sts4(hsb + (sq + 4) * SH2 + 4 * jq, o1);
            }
          }
          fence_proxy_async_smem();
          named_sync(1, kComputeThreads);
          if (tid == 0) {
            mbar_arrive(&bb->empty[st], kComputeWarps);  // the producer stores d_h_s2 from the stage
            TRACE_AT(0, 33);
          }
        } else {
          if (tid == 0) TRACE_AT(0, 41);
          float* hb = stg;
          const int r0 = k * kRowItem, nr = min(kRowItem, R_t - r0);
          const bool full_item = nr == kRowItem && jok;
          if (ri >= 2) bounded_wait(&bb->htfree[ri & 1], ((ri - 2) >> 1) & 1, a.err);
          tc_fence_after();
          {
            // this thread's column j of the 16 rows: h and h - trunc(h)
            float raw[16], lo[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
              const float x = (full_item || (r < nr && jok)) ? hb[r * SH2 + jrow] : 0.f;
              raw[r] = x;
              lo[r] = x - tf32_trunc(x);
            }
            const uint32_t tb = lane_base + kColHT + 64u * (ri & 1) + 32u * sub;
            tmem_st16(tb, raw);
            tmem_st16(tb + 16u, lo);
          }
          {  // dA|dB of these rows, transposed: [hi 32 | lo 32] x 16 rows; zero past the tile
            const int m = tid >> 2, rr = 4 * (tid & 3);
            const float* src = m < TD ? sPh : sPl;
            const int col = m & (TD - 1);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int r = rr + v;
              sDT[sw128_idx(m, 16 * (ri & 1) + r)] = r < nr ? src[sw128_idx(r0 + r, col)] : 0.f;
            }
          }
          tmem_st_wait();
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bb->htready[ri & 1]);
          const int rh = k >> 2;
          if ((k & 3) == 0) {
            if (tid == 0) TRACE_AT(0, 44);
            bounded_wait(&bb->dhready[rh], t & 1, a.err);
            if (tid == 0) TRACE_AT(0, 45);
          }
          tc_fence_after();
          {
            // each thread overwrites exactly the elements it read (column j
            // of the 16 rows), so no other thread's read is in the way
            float v[16];
            tmem_ld<16>(lane_base + 64u * sub + 16u * (k & 3), v);
            if (full_item) {
#pragma unroll
              for (int r = 0; r < 16; ++r) hb[r * SH2 + jrow] = v[r];
            } else {
#pragma unroll
              for (int r = 0; r < 16; ++r)
                if (r < nr && jok) hb[r * SH2 + jrow] = v[r];
            }
          }
          const bool last_of_half = (k & 3) == 3 || k == NRI - 1;
          tc_fence_before();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {  // per warp: its part of d_h read, its rows written
            if (last_of_half) mbar_arrive(&bb->dhfree[rh]);
            mbar_arrive(&bb->empty[st]);  // the producer stores the d_h rows from the stage
          }
          if (tid == 0) TRACE_AT(0, 42);
          ++ri;
        }
      }
      if (NRI <= 4 && lane == 0) mbar_arrive(&bb->dhfree[1]);
      if (tid == 0) TRACE_AT(0, 46);
    }
    // ===================================== partial sums into the CTA's slot
    // the slot holds the layer's Dr states: [4][SH2 * Dr]
    float* slot = a.ws + static_cast<size_t>(cta) * 4 * SH2 * Dr;
    const int n = SH2 * Dr;
    bounded_wait(&bb->dwdone, 0, a.err);
    tc_fence_after();
    {
      // row j of dW_A and dW_B: main sums (columns k) plus corrections (32 + k)
      float m[16], r[16];
#pragma unroll
      for (int cp = 0; cp < 2; ++cp) {
        tmem_ld<16>(lane_base + kColDW + 64u * sub + 16u * cp, m);
        tmem_ld<16>(lane_base + kColDW + 64u * sub + TD + 16u * cp, r);
        if (jok) {
          float4* dst = reinterpret_cast<float4*>(slot + cp * n + jrow * Dr);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (4 * i < Dr)
              dst[i] = make_float4(m[4 * i] + r[4 * i], m[4 * i + 1] + r[4 * i + 1], m[4 * i + 2] + r[4 * i + 2],
                                   m[4 * i + 3] + r[4 * i + 3]);
        }
      }
    }
    if (cw_own) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = 4 * cw_jq + i;
        if (cw_role == 0) {
          float4* dst = reinterpret_cast<float4*>(slot + 2 * n + j * Dr + 8 * cw_dh);
          if (8 * cw_dh < Dr) dst[0] = make_float4(cacc[i][0], cacc[i][1], cacc[i][2], cacc[i][3]);
          if (8 * cw_dh + 4 < Dr) dst[1] = make_float4(cacc[i][4], cacc[i][5], cacc[i][6], cacc[i][7]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (8 * cw_dh + e < Dr) slot[3 * n + (8 * cw_dh + e) * SH2 + j] = a.tw * cacc[i][e];
        }
      }
    }
    if (tid == 0) TRACE_AT(0, 50);
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0) signal_dependent_launch();
  if (tid == 0) TRACE_CTA(2);
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

int round_up_b(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

// D = 4 and 8 run the same kernel with 16 states, the others zero-padded
// (their weights read as zero, their gradients not written): every term they
// add is an exact zero.
bool bwd_tc_plan(int K, int SH2, int Dr, FastArgs* a) {
  if (!fast_path_ok(K, SH2, Dr)) return false;
  constexpr int D = 16;
  int S_max = kTileRows / K;
  if (S_max > 16) S_max = 16;  // the dots cover two halves of 8 samples, the scan 16 x D threads
  const int hc = S_max * K * 128, sc = S_max * 128;
  const int off_S = round_up_b(hc, 1024);
  const int off_G = off_S + round_up_b(sc, 1024);
  int stage = off_G + sc;
  if (2 * kBwdSampleItem * SH2 * 4 > stage) stage = 2 * kBwdSampleItem * SH2 * 4;
  if (kRowItem * SH2 * 4 > stage) stage = kRowItem * SH2 * 4;
  // the projection MMAs read 128 rows of 128 bytes from the start of a stage
  if (kTileRows * 128 > stage) stage = kTileRows * 128;
  stage = round_up_b(stage, 1024);
  const int wbytes = SH2 * 4 * D * 4;
  const int rest = wbytes + 2 * kTileRows * 128 + 64 * 32 * 4 + D * SH2 * 4 +
                   4 * S_max * D * 4 + static_cast<int>(sizeof(BwdBars)) + 16 + 1024;
  int n_stages = kMaxStages;
  while (n_stages > 2 && n_stages * stage + rest > 227 * 1024) --n_stages;
  int off = n_stages * stage;
  a->off_wt = off;   off += wbytes;
  a->off_p = off;    off += kTileRows * 128;
  a->off_hlo = off;  off += kTileRows * 128;
  a->off_wab = off;  off += 64 * 32 * 4;
  a->off_wct = off;  off += D * SH2 * 4;
  a->off_cs = off;   off += S_max * D * 4;
  a->off_ctx = off;  off += S_max * D * 4;
  a->off_dctx = off; off += S_max * D * 4;
  a->off_dc = off;   off += S_max * D * 4;
  off = round_up_b(off, 16);
  a->off_bar = off;  off += static_cast<int>(sizeof(BwdBars));
  a->smem_bytes = off + 1024;
  a->S_max = S_max;
  a->SG = kBwdSampleItem;
  a->stage_bytes = stage;
  a->hc_bytes = hc;
  a->sc_bytes = sc;
  a->off_S = off_S;
  a->off_G = off_G;
  a->K = K;
  a->SH2 = SH2;
  a->n_stages = n_stages;
  a->tc = 1;
  a->tmem_cols = 512;
  a->Dr = Dr;
  return a->smem_bytes <= 227 * 1024;
}

cudaError_t launch_bwd_tc(const FastArgs& a, int grid, cudaStream_t stream) {
  switch (a.Dr) {
    case 4: bwd_tc_kernel<4><<<grid, kBwdThreads, a.smem_bytes, stream>>>(a); break;
    case 8: bwd_tc_kernel<8><<<grid, kBwdThreads, a.smem_bytes, stream>>>(a); break;
    default: bwd_tc_kernel<16><<<grid, kBwdThreads, a.smem_bytes, stream>>>(a); break;
  }
  return cudaGetLastError();
}

cudaError_t prepare_bwd_tc_kernels(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  return e;
}

}  // namespace m2scan
