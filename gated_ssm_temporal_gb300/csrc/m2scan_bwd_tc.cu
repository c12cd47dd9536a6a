// Backward of the gated temporal scan layer with two of its three large
// contractions on the tensor cores, warp-specialised (D = 16, SH2 % 32 == 0,
// SH2 <= 256, K <= 128).
//
// Per tile of at most 128 rows (S samples x K) of one persistent CTA:
//   pass 1   (as in the forward) the producer warp streams 32-column chunks of
//            h_history, h_s2 and d_h_enriched; the compute warps split each h
//            row into tf32 hi/lo parts stored in TMEM; the MMA warp accumulates
//            A|B = h . [W_A|W_B] (3 x tf32); the compute warps also form
//            C = h_s2 . W_C and d_ctx = tw dY . W_O^T on the FMA pipe.
//   scan     replay of the forward scan and the reverse scan of the
//            implementation plan's Task 2 ("Custom Kernel Optimization
//            Implementation Plan"): dB_t = dx, dA_t = dx x_{t-1} sigmoid'(A_t),
//            dx <- dx sigmoid(A_t); dA|dB are left in shared memory split into a
//            tf32 part and an exact remainder (the MMA's B operand).
//   d_h      the MMA warp computes d_h_history transposed,
//            D[j, row] = [W_A|W_B][j, :] . dA|dB[row, :], A operand [W_A|W_B]
//            (hi/lo, kept in TMEM for the whole kernel), B operand dA|dB
//            (hi/lo), 3 x tf32; the compute warps read D back (thread = column
//            j, so each store instruction writes one contiguous row segment).
//   per row  dW_A|dW_B partial sums on the FMA pipe over the tile's rows,
//            streamed again as 16-row items (register accumulators).
//   per sample dW_C, dW_O partial sums and d_h_s2 = dY + dC . W_C^T.
// Weight-gradient partial sums are written once to the CTA's workspace slot;
// the slot reduction adds the slots in a fixed order.
#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kBwdThreads = kComputeThreads + 64;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kRowItem = 16;      // h_history rows per dW item
constexpr int kBwdSampleItem = 8;  // samples per dW_C/dW_O/d_h_s2 item

struct BwdBars {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t aready[2];
  uint64_t afree[2];
  uint64_t accfull;  // MMA -> compute: projections of the tile done
  uint64_t bready;   // compute -> MMA: dA|dB operand tiles written
  uint64_t bdone;    // MMA -> compute: d_h MMAs of the tile done
  uint64_t dhfree;   // compute -> MMA: d_h read back, TMEM [0, 256) free
  uint32_t tslot;
  uint32_t pad;
};

// TMEM columns: [0, 256) projection accumulators (4 pairs of [main | corrections],
// 64 columns each), later the transposed d_h (two 128-row halves of SH2);
// [256, 384) two A-operand buffers of the projection (32 hi + 32 lo);
// [384, 512) [W_A|W_B] as the d_h A operand: per half of SH2, 32 hi + 32 lo.
constexpr uint32_t kAcolA = 256;
constexpr uint32_t kWcol = 384;

__global__ void __launch_bounds__(kBwdThreads, 1) bwd_tc_kernel(const __grid_constant__ FastArgs a) {
  constexpr int D = 16, TD = 32, FD = 64;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  float* sW = reinterpret_cast<float*>(base + a.off_wt);      // NC tiles [FD][32], swizzled
  float* sW_Ct = reinterpret_cast<float*>(base + a.off_wct);  // W_C transposed [D][SH2]
  float* sW_O = reinterpret_cast<float*>(base + a.off_wo);    // W_O [D][SH2]
  float* sPh = reinterpret_cast<float*>(base + a.off_p);      // A|B, then dA|dB (tf32 part) [128][32] swizzled
  float* sPl = reinterpret_cast<float*>(base + a.off_hlo);    // dA|dB remainder, same layout
  float* sC = reinterpret_cast<float*>(base + a.off_cs);      // C [S_max][D]
  float* sCtx = reinterpret_cast<float*>(base + a.off_ctx);   // ctx [S_max][D]
  float* sDctx = reinterpret_cast<float*>(base + a.off_dctx); // d_ctx [S_max][D]
  float* sDC = reinterpret_cast<float*>(base + a.off_dc);     // dC [S_max][D]
  BwdBars* bb = reinterpret_cast<BwdBars*>(base + a.off_bar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int trace_n = 0;
  (void)trace_n;
  if (tid == 0) TRACE_AT(0, 1);
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max, NST = a.n_stages;
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

  if (tid == kProducerWarp * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_hs)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_g)) : "memory");
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bb->full[s], 1);
      mbar_init(&bb->empty[s], kComputeWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bb->aready[s], kComputeWarps);
      mbar_init(&bb->afree[s], 1);
    }
    mbar_init(&bb->accfull, 1);
    mbar_init(&bb->bready, 1);
    mbar_init(&bb->bdone, 1);
    mbar_init(&bb->dhfree, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&bb->tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bb->tslot;
  if (tid == 0) TRACE_AT(0, 3);

  // ---- producer state: items per tile are NC chunks, sample items, row items
  int pseq = 0, ptile = 0, pit = 0;
  auto produce_one = [&]() {
    const long long tb0 = tile_start(ptile);
    const int S_t = static_cast<int>(tile_start(ptile + 1) - tb0);
    const int NSI = n_sample_items(S_t), NRI = n_row_items(S_t);
    const int st = pseq % NST, use = pseq / NST;
    if (use > 0) bounded_wait(&bb->empty[st], (use - 1) & 1, a.err);
    unsigned char* sp = base + static_cast<size_t>(st) * a.stage_bytes;
    uint64_t* bar = &bb->full[st];
    if (pit < NC) {
      mbar_arrive_expect_tx(bar, a.hc_bytes + 2 * a.sc_bytes);
      tma_load_3d(sp, &a.tm_h, pit * kChunk, 0, static_cast<int>(tb0), bar);
      tma_load_2d(sp + a.off_S, &a.tm_hs, pit * kChunk, static_cast<int>(tb0), bar);
      tma_load_2d(sp + a.off_G, &a.tm_g, pit * kChunk, static_cast<int>(tb0), bar);
    } else if (pit < NC + NSI) {
      const int s0 = (pit - NC) * kBwdSampleItem;
      const int ns = min(kBwdSampleItem, S_t - s0);
      const uint32_t rb = static_cast<uint32_t>(ns) * SH2 * 4u;
      mbar_arrive_expect_tx(bar, 2u * rb);
      bulk_load(sp, a.h_s2 + (tb0 + s0) * SH2, rb, bar);
      bulk_load(sp + static_cast<size_t>(kBwdSampleItem) * SH2 * 4, a.g + (tb0 + s0) * SH2, rb, bar);
    } else {
      const int r0 = (pit - NC - NSI) * kRowItem;
      const int nr = min(kRowItem, S_t * K - r0);
      const uint32_t rb = static_cast<uint32_t>(nr) * SH2 * 4u;
      mbar_arrive_expect_tx(bar, rb);
      bulk_load(sp, a.h_history + (tb0 * K + r0) * SH2, rb, bar);
    }
    ++pseq;
    if (++pit == NC + NSI + NRI) {
      pit = 0;
      ++ptile;
    }
  };
  if (warp == kProducerWarp && lane == 0)
    for (int i = 0; i < NST && ptile < T; ++i) produce_one();

  // ---- weights: projection B tiles and W_C^T, W_O into shared memory;
  // [W_A|W_B] rows (hi/lo) into TMEM as the d_h A operand (compute warps)
  constexpr int kWPer = (4096 + kBwdThreads - 1) / kBwdThreads;
  {
    float wa[kWPer], wb[kWPer], wc[kWPer], wo[kWPer];
#pragma unroll
    for (int u = 0; u < kWPer; ++u) {
      const int i = tid + u * kBwdThreads;
      const bool ok = i < SH2 * D;
      wa[u] = ok ? __ldg(a.W_A + i) : 0.f;
      wb[u] = ok ? __ldg(a.W_B + i) : 0.f;
      wc[u] = ok ? __ldg(a.W_C + i) : 0.f;
      wo[u] = ok ? __ldg(a.W_O + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kWPer; ++u) {
      const int i = tid + u * kBwdThreads;
      if (i >= SH2 * D) break;
      const int j = i / D, d = i - (i / D) * D;
      float* tile = sW + (j >> 5) * FD * 32;
      const int jj = j & 31;
      const float ha = tf32_rna(wa[u]), hb = tf32_rna(wb[u]);
      tile[sw128_idx(d, jj)] = ha;
      tile[sw128_idx(D + d, jj)] = hb;
      tile[sw128_idx(TD + d, jj)] = wa[u] - ha;
      tile[sw128_idx(TD + D + d, jj)] = wb[u] - hb;
      sW_Ct[d * SH2 + j] = wc[u];
      sW_O[i] = wo[u];
    }
  }
  if (warp < kComputeWarps) {
    // thread = TMEM lane = row j of [W_A|W_B] within its half of SH2
    const int half = warp >> 2, j = 128 * half + 32 * (warp & 3) + lane;
    float hi[32], lo[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float w = j < SH2 ? __ldg((k < D ? a.W_A : a.W_B) + j * D + (k & (D - 1))) : 0.f;
      hi[k] = tf32_rna(w);
      lo[k] = w - hi[k];
    }
    const uint32_t tw0 = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + kWcol + 64u * half;
    tmem_st16(tw0, hi);
    tmem_st16(tw0 + 16u, hi + 16);
    tmem_st16(tw0 + 32u, lo);
    tmem_st16(tw0 + 48u, lo + 16);
    tmem_st_wait();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) TRACE_AT(0, 2);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0)
      while (ptile < T) {
        TRACE_AT(1, 100 + pit);
        produce_one();
      }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_f = umma_idesc_tf32(128, FD);
      constexpr uint32_t idesc_t = umma_idesc_tf32(128, TD);
      constexpr uint32_t idesc_d = umma_idesc_tf32(128, 128);
      const uint32_t ph = smem_addr(sPh), pl = smem_addr(sPl);
      int c = 0;
      for (int t = 0; t < T; ++t) {
        if (t > 0) bounded_wait(&bb->dhfree, (t - 1) & 1, a.err);
        TRACE_AT(2, 290);
        for (int q = 0; q < NC; ++q, ++c) {
          bounded_wait(&bb->aready[c & 1], (c >> 1) & 1, a.err);
          TRACE_AT(2, 400 + q);
          tc_fence_after();
          const uint32_t ah = tmem + kAcolA + 64u * (c & 1), al = ah + 32u;
          const uint32_t wt = smem_addr(sW + q * FD * 32);
          const uint32_t d_pair = tmem + static_cast<uint32_t>((q >> 1) * FD);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bdesc = umma_desc_sw128(wt + 32u * ks);
            umma_tf32_ta(d_pair, ah + 8u * ks, bdesc, idesc_f, ((q & 1) | ks) != 0);
            umma_tf32_ta(d_pair + TD, al + 8u * ks, bdesc, idesc_t, 1u);
          }
          umma_commit(&bb->afree[c & 1]);
        }
        umma_commit(&bb->accfull);
        TRACE_AT(2, 500);
        // d_h^T[j, row] = W[j, :] . dAB[row, :] per 128-row half of SH2
        bounded_wait(&bb->bready, t & 1, a.err);
        TRACE_AT(2, 600);
        tc_fence_after();
        for (int hh = 0; hh * 128 < SH2; ++hh) {
          const uint32_t dd = tmem + 128u * hh;
          const uint32_t wh = tmem + kWcol + 64u * hh, wl = wh + 32u;
          // the two small cross terms first, then the main products on top
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bh = umma_desc_sw128(ph + 32u * ks), bl = umma_desc_sw128(pl + 32u * ks);
            umma_tf32_ta(dd, wh + 8u * ks, bl, idesc_d, ks != 0);
            umma_tf32_ta(dd, wl + 8u * ks, bh, idesc_d, 1u);
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_tf32_ta(dd, wh + 8u * ks, umma_desc_sw128(ph + 32u * ks), idesc_d, 1u);
        }
        umma_commit(&bb->bdone);
        TRACE_AT(2, 601);
      }
    }
  } else {
    // ------------------------------------------------------------- compute
    const int row = 32 * (warp & 3) + lane, half = warp >> 2;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    const int sd_jo = tid & 3, sd_dq = (tid >> 2) & 3, sd_s = tid >> 4;  // D = 16: 4 state groups
    // weight-gradient ownership: dW_A|dW_B 4 rows x 8 columns, dW_C, dW_O 4 x 4
    const int pjq_ab = tid >> 2, pkq = tid & 3;
    const bool own_ab = pjq_ab < SH2 / 4;
    const int pjq_c = tid >> 2, pdq = tid & 3;
    const bool own_c = pjq_c < SH2 / 4;
    float accAB[4][8], accC[4][4], accO[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int e = 0; e < 8; ++e) accAB[i][e] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) accC[i][e] = accO[i][e] = 0.f;
    }
    int seq = 0, c = 0;
    for (int t = 0; t < T; ++t) {
      const long long tb0 = tile_start(t);
      const int S_t = static_cast<int>(tile_start(t + 1) - tb0);
      const int R_t = S_t * K;
      const int NSI = n_sample_items(S_t), NRI = n_row_items(S_t);
      const bool sd_active = sd_s < S_t;
      float cacc[4] = {0.f, 0.f, 0.f, 0.f}, dacc[4] = {0.f, 0.f, 0.f, 0.f};
      // ====================================================== pass 1 chunks
      for (int q = 0; q < NC; ++q, ++seq, ++c) {
        const int st = seq % NST;
        if (tid == 0) TRACE_AT(0, 10);
        bounded_wait(&bb->full[st], (seq / NST) & 1, a.err);
        if (tid == 0) TRACE_AT(0, 11);
        const float* Hc = reinterpret_cast<const float*>(base + static_cast<size_t>(st) * a.stage_bytes);
        const float* Sc = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(Hc) + a.off_S);
        const float* Gc = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(Hc) + a.off_G);
        if (c >= 2) bounded_wait(&bb->afree[c & 1], ((c - 2) >> 1) & 1, a.err);
        float hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = lds4(Hc + row * 32 + ((((4 * half + i) ^ (row & 7))) << 2));
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[4 * i + e] = tf32_rna(vv[e]);
            lo[4 * i + e] = vv[e] - hi[4 * i + e];
          }
        }
        const uint32_t ta = lane_base + kAcolA + 64u * (c & 1) + 16u * half;
        tmem_st16(ta, hi);
        tmem_st16(ta + 32u, lo);
        if (sd_active) {  // C and d_ctx partial dot products, 8 columns of this chunk
          const int s = sd_s, ch0 = 2 * sd_jo;
          const float4 h0 = lds4(Sc + s * 32 + ((ch0 ^ (s & 7)) << 2));
          const float4 h1 = lds4(Sc + s * 32 + (((ch0 + 1) ^ (s & 7)) << 2));
          const float4 g0 = lds4(Gc + s * 32 + ((ch0 ^ (s & 7)) << 2));
          const float4 g1 = lds4(Gc + s * 32 + (((ch0 + 1) ^ (s & 7)) << 2));
          const int jb = q * kChunk + 8 * sd_jo;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* wc = sW_Ct + (4 * sd_dq + i) * SH2 + jb;
            const float* wo = sW_O + (4 * sd_dq + i) * SH2 + jb;
            const float4 c0 = lds4(wc), c1 = lds4(wc + 4), o0 = lds4(wo), o1 = lds4(wo + 4);
            float x = cacc[i], y = dacc[i];
            x = fmaf(h0.x, c0.x, x); x = fmaf(h0.y, c0.y, x); x = fmaf(h0.z, c0.z, x); x = fmaf(h0.w, c0.w, x);
            x = fmaf(h1.x, c1.x, x); x = fmaf(h1.y, c1.y, x); x = fmaf(h1.z, c1.z, x); x = fmaf(h1.w, c1.w, x);
            y = fmaf(g0.x, o0.x, y); y = fmaf(g0.y, o0.y, y); y = fmaf(g0.z, o0.z, y); y = fmaf(g0.w, o0.w, y);
            y = fmaf(g1.x, o1.x, y); y = fmaf(g1.y, o1.y, y); y = fmaf(g1.z, o1.z, y); y = fmaf(g1.w, o1.w, y);
            cacc[i] = x;
            dacc[i] = y;
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bb->aready[c & 1]);
          mbar_arrive(&bb->empty[st]);
        }
        if (tid == 0) TRACE_AT(0, 13);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        cacc[i] += __shfl_xor_sync(0xffffffffu, cacc[i], 1);
        cacc[i] += __shfl_xor_sync(0xffffffffu, cacc[i], 2);
        dacc[i] += __shfl_xor_sync(0xffffffffu, dacc[i], 1);
        dacc[i] += __shfl_xor_sync(0xffffffffu, dacc[i], 2);
      }
      if (sd_active && sd_jo == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sC[sd_s * D + 4 * sd_dq + i] = cacc[i];
          sDctx[sd_s * D + 4 * sd_dq + i] = a.tw * dacc[i];
        }
      }
      // ==================================== projections: TMEM -> shared memory
      if (tid == 0) TRACE_AT(0, 20);
      bounded_wait(&bb->accfull, t & 1, a.err);
      if (tid == 0) TRACE_AT(0, 21);
      tc_fence_after();
      {
        const int c0 = half * D;  // warps 0-3: A columns, 4-7: B columns
        float v[D];
#pragma unroll
        for (int i = 0; i < D; ++i) v[i] = 0.f;
        for (int p = 0; 2 * p < NC; ++p) {
          uint32_t r0[D], r1[D];
          tmem_ld16_nowait(lane_base + p * FD + c0, r0);
          tmem_ld16_nowait(lane_base + p * FD + TD + c0, r1);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < D; ++i) v[i] += __uint_as_float(r0[i]);
#pragma unroll
          for (int i = 0; i < D; ++i) v[i] += __uint_as_float(r1[i]);
        }
#pragma unroll
        for (int i = 0; i < D; i += 4)
          sts4(sPh + sw128_idx(row, c0 + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
      }
      tc_fence_before();
      named_sync(1, kComputeThreads);
      if (tid == 0) TRACE_AT(0, 22);
      // ================================ scan and reverse scan per (sample, state)
      if (tid < S_t * D) {
        const int s = tid >> 4, d = tid & 15;
        float x = 0.f;
        for (int k = 0; k < K; ++k) {  // replay: A stays, B_t is replaced by x_t
          const int r = s * K + k;
          float* pb = sPh + sw128_idx(r, D + d);
          x = fmaf(sigmoidf_(sPh[sw128_idx(r, d)]), x, *pb);
          *pb = x;
        }
        const float Cv = sC[s * D + d], dctx = sDctx[s * D + d];
        sCtx[s * D + d] = Cv * x;
        sDC[s * D + d] = dctx * x;
        float dx = dctx * Cv;
        for (int k = K - 1; k >= 0; --k) {
          const int r = s * K + k;
          float* pa = sPh + sw128_idx(r, d);
          float* pb = sPh + sw128_idx(r, D + d);
          const float at = *pa;
          const float sg = sigmoidf_(at);
          const float dsg = sg * sigmoidf_(-at);
          const float xprev = k > 0 ? sPh[sw128_idx(r - 1, D + d)] : 0.f;
          *pb = dx;                   // dB
          *pa = dx * xprev * dsg;     // dA
          dx *= sg;
        }
      }
      named_sync(1, kComputeThreads);
      if (tid == 0) TRACE_AT(0, 23);
      // dA|dB = hi + lo: hi stays in sPh, the exact remainder goes to sPl
      for (int i = 4 * tid; i < kTileRows * 32; i += 4 * kComputeThreads) {
        const float4 v = lds4(sPh + i);
        const float4 h = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
        sts4(sPh + i, h);
        sts4(sPl + i, make_float4(v.x - h.x, v.y - h.y, v.z - h.z, v.w - h.w));
      }
      fence_proxy_async_smem();
      named_sync(1, kComputeThreads);
      if (tid == 0) mbar_arrive(&bb->bready);
      if (tid == 0) TRACE_AT(0, 24);
      // ===================== per sample: dW_C, dW_O partial sums and d_h_s2
      const int njq = SH2 / 4;
      for (int k = 0; k < NSI; ++k, ++seq) {
        const int st = seq % NST;
        bounded_wait(&bb->full[st], (seq / NST) & 1, a.err);
        if (tid == 0) TRACE_AT(0, 31);
        float* hsb = reinterpret_cast<float*>(base + static_cast<size_t>(st) * a.stage_bytes);
        float* gb = hsb + static_cast<size_t>(kBwdSampleItem) * SH2;
        const int s0 = k * kBwdSampleItem, ns = min(kBwdSampleItem, S_t - s0);
        if (own_c) {
          for (int s = 0; s < ns; ++s) {
            const float4 hv = lds4(hsb + s * SH2 + 4 * pjq_c);
            const float4 gv = lds4(gb + s * SH2 + 4 * pjq_c);
            const float4 dc = lds4(sDC + (s0 + s) * D + 4 * pdq);
            const float4 cx = lds4(sCtx + (s0 + s) * D + 4 * pdq);
            const float hvv[4] = {hv.x, hv.y, hv.z, hv.w}, gvv[4] = {gv.x, gv.y, gv.z, gv.w};
            const float dcv[4] = {dc.x, dc.y, dc.z, dc.w}, cxv[4] = {cx.x, cx.y, cx.z, cx.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                accC[i][e] = fmaf(hvv[i], dcv[e], accC[i][e]);
                accO[i][e] = fmaf(gvv[i], cxv[e], accO[i][e]);
              }
          }
        }
        named_sync(1, kComputeThreads);  // h_s2 rows no longer needed: d_h_s2 goes there
        const int nit = ((ns + 3) / 4) * njq;
        for (int it = tid; it < nit; it += kComputeThreads) {
          const int jq = it % njq, sq = it / njq;
          float o[4][4];
          int sidx[4];
#pragma unroll
          for (int si = 0; si < 4; ++si) {
            sidx[si] = min(4 * sq + si, ns - 1);
            const float4 gv = lds4(gb + sidx[si] * SH2 + 4 * jq);
            o[si][0] = gv.x; o[si][1] = gv.y; o[si][2] = gv.z; o[si][3] = gv.w;
          }
#pragma unroll 4
          for (int d = 0; d < D; ++d) {
            const float4 w = lds4(sW_Ct + d * SH2 + 4 * jq);
#pragma unroll
            for (int si = 0; si < 4; ++si) {
              const float dcv = sDC[(s0 + sidx[si]) * D + d];
              o[si][0] = fmaf(dcv, w.x, o[si][0]);
              o[si][1] = fmaf(dcv, w.y, o[si][1]);
              o[si][2] = fmaf(dcv, w.z, o[si][2]);
              o[si][3] = fmaf(dcv, w.w, o[si][3]);
            }
          }
#pragma unroll
          for (int si = 0; si < 4; ++si) {
            const int s = 4 * sq + si;
            if (s < ns) sts4(hsb + s * SH2 + 4 * jq, make_float4(o[si][0], o[si][1], o[si][2], o[si][3]));
          }
        }
        fence_proxy_async_smem();
        named_sync(1, kComputeThreads);
        if (tid == 0) {
          bulk_store(a.out1 + (tb0 + s0) * SH2, hsb, static_cast<uint32_t>(ns) * SH2 * 4u);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(&bb->empty[st], kComputeWarps);
          TRACE_AT(0, 33);
        }
      }
      // ================================= per 16 rows: dW_A|dW_B partial sums
      for (int k = 0; k < NRI; ++k, ++seq) {
        const int st = seq % NST;
        bounded_wait(&bb->full[st], (seq / NST) & 1, a.err);
        if (tid == 0) TRACE_AT(0, 41);
        const float* hb = reinterpret_cast<const float*>(base + static_cast<size_t>(st) * a.stage_bytes);
        const int r0 = k * kRowItem, nr = min(kRowItem, R_t - r0);
        if (own_ab) {
          const float* hrow = hb + 4 * pjq_ab;
#pragma unroll 2
          for (int r = 0; r < nr; ++r) {
            const int rr = r0 + r;
            const float4 hv = lds4(hrow + r * SH2);
            const float4 p0 = lds4(sPh + sw128_idx(rr, 8 * pkq)), p1 = lds4(sPh + sw128_idx(rr, 8 * pkq + 4));
            const float4 q0 = lds4(sPl + sw128_idx(rr, 8 * pkq)), q1 = lds4(sPl + sw128_idx(rr, 8 * pkq + 4));
            const float hvv[4] = {hv.x, hv.y, hv.z, hv.w};
            const float pv[8] = {p0.x + q0.x, p0.y + q0.y, p0.z + q0.z, p0.w + q0.w,
                                 p1.x + q1.x, p1.y + q1.y, p1.z + q1.z, p1.w + q1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int e = 0; e < 8; ++e) accAB[i][e] = fmaf(hvv[i], pv[e], accAB[i][e]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb->empty[st]);
        if (tid == 0) TRACE_AT(0, 42);
      }
      // ========================= d_h_history from TMEM: thread = column j
      bounded_wait(&bb->bdone, t & 1, a.err);
      if (tid == 0) TRACE_AT(0, 45);
      tc_fence_after();
      {
        const int j = 128 * half + 32 * (warp & 3) + lane;
        float* dst = a.out0 + tb0 * K * SH2 + j;
        for (int cb = 0; cb * 32 < R_t; ++cb) {
          float v[32];
          tmem_ld<16>(lane_base + 128u * half + 32u * cb, v);
          tmem_ld<16>(lane_base + 128u * half + 32u * cb + 16u, v + 16);
          if (j < SH2) {
            const int nrow = R_t - 32 * cb;
            float* d0 = dst + static_cast<long long>(32 * cb) * SH2;
#pragma unroll
            for (int r = 0; r < 32; ++r)
              if (r < nrow) d0[static_cast<long long>(r) * SH2] = v[r];
          }
        }
      }
      tc_fence_before();
      named_sync(1, kComputeThreads);
      if (tid == 0) mbar_arrive(&bb->dhfree);
      if (tid == 0) TRACE_AT(0, 46);
    }
    // ===================================== partial sums into the CTA's slot
    float* slot = a.ws + static_cast<size_t>(cta) * 4 * SH2 * D;
    const int n = SH2 * D;
    if (own_ab) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = 4 * pjq_ab + i, col = 8 * pkq + e;
          if (col < D)
            slot[j * D + col] = accAB[i][e];
          else
            slot[n + j * D + (col - D)] = accAB[i][e];
        }
    }
    if (own_c) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * pjq_c + i, d = 4 * pdq + e;
          slot[2 * n + j * D + d] = accC[i][e];
          slot[3 * n + d * SH2 + j] = a.tw * accO[i][e];
        }
    }
    if (tid == 0) bulk_wait_all();
    if (tid == 0) TRACE_AT(0, 50);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

int round_up_b(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

bool bwd_tc_plan(int K, int SH2, int D, FastArgs* a) {
  if (!fast_path_ok(K, SH2, D) || D != 16) return false;
  int S_max = kTileRows / K;
  if (S_max > 32) S_max = 32;
  if (S_max > kComputeThreads / D) S_max = kComputeThreads / D;
  const int hc = S_max * K * 128, sc = S_max * 128;
  const int off_S = round_up_b(hc, 1024);
  const int off_G = off_S + round_up_b(sc, 1024);
  int stage = off_G + sc;
  if (2 * kBwdSampleItem * SH2 * 4 > stage) stage = 2 * kBwdSampleItem * SH2 * 4;
  if (kRowItem * SH2 * 4 > stage) stage = kRowItem * SH2 * 4;
  if (kTileRows * 128 > stage) stage = kTileRows * 128;
  stage = round_up_b(stage, 1024);
  const int wbytes = SH2 * 4 * D * 4;
  const int rest = wbytes + 2 * D * SH2 * 4 + 2 * kTileRows * 128 + 4 * S_max * D * 4 +
                   static_cast<int>(sizeof(BwdBars)) + 1024 + 64;
  int n_stages = kMaxStages;
  while (n_stages > 2 && n_stages * stage + rest > 227 * 1024) --n_stages;
  int off = n_stages * stage;
  a->off_wt = off;  off += wbytes;
  a->off_p = off;   off += kTileRows * 128;
  a->off_hlo = off; off += kTileRows * 128;
  a->off_wct = off; off += D * SH2 * 4;
  a->off_wo = off;  off += D * SH2 * 4;
  a->off_cs = off;  off += S_max * D * 4;
  a->off_ctx = off; off += S_max * D * 4;
  a->off_dctx = off; off += S_max * D * 4;
  a->off_dc = off;  off += S_max * D * 4;
  off = round_up_b(off, 16);
  a->off_bar = off; off += static_cast<int>(sizeof(BwdBars));
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
  return a->smem_bytes <= 227 * 1024;
}

cudaError_t launch_bwd_tc(const FastArgs& a, int grid, cudaStream_t stream) {
  bwd_tc_kernel<<<grid, kBwdThreads, a.smem_bytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t prepare_bwd_tc_kernels(int max_smem) {
  return cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

}  // namespace m2scan
