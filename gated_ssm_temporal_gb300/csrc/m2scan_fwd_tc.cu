// Forward of the gated temporal scan layer with the projections on the
// tensor cores, warp-specialised (D in {8, 16}, SH2 % 32 == 0, SH2 <= 256,
// K <= 128).
//
// Roles inside each persistent CTA (one CTA per weight-gradient slot range of
// samples, tiles of at most 128 rows = S samples x K):
//   warp 8 (producer)  streams the items of every tile into a ring of shared
//                      memory stages: per 32-column chunk of SH2 a TMA box of
//                      h_history [S, K, 32] and of h_s2 [S, 32] (128-byte
//                      swizzle), then the h_s2 rows for the output step.
//   warps 0-7 (compute) per chunk: split h = hi + lo (hi = tf32 round to
//                      nearest) and store both into a TMEM A-operand buffer
//                      (thread = tile row); partial dot products of
//                      C = h_s2 . W_C. Per tile: read the projections back from
//                      TMEM, run the scan x_t = sigmoid(A_t) x_{t-1} + B_t,
//                      ctx = C x_{K-1} and h_enriched = h_s2 + tw ctx . W_O
//                      ("Custom Kernel Optimization -- cuBLAS Projections +
//                      Batch-Parallel Scans", Design 1, Steps 1-2; output step
//                      as the layer fixes it).
//   warp 9 (MMA)       per chunk, for each 8-column K step: one tf32 MMA
//                      hi . [W_hi ; W_lo] (N = 4D) into the accumulator pair of
//                      the chunk pair, one lo . W_hi (N = 2D) into a shared
//                      correction accumulator. A|B = sum of the main and
//                      correction accumulators, added in a fixed order in
//                      registers: fp32-level accuracy from 3 x tf32 products.
// Hand-offs use shared-memory mbarriers only; no CTA-wide barrier per chunk.
#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kFwdThreads = kComputeThreads + 64;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

struct FwdBars {
  uint64_t full[kMaxStages];   // producer -> compute: stage loaded
  uint64_t empty[kMaxStages];  // compute warps -> producer: stage consumed
  uint64_t aready[2];          // compute warps -> MMA: TMEM A buffer written
  uint64_t afree[2];           // MMA -> compute: TMEM A buffer consumed
  uint64_t accfull;            // MMA -> compute: every MMA of the tile done
  uint64_t accempty;           // compute -> MMA: accumulators read out
  uint32_t tslot;              // TMEM base address from tcgen05.alloc
  uint32_t pad;
};

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_tc_kernel(const __grid_constant__ FastArgs a) {
  constexpr int TD = 2 * D;   // columns of A|B
  constexpr int FD = 4 * D;   // rows of a weight tile: tf32 part, then remainder
  constexpr int PS = TD + 4;  // row stride of the A|B tile in shared memory
  constexpr int NQ = D / 4;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  float* sW = reinterpret_cast<float*>(base + a.off_wt);      // NC tiles [FD][32], swizzled
  float* sW_Ct = reinterpret_cast<float*>(base + a.off_wct);  // W_C transposed [D][SH2]
  float* sW_O = reinterpret_cast<float*>(base + a.off_wo);    // W_O [D][SH2]
  float* sP = reinterpret_cast<float*>(base + a.off_p);       // A|B tile [128][PS]
  float* sC = reinterpret_cast<float*>(base + a.off_cs);      // C [S_max][D]
  float* sCtx = reinterpret_cast<float*>(base + a.off_ctx);   // ctx [S_max][D]
  FwdBars* bb = reinterpret_cast<FwdBars*>(base + a.off_bar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int trace_n = 0;
  (void)trace_n;
  if (tid == 0) TRACE_AT(0, 1);
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max, SG = a.SG, NST = a.n_stages;
  const int NC = SH2 / kChunk, NP = (NC + 1) / 2;
  const uint32_t corr_col = static_cast<uint32_t>(NP * FD);
  const uint32_t acol0 = corr_col + TD;
  const long long B = a.B;
  const int P = gridDim.x, cta = blockIdx.x;
  const long long cb0 = B * cta / P;
  const int n_c = static_cast<int>(B * (cta + 1) / P - cb0);
  const int T = (n_c + S_max - 1) / S_max;
  const int t_base = n_c / T, t_extra = n_c - (n_c / T) * T;
  auto tile_start = [&](int i) -> long long {
    return cb0 + static_cast<long long>(i) * t_base + (i < t_extra ? i : t_extra);
  };

  if (tid == kProducerWarp * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_hs)) : "memory");
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bb->full[s], 1);
      mbar_init(&bb->empty[s], kComputeWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bb->aready[s], kComputeWarps);
      mbar_init(&bb->afree[s], 1);
    }
    mbar_init(&bb->accfull, 1);
    mbar_init(&bb->accempty, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&bb->tslot, a.tmem_cols);
  __syncthreads();  // barriers initialised: the producer may start while the weights load

  int pseq = 0;  // producer: next item to load
  int ptile = 0, pit = 0;
  auto produce_one = [&]() {
    const long long tb0 = tile_start(ptile);
    const int S_t = static_cast<int>(tile_start(ptile + 1) - tb0);
    const int NSI = (S_t + SG - 1) / SG;
    const int st = pseq % NST, use = pseq / NST;
    if (use > 0) bounded_wait(&bb->empty[st], (use - 1) & 1, a.err);
    unsigned char* sp = base + static_cast<size_t>(st) * a.stage_bytes;
    uint64_t* bar = &bb->full[st];
    if (pit < NC) {
      mbar_arrive_expect_tx(bar, a.hc_bytes + a.sc_bytes);
      tma_load_3d(sp, &a.tm_h, pit * kChunk, 0, static_cast<int>(tb0), bar);
      tma_load_2d(sp + a.off_S, &a.tm_hs, pit * kChunk, static_cast<int>(tb0), bar);
    } else {
      const int s0 = (pit - NC) * SG;
      const int ns = min(SG, S_t - s0);
      const uint32_t rb = static_cast<uint32_t>(ns) * SH2 * 4u;
      mbar_arrive_expect_tx(bar, rb);
      bulk_load(sp, a.h_s2 + (tb0 + s0) * SH2, rb, bar);
    }
    ++pseq;
    if (++pit == NC + NSI) {
      pit = 0;
      ++ptile;
    }
  };
  if (warp == kProducerWarp && lane == 0)
    for (int i = 0; i < NST && ptile < T; ++i) produce_one();

  // weights into shared memory: SH2*D <= 4096, all global loads first
  constexpr int kWPer = (4096 + kFwdThreads - 1) / kFwdThreads;
  {
    float wa[kWPer], wb[kWPer], wc[kWPer], wo[kWPer];
#pragma unroll
    for (int u = 0; u < kWPer; ++u) {
      const int i = tid + u * kFwdThreads;
      const bool ok = i < SH2 * D;
      wa[u] = ok ? __ldg(a.W_A + i) : 0.f;
      wb[u] = ok ? __ldg(a.W_B + i) : 0.f;
      wc[u] = ok ? __ldg(a.W_C + i) : 0.f;
      wo[u] = ok ? __ldg(a.W_O + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kWPer; ++u) {
      const int i = tid + u * kFwdThreads;
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
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bb->tslot;
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
      int c = 0;
      for (int t = 0; t < T; ++t) {
        if (t > 0) bounded_wait(&bb->accempty, (t - 1) & 1, a.err);
        for (int q = 0; q < NC; ++q, ++c) {
          TRACE_AT(2, 300 + q);
          bounded_wait(&bb->aready[c & 1], (c >> 1) & 1, a.err);
          TRACE_AT(2, 400 + q);
          tc_fence_after();
          const uint32_t ah = tmem + acol0 + 64u * (c & 1), al = ah + 32u;
          const uint32_t wt = smem_addr(sW + q * FD * 32);
          const uint32_t d_pair = tmem + static_cast<uint32_t>((q >> 1) * FD);
          const uint32_t d_corr = tmem + corr_col;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bdesc = umma_desc_sw128(wt + 32u * ks);
            umma_tf32_ta(d_pair, ah + 8u * ks, bdesc, idesc_f, ((q & 1) | ks) != 0);
            umma_tf32_ta(d_corr, al + 8u * ks, bdesc, idesc_t, (q | ks) != 0);
          }
          umma_commit(&bb->afree[c & 1]);
          TRACE_AT(2, 500 + q);
        }
        umma_commit(&bb->accfull);
      }
    }
  } else {
    // ------------------------------------------------------------- compute
    const int row = 32 * (warp & 3) + lane, half = warp >> 2;
    const int sd_jo = tid & 3, sd_dq = (tid >> 2) % NQ, sd_s = (tid >> 2) / NQ;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    int seq = 0, c = 0;
    for (int t = 0; t < T; ++t) {
      const long long tb0 = tile_start(t);
      const int S_t = static_cast<int>(tile_start(t + 1) - tb0);
      const int NSI = (S_t + SG - 1) / SG;
      const bool sd_active = sd_s < S_t;
      float cacc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = 0; q < NC; ++q, ++seq, ++c) {
        const int st = seq % NST;
        if (tid == 0) TRACE_AT(0, 10);
        bounded_wait(&bb->full[st], (seq / NST) & 1, a.err);
        if (tid == 0) TRACE_AT(0, 11);
        const float* Hc = reinterpret_cast<const float*>(base + static_cast<size_t>(st) * a.stage_bytes);
        const float* Sc = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(Hc) + a.off_S);
        if (c >= 2) bounded_wait(&bb->afree[c & 1], ((c - 2) >> 1) & 1, a.err);
        if (tid == 0) TRACE_AT(0, 12);
        // A operand: this thread's row, 16 of the chunk's 32 columns
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
        const uint32_t ta = lane_base + acol0 + 64u * (c & 1) + 16u * half;
        tmem_st16(ta, hi);
        tmem_st16(ta + 32u, lo);
        // C partial dot products over this chunk while the TMEM stores land:
        // sample sd_s, states 4*sd_dq.., 8 columns
        if (sd_active) {
          const int s = sd_s, ch0 = 2 * sd_jo;
          const float4 h0 = lds4(Sc + s * 32 + ((ch0 ^ (s & 7)) << 2));
          const float4 h1 = lds4(Sc + s * 32 + (((ch0 + 1) ^ (s & 7)) << 2));
          const int jb = q * kChunk + 8 * sd_jo;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* w = sW_Ct + (4 * sd_dq + i) * SH2 + jb;
            const float4 w0 = lds4(w), w1 = lds4(w + 4);
            float acc = cacc[i];
            acc = fmaf(h0.x, w0.x, acc); acc = fmaf(h0.y, w0.y, acc);
            acc = fmaf(h0.z, w0.z, acc); acc = fmaf(h0.w, w0.w, acc);
            acc = fmaf(h1.x, w1.x, acc); acc = fmaf(h1.y, w1.y, acc);
            acc = fmaf(h1.z, w1.z, acc); acc = fmaf(h1.w, w1.w, acc);
            cacc[i] = acc;
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
      // C: sum the four column groups in a fixed order
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        cacc[i] += __shfl_xor_sync(0xffffffffu, cacc[i], 1);
        cacc[i] += __shfl_xor_sync(0xffffffffu, cacc[i], 2);
      }
      if (sd_active && sd_jo == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) sC[sd_s * D + 4 * sd_dq + i] = cacc[i];
      }
      // A|B: main and correction accumulators, added in a fixed order
      if (tid == 0) TRACE_AT(0, 20);
      bounded_wait(&bb->accfull, t & 1, a.err);
      if (tid == 0) TRACE_AT(0, 21);
      tc_fence_after();
      {
        const int c0 = half * D;  // warps 0-3: A columns, 4-7: B columns
        float v[D];
#pragma unroll
        for (int i = 0; i < D; ++i) v[i] = 0.f;
        // per pair: main and correction block issued together, one wait
        for (int p = 0; p < NP; ++p) {
          uint32_t r0[D], r1[D];
          if constexpr (D == 16) {
            tmem_ld16_nowait(lane_base + p * FD + c0, r0);
            tmem_ld16_nowait(lane_base + p * FD + TD + c0, r1);
          } else {
            tmem_ld8_nowait(lane_base + p * FD + c0, r0);
            tmem_ld8_nowait(lane_base + p * FD + TD + c0, r1);
          }
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < D; ++i) v[i] += __uint_as_float(r0[i]);
#pragma unroll
          for (int i = 0; i < D; ++i) v[i] += __uint_as_float(r1[i]);
        }
        {
          float w[D];
          tmem_ld<D>(lane_base + corr_col + c0, w);
#pragma unroll
          for (int i = 0; i < D; ++i) v[i] += w[i];
        }
        float* pr = sP + row * PS + c0;
#pragma unroll
        for (int i = 0; i < D; i += 4) sts4(pr + i, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
      }
      tc_fence_before();
      named_sync(1, kComputeThreads);
      if (tid == 0) TRACE_AT(0, 22);
      if (tid == 0) mbar_arrive(&bb->accempty);
      // scan: one thread per (sample, state)
      if (tid < S_t * D) {
        const int s = tid / D, d = tid - (tid / D) * D;
        const float* pcol = sP + s * K * PS;
        const float gsc = load_gate_scale(a.gate_scale);
        float x = 0.f;
        int k = 0;
        for (; k + 8 <= K; k += 8) {  // 8 independent gates, then the 8-step chain
          float g8[8], b8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float* pr = pcol + (k + u) * PS;
            g8[u] = gsc * sigmoidf_(pr[d]);
            b8[u] = pr[D + d];
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) x = fmaf(g8[u], x, b8[u]);
        }
        for (; k < K; ++k) {
          const float* pr = pcol + k * PS;
          x = fmaf(gsc * sigmoidf_(pr[d]), x, pr[D + d]);
        }
        sCtx[d * S_max + s] = sC[s * D + d] * x;  // transposed: [D][S_max]
      }
      named_sync(1, kComputeThreads);
      if (tid == 0) TRACE_AT(0, 23);
      // output step: h_enriched = h_s2 + tw * ctx . W_O, in place over the h_s2 rows
      const int njq = SH2 / 4;
      for (int k = 0; k < NSI; ++k, ++seq) {
        const int st = seq % NST;
        bounded_wait(&bb->full[st], (seq / NST) & 1, a.err);
        float* hsb = reinterpret_cast<float*>(base + static_cast<size_t>(st) * a.stage_bytes);
        const int s0 = k * SG, ns = min(SG, S_t - s0);
        const int nit = ((ns + 3) / 4) * njq;
        for (int it = tid; it < nit; it += kComputeThreads) {
          const int jq = it % njq, sq = it / njq;
          float o[4][4];
#pragma unroll
          for (int si = 0; si < 4; ++si)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[si][e] = 0.f;
          // four samples 4*sq.. (clamped into the item; rows past ns are not stored)
          int sidx[4];
#pragma unroll
          for (int si = 0; si < 4; ++si) sidx[si] = s0 + min(4 * sq + si, ns - 1);
#pragma unroll 4
          for (int d = 0; d < D; ++d) {
            const float4 w = lds4(sW_O + d * SH2 + 4 * jq);
            const float* cr = sCtx + d * S_max;
            const float cxv[4] = {cr[sidx[0]], cr[sidx[1]], cr[sidx[2]], cr[sidx[3]]};
#pragma unroll
            for (int si = 0; si < 4; ++si) {
              o[si][0] = fmaf(cxv[si], w.x, o[si][0]);
              o[si][1] = fmaf(cxv[si], w.y, o[si][1]);
              o[si][2] = fmaf(cxv[si], w.z, o[si][2]);
              o[si][3] = fmaf(cxv[si], w.w, o[si][3]);
            }
          }
#pragma unroll
          for (int si = 0; si < 4; ++si) {
            const int s = 4 * sq + si;
            if (s < ns) {
              float* hp = hsb + s * SH2 + 4 * jq;
              float4 h = lds4(hp);
              h.x = fmaf(a.tw, o[si][0], h.x);
              h.y = fmaf(a.tw, o[si][1], h.y);
              h.z = fmaf(a.tw, o[si][2], h.z);
              h.w = fmaf(a.tw, o[si][3], h.w);
              sts4(hp, h);
            }
          }
        }
        fence_proxy_async_smem();
        named_sync(1, kComputeThreads);
        if (tid == 0) TRACE_AT(0, 30);
        if (tid == 0) {
          bulk_store(a.out0 + (tb0 + s0) * SH2, hsb, static_cast<uint32_t>(ns) * SH2 * 4u);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(&bb->empty[st], kComputeWarps);
          TRACE_AT(0, 31);
        }
      }
    }
    if (tid == 0) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) tmem_dealloc(tmem, a.tmem_cols);
}

int round_up_i(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

bool fwd_tc_plan(int K, int SH2, int D, FastArgs* a) {
  if (!fast_path_ok(K, SH2, D) || !(D == 8 || D == 16)) return false;
  int S_max = kTileRows / K;
  if (S_max > 32) S_max = 32;
  if (S_max > kComputeThreads / D) S_max = kComputeThreads / D;
  const int hc = S_max * K * 128, sc = S_max * 128;
  const int off_S = round_up_i(hc, 1024);
  int stage = off_S + sc;
  if (S_max * SH2 * 4 > stage) stage = S_max * SH2 * 4;
  if (kTileRows * 128 > stage) stage = kTileRows * 128;  // the A tile always spans 128 rows
  stage = round_up_i(stage, 1024);
  const int wbytes = SH2 * 4 * D * 4;  // weight tiles: 4D rows x SH2 columns
  int rest = wbytes + 2 * D * SH2 * 4 + kTileRows * (2 * D + 4) * 4 + 2 * S_max * D * 4 +
             static_cast<int>(sizeof(FwdBars)) + 1024 + 64;
  int n_stages = kMaxStages;
  while (n_stages > 2 && n_stages * stage + rest > 227 * 1024) --n_stages;
  int off = n_stages * stage;
  a->off_wt = off;  off += wbytes;
  a->off_wct = off; off += D * SH2 * 4;
  a->off_wo = off;  off += D * SH2 * 4;
  a->off_p = off;   off += kTileRows * (2 * D + 4) * 4;
  a->off_cs = off;  off += S_max * D * 4;
  a->off_ctx = off; off += S_max * D * 4;
  off = round_up_i(off, 16);
  a->off_bar = off; off += static_cast<int>(sizeof(FwdBars));
  a->smem_bytes = off + 1024;
  a->S_max = S_max;
  a->SG = S_max;
  a->stage_bytes = stage;
  a->hc_bytes = hc;
  a->sc_bytes = sc;
  a->off_S = off_S;
  a->off_G = off_S;
  a->K = K;
  a->SH2 = SH2;
  a->n_stages = n_stages;
  a->tc = 1;
  const int NP = (SH2 / kChunk + 1) / 2;
  int cols = 32;
  while (cols < NP * 4 * D + 2 * D + 128) cols *= 2;
  a->tmem_cols = cols;
  return a->smem_bytes <= 227 * 1024 && cols <= 512;
}

cudaError_t launch_fwd_tc(int D, const FastArgs& a, int grid, cudaStream_t stream) {
  switch (D) {
    case 8: fwd_tc_kernel<8><<<grid, kFwdThreads, a.smem_bytes, stream>>>(a); break;
    case 16: fwd_tc_kernel<16><<<grid, kFwdThreads, a.smem_bytes, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t prepare_fwd_tc_kernels(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fwd_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             max_smem);
  return e;
}

}  // namespace m2scan
