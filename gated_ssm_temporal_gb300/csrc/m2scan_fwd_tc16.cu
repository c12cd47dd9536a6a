// Forward of the gated temporal scan layer for D = 16 with the projections on
// the tensor cores, warp-specialised like the backward kernel (SH2 % 32 == 0,
// SH2 <= 256, K <= 128).
//
// One persistent CTA per slot range of samples walks them in tiles of at most
// 128 rows (S samples x K) ("Custom Kernel Optimization -- cuBLAS Projections
// + Batch-Parallel Scans", Design 1, Steps 1-2; output step as the layer fixes
// it). Per tile:
//   pass 1   the producer warp streams 32-column chunks of h_history and h_s2
//            (TMA boxes, 128-byte swizzle). One MMA thread computes
//            A|B = h . [W_A|W_B] with the chunk as the A operand straight from
//            shared memory (the tensor core reads trunc(h)); the compute warps
//            write h - trunc(h) (rounded to tf32) into tensor memory and a
//            second MMA thread adds that product (3 x tf32 in all). A stage is
//            free once its main MMAs are done and the compute warps have read
//            it. The compute warps form C = h_s2 . W_C on the FMA pipe
//            meanwhile.
//   scan     x_t = sigmoid(A_t) x_{t-1} + B_t, one thread per (sample, state);
//            ctx = C x_{K-1}.
//   output   h_enriched = h_s2 + tw ctx . W_O from the tile's h_s2 rows
//            (a stage of their own, loaded after the next tile's chunks),
//            written straight to global memory.
#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kFwdThreads = kComputeThreads + 96;
constexpr int kProducerWarp = kComputeWarps;
constexpr int kMmaWarp = kComputeWarps + 1;    // main products trunc(h) . [W_hi | W_lo]
constexpr int kCorrWarp = kComputeWarps + 2;   // remainder products (h - trunc h) . W_hi
constexpr int kChunkRing = 6;
constexpr int kLoBufs = 3;

// Two threads issue the tensor-core work, each with its own commits: a
// commit stalls only the stream of the thread that issues it, so the main
// and the remainder products of a chunk overlap each other's stalls.
struct FwdBars {
  uint64_t full[kMaxStages];     // producer -> MMA, compute: chunk loaded into stage s
  uint64_t fullo[kMaxStages];    // producer -> compute: h_s2 rows loaded into stage s (the MMA
                                 // threads skip these items, so they have a barrier of their own)
  uint64_t empty[kMaxStages];    // chunk stage s free: main products done (commit) + compute read (arrive)
  uint64_t outdone[kMaxStages];  // compute -> producer: h_s2 item in stage s read (one arrival per warp)
  uint64_t loready[kChunkRing];  // compute -> remainder MMA thread: chunk c read, h - trunc(h) in TMEM
  uint64_t lofree[kLoBufs];      // remainder MMA thread -> all: remainder buffer's products done
  uint64_t mdone[2];             // main MMA thread -> compute: main products of tile t (set t & 1) done
  uint64_t accempty[2];          // compute -> MMA threads: projections of accumulator set s read back
  uint32_t tslot;
  uint32_t pad;
};

// TMEM columns: two accumulator sets, tile t using set t & 1 at 256 (t & 1),
// so that the MMA threads start the next tile's products while the compute
// warps still read back, scan and write out this one. Within a set: [0, 128)
// trunc(h) . [W_hi | W_lo] of the even and of the odd chunks, [224, 256)
// (h - trunc h) . W_hi. [128, 224): three buffers of h - trunc(h), shared
// by both sets.
constexpr uint32_t kColLo = 128;
constexpr uint32_t kColCorr = 224;
constexpr uint32_t kSetCols = 256;

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

// DR: the layer's states (4 or 16; a compile-time constant, so that the
// D = 16 kernel is exactly the unpadded one).
template <int DR>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_tc16_kernel(const __grid_constant__ FastArgs a) {
  constexpr int D = 16, TD = 32, FD = 64;  // states inside the kernel
  constexpr int Dr = DR;  // the layer's states; the others have zero weights
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  float* sW = reinterpret_cast<float*>(base + a.off_wt);      // NC tiles [FD][32], swizzled
  float* sW_Ct = reinterpret_cast<float*>(base + a.off_wct);  // W_C transposed [D][SH2]
  float* sW_O = reinterpret_cast<float*>(base + a.off_wo);    // W_O [D][SH2]
  float* sP = reinterpret_cast<float*>(base + a.off_p);       // A|B [128][32] swizzled
  float* sC = reinterpret_cast<float*>(base + a.off_cs);      // C [S_max][D]
  float* sCtx = reinterpret_cast<float*>(base + a.off_ctx);   // ctx [S_max][D]
  FwdBars* bb = reinterpret_cast<FwdBars*>(base + a.off_bar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max, NST = a.n_stages;
  int trace_n = 0;
  (void)trace_n;
  if (tid == 0) TRACE_CTA(0);
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
  auto stage_ptr = [&](int st) { return base + static_cast<uint32_t>(st) * stage_bytes; };

  if (tid == kProducerWarp * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_hs)) : "memory");
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bb->full[s], 1);
      mbar_init(&bb->fullo[s], 1);
      mbar_init(&bb->empty[s], 2);
      mbar_init(&bb->outdone[s], kComputeWarps);
    }
    for (int s = 0; s < kChunkRing; ++s) mbar_init(&bb->loready[s], kComputeWarps);
    for (int s = 0; s < kLoBufs; ++s) mbar_init(&bb->lofree[s], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bb->mdone[s], 1);
      mbar_init(&bb->accempty[s], 1);  // waited for by both MMA threads
    }
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&bb->tslot, 2 * kSetCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bb->tslot;

  // ---- producer: in round u = 0 .. T the NC chunks of tile u (u < T), then
  // the item of tile u - 1's h_s2 rows (u >= 1): the compute warps read a
  // tile's h_s2 rows after the next tile's chunks and write its output
  // straight to global memory
  RingPos lp, rp;
  uint32_t rch = 0;     // bit s: parity of the next empty[s] phase (chunks only)
  uint32_t rout = 0;    // bit s: parity of the next outdone[s] phase (h_s2 items only)
  int pn = 0, pround = 0, pit = 0;
  int rround = 0, rit = 0;
  auto round_items = [&](int u) { return (u < T ? NC : 0) + (u >= 1 ? 1 : 0); };
  auto release_one = [&]() {
    if (rit < (rround < T ? NC : 0)) {
      // a chunk: free once its main products are done and the compute warps
      // have read it
      bounded_wait(&bb->empty[rp.i], (rch >> rp.i) & 1u, a.err);
      rch ^= 1u << rp.i;
    } else {
      bounded_wait(&bb->outdone[rp.i], (rout >> rp.i) & 1u, a.err);
      rout ^= 1u << rp.i;
    }
    rp.next(NST);
    if (++rit == round_items(rround)) {
      rit = 0;
      ++rround;
    }
  };
  auto produce_one = [&]() {
    if (pn >= NST) release_one();
    unsigned char* sp = stage_ptr(lp.i);
    const bool chunk = pit < (pround < T ? NC : 0);
    uint64_t* bar = chunk ? &bb->full[lp.i] : &bb->fullo[lp.i];
    if (chunk) {
      const long long tb0 = tile_start(pround);
      mbar_arrive_expect_tx(bar, a.hc_bytes + a.sc_bytes);
      tma_load_3d(sp, &a.tm_h, pit * kChunk, 0, static_cast<int>(tb0), bar);
      tma_load_2d(sp + a.off_S, &a.tm_hs, pit * kChunk, static_cast<int>(tb0), bar);
    } else {
      const long long tb0 = tile_start(pround - 1);
      const int S_t = static_cast<int>(tile_start(pround) - tb0);
      const uint32_t rb = static_cast<uint32_t>(S_t) * SH2 * 4u;
      mbar_arrive_expect_tx(bar, rb);
      bulk_load(sp, a.h_s2 + tb0 * SH2, rb, bar);
    }
    lp.next(NST);
    ++pn;
    if (++pit == round_items(pround)) {
      pit = 0;
      ++pround;
    }
  };

  // ---- weights: projection B tiles, W_C^T and W_O into shared memory.
  // Thread = (state quad dq, row j), j fastest: one float4 of each of W_A, W_B,
  // W_C row j, so that the transposed and swizzled stores of a warp go to 32
  // consecutive columns (no bank conflicts); W_O is copied as float4.
  constexpr int kWPer = (256 * 4 + kFwdThreads - 1) / kFwdThreads;  // SH2 x D/4 items, SH2 <= 256
  {
    float4 wa[kWPer], wb[kWPer], wc[kWPer], wo[kWPer];
#pragma unroll
    for (int u = 0; u < kWPer; ++u) {
      const int i = tid + u * kFwdThreads;
      const bool ok = i < SH2 * 4;
      const int j = i % SH2, dq = i / SH2;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      // states Dr .. 15 of a layer with fewer states: zero weights
      const bool okd = ok && 4 * dq < Dr;
      wa[u] = okd ? __ldg(reinterpret_cast<const float4*>(a.W_A + j * Dr + 4 * dq)) : z;
      wb[u] = okd ? __ldg(reinterpret_cast<const float4*>(a.W_B + j * Dr + 4 * dq)) : z;
      wc[u] = okd ? __ldg(reinterpret_cast<const float4*>(a.W_C + j * Dr + 4 * dq)) : z;
      wo[u] = ok && i < Dr * SH2 / 4 ? __ldg(reinterpret_cast<const float4*>(a.W_O) + i) : z;
    }
    // the first stages are requested after the weights, so that the weight
    // loads are not queued behind them
    if (warp == kProducerWarp && lane == 0)
      for (int i = 0; i < NST && pround <= T; ++i) produce_one();
#pragma unroll
    for (int u = 0; u < kWPer; ++u) {
      const int i = tid + u * kFwdThreads;
      if (i >= SH2 * 4) break;
      const int j = i % SH2, dq = i / SH2;
      float* tile = sW + (j >> 5) * FD * 32;
      const int jj = j & 31;
      const float va[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
      const float vb[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
      const float vc[4] = {wc[u].x, wc[u].y, wc[u].z, wc[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = 4 * dq + e;
        const float ha = tf32_rn(va[e]), hb = tf32_rn(vb[e]);
        tile[sw128_idx(d, jj)] = ha;
        tile[sw128_idx(D + d, jj)] = hb;
        tile[sw128_idx(TD + d, jj)] = va[e] - ha;
        tile[sw128_idx(TD + D + d, jj)] = vb[e] - hb;
        sW_Ct[d * SH2 + j] = vc[e];
      }
      sts4(sW_O + 4 * i, wo[u]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      while (pround <= T) produce_one();
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------- MMA: main products
    // trunc(h) . [W_hi | W_lo] of each chunk as it lands, into the even- or
    // odd-chunk accumulator of the tile's set; a commit per chunk frees the
    // stage (with the remainder thread's arrival), one per tile hands the
    // main products to the compute warps. descriptor + 2 u = 32 u bytes on.
    if (lane == 0) {
      constexpr uint32_t idesc64 = umma_idesc_tf32(128, 64);
      const uint32_t ring = smem_addr(base);
      const uint32_t w0 = smem_addr(sW);
      RingPos tp;
      uint32_t fph = 0;  // bit s: parity of the next full[s] phase (chunks only)
      for (int t = 0; t < T; ++t) {
        // the set's previous tile (t - 2) has been read back
        if (t >= 2) bounded_wait(&bb->accempty[t & 1], ((t - 2) >> 1) & 1, a.err);
        const uint32_t acc = tmem + kSetCols * static_cast<uint32_t>(t & 1);
        RingPos pm = tp;
        for (int qm = 0; qm < NC; ++qm) {
          bounded_wait(&bb->full[pm.i], (fph >> pm.i) & 1u, a.err);
          fph ^= 1u << pm.i;
          tc_fence_after();
          TRACE_AT(2, 600 + qm);
          const uint64_t ad = umma_desc_sw128(ring + static_cast<uint32_t>(pm.i) * stage_bytes);
          const uint64_t bd = umma_desc_sw128(w0 + static_cast<uint32_t>(qm * FD * 128));
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_tf32(acc + 64u * (qm & 1), ad + 2u * ks, bd + 2u * ks, idesc64, (qm >= 2 || ks > 0) ? 1u : 0u);
          umma_commit(&bb->empty[pm.i]);
          TRACE_AT(2, 300 + qm);
          pm.next(NST);
        }
        umma_commit(&bb->mdone[t & 1]);
        for (int i = 0; i < round_items(t); ++i) tp.next(NST);  // this tile's chunks, the previous tile's rows
      }
    }
  } else if (warp == kCorrWarp) {
    // ------------------------------------- MMA: remainder products
    // (h - trunc h) . W_hi of each chunk once the compute warps have written
    // its remainder; a commit per chunk frees the remainder buffer, and the
    // one after the tile's last chunk hands the tile over.
    if (lane == 0) {
      constexpr uint32_t idesc32 = umma_idesc_tf32(128, 32);
      const uint32_t w0 = smem_addr(sW);
      RingPos tp, lr, lf;
      for (int t = 0; t < T; ++t) {
        if (t >= 2) bounded_wait(&bb->accempty[t & 1], ((t - 2) >> 1) & 1, a.err);
        const uint32_t acc = tmem + kSetCols * static_cast<uint32_t>(t & 1);
        RingPos pc = tp;
        for (int qc = 0; qc < NC; ++qc) {
          bounded_wait(&bb->loready[lr.i], lr.ph, a.err);
          tc_fence_after();
          TRACE_AT(3, 700 + qc);
          mbar_arrive(&bb->empty[pc.i]);  // the compute warps are done with the stage
          const uint32_t al = tmem + kColLo + 32u * lf.i;
          const uint64_t bd = umma_desc_sw128(w0 + static_cast<uint32_t>(qc * FD * 128));
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_tf32_ta(acc + kColCorr, al + 8u * ks, bd + 2u * ks, idesc32, (qc > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bb->lofree[lf.i]);
          TRACE_AT(3, 400 + qc);
          lr.next(kChunkRing);
          lf.next(kLoBufs);
          pc.next(NST);
        }
        for (int i = 0; i < round_items(t); ++i) tp.next(NST);
      }
    }
  } else {
    // ------------------------------------------------------------- compute
    // 8 warps, two per TMEM lane quadrant: sub = 0 / 1 selects the half of a
    // row's columns
    const int qd = warp & 3, sub = warp >> 2;
    const int row = 32 * qd + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    const float gsc = load_gate_scale(a.gate_scale);
    // C partial dots: thread = (state quad sd_dq, sample pair sd_sp, column
    // quad sd_jq): samples 2 sd_sp, 2 sd_sp + 1 x states 4 sd_dq .. + 3 over 4
    // columns of each chunk
    const int sd_jq = tid & 7, sd_sp = (tid >> 3) & 7, sd_dq = tid >> 6;
    const float* sd_w = sW_Ct + 4 * sd_dq * SH2 + 4 * sd_jq;
    int lo_off[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) lo_off[v] = row * 32 + (((4 * sub + v) ^ (row & 7)) << 2);
    RingPos ip, lr, lf;
    uint32_t cph = 0, oph = 0;  // bit s: parity of the next full[s] / fullo[s] phase
    int c = 0;
    PROF_DECL;
    // ====== output of tile tt: h_enriched = h_s2 + tw ctx . W_O from its h_s2
    // rows, straight to global memory; runs after the next tile's chunks,
    // while the MMA threads finish that tile's projections
    auto output_tile = [&](int tt) {
      const int S_t = static_cast<int>(tile_start(tt + 1) - tile_start(tt));
      {
        PROF_BEGIN();
        bounded_wait(&bb->fullo[ip.i], (oph >> ip.i) & 1u, a.err);
        oph ^= 1u << ip.i;
        PROF_END(9);
        PROF_BEGIN();
        float* hs = reinterpret_cast<float*>(stage_ptr(ip.i));
        const int st = ip.i;
        ip.next(NST);
        // thread = 4 columns x samples sq, sq + 4, sq + 8, sq + 12: each W_O
        // element serves four samples
        const int jq = tid & 63, sq = tid >> 6;
        if (4 * jq < SH2) {
          float4 o[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int dq = 0; dq < D / 4; ++dq) {
            float cx[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int s = min(sq + 4 * u, S_max - 1);
              const float4 cv = lds4(sCtx + s * D + 4 * dq);
              cx[u][0] = cv.x; cx[u][1] = cv.y; cx[u][2] = cv.z; cx[u][3] = cv.w;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 wv = lds4(sW_O + (4 * dq + e) * SH2 + 4 * jq);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                o[u].x = fmaf(cx[u][e], wv.x, o[u].x);
                o[u].y = fmaf(cx[u][e], wv.y, o[u].y);
                o[u].z = fmaf(cx[u][e], wv.z, o[u].z);
                o[u].w = fmaf(cx[u][e], wv.w, o[u].w);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int s = sq + 4 * u;
            if (s < S_t) {
              float4 h = lds4(hs + s * SH2 + 4 * jq);
              h.x = fmaf(a.tw, o[u].x, h.x);
              h.y = fmaf(a.tw, o[u].y, h.y);
              h.z = fmaf(a.tw, o[u].z, h.z);
              h.w = fmaf(a.tw, o[u].w, h.w);
              *reinterpret_cast<float4*>(a.out0 + (tile_start(tt) + s) * SH2 + 4 * jq) = h;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb->outdone[st]);  // per warp: its reads of the h_s2 rows are done
        PROF_END(10);
      }
    };
    for (int t = 0; t < T; ++t) {
      const long long tb0 = tile_start(t);
      const int S_t = static_cast<int>(tile_start(t + 1) - tb0);
      float sacc[2][4];  // [sample 2 sd_sp + i][state 4 sd_dq + e]
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[i][e] = 0.f;
      // ====================================================== pass 1 chunks
      RingPos lr_prev = lr;
      for (int q = 0; q < NC; ++q, ++c) {
        float4 w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = lds4(sd_w + e * SH2 + q * kChunk);
        PROF_BEGIN();
        if (tid == 0) TRACE_AT(0, 10);
        bounded_wait(&bb->full[ip.i], (cph >> ip.i) & 1u, a.err);
        cph ^= 1u << ip.i;
        if (tid == 0) TRACE_AT(0, 11);
        PROF_END(0);
        PROF_BEGIN();
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
        PROF_END(1);
        if (q > 0) {  // the previous chunk's remainder has landed: hand it over
          PROF_BEGIN();
          tmem_st_wait();
          PROF_END(2);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bb->loready[lr_prev.i]);
          lr_prev = lr;
        }
        PROF_BEGIN();
        // the buffer's previous chunk c - 3 is done
        if (c >= kLoBufs) bounded_wait(&bb->lofree[lf.i], lf.ph ^ 1u, a.err);
        PROF_END(3);
        PROF_BEGIN();
        tc_fence_after();
        tmem_st16(lane_base + kColLo + 32u * lf.i + 16u * sub, lo);
        lr.next(kChunkRing);
        lf.next(kLoBufs);
        {
          // all 16 rows of the box even past S_max: the reads stay inside
          // shared memory and the sums of missing samples are never stored
          const float* bp = reinterpret_cast<const float*>(sp + a.off_S);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int r = 2 * sd_sp + i;
            const float4 v = lds4(bp + r * 32 + ((sd_jq ^ (r & 7)) << 2));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float x = sacc[i][e];
              x = fmaf(v.x, w[e].x, x); x = fmaf(v.y, w[e].y, x); x = fmaf(v.z, w[e].z, x); x = fmaf(v.w, w[e].w, x);
              sacc[i][e] = x;
            }
          }
        }
        ip.next(NST);
        if (tid == 0) TRACE_AT(0, 13);
        PROF_END(4);
      }
      PROF_BEGIN();
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bb->loready[lr_prev.i]);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int m = 1; m < 8; m <<= 1) sacc[i][e] += __shfl_xor_sync(0xffffffffu, sacc[i][e], m);
      if (sd_jq == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int s = 2 * sd_sp + i;
          if (s < S_t) sts4(sC + s * D + 4 * sd_dq, make_float4(sacc[i][0], sacc[i][1], sacc[i][2], sacc[i][3]));
        }
      }
      PROF_END(5);
      if (t >= 1) output_tile(t - 1);
      // ==================================== projections: TMEM -> shared memory
      PROF_BEGIN();
      if (tid == 0) TRACE_AT(0, 20);
      // the tile's main products and the remainder products of its last chunk
      bounded_wait(&bb->mdone[t & 1], (t >> 1) & 1, a.err);
      bounded_wait(&bb->lofree[(c - 1) % kLoBufs], ((c - 1) / kLoBufs) & 1, a.err);
      if (tid == 0) TRACE_AT(0, 21);
      PROF_END(6);
      PROF_BEGIN();
      tc_fence_after();
      {
        const int c0 = 16 * sub;  // columns c0 .. c0 + 15 of A|B
        const uint32_t tc0 = lane_base + kSetCols * static_cast<uint32_t>(t & 1) + c0;
        uint32_t r0[16], r1[16], r2[16], r3[16], r4[16];
        tmem_ld16_nowait(tc0, r0);
        tmem_ld16_nowait(tc0 + TD, r1);
        tmem_ld16_nowait(tc0 + 64u, r2);
        tmem_ld16_nowait(tc0 + 64u + TD, r3);
        tmem_ld16_nowait(tc0 + kColCorr, r4);
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
          sts4(sP + sw128_idx(row, c0 + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
      }
      tc_fence_before();
      named_sync(1, kComputeThreads);
      if (tid == 0) mbar_arrive(&bb->accempty[t & 1]);
      PROF_END(7);
      PROF_BEGIN();
      // ============================== scan: one thread per (sample, state)
      if (tid < S_t * D && (K & 7) == 0) {
        // K a multiple of 8: the swizzle offsets within a group of 8 rows are
        // the same for every group
        const int s = tid >> 4, d = tid & 15, rb = s * K;
        int oa[8], ob[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          oa[u] = u * 32 + (((d >> 2) ^ u) << 2) + (d & 3);
          ob[u] = u * 32 + (((4 + (d >> 2)) ^ u) << 2) + (d & 3);
        }
        float x = 0.f;
        for (int g = 0; g < K; g += 8) {
          const float* pg = sP + (rb + g) * 32;
          float av[8], bv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            av[u] = pg[oa[u]];
            bv[u] = pg[ob[u]];
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) av[u] = gsc * sigmoid_fast(av[u]);
#pragma unroll
          for (int u = 0; u < 8; ++u) x = fmaf(av[u], x, bv[u]);
        }
        sCtx[s * D + d] = sC[s * D + d] * x;
      } else if (tid < S_t * D) {
        const int s = tid >> 4, d = tid & 15, rb = s * K;
        float x = 0.f;
        for (int k0 = 0; k0 < K; k0 += 8) {
          const int n = min(8, K - k0);
          float av[8], bv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (u < n) {
              av[u] = sP[sw128_idx(rb + k0 + u, d)];
              bv[u] = sP[sw128_idx(rb + k0 + u, D + d)];
            }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (u < n) av[u] = gsc * sigmoid_fast(av[u]);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (u < n) x = fmaf(av[u], x, bv[u]);
        }
        sCtx[s * D + d] = sC[s * D + d] * x;
      }
      named_sync(1, kComputeThreads);
      PROF_END(8);
    }
    if (T > 0) output_tile(T - 1);
    if (tid == 0) PROF_FLUSH(0);
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0) TRACE_CTA(2);
  if (warp == kMmaWarp) tmem_dealloc(tmem, 2 * kSetCols);
}

int round_up_f(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

// D = 4 runs the same kernel with 16 states, 12 of them zero-padded (their
// weights read as zero): every term they add is an exact zero. (D = 8 has a
// kernel of its own.)
bool fwd_tc16_plan(int K, int SH2, int Dr, FastArgs* a) {
  if (!fast_path_ok(K, SH2, Dr) || (Dr != 16 && Dr != 4)) return false;
  constexpr int D = 16;
  int S_max = kTileRows / K;
  if (S_max > 16) S_max = 16;  // the dots cover two halves of 8 samples, the output four groups of 4
  const int hc = S_max * K * 128, sc = S_max * 128;
  const int off_S = round_up_f(hc, 1024);
  int stage = off_S + sc;
  if (S_max * SH2 * 4 > stage) stage = S_max * SH2 * 4;
  // the projection MMAs read 128 rows of 128 bytes from the start of a stage
  if (kTileRows * 128 > stage) stage = kTileRows * 128;
  stage = round_up_f(stage, 1024);
  const int wbytes = SH2 * 4 * D * 4;
  const int rest = wbytes + 2 * D * SH2 * 4 + kTileRows * 128 + 2 * S_max * D * 4 +
                   static_cast<int>(sizeof(FwdBars)) + 16 + 1024;
  int n_stages = kMaxStages;
  while (n_stages > 2 && n_stages * stage + rest > 227 * 1024) --n_stages;
  int off = n_stages * stage;
  a->off_wt = off;  off += wbytes;
  a->off_wct = off; off += D * SH2 * 4;
  a->off_wo = off;  off += D * SH2 * 4;
  a->off_p = off;   off += kTileRows * 128;
  a->off_cs = off;  off += S_max * D * 4;
  a->off_ctx = off; off += S_max * D * 4;
  off = round_up_f(off, 16);
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
  a->tc = 2;
  a->tmem_cols = 512;
  a->Dr = Dr;
  return a->smem_bytes <= 227 * 1024;
}

cudaError_t launch_fwd_tc16(const FastArgs& a, int grid, cudaStream_t stream) {
  if (a.Dr == 4)
    fwd_tc16_kernel<4><<<grid, kFwdThreads, a.smem_bytes, stream>>>(a);
  else
    fwd_tc16_kernel<16><<<grid, kFwdThreads, a.smem_bytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t prepare_fwd_tc16_kernels(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(fwd_tc16_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fwd_tc16_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  return e;
}

}  // namespace m2scan
