// Fused forward and backward kernels of the gated temporal scan layer (fast
// path: D in {4, 8, 16}, SH2 % 32 == 0, SH2 <= 256, SH2*D <= 4096, K <= 128).
//
// Work split. One persistent CTA per weight-gradient slot; CTA c owns the
// samples [c*B/P, (c+1)*B/P) and walks them in tiles of at most S_max samples
// (S_max*K <= 128 rows). Each tile is processed in three phases:
//
//  pass 1  The tile's h_history rows are streamed through a ring of shared
//          memory stages in chunks of 32 columns of SH2 (TMA, 128-byte
//          swizzle). Each chunk adds its part of the projections
//          A|B = h_history . [W_A|W_B] (registers, FP32 FMA) and of the small
//          projections C = h_s2 . W_C and (backward) d_ctx = dY . W_O^T.
//          ("Custom Kernel Optimization -- cuBLAS Projections +
//          Batch-Parallel Scans", Design 1, Step 1: the same three
//          projections, kept on chip instead of written to HBM.)
//  scan    One thread per (sample, state): x_t = sigmoid(A_t) x_{t-1} + B_t,
//          ctx = C x_{K-1} (design spec Step 2). The backward replays the
//          scan, then runs the reverse scan of the implementation plan's
//          Task 2 and leaves dA|dB in shared memory.
//  pass 2  Forward: h_enriched = h_s2 + tw * ctx . W_O, per group of samples,
//          written back with a 1-D bulk store. Backward: per group of samples,
//          dW_C and dW_O partial sums and d_h_s2 = dY + dC . W_C^T; per block of
//          32 rows, dW_A|dW_B partial sums (registers) and
//          d_h_history = dA|dB . [W_A|W_B]^T (bulk store).
//
// The weight-gradient partial sums of each CTA stay in registers for the
// whole kernel and are written once to the CTA's slot of the workspace; a
// second kernel adds the slots in slot order (the two-phase deterministic
// reduction of "Phase 3 Kernel Optimization Implementation Plan", Task 2).
#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

// Debug timeline (compiled in with -DM2SCAN_TRACE only): thread 0 of CTA 0
// records %globaltimer at phase boundaries into FastArgs::trace.
#ifdef M2SCAN_TRACE
#define M2_TRACE(tag)                                                        \
  do {                                                                       \
    if (a.trace && blockIdx.x == 0 && threadIdx.x == 0 && trace_n < 4096) {  \
      a.trace[2 * trace_n] = (tag);                                          \
      a.trace[2 * trace_n + 1] = global_timer_ns();                          \
      ++trace_n;                                                             \
    }                                                                        \
  } while (0)
#else
#define M2_TRACE(tag) \
  do {                \
  } while (0)
#endif

// Index of W_A|W_B element (j, col) in the swizzled shared copy: rows of 2D
// floats, 16-byte chunk index XORed with bits of j so that both the
// projection loop (one row, four lanes) and the d_h_history loop (rows
// 4*lane + a) read without bank conflicts.
template <int D>
__device__ __forceinline__ int wab_idx(int j, int col) {
  constexpr int NCH = (2 * D) / 4;
  return j * (2 * D) + ((((col >> 2) ^ ((j >> 2) & (NCH - 1)))) << 2) + (col & 3);
}

template <int NQ>
__device__ __forceinline__ void load_run(const float* p, float* v) {
  if constexpr (NQ == 4) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else if constexpr (NQ == 2) {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x; v[1] = t.y;
  } else {
    v[0] = p[0];
  }
}

__device__ __forceinline__ float comp(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ float dot4(const float4& a, const float4& b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

template <int D, bool BWD, bool TC>
__global__ void __launch_bounds__(kThreads, 1) fast_kernel(const __grid_constant__ FastArgs a) {
  constexpr int NQ = D / 4;    // A (and B) columns per lane in the projection loop
  constexpr int TD = 2 * D;    // columns of A|B
  constexpr int NCH = TD / 4;  // 16-byte chunks per A|B row
  constexpr int PS = TD + 4;   // row stride of the A|B tile (padded)
  constexpr int KQN = TD / 8;  // groups of 8 columns in dW_A|dW_B

  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  float* sW_AB = reinterpret_cast<float*>(base + a.off_wab);
  float* sW_Ct = reinterpret_cast<float*>(base + a.off_wct);  // W_C transposed [D][SH2]
  float* sW_O = reinterpret_cast<float*>(base + a.off_wo);    // W_O [D][SH2]
  float* sP = reinterpret_cast<float*>(base + a.off_p);       // A|B tile [128][PS]
  float* sC = reinterpret_cast<float*>(base + a.off_cs);      // C [S_max][D]
  float* sCtx = reinterpret_cast<float*>(base + a.off_ctx);   // ctx [S_max][D]
  float* sDctx = reinterpret_cast<float*>(base + a.off_dctx); // d_ctx [S_max][D]
  float* sDC = reinterpret_cast<float*>(base + a.off_dc);     // dC [S_max][D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + a.off_bar);
  // tensor-core path
  float* sWt = reinterpret_cast<float*>(base + a.off_wt);     // NC tiles [2D][32], swizzled
  float* sWtlo = reinterpret_cast<float*>(base + a.off_wtlo);
  uint64_t* mbars = reinterpret_cast<uint64_t*>(base + a.off_mbar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(base + a.off_tslot);
  const int NST = a.n_stages;
  // loads are issued this many items ahead (a stage is free once the threads
  // have read it: the MMAs read their operands from TMEM and the weight tiles)
  const int PF = NST;


  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int trace_n = 0;
  (void)trace_n;
  M2_TRACE(1);
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max, SG = a.SG;
  const int NC = SH2 / kChunk;
  // TMEM columns: [0, NC*2D) one accumulator per chunk, then the corrections,
  // then two A-operand buffers of 64 columns (32 hi + 32 lo) at a_col0
  const uint32_t a_col0 = static_cast<uint32_t>((NC + 1) * TD);
  const long long B = a.B;
  const int P = gridDim.x, cta = blockIdx.x;
  const long long cb0 = B * cta / P;
  const int n_c = static_cast<int>(B * (cta + 1) / P - cb0);
  const int T = (n_c + S_max - 1) / S_max;

  // tile i holds base (+1 for the first `extra` tiles) samples: no division per tile
  const int t_base = n_c / T, t_extra = n_c - (n_c / T) * T;
  auto tile_start = [&](int i) -> long long {
    return cb0 + static_cast<long long>(i) * t_base + (i < t_extra ? i : t_extra);
  };
  auto tile_items = [&](int S_t) -> int {
    int n = NC + (S_t + SG - 1) / SG;
    if (BWD) n += (S_t * K + kRowsPerItem - 1) / kRowsPerItem;
    return n;
  };

  // ---- copy producer (thread 0): issues the loads of the next item into the
  // ring, PF items ahead of the consumers.
  int pf_tile = 0, pf_idx = 0, pf_seq = 0;
  auto issue_next = [&]() {
    if (pf_tile >= T) return;
    const long long tb0 = tile_start(pf_tile);
    const int S_t = static_cast<int>(tile_start(pf_tile + 1) - tb0);
    const int NSI = (S_t + SG - 1) / SG;
    const int stage = pf_seq % NST;
    unsigned char* st = base + static_cast<size_t>(stage) * a.stage_bytes;
    uint64_t* bar = &bars[stage];
    const int idx = pf_idx;
    M2_TRACE(60);
    if (idx < NC) {
      const uint32_t bytes = a.hc_bytes + a.sc_bytes * (BWD ? 2 : 1);
      mbar_arrive_expect_tx(bar, bytes);
      M2_TRACE(61);
      tma_load_3d(st, &a.tm_h, idx * kChunk, 0, static_cast<int>(tb0), bar);
      tma_load_2d(st + a.off_S, &a.tm_hs, idx * kChunk, static_cast<int>(tb0), bar);
      if (BWD) tma_load_2d(st + a.off_G, &a.tm_g, idx * kChunk, static_cast<int>(tb0), bar);
      M2_TRACE(62);
    } else if (idx < NC + NSI) {
      const int s0 = (idx - NC) * SG;
      const int ns = min(SG, S_t - s0);
      const uint32_t rb = static_cast<uint32_t>(ns) * SH2 * 4u;
      mbar_arrive_expect_tx(bar, BWD ? 2u * rb : rb);
      bulk_load(st, a.h_s2 + (tb0 + s0) * SH2, rb, bar);
      if (BWD) bulk_load(st + static_cast<size_t>(SG) * SH2 * 4, a.g + (tb0 + s0) * SH2, rb, bar);
    } else {
      const int r0 = (idx - NC - NSI) * kRowsPerItem;
      const int nr = min(kRowsPerItem, S_t * K - r0);
      const uint32_t rb = static_cast<uint32_t>(nr) * SH2 * 4u;
      mbar_arrive_expect_tx(bar, rb);
      bulk_load(st, a.h_history + (tb0 * K + r0) * SH2, rb, bar);
    }
    ++pf_seq;
    if (++pf_idx == tile_items(S_t)) {
      pf_idx = 0;
      ++pf_tile;
    }
  };

  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_hs)) : "memory");
    if (BWD) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_g)) : "memory");
    for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
    if (TC)
      for (int s = 0; s < 2; ++s) mbar_init(&mbars[s], 1);
    fence_barrier_init();
  }
  if (TC && warp == 0) tmem_alloc(tslot, a.tmem_cols);
  if (TC) tc_fence_before();
  __syncthreads();
  if (TC) tc_fence_after();
  const uint32_t tmem_acc = TC ? *tslot : 0u;
  if (tid == 0)
    for (int s = 0; s < PF; ++s) issue_next();

  // weights into shared memory (overlaps the first loads); SH2*D <= 4096 gives at
  // most 16 elements per thread: all global loads are issued before any store
  constexpr int kWPer = 4096 / kThreads;
  float wa[kWPer], wb[kWPer], wc[kWPer], wo[kWPer];
#pragma unroll
  for (int u = 0; u < kWPer; ++u) {
    const int i = tid + u * kThreads;
    const bool ok = i < SH2 * D;
    wa[u] = ok ? __ldg(a.W_A + i) : 0.f;
    wb[u] = ok ? __ldg(a.W_B + i) : 0.f;
    wc[u] = ok ? __ldg(a.W_C + i) : 0.f;
    wo[u] = ok ? __ldg(a.W_O + i) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < kWPer; ++u) {
    const int i = tid + u * kThreads;
    if (i >= SH2 * D) break;
    const int j = i / D, d = i - j * D;
    if (!TC || BWD) {
      sW_AB[wab_idx<D>(j, d)] = wa[u];
      sW_AB[wab_idx<D>(j, D + d)] = wb[u];
    }
    if (TC) {  // B operand of the projection MMA: tile q = [2D rows][32 columns of SH2]
      const int tq = (j >> 5) * TD * 32, jj = j & 31;
      const float ha = tf32_rn(wa[u]), hb = tf32_rn(wb[u]);
      sWt[tq + sw128_idx(d, jj)] = ha;
      sWtlo[tq + sw128_idx(d, jj)] = wa[u] - ha;
      sWt[tq + sw128_idx(D + d, jj)] = hb;
      sWtlo[tq + sw128_idx(D + d, jj)] = wb[u] - hb;
    }
    sW_Ct[d * SH2 + j] = wc[u];
    sW_O[i] = wo[u];
  }
  if (TC) fence_proxy_async_smem();
  __syncthreads();
  M2_TRACE(2);

  // ---- per-thread ownership of weight-gradient entries (backward)
  const int pjq_ab = tid / KQN, pkq = tid - (tid / KQN) * KQN;  // dW_A|dW_B: 4 rows x 8 cols
  const bool own_ab = pjq_ab < SH2 / 4;
  const int pjq_c = tid / NQ, pdq = tid - (tid / NQ) * NQ;      // dW_C, dW_O: 4 x 4
  const bool own_c = pjq_c < SH2 / 4;
  float accAB[4][8], accC[4][4], accO[4][4];
  if constexpr (BWD) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int k = 0; k < 8; ++k) accAB[i][k] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) accC[i][k] = accO[i][k] = 0.f;
    }
  }

  const int r_lane = lane >> 2, c_lane = lane & 3;
  const int wrow0 = 32 * (warp & 3);
  const int jh = warp >> 2;
  const int sd_jo = tid & 3;
  const int sd_dq = (tid >> 2) % NQ;
  const int sd_s = (tid >> 2) / NQ;

  int seq = 0;
  int mma_id = 0;  // chunks whose MMAs have been issued (all threads count)
  for (int tile = 0; tile < T; ++tile) {
    const long long tb0 = tile_start(tile);
    const int S_t = static_cast<int>(tile_start(tile + 1) - tb0);
    const int R_t = S_t * K;
    const int NSI = (S_t + SG - 1) / SG;

    // ================= pass 1: projections over 32-column chunks =========
    const bool gemm_active = wrow0 < R_t;
    const bool sd_active = sd_s < S_t;
    float acc[4][2 * NQ];
#pragma unroll
    for (int rg = 0; rg < 4; ++rg)
#pragma unroll
      for (int k = 0; k < 2 * NQ; ++k) acc[rg][k] = 0.f;
    float cacc[4] = {0.f, 0.f, 0.f, 0.f}, dacc[4] = {0.f, 0.f, 0.f, 0.f};

    for (int q = 0; q < NC; ++q, ++seq) {
      const int stage = seq % NST;
      M2_TRACE(10);
      bounded_wait(&bars[stage], (seq / NST) & 1, a.err);
      M2_TRACE(11);
      const float* Hc = reinterpret_cast<const float*>(base + static_cast<size_t>(stage) * a.stage_bytes);
      const float* Sc = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(Hc) + a.off_S);
      const float* Gc = reinterpret_cast<const float*>(reinterpret_cast<const unsigned char*>(Hc) + a.off_G);
      if constexpr (TC) {
        // A operand into TMEM: thread = tile row (lane), warps 0-3 take columns
        // 0-15 of the chunk and warps 4-7 columns 16-31; h = hi + lo with
        // hi = tf32_rn(h). Rows past the h box hold don't-care values.
        // The MMAs of chunk mma_id-2 read this TMEM buffer: wait for them.
        if (mma_id >= 2) bounded_wait(&mbars[mma_id & 1], ((mma_id - 2) >> 1) & 1, a.err);
        const int row = 32 * (warp & 3) + lane, half = warp >> 2;
        float hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = lds4(Hc + row * 32 + ((((4 * half + i) ^ (row & 7))) << 2));
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            hi[4 * i + e] = tf32_rn(vv[e]);
            lo[4 * i + e] = vv[e] - hi[4 * i + e];
          }
        }
        const uint32_t ta = tmem_acc + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + a_col0 +
                            64u * (mma_id & 1) + 16u * half;
        tmem_st16(ta, hi);
        tmem_st16(ta + 32, lo);
        tmem_st_wait();
        tc_fence_before();
      } else if (gemm_active) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jj = 16 * jh + 4 * u;  // first column (within the chunk) of this step
          float4 hv[4];
#pragma unroll
          for (int rg = 0; rg < 4; ++rg) {
            const int row = wrow0 + r_lane + 8 * rg;
            hv[rg] = lds4(Hc + row * 32 + (((jj >> 2) ^ (row & 7)) << 2));
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int j = q * kChunk + jj + i;
            float wa[NQ], wb[NQ];
            load_run<NQ>(sW_AB + wab_idx<D>(j, c_lane * NQ), wa);
            load_run<NQ>(sW_AB + wab_idx<D>(j, D + c_lane * NQ), wb);
#pragma unroll
            for (int rg = 0; rg < 4; ++rg) {
              const float hval = comp(hv[rg], i);
#pragma unroll
              for (int k = 0; k < NQ; ++k) {
                acc[rg][k] = fmaf(hval, wa[k], acc[rg][k]);
                acc[rg][NQ + k] = fmaf(hval, wb[k], acc[rg][NQ + k]);
              }
            }
          }
        }
      }
      if (sd_active) {
        const int s = sd_s, ch0 = 2 * sd_jo;
        const float4 h0 = lds4(Sc + s * 32 + ((ch0 ^ (s & 7)) << 2));
        const float4 h1 = lds4(Sc + s * 32 + (((ch0 + 1) ^ (s & 7)) << 2));
        const int jb = q * kChunk + 8 * sd_jo;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float* w = sW_Ct + (4 * sd_dq + i) * SH2 + jb;
          cacc[i] = dot4(h1, lds4(w + 4), dot4(h0, lds4(w), cacc[i]));
        }
        if constexpr (BWD) {
          const float4 g0 = lds4(Gc + s * 32 + ((ch0 ^ (s & 7)) << 2));
          const float4 g1 = lds4(Gc + s * 32 + (((ch0 + 1) ^ (s & 7)) << 2));
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float* w = sW_O + (4 * sd_dq + i) * SH2 + jb;
            dacc[i] = dot4(g1, lds4(w + 4), dot4(g0, lds4(w), dacc[i]));
          }
        }
      }
      M2_TRACE(12);
      __syncthreads();
      M2_TRACE(13);
      if (tid == 0) {
        if constexpr (TC) {
          // A|B = sum over chunks of h_hi.W_hi, plus the corrections
          // h_hi.W_lo + h_lo.W_hi (3 x tf32, hi = tf32_rn, lo = remainder). Each chunk's main
          // product has its own TMEM accumulator (columns q*2D) and the corrections
          // share one (columns NC*2D): few accumulation steps per accumulator keep
          // the tensor cores' accumulation error at the level of fp32 FMA.
          tc_fence_after();
          M2_TRACE(14);
          issue_next();  // the stage just read is free
          M2_TRACE(15);
          constexpr uint32_t idesc = umma_idesc_tf32(128, TD);
          const uint32_t ah = tmem_acc + a_col0 + 64u * (mma_id & 1), al = ah + 32u;
          const uint32_t bh = smem_addr(sWt + q * TD * 32), bl = smem_addr(sWtlo + q * TD * 32);
          const uint32_t d_main = tmem_acc + q * TD, d_corr = tmem_acc + NC * TD;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t o = 32u * ks;
            umma_tf32_ta(d_main, ah + 8u * ks, umma_desc_sw128(bh + o), idesc, ks != 0);
            umma_tf32_ta(d_corr, ah + 8u * ks, umma_desc_sw128(bl + o), idesc, (q | ks) != 0);
            umma_tf32_ta(d_corr, al + 8u * ks, umma_desc_sw128(bh + o), idesc, 1u);
          }
          M2_TRACE(16);
          umma_commit(&mbars[mma_id & 1]);
          M2_TRACE(17);
        } else {
          issue_next();
        }
      }
      if (TC) ++mma_id;
    }

    M2_TRACE(20);
    // ---- A|B tile into shared memory; finish C, d_ctx
    if constexpr (TC) {
      const int last = mma_id - 1;
      bounded_wait(&mbars[last & 1], (last >> 1) & 1, a.err);
      tc_fence_after();
      float v[D], w[D];
      const int c0 = (warp >> 2) * D;  // warps 0-3: A columns, warps 4-7: B columns
      const uint32_t lane_base = tmem_acc + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + c0;
      tmem_ld<D>(lane_base, v);
      for (int qq = 1; qq < NC; ++qq) {  // fixed order: chunk 0, 1, ..., then the corrections
        tmem_ld<D>(lane_base + qq * TD, w);
#pragma unroll
        for (int i = 0; i < D; ++i) v[i] += w[i];
      }
      tmem_ld<D>(lane_base + NC * TD, w);
#pragma unroll
      for (int i = 0; i < D; ++i) v[i] += w[i];
      float* pr = sP + (32 * (warp & 3) + lane) * PS + c0;
#pragma unroll
      for (int i = 0; i < D; i += 4) sts4(pr + i, make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
      tc_fence_before();
    }
    if (!TC && gemm_active && jh == 1) {
#pragma unroll
      for (int rg = 0; rg < 4; ++rg) {
        float* pr = sP + (wrow0 + r_lane + 8 * rg) * PS;
#pragma unroll
        for (int k = 0; k < NQ; ++k) {
          pr[c_lane * NQ + k] = acc[rg][k];
          pr[D + c_lane * NQ + k] = acc[rg][NQ + k];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cacc[i] += __shfl_xor_sync(0xffffffffu, cacc[i], 1);
      cacc[i] += __shfl_xor_sync(0xffffffffu, cacc[i], 2);
      if constexpr (BWD) {
        dacc[i] += __shfl_xor_sync(0xffffffffu, dacc[i], 1);
        dacc[i] += __shfl_xor_sync(0xffffffffu, dacc[i], 2);
      }
    }
    if (sd_active && sd_jo == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sC[sd_s * D + 4 * sd_dq + i] = cacc[i];
        if constexpr (BWD) sDctx[sd_s * D + 4 * sd_dq + i] = a.tw * dacc[i];
      }
    }
    __syncthreads();
    if (!TC && gemm_active && jh == 0) {
#pragma unroll
      for (int rg = 0; rg < 4; ++rg) {
        float* pr = sP + (wrow0 + r_lane + 8 * rg) * PS;
#pragma unroll
        for (int k = 0; k < NQ; ++k) {
          pr[c_lane * NQ + k] = acc[rg][k] + pr[c_lane * NQ + k];
          pr[D + c_lane * NQ + k] = acc[rg][NQ + k] + pr[D + c_lane * NQ + k];
        }
      }
    }
    __syncthreads();

    M2_TRACE(21);
    // ================= scan (one thread per sample and state) ============
    if (tid < S_t * D) {
      const int s = tid / D, d = tid - (tid / D) * D;
      float* pcol = sP + s * K * PS;
      const float gsc = load_gate_scale(a.gate_scale);
      float x = 0.f;
      if constexpr (!BWD) {
        for (int t = 0; t < K; ++t) {
          const float* pr = pcol + t * PS;
          x = fmaf(gsc * sigmoidf_(pr[d]), x, pr[D + d]);
        }
        sCtx[s * D + d] = sC[s * D + d] * x;
      } else {
        for (int t = 0; t < K; ++t) {  // replay: A stays in place, B_t is replaced by x_t
          float* pr = pcol + t * PS;
          x = fmaf(gsc * sigmoidf_(pr[d]), x, pr[D + d]);
          pr[D + d] = x;
        }
        const float Cv = sC[s * D + d], dctx = sDctx[s * D + d];
        sCtx[s * D + d] = Cv * x;
        sDC[s * D + d] = dctx * x;
        float dx = dctx * Cv;  // gradient with respect to x_{K-1}
        for (int t = K - 1; t >= 0; --t) {
          float* pr = pcol + t * PS;
          const float at = pr[d];
          const float sg0 = sigmoidf_(at);
          // sigmoid'(a) = sigmoid(a) * sigmoid(-a): 1 - sigmoid(a) taken as sigmoid(-a)
          // keeps full relative precision when the gate is saturated near 1.
          const float dsg = gsc * (sg0 * sigmoidf_(-at));
          const float sg = gsc * sg0;
          const float xprev = t > 0 ? pr[D + d - PS] : 0.f;
          pr[D + d] = dx;                   // dB_t
          pr[d] = dx * xprev * dsg;         // dA_t
          dx *= sg;
        }
      }
    }
    __syncthreads();

    M2_TRACE(22);
    // ================= pass 2a: per-sample outputs =======================
    const int njq = SH2 / 4;
    for (int k = 0; k < NSI; ++k, ++seq) {
      const int stage = seq % NST;
      M2_TRACE(30);
      bounded_wait(&bars[stage], (seq / NST) & 1, a.err);
      M2_TRACE(31);
      float* hsb = reinterpret_cast<float*>(base + static_cast<size_t>(stage) * a.stage_bytes);
      const int s0 = k * SG, ns = min(SG, S_t - s0);
      const int nit = ((ns + 3) / 4) * njq;
      if constexpr (!BWD) {
        // h_enriched = h_s2 + tw * ctx . W_O, in place over the h_s2 rows
        for (int it = tid; it < nit; it += kThreads) {
          const int jq = it % njq, sq = it / njq;
          float o[4][4];
#pragma unroll
          for (int si = 0; si < 4; ++si)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[si][e] = 0.f;
          for (int d = 0; d < D; ++d) {
            const float4 w = lds4(sW_O + d * SH2 + 4 * jq);
#pragma unroll
            for (int si = 0; si < 4; ++si) {
              const int s = min(4 * sq + si, ns - 1);
              const float cx = sCtx[(s0 + s) * D + d];
              o[si][0] = fmaf(cx, w.x, o[si][0]);
              o[si][1] = fmaf(cx, w.y, o[si][1]);
              o[si][2] = fmaf(cx, w.z, o[si][2]);
              o[si][3] = fmaf(cx, w.w, o[si][3]);
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
      } else {
        float* gb = hsb + static_cast<size_t>(SG) * SH2;
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
        __syncthreads();  // h_s2 rows no longer needed: d_h_s2 goes there
        for (int it = tid; it < nit; it += kThreads) {
          const int jq = it % njq, sq = it / njq;
          float o[4][4];
#pragma unroll
          for (int si = 0; si < 4; ++si) {
            const int s = min(4 * sq + si, ns - 1);
            const float4 gv = lds4(gb + s * SH2 + 4 * jq);
            o[si][0] = gv.x; o[si][1] = gv.y; o[si][2] = gv.z; o[si][3] = gv.w;
          }
          for (int d = 0; d < D; ++d) {
            const float4 w = lds4(sW_Ct + d * SH2 + 4 * jq);
#pragma unroll
            for (int si = 0; si < 4; ++si) {
              const int s = min(4 * sq + si, ns - 1);
              const float dcv = sDC[(s0 + s) * D + d];
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
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        float* dst = (BWD ? a.out1 : a.out0) + (tb0 + s0) * SH2;
        M2_TRACE(32);
        bulk_store(dst, hsb, static_cast<uint32_t>(ns) * SH2 * 4u);
        bulk_commit();
        bulk_wait_read_all();
        M2_TRACE(33);
        issue_next();
      }
    }

    // ================= pass 2b: per-row outputs (backward) ===============
    if constexpr (BWD) {
      const int NRI = (R_t + kRowsPerItem - 1) / kRowsPerItem;
      for (int k = 0; k < NRI; ++k, ++seq) {
        const int stage = seq % NST;
        M2_TRACE(40);
        bounded_wait(&bars[stage], (seq / NST) & 1, a.err);
        M2_TRACE(41);
        float* hb = reinterpret_cast<float*>(base + static_cast<size_t>(stage) * a.stage_bytes);
        const int r0 = k * kRowsPerItem, nr = min(kRowsPerItem, R_t - r0);
        // dW_A | dW_B partial sums: sum over rows of h[row, j] * dAB[row, col]
        if (own_ab) {
          const float* prow = sP + r0 * PS + 8 * pkq;
          const float* hrow = hb + 4 * pjq_ab;
          for (int r = 0; r < nr; ++r) {
            const float4 hv = lds4(hrow + r * SH2);
            const float4 p0 = lds4(prow + r * PS), p1 = lds4(prow + r * PS + 4);
            const float hvv[4] = {hv.x, hv.y, hv.z, hv.w};
            const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int e = 0; e < 8; ++e) accAB[i][e] = fmaf(hvv[i], pv[e], accAB[i][e]);
          }
        }
        // d_h_history rows: dA|dB . [W_A|W_B]^T, 8 rows x 4 columns per lane
        const int rg0 = 8 * (warp & 3);
        const int jd = 128 * (warp >> 2) + 4 * lane;
        const bool dh_active = rg0 < nr && jd < SH2;
        float dh[8][4];
        if (dh_active) {
#pragma unroll
          for (int rr = 0; rr < 8; ++rr)
#pragma unroll
            for (int e = 0; e < 4; ++e) dh[rr][e] = 0.f;
#pragma unroll
          for (int kk = 0; kk < TD / 4; ++kk) {
            float4 w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = jd + e;
              w[e] = lds4(sW_AB + j * TD + ((kk ^ ((j >> 2) & (NCH - 1))) << 2));
            }
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
              const float4 pv = lds4(sP + (r0 + rg0 + rr) * PS + 4 * kk);
#pragma unroll
              for (int e = 0; e < 4; ++e) dh[rr][e] = dot4(pv, w[e], dh[rr][e]);
            }
          }
        }
        __syncthreads();  // every read of the h rows is done: d_h_history goes there
        if (dh_active) {
#pragma unroll
          for (int rr = 0; rr < 8; ++rr)
            if (rg0 + rr < nr)
              sts4(hb + (rg0 + rr) * SH2 + jd, make_float4(dh[rr][0], dh[rr][1], dh[rr][2], dh[rr][3]));
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
          M2_TRACE(42);
          bulk_store(a.out0 + (tb0 * K + r0) * SH2, hb, static_cast<uint32_t>(nr) * SH2 * 4u);
          bulk_commit();
          bulk_wait_read_all();
          M2_TRACE(43);
          issue_next();
        }
      }
    }
  }

  if constexpr (BWD) {
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
  }
  M2_TRACE(50);
  if (tid == 0) bulk_wait_all();
  if constexpr (TC) {
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_acc, a.tmem_cols);
  }
  if constexpr (BWD) {
    __syncthreads();
    if (tid == 0) signal_dependent_launch();
  }
}

}  // namespace

bool fast_path_ok(int K, int SH2, int D) {
  return (D == 4 || D == 8 || D == 16) && SH2 >= kChunk && SH2 % kChunk == 0 && SH2 <= 256 &&
         SH2 * D <= 4096 && K >= 1 && K <= kTileRows;
}

// The TC variant of this kernel is not used (the forward has its own
// warp-specialised tensor-core kernel).
bool tc_path_ok(bool bwd, int D) {
  (void)bwd;
  (void)D;
  return false;
}

static int round_up(int x, int m) { return (x + m - 1) / m * m; }

bool fast_plan(bool bwd, int K, int SH2, int D, FastArgs* a) {
  if (!fast_path_ok(K, SH2, D)) return false;
  const bool tc = tc_path_ok(bwd, D);
  int S_max = kTileRows / K;
  if (S_max > 32) S_max = 32;
  if (S_max > kThreads / D) S_max = kThreads / D;
  const int SG = bwd ? (S_max < kMaxSampleItem ? S_max : kMaxSampleItem) : S_max;
  const int hc = S_max * K * 128, sc = S_max * 128;
  const int off_S = round_up(hc, 1024);
  const int off_G = off_S + round_up(sc, 1024);
  const int chunk_end = bwd ? off_G + round_up(sc, 1024) : off_G;
  int stage = chunk_end;
  const int sample_bytes = (bwd ? 2 : 1) * SG * SH2 * 4;
  if (sample_bytes > stage) stage = sample_bytes;
  if (bwd && kRowsPerItem * SH2 * 4 > stage) stage = kRowsPerItem * SH2 * 4;
  if (kTileRows * 128 > stage) stage = kTileRows * 128;  // a 128-row tile is always read
  stage = round_up(stage, 1024);
  // the rest of the plan does not depend on the ring depth: lay it out after a
  // ring of kMaxStages and shrink the ring if that does not fit
  int rest = 0;
  if (tc) rest += 2 * SH2 * 2 * D * 4;
  if (!tc || bwd) rest += SH2 * 2 * D * 4;
  rest += 2 * D * SH2 * 4 + kTileRows * (2 * D + 4) * 4 + 4 * S_max * D * 4 + 1024 + 1024;
  int n_stages = tc ? kMaxStages : kStages;
  while (n_stages > 2 && n_stages * stage + rest > 227 * 1024) --n_stages;
  int off = n_stages * stage;
  a->off_hlo = a->off_wt = a->off_wtlo = off;
  if (tc) {
    a->off_wt = off;   off += SH2 * 2 * D * 4;
    a->off_wtlo = off; off += SH2 * 2 * D * 4;
  }
  a->off_wab = off;
  if (!tc || bwd) off += SH2 * 2 * D * 4;
  a->off_wct = off; off += D * SH2 * 4;
  a->off_wo = off;  off += D * SH2 * 4;
  a->off_p = off;   off += kTileRows * (2 * D + 4) * 4;
  a->off_cs = off;  off += S_max * D * 4;
  a->off_ctx = off; off += S_max * D * 4;
  a->off_dctx = off; off += S_max * D * 4;
  a->off_dc = off;  off += S_max * D * 4;
  off = round_up(off, 16);
  a->off_bar = off;  off += kMaxStages * 8;
  a->off_mbar = off; off += 2 * 8;
  a->off_tslot = off; off += 16;
  a->smem_bytes = off + 1024;  // slack to align the start to 1024 bytes
  a->S_max = S_max;
  a->SG = SG;
  a->stage_bytes = stage;
  a->hc_bytes = hc;
  a->sc_bytes = sc;
  a->off_S = off_S;
  a->off_G = off_G;
  a->K = K;
  a->SH2 = SH2;
  a->n_stages = n_stages;
  a->tc = tc ? 1 : 0;
  // TMEM: one accumulator block per SH2 chunk, one for the correction terms and
  // two 64-column A-operand buffers
  int cols = 32;
  while (cols < (SH2 / kChunk + 1) * 2 * D + 128) cols *= 2;
  a->tmem_cols = cols;
  return a->smem_bytes <= 227 * 1024;
}

template <int D, bool BWD, bool TC>
static cudaError_t launch_one(const FastArgs& a, int grid, cudaStream_t stream) {
  static_assert(D % 4 == 0, "D must be a multiple of 4");
  fast_kernel<D, BWD, TC><<<grid, kThreads, a.smem_bytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fast(bool bwd, int D, const FastArgs& a, int grid, cudaStream_t stream) {
  switch (D) {
    case 4: return bwd ? launch_one<4, true, false>(a, grid, stream) : launch_one<4, false, false>(a, grid, stream);
    case 8: return bwd ? launch_one<8, true, false>(a, grid, stream) : launch_one<8, false, false>(a, grid, stream);
    case 16: return bwd ? launch_one<16, true, false>(a, grid, stream) : launch_one<16, false, false>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t prepare_fast_kernels(int max_smem) {
  cudaError_t e = cudaSuccess;
#define M2_SET(DD, BB, TT)                                                                       \
  if (e == cudaSuccess)                                                                          \
    e = cudaFuncSetAttribute(fast_kernel<DD, BB, TT>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             max_smem);
  M2_SET(4, false, false) M2_SET(4, true, false) M2_SET(8, false, false) M2_SET(8, true, false)
  M2_SET(16, false, false) M2_SET(16, true, false)
#undef M2_SET
  return e;
}

}  // namespace m2scan
