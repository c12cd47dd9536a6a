// Forward of the gated temporal scan layer with bf16 activations: h_history,
// h_s2 and h_enriched are bfloat16 in memory, the weights fp32, every sum in
// fp32 (the pages' "bf16 inputs/outputs with fp32 accumulation", which halves
// the bytes of this memory-bound pass). D = 16, SH2 % 64 == 0, SH2 <= 256,
// K <= 128.
//
// Same tiling and roles as the fp32 tensor-core forward: one persistent CTA
// per slot range of samples, tiles of at most 128 rows (S samples x K). Per
// tile:
//   pass 1   the producer warp streams 64-column chunks of h_history and h_s2
//            (TMA boxes of bf16, 128-byte rows, 128-byte swizzle). A bf16
//            value is exact in the tensor core's bf16 input, so one MMA
//            thread forms A|B = h . [W1 | W2] with kind::f16 (bf16 x bf16
//            products, exact in the fp32 accumulator), W = W1 + W2 split
//            into two bf16 parts (16 significant bits; the output is bf16, 8).
//            A stage is free once its MMAs are done (commit) and the compute
//            warps, which form C = h_s2 . W_C on the FMA pipe meanwhile, have
//            read it.
//   scan     x_t = g sigmoid(A_t) x_{t-1} + B_t, one thread per (sample,
//            state); ctx = C x_{K-1}.
//   output   h_enriched = h_s2 + tw ctx . W_O, rounded to bf16, from the
//            tile's h_s2 rows (a stage of their own, after the next tile's
//            chunks), straight to global memory.
#include <cuda_bf16.h>

#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

constexpr int kBfComputeWarps = 8;
constexpr int kBfComputeThreads = kBfComputeWarps * 32;
constexpr int kBfThreads = kBfComputeThreads + 64;
constexpr int kBfProducerWarp = kBfComputeWarps;
constexpr int kBfMmaWarp = kBfComputeWarps + 1;
constexpr int kBfChunk = 64;   // SH2 columns (bf16) per chunk: one 128-byte row
constexpr int kBfStages = 6;   // copy ring depth, at most
constexpr int kBfN = 64;       // MMA N: [W1_A | W1_B | W2_A | W2_B], 16 columns each
constexpr uint32_t kBfSetCols = 64;

struct BfBars {
  uint64_t full[kBfStages];     // producer -> MMA, compute: chunk loaded into stage s
  uint64_t fullo[kBfStages];    // producer -> compute: h_s2 rows loaded into stage s (the MMA
                                // thread skips these items, so they have a barrier of their own)
  uint64_t empty[kBfStages];    // chunk stage free: MMA commit + one arrival per compute warp
  uint64_t outdone[kBfStages];  // compute -> producer: h_s2 item read (one arrival per warp)
  uint64_t mdone[2];            // MMA -> compute: tile t's products (set t & 1) done
  uint64_t accempty[2];         // compute -> MMA: set s read back
  uint32_t tslot;
  uint32_t pad;
};

struct BfPos {
  int i = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++i == n) {
      i = 0;
      ph ^= 1u;
    }
  }
};

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__global__ void __launch_bounds__(kBfThreads, 1) fwd_bf16_kernel(const __grid_constant__ FastArgs a) {
  constexpr int D = 16, TD = 32;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* sW = base + a.off_wt;                         // NC tiles [kBfN][64] bf16, swizzled
  float* sW_Ct = reinterpret_cast<float*>(base + a.off_wct);  // W_C transposed [D][SH2]
  float* sW_O = reinterpret_cast<float*>(base + a.off_wo);    // W_O [D][SH2]
  float* sP = reinterpret_cast<float*>(base + a.off_p);       // A|B [128][32] fp32 swizzled
  float* sC = reinterpret_cast<float*>(base + a.off_cs);      // C [S_max][D]
  float* sCtx = reinterpret_cast<float*>(base + a.off_ctx);   // ctx [S_max][D]
  BfBars* bb = reinterpret_cast<BfBars*>(base + a.off_bar);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, SH2 = a.SH2, S_max = a.S_max, NST = a.n_stages;
  const uint32_t stage_bytes = static_cast<uint32_t>(a.stage_bytes);
  const int NC = SH2 / kBfChunk;
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
  const __nv_bfloat16* hs2 = reinterpret_cast<const __nv_bfloat16*>(a.h_s2);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out0);

  if (tid == kBfProducerWarp * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.tm_hs)) : "memory");
    for (int s = 0; s < NST; ++s) {
      mbar_init(&bb->full[s], 1);
      mbar_init(&bb->fullo[s], 1);
      mbar_init(&bb->empty[s], 1 + kBfComputeWarps);
      mbar_init(&bb->outdone[s], kBfComputeWarps);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bb->mdone[s], 1);
      mbar_init(&bb->accempty[s], 1);
    }
    fence_barrier_init();
  }
  if (warp == kBfMmaWarp) tmem_alloc(&bb->tslot, 2 * kBfSetCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bb->tslot;

  // ---- producer: in round u = 0 .. T the NC chunks of tile u (u < T), then
  // the h_s2 rows of tile u - 1 (u >= 1)
  BfPos lp, rp;
  uint32_t rch = 0, rout = 0;  // bit s: parity of the next empty[s] / outdone[s] phase
  int pn = 0, pround = 0, pit = 0;
  int rround = 0, rit = 0;
  auto round_items = [&](int u) { return (u < T ? NC : 0) + (u >= 1 ? 1 : 0); };
  auto release_one = [&]() {
    if (rit < (rround < T ? NC : 0)) {
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
      tma_load_3d(sp, &a.tm_h, pit * kBfChunk, 0, static_cast<int>(tb0), bar);
      tma_load_2d(sp + a.off_S, &a.tm_hs, pit * kBfChunk, static_cast<int>(tb0), bar);
    } else {
      const long long tb0 = tile_start(pround - 1);
      const int S_t = static_cast<int>(tile_start(pround) - tb0);
      const uint32_t rb = static_cast<uint32_t>(S_t) * SH2 * 2u;
      mbar_arrive_expect_tx(bar, rb);
      bulk_load(sp, hs2 + tb0 * SH2, rb, bar);
    }
    lp.next(NST);
    ++pn;
    if (++pit == round_items(pround)) {
      pit = 0;
      ++pround;
    }
  };

  // ---- weights: the projection B tiles as bf16 pairs W = W1 + W2, and
  // W_C^T, W_O in fp32. Thread = (state quad dq, row j), j fastest.
  constexpr int kWPer = (256 * 4 + kBfThreads - 1) / kBfThreads;
  {
    float4 wa[kWPer], wb[kWPer], wc[kWPer], wo[kWPer];
#pragma unroll
    for (int u = 0; u < kWPer; ++u) {
      const int i = tid + u * kBfThreads;
      const bool ok = i < SH2 * 4;
      const int j = i % SH2, dq = i / SH2;
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      wa[u] = ok ? __ldg(reinterpret_cast<const float4*>(a.W_A + j * D + 4 * dq)) : z;
      wb[u] = ok ? __ldg(reinterpret_cast<const float4*>(a.W_B + j * D + 4 * dq)) : z;
      wc[u] = ok ? __ldg(reinterpret_cast<const float4*>(a.W_C + j * D + 4 * dq)) : z;
      wo[u] = ok ? __ldg(reinterpret_cast<const float4*>(a.W_O) + i) : z;
    }
    if (warp == kBfProducerWarp && lane == 0)
      for (int i = 0; i < NST && pround <= T; ++i) produce_one();
#pragma unroll
    for (int u = 0; u < kWPer; ++u) {
      const int i = tid + u * kBfThreads;
      if (i >= SH2 * 4) break;
      const int j = i % SH2, dq = i / SH2;
      // tile of chunk j / 64: row n (output column), K index jj = j % 64 at
      // byte 2 jj of the row, 16-byte units swizzled with the row
      unsigned char* tile = sW + (j / kBfChunk) * (kBfN * 128);
      const int jj = j % kBfChunk;
      const float va[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
      const float vb[4] = {wb[u].x, wb[u].y, wb[u].z, wb[u].w};
      const float vc[4] = {wc[u].x, wc[u].y, wc[u].z, wc[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = 4 * dq + e;
        const __nv_bfloat16 a1 = __float2bfloat16_rn(va[e]), b1 = __float2bfloat16_rn(vb[e]);
        const __nv_bfloat16 a2 = __float2bfloat16_rn(va[e] - __bfloat162float(a1));
        const __nv_bfloat16 b2 = __float2bfloat16_rn(vb[e] - __bfloat162float(b1));
        const int rows[4] = {d, D + d, TD + d, TD + D + d};
        const __nv_bfloat16 vals[4] = {a1, b1, a2, b2};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int n = rows[r];
          const int off = n * 128 + ((((jj >> 3) ^ (n & 7)) << 4)) + 2 * (jj & 7);
          *reinterpret_cast<__nv_bfloat16*>(tile + off) = vals[r];
        }
        sW_Ct[d * SH2 + j] = vc[e];
      }
      sts4(sW_O + 4 * i, wo[u]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kBfProducerWarp) {
    if (lane == 0) {
      while (pround <= T) produce_one();
    }
  } else if (warp == kBfMmaWarp) {
    // ------------------------------------------------------------- MMA
    // h (bf16) . [W1 | W2] of each chunk as it lands into the tile's set; a
    // commit per chunk frees the stage (with the compute warps' arrivals),
    // one per tile hands the projections over. descriptor + 2 u = 32 u bytes
    // on = 16 u bf16 values (one K step).
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(128, kBfN);
      const uint32_t ring = smem_addr(base);
      const uint32_t w0 = smem_addr(sW);
      BfPos tp;
      uint32_t fph = 0;  // bit s: parity of the next full[s] phase (chunks only)
      for (int t = 0; t < T; ++t) {
        if (t >= 2) bounded_wait(&bb->accempty[t & 1], ((t - 2) >> 1) & 1, a.err);
        const uint32_t acc = tmem + kBfSetCols * static_cast<uint32_t>(t & 1);
        BfPos pm = tp;
        for (int q = 0; q < NC; ++q) {
          bounded_wait(&bb->full[pm.i], (fph >> pm.i) & 1u, a.err);
          fph ^= 1u << pm.i;
          tc_fence_after();
          const uint64_t ad = umma_desc_sw128(ring + static_cast<uint32_t>(pm.i) * stage_bytes);
          const uint64_t bd = umma_desc_sw128(w0 + static_cast<uint32_t>(q * kBfN * 128));
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_bf16(acc, ad + 2u * ks, bd + 2u * ks, idesc, (q > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&bb->empty[pm.i]);
          pm.next(NST);
        }
        umma_commit(&bb->mdone[t & 1]);
        for (int i = 0; i < round_items(t); ++i) tp.next(NST);
      }
    }
  } else {
    // ------------------------------------------------------------- compute
    const int qd = warp & 3, sub = warp >> 2;
    const int row = 32 * qd + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * qd) << 16);
    const float gsc = load_gate_scale(a.gate_scale);
    // C partial dots: thread = (state quad sd_dq, sample pair sd_sp, column
    // octet sd_jo): samples 2 sd_sp, 2 sd_sp + 1 x states 4 sd_dq .. + 3 over
    // 8 columns of each chunk
    const int sd_jo = tid & 7, sd_sp = (tid >> 3) & 7, sd_dq = tid >> 6;
    BfPos ip;
    uint32_t cph = 0, oph = 0;  // bit s: parity of the next full[s] / fullo[s] phase
    auto output_tile = [&](int tt) {
      const long long tb0 = tile_start(tt);
      const int S_t = static_cast<int>(tile_start(tt + 1) - tb0);
      bounded_wait(&bb->fullo[ip.i], (oph >> ip.i) & 1u, a.err);
      oph ^= 1u << ip.i;
      const unsigned char* hs = stage_ptr(ip.i);
      const int st = ip.i;
      ip.next(NST);
      // thread = 4 columns x samples sq, sq + 4, sq + 8, sq + 12
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
            const uint2 hv = *reinterpret_cast<const uint2*>(hs + (static_cast<size_t>(s) * SH2 + 4 * jq) * 2);
            const float y0 = fmaf(a.tw, o[u].x, bf_lo(hv.x)), y1 = fmaf(a.tw, o[u].y, bf_hi(hv.x));
            const float y2 = fmaf(a.tw, o[u].z, bf_lo(hv.y)), y3 = fmaf(a.tw, o[u].w, bf_hi(hv.y));
            __nv_bfloat162 p0 = __floats2bfloat162_rn(y0, y1), p1 = __floats2bfloat162_rn(y2, y3);
            uint2 ov;
            ov.x = *reinterpret_cast<uint32_t*>(&p0);
            ov.y = *reinterpret_cast<uint32_t*>(&p1);
            *reinterpret_cast<uint2*>(out + (tb0 + s) * SH2 + 4 * jq) = ov;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bb->outdone[st]);  // per warp: its reads of the h_s2 rows are done
    };
    for (int t = 0; t < T; ++t) {
      const long long tb0 = tile_start(t);
      const int S_t = static_cast<int>(tile_start(t + 1) - tb0);
      float sacc[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[i][e] = 0.f;
      // ====================================================== pass 1 chunks
      for (int q = 0; q < NC; ++q) {
        float4 w[4][2];  // states 4 sd_dq + e, columns 8 sd_jo .. + 7 of the chunk
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float* wp = sW_Ct + (4 * sd_dq + e) * SH2 + q * kBfChunk + 8 * sd_jo;
          w[e][0] = lds4(wp);
          w[e][1] = lds4(wp + 4);
        }
        bounded_wait(&bb->full[ip.i], (cph >> ip.i) & 1u, a.err);
        cph ^= 1u << ip.i;
        const unsigned char* sp = stage_ptr(ip.i);
        // all 16 rows of the box even past S_max: the reads stay inside shared
        // memory and the sums of missing samples are never stored
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = 2 * sd_sp + i;
          const uint4 hv = *reinterpret_cast<const uint4*>(sp + a.off_S + r * 128 + ((sd_jo ^ (r & 7)) << 4));
          const float h[8] = {bf_lo(hv.x), bf_hi(hv.x), bf_lo(hv.y), bf_hi(hv.y),
                              bf_lo(hv.z), bf_hi(hv.z), bf_lo(hv.w), bf_hi(hv.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float wv[8] = {w[e][0].x, w[e][0].y, w[e][0].z, w[e][0].w,
                                 w[e][1].x, w[e][1].y, w[e][1].z, w[e][1].w};
            float x = sacc[i][e];
#pragma unroll
            for (int k = 0; k < 8; ++k) x = fmaf(h[k], wv[k], x);
            sacc[i][e] = x;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bb->empty[ip.i]);  // per warp: its reads of the stage are done
        ip.next(NST);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int m = 1; m < 8; m <<= 1) sacc[i][e] += __shfl_xor_sync(0xffffffffu, sacc[i][e], m);
      if (sd_jo == 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int s = 2 * sd_sp + i;
          if (s < S_t) sts4(sC + s * D + 4 * sd_dq, make_float4(sacc[i][0], sacc[i][1], sacc[i][2], sacc[i][3]));
        }
      }
      if (t >= 1) output_tile(t - 1);
      // ==================================== projections: TMEM -> shared memory
      bounded_wait(&bb->mdone[t & 1], (t >> 1) & 1, a.err);
      tc_fence_after();
      {
        const int c0 = 16 * sub;  // columns c0 .. c0 + 15 of A|B
        const uint32_t tc0 = lane_base + kBfSetCols * static_cast<uint32_t>(t & 1) + c0;
        uint32_t r0[16], r1[16];
        tmem_ld16_nowait(tc0, r0);       // h . W1
        tmem_ld16_nowait(tc0 + TD, r1);  // h . W2
        tmem_ld_wait();
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r0[i]) + __uint_as_float(r1[i]);
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          sts4(sP + sw128_idx(row, c0 + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
      }
      tc_fence_before();
      named_sync(1, kBfComputeThreads);
      if (tid == 0) mbar_arrive(&bb->accempty[t & 1]);
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
        for (int g8 = 0; g8 < K; g8 += 8) {
          const float* pg = sP + (rb + g8) * 32;
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
      named_sync(1, kBfComputeThreads);
    }
    if (T > 0) output_tile(T - 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kBfMmaWarp) tmem_dealloc(tmem, 2 * kBfSetCols);
}

int round_up_bf(int x, int m) { return (x + m - 1) / m * m; }

}  // namespace

bool fwd_bf16_plan(int K, int SH2, int D, FastArgs* a) {
  if (D != 16 || K < 1 || K > 128 || SH2 < kBfChunk || SH2 > 256 || SH2 % kBfChunk != 0) return false;
  int S_max = kTileRows / K;
  if (S_max > 16) S_max = 16;
  const int hc = S_max * K * 128, sc = S_max * 128;
  const int off_S = round_up_bf(hc, 1024);
  int stage = off_S + sc;
  if (S_max * SH2 * 2 > stage) stage = S_max * SH2 * 2;
  // the projection MMAs read 128 rows of 128 bytes from the start of a stage
  if (kTileRows * 128 > stage) stage = kTileRows * 128;
  stage = round_up_bf(stage, 1024);
  const int wbytes = (SH2 / kBfChunk) * kBfN * 128;
  const int rest = wbytes + 2 * D * SH2 * 4 + kTileRows * 128 + 2 * S_max * D * 4 +
                   static_cast<int>(sizeof(BfBars)) + 16 + 1024;
  int n_stages = kBfStages;
  while (n_stages > 2 && n_stages * stage + rest > 227 * 1024) --n_stages;
  int off = n_stages * stage;
  a->off_wt = off;  off += wbytes;
  a->off_wct = off; off += D * SH2 * 4;
  a->off_wo = off;  off += D * SH2 * 4;
  a->off_p = off;   off += kTileRows * 128;
  a->off_cs = off;  off += S_max * D * 4;
  a->off_ctx = off; off += S_max * D * 4;
  off = round_up_bf(off, 16);
  a->off_bar = off; off += static_cast<int>(sizeof(BfBars));
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
  a->tc = 3;
  a->tmem_cols = 2 * kBfSetCols;
  return a->smem_bytes <= 227 * 1024;
}

cudaError_t launch_fwd_bf16(const FastArgs& a, int grid, cudaStream_t stream) {
  fwd_bf16_kernel<<<grid, kBfThreads, a.smem_bytes, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t prepare_fwd_bf16_kernels(int max_smem) {
  return cudaFuncSetAttribute(fwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

}  // namespace m2scan
