// Device helpers for the m2scan kernels: shared-memory barriers (mbarrier),
// TMA tensor loads, 1-D bulk copies and the bounded wait used everywhere a
// thread waits for an asynchronous copy. Inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace m2scan {

// Bit set in the device error word when a wait gives up (see bounded_wait).
constexpr unsigned kErrWaitTimeout = 1u;
// A wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA engine).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads of the same bytes (a bulk store).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Lets the next kernel of the stream, when it was launched as a programmatic
// dependent (the weight-gradient slot sum), be scheduled once every CTA of
// this grid has signalled or exited. It orders no memory: the dependent
// still waits for this grid to complete (griddepcontrol.wait) before it
// reads anything this grid wrote. Called by one thread after the CTA's last
// barrier, so the dependent's CTAs take SMs only as this grid's CTAs leave.
__device__ __forceinline__ void signal_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Arrives `count` times on the barrier (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar, uint32_t count = 1) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Barrier among `nthreads` threads (a multiple of 32) on hardware barrier `id`.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Non-blocking test of the same condition (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Same test, but a thread whose phase is not complete is suspended until it
// completes or about `hint_ns` nanoseconds have passed, instead of returning
// at once: a waiting warp then takes no issue slots from the working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

// Waits until the barrier phase with the given parity has completed. Gives up
// after kWaitLimitNs, sets kErrWaitTimeout in *err and returns false; the
// caller then carries on (its results are garbage but the kernel ends). Once
// any wait of any kernel has given up (the bit is set), every later wait that
// has to spin gives up at its next check instead of waiting out its own
// limit, so a broken hand-off ends the kernel in about one limit.
// `limit_ns` is kWaitLimitNs everywhere except in the library's self-test of
// this give-up path, which waits on a barrier nobody arrives on.
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, unsigned* err,
                                             unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if ((i & 15u) == 0u) {
      if ((*reinterpret_cast<volatile unsigned*>(err) & kErrWaitTimeout) != 0u) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        atomicOr(err, kErrWaitTimeout);
        return false;
      }
    }
  }
}

// TMA tiled loads, completion signalled on `bar` (complete_tx bytes).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 1-D bulk copy shared -> global, tracked by the bulk async-group of this thread.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every committed bulk store of this thread has finished reading
// shared memory (the source may then be overwritten).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float4 lds4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

__device__ __forceinline__ void sts4(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}

__device__ __forceinline__ float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }

// The optional gate multiplier: every gate is gate_scale * sigmoid(A).
__device__ __forceinline__ float load_gate_scale(const float* p) { return p ? __ldg(p) : 1.0f; }

// sigmoid(a) from e = exp(-|a|) and r = 1 / (1 + e): sigmoid(|a|) = r and
// sigmoid(-|a|) = e r, so neither side cancels. Uses the fast exponential and
// division intrinsics (a few ulp; the layer's results are checked to 1e-4).
__device__ __forceinline__ float sigmoid_fast(float a) {
  const float e = __expf(-fabsf(a));
  const float r = __fdividef(1.0f, 1.0f + e);
  return a >= 0.f ? r : e * r;
}

// sigmoid(a) and its slope sigmoid(a) sigmoid(-a) = e r^2 from one exponential.
__device__ __forceinline__ void sigmoid_and_slope(float a, float& sg, float& slope) {
  const float e = __expf(-fabsf(a));
  const float r = __fdividef(1.0f, 1.0f + e);
  const float er = e * r;
  sg = a >= 0.f ? r : er;
  slope = er * r;
}

// ---------------------------------------------------------------- tcgen05
// Tensor-core MMA with the accumulator in tensor memory (TMEM), operands in
// shared memory as K-major, 128-byte-swizzled tiles (rows of 128 bytes, the
// 16-byte chunk index XORed with the row index mod 8, 8-row groups 1024 bytes
// apart). kind::tf32 reads the top 19 bits of each fp32 operand (the low 13
// mantissa bits are dropped). Operands are split as x = hi + lo with
// hi = tf32_rn(x) stored explicitly and lo = x - hi exact in fp32.

// Element (r, c) of a [rows x 32] fp32 tile in that layout.
__device__ __forceinline__ int sw128_idx(int r, int c) {
  return r * 32 + ((((c >> 2) ^ (r & 7))) << 2) + (c & 3);
}

__device__ __forceinline__ float tf32_trunc(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}

// x rounded to the nearest tf32 value by the conversion instruction (ties away
// from zero); x - tf32_rna(x) is exact and at most half a tf32 ulp.
__device__ __forceinline__ float tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// x rounded to the nearest tf32 value (ties to even on the 13 dropped bits);
// x - tf32_rn(x) is exact, at most half a tf32 ulp and unbiased.
__device__ __forceinline__ float tf32_rn(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0xfffu + ((u >> 13) & 1u);
  return __uint_as_float(u & 0xffffe000u);
}

// Shared-memory matrix descriptor: start address, LBO (unused for swizzled
// K-major tiles), SBO = 1024 bytes between 8-row groups, descriptor version 1,
// layout 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>((1024u >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor: fp32 accumulator, tf32 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of kind::tf32 with either operand MN-major.
__host__ __device__ constexpr uint32_t idesc_tf32_mn(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory descriptor of an MN-major tf32 operand in the layout TMA
// writes with 128-byte swizzle and 32-byte atoms: rows of 128 bytes (32
// elements along M or N) one per K index, groups of 4 rows 512 bytes apart
// (SBO), 32-element blocks along M/N `lbo` bytes apart, layout type 1.
// The next 8 K indices (one MMA step) start 1024 bytes further.
__device__ __forceinline__ uint64_t desc_mn32(uint32_t saddr, uint32_t lbo) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((512u >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(1u) << 61;
  return d;
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same, with the A operand in TMEM (lane = row, one column per K element).
__device__ __forceinline__ void umma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Whole warp: lane l writes 16 consecutive columns of TMEM lane (taddr.lane + l).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

// Whole warp: lane l writes 8 consecutive columns of TMEM lane (taddr.lane + l).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Arrives on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                   "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `ncols` TMEM columns, address written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Whole warp: lane l reads TMEM lane (taddr.lane + l), columns [col, col + N).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float* v);

template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Issue-only variants: results are valid after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Debug timeline (builds with -DM2SCAN_TRACE): CTA 0 records %globaltimer per
// role into the kernel argument's trace buffer (compute thread 0: entries 0.., producer: 1024..,
// MMA issuer: 2048..).
#ifdef M2SCAN_TRACE
#define TRACE_AT(region, tag)                                                    \
  do {                                                                           \
    if (a.trace && blockIdx.x == 0 && trace_n < 1000) {                          \
      a.trace[2 * ((region) * 1024 + trace_n)] = (tag);                          \
      a.trace[2 * ((region) * 1024 + trace_n) + 1] = global_timer_ns();          \
      ++trace_n;                                                                 \
    }                                                                            \
  } while (0)
// Per-CTA marks (entries 4096 + 4 cta + slot): start, end of the prologue, end.
#define TRACE_CTA(slot)                                                              \
  do {                                                                               \
    if (a.trace) a.trace[2 * (4096 + 4 * blockIdx.x + (slot)) + 1] = global_timer_ns(); \
  } while (0)
#else
#define TRACE_AT(region, tag) \
  do {                        \
  } while (0)
#define TRACE_CTA(slot) \
  do {                  \
  } while (0)
#endif

// Debug time accounting (builds with -DM2SCAN_TRACE): a thread adds the time
// between PROF_BEGIN() and PROF_END(slot) to its slot (0..15); PROF_FLUSH(tag)
// writes the slots of CTA 0 to trace entries 3072 + 16 * tag ...
#ifdef M2SCAN_TRACE
#define PROF_DECL                            \
  unsigned long long prof_acc[16] = {};     \
  unsigned long long prof_t0 = 0;           \
  (void)prof_acc;                           \
  (void)prof_t0
#define PROF_BEGIN() (prof_t0 = global_timer_ns())
#define PROF_END(slot) (prof_acc[slot] += global_timer_ns() - prof_t0)
#define PROF_FLUSH(tag)                                                         \
  do {                                                                          \
    if (a.trace && blockIdx.x == 0)                                             \
      for (int pi_ = 0; pi_ < 16; ++pi_) {                                      \
        a.trace[2 * (3072 + 16 * (tag) + pi_)] = 1000 + 16 * (tag) + pi_;       \
        a.trace[2 * (3072 + 16 * (tag) + pi_) + 1] = prof_acc[pi_];             \
      }                                                                         \
  } while (0)
#else
#define PROF_DECL \
  do {            \
  } while (0)
#define PROF_BEGIN() \
  do {               \
  } while (0)
#define PROF_END(slot) \
  do {                 \
  } while (0)
#define PROF_FLUSH(tag) \
  do {                  \
  } while (0)
#endif

}  // namespace m2scan
