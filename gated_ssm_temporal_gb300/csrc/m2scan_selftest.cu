// Self-test of the bounded barrier wait that every kernel of the library uses
// (m2scan_device.cuh, bounded_wait): one thread initialises a shared-memory
// barrier that expects one arrival, never arrives on it, and waits twice with
// a short limit. The first wait must give up after the limit and set the
// device error bit; the second must then give up at its first check of that
// bit instead of waiting out its own limit. Nothing faults, traps or hangs:
// both waits end, and the kernel returns.
#include "m2scan_device.cuh"
#include "m2scan_internal.h"

namespace m2scan {
namespace {

// out[0], out[1]: nanoseconds each wait took; out[2]: bit 0 / bit 1 set when
// the first / second wait returned false (gave up).
__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(unsigned* err, unsigned long long limit_ns,
                                                             unsigned long long* out) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  const unsigned long long t0 = global_timer_ns();
  const bool r0 = bounded_wait(&bar, 0u, err, limit_ns);
  const unsigned long long t1 = global_timer_ns();
  const bool r1 = bounded_wait(&bar, 0u, err, limit_ns);
  const unsigned long long t2 = global_timer_ns();
  out[0] = t1 - t0;
  out[1] = t2 - t1;
  out[2] = (r0 ? 0ull : 1ull) | (r1 ? 0ull : 2ull);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned* err, unsigned long long limit_ns,
                                         unsigned long long* out, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err, limit_ns, out);
  return cudaGetLastError();
}

}  // namespace m2scan
