// Probe of the bounded wait that every kernel of the library uses on its
// mbarriers.  One thread initialises a barrier that expects one arrival,
// never arrives, and waits on its first phase through mbar_wait_bounded with
// a caller-chosen poll limit.  The wait gives up, the probe records the
// timeout bit in the error word -- the path a kernel takes when a copy or an
// MMA never completes -- and the kernel returns, leaving the context usable.
// Nothing faults and nothing waits without a bound.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

static __device__ unsigned g_probe_error = 0;

__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(uint32_t polls,
                                                                unsigned long long* cycles) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  const long long t0 = clock64();
  const bool done = mbar_wait_bounded(b, 0, polls);  // phase 0 never completes
  const long long t1 = clock64();
  if (cycles) *cycles = static_cast<unsigned long long>(t1 - t0);
  if (!done) atomicOr(&g_probe_error, kErrWaitTimeout);
}

cudaError_t launch_wait_timeout_probe(uint32_t polls, unsigned long long* cycles,
                                      cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(polls, cycles);
  return cudaGetLastError();
}

uint32_t wait_poll_limit() { return kWaitPollLimit; }

// Device address of this unit's error word on the current device.
cudaError_t probe_error_word(unsigned** word) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(word), g_probe_error);
}

unsigned read_probe_error(bool clear) {
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_probe_error, sizeof(word)) != cudaSuccess) return ~0u;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_probe_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
  }
  return word;
}

}  // namespace pkv
