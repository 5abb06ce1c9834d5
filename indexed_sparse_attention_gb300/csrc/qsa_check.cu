// Test hook for the reporting of expired device-side waits: the pipelined
// kernels bound every wait on a shared-memory barrier by a time limit and
// count the waits that gave up; qsa_check_device_status reports them as
// QSA_ERR_TIMEOUT.  This kernel makes one such wait run out on purpose --
// one thread waits on a barrier that nothing completes -- so the reporting
// can be tested without disturbing the GPU: the wait is bounded by the
// global timer and by an iteration cap, and the kernel then ends.
#include "qsa_internal.cuh"

namespace qsa {

namespace {

__device__ int g_selftest_timeouts;

__device__ __forceinline__ uint64_t timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void expired_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = (uint32_t)__cvta_generic_to_shared(&bar);
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(b) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  const uint64_t t0 = timer_ns();
  const uint64_t max_iter = (limit_ns >> 4) + 4096;   // ends even if the timer stood still
  for (uint64_t it = 0; it < max_iter; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(b)
        : "memory");
    if (done) return;   // the phase completed (nothing arrives: never)
    if (timer_ns() - t0 > limit_ns) break;
  }
  atomicAdd(&g_selftest_timeouts, 1);
}

}  // namespace

cudaError_t launch_selftest_wait(int32_t limit_us, cudaStream_t st) {
  expired_wait_kernel<<<1, 1, 0, st>>>((uint64_t)limit_us * 1000u);
  return cudaGetLastError();
}

int selftest_timeouts_take() { return take_counter(g_selftest_timeouts); }

}  // namespace qsa
