// Test support: the library's bounded mbarrier wait, run on its own.
//
// Every tensor-core kernel of the library waits on shared-memory mbarriers (TMA copies landed,
// MMAs complete) through mbar_wait, which gives up after a bounded number of polls; the kernel
// then records TV_ERR_TIMEOUT in err[b] and leaves.  Making such a wait run out inside those
// kernels would need a copy or an MMA that never completes, which a test must not cause.  This
// kernel runs the same mbar_wait on a barrier that nothing arrives on -- no copy, no MMA and no
// other thread is involved -- so a test can drive the wait to its limit and check the status
// and the time it took.  With `arrive` set, the one thread arrives first and the wait succeeds.
#include "tv.h"
#include "tv_async.cuh"
#include "tv_internal.h"
#include "tv_tc.cuh"

namespace tv {
namespace {

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__global__ void bounded_wait_kernel(uint32_t max_polls, int arrive, int32_t* status, int64_t* elapsed_ns) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  mbar_fence_init();
  if (arrive) mbar_arrive(&bar);
  const uint64_t t0 = global_ns();
  const bool done = max_polls ? mbar_wait(&bar, 0, max_polls) : mbar_wait(&bar, 0);
  const uint64_t t1 = global_ns();
  *status = done ? TV_OK : TV_ERR_TIMEOUT;
  *elapsed_ns = (int64_t)(t1 - t0);
}

}  // namespace
}  // namespace tv

extern "C" {

int tv_test_bounded_wait(unsigned max_polls, int arrive, int32_t* status, int64_t* elapsed_ns,
                         tv_stream_t stream) {
  if (status == nullptr || elapsed_ns == nullptr || (reinterpret_cast<uintptr_t>(status) & 3u) ||
      (reinterpret_cast<uintptr_t>(elapsed_ns) & 7u))
    return TV_ERR_INVALID_ARG;
  tv::bounded_wait_kernel<<<1, 1, 0, stream>>>(max_polls, arrive, status, elapsed_ns);
  return tv::cuda_status_of(cudaGetLastError());
}

}  // extern "C"
