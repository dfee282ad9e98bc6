// selftest.cu -- a kernel whose awaited work never completes, to exercise the
// failure path the prefill kernel takes on a timed-out wait: the bounded
// mbarrier wait, the error word, the TMEM release, the early return.
#include "launch.h"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace umma;

__global__ void __launch_bounds__(128, 1) wait_selftest_kernel(unsigned int *err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) bar_init(&bar, 1);  // expects one arrival; none is ever made
  if (warp == 0) tmem_alloc(&tmem_slot, 32);
  fence_before();
  __syncthreads();
  fence_after();
  const bool ok = bar_wait(&bar, 0, limit_ns);
  const int bad = __syncthreads_or(!ok);
  if (bad && threadIdx.x == 0) atomicOr(err, kErrTimeout);
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tmem_slot, 32);
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned int *err, unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 128, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace gdn
