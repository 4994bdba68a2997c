// Self-test of failure detection: the bounded mbarrier wait that every
// pipeline stage and MMA completion of the apply kernel goes through, run on
// a barrier that never completes (no GPU fault, no hang: the wait gives up
// after its limit and the block raises the timeout flag).
#include "lopt_internal.cuh"
#include "tc_layout.cuh"

namespace lopt {

// Self-test of the bounded wait the kernels use: 32 threads wait on an
// mbarrier that expects two arrivals and gets one, so its phase never
// completes; each wait gives up after limit_ns (or when another thread has
// given up) and the block raises the timeout flag.
__global__ void k_wait_probe(int64_t limit_ns, int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 2);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(&bar);   // one of the two arrivals
  const bool done = mbar_wait_or_abort(&bar, 0u, (uint64_t)limit_ns, &abort_flag);
  __syncthreads();
  if (threadIdx.x == 0) atomicOr(status, (!done && abort_flag) ? kStatusTimeout : 0);
}

cudaError_t launch_wait_probe(int64_t limit_ns, int32_t* status, cudaStream_t s) {
  k_wait_probe<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace lopt
