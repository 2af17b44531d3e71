// diag.cu -- a self-check of the bounded waits every kernel here relies on:
// one wait on an mbarrier that nobody arrives on and one on a global flag
// that nobody sets.  Both must give up after the library's wait limit,
// record PE_DEV_TIMEOUT in the handle's error word and return, leaving the
// context usable.  No asynchronous copy or tensor-core work is in flight
// while they wait, so giving up is safe.
#include "pe_common.cuh"
#include "pe_kernels.h"

namespace pe {

__global__ void bounded_wait_check_kernel(int* flag, int32_t* out, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_fence_init();
  // phase 0 never completes: no thread arrives
  out[0] = mbar_wait(&bar, 0, err) ? 0 : 1;
  // the flag stays 0: nothing publishes it
  out[1] = flag_wait_geq(flag, 1, err) ? 0 : 1;
}

cudaError_t launch_bounded_wait_check(int* flag, int32_t* out, int* err, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  bounded_wait_check_kernel<<<1, 32, 0, s>>>(flag, out, err);
  return cudaGetLastError();
}

}  // namespace pe
