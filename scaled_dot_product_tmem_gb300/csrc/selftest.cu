// selftest.cu -- a check of the library's failure path that faults nothing: one
// warp waits on an mbarrier that nobody arrives at, through the same bounded wait
// every pipeline wait uses.  After the wait limit (about one second) it records its
// site code in the device error word and returns, as a stalled pipeline would.
#include <cuda_runtime.h>

#include "attn_kernels.h"
#include "ptx.cuh"

namespace sdpa {

__global__ void __launch_bounds__(32) selftest_wait_kernel(int* err, int site) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  // phase 0 never completes: the wait gives up after the limit and records the site
  mbar_wait_warp(&bar, 0, err, site);
  // once the word is set, a further wait returns at its first check
  mbar_wait_warp(&bar, 0, err, site + 1);
}

int launch_selftest_wait(int* err, int site, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, site);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sdpa
