// A kernel whose bounded waits are made to run out, so that the timeout path every kernel of
// the library relies on can be checked without hanging a GPU.  One CTA of four warps takes
// tensor memory like the warp-specialised kernels do; warp 0 waits on an mbarrier that nothing
// will complete with one thread (the MMA-issuer form), warps 1-3 with every lane (the
// warp-uniform form).  Each wait gives up after limit_ns and sets ERR_TIMEOUT in the device
// error word; the CTA then frees its tensor memory and returns.
#include "kernels.cuh"

namespace pisa {
namespace {

__global__ void __launch_bounds__(128, 1) wait_check_kernel(uint64_t limit_ns, uint32_t* err) {
  __shared__ uint64_t never;  // no thread arrives on it and no copy completes it
  __shared__ uint32_t tmem_base_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base_s, 32);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_base_s;
  if (warp == 0) {
    if (lane == 0) mbar_wait(&never, 0, err, limit_ns);
    __syncwarp();
  } else {
    mbar_wait_warp(&never, 0, err, limit_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 32);
  }
}

}  // namespace

cudaError_t launch_wait_check(uint64_t limit_ns, uint32_t* err, cudaStream_t s) {
  wait_check_kernel<<<1, 128, 0, s>>>(limit_ns, err);
  return cudaGetLastError();
}

}  // namespace pisa
