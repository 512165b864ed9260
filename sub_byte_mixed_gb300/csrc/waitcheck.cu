// waitcheck.cu -- a self-check of the library's failure path: the bounded
// mbarrier wait that every pipeline role of the GEMMs uses.  One CTA, two
// waiting threads, on two mbarrier phases that nothing completes:
//   thread 0   waits with the caller's limit; when it runs out it raises the
//              timeout bit of the workspace status word and the CTA's abort
//              flag, and returns;
//   thread 32  waits with four times that limit, and leaves as soon as it
//              sees the abort flag -- the way the GEMM's other roles fall
//              through after one of them gives up.
// out[0] / out[1]: 1 if the thread's wait completed (it cannot), 0 if it gave
// up; out[2]: thread 32's time in the wait, in ns.  Nothing traps: the GPU
// context stays usable and the host reads the status word.
#include "snip_kernels.cuh"

namespace snip {

__global__ void wait_check_kernel(uint32_t* status, uint64_t limit_ns, uint32_t* out) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* flag = &abort_flag;
  if (threadIdx.x == 0) {
    out[0] = mbar_wait_bounded(smem_u32(&bars[0]), 0, flag, status, limit_ns) ? 1u : 0u;
  } else if (threadIdx.x == 32) {
    const uint64_t t0 = globaltimer_ns();
    out[1] = mbar_wait_bounded(smem_u32(&bars[1]), 0, flag, status, 4 * limit_ns) ? 1u : 0u;
    out[2] = (uint32_t)(globaltimer_ns() - t0);
  }
}

cudaError_t launch_wait_check(uint32_t* status, uint64_t limit_ns, uint32_t* out, cudaStream_t st) {
  wait_check_kernel<<<1, 64, 0, st>>>(status, limit_ns, out);
  return cudaGetLastError();
}

}  // namespace snip
