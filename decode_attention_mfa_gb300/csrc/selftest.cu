// selftest.cu -- exercises the bounded mbarrier wait that every pipeline wait
// of the decode kernels goes through: one thread waits on an mbarrier that
// nothing arrives on; the wait must give up after its budget, record
// MFA_DEVERR_TIMEOUT and let the kernel return normally.
#include "mfa_device.cuh"

namespace mfa {
namespace {

__global__ void selftest_wait_kernel(uint32_t* err, uint64_t budget_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: no thread arrives and no copy is pending
    (void)mbar_wait(smem_u32(&bar), 0u, budget_ns, &abort_flag, err);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t* err, uint64_t budget_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err, budget_ns);
  return cudaGetLastError();
}

}  // namespace mfa
