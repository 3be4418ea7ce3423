// Self-test of the device-side failure path shared by the attention kernels:
// one thread waits on an mbarrier that nothing ever arrives at, with the same
// bounded wait (ptx::mbar_wait) the kernels use.  The wait must give up after
// `limit_ns`, report TPK_E_TIMEOUT through *dev_err and let the kernel exit,
// leaving the context usable.  Nothing faults, traps or spins unbounded.
#include "common.cuh"
#include "ptx.cuh"

namespace tpk {
namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);   // expects one arrival; none will come
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns);
    if (!ok && abort_flag && err) atomicExch(err, TPK_E_TIMEOUT);
  }
  __syncthreads();
}

}  // namespace
}  // namespace tpk

extern "C" int tpk_selftest_wait_timeout(uint64_t limit_ns, int32_t* dev_err, void* stream) {
  using namespace tpk;
  if (!dev_err || limit_ns == 0 || limit_ns > kWaitLimitNs) return TPK_E_ARG;
  int st = check_device();
  if (st != TPK_OK) return st;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, dev_err);
  return cuda_status(cudaGetLastError());
}
