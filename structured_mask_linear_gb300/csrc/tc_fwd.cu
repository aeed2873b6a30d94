// Tensor-core (tcgen05) path of the log-linear Mamba-2 forward.  Not enabled yet:
// tc_supported() returns false and every shape runs the generic path.
#include <cuda_runtime.h>

#include "ll_internal.cuh"
#include "ptx.cuh"

namespace ll {

namespace {

// One thread waits on an mbarrier phase that nothing completes and gives up after
// `spins` polls, recording a timeout in the status word.
__global__ void wait_selftest_kernel(unsigned* status, long long spins) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!ptx::mbar_wait(&bar, 0, spins)) atomicExch(status, kStatusTimeout);
  }
}

}  // namespace

cudaError_t launch_wait_selftest(unsigned* status, long long spins, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, spins);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) note_launch();
  return e;
}

bool tc_supported(const ll_shape&) { return false; }

const char* tc_kernel_names(bool) { return ""; }

bool make_tc_plan(const ll_shape&, TcPlan*) { return false; }

cudaError_t launch_tc_fwd(const TcPlan&, const FwdArgs&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ll
