// Diagnostic kernel: a bounded device wait that is made to expire.
//
// Every kernel of the library waits on mbarriers with a wall-clock limit; when
// a wait expires it records LCATTN_ERR_DEVICE_TIMEOUT in the status words of the
// tile metadata and the kernel returns.  This kernel waits on a barrier that
// nothing ever completes, so that the host can check the whole path (expiry,
// status word, lcattn_read_status, a usable context afterwards) without any
// fault or hang on the GPU.
#include "lcattn_internal.cuh"
#include "sm103_primitives.cuh"

namespace lcattn {
namespace {

__global__ void wait_timeout_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    dev::mbar_init(&bar, 1);  // expects one arrival that never comes
    abort_flag = 0;
    dev::fence_barrier_init();
  }
  __syncthreads();
  dev::mbar_wait(&bar, 0, &abort_flag, status, LCATTN_ERR_DEVICE_TIMEOUT);
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(int32_t* status, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

}  // namespace lcattn
