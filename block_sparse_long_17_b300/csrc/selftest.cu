// Diagnostic kernel for the bounded-wait path: one thread waits, with the same
// bounded mbarrier wait the fused indexer uses, on a barrier that nothing
// arrives on.  The wait gives up after `limit` SM cycles, raises the CTA's
// abort flag and records kDevErrTimeout in the device error word; the kernel
// then returns normally, so the context stays usable.
#include "common.cuh"
#include "sm100.cuh"

namespace qsa {

__global__ void wait_timeout_selftest_kernel(long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    abort_flag = 0;
    sm100::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) sm100::mbar_wait(&bar, 0, &abort_flag, limit);  // phase 0 never completes
}

}  // namespace qsa

extern "C" qsa_status qsa_selftest_wait_timeout(int64_t limit_cycles, qsa_stream_t stream) {
  if (limit_cycles < 1000 || limit_cycles > qsa::sm100::kWaitCycles) return QSA_ERR_INVALID_ARG;
  qsa::wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>((long long)limit_cycles);
  return qsa::count_launch(cudaGetLastError()) == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
