// Device health check of the failure path every pipelined kernel relies on: a bounded mbarrier
// wait that nothing completes.  The GEMMs' waits give up after 2 s, raise their CTA's abort flag,
// record MOE_ERR_TIMEOUT in the device status word and return instead of hanging; this kernel runs
// the same wait (mbar_wait) on a barrier no thread arrives at, with a short limit, so that a caller
// (or a test) can see the timeout reported and the context stay usable afterwards.
#include "common.cuh"
#include "internal.h"

namespace moe {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns, int* status, int* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);   // one arrival completes phase 0; none comes
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait(&bar, 0u, &abort_flag, status, limit_ns);
    const uint64_t waited = globaltimer_ns() - t0;
    // result: 1 = gave up after at least the limit with the abort flag raised; 0 otherwise
    result[0] = (!ok && abort_flag && waited >= limit_ns) ? 1 : 0;
    result[1] = (int)(waited / 1000000ull);   // milliseconds waited
  }
}

__device__ int g_wait_check[2];

cudaError_t launch_wait_timeout_check(uint64_t limit_ns, int* status, int* result_host, cudaStream_t st) {
  void* res = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&res, g_wait_check);
  if (e != cudaSuccess) return e;
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, status, static_cast<int*>(res));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(result_host, res, 2 * sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(st);
}

}  // namespace moe
