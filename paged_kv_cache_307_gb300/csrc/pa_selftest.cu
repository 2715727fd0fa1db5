// pa_selftest.cu — a health check of the bounded pipeline waits.
//
// Every mbarrier wait in the decode and prefill kernels gives up after a
// time limit instead of spinning forever: it records PA_DEV_TIMEOUT, the
// kernel winds down, the CUDA context stays usable and pa_last_error reports
// the condition.  pa_selftest_bounded_wait runs that mechanism on purpose,
// with nothing else involved: one warp waits on an mbarrier that nothing
// arrives at.  No memory is touched outside the CTA's own shared memory.
#include "pa_common.cuh"

namespace pa {
namespace {

__device__ unsigned g_status_selftest;

__global__ void __launch_bounds__(32) bounded_wait_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);       // phase 0 completes after one arrival, and none comes
    fence_mbar_init();
  }
  __syncwarp();
  const bool done = mbar_wait_for(&bar, 0, limit_ns);
  if (!done && threadIdx.x == 0) atomicOr(&g_status_selftest, PA_DEV_TIMEOUT);
}

}  // namespace

unsigned fetch_status_selftest() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_selftest, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v && cudaMemcpyToSymbol(g_status_selftest, &zero, sizeof(zero)) != cudaSuccess) return 0xffffffffu;
  return v;
}

}  // namespace pa

extern "C" int pa_selftest_bounded_wait(unsigned long long limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > pa::kWaitLimitNs) return PA_ERR_SHAPE;
  pa::bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns);
  if (!pa::ck(cudaGetLastError(), "bounded_wait_kernel launch")) return PA_ERR_CUDA;
  return PA_OK;
}
