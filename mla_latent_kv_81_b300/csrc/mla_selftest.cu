// Self-check of the failure detection built into every kernel of the library: a wait on an mbarrier
// that nothing completes gives up after a bounded number of cycles, records the timeout in the
// caller's status word and returns, leaving the context usable.
#include "mla_sm100.cuh"
#include "mla_tc.cuh"

namespace mla {
namespace {

__global__ void wait_timeout_kernel(uint32_t* status, long long limit_cycles) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    abort_flag = 0;
    sm100::fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the kernels' wait routine runs out after limit_cycles
  if (threadIdx.x == 0) (void)sm100::mbar_wait_limit(&bar, 0, status, &abort_flag, limit_cycles);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_check(const Ctx& ctx, long long limit_cycles) {
  wait_timeout_kernel<<<1, 32, 0, ctx.stream>>>(ctx.status, limit_cycles);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
