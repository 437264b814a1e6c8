// Self-test of the bounded waits every kernel of this library uses.
//
// One CTA of two warps.  Warp 0 waits, through the same mbar_wait_limit the
// kernels use, on an mbarrier that nothing ever arrives on, with a limit the
// caller chooses; when the limit runs out it records ERR_TIMEOUT_OTHER in this
// unit's error word and raises the CTA's abort flag.  Warp 1 waits on a second
// mbarrier that nothing arrives on either, with the kernels' own (much longer)
// limit, and must leave as soon as it sees the abort flag: that is how one
// role's failure ends every other role of a CTA.  No copy or MMA is in
// flight, nothing is allocated in TMEM, and both waits are bounded, so the
// kernel always returns and the context stays usable.
#include "common.cuh"
#include "launch.h"

namespace zl {
namespace {

__device__ uint32_t g_selftest_err;

__global__ void __launch_bounds__(64, 1) wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* af = &abort_flag;
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    if (warp == 0)
      mbar_wait_limit(&bars[0], 0, af, &g_selftest_err, ERR_TIMEOUT_OTHER, limit_ns);
    else
      mbar_wait(&bars[1], 0, af, &g_selftest_err, ERR_TIMEOUT_MMA);
  }
  __syncwarp();
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

uint32_t selftest_take_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_selftest_err, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (v != 0) cudaMemcpyToSymbol(g_selftest_err, &zero, sizeof(zero));
  return v;
}

}  // namespace zl
