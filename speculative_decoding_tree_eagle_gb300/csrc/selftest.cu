// ts_selftest_bounded_wait: exercises the bounded pipeline wait that every mbarrier wait of
// the library goes through (mbar_wait / mbar_wait_warp in common.cuh).  One CTA, two waiting
// warps on two mbarriers:
//   mode 0  nothing ever arrives on either barrier.  The waits give up after the wait limit
//           (2 s of %globaltimer), the first to give up raises the CTA's abort flag and stores
//           TS_ERR_TIMEOUT in the status word, the other leaves on the flag, and the kernel
//           returns normally: no trap, the context stays usable.
//   mode 1  thread 0 completes both barriers first; both waits succeed at once.
// result[w] = 1 when warp w's wait succeeded, else 0.
#include "common.cuh"
#include "internal.h"

namespace ts {
namespace {

__global__ void __launch_bounds__(64) bounded_wait_kernel(int mode, int32_t* result, int32_t* status) {
  __shared__ alignas(8) uint64_t s_bar[2];
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&s_bar[0]), 1);
    mbar_init(smem_u32(&s_bar[1]), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (mode == 1 && threadIdx.x == 0) {
    mbar_arrive(smem_u32(&s_bar[0]));
    mbar_arrive(smem_u32(&s_bar[1]));
  }
  const int warp = threadIdx.x >> 5;
  const bool ok = mbar_wait_warp(smem_u32(&s_bar[warp]), 0, &s_abort, status);
  if ((threadIdx.x & 31) == 0) result[warp] = ok ? 1 : 0;
}

}  // namespace

int selftest_bounded_wait_launch(int mode, int32_t* result, int32_t* dev_status, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 64, 0, stream>>>(mode, result, dev_status);
  if (cudaGetLastError() != cudaSuccess) return TS_ERR_CUDA;
  count_launches(1);
  return TS_OK;
}

}  // namespace ts
