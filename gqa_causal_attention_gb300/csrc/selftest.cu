// attn_selftest_wait_timeout: the failure path of the pipeline waits, run on purpose.
//
// The tensor-core kernels never wait without a limit: every mbarrier wait gives
// up after tc::kWaitLimitNs of %globaltimer, raises the block's abort flag so
// that its other roles stop waiting too, and the block reports ATTN_DEV_TIMEOUT
// in the caller's status word instead of hanging. This kernel runs exactly that
// code (tc::mbar_wait) on barriers that nothing ever signals: role 0 waits
// until its limit and raises abort, role 1 waits on a second barrier and returns
// as soon as it sees the abort, and the block then reports the timeout. No
// memory is touched but the status word, so the context stays usable.
#include "../../include/gqa_attn.h"
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace {

__global__ void __launch_bounds__(64) wait_timeout_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    gqa::tc::mbar_init(&bars[0], 1);
    gqa::tc::mbar_init(&bars[1], 1);
    abort_flag = 0;
    gqa::tc::fence_mbar_init();
  }
  __syncthreads();
  const int role = threadIdx.x / 32;
  if ((threadIdx.x & 31) == 0) {
    // phase 0 of a fresh barrier completes only when someone arrives: nobody does
    gqa::tc::mbar_wait(&bars[role], 0u, reinterpret_cast<volatile int*>(&abort_flag));
  }
  __syncthreads();
  if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(&abort_flag))
    gqa::report(status, ATTN_DEV_TIMEOUT);
}

}  // namespace

extern "C" int attn_selftest_wait_timeout(int32_t* status, void* stream) {
  if (!status) return ATTN_ERR_NULL;
  wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(status);
  return gqa::record_cuda_error(cudaGetLastError());
}
