// Diagnostic of the library's bounded waits (not a step of the method).
//
// Every mbarrier wait in the library's kernels gives up after a fixed limit
// of global time (tc::kWaitNs), records MLA_ERR_TIMEOUT in the error word and
// lets the kernel return, so that a copy or a peer that never arrives cannot
// hang the GPU.  This kernel waits on an mbarrier that nothing completes, so
// that a test can watch that path end with the status and a usable context.
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace {

__global__ void bounded_wait_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc::mbar_init(tc::smem_u32(&bar), 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait(tc::smem_u32(&bar), 0, &abort_flag, err);  // no arrival comes
}

}  // namespace
}  // namespace mla

extern "C" mla_status mla_selftest_bounded_wait(void* workspace, mla_stream_t stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  mla::bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(static_cast<int*>(workspace));
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
