// diag.cu -- poetx_diag_expire_wait: one bounded device wait that runs out.
//
// Every kernel of the tensor-core path waits on mbarriers through bounded
// polls (tc_ptx.cuh); when a wait gives up, the kernel records
// POETX_ERR_TIMEOUT in the library's device error word and winds down
// instead of hanging, and poetx_stream_status() reports it.  This entry point
// exercises exactly that path without a fault: one thread initialises an
// mbarrier in its own shared memory that nothing ever arrives on (no TMA, no
// MMA, no remote arrive is in flight) and waits on it with the ordinary
// bounded wait, given a short poll limit.
#include "common.cuh"
#include "profile.cuh"
#include "tc_ptx.cuh"

namespace poetx {
namespace {

__global__ void expire_wait_kernel(int cluster_scope, uint32_t polls, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    // phase 0 of a fresh barrier completes only after one arrival; none comes
    if (cluster_scope) tc::mbar_wait_cluster_bounded(&bar, 0, polls, err);
    else tc::mbar_wait_bounded(&bar, 0, polls, err);
  }
}

}  // namespace
}  // namespace poetx

extern "C" poetx_status poetx_diag_expire_wait(int cluster_scope, unsigned polls,
                                               cudaStream_t stream) {
  if ((cluster_scope != 0 && cluster_scope != 1) || polls < 1 || polls > (1u << 20))
    return POETX_ERR_INVALID_ARG;
  int* err = poetx::device_error_word();
  if (!err) return POETX_ERR_CUDA;
  {
    poetx::KernelScope ks_("diag_expire_wait", stream);
    poetx::expire_wait_kernel<<<1, 32, 0, stream>>>(cluster_scope, polls, err);
  }
  return poetx::check_launch();
}
