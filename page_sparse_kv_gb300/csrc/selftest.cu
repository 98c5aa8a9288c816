// psk_selftest_bounded_wait: runs the kernels' bounded mbarrier wait on a phase that can never
// complete, so a test can see the timeout path work on the GPU without anything hanging: the wait
// gives up after `spin_limit` polls, sets PSK_DEV_TIMEOUT in the workspace status word and the
// kernel returns. Nothing is in flight (no copy was issued), so the context stays usable.
//
// The phase: one thread initialises an mbarrier for one arrival, arrives with an expected
// transaction count of 16 bytes and issues no copy, leaving the phase waiting for bytes that
// never come. mbar_wait_limit is the function every streaming kernel of the library waits with
// (there with kMbarSpinLimit polls).
#include "psk_common.cuh"
#include "psk_internal.h"

namespace psk {
namespace {

__global__ void bounded_wait_kernel(void *ws, uint32_t spin_limit) {
  __shared__ __align__(8) uint64_t bar;
  pdl_begin();  // stream order with the kernels around it, as every kernel of the library
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  mbar_arrive_expect_tx(b, 16u);  // the phase now also waits for 16 bytes that no copy delivers
  (void)mbar_wait_limit(b, 0u, ws, spin_limit);
}

}  // namespace
}  // namespace psk

extern "C" int psk_selftest_bounded_wait(void *workspace, size_t workspace_bytes, uint32_t spin_limit,
                                         psk_stream_t stream) {
  using namespace psk;
  if (!workspace) return PSK_ERR_INVALID_ARG;
  if (workspace_bytes < kWsHeader) return PSK_ERR_WORKSPACE;
  if (spin_limit < 1 || spin_limit > kMbarSpinLimit) return PSK_ERR_INVALID_ARG;
  const cudaError_t e =
      launch_kernel(true, bounded_wait_kernel, 1, 32, 0, static_cast<cudaStream_t>(stream), workspace, spin_limit);
  return e == cudaSuccess ? PSK_OK : PSK_ERR_CUDA;
}
