// Self-test of the bounded device waits (failure detection; not a step of the
// MoE method).  One thread waits, through the same bounded-wait routine as
// the grouped GEMM's pipeline, on an mbarrier that nothing arrives on.  The
// wait gives up after `limit` SM cycles, the kernel records MOE_ERR_TIMEOUT
// in the workspace error word and returns normally, so the CUDA context
// stays usable and moe_check() reports the timeout.
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace moe {
namespace {

__global__ void wait_timeout_selftest_kernel(long long limit, int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  ptx::mbar_init(ptx::smem_u32(&bar), 1);  // expects one arrival; none comes
  ptx::fence_mbar_init();
  abort_flag = 0;
  bool timed_out = false;
  if (!ptx::mbar_wait_bounded(ptx::smem_u32(&bar), 0, limit, &abort_flag, true, &timed_out) &&
      timed_out)
    report_error(err, DEV_ERR_TIMEOUT, 99);
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_cycles,
                                                moe_stream_t stream) {
  if (ws == nullptr || ws_bytes < moe::kErrBytes || limit_cycles <= 0 ||
      reinterpret_cast<uintptr_t>(ws) % 16 != 0)
    return MOE_ERR_INVALID_ARG;
  moe::wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(static_cast<long long>(limit_cycles),
                                                          static_cast<int*>(ws));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
