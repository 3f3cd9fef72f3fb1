// selftest.cu -- moe_selftest_wait_timeout: runs the bounded mbarrier wait
// of the grouped GEMMs to its limit on purpose, so that a test can check
// that an expired wait reports MOE_ERR_TIMEOUT through the device error word
// and that the other roles of the CTA stop through its abort flag, with the
// context still usable afterwards. No copy or MMA is in flight in this kernel.
#include "kernels.h"
#include "tc_common.cuh"

namespace moe {
namespace {

// Warp 0 waits (bounded by `cycles`) on an mbarrier that nothing arrives on;
// warp 1 waits on another one with the GEMMs' full limit and has to leave
// through the abort flag that warp 0 raises when its wait expires. out[w] = 1
// if warp w's wait completed, 0 if it gave up.
__global__ void __launch_bounds__(64) wait_selftest_kernel(long long cycles, int* err, int32_t* out) {
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar[0], 1);
    ptx::mbar_init(&bar[1], 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    // phase 0 of a fresh mbarrier completes only when one arrival lands
    const bool ok = warp == 0 ? tc::wait_bar_for(&bar[0], 0, &abort_flag, err, cycles)
                              : tc::wait_bar_for(&bar[1], 0, &abort_flag, err, tc::kWaitLimitCycles);
    out[warp] = ok ? 1 : 0;
  }
  __syncthreads();
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_wait_timeout(long long cycles, int32_t* out, void* stream) {
  if (cycles <= 0 || cycles > moe::tc::kWaitLimitCycles || out == nullptr) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(out) & 15u) != 0) return MOE_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_COUNTED_AS("wait_selftest", st) moe::wait_selftest_kernel<<<1, 64, 0, st>>>(cycles, moe::device_error_word(), out);
  MOE_CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}
