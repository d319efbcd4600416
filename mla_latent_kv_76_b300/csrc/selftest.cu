// mla_selftest_bounded_wait: runs the library's bounded device wait against an
// mbarrier that nothing arrives on, so the timeout path (abort flag, status
// MLA_ERR_DEVICE_TIMEOUT, every role of the CTA leaving its wait, the kernel
// returning) can be exercised on a GPU without a fault or a hang.
#include "../../include/mla.h"
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace {

// Thread 0 waits with the short budget on barrier 0 (never completed);
// thread 32 waits with the library's full budget on barrier 1 (never
// completed either) and must leave once thread 0 raises the CTA's abort
// flag.  With `arrive` set both barriers are completed first, the control
// case: both waits succeed and nothing is reported.
__global__ void bounded_wait_selftest_kernel(long long budget, int arrive, int32_t* status, int32_t* out) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (arrive && threadIdx.x == 0) {
    tc::mbar_arrive(&bar[0]);
    tc::mbar_arrive(&bar[1]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const tc::Abort ab{&abort_flag, status, budget};
    out[0] = tc::wait<false>(&bar[0], 0, ab) ? 1 : 0;
  } else if (threadIdx.x == 32) {
    const tc::Abort ab{&abort_flag, status};
    out[1] = tc::wait<false>(&bar[1], 0, ab) ? 1 : 0;
  }
}

}  // namespace
}  // namespace mla

extern "C" int mla_selftest_bounded_wait(int64_t budget_cycles, int32_t arrive, int32_t* dev_status,
                                         int32_t* dev_out, void* stream) {
  if (budget_cycles < 1 || budget_cycles > mla::tc::kWaitCycles || !dev_out) return MLA_ERR_INVALID_ARG;
  mla::bounded_wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      (long long)budget_cycles, arrive ? 1 : 0, dev_status, dev_out);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
