// debug_wait.cu -- test entry for the kernels' failure path: one thread waits, with the
// library's bounded mbarrier wait, on a barrier that nothing ever arrives on.  The wait
// gives up after the requested limit, sets the device error word as any expired wait in
// the attention kernels does, and the kernel returns normally; qat_attn_device_status
// then reports QAT_ERR_TIMEOUT and clears the word.  Nothing faults, traps or hangs.
#include "qat_attn.h"
#include "qat_internal.h"
#include "sm100.cuh"

namespace qat {
namespace {

using namespace sm100;

__global__ void __launch_bounds__(32) wait_timeout_kernel(unsigned int* err,
                                                          unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar_word;
  __shared__ WaitCtl ctl;
  if (threadIdx.x == 0) {
    ctl.abort = 0;
    ctl.limit_ns = limit_ns;
    mbar_init(smem_addr(&bar_word), 1);
    fence_barrier_init();
    // phase 0 of a fresh barrier completes only after one arrival, and none comes
    mbar_wait(smem_addr(&bar_word), 0, &ctl, err, limit_ns);
  }
}

}  // namespace
}  // namespace qat

extern "C" qat_status_t qat_debug_wait_timeout(int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 4000) return QAT_ERR_INVALID_ARG;
  unsigned int* err = nullptr;
  int num_sms = 0;
  cudaError_t e = qat::device_context(&err, &num_sms);
  if (e == cudaSuccess) {
    qat::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        err, static_cast<unsigned long long>(limit_ms) * 1000000ull);
    e = cudaGetLastError();
  }
  return e == cudaSuccess ? QAT_OK : QAT_ERR_CUDA;
}
