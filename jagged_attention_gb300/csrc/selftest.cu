// selftest.cu -- exercises the bounded-wait failure path on a GPU.
//
// Every kernel of the library waits on mbarriers with a time limit: a wait
// that runs out raises the CTA's abort flag and records a timeout in a status
// word the host reads, and the kernel then winds down and returns (no trap,
// no fault, no hang).  jfa_selftest_wait_timeout runs that same wait on a
// barrier that nothing arrives on, with a short limit, so a test can check
// the outcome and then keep using the context.
#include <cuda_runtime.h>

#include "jfa.h"
#include "sm103_ptx.cuh"

namespace {

__device__ int g_selftest_status;
__device__ unsigned long long g_selftest_waited_ns;

__global__ void jfa_selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    jfa::mbar_init(jfa::smem_u32(&bar), 1);
    flag = 0;
    jfa::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const jfa::Abort ab{&flag, &g_selftest_status};
    const uint64_t t0 = jfa::globaltimer_ns();
    // phase 0 of a fresh barrier with an expected count of one: never completes
    const bool done = jfa::mbar_wait(jfa::smem_u32(&bar), 0, ab, limit_ns);
    g_selftest_waited_ns = jfa::globaltimer_ns() - t0;
    if (done) atomicOr(&g_selftest_status, 0x100);
  }
}

}  // namespace

extern "C" int jfa_selftest_wait_timeout(unsigned limit_us, unsigned long long* waited_ns,
                                         void* stream) {
  if (limit_us == 0 || limit_us > 2000000u) return JFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_selftest_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return JFA_ERR_CUDA;
  jfa_selftest_wait_kernel<<<1, 32, 0, s>>>(uint64_t(limit_us) * 1000u);
  if (cudaGetLastError() != cudaSuccess) return JFA_ERR_CUDA;
  int status = 0;
  unsigned long long waited = 0;
  if (cudaMemcpyFromSymbolAsync(&status, g_selftest_status, sizeof(status), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&waited, g_selftest_waited_ns, sizeof(waited), 0,
                                cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return JFA_ERR_CUDA;
  if (waited_ns) *waited_ns = waited;
  if (status & jfa::kDevWaitTimeout) return JFA_ERR_DEVICE_TIMEOUT;
  return status == 0x100 ? JFA_OK : JFA_ERR_CUDA;
}
