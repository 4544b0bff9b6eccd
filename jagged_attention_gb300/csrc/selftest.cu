// selftest.cu -- self-tests that run on a GPU apart from the attention
// kernels.
//
// Every kernel of the library waits on mbarriers with a time limit: a wait
// that runs out raises the CTA's abort flag and records a timeout in a status
// word the host reads, and the kernel then winds down and returns (no trap,
// no fault, no hang).  jfa_selftest_wait_timeout runs that same wait on a
// barrier that nothing arrives on, with a short limit, so a test can check
// the outcome and then keep using the context.
//
// jfa_selftest_mma_cycles measures what one tensor-core product costs: one
// CTA issues `count` products of one shape back to back into one TMEM
// accumulator, with the operand descriptors the kernels use, and times them
// to the completion of a final commit.  The kernels' products are of these
// shapes, so the figure bounds how fast a tile's products can run.
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

__device__ unsigned long long g_selftest_cycles, g_selftest_issue_cycles;

// forms: 0 M128 N128 (A, B in shared memory), 1 M128 N256, 2 M128 N128 with
// A in TMEM, 3 M128 N64.  Operands are zeros; K = 16 per product; the issue
// loop is unrolled by eight with the form fixed at compile time, so the
// thread spends next to nothing between products.  group > 0: after every
// `group` products the thread commits and waits for them to complete before
// issuing the next group (a dependent chain, as in the kernels).
template <int kForm>
__global__ void __launch_bounds__(128, 1) jfa_selftest_mma_kernel(int count, int group, uint64_t limit_ns) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tbase;
  __shared__ int flag;
  for (int i = threadIdx.x; i < 48 * 1024 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    jfa::mbar_init(jfa::smem_u32(&bar), 1);
    flag = 0;
    jfa::fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    jfa::tmem_alloc(jfa::smem_u32(&tbase), 512);
    jfa::tmem_relinquish();
  }
  jfa::fence_proxy_async_smem();
  jfa::tc_fence_before();
  __syncthreads();
  jfa::tc_fence_after();
  const uint32_t tm = tbase;
  {  // zero the 16 columns [384, 400) the TMEM-A form reads, lane = thread
    const uint32_t z[16] = {};
    jfa::tmem_st_x16(tm + (static_cast<uint32_t>((threadIdx.x >> 5) * 32) << 16) + 384, z);
    jfa::tmem_st_wait();
  }
  jfa::tc_fence_before();
  __syncthreads();
  jfa::tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t sA = jfa::smem_u32(sm), sB = jfa::smem_u32(sm + 16384);
    // forms 4-6 read A and / or B in the MN-major layout (64-element chunks
    // along M / N, 8 KB apart), as the kernels' transposed operands do
    constexpr bool kAmn = kForm == 5, kBmn = kForm >= 4;
    const uint64_t ad = jfa::smem_desc_sw128(sA, kAmn ? 8192 : 16, 1024);
    const uint64_t bd = jfa::smem_desc_sw128(sB, kBmn ? 8192 : 16, 1024);
    constexpr int N = kForm == 1 ? 256 : kForm == 3 ? 64 : 128;
    constexpr uint32_t id = jfa::idesc_bf16_f32(128, N, kAmn, kBmn);
    constexpr bool kTs = kForm == 2 || kForm == 6;
    const jfa::Abort ab{&flag, &g_selftest_status};
    const int G = group > 0 ? group : count;  // both multiples of 8 (checked on the host)
    uint32_t phase = 0;
    bool done = true;
    long long issue = 0;
    const long long t0 = clock64();
    for (int g0 = 0; g0 < count && done; g0 += G) {
      const long long ti = clock64();
      // the first product of the run overwrites the accumulator
      if constexpr (kTs) jfa::mma_bf16_ts(tm, tm + 384, bd, id, g0 > 0 ? 1u : 0u);
      else jfa::mma_bf16_ss(tm, ad, bd, id, g0 > 0 ? 1u : 0u);
#pragma unroll 8
      for (int i = 1; i < G; ++i) {
        if constexpr (kTs) jfa::mma_bf16_ts(tm, tm + 384, bd, id, 1u);
        else jfa::mma_bf16_ss(tm, ad, bd, id, 1u);
      }
      issue += clock64() - ti;
      jfa::mma_commit(jfa::smem_u32(&bar));
      done = jfa::mbar_wait(jfa::smem_u32(&bar), phase, ab, limit_ns);
      phase ^= 1;
    }
    g_selftest_cycles = done ? static_cast<unsigned long long>(clock64() - t0) : 0ull;
    g_selftest_issue_cycles = static_cast<unsigned long long>(issue);
  }
  jfa::tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    jfa::tc_fence_after();
    jfa::tmem_dealloc(tm, 512);
  }
}

}  // namespace

namespace {
template <int kForm>
cudaError_t launch_mma_selftest(int count, int group, int smem, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(jfa_selftest_mma_kernel<kForm>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  jfa_selftest_mma_kernel<kForm><<<1, 128, smem, s>>>(count, group, jfa::kWaitLimitNs);
  return cudaGetLastError();
}
}  // namespace

extern "C" int jfa_selftest_mma_cycles(int form, int count, int group, unsigned long long* cycles,
                                       unsigned long long* issue_cycles, void* stream) {
  if (form < 0 || form > 6 || count < 8 || count > (1 << 20) || count % 8 != 0 || !cycles)
    return JFA_ERR_INVALID_ARG;
  if (group < 0 || (group > 0 && (group % 8 != 0 || count % group != 0))) return JFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int smem = 48 * 1024 + 1024;
  const int zero = 0;
  if (cudaMemcpyToSymbolAsync(g_selftest_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return JFA_ERR_CUDA;
  const cudaError_t e = form == 0 ? launch_mma_selftest<0>(count, group, smem, s)
                        : form == 1 ? launch_mma_selftest<1>(count, group, smem, s)
                        : form == 2 ? launch_mma_selftest<2>(count, group, smem, s)
                        : form == 3 ? launch_mma_selftest<3>(count, group, smem, s)
                        : form == 4 ? launch_mma_selftest<4>(count, group, smem, s)
                        : form == 5 ? launch_mma_selftest<5>(count, group, smem, s)
                                    : launch_mma_selftest<6>(count, group, smem, s);
  if (e != cudaSuccess) return JFA_ERR_CUDA;
  int status = 0;
  unsigned long long c = 0, ci = 0;
  if (cudaMemcpyFromSymbolAsync(&status, g_selftest_status, sizeof(status), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&c, g_selftest_cycles, sizeof(c), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&ci, g_selftest_issue_cycles, sizeof(ci), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return JFA_ERR_CUDA;
  if (status & jfa::kDevWaitTimeout) return JFA_ERR_DEVICE_TIMEOUT;
  *cycles = c;
  if (issue_cycles) *issue_cycles = ci;
  return JFA_OK;
}

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
