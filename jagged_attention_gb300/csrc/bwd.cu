// bwd.cu -- jagged FlashAttention backward for GB300 (sm_103a).
#include <algorithm>
#include "kernels.h"
#include "sm103_ptx.cuh"

namespace jfa {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Delta_i = sum_d dO_id O_id for every (row, head): the row sum the backward
// subtracts inside dS = P o (dP - Delta) (the "Di" preprocessing of the TLX
// Block Attention page, "One Constraint, Five Eliminations").  D/8 lanes per
// row, 16-byte loads, a shuffle reduction; memory-bound.
__global__ void __launch_bounds__(256)
    delta_kernel(const uint16_t* __restrict__ out, const uint16_t* __restrict__ dout,
                 float* __restrict__ delta, int64_t n_o, int H, int D) {
  const int lanes = D / 8;
  const int64_t rows = n_o * H;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; gid - (threadIdx.x & 31) < rows * lanes;
       gid += stride) {
    const int64_t row = gid / lanes;  // row * H + head, in memory order
    const int sub = static_cast<int>(gid % lanes);
    float acc = 0.0f;
    if (row < rows) {
      const uint4 o = *reinterpret_cast<const uint4*>(out + row * D + sub * 8);
      const uint4 g = *reinterpret_cast<const uint4*>(dout + row * D + sub * 8);
      acc = bf16_lo(o.x) * bf16_lo(g.x) + bf16_hi(o.x) * bf16_hi(g.x) + bf16_lo(o.y) * bf16_lo(g.y) +
            bf16_hi(o.y) * bf16_hi(g.y) + bf16_lo(o.z) * bf16_lo(g.z) + bf16_hi(o.z) * bf16_hi(g.z) +
            bf16_lo(o.w) * bf16_lo(g.w) + bf16_hi(o.w) * bf16_hi(g.w);
    }
    for (int w = lanes / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w, lanes);
    if (sub == 0 && row < rows) {
      const int64_t i = row / H;
      const int h = static_cast<int>(row % H);
      delta[int64_t(h) * n_o + i] = acc;
    }
  }
}

}  // namespace

cudaError_t launch_delta(const uint16_t* out, const uint16_t* dout, float* delta, int64_t n_o,
                         int H, int D, cudaStream_t stream) {
  const int64_t threads = n_o * H * (D / 8);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((threads + 255) / 256, int64_t(152) * 64);
  delta_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(out, dout, delta, n_o, H, D);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdArgs&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                       const CUtensorMap&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace jfa
