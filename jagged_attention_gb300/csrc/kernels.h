// kernels.h -- parameter blocks and launchers of the device kernels (internal).
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace jfa {

// The dynamic shared-memory limit of kernel K raised to `bytes`, once for
// each device the process launches it on (the attribute is per device).
template <auto K>
cudaError_t set_smem_limit_once(int bytes) {
  static std::atomic<uint64_t> done{0};  // bit d: device d configured
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Problem description shared by every kernel.  Offsets are device int32
// [B+1]; q_off == nullptr selects broadcast mode (Q has Lq rows shared by all
// sequences, O / dO / LSE have B*Lq rows, b-major).
struct Problem {
  const int32_t* kv_off;
  const int32_t* q_off;
  int B, H, Lq, D;
  int64_t n_q, n_o, n_kv;
};

struct FwdArgs {
  Problem pb;
  const int32_t* tiles;    // [T][4] {b, h, m, cost}
  const int32_t* cta_ptr;  // [P+1]
  float scale_log2;        // scale * log2(e)
  uint16_t* out;           // bf16 [n_o, H, D]
  float* lse;              // [H, n_o]
  int* status;
  bool packed;             // the schedule may hold packed tiles {b0, h, -nseq, 1}
  int* dyn_counter = nullptr;  // dynamic schedule: claim counter (zeroed before the launch)
  int T = 0;                   // tiles in the schedule
  // failure-path test only (jfa_plan_selftest): a limit for every wait
  // (0: the default) and, with test_skip = 1, one arrival withheld
  uint64_t wait_limit_ns = 0;
  int test_skip = 0;
  // CTA pairs (D = 128, static, no packing): the schedule lists pair tiles
  // {b, h, mp, cost} -- query blocks 2 mp and 2 mp + 1 -- over grid / 2 slots
  bool pair = false;
};

struct BwdArgs {
  Problem pb;
  const int32_t* tiles;    // [T][4] {b, h, n, qblocks}
  const int32_t* cta_ptr;
  float scale;             // softmax scale
  float scale_log2;        // scale * log2(e)
  const float* lse;        // [H, n_o]
  const float* delta;      // [H, n_o]
  float* dq;               // fp32 [n_q, H, D]
  uint16_t* dk;            // bf16 [n_kv, H, D]
  uint16_t* dv;
  int* status;
  bool packed;             // the schedule may hold packed tiles {b0, h, -nseq, 1}
  bool own_rows = false;   // the pre-pass left the dQ rows of single-key-block
                           // sequences uncleared: their one tile stores them
  bool own_delta = false;  // every tile holds all the keys its queries meet: the
                           // kernel forms Delta itself and `delta` is not read
  int* dyn_counter = nullptr;  // dynamic schedule: claim counter (zeroed before the launch)
  int T = 0;                   // tiles in the schedule
  uint64_t wait_limit_ns = 0;  // failure-path test only, as in FwdArgs (test_skip = 2)
  int test_skip = 0;
};

// Forward: one persistent launch over the schedule (grid = P CTAs).  o_map:
// bf16 O as [rows, H*D] in boxes of 32 rows x 64 columns (128-byte swizzle).
cudaError_t launch_fwd(const FwdArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                       const CUtensorMap& v_map, const CUtensorMap& o_map, int grid,
                       cudaStream_t stream);

// Forward with two query tiles in flight per CTA (D = 128, static schedule
// over tiles {b, h, mp, cost} of query blocks 2 mp and 2 mp + 1; grid = P).
cudaError_t launch_fwd_two(const FwdArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, const CUtensorMap& o_map, int grid,
                           cudaStream_t stream);

// Backward pre-pass: delta[h, i] = sum_d dO[i,h,d] * O[i,h,d].
cudaError_t launch_delta(const uint16_t* out, const uint16_t* dout, float* delta, int64_t n_o,
                         int H, int D, cudaStream_t stream);

// Backward main pass (grid = P CTAs).  Output maps, [rows, H*D] with the
// 128-byte swizzle: dq_map fp32 in boxes of 32 x 32, dk_map / dv_map bf16 in
// boxes of 32 rows x 64 columns.
cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                       const CUtensorMap& v_map, const CUtensorMap& do_map,
                       const CUtensorMap& dq_map, const CUtensorMap& dk_map,
                       const CUtensorMap& dv_map, int grid, cudaStream_t stream);

}  // namespace jfa
