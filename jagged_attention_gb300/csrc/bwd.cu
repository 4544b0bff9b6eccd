// bwd.cu -- jagged FlashAttention backward for GB300 (sm_103a).
#include <algorithm>
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace jfa {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Delta_i = sum_d dO_id O_id for every (row, head): the row sum the backward
// subtracts inside dS = P o (dP - Delta) (the "Di" preprocessing of the TLX
// Block Attention page, "One Constraint, Five Eliminations").  D/8 lanes per
// row, 16-byte loads, a shuffle reduction; memory-bound, so each thread loads
// the pieces of two rows (one grid stride apart) before reducing either, to
// keep twice the bytes in flight.
__device__ __forceinline__ float dot_bf16x8(const uint4& o, const uint4& g) {
  return bf16_lo(o.x) * bf16_lo(g.x) + bf16_hi(o.x) * bf16_hi(g.x) + bf16_lo(o.y) * bf16_lo(g.y) +
         bf16_hi(o.y) * bf16_hi(g.y) + bf16_lo(o.z) * bf16_lo(g.z) + bf16_hi(o.z) * bf16_hi(g.z) +
         bf16_lo(o.w) * bf16_lo(g.w) + bf16_hi(o.w) * bf16_hi(g.w);
}

__global__ void __launch_bounds__(256)
    delta_kernel(const uint16_t* __restrict__ out, const uint16_t* __restrict__ dout,
                 float* __restrict__ delta, int64_t n_o, int H, int D) {
  const int lanes = D / 8;
  const int64_t rows = n_o * H;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  // the whole warp iterates while any of its lanes has a piece (the shuffles need all lanes)
  for (int64_t gid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; gid - (threadIdx.x & 31) < rows * lanes;
       gid += 2 * stride) {
    const int64_t row0 = gid / lanes, row1 = (gid + stride) / lanes;
    const int sub = static_cast<int>(gid % lanes);  // the same for both: stride is a multiple of lanes
    uint4 o0 = make_uint4(0, 0, 0, 0), g0 = o0, o1 = o0, g1 = o0;
    if (row0 < rows) {
      o0 = *reinterpret_cast<const uint4*>(out + row0 * D + sub * 8);
      g0 = *reinterpret_cast<const uint4*>(dout + row0 * D + sub * 8);
    }
    if (row1 < rows) {
      o1 = *reinterpret_cast<const uint4*>(out + row1 * D + sub * 8);
      g1 = *reinterpret_cast<const uint4*>(dout + row1 * D + sub * 8);
    }
    float acc0 = dot_bf16x8(o0, g0), acc1 = dot_bf16x8(o1, g1);
    for (int w = lanes / 2; w > 0; w >>= 1) {
      acc0 += __shfl_xor_sync(0xffffffffu, acc0, w, lanes);
      acc1 += __shfl_xor_sync(0xffffffffu, acc1, w, lanes);
    }
    if (sub == 0) {
      if (row0 < rows) delta[int64_t(row0 % H) * n_o + row0 / H] = acc0;
      if (row1 < rows) delta[int64_t(row1 % H) * n_o + row1 / H] = acc1;
    }
  }
}


// ===========================================================================
// Key/value-stationary backward.
//
// Tile (b, h, n): the 128 keys K_n and values V_n stay in shared memory while
// the CTA walks the sequence's query blocks m (broadcast mode: the blocks of
// the one dense Q).  Per query block, with S = Q K^T unscaled and
// c = scale*log2(e):
//   S^T   = K_n Q_m^T                  tcgen05.mma -> TMEM (kv rows = lanes)
//   dP^T  = V_n dO_m^T                 tcgen05.mma -> TMEM
//   P^T   = exp2(c S^T - LSE*log2 e)   WG0, written back to TMEM as bf16
//   dS^T  = P^T o (dP^T - Delta)       WG0, written to swizzled shared memory,
//                                      times the softmax scale (which dQ and
//                                      dK carry: the drain multiplies neither)
//   dV   += P^T dO_m                   A = P^T from TMEM
//   dK   += dS^T Q_m                   A = dS^T, K-major view
//   dQ_m  = dS K_n                     A = the same dS^T buffer, M-major view
// dQ_m leaves through the drain group: TMEM -> registers -> swizzled shared
// staging -> tensor reduce-add into the fp32 dq (in broadcast mode every
// sequence's tiles add into the same rows: the cross-batch reduction of the
// GEM page, "GEM's sequences do not fit a fixed grid").  The TMEM slice
// holding dQ_m is released as soon as all of it is in registers, before its
// last columns are staged (the pages' early TMEM release).  At the end of a
// tile the same group writes dV and scale*dK in bf16.
//
//   warps 0-7   two softmax groups: P^T and dS^T (thread = key row), query
//               columns split in halves
//   warp 8      TMA producer: K_n, V_n per tile; Q_m, dO_m double-buffered
//   warp 9      tcgen05.mma issuer, TMEM owner
//   warps 10-13 drain: dQ (thread = query row), dK / dV epilogue
// TMEM: S^T [0,128) (P^T bf16 pairs in columns [0,32) and [64,96)), dP^T
// [128,256) (dQ_m reuses it), dV [256, 256+D), dK [256+D, 256+2D).
// ===========================================================================

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kChunkBytes = 128 * 128;       // [128 rows x 64 bf16]
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kOffKV = 0;                    // two K/V buffers; see bwd_producer
  static constexpr int kOffQ = 2 * kTileBytes;        // 2 stages
  static constexpr int kOffDO = 4 * kTileBytes;       // 2 stages
  static constexpr int kOffDS = 6 * kTileBytes;       // dS^T [128 keys x 128 queries] bf16
  static constexpr int kOffLse = kOffDS + 32768;      // 128 -LSE*log2(e), 128 -scale*Delta (fp32)
  static constexpr int kOffBar = kOffLse + 1024;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 448;
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;
  static constexpr int kDrainWarp0 = 10;  // warps 10-13
};

struct BwdBars {
  uint64_t kv_full[2], kv_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full;
  uint64_t dv_done, ds_empty;
  uint64_t dq_full, dq_empty;
  uint64_t dkv_empty;
  uint64_t epi_done;  // a tile's last dQ has left the dS^T buffer
  uint64_t lse_ready[2], lse_done[2];  // per softmax group: LSE / Delta staging
  uint64_t dsum_part[2], dsum_ready[2];  // per softmax group: Delta formed in the kernel
  uint64_t drain;
  TileRing ring;  // dynamic schedules: tile indices from the producer to the other roles
  uint32_t tmem_base;
  int abort_flag;
};

struct BTile {
  int b, h, n, qblocks;
};
__device__ __forceinline__ BTile load_btile(const int32_t* tiles, int i) {
  const int4 t = __ldg(reinterpret_cast<const int4*>(tiles) + i);
  return {t.x, t.y, t.z, t.w};
}

__device__ __forceinline__ bool warp_wait_b(uint32_t bar, uint32_t parity, const Abort& ab) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
}
__device__ __forceinline__ void drain_wait_b(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
template <int D, bool kPack, class Seq>
__device__ void bwd_producer(const BwdArgs& a, const CUtensorMap* q_map, const CUtensorMap* k_map,
                             const CUtensorMap* v_map, const CUtensorMap* do_map, uint32_t sbase,
                             BwdBars& bars, const Abort& ab, Seq& seq) {
  using C = BwdCfg<D>;
  tma_prefetch_desc(q_map);
  tma_prefetch_desc(k_map);
  tma_prefetch_desc(v_map);
  tma_prefetch_desc(do_map);
  // Two K/V buffers swap roles every tile: tile u keeps K in buffer u % 2
  // and V in the other.  V is last read by the tile's last dP product, long
  // before K (last read by the last dQ product), so the next tile's K goes
  // into the buffer V frees and is resident by the time that tile starts; the
  // next V follows into the old K buffer, in time for the first dP (which
  // comes after the first S and P).  Each buffer is filled once per tile.
  uint32_t nq = 0, nf[2] = {0, 0};  // Q/dO stage loads, fills per K/V buffer
  bool ok = true;
  uint32_t u = 0;
  auto next = [&] { return seq.claim(a.dyn_counter, a.T, bars.ring, ab); };
  for (int i = next(); i >= 0 && ok; i = next(), ++u) {
    const BTile t = load_btile(a.tiles, i);
    const int x0 = t.h * D;
    const int k_row0 = a.pb.kv_off[t.b] + (kPack ? max(t.n, 0) : t.n) * 128;  // packed tiles: n < 0
    const int q_base = a.pb.q_off ? a.pb.q_off[t.b] : 0;
    const int o_base = a.pb.q_off ? a.pb.q_off[t.b] : t.b * a.pb.Lq;
    const uint32_t kb = u & 1, vb = kb ^ 1;
    auto load_kv = [&](uint32_t buf, const CUtensorMap* map) -> bool {
      if (!mbar_wait(smem_u32(&bars.kv_empty[buf]), (u & 1) ^ 1, ab)) return false;
      mbar_arrive_expect_tx(smem_u32(&bars.kv_full[buf]), C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_2d(sbase + C::kOffKV + buf * C::kTileBytes + c * C::kChunkBytes, map,
                    smem_u32(&bars.kv_full[buf]), x0 + c * 64, k_row0);
      ++nf[buf];
      return true;
    };
    ok = load_kv(kb, k_map);
    for (int m = 0; m < t.qblocks && ok; ++m) {
      const uint32_t qs = nq & 1, ph = (nq >> 1) & 1;
      ok = mbar_wait(smem_u32(&bars.q_empty[qs]), ph ^ 1, ab);
      if (!ok) break;
      mbar_arrive_expect_tx(smem_u32(&bars.q_full[qs]), 2 * C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        tma_load_2d(sbase + C::kOffQ + qs * C::kTileBytes + c * C::kChunkBytes, q_map,
                    smem_u32(&bars.q_full[qs]), x0 + c * 64, q_base + m * 128);
        tma_load_2d(sbase + C::kOffDO + qs * C::kTileBytes + c * C::kChunkBytes, do_map,
                    smem_u32(&bars.q_full[qs]), x0 + c * 64, o_base + m * 128);
      }
      ++nq;
      if (m == 0) ok = load_kv(vb, v_map);
    }
  }
  // let every issued copy land before the CTA may exit
  for (int b = 0; b < 2; ++b)
    if (nf[b] > 0) drain_wait_b(smem_u32(&bars.kv_full[b]), (nf[b] - 1) & 1);
  for (uint32_t qs = 0; qs < 2 && qs < nq; ++qs) {
    const uint32_t last = nq - 1 - ((nq - 1 - qs) & 1);
    drain_wait_b(smem_u32(&bars.q_full[qs]), (last >> 1) & 1);
  }
}

// ---------------------------------------------------------------------------
template <int D, class Seq>
__device__ void bwd_mma(const BwdArgs& a, uint32_t sbase, uint32_t tmem, BwdBars& bars,
                        const Abort& ab, Seq& seq) {
  using C = BwdCfg<D>;
  constexpr uint32_t id_sdp = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
  constexpr uint32_t id_kmaj = idesc_bf16_f32(128, D, false, true);    // dV (A in TMEM), dK
  constexpr uint32_t id_dq = idesc_bf16_f32(128, D, true, true);       // dQ: A = dS (M-major)
  const uint32_t sDS = sbase + C::kOffDS;
  const uint64_t dsd_k = smem_desc_sw128(sDS, 16, 1024), dsd_m = smem_desc_sw128(sDS, C::kChunkBytes, 1024);
  uint32_t gm = 0, tt = 0;
  bool ok = true;
  auto next = [&] { return seq.take(a.dyn_counter, bars.ring, ab); };
  for (int i = next(); i >= 0 && ok; i = next()) {
    const BTile t = load_btile(a.tiles, i);
    const uint32_t kb = tt & 1, vb = kb ^ 1;  // K and V buffers of this tile
    const uint32_t sK = sbase + C::kOffKV + kb * C::kTileBytes;
    const uint32_t sV = sbase + C::kOffKV + vb * C::kTileBytes;
    const uint64_t kd_k = smem_desc_sw128(sK, 16, 1024), kd_m = smem_desc_sw128(sK, C::kChunkBytes, 1024);
    const uint64_t vd_k = smem_desc_sw128(sV, 16, 1024);
    for (int m = 0; m < t.qblocks && ok; ++m, ++gm) {
      const uint32_t qs = gm & 1;
      const uint32_t sQ = sbase + C::kOffQ + qs * C::kTileBytes;
      const uint32_t sDO = sbase + C::kOffDO + qs * C::kTileBytes;
      // operand descriptors of this step: K-major (16, 1024) and MN-major
      // (chunk stride, 1024) views
      const uint64_t qd_k = smem_desc_sw128(sQ, 16, 1024), qd_m = smem_desc_sw128(sQ, C::kChunkBytes, 1024);
      const uint64_t dod_k = smem_desc_sw128(sDO, 16, 1024), dod_m = smem_desc_sw128(sDO, C::kChunkBytes, 1024);
      ok = mbar_wait(smem_u32(&bars.q_full[qs]), (gm >> 1) & 1, ab);
      if (ok && m == 0) ok = mbar_wait(smem_u32(&bars.kv_full[kb]), tt & 1, ab);
      // S^T region is free once the previous step's dV (which read P^T there) completed
      if (ok) ok = mbar_wait(smem_u32(&bars.dv_done), (gm & 1) ^ 1, ab);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
        mma_bf16_ss(tmem + C::kColS, desc_at(kd_k, koff), desc_at(qd_k, koff), id_sdp, kk > 0 ? 1u : 0u);
      }
      mma_commit(smem_u32(&bars.s_full));
      // dP^T region is free once the drain group has the previous dQ in registers
      ok = mbar_wait(smem_u32(&bars.dq_empty), (gm & 1) ^ 1, ab);
      if (ok && m == 0) ok = mbar_wait(smem_u32(&bars.kv_full[vb]), tt & 1, ab);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
        mma_bf16_ss(tmem + C::kColDP, desc_at(vd_k, koff), desc_at(dod_k, koff), id_sdp, kk > 0 ? 1u : 0u);
      }
      mma_commit(smem_u32(&bars.dp_full));
      if (m == t.qblocks - 1) mma_commit(smem_u32(&bars.kv_empty[vb]));  // V read for the last time
      if (m == 0) ok = mbar_wait(smem_u32(&bars.dkv_empty), (tt & 1) ^ 1, ab);
      if (ok) ok = mbar_wait(smem_u32(&bars.p_full), gm & 1, ab);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dV += P^T dO_m, K = 128 queries; P^T of query
                                       // half g sits at S columns [64g, 64g + 32)
        mma_bf16_ts(tmem + C::kColDV, tmem + C::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                    desc_at(dod_m, kk * 2048), id_kmaj,
                    (m > 0 || kk > 0) ? 1u : 0u);
      mma_commit(smem_u32(&bars.dv_done));
      ok = mbar_wait(smem_u32(&bars.ds_full), gm & 1, ab);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dK += dS^T Q_m
        mma_bf16_ss(tmem + C::kColDK,
                    desc_at(dsd_k, (kk >> 2) * C::kChunkBytes + (kk & 3) * 32),
                    desc_at(qd_m, kk * 2048), id_kmaj,
                    (m > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dQ_m = dS K_n, K = 128 keys
        mma_bf16_ss(tmem + C::kColDP, desc_at(dsd_m, kk * 2048), desc_at(kd_m, kk * 2048), id_dq,
                    kk > 0 ? 1u : 0u);
      mma_commit(smem_u32(&bars.dq_full));  // also: Q/dO stage qs read for the last time
      mma_commit(smem_u32(&bars.ds_empty));
      if (m == t.qblocks - 1) mma_commit(smem_u32(&bars.kv_empty[kb]));  // K read for the last time
    }
    ++tt;
  }
  mma_commit(smem_u32(&bars.drain));
  drain_wait_b(smem_u32(&bars.drain), 0);
}

// ---------------------------------------------------------------------------
// One step of a sum across the warp's lanes of 2N values per lane: lanes with
// bit N clear keep values [0, N), the others [N, 2N), and each adds its
// partner's copy of the half it keeps.  After the steps N = 16, 8, 4, 2, 1 on
// 32 values, x[0] of lane l is the sum over all lanes of value l (a fixed
// order of additions, so the result is deterministic).
template <int N>
__device__ __forceinline__ void lane_fold(float (&x)[32], int lane) {
  const bool hi = (lane & N) != 0;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const float send = hi ? x[k] : x[k + N];
    const float keep = hi ? x[k + N] : x[k];
    x[k] = keep + __shfl_xor_sync(0xffffffffu, send, N);
  }
}

// ---------------------------------------------------------------------------
// Softmax groups: P^T and dS^T.  Two warpgroups share every key row (TMEM
// lane): group g (warps 4g .. 4g+3) owns query columns [64g, 64g + 64).  With
// LSE and Delta given, the backward needs no reduction along a key row, so
// the halves are independent; splitting them puts two warps on every SM
// sub-partition, whose instruction issue is what bounds this work (hence the
// packed fp32 pairs below).  kOwnDelta: the tiles form Delta themselves, a
// sum down each query column within the group (a separate copy of the loop,
// so the common case carries none of that code).
template <int D, bool kPack, bool kOwnDelta, class Seq>
__device__ __forceinline__ void bwd_softmax_loop(const BwdArgs& a, uint8_t* smem, uint32_t sbase,
                                                 uint32_t tmem, BwdBars& bars, const Abort& ab,
                                                 Seq& seq, int g) {
  using C = BwdCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;  // key row of the tile = TMEM lane
  const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const int c0 = 64 * g;                 // first query column of this group
  float* lse2 = reinterpret_cast<float*>(smem + C::kOffLse);  // 128 -LSE*log2(e), then 128 -scale*Delta
  float* dlt = lse2 + 128;
  const uint32_t lse_ready = smem_u32(&bars.lse_ready[g]), lse_done = smem_u32(&bars.lse_done[g]);
  uint32_t gm = 0, tt = 0;
  auto next = [&] { return seq.take_warp(a.dyn_counter, bars.ring, ab); };
  for (int i = next(); i >= 0; i = next(), ++tt) {
    const BTile t = load_btile(a.tiles, i);
    // packed tile (n = -nseq): key and query rows [off[b], off[b + nseq]) of
    // nseq short sequences; a key row only meets its own sequence's queries
    const bool packed = kPack && t.n < 0;
    const int nb = packed ? 0 : t.n;
    const int b_end = t.b + (packed ? -t.n : 1);
    const int64_t klen = a.pb.kv_off[b_end] - a.pb.kv_off[t.b];
    const bool kv_ok = int64_t(nb) * 128 + r < klen;
    const int64_t qlen = a.pb.q_off ? (a.pb.q_off[b_end] - a.pb.q_off[t.b]) : a.pb.Lq;
    int q_lo = 0, q_hi = 128;  // query columns this key row may meet
    if (packed && kv_ok) {
      const int base = a.pb.kv_off[t.b], row = base + r;
      int sq = t.b;
      while (a.pb.kv_off[sq + 1] <= row) ++sq;
      q_lo = a.pb.kv_off[sq] - base;
      q_hi = a.pb.kv_off[sq + 1] - base;
    }
    const int64_t o_base = a.pb.q_off ? a.pb.q_off[t.b] : int64_t(t.b) * a.pb.Lq;
    for (int m = 0; m < t.qblocks; ++m, ++gm) {
      // this group's 64 LSE (log2 units) and -scale * Delta values, masked
      // past the sequence; mbarriers (bounded waits) rather than hardware
      // barriers, so a timed-out warp can never strand the others
      if (!warp_wait_b(lse_done, (gm & 1) ^ 1, ab)) return;  // previous block's values read
      if (r < 64) {
        const int64_t q = int64_t(m) * 128 + c0 + r;
        const bool q_ok = q < qlen;
        const int64_t idx = int64_t(t.h) * a.pb.n_o + o_base + q;
        lse2[c0 + r] = q_ok ? -(a.lse[idx] * 1.4426950408889634f) : -INFINITY;  // -LSE, log2 units
        if constexpr (!kOwnDelta) dlt[c0 + r] = q_ok ? -(a.scale * a.delta[idx]) : 0.0f;
      }
      mbar_arrive(lse_ready);
      if (!warp_wait_b(lse_ready, gm & 1, ab)) return;

      if (!warp_wait_b(smem_u32(&bars.s_full), gm & 1, ab)) return;
      tc_fence_after();
      // P^T goes back into TMEM a 32-column half at a time, over this group's
      // own S columns read in the first half
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld_x32(tl + C::kColS + c0 + c * 32, v);
        uint32_t ph[16];
        if (!packed) {
          const uint64_t sl2x2 = f2_pack(a.scale_log2, a.scale_log2);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = c0 + c * 32 + 2 * e;
            float p0, p1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sl2x2,
                             *reinterpret_cast<const uint64_t*>(lse2 + j)), p0, p1);
            p0 = fast_exp2(p0);
            p1 = fast_exp2(p1);
            ph[e] = pack_bf16x2(p0, p1);
          }
        } else {  // packed tile: only this key row's own sequence
          const uint64_t sl2x2 = f2_pack(a.scale_log2, a.scale_log2);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = c0 + c * 32 + 2 * e;
            float p0, p1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sl2x2,
                             *reinterpret_cast<const uint64_t*>(lse2 + j)), p0, p1);
            p0 = fast_exp2(p0);
            p1 = fast_exp2(p1);
            if (!kv_ok || j < q_lo || j >= q_hi) p0 = 0.0f;
            if (!kv_ok || j + 1 < q_lo || j + 1 >= q_hi) p1 = 0.0f;
            ph[e] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st_x16(tl + C::kColS + c0 + c * 16, ph);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_full));

      if (!warp_wait_b(smem_u32(&bars.dp_full), gm & 1, ab)) return;
      // the dS^T buffer is free once the previous step's dK and dQ products
      // completed and, at a tile's first step, once the previous tile's last
      // dQ has left through it
      if (!warp_wait_b(smem_u32(&bars.ds_empty), (gm & 1) ^ 1, ab)) return;
      if (m == 0 && !warp_wait_b(smem_u32(&bars.epi_done), (tt & 1) ^ 1, ab)) return;
      tc_fence_after();
      if constexpr (kOwnDelta) {
        // The tile holds every key its queries meet, so Delta_i = sum_d dO_id
        // O_id equals sum_j P_ij dP_ij over the tile's key rows (O = P V and
        // dP = dO V^T).  Each warp sums its 32 key rows across lanes, the four
        // warps' sums meet in the first kilobyte of this group's dS^T chunk
        // (free since ds_empty; overwritten by dS^T only after dsum_ready),
        // and 64 threads add them in a fixed order.
        float* part = reinterpret_cast<float*>(smem + C::kOffDS + g * C::kChunkBytes);
        uint32_t pq[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          if (c == 0) {
            tmem_ld_x32_nw(tl + C::kColS + c0, pq);
            tmem_ld_x32_nw(tl + C::kColDP + c0, v);
            tmem_ld_wait2(pq, v);
          } else {
            tmem_ld_x32(tl + C::kColDP + c0 + 32, v);
          }
          float x[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t pp = pq[c * 16 + e];
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(pp << 16), __uint_as_float(pp & 0xffff0000u)),
                             f2_pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]))),
                      x0, x1);
            x[2 * e] = kv_ok ? x0 : 0.0f;  // key rows past the sequence hold another's P^T
            x[2 * e + 1] = kv_ok ? x1 : 0.0f;
          }
          lane_fold<16>(x, lane);
          lane_fold<8>(x, lane);
          lane_fold<4>(x, lane);
          lane_fold<2>(x, lane);
          lane_fold<1>(x, lane);
          part[(warp & 3) * 64 + c * 32 + lane] = x[0];
        }
        mbar_arrive(smem_u32(&bars.dsum_part[g]));
        if (!warp_wait_b(smem_u32(&bars.dsum_part[g]), gm & 1, ab)) return;
        if (r < 64) dlt[c0 + r] = -(a.scale * ((part[r] + part[64 + r]) + (part[128 + r] + part[192 + r])));
        mbar_arrive(smem_u32(&bars.dsum_ready[g]));
        if (!warp_wait_b(smem_u32(&bars.dsum_ready[g]), gm & 1, ab)) return;
      }
      const uint32_t sDS = sbase + C::kOffDS + g * C::kChunkBytes;  // 128-byte chunk g of each row
      uint32_t p[32];  // P^T of this row, back from TMEM
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        if (c == 0) {
          tmem_ld_x32_nw(tl + C::kColS + c0, p);
          tmem_ld_x32_nw(tl + C::kColDP + c0, v);
          tmem_ld_wait2(p, v);
        } else {
          tmem_ld_x32(tl + C::kColDP + c0 + 32, v);
        }
        // Key rows past the sequence get dS^T = 0 (it reaches dQ through K);
        // their P^T is left unmasked, since it only reaches rows of dV and dK
        // that are never stored.
        // scale * dS^T = P^T o (scale dP^T - scale Delta): one packed fma in
        // place of the subtraction
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = 0u;
        if (kv_ok) {
          const uint64_t sc2 = f2_pack(a.scale, a.scale);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = c0 + c * 32 + 2 * e;
            const uint32_t pp = p[c * 16 + e];
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(pp << 16), __uint_as_float(pp & 0xffff0000u)),
                             f2_fma(f2_pack(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sc2,
                                    *reinterpret_cast<const uint64_t*>(dlt + j))),
                      d0, d1);
            w[e] = pack_bf16x2(d0, d1);
          }
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(sDS + sw128_offset(r, c * 4 + q4), w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2],
                       w[4 * q4 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      // (failure-path test: CTA 0's first warp withholds its first arrival)
      if (!(a.test_skip == 2 && blockIdx.x == 0 && warp == 0 && gm == 0))
        mbar_arrive(smem_u32(&bars.ds_full));
      mbar_arrive(lse_done);  // this block's LSE / Delta no longer read by this thread
    }
  }
}

template <int D, bool kPack, class Seq>
__device__ void bwd_softmax(const BwdArgs& a, uint8_t* smem, uint32_t sbase, uint32_t tmem,
                            BwdBars& bars, const Abort& ab, Seq& seq, int g) {
  if (a.own_delta)
    bwd_softmax_loop<D, kPack, true>(a, smem, sbase, tmem, bars, ab, seq, g);
  else
    bwd_softmax_loop<D, kPack, false>(a, smem, sbase, tmem, bars, ab, seq, g);
}

// ---------------------------------------------------------------------------
// Drain group (warps 10-13): dQ_m leaves TMEM (thread = query row), the TMEM
// columns are released as soon as all of it is in registers, and tensor
// reduce-adds into dq follow each staged pair of boxes (the cross-batch
// reduction of the broadcast mode happens here, in the memory system).  At the end of a tile the group also writes dV
// and scale * dK (thread = key row) as bf16 boxes of 32 x 64.
// Whether key row r of tile t belongs to the tile's sequence(s).
template <bool kPack>
__device__ __forceinline__ bool key_row_ok(const BwdArgs& a, const BTile& t, int r) {
  const bool packed = kPack && t.n < 0;
  const int nb = packed ? 0 : t.n;
  const int64_t klen = a.pb.kv_off[t.b + (packed ? -t.n : 1)] - a.pb.kv_off[t.b];
  return int64_t(nb) * 128 + r < klen;
}

// 32 dQ columns of one row: reduce-added, or stored when this tile owns the row.
__device__ __forceinline__ void dq_row_out(float* row, const uint32_t (&v)[32], bool store) {
  float4* dst = reinterpret_cast<float4*>(row);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float4 val = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                   __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
    if (store) dst[e] = val;
    else atomicAdd(dst + e, val);
  }
}

// dQ leaves TMEM a thread per query row, but the memory system takes row-wise
// scattered 16-byte pieces at a fraction of the rate of whole rows.  So each
// drain warp writes its 32 rows into shared memory in the 128-byte-swizzled
// box layout and hands them to the tensor-memory-access unit as D/32 boxes of
// 32 x 32 fp32 (reduce-add, or store when the tile owns the rows), reading
// TMEM two 32-column loads per wait.  The staging space is
// the Q/dO stage of the step just finished, free once dq_full has fired: its
// D/32 boxes of 16 KB fill the Q stage first, then the dO stage.  The stage
// returns to the producer when every drain warp's boxes have been read out.
// A warp whose rows run past the sequence writes its valid rows directly.
// kSelf: queries have their own offsets, so a tile can own its dQ rows.
template <int D, bool kPack, bool kSelf, class Seq>
__device__ void bwd_drain(const BwdArgs& a, const CUtensorMap* dq_map, const CUtensorMap* dk_map,
                          const CUtensorMap* dv_map, uint32_t sbase, uint32_t tmem, BwdBars& bars,
                          const Abort& ab, Seq& seq) {
  using C = BwdCfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;  // TMEM lane of this thread
  const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const int H = a.pb.H;
  uint32_t gm = 0, tt = 0;
  auto next = [&] { return seq.take_warp(a.dyn_counter, bars.ring, ab); };
  for (int i = next(); i >= 0; i = next()) {
    const BTile t = load_btile(a.tiles, i);
    // a tile that is the only one touching its dQ rows stores them instead of
    // reduce-adding: a packed tile, or (queries with their own offsets) the one
    // tile of a sequence with a single key block
    const bool packed = kPack && t.n < 0;
    const bool store = packed || (kSelf && a.pb.kv_off[t.b + 1] - a.pb.kv_off[t.b] <= 128);
    const int64_t qlen = a.pb.q_off ? (a.pb.q_off[t.b + (packed ? -t.n : 1)] - a.pb.q_off[t.b]) : a.pb.Lq;
    const int64_t q_base = a.pb.q_off ? a.pb.q_off[t.b] : 0;
    for (int m = 0; m < t.qblocks; ++m, ++gm) {
      const uint32_t qs = gm & 1;
      if (!warp_wait_b(smem_u32(&bars.dq_full), gm & 1, ab)) return;
      tc_fence_after();
      const bool last = m == t.qblocks - 1;
      const bool q_ok = int64_t(m) * 128 + r < qlen;
      const bool whole = __all_sync(0xffffffffu, q_ok);
      float* row = a.dq + ((q_base + int64_t(m) * 128 + r) * H + t.h) * D;
      auto box_addr = [&](int k) -> uint32_t {  // this warp's 32 rows of box k
        return sbase + (k < D / 64 ? C::kOffQ + qs * C::kTileBytes + k * 16384
                                   : C::kOffDO + qs * C::kTileBytes + (k - D / 64) * 16384) +
               wq * 4096;
      };
      uint32_t vv[2][32];
      auto load_pair = [&](int k2) {
        tmem_ld_x32_nw(tl + C::kColDP + k2 * 32, vv[0]);
        tmem_ld_x32_nw(tl + C::kColDP + (k2 + 1) * 32, vv[1]);
        tmem_ld_wait2(vv[0], vv[1]);
      };
      auto put = [&](int k, uint32_t dst_box, const uint32_t (&v)[32]) {  // dQ columns [32k, 32k + 32)
        if (whole) {
          const uint32_t dst = dst_box + lane * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            st_shared_v4(dst + ((u ^ (lane & 7)) << 4), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
        } else if (q_ok) {
          dq_row_out(row + k * 32, v, store);
        }
      };
      const int y = static_cast<int>(q_base + int64_t(m) * 128 + wq * 32);
      auto send = [&](int k, uint32_t src_box) {  // lane 0: one box out
        if (store) tma_store_2d(dq_map, src_box, t.h * D + k * 32, y);
        else tma_reduce_add_2d(dq_map, src_box, t.h * D + k * 32, y);
      };
      if (!last) {
        // a staged pair of boxes goes to its reduce-adds while the next pair
        // is staged (packed plans, whose tiles hold one step each, send all
        // four at once); TMEM is read and released first
        auto send_pair = [&](int k2) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            send(k2, box_addr(k2));
            send(k2 + 1, box_addr(k2 + 1));
            bulk_commit();
          }
        };
#pragma unroll
        for (int k2 = 0; k2 < D / 32; k2 += 2) {
          load_pair(k2);
          if (k2 + 2 == D / 32) {  // every TMEM read of dQ done: its columns are free for the next dP
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.dq_empty));
          }
          if (!kPack && whole && k2 > 0) send_pair(k2 - 2);
          put(k2, box_addr(k2), vv[0]);
          put(k2 + 1, box_addr(k2 + 1), vv[1]);
        }
        if (!kPack && whole) send_pair(D / 32 - 2);
        if (kPack && whole) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (kPack && whole) {
#pragma unroll
            for (int k = 0; k < D / 32; ++k) send(k, box_addr(k));
            bulk_commit();
          }
          if (whole) bulk_wait_read_all();
          mbar_arrive(smem_u32(&bars.q_empty[qs]));
        }
      } else {
        // A tile's last step (dq_full: dV and dK are complete too): dQ, dV and
        // dK leave together, and the next tile's first dP and first dV wait
        // for their TMEM columns, while boxes take a while to be read out of
        // shared memory (the memory system drains reduce-adds slowly).  So
        // every TMEM read comes first: dQ's first half goes out through the
        // dO half of the stage, its second through the dS^T buffer (the
        // next tile's first dS^T waits for epi_done), dV through the Q half,
        // and dK waits in registers as bf16 until dQ's first half is read out.
        const uint32_t do_box = sbase + C::kOffDO + qs * C::kTileBytes + wq * 4096;  // box j at + j * 16384
        const uint32_t ds_box = sbase + C::kOffDS + wq * 4096;
        constexpr int kHalf = D / 64;  // dQ boxes per half
        // D = 128 (unpacked): one pair = one half.  Group 1 (the dO-half
        // boxes) leaves once TMEM is read and released, while the second pair
        // is staged; group 2 (the dS^T-buffer boxes) after it
        auto send_half = [&](int k2, uint32_t base) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            send(k2, base);
            send(k2 + 1, base + 16384);
            bulk_commit();
          }
        };
#pragma unroll
        for (int k2 = 0; k2 < D / 32; k2 += 2) {
          load_pair(k2);
          if (k2 + 2 == D / 32) {  // every TMEM read of dQ done
            tc_fence_before();
            mbar_arrive(smem_u32(&bars.dq_empty));
          }
          if constexpr (D == 128 && !kPack) {
            if (whole && k2 > 0) send_half(k2 - 2, do_box);
          }
          const uint32_t base = k2 < kHalf ? do_box + k2 * 16384 : ds_box + (k2 - kHalf) * 16384;
          put(k2, base, vv[0]);
          put(k2 + 1, kHalf == 1 ? ds_box : base + 16384, vv[1]);
        }
        if constexpr (D == 128 && !kPack) {
          if (whole) send_half(D / 32 - 2, ds_box);
        }
        if constexpr (D != 128 || kPack) {
          if (whole) fence_proxy_async_smem();
          __syncwarp();
          if (whole && lane == 0) {  // group 1: the dO-half boxes, group 2: the dS^T-buffer boxes
#pragma unroll
            for (int j = 0; j < kHalf; ++j) send(j, do_box + j * 16384);
            bulk_commit();
#pragma unroll
            for (int j = 0; j < kHalf; ++j) send(kHalf + j, ds_box + j * 16384);
            bulk_commit();
          }
        }
        // dV through the Q half (group 3), dK into registers
        const bool kv_ok = key_row_ok<kPack>(a, t, r);
        const bool kv_whole = __all_sync(0xffffffffu, kv_ok);
        const int nb = (kPack && t.n < 0) ? 0 : t.n;
        const int64_t krow = int64_t(a.pb.kv_off[t.b]) + nb * 128 + r;
        const int yk = static_cast<int>(int64_t(a.pb.kv_off[t.b]) + nb * 128 + wq * 32);
        const uint32_t qh = sbase + C::kOffQ + qs * C::kTileBytes + wq * 4096;  // chunk c at + c * 16384
        auto put_bf16 = [&](uint32_t region, uint16_t* dst_row, int c, const uint32_t (&pk)[16]) {
          if (kv_whole) {  // 32 columns = units 4(c&1) .. 4(c&1)+3 of the row in chunk c/2
            const uint32_t dst = region + lane * 128 + (c >> 1) * 16384;
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(dst + (((4 * (c & 1) + q) ^ (lane & 7)) << 4), pk[4 * q], pk[4 * q + 1],
                           pk[4 * q + 2], pk[4 * q + 3]);
          } else if (kv_ok) {
            uint4* dst = reinterpret_cast<uint4*>(dst_row + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        };
        uint16_t* dv_row = a.dv + (krow * H + t.h) * D;
        uint16_t* dk_row = a.dk + (krow * H + t.h) * D;
#pragma unroll
        for (int c2 = 0; c2 < D / 32; c2 += 2) {
          uint32_t ww[2][32];
          tmem_ld_x32_nw(tl + C::kColDV + c2 * 32, ww[0]);
          tmem_ld_x32_nw(tl + C::kColDV + (c2 + 1) * 32, ww[1]);
          tmem_ld_wait2(ww[0], ww[1]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(__uint_as_float(ww[h][2 * e]), __uint_as_float(ww[h][2 * e + 1]));
            put_bf16(qh, dv_row, c2 + h, pk);
          }
        }
        uint32_t dkp[D / 32][16];  // dK of this row (dS^T carried the scale), bf16 pairs
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t w[32];
          tmem_ld_x32(tl + C::kColDK + c * 32, w);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            dkp[c][e] = pack_bf16x2(__uint_as_float(w[2 * e]), __uint_as_float(w[2 * e + 1]));
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.dkv_empty));  // dV / dK columns free for the next tile
        if (kv_whole) fence_proxy_async_smem();
        __syncwarp();
        if (kv_whole && lane == 0) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c) tma_store_2d(dv_map, qh + c * 16384, t.h * D + c * 64, yk);
          bulk_commit();
          if (whole) bulk_wait_read_keep2();  // dQ's dO-half boxes are read out
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) put_bf16(do_box, dk_row, c, dkp[c]);
        if (kv_whole) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (kv_whole) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_store_2d(dk_map, do_box + c * 16384, t.h * D + c * 64, yk);
            bulk_commit();
          }
          // open groups, oldest first: dQ dO half, dQ dS^T buffer, dV, dK
          if (whole && kv_whole) bulk_wait_read_keep2();
          else if (whole) bulk_wait_read_all();
          mbar_arrive(smem_u32(&bars.epi_done));  // the dS^T buffer is read out
          bulk_wait_read_all();                   // the stage is read out
          mbar_arrive(smem_u32(&bars.q_empty[qs]));
        }
        ++tt;
      }
      __syncwarp();
    }
  }
}

template <int D, bool kPack, bool kSelf, bool kDyn>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1)
    jfa_bwd_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap do_map,
                   const __grid_constant__ CUtensorMap dq_map, const __grid_constant__ CUtensorMap dk_map,
                   const __grid_constant__ CUtensorMap dv_map, const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  BwdBars& bars = *reinterpret_cast<BwdBars*>(smem + C::kOffBar);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tile_ring_init(bars.ring, 1 + 8 + 4);  // consumers: MMA thread, 8 softmax and 4 drain warps
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars.kv_full[b]), 1);
      mbar_init(smem_u32(&bars.kv_empty[b]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars.q_full[s]), 1);
      mbar_init(smem_u32(&bars.q_empty[s]), 4);  // one arrival per drain warp
    }
    mbar_init(smem_u32(&bars.s_full), 1);
    mbar_init(smem_u32(&bars.dp_full), 1);
    mbar_init(smem_u32(&bars.p_full), 256);
    mbar_init(smem_u32(&bars.ds_full), 256);
    mbar_init(smem_u32(&bars.dv_done), 1);
    mbar_init(smem_u32(&bars.ds_empty), 1);
    mbar_init(smem_u32(&bars.dq_full), 1);
    mbar_init(smem_u32(&bars.dq_empty), 128);
    mbar_init(smem_u32(&bars.dkv_empty), 128);
    mbar_init(smem_u32(&bars.epi_done), 4);  // one arrival per drain warp
    for (int g = 0; g < 2; ++g) {
      mbar_init(smem_u32(&bars.lse_ready[g]), 128);
      mbar_init(smem_u32(&bars.lse_done[g]), 128);
      mbar_init(smem_u32(&bars.dsum_part[g]), 128);
      mbar_init(smem_u32(&bars.dsum_ready[g]), 128);
    }
    mbar_init(smem_u32(&bars.drain), 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    tmem_alloc(smem_u32(&bars.tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const Abort ab{&bars.abort_flag, a.status, a.wait_limit_ns ? a.wait_limit_ns : kWaitLimitNs};
  TileSeq<kDyn> seq(a.cta_ptr, a.dyn_counter);
  if (warp < 8) {
    bwd_softmax<D, kPack>(a, smem, sbase, tmem, bars, ab, seq, warp >> 2);
  } else if (warp >= C::kDrainWarp0) {
    bwd_drain<D, kPack, kSelf>(a, &dq_map, &dk_map, &dv_map, sbase, tmem, bars, ab, seq);
    if (lane == 0) bulk_wait_all();  // dQ, dK, dV boxes written before the CTA exits
  } else if (warp == C::kProducerWarp) {
    if (lane == 0) bwd_producer<D, kPack>(a, &q_map, &k_map, &v_map, &do_map, sbase, bars, ab, seq);
    __syncwarp();
  } else {
    if (lane == 0) bwd_mma<D>(a, sbase, tmem, bars, ab, seq);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool kPack, bool kSelf, bool kDyn>
cudaError_t launch_bwd_d(const BwdArgs& a, const CUtensorMap& q, const CUtensorMap& k,
                         const CUtensorMap& v, const CUtensorMap& dO, const CUtensorMap& dq,
                         const CUtensorMap& dk, const CUtensorMap& dv, int grid, cudaStream_t stream) {
  using C = BwdCfg<D>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  static_assert(sizeof(BwdBars) <= C::kBarBytes, "barrier block");
  cudaError_t e = set_smem_limit_once<jfa_bwd_kernel<D, kPack, kSelf, kDyn>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  jfa_bwd_kernel<D, kPack, kSelf, kDyn><<<grid, C::kThreads, C::kSmemBytes, stream>>>(q, k, v, dO, dq, dk, dv, a);
  return cudaGetLastError();
}

// packed plans, owned-dQ plans, reduce-only plans and dynamic schedules run
// their own instantiations
template <int D, bool kDyn>
cudaError_t launch_bwd_m(bool packed, bool self, const BwdArgs& a, const CUtensorMap& q,
                         const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dO,
                         const CUtensorMap& dq, const CUtensorMap& dk, const CUtensorMap& dv, int grid,
                         cudaStream_t stream) {
  if (packed) return launch_bwd_d<D, true, true, kDyn>(a, q, k, v, dO, dq, dk, dv, grid, stream);
  if (self) return launch_bwd_d<D, false, true, kDyn>(a, q, k, v, dO, dq, dk, dv, grid, stream);
  return launch_bwd_d<D, false, false, kDyn>(a, q, k, v, dO, dq, dk, dv, grid, stream);
}

}  // namespace

cudaError_t launch_delta(const uint16_t* out, const uint16_t* dout, float* delta, int64_t n_o,
                         int H, int D, cudaStream_t stream) {
  const int64_t threads = n_o * H * (D / 8);
  if (threads == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // a grid-stride loop over enough blocks to fill every SM of this device
  const int64_t blocks = std::min<int64_t>((threads + 255) / 256, int64_t(sms) * 64);
  delta_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(out, dout, delta, n_o, H, D);
  return cudaGetLastError();
}


}  // namespace jfa

namespace jfa {
cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                       const CUtensorMap& v_map, const CUtensorMap& do_map,
                       const CUtensorMap& dq_map, const CUtensorMap& dk_map,
                       const CUtensorMap& dv_map, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
#define JFA_BWD_ARGS a, q_map, k_map, v_map, do_map, dq_map, dk_map, dv_map, grid, stream
  // packed plans, plans whose single-key-block tiles store their dQ rows, and
  // plans where every tile reduce-adds run separate instantiations
  const bool self = a.own_rows;
  if (a.pb.D == 128)
    return a.dyn_counter ? launch_bwd_m<128, true>(a.packed, self, JFA_BWD_ARGS)
                         : launch_bwd_m<128, false>(a.packed, self, JFA_BWD_ARGS);
  return a.dyn_counter ? launch_bwd_m<64, true>(a.packed, self, JFA_BWD_ARGS)
                       : launch_bwd_m<64, false>(a.packed, self, JFA_BWD_ARGS);
#undef JFA_BWD_ARGS
}
}  // namespace jfa
