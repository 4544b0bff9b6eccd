// fwd2.cu -- jagged FlashAttention forward with two query tiles in flight per
// CTA (D = 128), for GB300 (sm_103a).
//
// A schedule tile {b, h, mp, cost} covers query blocks A = 2 mp and B = 2 mp + 1
// of sequence b (rows [256 mp, 256 mp + 256)); both share every K/V block.
// The one-tile forward (fwd.cu) keeps the tensor pipe busy less than half the
// time: each key block's products wait for that block's softmax, and the
// softmax waits for the products.  Here the two tiles alternate: while the
// softmax warps work on one tile's block, the pipe runs the other tile's
// products (the pages' two query tiles per CTA: alphasignal JFA page,
// "Specialized warps keep tensor cores busy").  Per key block j the MMA
// thread issues
//
//   PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
//
// -- one issuing thread per tile (warps 9 and 10), each walking its tile's
// chain, the tensor pipe interleaving their products: a single issuer stays
// held by the products it has just issued and would serialise the two chains
// -- and the softmax warps process A(j), B(j), A(j+1), ... with the same
// column split as the one-tile kernel (warps 0-3 take key columns [0, 64) of
// each block, warps 4-7 [64, 128), exchanging row maxima per block and row
// sums per tile).
//
// TMEM (512 columns): S_A [0, 128), S_B [128, 256), O_A [256, 384), O_B
// [384, 512).  A tile's P (bf16) is written back over its own S columns --
// each softmax group over the half it read -- and the next S of that tile
// waits until the PV that read P has completed.  Since that S's commit comes
// after the PV in the issue order, the softmax that waits for S finds O
// already holding the PV.
//
// Shared memory: Q_A, Q_B (32 KB each), a two-stage K and V ring (32 KB
// stages), row statistics.  There is no room left for a separate O staging
// area.  At a tile's end both tiles' products on the K and V stages of its
// last block have completed, and the producer's next loads into those two
// stages come one block into the next tile: O_A leaves through that K stage
// and O_B through that V stage, the producer's next load into either waiting
// until O's boxes have been read out of it.  The Q buffers are released as
// soon as each tile's last QK^T completes, so the next tile's Q loads run
// while the softmax warps write O.
#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace jfa {
namespace {

constexpr float kLn2f = 0.693147180559945309f;
constexpr float kRescaleLog2 = 8.0f;  // O is rescaled when a row's max grows by more than 2^8

struct Fwd2Cfg {
  static constexpr int D = 128;
  static constexpr int kChunkBytes = 128 * 128;  // [128 rows x 64 bf16]
  static constexpr int kTileBytes = 128 * D * 2;  // Q, K or V block
  static constexpr int kStages = 2;
  static constexpr int kOffQ = 0;                 // Q_A, Q_B
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kTileBytes;
  static constexpr int kOffXMax = kOffV + kStages * kTileBytes;  // [tile][buf][group][128] f32
  static constexpr int kOffXSum = kOffXMax + 2 * 2 * 2 * 128 * 4;  // [tile][buf][group][2][128] f32
  static constexpr int kOffBar = kOffXSum + 2 * 2 * 2 * 2 * 128 * 4;
  static constexpr int kBarBytes = 1024;
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + alignment slack
  static constexpr uint32_t kColS = 0;    // S_X at kColS + 128 X
  static constexpr uint32_t kColO = 256;  // O_X at kColO + 128 X
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 352;
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;  // slot A's issuer (and TMEM owner); warp 10 issues for slot B
};

struct Fwd2Bars {
  uint64_t q_full[2], q_free[2];  // per tile slot X (A = 0, B = 1)
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t ko_free[2], vo_free[2];  // per stage: O boxes staged there at a tile end read out
  uint64_t s_full[2], p_full[2], pv_done[2], o_empty[2];
  uint64_t max_ready[2][2][4];  // [slot][buffer][TMEM lane quadrant]
  uint64_t sum_ready[2][2][4];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct PTile {
  int b, h, mp, cost;
};
__device__ __forceinline__ PTile load_ptile(const int32_t* tiles, int i) {
  const int4 t = __ldg(reinterpret_cast<const int4*>(tiles) + i);
  return {t.x, t.y, t.z, t.w};
}

__device__ __forceinline__ bool warp_wait2(uint32_t bar, uint32_t parity, const Abort& ab) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
}

__device__ __forceinline__ void drain_wait2(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
// TMA producer (one thread): per tile Q_A and Q_B (each once its buffer's O
// boxes from the previous tile are read out), then K one block ahead of V.
// ---------------------------------------------------------------------------
__device__ void fwd2_producer(const FwdArgs& a, const CUtensorMap* q_map, const CUtensorMap* k_map,
                              const CUtensorMap* v_map, uint32_t sbase, Fwd2Bars& bars,
                              const Abort& ab) {
  using C = Fwd2Cfg;
  tma_prefetch_desc(q_map);
  tma_prefetch_desc(k_map);
  tma_prefetch_desc(v_map);
  uint32_t nq[2] = {0, 0}, nk = 0, nv = 0;  // Q loads per slot, K and V loads issued
  // per stage: an epilogue stages O there (set when a tile's last block is
  // loaded into it) and the waits done for that so far
  bool k_held[2] = {false, false}, v_held[2] = {false, false};
  uint32_t k_waits[2] = {0, 0}, v_waits[2] = {0, 0};
  bool ok = true;
  for (int i = a.cta_ptr[blockIdx.x]; i < a.cta_ptr[blockIdx.x + 1] && ok; ++i) {
    const PTile t = load_ptile(a.tiles, i);
    if (t.cost == 0) continue;
    const int kv0 = a.pb.kv_off[t.b];
    const int q0 = (a.pb.q_off ? a.pb.q_off[t.b] : 0) + t.mp * 256;
    const int x0 = t.h * C::D;
    auto load_k = [&](int j) -> bool {
      const uint32_t st = nk % C::kStages, ph = (nk / C::kStages) & 1;
      if (!mbar_wait(smem_u32(&bars.k_empty[st]), ph ^ 1, ab)) return false;
      if (k_held[st]) {  // O_A of an earlier tile leaves through this stage
        if (!mbar_wait(smem_u32(&bars.ko_free[st]), k_waits[st] & 1, ab)) return false;
        ++k_waits[st];
        k_held[st] = false;
      }
      mbar_arrive_expect_tx(smem_u32(&bars.k_full[st]), C::kTileBytes);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tma_load_2d(sbase + C::kOffK + st * C::kTileBytes + c * C::kChunkBytes, k_map,
                    smem_u32(&bars.k_full[st]), x0 + c * 64, kv0 + j * 128);
      ++nk;
      if (j == t.cost - 1) k_held[st] = true;
      return true;
    };
    auto load_v = [&](int j) -> bool {
      const uint32_t st = nv % C::kStages, ph = (nv / C::kStages) & 1;
      if (!mbar_wait(smem_u32(&bars.v_empty[st]), ph ^ 1, ab)) return false;
      if (v_held[st]) {  // O_B of an earlier tile leaves through this stage
        if (!mbar_wait(smem_u32(&bars.vo_free[st]), v_waits[st] & 1, ab)) return false;
        ++v_waits[st];
        v_held[st] = false;
      }
      mbar_arrive_expect_tx(smem_u32(&bars.v_full[st]), C::kTileBytes);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tma_load_2d(sbase + C::kOffV + st * C::kTileBytes + c * C::kChunkBytes, v_map,
                    smem_u32(&bars.v_full[st]), x0 + c * 64, kv0 + j * 128);
      ++nv;
      if (j == t.cost - 1) v_held[st] = true;
      return true;
    };
    ok = load_k(0);
    for (int X = 0; X < 2 && ok; ++X) {
      ok = mbar_wait(smem_u32(&bars.q_free[X]), (nq[X] & 1) ^ 1, ab);
      if (!ok) break;
      mbar_arrive_expect_tx(smem_u32(&bars.q_full[X]), C::kTileBytes);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        tma_load_2d(sbase + C::kOffQ + X * C::kTileBytes + c * C::kChunkBytes, q_map,
                    smem_u32(&bars.q_full[X]), x0 + c * 64, q0 + X * 128);
      ++nq[X];
    }
    if (!ok) break;
    for (int j = 0; j < t.cost && ok; ++j) {
      if (j + 1 < t.cost) ok = load_k(j + 1);
      if (ok) ok = load_v(j);
    }
  }
  // every copy issued lands before the CTA may exit
  for (int X = 0; X < 2; ++X)
    if (nq[X] > 0) drain_wait2(smem_u32(&bars.q_full[X]), (nq[X] - 1) & 1);
  for (uint32_t st = 0; st < C::kStages; ++st) {
    if (st < nk) {
      const uint32_t last = nk - 1 - ((nk - 1 - st) % C::kStages);
      drain_wait2(smem_u32(&bars.k_full[st]), (last / C::kStages) & 1);
    }
    if (st < nv) {
      const uint32_t last = nv - 1 - ((nv - 1 - st) % C::kStages);
      drain_wait2(smem_u32(&bars.v_full[st]), (last / C::kStages) & 1);
    }
  }
}

// ---------------------------------------------------------------------------
// MMA issuer of tile slot X (one thread each for A and B).  K and V stages are
// released by both issuers (two arrivals), the other barriers per slot.
// ---------------------------------------------------------------------------
__device__ void fwd2_mma(const FwdArgs& a, uint32_t sbase, uint32_t tmem, Fwd2Bars& bars, const Abort& ab,
                         int X) {
  using C = Fwd2Cfg;
  constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(128, C::D, false, true);
  const uint64_t qd = smem_desc_sw128(sbase + C::kOffQ + X * C::kTileBytes, 16, 1024);
  uint32_t g = 0, tq = 0;  // blocks and tiles done
  // S_X(gj) = Q_X K_gj^T into S_X, once PV_X(gj - 1) has read the P over it
  auto issue_s = [&](uint32_t gj) -> bool {
    const uint32_t st = gj % C::kStages, ph = (gj / C::kStages) & 1;
    if (!mbar_wait(smem_u32(&bars.k_full[st]), ph, ab)) return false;
    if (gj > 0 && !mbar_wait(smem_u32(&bars.pv_done[X]), (gj - 1) & 1, ab)) return false;
    tc_fence_after();
    const uint64_t kd = smem_desc_sw128(sbase + C::kOffK + st * C::kTileBytes, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < C::D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
      mma_bf16_ss(tmem + C::kColS + X * 128, desc_at(qd, off), desc_at(kd, off), idesc_qk, kk > 0 ? 1u : 0u);
    }
    mma_commit(smem_u32(&bars.s_full[X]));
    mma_commit(smem_u32(&bars.k_empty[st]));  // this slot's read of K_gj
    return true;
  };
  // O_X (+)= P_X(gj) V_gj; P of key columns [64 g, 64 g + 64) sits at S_X
  // columns [64 g, 64 g + 32)
  auto issue_pv = [&](uint32_t gj, bool first) -> bool {
    const uint32_t st = gj % C::kStages, ph = (gj / C::kStages) & 1;
    if (first && !mbar_wait(smem_u32(&bars.o_empty[X]), (tq & 1) ^ 1, ab)) return false;
    if (!mbar_wait(smem_u32(&bars.p_full[X]), gj & 1, ab)) return false;
    if (!mbar_wait(smem_u32(&bars.v_full[st]), ph, ab)) return false;
    tc_fence_after();
    const uint64_t vd = smem_desc_sw128(sbase + C::kOffV + st * C::kTileBytes, C::kChunkBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16_ts(tmem + C::kColO + X * 128, tmem + C::kColS + X * 128 + (kk >> 2) * 64 + (kk & 3) * 8,
                  desc_at(vd, kk * 2048), idesc_pv, (first && kk == 0) ? 0u : 1u);
    mma_commit(smem_u32(&bars.pv_done[X]));
    mma_commit(smem_u32(&bars.v_empty[st]));  // this slot's read of V_gj
    return true;
  };

  bool ok = true;
  for (int i = a.cta_ptr[blockIdx.x]; i < a.cta_ptr[blockIdx.x + 1] && ok; ++i) {
    const PTile t = load_ptile(a.tiles, i);
    if (t.cost == 0) continue;
    ok = mbar_wait(smem_u32(&bars.q_full[X]), tq & 1, ab);
    if (ok) ok = issue_s(g);
    // Q_X is free for the next tile once this tile's last QK^T has completed
    if (ok && t.cost == 1) mma_commit(smem_u32(&bars.q_free[X]));
    for (int j = 0; j < t.cost && ok; ++j) {
      ok = issue_pv(g + j, j == 0);
      if (ok && j + 1 < t.cost) {
        ok = issue_s(g + j + 1);
        if (ok && j + 2 == t.cost) mma_commit(smem_u32(&bars.q_free[X]));
      }
    }
    g += t.cost;
    ++tq;
  }
  // every product this thread issued has completed once this commit arrives
  // (the barrier completes when both issuers' commits have)
  mma_commit(smem_u32(&bars.drain));
  drain_wait2(smem_u32(&bars.drain), 0);
}

// ---------------------------------------------------------------------------
// softmax / epilogue (warps 0-7: group = warp / 4, thread = query row)
// ---------------------------------------------------------------------------
__device__ void fwd2_softmax(const FwdArgs& a, const CUtensorMap* o_map, uint8_t* smem, uint32_t tmem,
                             Fwd2Bars& bars, const Abort& ab, int grp) {
  using C = Fwd2Cfg;
  constexpr int D = C::D;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, wq = warp & 3;
  const int r = wq * 32 + lane;  // row of a tile, TMEM lane
  const uint32_t tl = tmem + (static_cast<uint32_t>(wq * 32) << 16);
  const int c0 = 64 * grp;  // this group's key columns of a block and O columns
  float* xmax = reinterpret_cast<float*>(smem + C::kOffXMax);
  float* xsum = reinterpret_cast<float*>(smem + C::kOffXSum);
  const float sl2 = a.scale_log2;
  const int H = a.pb.H;
  uint32_t g = 0, tq = 0;
  for (int i = a.cta_ptr[blockIdx.x]; i < a.cta_ptr[blockIdx.x + 1]; ++i) {
    const PTile t = load_ptile(a.tiles, i);
    const int64_t qlen = a.pb.q_off ? (a.pb.q_off[t.b + 1] - a.pb.q_off[t.b]) : a.pb.Lq;
    const int64_t o_base = (a.pb.q_off ? a.pb.q_off[t.b] : int64_t(t.b) * a.pb.Lq) + int64_t(t.mp) * 256;
    bool row_ok[2];
#pragma unroll
    for (int X = 0; X < 2; ++X) row_ok[X] = int64_t(t.mp) * 256 + X * 128 + r < qlen;
    if (t.cost == 0) {  // no keys: O = 0, LSE = -inf
      for (int X = 0; X < 2; ++X) {
        if (!row_ok[X]) continue;
        const int64_t orow = o_base + X * 128 + r;
        uint4* dst = reinterpret_cast<uint4*>(a.out + (orow * H + t.h) * D + c0);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        if (grp == 0) a.lse[int64_t(t.h) * a.pb.n_o + orow] = -INFINITY;
      }
      continue;
    }
    const int k_hi = (a.pb.kv_off[t.b + 1] - a.pb.kv_off[t.b]) - (t.cost - 1) * 128;  // keys of the last block
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f}, lr_run[2] = {0.0f, 0.0f};
    for (int j = 0; j < t.cost; ++j) {
      const uint32_t gj = g + j;
#pragma unroll
      for (int X = 0; X < 2; ++X) {
        const uint32_t sx = C::kColS + X * 128;
        if (!warp_wait2(smem_u32(&bars.s_full[X]), gj & 1, ab)) return;
        tc_fence_after();
        float s[64];
        {
          uint32_t vv[2][32];
          tmem_ld_x32_nw(tl + sx + c0, vv[0]);
          tmem_ld_x32_nw(tl + sx + c0 + 32, vv[1]);
          tmem_ld_wait2(vv[0], vv[1]);
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(vv[c][e]);
        }
        if (j == t.cost - 1 && k_hi < 128) {  // the peeled tail: keys past the sequence
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (c0 + e >= k_hi) s[e] = -INFINITY;
        }
        float mx = s[0];
#pragma unroll
        for (int e = 1; e < 64; ++e) mx = fmaxf(mx, s[e]);
        // combine with the other group's maximum of this row
        float* xm = xmax + ((X * 2 + (gj & 1)) * 2) * 128;
        xm[grp * 128 + r] = mx;
        mbar_arrive(smem_u32(&bars.max_ready[X][gj & 1][wq]));
        if (!warp_wait2(smem_u32(&bars.max_ready[X][gj & 1][wq]), (gj >> 1) & 1, ab)) return;
        mx = fmaxf(mx, xm[(grp ^ 1) * 128 + r]);
        const float m_cand = mx * sl2;
        const bool resc = m_cand > m_run[X] + kRescaleLog2;
        const float m_new = resc ? m_cand : m_run[X];
        const float alpha = resc ? fast_exp2(m_run[X] - m_new) : 1.0f;
        uint32_t p[32];
        uint64_t acc = f2_pack(0.0f, 0.0f);
        float r_lo = 0.0f, r_hi = 0.0f;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), negm = f2_pack(-m_new, -m_new);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(s[2 * e], s[2 * e + 1]), sl2x2, negm), x0, x1);
          const float p0 = fast_exp2(x0);
          const float p1 = fast_exp2(x1);
          p[e] = pack_bf16x2(p0, p1);
          acc = f2_add(acc, f2_pack(p0, p1));
          // O is normalised by the sum of the rounded weights the PV product
          // uses; LSE keeps the sum of the unrounded ones
          acc_bf16x2(p[e], r_lo, r_hi);
        }
        float a0, a1;
        f2_unpack(acc, a0, a1);
        l_run[X] = l_run[X] * alpha + (a0 + a1);
        lr_run[X] = lr_run[X] * alpha + (r_lo + r_hi);
        // S_X(gj) is committed after PV_X(gj - 1), so O_X holds it now
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t v[32];
            tmem_ld_x32(tl + C::kColO + X * 128 + c0 + c * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st_x32(tl + C::kColO + X * 128 + c0 + c * 32, v);
          }
        }
        // P over the S columns this group read: key columns [c0, c0 + 64)
        tmem_st_x32(tl + sx + c0, p);
        tmem_st_wait();
        tc_fence_before();
        // (failure-path test: CTA 0's first warp withholds its first arrival)
        if (!(a.test_skip == 1 && blockIdx.x == 0 && warp == 0 && gj == 0 && X == 0))
          mbar_arrive(smem_u32(&bars.p_full[X]));
        m_run[X] = m_new;
      }
    }
    // epilogues: combine the groups' row sums, wait for the tile's last PV,
    // normalise this group's O columns and store them through the K (tile A)
    // or V (tile B) stage of the last block, then hand the stage back
    const uint32_t gl = g + t.cost - 1, sl = gl % C::kStages;
#pragma unroll
    for (int X = 0; X < 2; ++X) {
      float* xs = xsum + ((X * 2 + (tq & 1)) * 2) * 256;  // [group][exact, rounded][128]
      xs[grp * 256 + r] = l_run[X];
      xs[grp * 256 + 128 + r] = lr_run[X];
      mbar_arrive(smem_u32(&bars.sum_ready[X][tq & 1][wq]));
      if (!warp_wait2(smem_u32(&bars.sum_ready[X][tq & 1][wq]), (tq >> 1) & 1, ab)) return;
      const float l_all = l_run[X] + xs[(grp ^ 1) * 256 + r];
      const float lr_all = lr_run[X] + xs[(grp ^ 1) * 256 + 128 + r];
      if (!warp_wait2(smem_u32(&bars.pv_done[X]), gl & 1, ab)) return;
      tc_fence_after();
      uint32_t ov[2][32];
      tmem_ld_x32_nw(tl + C::kColO + X * 128 + c0, ov[0]);
      tmem_ld_x32_nw(tl + C::kColO + X * 128 + c0 + 32, ov[1]);
      tmem_ld_wait2(ov[0], ov[1]);
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.o_empty[X]));  // O_X's columns are free for the next tile
      const float inv_l = 1.0f / lr_all;
      const int64_t orow = o_base + X * 128 + r;
      // a warp whose 32 rows all belong to the sequence stores them as one
      // swizzled box through that stage; others store their valid rows
      const bool staged = __all_sync(0xffffffffu, row_ok[X]);
      const uint32_t stg = smem_u32(smem + (X == 0 ? C::kOffK : C::kOffV) + sl * C::kTileBytes) +
                           grp * C::kChunkBytes + wq * 4096;
      uint16_t* orow_ptr = a.out + (orow * H + t.h) * D + c0;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(ov[c][2 * e]) * inv_l, __uint_as_float(ov[c][2 * e + 1]) * inv_l);
        if (staged) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_shared_v4(stg + lane * 128 + (((4 * c + q) ^ (lane & 7)) << 4), w[4 * q], w[4 * q + 1],
                         w[4 * q + 2], w[4 * q + 3]);
        } else if (row_ok[X]) {
          uint4* dst = reinterpret_cast<uint4*>(orow_ptr + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      if (staged) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (staged) {
          tma_store_2d(o_map, stg, t.h * D + c0, static_cast<int>(orow - lane));
          bulk_commit();
          bulk_wait_read_all();  // the box has left the stage
        }
        mbar_arrive(smem_u32(X == 0 ? &bars.ko_free[sl] : &bars.vo_free[sl]));
      }
      if (row_ok[X] && grp == 0) a.lse[int64_t(t.h) * a.pb.n_o + orow] = (m_run[X] + __log2f(l_all)) * kLn2f;
    }
    g += t.cost;
    ++tq;
  }
}

__global__ void __launch_bounds__(Fwd2Cfg::kThreads, 1)
    jfa_fwd2_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap o_map,
                    const FwdArgs a) {
  using C = Fwd2Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Fwd2Bars& bars = *reinterpret_cast<Fwd2Bars*>(smem + C::kOffBar);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int X = 0; X < 2; ++X) {
      mbar_init(smem_u32(&bars.q_full[X]), 1);
      mbar_init(smem_u32(&bars.q_free[X]), 1);   // slot X's issuer
      mbar_init(smem_u32(&bars.ko_free[X]), 8);  // lane 0 of each softmax warp (stage X)
      mbar_init(smem_u32(&bars.vo_free[X]), 8);
      mbar_init(smem_u32(&bars.k_full[X]), 1);
      mbar_init(smem_u32(&bars.k_empty[X]), 2);  // both issuers
      mbar_init(smem_u32(&bars.v_full[X]), 1);
      mbar_init(smem_u32(&bars.v_empty[X]), 2);
      mbar_init(smem_u32(&bars.s_full[X]), 1);
      mbar_init(smem_u32(&bars.p_full[X]), 256);
      mbar_init(smem_u32(&bars.pv_done[X]), 1);
      mbar_init(smem_u32(&bars.o_empty[X]), 256);
      for (int b = 0; b < 2; ++b)
        for (int q = 0; q < 4; ++q) {
          mbar_init(smem_u32(&bars.max_ready[X][b][q]), 64);
          mbar_init(smem_u32(&bars.sum_ready[X][b][q]), 64);
        }
    }
    mbar_init(smem_u32(&bars.drain), 2);
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
  if (warp == C::kProducerWarp) {
    if (lane == 0) fwd2_producer(a, &q_map, &k_map, &v_map, sbase, bars, ab);
    __syncwarp();
  } else if (warp == C::kMmaWarp || warp == C::kMmaWarp + 1) {
    if (lane == 0) fwd2_mma(a, sbase, tmem, bars, ab, warp - C::kMmaWarp);
    __syncwarp();
  } else {
    fwd2_softmax(a, &o_map, smem, tmem, bars, ab, warp >> 2);
    if (lane == 0) bulk_wait_all();  // O boxes written before the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace

cudaError_t launch_fwd_two(const FwdArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, const CUtensorMap& o_map, int grid, cudaStream_t stream) {
  using C = Fwd2Cfg;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  static_assert(sizeof(Fwd2Bars) <= C::kBarBytes, "barrier block");
  if (grid <= 0) return cudaSuccess;
  cudaError_t e = set_smem_limit_once<jfa_fwd2_kernel>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  jfa_fwd2_kernel<<<grid, C::kThreads, C::kSmemBytes, stream>>>(q_map, k_map, v_map, o_map, a);
  return cudaGetLastError();
}

}  // namespace jfa
