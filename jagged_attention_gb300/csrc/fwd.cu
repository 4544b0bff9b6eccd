// fwd.cu -- jagged FlashAttention forward for GB300 (sm_103a).
//
// One persistent CTA per SM walks its slice of the host-built schedule
// (tiles (b, h, query block m), zigzag-dealt by key/value cost).  For each
// tile it streams the sequence's key/value blocks through a TMA-fed shared
// memory ring and runs FlashAttention's online softmax:
//
//   S_j = Q K_j^T                  tcgen05.mma, fp32 accumulator in TMEM
//   m, l   running row max / sum   fp32 in registers, exp2 with scale*log2(e) folded in
//   P_j = exp2(S_j*c - m)          bf16, written back into TMEM
//   O  += P_j V_j                  tcgen05.mma with A = P_j from TMEM
//   O  /= l, LSE = m ln2 + ln l    epilogue
//
// The structure follows the roles the jagged FlashAttention pages describe
// (alphasignal page, "Specialized warps keep tensor cores busy": a load warp,
// an MMA warp, softmax/correction warps, output stores; a multi-stage K/V
// pipeline; persistent CTAs), re-derived for sm_103a:
//   warp 8      TMA producer (Q once per tile, K and V per block)
//   warp 9      tcgen05.mma issuer; owns the TMEM allocation
//   warps 0-3,  softmax + correction + epilogue: two groups share every query
//   warps 4-7   row (key columns [0, 64) and [64, 128) of each block, O
//               columns [0, D/2) and [D/2, D)) and exchange row maxima and
//               sums through shared memory
// TMEM (512 columns): two 128-column score buffers (so QK^T of block j+1
// overlaps the softmax of block j), the D-column O accumulator and two
// 64-column bf16 P buffers.  O is rescaled only when a row's max grows by
// more than 2^8 (the stale max keeps every P <= 256, exact after the final
// division by l).  The last, partial key block is the only one that masks
// (the pages' "loop peeling": the bulk pass is branch-free).
#include <type_traits>

#include "kernels.h"
#include "sm103_ptx.cuh"
#include "tiles.cuh"

namespace jfa {
namespace {

constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// kPair: a CTA of a pair (the 2-CTA form below) holds half of each K/V
// block: K rows [64 r, 64 r + 64) of the block with all D columns, and V's
// 64 columns [64 r, 64 r + 64) of all 128 rows (r = the CTA's rank).
template <int D, bool kPair = false>
struct FwdCfg {
  static constexpr int kChunks = D / 64;             // 128-byte column chunks per row
  static constexpr int kChunkBytes = 128 * 128;      // one [128 rows x 64 bf16] chunk
  static constexpr int kTileBytes = 128 * D * 2;     // one 128-row tile of Q, K or V
  static constexpr int kStages = kPair ? 4 : (D == 128) ? 2 : 4;  // K and V ring depth (keeps 1 CTA/SM)
  static constexpr int kKChunkBytes = kPair ? 64 * 128 : kChunkBytes;  // one 64-column chunk of K
  static constexpr int kKBytes = kPair ? 64 * D * 2 : kTileBytes;      // a K stage
  // K/V blocks the L2 prefetch runs ahead of the loads: the pair's ring
  // waits on load latency (two blocks ahead measured best); one CTA per
  // block is faster without it
  static constexpr int kPrefetch = kPair ? 2 : 0;
  static constexpr int kVBytes = kPair ? 128 * 64 * 2 : kTileBytes;    // a V stage
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTileBytes;
  static constexpr int kOffV = kOffK + kStages * kKBytes;
  // row statistics the two softmax groups exchange: per-block partial maxima
  // (2 buffers x 2 groups x 128 rows) and per-tile partial sums (2 buffers x
  // 2 groups x 2 sums x 128 rows)
  static constexpr int kOffXMax = kOffV + kStages * kVBytes;
  static constexpr int kOffXSum = kOffXMax + 2 * 2 * 128 * 4;
  // O leaves through shared memory at D = 128: per softmax group a
  // 128-byte-swizzled [128 rows x 64 bf16] box, stored by TMA a warp (32
  // rows) at a time
  static constexpr int kOffOStg = kOffXSum + 2 * 2 * 2 * 128 * 4;
  static constexpr int kOffBar = kOffOStg + (D == 128 ? 2 * 16384 : 0);
  static constexpr int kBarBytes = 640;
  static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;  // + barriers + alignment slack
  static constexpr uint32_t kColS = 0;               // 2 x 128 fp32 columns
  static constexpr uint32_t kColO = 256;             // D fp32 columns
  static constexpr uint32_t kColP = 256 + D;         // 2 x 64 columns of bf16 pairs
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 320;
  static constexpr int kProducerWarp = 8;
  static constexpr int kMmaWarp = 9;
};

struct FwdBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  // CTA pairs, in the even CTA: the odd CTA's loads of the same stages
  uint64_t q_pair, k_pair[4], v_pair[4];
  uint64_t s_full[2], s_empty[2], p_full[2], pv_done[2];
  uint64_t o_empty;
  // per buffer and TMEM lane quadrant (the two warps, one per group, that
  // share those 32 rows): both groups' partial row maxima of a block, and
  // partial row sums of a tile, are in shared memory
  uint64_t max_ready[2][4];
  uint64_t sum_ready[2][4];
  uint64_t drain;
  TileRing ring;  // dynamic schedules: tile indices from the producer to the other roles
  uint32_t tmem_base;
  int abort_flag;
};

struct Tile {
  int b, h, blk, cost;
};
__device__ __forceinline__ Tile load_tile(const int32_t* tiles, int i) {
  const int4 t = __ldg(reinterpret_cast<const int4*>(tiles) + i);
  return {t.x, t.y, t.z, t.w};
}

// Wait with every lane of the warp, and agree on the outcome so that the
// warp stays converged for the .sync.aligned tcgen05 instructions after it.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Abort& ab) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
}

// Bounded wait used only while draining at exit: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// ---------------------------------------------------------------------------
// TMA producer (one thread)
// ---------------------------------------------------------------------------
// CTA pairs (kPair): both CTAs of a pair walk the same pair tiles
// {b, h, mp, cost}; CTA r takes query block 2 mp + r and loads its half of
// every K/V block (see FwdCfg).
template <int D, bool kPack, bool kPair, class Seq>
__device__ void fwd_producer(const FwdArgs& a, const CUtensorMap* q_map, const CUtensorMap* k_map,
                             const CUtensorMap* v_map, uint32_t sbase, FwdBars& bars,
                             const Abort& ab, Seq& seq, uint32_t rank) {
  using C = FwdCfg<D, kPair>;
  tma_prefetch_desc(q_map);
  tma_prefetch_desc(k_map);
  tma_prefetch_desc(v_map);
  const uint32_t sQ = sbase + C::kOffQ;
  uint32_t nq = 0, nk = 0, nv = 0;  // loads issued
  bool ok = true;
  // L2 prefetch cursor (static schedules): walks this CTA's blocks, across
  // tile boundaries, kPrefetch blocks ahead of the K loads, so that DRAM
  // reads start earlier than the shared-memory ring alone would let them
  [[maybe_unused]] int pf_i = 0, pf_end = 0, pf_j = 0;
  [[maybe_unused]] uint32_t npf = 0;
  constexpr bool kStatic = std::is_same_v<Seq, TileSeq<false>>;
  if constexpr (kStatic) {
    pf_i = seq.i;
    pf_end = seq.end;
  }
  auto prefetch_to = [&](uint32_t target) {
    if constexpr (kStatic && C::kPrefetch > 0) {
      while (npf < target && pf_i < pf_end) {
        const Tile u = load_tile(a.tiles, pf_i);
        if (pf_j >= u.cost) {
          ++pf_i;
          pf_j = 0;
          continue;
        }
        const int y = a.pb.kv_off[u.b] + pf_j * 128, x = u.h * D;
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_prefetch_l2_2d(k_map, x + c * 64, y + (kPair ? 64 * int(rank) : 0));
        if constexpr (kPair) {
          tma_prefetch_l2_2d(v_map, x + 64 * int(rank), y);
        } else {
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c) tma_prefetch_l2_2d(v_map, x + c * 64, y);
        }
        ++pf_j;
        ++npf;
      }
    }
  };
  auto next = [&] { return seq.claim(a.dyn_counter, a.T, bars.ring, ab); };
  for (int i = next(); i >= 0 && ok; i = next()) {
    const Tile t = load_tile(a.tiles, i);
    if (t.cost == 0) continue;
    const int kv0 = a.pb.kv_off[t.b];
    const int mblk = kPair ? 2 * t.blk + int(rank) : (kPack ? max(t.blk, 0) : t.blk);
    const int qrow = (a.pb.q_off ? a.pb.q_off[t.b] : 0) + mblk * 128;
    const int x0 = t.h * D;
    ok = mbar_wait(smem_u32(&bars.q_empty), (nq & 1) ^ 1, ab);
    if (!ok) break;
    mbar_arrive_expect_tx(smem_u32(&bars.q_full), C::kTileBytes);
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c)
      tma_load_2d(sQ + c * C::kChunkBytes, q_map, smem_u32(&bars.q_full), x0 + c * 64, qrow);
    ++nq;
    // K runs one block ahead of V: a V load waits for the PV two blocks
    // back, which must not hold up the K the next QK^T needs
    auto load_k = [&](int j) -> bool {
      const uint32_t st = nk % C::kStages, ph = (nk / C::kStages) & 1;
      if (!mbar_wait(smem_u32(&bars.k_empty[st]), ph ^ 1, ab)) return false;
      mbar_arrive_expect_tx(smem_u32(&bars.k_full[st]), C::kKBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)  // a pair's CTA: its 64 of the block's keys
        tma_load_2d(sbase + C::kOffK + st * C::kKBytes + c * C::kKChunkBytes, k_map,
                    smem_u32(&bars.k_full[st]), x0 + c * 64, kv0 + j * 128 + (kPair ? 64 * int(rank) : 0));
      ++nk;
      prefetch_to(nk + C::kPrefetch);
      return true;
    };
    auto load_v = [&](int j) -> bool {
      const uint32_t st = nv % C::kStages, ph = (nv / C::kStages) & 1;
      if (!mbar_wait(smem_u32(&bars.v_empty[st]), ph ^ 1, ab)) return false;
      mbar_arrive_expect_tx(smem_u32(&bars.v_full[st]), C::kVBytes);
      if constexpr (kPair) {  // its 64 of the head's D columns, all 128 keys
        tma_load_2d(sbase + C::kOffV + st * C::kVBytes, v_map, smem_u32(&bars.v_full[st]),
                    x0 + 64 * int(rank), kv0 + j * 128);
      } else {
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_2d(sbase + C::kOffV + st * C::kVBytes + c * C::kChunkBytes, v_map,
                      smem_u32(&bars.v_full[st]), x0 + c * 64, kv0 + j * 128);
      }
      ++nv;
      return true;
    };
    ok = load_k(0);
    for (int j = 0; j < t.cost && ok; ++j) {
      if (j + 1 < t.cost) ok = load_k(j + 1);
      if (ok) ok = load_v(j);
    }
  }
  // Let every copy this thread issued land before the CTA can exit: the last
  // phase issued on each full barrier completes when its bytes arrive, and
  // nothing else completes phases of the full barriers.
  if (nq > 0) drain_wait(smem_u32(&bars.q_full), (nq - 1) & 1);
  for (uint32_t st = 0; st < C::kStages; ++st) {
    if (st < nk) {
      const uint32_t last = nk - 1 - ((nk - 1 - st) % C::kStages);  // last K load into stage st
      drain_wait(smem_u32(&bars.k_full[st]), (last / C::kStages) & 1);
    }
    if (st < nv) {
      const uint32_t last = nv - 1 - ((nv - 1 - st) % C::kStages);
      drain_wait(smem_u32(&bars.v_full[st]), (last / C::kStages) & 1);
    }
  }
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread).  kPair: the even CTA's thread issues the pair's
// products -- S = Q K^T with M = 256 (each CTA's 128 query rows) and N = 128
// keys (each CTA's 64-key half of K), and O += P V with P from each CTA's
// TMEM and V's D columns split in halves -- and commits each to the barrier
// of that name in both CTAs.  It waits for the odd CTA's loads through the
// *_pair barriers (the odd CTA's forwarder arrives on them) and for the
// softmax warps of both CTAs (s_empty, p_full, o_empty count one arrival per
// warp of either CTA).
// ---------------------------------------------------------------------------
template <int D, bool kPair, class Seq>
__device__ void fwd_mma(const FwdArgs& a, uint32_t sbase, uint32_t tmem, FwdBars& bars,
                        const Abort& ab, Seq& seq) {
  using C = FwdCfg<D, kPair>;
  constexpr int M = kPair ? 256 : 128;
  constexpr uint32_t idesc_qk = idesc_bf16_f32(M, 128, false, false);
  constexpr uint32_t idesc_pv = idesc_bf16_f32(M, D, false, true);
  const uint64_t qd = smem_desc_sw128(sbase + C::kOffQ, 16, 1024);
  uint32_t g = 0, tq = 0;
  // phases the other CTA's threads arrive on are acquired at cluster scope
  auto wait_x = [&](uint32_t bar, uint32_t parity) -> bool {
    if constexpr (kPair) return mbar_wait_cluster(bar, parity, ab);
    else return mbar_wait(bar, parity, ab);
  };
  auto commit = [&](uint32_t bar) {
    if constexpr (kPair) mma_commit_pair(bar);
    else mma_commit(bar);
  };

  // O += P_gp V_gp; `first` marks the first block of a tile (overwrite O).
  auto issue_pv = [&](uint32_t gp, bool first) -> bool {
    const uint32_t pb = gp & 1, st = gp % C::kStages, ph = (gp / C::kStages) & 1;
    if (first && !wait_x(smem_u32(&bars.o_empty), (tq & 1) ^ 1)) return false;
    if (!wait_x(smem_u32(&bars.p_full[pb]), (gp >> 1) & 1)) return false;
    if (!mbar_wait(smem_u32(&bars.v_full[st]), ph, ab)) return false;
    if (kPair && !wait_x(smem_u32(&bars.v_pair[st]), ph)) return false;
    tc_fence_after();
    const uint64_t vd = smem_desc_sw128(sbase + C::kOffV + st * C::kVBytes, C::kChunkBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      if constexpr (kPair)
        mma_pair_ts(tmem + C::kColO, tmem + C::kColP + pb * 64 + kk * 8, desc_at(vd, kk * 2048), idesc_pv,
                    (first && kk == 0) ? 0u : 1u);
      else
        mma_bf16_ts(tmem + C::kColO, tmem + C::kColP + pb * 64 + kk * 8, desc_at(vd, kk * 2048), idesc_pv,
                    (first && kk == 0) ? 0u : 1u);
    }
    commit(smem_u32(&bars.v_empty[st]));
    commit(smem_u32(&bars.pv_done[pb]));
    return true;
  };

  bool ok = true;
  auto next = [&] { return seq.take(a.dyn_counter, bars.ring, ab); };
  for (int i = next(); i >= 0 && ok; i = next()) {
    const Tile t = load_tile(a.tiles, i);
    if (t.cost == 0) continue;
    ok = mbar_wait(smem_u32(&bars.q_full), tq & 1, ab);
    if (kPair && ok) ok = wait_x(smem_u32(&bars.q_pair), tq & 1);
    for (int j = 0; j < t.cost && ok; ++j) {
      const uint32_t gj = g + j, st = gj % C::kStages, sb = gj & 1, ph = (gj / C::kStages) & 1;
      ok = mbar_wait(smem_u32(&bars.k_full[st]), ph, ab) &&
           (!kPair || wait_x(smem_u32(&bars.k_pair[st]), ph)) &&
           wait_x(smem_u32(&bars.s_empty[sb]), ((gj >> 1) & 1) ^ 1);
      if (!ok) break;
      tc_fence_after();
      const uint64_t kd = smem_desc_sw128(sbase + C::kOffK + st * C::kKBytes, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t koff = (kk & 3) * 32;
        if constexpr (kPair)
          mma_pair_ss(tmem + C::kColS + sb * 128, desc_at(qd, (kk >> 2) * C::kChunkBytes + koff),
                      desc_at(kd, (kk >> 2) * C::kKChunkBytes + koff), idesc_qk, kk > 0 ? 1u : 0u);
        else
          mma_bf16_ss(tmem + C::kColS + sb * 128, desc_at(qd, (kk >> 2) * C::kChunkBytes + koff),
                      desc_at(kd, (kk >> 2) * C::kKChunkBytes + koff), idesc_qk, kk > 0 ? 1u : 0u);
      }
      commit(smem_u32(&bars.s_full[sb]));
      commit(smem_u32(&bars.k_empty[st]));
      if (j == t.cost - 1) commit(smem_u32(&bars.q_empty));
      if (j >= 1) ok = issue_pv(gj - 1, j == 1);
    }
    if (ok) ok = issue_pv(g + t.cost - 1, t.cost == 1);
    g += t.cost;
    ++tq;
  }
  // every MMA issued above has completed once this commit arrives
  commit(smem_u32(&bars.drain));
  drain_wait(smem_u32(&bars.drain), 0);
}

// The odd CTA of a pair: after each of its own loads lands, tell the even
// CTA's MMA issuer (which cannot wait on another CTA's barrier) through the
// matching *_pair barrier there.  One thread, walking the same loads as the
// producer.
template <int D, class Seq>
__device__ void fwd_pair_forwarder(const FwdArgs& a, FwdBars& bars, const Abort& ab, Seq& seq) {
  using C = FwdCfg<D, true>;
  uint32_t nq = 0, nk = 0, nv = 0;
  auto next = [&] { return seq.take(a.dyn_counter, bars.ring, ab); };
  for (int i = next(); i >= 0; i = next()) {
    const Tile t = load_tile(a.tiles, i);
    if (t.cost == 0) continue;
    if (!mbar_wait(smem_u32(&bars.q_full), nq & 1, ab)) return;
    mbar_arrive_rank0(smem_u32(&bars.q_pair));
    ++nq;
    for (int j = 0; j < t.cost; ++j) {
      uint32_t st = nk % C::kStages;
      if (!mbar_wait(smem_u32(&bars.k_full[st]), (nk / C::kStages) & 1, ab)) return;
      mbar_arrive_rank0(smem_u32(&bars.k_pair[st]));
      ++nk;
      st = nv % C::kStages;
      if (!mbar_wait(smem_u32(&bars.v_full[st]), (nv / C::kStages) & 1, ab)) return;
      mbar_arrive_rank0(smem_u32(&bars.v_pair[st]));
      ++nv;
    }
  }
}

// ---------------------------------------------------------------------------
// softmax / correction / epilogue (warps 0-7 in two groups, thread = query row = TMEM lane)
// ---------------------------------------------------------------------------
template <int D, bool kPack, bool kPair, class Seq>
__device__ void fwd_softmax(const FwdArgs& a, const CUtensorMap* o_map, uint8_t* smem, uint32_t tmem,
                            FwdBars& bars, const Abort& ab, Seq& seq, int grp, uint32_t rank) {
  using C = FwdCfg<D, kPair>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = (warp & 3) * 32 + lane;  // row of the tile, TMEM lane
  const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  const int c0 = 64 * grp;               // this group's key columns in a block
  const int o0 = grp * (D / 2);          // and O columns
  float* xmax = reinterpret_cast<float*>(smem + C::kOffXMax);  // [2][2][128]
  float* xsum = reinterpret_cast<float*>(smem + C::kOffXSum);  // [2][2][2][128]
  const float sl2 = a.scale_log2;
  const int H = a.pb.H;
  uint32_t g = 0, tq = 0;
  // an arrival the MMA issuer waits for: each thread's, or (CTA pairs) one per
  // warp, on the barrier in the even CTA, whose thread issues for both.  These
  // report tensor-memory reads and stores the warp has waited for, so the odd
  // CTA's remote arrival needs no release of its other memory writes.
  auto arrive_mma = [&](uint32_t bar) {
    if constexpr (kPair) {
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(bar);
        else mbar_arrive_rank0_relaxed(bar);
      }
    } else {
      mbar_arrive(bar);
    }
  };

  auto next = [&] { return seq.take_warp(a.dyn_counter, bars.ring, ab); };
  for (int i = next(); i >= 0; i = next()) {
    const Tile t = load_tile(a.tiles, i);
    // packed tile (blk = -nseq): rows [off[b], off[b + nseq]) of nseq short
    // sequences, one key block, each row masked to its own sequence's keys
    const bool packed = kPack && t.blk < 0;
    const int mblk = kPair ? 2 * t.blk + int(rank) : packed ? 0 : t.blk;
    const int64_t qlen = a.pb.q_off ? (a.pb.q_off[t.b + (packed ? -t.blk : 1)] - a.pb.q_off[t.b]) : a.pb.Lq;
    const int64_t o_first = (a.pb.q_off ? a.pb.q_off[t.b] : int64_t(t.b) * a.pb.Lq) + mblk * 128;
    const bool row_ok = int64_t(mblk) * 128 + r < qlen;
    const int64_t orow = o_first + r;
    uint16_t* orow_ptr = a.out + (orow * H + t.h) * D + o0;
    if (t.cost == 0) {  // no keys: O = 0, LSE = -inf
      if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow_ptr);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        if (grp == 0) a.lse[int64_t(t.h) * a.pb.n_o + orow] = -INFINITY;
      }
      continue;
    }
    // keys this row may see in the last (peeled) block: [k_lo, k_hi); a
    // packed tile's single block limits each row to its own sequence
    int k_lo = 0, k_hi = (a.pb.kv_off[t.b + 1] - a.pb.kv_off[t.b]) - (t.cost - 1) * 128;
    if (packed) {
      k_hi = 128;  // rows past the pack: never stored
      if (row_ok) {
        const int base = a.pb.kv_off[t.b], row = base + r;
        int sq = t.b;
        while (a.pb.kv_off[sq + 1] <= row) ++sq;  // the sequence holding this row
        k_lo = a.pb.kv_off[sq] - base;
        k_hi = a.pb.kv_off[sq + 1] - base;
      }
    }
    // the group's partial sums (exact and of the bf16-rounded weights); the
    // running max is the same in both groups (they combine their maxima)
    float m_run = -INFINITY, l_run = 0.0f, lr_run = 0.0f;
    for (int j = 0; j < t.cost; ++j) {
      const uint32_t gj = g + j, sb = gj & 1;
      if (!warp_wait(smem_u32(&bars.s_full[sb]), (gj >> 1) & 1, ab)) return;
      tc_fence_after();
      float s[64];
      {  // both halves of this group's columns, one wait
        uint32_t vv[2][32];
        tmem_ld_x32_nw(tl + C::kColS + sb * 128 + c0, vv[0]);
        tmem_ld_x32_nw(tl + C::kColS + sb * 128 + c0 + 32, vv[1]);
        tmem_ld_wait2(vv[0], vv[1]);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(vv[c][e]);
      }
      tc_fence_before();
      arrive_mma(smem_u32(&bars.s_empty[sb]));
      if (j == t.cost - 1) {  // peeled tail: keys outside the sequence
        if (packed) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (c0 + e < k_lo || c0 + e >= k_hi) s[e] = -INFINITY;
        } else if (k_hi < 128) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (c0 + e >= k_hi) s[e] = -INFINITY;
        }
      }
      float mx = s[0];
#pragma unroll
      for (int e = 1; e < 64; ++e) mx = fmaxf(mx, s[e]);
      // combine with the other group's maximum of this row
      float* xm = xmax + (gj & 1) * 256;
      xm[grp * 128 + r] = mx;
      mbar_arrive(smem_u32(&bars.max_ready[gj & 1][warp & 3]));
      if (!warp_wait(smem_u32(&bars.max_ready[gj & 1][warp & 3]), (gj >> 1) & 1, ab)) return;
      mx = fmaxf(mx, xm[(grp ^ 1) * 128 + r]);
      const float m_cand = mx * sl2;
      const bool resc = m_cand > m_run + kRescaleThreshold;
      const float m_new = resc ? m_cand : m_run;
      const float alpha = resc ? fast_exp2(m_run - m_new) : 1.0f;
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
        // uses (an exact convex combination of V rows under those weights);
        // LSE keeps the sum of the unrounded ones
        acc_bf16x2(p[e], r_lo, r_hi);
      }
      float rowsum, rowsum_r;
      {
        float a0, a1;
        f2_unpack(acc, a0, a1);
        rowsum = a0 + a1;
        rowsum_r = r_lo + r_hi;
      }
      l_run = l_run * alpha + rowsum;
      lr_run = lr_run * alpha + rowsum_r;
      // the P buffer is free once PV of block gj-2 has completed
      if (!warp_wait(smem_u32(&bars.pv_done[sb]), ((gj >> 1) & 1) ^ 1, ab)) return;
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        const uint32_t gp = gj - 1;  // O must hold PV of block gj-1 before rescaling
        if (!warp_wait(smem_u32(&bars.pv_done[gp & 1]), (gp >> 1) & 1, ab)) return;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t v[32];
          tmem_ld_x32(tl + C::kColO + o0 + c * 32, v);
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tmem_st_x32(tl + C::kColO + o0 + c * 32, v);
        }
      }
      // P of key columns [c0, c0 + 64) = packed columns [32 grp, 32 grp + 32)
      tmem_st_x32(tl + C::kColP + sb * 64 + grp * 32, p);
      tmem_st_wait();
      tc_fence_before();
      // (failure-path test: CTA 0's first warp withholds its first arrival)
      if (!(a.test_skip == 1 && blockIdx.x == 0 && warp == 0 && gj == 0))
        arrive_mma(smem_u32(&bars.p_full[sb]));
      m_run = m_new;
    }
    // epilogue: combine the groups' row sums, wait for the last PV,
    // normalise this group's O columns, store O and LSE
    float* xs = xsum + (tq & 1) * 512;  // [group][exact, rounded][128]
    xs[grp * 256 + r] = l_run;
    xs[grp * 256 + 128 + r] = lr_run;
    mbar_arrive(smem_u32(&bars.sum_ready[tq & 1][warp & 3]));
    if (!warp_wait(smem_u32(&bars.sum_ready[tq & 1][warp & 3]), (tq >> 1) & 1, ab)) return;
    l_run += xs[(grp ^ 1) * 256 + r];
    lr_run += xs[(grp ^ 1) * 256 + 128 + r];
    const uint32_t gl = g + t.cost - 1;
    if (!warp_wait(smem_u32(&bars.pv_done[gl & 1]), (gl >> 1) & 1, ab)) return;
    tc_fence_after();
    const float inv_l = 1.0f / lr_run;
    // a warp whose 32 rows all belong to the tile stages them for one TMA
    // store (row-wise scattered 16-byte stores reach a fraction of the memory
    // system's rate); a warp with rows past the sequence stores its valid rows
    const bool staged = D == 128 && __all_sync(0xffffffffu, row_ok);
    const uint32_t stg_warp = smem_u32(smem + C::kOffOStg) + grp * 16384 + (warp & 3) * 4096;
    if (staged) {
      if (lane == 0) bulk_wait_read_all();  // this warp's previous O box has been read out
      __syncwarp();
    }
    uint32_t ov[D / 64][32];
    if constexpr (D == 128) {
      tmem_ld_x32_nw(tl + C::kColO + o0, ov[0]);
      tmem_ld_x32_nw(tl + C::kColO + o0 + 32, ov[D / 64 - 1]);
      tmem_ld_wait2(ov[0], ov[D / 64 - 1]);
    } else {
      tmem_ld_x32(tl + C::kColO + o0, ov[0]);
    }
    tc_fence_before();
    arrive_mma(smem_u32(&bars.o_empty));  // O's columns are free for the next tile
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      const uint32_t (&v)[32] = ov[c];
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * inv_l, __uint_as_float(v[2 * e + 1]) * inv_l);
      if (staged) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_shared_v4(stg_warp + lane * 128 + (((4 * c + q) ^ (lane & 7)) << 4), w[4 * q], w[4 * q + 1],
                       w[4 * q + 2], w[4 * q + 3]);
      } else if (row_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow_ptr + c * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      }
    }
    if (staged) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(o_map, stg_warp, t.h * D + o0, static_cast<int>(orow - lane));
        bulk_commit();
      }
    }
    if (row_ok && grp == 0) a.lse[int64_t(t.h) * a.pb.n_o + orow] = (m_run + __log2f(l_run)) * kLn2;
    g += t.cost;
    ++tq;
  }
}

template <int D, bool kPack, bool kDyn, bool kPair>
__global__ void __launch_bounds__(FwdCfg<D, kPair>::kThreads, 1)
    jfa_fwd_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap k_map,
                   const __grid_constant__ CUtensorMap v_map,
                   const __grid_constant__ CUtensorMap o_map, const FwdArgs a) {
  using C = FwdCfg<D, kPair>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  FwdBars& bars = *reinterpret_cast<FwdBars*>(smem + C::kOffBar);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = kPair ? cluster_rank() : 0;
  // arrivals the MMA issuer waits for: every softmax thread, or one per softmax
  // warp of both CTAs of a pair
  constexpr uint32_t kSoftmaxArrivals = kPair ? 16 : 256;
  if (tid == 0) {
    tile_ring_init(bars.ring, 1 + 8);  // consumers: the MMA thread and the 8 softmax warps
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_empty), 1);
    mbar_init(smem_u32(&bars.q_pair), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.v_empty[s]), 1);
      mbar_init(smem_u32(&bars.k_pair[s]), 1);
      mbar_init(smem_u32(&bars.v_pair[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars.s_full[s]), 1);
      mbar_init(smem_u32(&bars.s_empty[s]), kSoftmaxArrivals);
      mbar_init(smem_u32(&bars.p_full[s]), kSoftmaxArrivals);
      for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&bars.max_ready[s][q]), 64);
      for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&bars.sum_ready[s][q]), 64);
      mbar_init(smem_u32(&bars.pv_done[s]), 1);
    }
    mbar_init(smem_u32(&bars.o_empty), kSoftmaxArrivals);
    mbar_init(smem_u32(&bars.drain), 1);
    bars.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kMmaWarp) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(&bars.tmem_base), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&bars.tmem_base), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  const Abort ab{&bars.abort_flag, a.status, a.wait_limit_ns ? a.wait_limit_ns : kWaitLimitNs};
  // a pair's two CTAs walk the pair's slice of the schedule
  TileSeq<kDyn> seq(a.cta_ptr, a.dyn_counter, kPair ? int(blockIdx.x >> 1) : int(blockIdx.x));

  if (warp == C::kProducerWarp) {
    if (lane == 0) fwd_producer<D, kPack, kPair>(a, &q_map, &k_map, &v_map, sbase, bars, ab, seq, rank);
    __syncwarp();
  } else if (warp == C::kMmaWarp) {
    if (lane == 0) {
      if (rank == 0) {
        fwd_mma<D, kPair>(a, sbase, tmem, bars, ab, seq);
      } else if constexpr (kPair) {
        fwd_pair_forwarder<D>(a, bars, ab, seq);
        drain_wait(smem_u32(&bars.drain), 0);  // the even CTA's last products have completed
      }
    }
    __syncwarp();
  } else {
    fwd_softmax<D, kPack, kPair>(a, &o_map, smem, tmem, bars, ab, seq, warp >> 2, rank);
    if (lane == 0) bulk_wait_all();  // O boxes written before the CTA exits
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // neither CTA leaves while the pair's products run
  if (warp == C::kMmaWarp) {
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tmem, C::kTmemCols);
    else tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool kPack, bool kDyn, bool kPair>
cudaError_t launch_fwd_d(const FwdArgs& a, const CUtensorMap& q, const CUtensorMap& k,
                         const CUtensorMap& v, const CUtensorMap& o, int grid, cudaStream_t stream) {
  using C = FwdCfg<D, kPair>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  static_assert(sizeof(FwdBars) <= C::kBarBytes, "barrier block");
  cudaError_t e = set_smem_limit_once<jfa_fwd_kernel<D, kPack, kDyn, kPair>>(C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if constexpr (kPair) {  // clusters of two CTAs, grid = 2 x pairs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, jfa_fwd_kernel<D, kPack, kDyn, kPair>, q, k, v, o, a);
    if (e != cudaSuccess) return e;
  } else {
    jfa_fwd_kernel<D, kPack, kDyn, kPair><<<grid, C::kThreads, C::kSmemBytes, stream>>>(q, k, v, o, a);
  }
  return cudaGetLastError();
}

// packed plans, dynamic schedules and CTA pairs run their own instantiations
template <int D>
cudaError_t launch_fwd_m(const FwdArgs& a, const CUtensorMap& q, const CUtensorMap& k,
                         const CUtensorMap& v, const CUtensorMap& o, int grid, cudaStream_t stream) {
  if (a.dyn_counter)
    return a.packed ? launch_fwd_d<D, true, true, false>(a, q, k, v, o, grid, stream)
                    : launch_fwd_d<D, false, true, false>(a, q, k, v, o, grid, stream);
  return a.packed ? launch_fwd_d<D, true, false, false>(a, q, k, v, o, grid, stream)
                  : launch_fwd_d<D, false, false, false>(a, q, k, v, o, grid, stream);
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, const CUtensorMap& q_map, const CUtensorMap& k_map,
                       const CUtensorMap& v_map, const CUtensorMap& o_map, int grid,
                       cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  // plans with packed short sequences run an instantiation that handles
  // packed tiles; the others keep the plain code path
  if (a.pair) {  // D = 128, static schedule, plain tiles: grid = 2 x pairs
    if (a.pb.D != 128 || a.packed || a.dyn_counter || (grid & 1)) return cudaErrorInvalidValue;
    return launch_fwd_d<128, false, false, true>(a, q_map, k_map, v_map, o_map, grid, stream);
  }
  if (a.pb.D == 128)
    return launch_fwd_m<128>(a, q_map, k_map, v_map, o_map, grid, stream);
  return launch_fwd_m<64>(a, q_map, k_map, v_map, o_map, grid, stream);
}

}  // namespace jfa
