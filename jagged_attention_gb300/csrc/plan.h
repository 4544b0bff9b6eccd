// plan.h -- host-side tile schedules and the plan object behind jfa_plan_t.
#pragma once
#include <cstdint>
#include <utility>
#include <vector>

namespace jfa {

constexpr int kBM = 128;  // query rows per forward tile / per backward query block
constexpr int kBN = 128;  // key rows per key/value block / per backward tile

// A schedule: T tiles of four int32 {b, h, block, cost}, grouped by CTA, and
// the CSR row pointer over the P CTAs that receive work.
struct Schedule {
  std::vector<int32_t> tiles;    // 4 * T
  std::vector<int32_t> cta_ptr;  // P + 1
  int T = 0;
  int P = 0;
};

// Check offsets: off[0] == 0, non-decreasing, total < 2^31.  Returns the
// total through *total.  false on any violation.
bool validate_offsets(const int32_t* off, int B, int64_t* total);

// Packing of short sequences (self mode with one shared offsets array): a run
// of consecutive sequences whose lengths add up to at most 128 rows, with at
// least two non-empty ones, becomes one tile {b0, h, -nseq, 1} covering rows
// [off[b0], off[b0 + nseq]) with a block-diagonal mask.  pack[b] is nseq for a
// pack starting at b, 0 for a sequence inside a pack, and 1 otherwise.
std::vector<int> short_packs(const std::vector<int64_t>& len);

// Forward schedule: tiles (b, h, m) for m < ceil(Lq_b / BM) with cost
// ceil(Lk_b / BN), stable-sorted by cost descending, dealt zigzag to
// P = min(num_ctas, T) CTAs.
// `pack` (optional) replaces packed runs by one tile each.  dynamic: instead
// of the deal, every tile once in claim order (stable sort by the last field,
// descending) with cta_ptr = {0, T, ..., T}; the CTAs claim tiles at run time.
Schedule build_fwd_schedule(const std::vector<int64_t>& q_len, const std::vector<int64_t>& kv_len,
                            int H, int num_ctas, const std::vector<int>* pack = nullptr,
                            bool dynamic = false);
// Backward schedule: tiles (b, h, n) for n < ceil(Lk_b / BN) where Lq_b > 0,
// cost ceil(Lq_b / BM), dealt round-robin (or in claim order, as above).
Schedule build_bwd_schedule(const std::vector<int64_t>& q_len, const std::vector<int64_t>& kv_len,
                            int H, int num_ctas, const std::vector<int>* pack = nullptr,
                            bool dynamic = false);

}  // namespace jfa

struct jfa_plan {
  int B = 0, H = 0, Lq = 0, D = 0;
  bool broadcast = false;
  bool packed = false;       // short sequences packed into shared tiles
  // query row ranges [begin, end) whose dQ the backward reduce-adds (or never
  // writes) and the pre-pass therefore clears: broadcast mode's shared rows,
  // and in self mode the sequences with no key or more than one key block
  // (a sequence with one key block, or in a packed tile, has one tile that
  // stores its rows)
  std::vector<std::pair<int64_t, int64_t>> dq_rows_to_clear;
  bool dq_own_rows = false;  // some rows are left to the tiles that own them
  bool fwd_dynamic = false;  // forward tiles claimed at run time
  bool bwd_dynamic = false;  // backward tiles claimed at run time
  // every sequence with queries has at most one key block, so each backward
  // tile meets all the keys of its queries and forms Delta itself: the
  // pre-pass skips the Delta kernel (unless JFA_PLAN_DELTA_PREPASS)
  bool own_delta = false;
  // the forward runs as CTA pairs over pairs of query blocks; `fwd` then
  // holds the pair schedule, P pairs (2 P CTAs)
  bool fwd_pair = false;
  // the forward runs two query tiles per CTA; `fwd` then holds the tiles of
  // two query blocks, over P CTAs
  bool fwd_two = false;
  // failure-path test only (jfa_plan_selftest)
  int test_skip = 0;
  uint64_t test_limit_ns = 0;
  int* d_counters = nullptr; // dynamic: claim counters [fwd, bwd]
  int device = 0;
  int num_ctas = 0;
  int64_t n_q = 0;   // rows of Q
  int64_t n_o = 0;   // rows of O / dO / LSE
  int64_t n_kv = 0;  // rows of K / V
  jfa::Schedule fwd, bwd;
  // key/value row ranges [begin, end) of sequences that have keys but no
  // queries: no backward tile covers them, so their dK / dV are cleared
  std::vector<std::pair<int64_t, int64_t>> kv_rows_without_queries;
  // device copies (one allocation)
  void* dev_block = nullptr;
  int32_t* d_kv_off = nullptr;
  int32_t* d_q_off = nullptr;  // null in broadcast mode
  int32_t* d_fwd_tiles = nullptr;
  int32_t* d_fwd_ptr = nullptr;
  int32_t* d_bwd_tiles = nullptr;
  int32_t* d_bwd_ptr = nullptr;
  int* d_status = nullptr;
};
