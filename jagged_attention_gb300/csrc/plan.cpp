// plan.cpp -- host-side tile schedules for the persistent kernels.
//
// Forward: the jagged FlashAttention pages balance forward work on the host:
// tiles are sorted by key/value workload and dealt to the SMs back and forth
// (alphasignal page, "Five changes unlocked the gains", item 1; yuxiaoba
// note, "Why both static and dynamic balancing help").  Backward: the valid
// (batch, head, key/value-block) tiles are precomputed and dealt round-robin
// (same note; asivanadi0 blog, "Structural changes and layered opts",
// item 1).  The exact order (enumeration b, h, block; stable sort by cost
// descending; CTA k on even rounds, P-1-k on odd rounds) is this library's
// reading of those passages.
#include "plan.h"

#include <algorithm>
#include <numeric>

namespace jfa {

static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool validate_offsets(const int32_t* off, int B, int64_t* total) {
  if (off == nullptr || B < 1) return false;
  if (off[0] != 0) return false;
  for (int b = 0; b < B; ++b)
    if (off[b + 1] < off[b]) return false;
  // int32 offsets already bound the total below 2^31
  *total = off[B];
  return true;
}

std::vector<int> short_packs(const std::vector<int64_t>& len) {
  const int B = static_cast<int>(len.size());
  std::vector<int> pack(B, 1);
  int b = 0;
  while (b < B) {
    if (len[b] == 0 || len[b] > kBM) {
      ++b;
      continue;
    }
    int64_t total = len[b];
    int e = b + 1, nonempty = 1;
    while (e < B && total + len[e] <= kBM) {
      total += len[e];
      nonempty += len[e] > 0;
      ++e;
    }
    if (nonempty >= 2) {
      pack[b] = e - b;
      for (int i = b + 1; i < e; ++i) pack[i] = 0;
      b = e;
    } else {
      ++b;
    }
  }
  return pack;
}

// Indices of the T tiles in `flat` by cost field, largest first, equal costs
// in enumeration order (a stable sort).  Costs are block counts, so their
// range is usually small next to T and a counting sort does this in linear
// time (block-diagonal batches have hundreds of thousands of tiles); a
// comparison sort covers wide ranges.
static std::vector<int> by_cost_descending(const std::vector<int32_t>& flat, int T) {
  std::vector<int> order(T);
  if (T == 0) return order;
  int32_t lo = flat[3], hi = flat[3];
  for (int i = 1; i < T; ++i) {
    lo = std::min(lo, flat[4 * static_cast<size_t>(i) + 3]);
    hi = std::max(hi, flat[4 * static_cast<size_t>(i) + 3]);
  }
  const int64_t range = int64_t(hi) - lo + 1;
  if (range <= 4 * int64_t(T) + 1024) {
    std::vector<int> next(static_cast<size_t>(range) + 1, 0);  // bucket hi - cost
    for (int i = 0; i < T; ++i) ++next[static_cast<size_t>(hi - flat[4 * static_cast<size_t>(i) + 3]) + 1];
    for (int64_t k = 0; k < range; ++k) next[k + 1] += next[k];
    for (int i = 0; i < T; ++i) order[next[static_cast<size_t>(hi - flat[4 * static_cast<size_t>(i) + 3])]++] = i;
    return order;
  }
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return flat[4 * size_t(a) + 3] > flat[4 * size_t(b) + 3]; });
  return order;
}

// Dynamic schedules: the tiles in claim order, one queue for every CTA.
static Schedule claim_order(const std::vector<int32_t>& flat, int num_ctas) {
  Schedule s;
  s.T = static_cast<int>(flat.size() / 4);
  s.P = std::min(num_ctas, s.T);
  s.cta_ptr.assign(s.P + 1, s.T);  // one queue: [0, T), the same for every CTA
  s.cta_ptr[0] = 0;
  const std::vector<int> order = by_cost_descending(flat, s.T);
  s.tiles.resize(4 * static_cast<size_t>(s.T));
  for (int i = 0; i < s.T; ++i)
    std::copy_n(&flat[4 * static_cast<size_t>(order[i])], 4, &s.tiles[4 * static_cast<size_t>(i)]);
  return s;
}

Schedule build_fwd_schedule(const std::vector<int64_t>& q_len, const std::vector<int64_t>& kv_len,
                            int H, int num_ctas, const std::vector<int>* pack, bool dynamic) {
  const int B = static_cast<int>(q_len.size());
  std::vector<int32_t> flat;  // enumeration order
  int64_t count = 0;
  for (int b = 0; b < B; ++b)
    count += (pack && (*pack)[b] != 1) ? ((*pack)[b] >= 2 ? H : 0) : H * cdiv(q_len[b], kBM);
  flat.reserve(4 * static_cast<size_t>(count));
  for (int b = 0; b < B; ++b) {
    if (pack && (*pack)[b] != 1) {
      if ((*pack)[b] >= 2)
        for (int h = 0; h < H; ++h) {
          flat.push_back(b);
          flat.push_back(h);
          flat.push_back(-(*pack)[b]);
          flat.push_back(1);
        }
      continue;
    }
    const int32_t cost = static_cast<int32_t>(cdiv(kv_len[b], kBN));
    const int64_t mblocks = cdiv(q_len[b], kBM);
    for (int h = 0; h < H; ++h)
      for (int64_t m = 0; m < mblocks; ++m) {
        flat.push_back(b);
        flat.push_back(h);
        flat.push_back(static_cast<int32_t>(m));
        flat.push_back(cost);
      }
  }
  if (dynamic) return claim_order(flat, num_ctas);
  Schedule s;
  s.T = static_cast<int>(flat.size() / 4);
  s.P = std::min(num_ctas, s.T);
  s.cta_ptr.assign(s.P + 1, 0);
  if (s.T == 0) return s;
  const std::vector<int> order = by_cost_descending(flat, s.T);
  // deal: sorted tile i -> round r = i / P, position k = i % P, zigzag across
  // rounds (r and k kept as running counters: no division per tile)
  std::vector<int> cta_of(s.T);
  for (int i = 0, r = 0, k = 0; i < s.T; ++i) {
    cta_of[i] = (r % 2 == 0) ? k : s.P - 1 - k;
    ++s.cta_ptr[cta_of[i] + 1];
    if (++k == s.P) {
      k = 0;
      ++r;
    }
  }
  for (int c = 0; c < s.P; ++c) s.cta_ptr[c + 1] += s.cta_ptr[c];
  s.tiles.resize(4 * static_cast<size_t>(s.T));
  std::vector<int32_t> fill(s.cta_ptr.begin(), s.cta_ptr.end() - 1);
  for (int i = 0; i < s.T; ++i) {  // i increases with the round, so each CTA's list is in round order
    const int dst = fill[cta_of[i]]++;
    std::copy_n(&flat[4 * static_cast<size_t>(order[i])], 4, &s.tiles[4 * static_cast<size_t>(dst)]);
  }
  return s;
}

Schedule build_bwd_schedule(const std::vector<int64_t>& q_len, const std::vector<int64_t>& kv_len,
                            int H, int num_ctas, const std::vector<int>* pack, bool dynamic) {
  const int B = static_cast<int>(q_len.size());
  std::vector<int32_t> flat;
  int64_t count = 0;
  for (int b = 0; b < B; ++b)
    count += (pack && (*pack)[b] != 1) ? ((*pack)[b] >= 2 ? H : 0)
                                       : (q_len[b] == 0 ? 0 : H * cdiv(kv_len[b], kBN));
  flat.reserve(4 * static_cast<size_t>(count));
  for (int b = 0; b < B; ++b) {
    if (pack && (*pack)[b] != 1) {
      if ((*pack)[b] >= 2)
        for (int h = 0; h < H; ++h) {
          flat.push_back(b);
          flat.push_back(h);
          flat.push_back(-(*pack)[b]);
          flat.push_back(1);
        }
      continue;
    }
    if (q_len[b] == 0) continue;
    const int32_t qblocks = static_cast<int32_t>(cdiv(q_len[b], kBM));
    const int64_t nblocks = cdiv(kv_len[b], kBN);
    for (int h = 0; h < H; ++h)
      for (int64_t n = 0; n < nblocks; ++n) {
        flat.push_back(b);
        flat.push_back(h);
        flat.push_back(static_cast<int32_t>(n));
        flat.push_back(qblocks);
      }
  }
  if (dynamic) return claim_order(flat, num_ctas);
  Schedule s;
  s.T = static_cast<int>(flat.size() / 4);
  s.P = std::min(num_ctas, s.T);
  s.cta_ptr.assign(s.P + 1, 0);
  if (s.T == 0) return s;
  // tile i -> CTA i % P: CTA c receives T / P tiles, one more when c < T % P
  for (int c = 0; c < s.P; ++c) s.cta_ptr[c + 1] = s.cta_ptr[c] + s.T / s.P + (c < s.T % s.P ? 1 : 0);
  s.tiles.resize(4 * static_cast<size_t>(s.T));
  std::vector<int32_t> fill(s.cta_ptr.begin(), s.cta_ptr.end() - 1);
  for (int i = 0, c = 0; i < s.T; ++i) {
    const int dst = fill[c]++;
    std::copy_n(&flat[4 * static_cast<size_t>(i)], 4, &s.tiles[4 * static_cast<size_t>(dst)]);
    if (++c == s.P) c = 0;
  }
  return s;
}

}  // namespace jfa
