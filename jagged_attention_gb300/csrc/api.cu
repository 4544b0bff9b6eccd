// api.cu -- the C ABI declared in include/jfa.h: argument checks, plans,
// TMA descriptors and kernel launches.  No allocation happens in jfa_fwd /
// jfa_bwd; plans own their (small) device copies of offsets and schedules.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "jfa.h"
#include "kernels.h"
#include "plan.h"

using jfa::Schedule;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// TMA descriptor of a packed bf16 tensor viewed as 2-D [rows, H*D]: boxes of
// 128 rows x 64 columns (128 bytes) with the 128-byte swizzle the MMA
// descriptors expect.  Rows past the end read as zeros.  An empty tensor gets
// a zeroed descriptor that no tile ever uses.
// box_rows = 32: the unit one warp stores O (forward) or dK / dV (backward) in.
int make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, unsigned box_rows = 128) {
  std::memset(m, 0, sizeof(*m));
  if (rows == 0) return JFA_OK;
  auto enc = tensor_map_encoder();
  if (!enc) return JFA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? JFA_OK : JFA_ERR_CUDA;
}

// TMA descriptor of the fp32 dQ viewed as 2-D [rows, H*D]: boxes of 32 rows x
// 32 columns (128 bytes, 128-byte swizzle), the unit one warp of the backward
// reduce-adds (or stores) from shared memory.  Out-of-range rows are skipped.
int make_map_dq(CUtensorMap* m, const float* ptr, int64_t rows, int64_t cols) {
  std::memset(m, 0, sizeof(*m));
  if (rows == 0) return JFA_OK;
  auto enc = tensor_map_encoder();
  if (!enc) return JFA_ERR_CUDA;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? JFA_OK : JFA_ERR_CUDA;
}

jfa::Problem problem_of(const jfa_plan* p) {
  jfa::Problem pb;
  pb.kv_off = p->d_kv_off;
  pb.q_off = p->d_q_off;
  pb.B = p->B;
  pb.H = p->H;
  pb.Lq = p->Lq;
  pb.D = p->D;
  pb.n_q = p->n_q;
  pb.n_o = p->n_o;
  pb.n_kv = p->n_kv;
  return pb;
}

// A plan's device block and launches belong to the device that was current
// when it was created; calls that use them must run with that device current.
int check_device(const jfa_plan* p) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_CUDA;
  return dev == p->device ? JFA_OK : JFA_ERR_INVALID_ARG;
}

// Lengths from host offsets; q_off == nullptr means broadcast with Lq rows.
int lengths_of(const int32_t* kv_off, const int32_t* q_off, int B, int Lq,
               std::vector<int64_t>& qlen, std::vector<int64_t>& kvlen, int64_t* n_kv,
               int64_t* n_q) {
  if (!jfa::validate_offsets(kv_off, B, n_kv)) return JFA_ERR_BAD_OFFSETS;
  if (q_off) {
    if (!jfa::validate_offsets(q_off, B, n_q)) return JFA_ERR_BAD_OFFSETS;
  } else {
    if (Lq < 0) return JFA_ERR_INVALID_ARG;
    *n_q = Lq;
  }
  qlen.resize(B);
  kvlen.resize(B);
  for (int b = 0; b < B; ++b) {
    kvlen[b] = kv_off[b + 1] - kv_off[b];
    qlen[b] = q_off ? (q_off[b + 1] - q_off[b]) : Lq;
  }
  return JFA_OK;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Every sequence that has queries has at most one key block: each backward
// tile then meets all the keys of its queries and can form Delta itself.
bool tiles_hold_all_keys(const std::vector<int64_t>& qlen, const std::vector<int64_t>& kvlen) {
  for (size_t b = 0; b < qlen.size(); ++b)
    if (qlen[b] > 0 && kvlen[b] > jfa::kBN) return false;
  return true;
}

// Mean number of key rows the backward tiles hold (a packed tile counts the
// rows of all its sequences).
double mean_tile_keys(const jfa::Schedule& s, const int32_t* kv_off) {
  if (s.T == 0) return 0.0;
  double rows = 0.0;
  for (int t = 0; t < s.T; ++t) {
    const int b = s.tiles[4 * t], n = s.tiles[4 * t + 2];
    rows += n < 0 ? kv_off[b - n] - kv_off[b]
                  : std::min<int64_t>(jfa::kBN, int64_t(kv_off[b + 1] - kv_off[b]) - int64_t(n) * jfa::kBN);
  }
  return rows / s.T;
}

// Whether the backward tiles form Delta.  Forming it costs every step of a
// tile the same cross-lane sums however few key rows the tile holds, while
// the pre-pass it replaces costs in proportion to the rows: on the GB300 it
// paid with full tiles (64-token segments packed two per tile: step -11%)
// and came out even with half-full ones (the same segments one per tile:
// 15.08 against 15.05 ms), so by default tiles form it when they hold at
// least 96 key rows on average.
bool tiles_form_delta(unsigned flags, const std::vector<int64_t>& qlen,
                      const std::vector<int64_t>& kvlen, const jfa::Schedule& bwd,
                      const int32_t* kv_off) {
  if ((flags & JFA_PLAN_DELTA_PREPASS) || !tiles_hold_all_keys(qlen, kvlen)) return false;
  return (flags & JFA_PLAN_DELTA_IN_TILES) || mean_tile_keys(bwd, kv_off) >= 96.0;
}

// Whether the forward runs as CTA pairs (two CTAs of a cluster take the two
// query blocks of a pair tile and share each K/V block, the tensor-core
// products spanning both: cta_group::2): on request, where the pair kernel
// exists (D = 128, static schedule, no packed tiles) and there are queries.
bool use_fwd_pairs(unsigned flags, int D, bool packed, bool dynamic, int num_ctas,
                   const std::vector<int64_t>& qlen) {
  if (!(flags & JFA_PLAN_FWD_PAIRS) || D != 128 || packed || dynamic || num_ctas < 2) return false;
  for (const int64_t q : qlen)
    if (q > 0) return true;
  return false;
}

// Query lengths in units of pair tiles: the forward schedule over query
// blocks of 2 * 128 rows is the one over blocks of 128 rows of half-length
// sequences (ceil(ceil(q / 128) / 2) = ceil(ceil(q / 2) / 128)).
std::vector<int64_t> pair_lengths(const std::vector<int64_t>& qlen) {
  std::vector<int64_t> h(qlen.size());
  for (size_t b = 0; b < qlen.size(); ++b) h[b] = (qlen[b] + 1) / 2;
  return h;
}

// Which passes claim their tiles at run time: both with JFA_PLAN_DYNAMIC,
// neither with JFA_PLAN_STATIC, else the backward in self mode only.
bool claims_fwd(unsigned flags) { return (flags & JFA_PLAN_DYNAMIC) != 0; }
bool claims_bwd(unsigned flags, bool broadcast) {
  return (flags & JFA_PLAN_DYNAMIC) != 0 || (!(flags & JFA_PLAN_STATIC) && !broadcast);
}
bool bad_flags(unsigned flags) {
  return ((flags & JFA_PLAN_PACK_SHORT) && (flags & JFA_PLAN_NO_PACK)) ||
         ((flags & JFA_PLAN_DYNAMIC) && (flags & JFA_PLAN_STATIC)) ||
         __builtin_popcount(flags & (JFA_PLAN_FWD_PAIRS | JFA_PLAN_FWD_TWO | JFA_PLAN_FWD_ONE)) > 1;
}

// Whether the forward runs two query tiles per CTA: on request, or by default
// where the tiles of two query blocks hold at least 3 key blocks on average
// and at most a quarter of them have an empty second block; only where that
// kernel exists (D = 128, static schedule, no packed tiles) and there are
// queries.
bool use_fwd_two(unsigned flags, int D, int H, bool packed, bool dynamic, int num_ctas,
                 const std::vector<int64_t>& qlen, const std::vector<int64_t>& kvlen) {
  if ((flags & (JFA_PLAN_FWD_ONE | JFA_PLAN_FWD_PAIRS)) || D != 128 || packed || dynamic) return false;
  int64_t tiles = 0, half = 0, blocks = 0;
  for (size_t b = 0; b < qlen.size(); ++b) {
    const int64_t nb = (qlen[b] + jfa::kBM - 1) / jfa::kBM, nt = (nb + 1) / 2;
    tiles += nt;
    half += nb & 1;
    blocks += nt * ((kvlen[b] + jfa::kBN - 1) / jfa::kBN);
  }
  if (tiles == 0) return false;
  if (flags & JFA_PLAN_FWD_TWO) return true;
  // fewer than four tiles per CTA: halving the tile count costs more balance
  // than the second tile gains (jagged self, ~2 per CTA, measured 5% slower)
  return blocks >= 3 * tiles && 4 * half <= tiles && tiles * H >= 4 * int64_t(num_ctas);
}

// Whether the plan packs short sequences, and the packing (pack[b] as
// short_packs gives it) when it does.  Packing needs self mode with one
// offsets array for queries and keys.  JFA_PLAN_PACK_SHORT packs whenever a
// run forms, JFA_PLAN_NO_PACK never; by default a plan packs when that
// removes at least an eighth of its forward tiles (a pack of n non-empty
// sequences replaces n one-block tiles by one).
bool use_packing(unsigned flags, const int32_t* kv_off, const int32_t* q_off, int B,
                 const std::vector<int64_t>& kvlen, std::vector<int>* pack) {
  if ((flags & JFA_PLAN_NO_PACK) || !q_off) return false;
  if (std::memcmp(kv_off, q_off, (B + 1) * sizeof(int32_t)) != 0) return false;
  std::vector<int> p = jfa::short_packs(kvlen);
  int64_t saved = 0, tiles = 0;
  for (int b = 0; b < B; ++b) {
    tiles += (kvlen[b] + jfa::kBM - 1) / jfa::kBM;
    if (p[b] > 1) {
      int64_t nonempty = 0;
      for (int i = b; i < b + p[b]; ++i) nonempty += kvlen[i] > 0;
      saved += nonempty - 1;
    }
  }
  if (saved == 0 || (!(flags & JFA_PLAN_PACK_SHORT) && 8 * saved < tiles)) return false;
  *pack = std::move(p);
  return true;
}

// The schedule choices a plan makes from its sizes, offsets and flags (plan
// creation and the host-only jfa_plan_choices share this).
struct PlanChoices {
  bool packed = false, fwd_dynamic = false, bwd_dynamic = false, fwd_pair = false, fwd_two = false;
  std::vector<int> pack;
};
PlanChoices choose(unsigned flags, const int32_t* kv_off, const int32_t* q_off, int B, int H, int D,
                   int num_ctas, const std::vector<int64_t>& qlen, const std::vector<int64_t>& kvlen) {
  PlanChoices c;
  c.packed = use_packing(flags, kv_off, q_off, B, kvlen, &c.pack);
  c.fwd_dynamic = claims_fwd(flags);
  c.bwd_dynamic = claims_bwd(flags, q_off == nullptr);
  c.fwd_pair = use_fwd_pairs(flags, D, c.packed, c.fwd_dynamic, num_ctas, qlen);
  c.fwd_two = !c.fwd_pair && use_fwd_two(flags, D, H, c.packed, c.fwd_dynamic, num_ctas, qlen, kvlen);
  return c;
}

}  // namespace

extern "C" {

const char* jfa_status_string(int s) {
  switch (s) {
    case JFA_OK: return "ok";
    case JFA_ERR_INVALID_ARG: return "invalid argument";
    case JFA_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case JFA_ERR_BAD_OFFSETS: return "bad offsets";
    case JFA_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case JFA_ERR_WORKSPACE: return "workspace missing or too small";
    case JFA_ERR_CUDA: return "CUDA runtime error";
    case JFA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int jfa_build_tiles(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                    int Lq, int num_ctas, int dir, unsigned flags, int32_t* tiles_out,
                    int32_t* cta_ptr_out, int* T, int* P) {
  if (!kv_offsets_host || B < 1 || H < 1 || num_ctas < 1 || dir < 0 || dir > 2 || !T || !P)
    return JFA_ERR_INVALID_ARG;
  if (bad_flags(flags)) return JFA_ERR_INVALID_ARG;
  std::vector<int64_t> qlen, kvlen;
  int64_t n_kv = 0, n_q = 0;
  int rc = lengths_of(kv_offsets_host, q_offsets_host, B, Lq, qlen, kvlen, &n_kv, &n_q);
  if (rc != JFA_OK) return rc;
  std::vector<int> pack;
  const bool packing = use_packing(flags, kv_offsets_host, q_offsets_host, B, kvlen, &pack);
  const Schedule s =
      dir == 0 ? jfa::build_fwd_schedule(qlen, kvlen, H, num_ctas, packing ? &pack : nullptr, claims_fwd(flags))
      : dir == 1 ? jfa::build_bwd_schedule(qlen, kvlen, H, num_ctas, packing ? &pack : nullptr,
                                          claims_bwd(flags, q_offsets_host == nullptr))
                 : jfa::build_fwd_schedule(pair_lengths(qlen), kvlen, H, num_ctas, nullptr, false);
  *T = s.T;
  *P = s.P;
  if (tiles_out) std::memcpy(tiles_out, s.tiles.data(), s.tiles.size() * sizeof(int32_t));
  if (cta_ptr_out) std::memcpy(cta_ptr_out, s.cta_ptr.data(), s.cta_ptr.size() * sizeof(int32_t));
  return JFA_OK;
}

int jfa_delta_in_tiles(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B,
                       int Lq, unsigned flags, int* in_tiles) {
  if (!kv_offsets_host || B < 1 || !in_tiles) return JFA_ERR_INVALID_ARG;
  if ((flags & JFA_PLAN_DELTA_PREPASS) && (flags & JFA_PLAN_DELTA_IN_TILES)) return JFA_ERR_INVALID_ARG;
  if (bad_flags(flags)) return JFA_ERR_INVALID_ARG;
  std::vector<int64_t> qlen, kvlen;
  int64_t n_kv = 0, n_q = 0;
  int rc = lengths_of(kv_offsets_host, q_offsets_host, B, Lq, qlen, kvlen, &n_kv, &n_q);
  if (rc != JFA_OK) return rc;
  std::vector<int> pack;
  const bool packing = use_packing(flags, kv_offsets_host, q_offsets_host, B, kvlen, &pack);
  // the mean tile fill does not depend on the head count or the CTA count
  const Schedule s = jfa::build_bwd_schedule(qlen, kvlen, 1, 1, packing ? &pack : nullptr, false);
  *in_tiles = tiles_form_delta(flags, qlen, kvlen, s, kv_offsets_host) ? 1 : 0;
  return JFA_OK;
}

int jfa_plan_choices(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                     int Lq, int D, int num_ctas, unsigned flags, int* fwd_form, int* fwd_claims,
                     int* bwd_claims, int* packed) {
  if (!kv_offsets_host || B < 1 || H < 1 || num_ctas < 1) return JFA_ERR_INVALID_ARG;
  if ((flags & JFA_PLAN_DELTA_PREPASS) && (flags & JFA_PLAN_DELTA_IN_TILES)) return JFA_ERR_INVALID_ARG;
  if (bad_flags(flags)) return JFA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
  std::vector<int64_t> qlen, kvlen;
  int64_t n_kv = 0, n_q = 0;
  int rc = lengths_of(kv_offsets_host, q_offsets_host, B, Lq, qlen, kvlen, &n_kv, &n_q);
  if (rc != JFA_OK) return rc;
  const PlanChoices ch = choose(flags, kv_offsets_host, q_offsets_host, B, H, D, num_ctas, qlen, kvlen);
  if (fwd_form) *fwd_form = ch.fwd_pair ? 1 : ch.fwd_two ? 2 : 0;
  if (fwd_claims) *fwd_claims = ch.fwd_dynamic ? 1 : 0;
  if (bwd_claims) *bwd_claims = ch.bwd_dynamic ? 1 : 0;
  if (packed) *packed = ch.packed ? 1 : 0;
  return JFA_OK;
}

int jfa_plan_create(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                    int Lq, int D, int num_ctas, void* stream, jfa_plan_t* out) {
  return jfa_plan_create_ex(kv_offsets_host, q_offsets_host, B, H, Lq, D, num_ctas, 0u, stream, out);
}

int jfa_plan_create_ex(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                       int Lq, int D, int num_ctas, unsigned flags, void* stream, jfa_plan_t* out) {
  if (!out || !kv_offsets_host || B < 1 || H < 1 || num_ctas < 0) return JFA_ERR_INVALID_ARG;
  *out = nullptr;
  if ((flags & JFA_PLAN_DELTA_PREPASS) && (flags & JFA_PLAN_DELTA_IN_TILES)) return JFA_ERR_INVALID_ARG;
  if (bad_flags(flags)) return JFA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
  std::vector<int64_t> qlen, kvlen;
  int64_t n_kv = 0, n_q = 0;
  int rc = lengths_of(kv_offsets_host, q_offsets_host, B, Lq, qlen, kvlen, &n_kv, &n_q);
  if (rc != JFA_OK) return rc;
  const int64_t n_o = q_offsets_host ? n_q : int64_t(B) * Lq;
  if (n_o >= (int64_t(1) << 31) || int64_t(H) * D * 2 >= (int64_t(1) << 31))
    return JFA_ERR_UNSUPPORTED;

  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return JFA_ERR_CUDA;
  if (major != 10 || minor != 3) return JFA_ERR_UNSUPPORTED;  // built for sm_103a only

  auto* p = new jfa_plan();
  p->B = B;
  p->H = H;
  p->Lq = q_offsets_host ? 0 : Lq;
  p->D = D;
  p->broadcast = q_offsets_host == nullptr;
  p->device = dev;
  p->num_ctas = num_ctas > 0 ? num_ctas : sms;
  p->n_q = n_q;
  p->n_o = n_o;
  p->n_kv = n_kv;
  const PlanChoices ch = choose(flags, kv_offsets_host, q_offsets_host, B, H, D, p->num_ctas, qlen, kvlen);
  const std::vector<int>& pack = ch.pack;
  p->packed = ch.packed;
  if (!q_offsets_host) {
    if (n_q > 0) p->dq_rows_to_clear.emplace_back(0, n_q);
  } else {
    for (int b = 0; b < B; ++b) {
      const int64_t s = q_offsets_host[b], e = q_offsets_host[b + 1];
      if (e == s) continue;
      if (p->packed && pack[b] != 1) continue;   // a packed tile stores these rows
      if (kvlen[b] > 0 && kvlen[b] <= jfa::kBN) continue;  // one key block: its tile stores
      if (!p->dq_rows_to_clear.empty() && p->dq_rows_to_clear.back().second == s)
        p->dq_rows_to_clear.back().second = e;
      else
        p->dq_rows_to_clear.emplace_back(s, e);
    }
    // many runs, or most of the rows: one clear of the whole dQ costs less
    // than a launch per run (clearing rows a tile then stores is harmless)
    int64_t rows = 0;
    for (const auto& r : p->dq_rows_to_clear) rows += r.second - r.first;
    if (p->dq_rows_to_clear.size() > 4 || 2 * rows > n_q) {
      p->dq_rows_to_clear.clear();
      p->dq_rows_to_clear.emplace_back(0, n_q);
    } else {
      p->dq_own_rows = true;
    }
  }
  p->fwd_dynamic = ch.fwd_dynamic;
  p->bwd_dynamic = ch.bwd_dynamic;
  p->fwd_pair = ch.fwd_pair;
  p->fwd_two = ch.fwd_two;
  p->fwd = p->fwd_pair  ? jfa::build_fwd_schedule(pair_lengths(qlen), kvlen, H, p->num_ctas / 2, nullptr, false)
           : p->fwd_two ? jfa::build_fwd_schedule(pair_lengths(qlen), kvlen, H, p->num_ctas, nullptr, false)
                        : jfa::build_fwd_schedule(qlen, kvlen, H, p->num_ctas, p->packed ? &pack : nullptr,
                                                  p->fwd_dynamic);
  p->bwd = jfa::build_bwd_schedule(qlen, kvlen, H, p->num_ctas, p->packed ? &pack : nullptr, p->bwd_dynamic);
  p->own_delta = tiles_form_delta(flags, qlen, kvlen, p->bwd, kv_offsets_host);
  for (int b = 0; b < B; ++b) {
    if (qlen[b] == 0 && kvlen[b] > 0) {
      const int64_t s = kv_offsets_host[b], e = kv_offsets_host[b + 1];
      if (!p->kv_rows_without_queries.empty() && p->kv_rows_without_queries.back().second == s)
        p->kv_rows_without_queries.back().second = e;
      else
        p->kv_rows_without_queries.emplace_back(s, e);
    }
  }

  // one device block: offsets, schedules, status word and the two claim
  // counters of dynamic schedules (16-byte aligned pieces)
  const size_t o_kv = 0;
  const size_t o_q = align_up(o_kv + (B + 1) * 4, 16);
  const size_t o_ft = align_up(o_q + (q_offsets_host ? (B + 1) * 4 : 0), 16);
  const size_t o_fp = align_up(o_ft + p->fwd.tiles.size() * 4, 16);
  const size_t o_bt = align_up(o_fp + p->fwd.cta_ptr.size() * 4, 16);
  const size_t o_bp = align_up(o_bt + p->bwd.tiles.size() * 4, 16);
  const size_t o_st = align_up(o_bp + p->bwd.cta_ptr.size() * 4, 16);
  const size_t bytes = align_up(o_st + 16, 256);
  std::vector<uint8_t> host(bytes, 0);
  std::memcpy(&host[o_kv], kv_offsets_host, (B + 1) * 4);
  if (q_offsets_host) std::memcpy(&host[o_q], q_offsets_host, (B + 1) * 4);
  if (!p->fwd.tiles.empty()) std::memcpy(&host[o_ft], p->fwd.tiles.data(), p->fwd.tiles.size() * 4);
  std::memcpy(&host[o_fp], p->fwd.cta_ptr.data(), p->fwd.cta_ptr.size() * 4);
  if (!p->bwd.tiles.empty()) std::memcpy(&host[o_bt], p->bwd.tiles.data(), p->bwd.tiles.size() * 4);
  std::memcpy(&host[o_bp], p->bwd.cta_ptr.data(), p->bwd.cta_ptr.size() * 4);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMalloc(&p->dev_block, bytes) != cudaSuccess) {
    delete p;
    return JFA_ERR_CUDA;
  }
  if (cudaMemcpyAsync(p->dev_block, host.data(), bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaFree(p->dev_block);
    delete p;
    return JFA_ERR_CUDA;
  }
  auto* base = static_cast<uint8_t*>(p->dev_block);
  p->d_kv_off = reinterpret_cast<int32_t*>(base + o_kv);
  p->d_q_off = q_offsets_host ? reinterpret_cast<int32_t*>(base + o_q) : nullptr;
  p->d_fwd_tiles = reinterpret_cast<int32_t*>(base + o_ft);
  p->d_fwd_ptr = reinterpret_cast<int32_t*>(base + o_fp);
  p->d_bwd_tiles = reinterpret_cast<int32_t*>(base + o_bt);
  p->d_bwd_ptr = reinterpret_cast<int32_t*>(base + o_bp);
  p->d_status = reinterpret_cast<int*>(base + o_st);
  p->d_counters = reinterpret_cast<int*>(base + o_st + 4);
  *out = p;
  return JFA_OK;
}

int jfa_plan_destroy(jfa_plan_t plan) {
  if (!plan) return JFA_ERR_INVALID_ARG;
  int rc = JFA_OK;
  if (plan->dev_block && cudaFree(plan->dev_block) != cudaSuccess) rc = JFA_ERR_CUDA;
  delete plan;
  return rc;
}

int jfa_plan_claims(jfa_plan_t plan, int* fwd, int* bwd) {
  if (!plan) return JFA_ERR_INVALID_ARG;
  if (fwd) *fwd = plan->fwd_dynamic ? 1 : 0;
  if (bwd) *bwd = plan->bwd_dynamic ? 1 : 0;
  return JFA_OK;
}

int jfa_plan_forward_form(jfa_plan_t plan, int* form) {
  if (!plan || !form) return JFA_ERR_INVALID_ARG;
  *form = plan->fwd_pair ? 1 : plan->fwd_two ? 2 : 0;
  return JFA_OK;
}

int jfa_plan_forward_pairs(jfa_plan_t plan, int* pairs) {
  if (!plan || !pairs) return JFA_ERR_INVALID_ARG;
  *pairs = plan->fwd_pair ? 1 : 0;
  return JFA_OK;
}

int jfa_plan_selftest(jfa_plan_t plan, int skip, unsigned limit_us) {
  if (!plan || skip < 0 || skip > 2 || limit_us > 2000000u) return JFA_ERR_INVALID_ARG;
  plan->test_skip = skip;
  plan->test_limit_ns = uint64_t(limit_us) * 1000u;
  return JFA_OK;
}

int jfa_plan_tiles(jfa_plan_t plan, int dir, int32_t* tiles_host, int32_t* cta_ptr_host, int* T,
                   int* P) {
  if (!plan || (dir != 0 && dir != 1) || !T || !P) return JFA_ERR_INVALID_ARG;
  const Schedule& s = dir == 0 ? plan->fwd : plan->bwd;
  *T = s.T;
  *P = s.P;
  if (tiles_host) std::memcpy(tiles_host, s.tiles.data(), s.tiles.size() * sizeof(int32_t));
  if (cta_ptr_host) std::memcpy(cta_ptr_host, s.cta_ptr.data(), s.cta_ptr.size() * sizeof(int32_t));
  return JFA_OK;
}

int jfa_plan_device_status(jfa_plan_t plan, void* stream, int* raw) {
  if (!plan) return JFA_ERR_INVALID_ARG;
  if (int rc = check_device(plan)) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, plan->d_status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return JFA_ERR_CUDA;
  if (raw) *raw = word;
  if (word != 0) {
    if (cudaMemsetAsync(plan->d_status, 0, sizeof(int), s) != cudaSuccess) return JFA_ERR_CUDA;
    return JFA_ERR_DEVICE_TIMEOUT;
  }
  return JFA_OK;
}

int jfa_fwd(jfa_plan_t plan, const void* q, const void* k, const void* v, float scale, void* out,
            float* lse, void* stream) {
  if (!plan || !std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  if (int rc = check_device(plan)) return rc;
  if ((plan->n_q > 0 && !q) || (plan->n_kv > 0 && (!k || !v)) || (plan->n_o > 0 && (!out || !lse)))
    return JFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return JFA_ERR_ALIGNMENT;
  if (plan->fwd.P == 0) return JFA_OK;
  const int64_t cols = int64_t(plan->H) * plan->D;
  CUtensorMap qm, km, vm, om;
  // a CTA of a pair loads 64-row halves of each K block
  if (make_map(&qm, q, plan->n_q, cols) || make_map(&km, k, plan->n_kv, cols, plan->fwd_pair ? 64 : 128) ||
      make_map(&vm, v, plan->n_kv, cols) || make_map(&om, out, plan->n_o, cols, 32))
    return JFA_ERR_CUDA;
  jfa::FwdArgs a;
  a.pb = problem_of(plan);
  a.tiles = plan->d_fwd_tiles;
  a.cta_ptr = plan->d_fwd_ptr;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.status = plan->d_status;
  a.packed = plan->packed;
  a.T = plan->fwd.T;
  a.wait_limit_ns = plan->test_limit_ns;
  a.test_skip = plan->test_skip == 1 ? 1 : 0;
  if (plan->fwd_dynamic) {
    a.dyn_counter = plan->d_counters;
    if (cudaMemsetAsync(a.dyn_counter, 0, sizeof(int), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return JFA_ERR_CUDA;
  }
  a.pair = plan->fwd_pair;
  cudaError_t e = plan->fwd_two
                      ? jfa::launch_fwd_two(a, qm, km, vm, om, plan->fwd.P, static_cast<cudaStream_t>(stream))
                      : jfa::launch_fwd(a, qm, km, vm, om, plan->fwd_pair ? 2 * plan->fwd.P : plan->fwd.P,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

size_t jfa_bwd_workspace_bytes(jfa_plan_t plan) {
  if (!plan) return 0;
  return align_up(static_cast<size_t>(plan->n_o) * plan->H * sizeof(float), 256);
}

int jfa_bwd_preprocess(jfa_plan_t plan, const void* out, const void* dout, float* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan) return JFA_ERR_INVALID_ARG;
  if (int rc = check_device(plan)) return rc;
  if ((plan->n_q > 0 && !dq) || (plan->n_kv > 0 && (!dk || !dv)) ||
      (plan->n_o > 0 && (!out || !dout)))
    return JFA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(workspace))
    return JFA_ERR_ALIGNMENT;
  if (plan->n_o > 0 && (!workspace || workspace_bytes < jfa_bwd_workspace_bytes(plan)))
    return JFA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t cols = int64_t(plan->H) * plan->D;
  // dQ rows that tiles reduce-add into (or that no tile touches) start from
  // zero; rows a single tile owns are stored by it
  for (const auto& run : plan->dq_rows_to_clear) {
    const size_t off = static_cast<size_t>(run.first) * cols * sizeof(float);
    const size_t len = static_cast<size_t>(run.second - run.first) * cols * sizeof(float);
    if (cudaMemsetAsync(reinterpret_cast<uint8_t*>(dq) + off, 0, len, s) != cudaSuccess)
      return JFA_ERR_CUDA;
  }
  // keys of sequences without queries get no backward tile: their gradients are zero
  for (const auto& run : plan->kv_rows_without_queries) {
    const size_t off = static_cast<size_t>(run.first) * cols * 2;
    const size_t len = static_cast<size_t>(run.second - run.first) * cols * 2;
    if (cudaMemsetAsync(static_cast<uint8_t*>(dk) + off, 0, len, s) != cudaSuccess ||
        cudaMemsetAsync(static_cast<uint8_t*>(dv) + off, 0, len, s) != cudaSuccess)
      return JFA_ERR_CUDA;
  }
  if (plan->bwd.P == 0 || plan->n_o == 0 || plan->own_delta) return JFA_OK;
  cudaError_t e = jfa::launch_delta(static_cast<const uint16_t*>(out),
                                    static_cast<const uint16_t*>(dout),
                                    static_cast<float*>(workspace), plan->n_o, plan->H, plan->D, s);
  return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

int jfa_bwd_main(jfa_plan_t plan, const void* q, const void* k, const void* v, const void* dout,
                 const float* lse, float scale, float* dq, void* dk, void* dv,
                 const void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan || !std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  if (int rc = check_device(plan)) return rc;
  if ((plan->n_q > 0 && (!q || !dq)) || (plan->n_kv > 0 && (!k || !v || !dk || !dv)) ||
      (plan->n_o > 0 && (!dout || !lse)))
    return JFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return JFA_ERR_ALIGNMENT;
  if (plan->n_o > 0 && (!workspace || workspace_bytes < jfa_bwd_workspace_bytes(plan)))
    return JFA_ERR_WORKSPACE;
  if (plan->bwd.P == 0) return JFA_OK;
  const int64_t cols = int64_t(plan->H) * plan->D;
  CUtensorMap qm, km, vm, dom, dqm, dkm, dvm;
  if (make_map(&qm, q, plan->n_q, cols) || make_map(&km, k, plan->n_kv, cols) ||
      make_map(&vm, v, plan->n_kv, cols) || make_map(&dom, dout, plan->n_o, cols) ||
      make_map_dq(&dqm, dq, plan->n_q, cols) || make_map(&dkm, dk, plan->n_kv, cols, 32) ||
      make_map(&dvm, dv, plan->n_kv, cols, 32))
    return JFA_ERR_CUDA;
  jfa::BwdArgs a;
  a.pb = problem_of(plan);
  a.tiles = plan->d_bwd_tiles;
  a.cta_ptr = plan->d_bwd_ptr;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.lse = lse;
  a.delta = static_cast<const float*>(workspace);
  a.dq = dq;
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.status = plan->d_status;
  a.packed = plan->packed;
  a.own_rows = plan->dq_own_rows;
  a.own_delta = plan->own_delta;
  a.T = plan->bwd.T;
  a.wait_limit_ns = plan->test_limit_ns;
  a.test_skip = plan->test_skip == 2 ? 2 : 0;
  if (plan->bwd_dynamic) {
    a.dyn_counter = plan->d_counters + 1;
    if (cudaMemsetAsync(a.dyn_counter, 0, sizeof(int), static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return JFA_ERR_CUDA;
  }
  cudaError_t e =
      jfa::launch_bwd(a, qm, km, vm, dom, dqm, dkm, dvm, plan->bwd.P, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}

int jfa_bwd(jfa_plan_t plan, const void* q, const void* k, const void* v, const void* out,
            const void* dout, const float* lse, float scale, float* dq, void* dk, void* dv,
            void* workspace, size_t workspace_bytes, void* stream) {
  if (!plan || !std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  int rc = jfa_bwd_preprocess(plan, out, dout, dq, dk, dv, workspace, workspace_bytes, stream);
  if (rc != JFA_OK) return rc;
  return jfa_bwd_main(plan, q, k, v, dout, lse, scale, dq, dk, dv, workspace, workspace_bytes,
                      stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward without device allocation (jfa_bwd_noalloc in jfa.h).
// ---------------------------------------------------------------------------
namespace {

// The scratch every jfa_bwd_noalloc call uses: a status word, the offsets, the
// schedule and the Delta row sums.  Host code never hands this symbol to a
// kernel; it uses the device address cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[JFA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch on device `dev` (the current device),
// resolved on the first call for that device.
int noalloc_scratch(int dev, uint8_t** out) {
  if (dev < 0 || dev >= kMaxDevices) return JFA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return JFA_ERR_CUDA;
    g_noalloc_addr[dev] = ptr;
  }
  *out = static_cast<uint8_t*>(g_noalloc_addr[dev]);
  return JFA_OK;
}

}  // namespace

extern "C" int jfa_bwd_noalloc(const int32_t* kv_offsets_host, const int32_t* q_offsets_host,
                               int B, int H, int Lq, int D, const void* q, const void* k,
                               const void* v, const void* out, const void* dout, const float* lse,
                               float scale, float* dq, void* dk, void* dv, int* device_status,
                               void* stream) {
  if (!kv_offsets_host || B < 1 || H < 1 || !std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
  std::vector<int64_t> qlen, kvlen;
  int64_t n_kv = 0, n_q = 0;
  int rc = lengths_of(kv_offsets_host, q_offsets_host, B, Lq, qlen, kvlen, &n_kv, &n_q);
  if (rc != JFA_OK) return rc;
  const int64_t n_o = q_offsets_host ? n_q : int64_t(B) * Lq;
  if (n_o >= (int64_t(1) << 31) || int64_t(H) * D * 2 >= (int64_t(1) << 31))
    return JFA_ERR_UNSUPPORTED;
  if ((n_q > 0 && (!q || !dq)) || (n_kv > 0 && (!k || !v || !dk || !dv)) ||
      (n_o > 0 && (!out || !dout || !lse)))
    return JFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(device_status) & 3u))
    return JFA_ERR_ALIGNMENT;

  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return JFA_ERR_CUDA;
  if (major != 10 || minor != 3) return JFA_ERR_UNSUPPORTED;

  const Schedule sched = jfa::build_bwd_schedule(qlen, kvlen, H, sms);
  // scratch layout: status | kv offsets | q offsets | tiles | cta_ptr | Delta
  const size_t o_st = 0;
  const size_t o_kv = 256;
  const size_t o_q = align_up(o_kv + (B + 1) * 4, 256);
  const size_t o_t = align_up(o_q + (q_offsets_host ? (B + 1) * 4 : 0), 256);
  const size_t o_p = align_up(o_t + sched.tiles.size() * 4, 256);
  const size_t o_d = align_up(o_p + sched.cta_ptr.size() * 4, 256);
  const bool own_delta = tiles_form_delta(0u, qlen, kvlen, sched, kv_offsets_host);  // no Delta scratch
  const size_t need = o_d + (own_delta ? 0 : static_cast<size_t>(n_o) * H * sizeof(float));
  if (need > JFA_NOALLOC_SCRATCH_BYTES) return JFA_ERR_WORKSPACE;

  uint8_t* scratch = nullptr;
  rc = noalloc_scratch(dev, &scratch);
  if (rc != JFA_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // every byte before Delta is rewritten by this call (the status word
  // starts at 0); Delta, where there is a pre-pass, is written in full by it
  std::vector<uint8_t> host(o_d, 0);
  std::memcpy(&host[o_kv], kv_offsets_host, (B + 1) * 4);
  if (q_offsets_host) std::memcpy(&host[o_q], q_offsets_host, (B + 1) * 4);
  if (!sched.tiles.empty()) std::memcpy(&host[o_t], sched.tiles.data(), sched.tiles.size() * 4);
  std::memcpy(&host[o_p], sched.cta_ptr.data(), sched.cta_ptr.size() * 4);
  if (cudaMemcpyAsync(scratch, host.data(), o_d, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return JFA_ERR_CUDA;

  const int64_t cols = int64_t(H) * D;
  if (n_q > 0 &&
      cudaMemsetAsync(dq, 0, static_cast<size_t>(n_q) * cols * sizeof(float), s) != cudaSuccess)
    return JFA_ERR_CUDA;
  for (int b = 0; b < B; ++b) {  // keys without queries: zero gradients
    if (qlen[b] == 0 && kvlen[b] > 0) {
      const size_t off = static_cast<size_t>(kv_offsets_host[b]) * cols * 2;
      const size_t len = static_cast<size_t>(kvlen[b]) * cols * 2;
      if (cudaMemsetAsync(static_cast<uint8_t*>(dk) + off, 0, len, s) != cudaSuccess ||
          cudaMemsetAsync(static_cast<uint8_t*>(dv) + off, 0, len, s) != cudaSuccess)
        return JFA_ERR_CUDA;
    }
  }
  if (sched.P == 0 || n_o == 0) return JFA_OK;
  float* delta = own_delta ? nullptr : reinterpret_cast<float*>(scratch + o_d);
  cudaError_t e = cudaSuccess;
  if (!own_delta) {
    e = jfa::launch_delta(static_cast<const uint16_t*>(out), static_cast<const uint16_t*>(dout),
                          delta, n_o, H, D, s);
    if (e != cudaSuccess) return JFA_ERR_CUDA;
  }
  CUtensorMap qm, km, vm, dom, dqm, dkm, dvm;
  if (make_map(&qm, q, n_q, cols) || make_map(&km, k, n_kv, cols) || make_map(&vm, v, n_kv, cols) ||
      make_map(&dom, dout, n_o, cols) || make_map_dq(&dqm, dq, n_q, cols) ||
      make_map(&dkm, dk, n_kv, cols, 32) || make_map(&dvm, dv, n_kv, cols, 32))
    return JFA_ERR_CUDA;
  jfa::BwdArgs a;
  a.pb.kv_off = reinterpret_cast<const int32_t*>(scratch + o_kv);
  a.pb.q_off = q_offsets_host ? reinterpret_cast<const int32_t*>(scratch + o_q) : nullptr;
  a.pb.B = B;
  a.pb.H = H;
  a.pb.Lq = q_offsets_host ? 0 : Lq;
  a.pb.D = D;
  a.pb.n_q = n_q;
  a.pb.n_o = n_o;
  a.pb.n_kv = n_kv;
  a.tiles = reinterpret_cast<const int32_t*>(scratch + o_t);
  a.cta_ptr = reinterpret_cast<const int32_t*>(scratch + o_p);
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.lse = lse;
  a.delta = delta;
  a.dq = dq;
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.status = device_status ? device_status : reinterpret_cast<int*>(scratch + o_st);
  a.packed = false;
  a.own_delta = own_delta;
  e = jfa::launch_bwd(a, qm, km, vm, dom, dqm, dkm, dvm, sched.P, s);
  return e == cudaSuccess ? JFA_OK : JFA_ERR_CUDA;
}


// ---------------------------------------------------------------------------
// Plan-free entry points (jfa_fwd_simple / jfa_bwd_simple in jfa.h): a small
// cache of plans keyed by device, sizes and the offsets' contents.
// ---------------------------------------------------------------------------
namespace {

struct SimpleEntry {
  int device = 0, B = 0, H = 0, Lq = 0, D = 0;
  bool broadcast = false;
  std::vector<int32_t> kv, q;    // copies of the offsets the plan was built from
  jfa_plan_t plan = nullptr;
  void* ws = nullptr;            // backward workspace, allocated with the first backward
  uint64_t last_use = 0;
};

constexpr size_t kSimpleCapacity = 8;
std::mutex g_simple_mu;            // held for the whole of every plan-free call
std::vector<SimpleEntry> g_simple;
uint64_t g_simple_clock = 0;

void release_entry(SimpleEntry& e) {
  if (e.ws) cudaFree(e.ws);
  if (e.plan) jfa_plan_destroy(e.plan);
  e.ws = nullptr;
  e.plan = nullptr;
}

// Checks that need no device, so bad arguments fail before any CUDA call.
int simple_args_ok(const int32_t* kv, const int32_t* q, int B, int H, int Lq, int D) {
  if (!kv || B < 1 || H < 1) return JFA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return JFA_ERR_UNSUPPORTED;
  std::vector<int64_t> qlen, kvlen;
  int64_t n_kv = 0, n_q = 0;
  return lengths_of(kv, q, B, Lq, qlen, kvlen, &n_kv, &n_q);
}

// The cached plan for these arguments, built on a miss (the least recently
// used entry is released when the cache is full).  Caller holds g_simple_mu.
int simple_entry(const int32_t* kv, const int32_t* q, int B, int H, int Lq, int D, void* stream,
                 SimpleEntry** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_CUDA;
  const int lq = q ? 0 : Lq;
  for (auto& e : g_simple) {
    if (e.device == dev && e.B == B && e.H == H && e.Lq == lq && e.D == D &&
        e.broadcast == (q == nullptr) && std::equal(e.kv.begin(), e.kv.end(), kv) &&
        (!q || std::equal(e.q.begin(), e.q.end(), q))) {
      e.last_use = ++g_simple_clock;
      *out = &e;
      return JFA_OK;
    }
  }
  SimpleEntry e;
  int rc = jfa_plan_create_ex(kv, q, B, H, Lq, D, 0, 0u, stream, &e.plan);
  if (rc != JFA_OK) return rc;
  e.device = dev;
  e.B = B;
  e.H = H;
  e.Lq = lq;
  e.D = D;
  e.broadcast = q == nullptr;
  e.kv.assign(kv, kv + B + 1);
  if (q) e.q.assign(q, q + B + 1);
  e.last_use = ++g_simple_clock;
  if (g_simple.size() >= kSimpleCapacity) {
    size_t lru = 0;
    for (size_t i = 1; i < g_simple.size(); ++i)
      if (g_simple[i].last_use < g_simple[lru].last_use) lru = i;
    release_entry(g_simple[lru]);  // frees device memory: synchronises the device
    g_simple.erase(g_simple.begin() + static_cast<std::ptrdiff_t>(lru));
  }
  g_simple.push_back(std::move(e));
  *out = &g_simple.back();
  return JFA_OK;
}

}  // namespace

extern "C" int jfa_fwd_simple(const void* q, const void* k, const void* v,
                              const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B,
                              int H, int Lq, int D, float scale, void* out, float* lse,
                              void* stream) {
  int rc = simple_args_ok(kv_offsets_host, q_offsets_host, B, H, Lq, D);
  if (rc != JFA_OK) return rc;
  if (!std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_simple_mu);
  SimpleEntry* e = nullptr;
  rc = simple_entry(kv_offsets_host, q_offsets_host, B, H, Lq, D, stream, &e);
  if (rc != JFA_OK) return rc;
  return jfa_fwd(e->plan, q, k, v, scale, out, lse, stream);
}

extern "C" int jfa_bwd_simple(const void* q, const void* k, const void* v,
                              const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B,
                              int H, int Lq, int D, float scale, const void* out, const void* dout,
                              const float* lse, float* dq, void* dk, void* dv, void* stream) {
  int rc = simple_args_ok(kv_offsets_host, q_offsets_host, B, H, Lq, D);
  if (rc != JFA_OK) return rc;
  if (!std::isfinite(scale)) return JFA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_simple_mu);
  SimpleEntry* e = nullptr;
  rc = simple_entry(kv_offsets_host, q_offsets_host, B, H, Lq, D, stream, &e);
  if (rc != JFA_OK) return rc;
  const size_t ws_bytes = std::max<size_t>(jfa_bwd_workspace_bytes(e->plan), 256);
  if (!e->ws && cudaMalloc(&e->ws, ws_bytes) != cudaSuccess) {
    e->ws = nullptr;
    return JFA_ERR_CUDA;
  }
  return jfa_bwd(e->plan, q, k, v, out, dout, lse, scale, dq, dk, dv, e->ws, ws_bytes, stream);
}

extern "C" int jfa_simple_device_status(void* stream, int* raw) {
  std::lock_guard<std::mutex> lock(g_simple_mu);
  int dev = 0;
  if (!g_simple.empty() && cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_CUDA;
  int word = 0, rc = JFA_OK;
  for (auto& e : g_simple) {
    if (e.device != dev) continue;  // read with that device current
    int w = 0;
    const int r = jfa_plan_device_status(e.plan, stream, &w);
    if (r == JFA_ERR_CUDA) return r;
    if (r == JFA_ERR_DEVICE_TIMEOUT) rc = r;
    word |= w;
  }
  if (raw) *raw = word;
  return rc;
}

extern "C" int jfa_simple_release(void) {
  std::lock_guard<std::mutex> lock(g_simple_mu);
  for (auto& e : g_simple) release_entry(e);
  g_simple.clear();
  return JFA_OK;
}
