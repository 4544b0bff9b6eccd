/*
 * jfa.h -- C ABI of libjfa, jagged FlashAttention forward and backward for
 * GB300 (sm_103a).
 *
 * The operation (jagged FlashAttention pages: the alphasignal news page,
 * section "GEM's sequences do not fit a fixed grid"; the PyTorch-blog summary
 * on arc-codex, first key point): B variable-length sequences are packed
 * back to back, with no padding, and addressed by an offsets array, and
 * FlashAttention runs on them in that form; for every sequence b and head h
 *
 *     O_b = softmax(scale * Q_b K_b^T) V_b,   LSE_b = logsumexp(scale * Q_b K_b^T)
 *
 * row by row, with no mask inside a sequence.  In broadcast mode one dense
 * query block Q [Lq, H, D] attends to every sequence (same page and section:
 * all sequences of a batch share the query block, so their query gradients
 * add up) and the backward sums dQ over the batch.
 *
 * Layouts (all row-major, contiguous):
 *   K, V        bf16 [kv_offsets[B], H, D]
 *   Q           bf16 [q_offsets[B], H, D]            (self mode)
 *               bf16 [Lq, H, D]                      (broadcast mode)
 *   O, dO       bf16 [n_o, H, D], n_o = q_offsets[B] (self) or B*Lq (broadcast, b-major)
 *   LSE         fp32 [H, n_o], natural log of the row sum, scale included;
 *               -inf for rows of a sequence with no keys
 *   dQ          fp32, the shape of Q (broadcast: summed over all sequences)
 *   dK, dV      bf16, the shape of K
 * bf16 is IEEE-754 binary16-brain (8-bit exponent), passed as raw 16-bit
 * words.  Supported: D in {64, 128}; every device pointer 16-byte aligned.
 *
 * Ownership: the caller owns every tensor and the stream.  A plan owns a
 * small device copy of the offsets and of the tile schedule; it must outlive
 * the stream work that uses it.  A plan belongs to the device that was
 * current when it was created: jfa_fwd, jfa_bwd (and its stages) and
 * jfa_plan_device_status return JFA_ERR_INVALID_ARG when another device is
 * current.  jfa_fwd / jfa_bwd allocate nothing and are
 * asynchronous on the given stream (a cudaStream_t passed as void*; NULL is
 * the legacy default stream).
 *
 * Errors: every entry point returns a jfa_status; nothing throws across the
 * ABI.  Argument problems are reported before anything is launched.  Device
 * waits in the kernels are bounded: a wait that runs out records
 * JFA_ERR_DEVICE_TIMEOUT in the plan's device status word, which
 * jfa_plan_device_status reads back.
 */
#ifndef JFA_H
#define JFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum jfa_status {
  JFA_OK = 0,
  JFA_ERR_INVALID_ARG = 1,    /* null pointer, non-positive size, bad direction ... */
  JFA_ERR_UNSUPPORTED = 2,    /* D not in {64, 128}, no sm_100-family GPU */
  JFA_ERR_BAD_OFFSETS = 3,    /* offsets[0] != 0, decreasing, or total >= 2^31 */
  JFA_ERR_ALIGNMENT = 4,      /* a device pointer is not 16-byte aligned */
  JFA_ERR_WORKSPACE = 5,      /* workspace missing or smaller than jfa_bwd_workspace_bytes */
  JFA_ERR_CUDA = 6,           /* a CUDA runtime call failed */
  JFA_ERR_DEVICE_TIMEOUT = 7  /* a kernel wait ran out (see jfa_plan_device_status) */
} jfa_status;

/* Tile geometry: query rows per forward tile and key rows per backward tile. */
#define JFA_BLOCK_M 128
#define JFA_BLOCK_N 128

typedef struct jfa_plan* jfa_plan_t;

/*
 * Build a plan for one batch shape.
 *   kv_offsets_host  int32 [B+1], host memory: kv_offsets[0] = 0, non-decreasing.
 *   q_offsets_host   int32 [B+1] host offsets of the queries (self mode; may
 *                    equal kv_offsets), or NULL for broadcast mode.
 *   B, H             sequences and heads (B >= 1, H >= 1).
 *   Lq               broadcast mode: rows of the dense Q (>= 0); ignored in self mode.
 *   D                head dimension, 64 or 128.
 *   num_ctas         persistent CTAs per launch; 0 = one per SM of the current device.
 *   stream           stream for the host-to-device upload of offsets and tiles.
 * The tile schedule follows the pages' description: forward tiles
 * (b, h, query block) are sorted by key/value workload and dealt to the CTAs
 * in zigzag (boustrophedon) order (alphasignal page, "Five changes unlocked
 * the gains", item 1); backward tiles (b, h, key block) exist only where the
 * sequence has queries and are dealt round-robin (yuxiaoba note, "Why both
 * static and dynamic balancing help").  On success *out receives the plan.
 * Allocates device memory; the host arrays are not retained.
 */
int jfa_plan_create(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                    int Lq, int D, int num_ctas, void* stream, jfa_plan_t* out);

/*
 * Plan flags.
 * Packing of short sequences: in self mode with one offsets array shared by
 * queries and keys (q_offsets equal to kv_offsets element by element), runs
 * of consecutive short sequences whose lengths add up to at most 128 rows
 * (with at least two non-empty ones) share one 128-row tile, masked
 * block-diagonally so every row still sees only its own sequence.  This is
 * the block-diagonal case of the TLX Block Attention page ("One Constraint,
 * Five Eliminations": each query tile meets exactly one key tile), which an
 * unpacked schedule runs at half occupancy when segments are shorter than a
 * tile.  Such a tile is recorded as {b0, h, -nseq, 1}.  Never in broadcast
 * mode or when the offsets differ.  By default a plan packs when that removes
 * at least an eighth of its forward tiles (a pack of n non-empty sequences
 * replaces n tiles by one).
 * JFA_PLAN_PACK_SHORT: pack whenever a run forms.
 * JFA_PLAN_NO_PACK: never pack.  Setting both is JFA_ERR_INVALID_ARG.
 */
#define JFA_PLAN_PACK_SHORT 1u
#define JFA_PLAN_NO_PACK 32u

/*
 * JFA_PLAN_DYNAMIC: tiles are claimed at run time instead of dealt on the
 * host (the pages' dynamic balancing, which works alongside the static order):
 * each schedule lists every tile once in claim order -- the tiles stably
 * sorted by their cost field, largest first -- and the plan's P CTAs take
 * tile blockIdx.x, then the next unclaimed one from a device counter, until
 * none is left.  jfa_plan_tiles / jfa_build_tiles return that list with
 * cta_ptr = {0, T, ..., T} (P + 1 entries: one queue shared by the P CTAs
 * launched).  The
 * counter lives in the plan and is reset on the stream before each launch,
 * so a plan's launches must be stream-ordered.  Combines with
 * JFA_PLAN_PACK_SHORT.
 * JFA_PLAN_DYNAMIC claims the tiles of both passes; JFA_PLAN_STATIC deals
 * both on the host (the two together are invalid).  Without either, the
 * forward is dealt on the host, and the backward is claimed at run time when
 * queries have their own offsets (self mode, where a sequence's key blocks
 * make tiles of very different lengths) and dealt in broadcast mode, where
 * claiming measured slower; jfa_plan_claims reports the choice.
 */
#define JFA_PLAN_DYNAMIC 2u
#define JFA_PLAN_STATIC 128u

/*
 * Where Delta comes from.  When every sequence that has queries has at most
 * 128 keys (one key block: the block-diagonal and other short-sequence
 * cases), each backward tile meets all the keys of its queries and can form
 * Delta_i = sum_j P_ij dP_ij over them itself.  That is the same quantity as
 * sum_d dO_id O_id, because O = P V and dP = dO V^T, so the pre-pass that
 * reads O and dO only for Delta is skipped (the backward then does not read
 * O at all).  The sums cost every tile the same whatever its fill, so by
 * default the tiles form Delta only when they hold at least 96 key rows on
 * average (full tiles, as with JFA_PLAN_PACK_SHORT on 64-token segments).
 * JFA_PLAN_DELTA_PREPASS: always use the pre-pass.
 * JFA_PLAN_DELTA_IN_TILES: let the tiles form Delta whenever they hold all
 *   the keys of their queries, whatever their fill.
 * Setting both is JFA_ERR_INVALID_ARG.
 */
#define JFA_PLAN_DELTA_PREPASS 4u
#define JFA_PLAN_DELTA_IN_TILES 8u

/*
 * JFA_PLAN_FWD_PAIRS: run the forward as CTA pairs where the pair kernel
 * applies (D = 128, static schedule, no packed tiles, num_ctas >= 2).  Two
 * CTAs of a thread-block cluster take the two query blocks of a "pair tile"
 * (b, h, mp) -- query rows [256 mp, 256 mp + 256) of sequence b; a sequence
 * with an odd number of query blocks leaves its last pair tile half empty --
 * and share every K/V block, each loading half of it; one thread issues the
 * pair's tensor-core products, which span both CTAs' query rows (M = 256)
 * and so cost the pair fewer instructions than two single-CTA tiles (the
 * pages' 2-CTA collaborative MMA: alphasignal JFA page, "Five changes
 * unlocked the gains", closing paragraph).  The forward schedule then lists
 * pair tiles {b, h, mp, cost} over P = min(num_ctas / 2, T) pairs.
 * Without the flag a plan runs one CTA per query block: on GB300 that form
 * measures faster on every workload tried (the pair's K/V loads, half per
 * CTA plus the peer's half over the pair, arrive no sooner than a single
 * CTA's whole block, and its query blocks share no K/V through L2).
 */
#define JFA_PLAN_FWD_PAIRS 64u

/*
 * JFA_PLAN_FWD_TWO: run the forward with two query tiles in flight per CTA
 * where that kernel applies (D = 128, static schedule, no packed tiles):
 * each schedule tile {b, h, mp, cost} covers query blocks 2 mp and 2 mp + 1
 * of sequence b -- the list jfa_build_tiles dir 2 gives, over num_ctas CTAs
 * -- and the CTA alternates between them, so one tile's tensor-core products
 * run while the other tile's softmax works (the pages' two query tiles per
 * CTA: alphasignal JFA page, "Specialized warps keep tensor cores busy").
 * A sequence with an odd number of query blocks leaves its last tile half
 * empty.  By default a plan runs this form where it applies, its tiles
 * hold at least 3 key blocks on average with at most a quarter of them half
 * empty, and there are at least four of them per CTA (measured faster there,
 * slower on short tiles and on few tiles per CTA); JFA_PLAN_FWD_TWO
 * asks for it wherever it applies, JFA_PLAN_FWD_ONE never.  At most one of
 * JFA_PLAN_FWD_PAIRS, JFA_PLAN_FWD_TWO and JFA_PLAN_FWD_ONE (invalid
 * together).
 */
#define JFA_PLAN_FWD_TWO 256u
#define JFA_PLAN_FWD_ONE 512u

/* jfa_plan_create with flags (0 = the schedule described above). */
int jfa_plan_create_ex(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                       int Lq, int D, int num_ctas, unsigned flags, void* stream, jfa_plan_t* out);

/* Release a plan (synchronises the device first so in-flight work finishes). */
int jfa_plan_destroy(jfa_plan_t plan);

/*
 * Copy a plan's tile schedule to host memory.  dir: 0 forward (the schedule
 * the plan launches: over tiles of two query blocks when it runs CTA pairs or
 * two tiles per CTA, see jfa_plan_forward_form), 1 backward.
 * tiles_host receives T records of four int32 {b, h, block, cost} grouped by
 * CTA (or pair), cta_ptr_host receives P+1 CSR offsets (P = min(num_ctas, T),
 * or the number of pairs).  Either
 * buffer may be NULL to query only *T and *P.  Buffers must hold 4*T and P+1
 * int32.
 */
int jfa_plan_tiles(jfa_plan_t plan, int dir, int32_t* tiles_host, int32_t* cta_ptr_host, int* T,
                   int* P);

/* *fwd / *bwd = 1 when that pass's tiles are claimed at run time (JFA_PLAN_DYNAMIC
 * and the default rule given with it), 0 when they are dealt on the host.
 * Either pointer may be NULL. */
int jfa_plan_claims(jfa_plan_t plan, int* fwd, int* bwd);

/* *form = 0 when the plan's forward runs one query tile per CTA, 1 as CTA
 * pairs (JFA_PLAN_FWD_PAIRS), 2 with two query tiles per CTA (JFA_PLAN_FWD_TWO). */
int jfa_plan_forward_form(jfa_plan_t plan, int* form);

/* *pairs = 1 when the plan's forward runs as CTA pairs (JFA_PLAN_FWD_PAIRS), else 0. */
int jfa_plan_forward_pairs(jfa_plan_t plan, int* pairs);

/*
 * Host-only schedule builder (no GPU needed): the same lists a plan created
 * with the same flags holds.  dir: 0 forward (one CTA per query block), 1
 * backward, 2 forward over pair tiles (num_ctas then counts CTA pairs).
 * q_offsets_host == NULL means broadcast with Lq rows.  Call once with
 * tiles_out == NULL to learn *T and *P, then with buffers of 4*T and P+1
 * int32.
 */
int jfa_build_tiles(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                    int Lq, int num_ctas, int dir, unsigned flags, int32_t* tiles_out,
                    int32_t* cta_ptr_out, int* T, int* P);

/*
 * Host-only (no GPU needed): the schedule choices jfa_plan_create_ex makes
 * for these arguments on a device of num_ctas SMs (num_ctas >= 1 here):
 * *fwd_form as jfa_plan_forward_form, *fwd_claims / *bwd_claims as
 * jfa_plan_claims, *packed = 1 when short sequences are packed into shared
 * tiles (JFA_PLAN_PACK_SHORT's rule).  Any output pointer may be NULL.
 * Errors as jfa_plan_create_ex (offsets, sizes, conflicting flags).
 */
int jfa_plan_choices(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                     int Lq, int D, int num_ctas, unsigned flags, int* fwd_form, int* fwd_claims,
                     int* bwd_claims, int* packed);

/*
 * Host-only (no GPU needed): *in_tiles = 1 when a plan created from these
 * offsets and flags has its backward tiles form Delta (the rule given with
 * JFA_PLAN_DELTA_PREPASS), 0 when the pre-pass forms it.  With 1, jfa_bwd
 * does not read `out`; jfa_bwd_noalloc follows the flags-0 answer.  Errors as
 * jfa_plan_create_ex (offsets, conflicting Delta flags).
 */
int jfa_delta_in_tiles(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B,
                       int Lq, unsigned flags, int* in_tiles);

/*
 * Forward: out = softmax(scale Q K^T) V per sequence and head, lse as above.
 * q, k, v, out: bf16 device tensors in the layouts above; lse: fp32 device.
 * Rows of sequences without keys get O = 0 and LSE = -inf.
 */
int jfa_fwd(jfa_plan_t plan, const void* q, const void* k, const void* v, float scale, void* out,
            float* lse, void* stream);

/* Bytes of device workspace jfa_bwd needs (the fp32 row sums Delta = rowsum(dO * O)). */
size_t jfa_bwd_workspace_bytes(jfa_plan_t plan);

/*
 * Backward of jfa_fwd.  Inputs q, k, v, out (the forward's O), dout (dO), lse
 * (the forward's LSE) and the forward's scale.  Outputs dq (fp32, overwritten -- the library clears it
 * on the stream), dk and dv (bf16).  workspace: device memory of at least
 * jfa_bwd_workspace_bytes(plan) bytes, 16-byte aligned.  The backward first
 * forms Delta_i = sum_d dO_id O_id (the row sum the TLX Block Attention page
 * calls the "Di" preprocessing, "One Constraint, Five Eliminations"), then
 * runs the key/value-stationary pass that produces dK, dV and reduce-adds dQ.
 * Where every tile holds all the keys of its queries, the main pass may form
 * Delta itself instead (see JFA_PLAN_DELTA_PREPASS); the workspace is then
 * not written, but its size and alignment rules stay the same.
 */
int jfa_bwd(jfa_plan_t plan, const void* q, const void* k, const void* v, const void* out,
            const void* dout, const float* lse, float scale, float* dq, void* dk, void* dv,
            void* workspace, size_t workspace_bytes, void* stream);

/*
 * The two stages jfa_bwd runs, for callers that schedule them separately
 * (same arguments and rules as jfa_bwd).
 * jfa_bwd_preprocess: Delta (into workspace) from out and dout -- skipped when
 *   the main pass forms Delta itself (see JFA_PLAN_DELTA_PREPASS) --, clears the dq
 *   rows the main pass reduce-adds into or never writes (all of them in
 *   broadcast mode; with query offsets, those of sequences with no key or
 *   more than one key block -- a sequence with one key block, or in a packed
 *   tile, has its dQ rows stored outright by its one tile), and zeroes dk / dv
 *   rows of sequences with keys but no queries.
 * jfa_bwd_main: the key/value-stationary pass; needs the workspace written by
 *   jfa_bwd_preprocess (stream order) and the dq rows it cleared.
 */
int jfa_bwd_preprocess(jfa_plan_t plan, const void* out, const void* dout, float* dq, void* dk,
                       void* dv, void* workspace, size_t workspace_bytes, void* stream);
int jfa_bwd_main(jfa_plan_t plan, const void* q, const void* k, const void* v, const void* dout,
                 const float* lse, float scale, float* dq, void* dk, void* dv,
                 const void* workspace, size_t workspace_bytes, void* stream);

/*
 * Read the plan's device status word (synchronises `stream`), then clear it.
 * Returns JFA_ERR_DEVICE_TIMEOUT when a kernel recorded a wait that ran out,
 * JFA_OK otherwise; *raw (optional) receives the raw word.
 */
int jfa_plan_device_status(jfa_plan_t plan, void* stream, int* raw);

/*
 * Backward for callers that cannot allocate device memory: code that runs
 * inside a framework whose caching or pool allocator owns all device memory
 * (a stray cudaMalloc there fragments or oversubscribes the pool, and
 * cudaFree synchronises the device), and embedded or serving runtimes that
 * are handed a fixed budget of pre-allocated buffers and may not grow it.
 * There is no counterpart of this entry point on the jagged FlashAttention
 * pages; it computes exactly what jfa_bwd computes (same inputs, outputs,
 * layouts and tolerances) but needs neither a plan nor a workspace.
 *
 * Arguments are those of jfa_plan_create (host offsets, B, H, Lq, D) followed
 * by those of jfa_bwd without workspace; device_status is an optional device
 * int the kernels set when a wait runs out (NULL: not reported).
 *
 * Scratch: the schedule, the device copy of the offsets and the Delta row
 * sums live in one file-scope static __device__ array of
 * JFA_NOALLOC_SCRATCH_BYTES, which every GPU that loads this library holds
 * until the process exits.  A problem whose scratch (about 4 * H * n_o bytes
 * of Delta plus 16 bytes per backward tile; no Delta where the tiles form it,
 * under the default rule given with JFA_PLAN_DELTA_PREPASS) does not fit is
 * rejected with
 * JFA_ERR_WORKSPACE before anything is launched, as is (JFA_ERR_UNSUPPORTED)
 * any problem jfa_plan_create would refuse.  The call allocates no device
 * memory and calls no allocating library routine.  It uploads the schedule
 * and offsets with cudaMemcpyAsync from a host buffer that lives only for
 * the call (pageable memory), so the call returns once that copy has been
 * taken from the host buffer, and the call cannot be captured into a CUDA
 * graph (a replay would read that buffer after the call has returned).
 *
 * The first call on a device resolves the array's device address
 * (cudaGetSymbolAddress, with that device current).  All calls share the one array and each call
 * rewrites what it needs (nothing is assumed to start at zero), so calls
 * that overlap on the GPU -- different streams, or different host threads
 * without ordering -- race; issue them on one stream or order them.
 */
#define JFA_NOALLOC_SCRATCH_BYTES (32u << 20)
int jfa_bwd_noalloc(const int32_t* kv_offsets_host, const int32_t* q_offsets_host, int B, int H,
                    int Lq, int D, const void* q, const void* k, const void* v, const void* out,
                    const void* dout, const float* lse, float scale, float* dq, void* dk, void* dv,
                    int* device_status, void* stream);

/*
 * Test of the kernels' failure path (no counterpart in the pages; it exists
 * so that the timeout handling of the real kernels can be exercised on a GPU
 * without a fault).  Sets, for the plan's later launches, a limit of
 * limit_us microseconds on every device wait (0: the normal 2 s; at most
 * 2,000,000) and, with skip != 0, has one softmax warp of CTA 0 withhold one
 * arrival so that a wait of the MMA issuer runs out:
 *   skip = 1  jfa_fwd: the arrival on the first P block of CTA 0's first tile
 *   skip = 2  jfa_bwd: the arrival on the first dS^T block of CTA 0
 *   skip = 0  nothing withheld (normal operation)
 * The wait that runs out raises the CTA's abort flag: every role leaves its
 * loop, the TMA producer and the MMA issuer wait (bounded) for their work in
 * flight, and the TMEM is freed before the CTA exits, so the context stays
 * usable; jfa_plan_device_status then reports JFA_ERR_DEVICE_TIMEOUT, and the
 * outputs of that launch are undefined.  Not for production use: nothing in
 * the library or its benchmark sets it.  Errors: JFA_ERR_INVALID_ARG.
 */
int jfa_plan_selftest(jfa_plan_t plan, int skip, unsigned limit_us);

/*
 * Self-test of the failure path (no counterpart in the pages; it exists so
 * the timeout handling every kernel relies on can be exercised on a GPU
 * without a fault).  Launches one CTA whose waiting thread runs the kernels'
 * bounded mbarrier wait on a barrier nothing arrives on, with the limit
 * shortened to limit_us microseconds (1 .. 2,000,000), and synchronises the
 * stream.  Expected result: JFA_ERR_DEVICE_TIMEOUT, with the wait's measured
 * duration in *waited_ns (may be NULL); the kernel returns normally, so the
 * context stays usable.  JFA_OK would mean the wait completed (it cannot);
 * JFA_ERR_CUDA reports a failed launch.  The status word is one static device
 * variable: calls on different streams race.
 */
int jfa_selftest_wait_timeout(unsigned limit_us, unsigned long long* waited_ns, void* stream);

/*
 * Diagnostic: what one tensor-core product costs on this GPU.  One CTA issues
 * `count` (a multiple of 8, up to 2^20) tcgen05.mma products of one form back
 * to back into one TMEM accumulator (bf16 operands, fp32 accumulation, K = 16
 * per product, the operand descriptors the attention kernels use) and times
 * them in SM clock cycles: *cycles to the completion of a final commit,
 * *issue_cycles (optional) the time the issuing thread spends handing them
 * over.  group = 0: one run of `count` products; group > 0 (a multiple of 8
 * dividing count): after every `group` products the thread commits and waits
 * for them to complete before the next group, the dependent chain of the
 * kernels (a group's results feed the work the next group needs).
 * form: 0 M = 128, N = 128 with A and B in shared memory, both K-major (the
 * forward's QK^T, the backward's S^T and dP^T), 1 M = 128, N = 256, 2 M = 128,
 * N = 128 with A in TMEM, 3 M = 128, N = 64, 4 as 0 with B MN-major (the
 * backward's dK), 5 as 0 with A and B MN-major (the backward's dQ), 6 as 2
 * with B MN-major (the forward's PV, the backward's dV).  Synchronises the
 * stream.  Errors: JFA_ERR_INVALID_ARG,
 * JFA_ERR_CUDA, JFA_ERR_DEVICE_TIMEOUT (the commit did not arrive within the
 * kernels' wait limit).
 */
int jfa_selftest_mma_cycles(int form, int count, int group, unsigned long long* cycles,
                            unsigned long long* issue_cycles, void* stream);

/*
 * Plan-free forward and backward: the tensors, the host offsets and the sizes
 * in one call, as a framework op calls attention, with no plan handle and no
 * workspace.  Arguments mean what they mean for jfa_plan_create (kv_offsets
 * and q_offsets on the host, q_offsets NULL for broadcast mode with Lq query
 * rows), jfa_fwd and jfa_bwd (device tensors in the same layouts, 16-byte
 * aligned; dq fp32, overwritten).
 *
 * The library keeps a plan for each distinct (device, B, H, Lq, D, offsets)
 * it has seen, up to 8, releasing the least recently used one when a ninth
 * arrives; each cached plan owns the backward's workspace.  The first call
 * with new offsets builds the plan (host schedule, one device allocation and
 * an upload synchronised on `stream`), the first backward allocates the
 * workspace; later calls with the same offsets allocate nothing and are
 * asynchronous.  Releasing a plan frees device memory, which synchronises the
 * device.  Calls are serialised by a lock; backward calls with the same
 * offsets that overlap on the GPU (different streams, no ordering) share the
 * workspace and race: order them.
 *
 * Errors: the plan-creation codes (checked before any CUDA call where they
 * need no device), then those of jfa_fwd / jfa_bwd.  A wait that ran out is
 * recorded in the cached plan; jfa_simple_device_status reports it.
 */
int jfa_fwd_simple(const void* q, const void* k, const void* v, const int32_t* kv_offsets_host,
                   const int32_t* q_offsets_host, int B, int H, int Lq, int D, float scale,
                   void* out, float* lse, void* stream);
int jfa_bwd_simple(const void* q, const void* k, const void* v, const int32_t* kv_offsets_host,
                   const int32_t* q_offsets_host, int B, int H, int Lq, int D, float scale,
                   const void* out, const void* dout, const float* lse, float* dq, void* dk,
                   void* dv, void* stream);

/* Device status of every cached plan of the current device (synchronises
 * `stream`, then clears the words): JFA_ERR_DEVICE_TIMEOUT when any recorded
 * a wait that ran out; *raw (optional) receives the words or-ed together. */
int jfa_simple_device_status(void* stream, int* raw);

/* Release every cached plan and workspace (synchronises the device). */
int jfa_simple_release(void);

/* Human-readable text of a status code (static storage). */
const char* jfa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* JFA_H */
