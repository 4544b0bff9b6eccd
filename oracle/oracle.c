/*
 * oracle.c -- plain fp64 CPU restatement of jagged attention, forward and
 * backward.  TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check
 * and the benchmark's CPU-baseline leg call it; the CUDA library never does.
 * It shares no code, header or constant with the CUDA path.
 *
 * What it computes (the jagged FlashAttention pages describe FlashAttention
 * computed straight from the packed, unpadded tensors and their offsets: the
 * PyTorch-blog summary on arc-codex, first key point, and the asivanadi0
 * blog, section "What it is selling").  For each sequence b and
 * head h, with Q_b the query rows of b (broadcast mode: every row of the one
 * dense Q) and K_b, V_b the packed key/value rows of b:
 *
 *   S      = scale * Q_b K_b^T
 *   LSE_i  = max_j S_ij + ln sum_j exp(S_ij - max_j S_ij)      (natural log)
 *   P      = exp(S - LSE)                                      (row softmax)
 *   O_b    = P V_b
 *
 * and, given dO_b, the textbook gradients of that definition (the pages print
 * none; the row sum Delta is the "Di" preprocessing named on the TLX Block
 * Attention page, "One Constraint, Five Eliminations"):
 *
 *   Delta_i = sum_d dO_id O_id
 *   dV_b    = P^T dO_b
 *   dP      = dO_b V_b^T
 *   dS      = P o (dP - Delta)
 *   dQ_b    = scale * dS K_b
 *   dK_b    = scale * dS^T Q_b
 *
 * Broadcast mode (one dense Q shared by every sequence; the alphasignal page,
 * "GEM's sequences do not fit a fixed grid"): O, dO and LSE hold B*Lq rows,
 * b-major, and dQ = sum_b dQ_b.
 *
 * Conventions where the pages are silent: LSE is natural-log and includes
 * scale; a sequence with no keys gives O = 0 and LSE = -inf and contributes
 * nothing to any gradient; a sequence with no queries writes nothing.
 *
 * Layouts: packed tensors are [rows, H, D] row-major; LSE is [H, rows];
 * offsets are int64 [B+1].  Inputs are doubles (exact copies of the bf16
 * values); every product and sum is in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- one query row ------------------------------------------------------ */

/* Forward for one query row qi against nk keys: fills p[nk] with the softmax
 * row, o[D] with the output row and returns LSE.  With nk == 0 the row is
 * O = 0, LSE = -inf. */
static double row_forward(const double* qi, const double* k, const double* v,
                          int64_t ldk, int64_t nk, int D, double scale,
                          double* p, double* o)
{
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (nk == 0) return -INFINITY;
    double mx = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) {
        const double* kj = k + j * ldk;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qi[d] * kj[d];
        p[j] = scale * dot;                 /* S_ij for now */
        if (p[j] > mx) mx = p[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < nk; ++j) sum += exp(p[j] - mx);
    const double lse = mx + log(sum);
    for (int64_t j = 0; j < nk; ++j) {
        p[j] = exp(p[j] - lse);             /* P_ij */
        const double* vj = v + j * ldk;
        for (int d = 0; d < D; ++d) o[d] += p[j] * vj[d];
    }
    return lse;
}

/* dS row for one query row, given its softmax row p, output row o and the
 * incoming gradient row doi: dS_ij = P_ij (dP_ij - Delta_i). */
static void row_dS(const double* p, const double* o, const double* doi,
                   const double* v, int64_t ldk, int64_t nk, int D, double* ds)
{
    double delta = 0.0;
    for (int d = 0; d < D; ++d) delta += doi[d] * o[d];
    for (int64_t j = 0; j < nk; ++j) {
        const double* vj = v + j * ldk;
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += doi[d] * vj[d];
        ds[j] = p[j] * (dp - delta);
    }
}

/* ---- one (sequence, head) ---------------------------------------------- */

/* Forward of one (sequence, head).  q: nq rows with stride ldq; k, v: nk rows
 * with stride ldk; o: nq rows with stride ldo; lse: nq values with stride
 * lse_stride. */
void oracle_seq_fwd(const double* q, int64_t ldq, int64_t nq,
                    const double* k, const double* v, int64_t ldk, int64_t nk,
                    int D, double scale,
                    double* o, int64_t ldo, double* lse, int64_t lse_stride)
{
    double* p = (double*)malloc((size_t)(nk > 0 ? nk : 1) * sizeof(double));
    for (int64_t i = 0; i < nq; ++i)
        lse[i * lse_stride] = row_forward(q + i * ldq, k, v, ldk, nk, D, scale, p, o + i * ldo);
    free(p);
}

/* Backward of one (sequence, head): recomputes P and O from the definition,
 * then writes dK, dV (nk rows, stride lddk) and adds dQ_b into dq (nq rows,
 * stride lddq) -- callers zero dq first. */
void oracle_seq_bwd(const double* q, int64_t ldq, int64_t nq,
                    const double* k, const double* v, int64_t ldk, int64_t nk,
                    const double* dout, int64_t lddo, int D, double scale,
                    double* dq, int64_t lddq, double* dk, double* dv, int64_t lddk)
{
    for (int64_t j = 0; j < nk; ++j)
        for (int d = 0; d < D; ++d) { dk[j * lddk + d] = 0.0; dv[j * lddk + d] = 0.0; }
    if (nq == 0 || nk == 0) return;
    double* P = (double*)malloc((size_t)(nq * nk) * sizeof(double));
    double* dS = (double*)malloc((size_t)(nq * nk) * sizeof(double));
    double* o = (double*)malloc((size_t)D * sizeof(double));
    for (int64_t i = 0; i < nq; ++i) {
        (void)row_forward(q + i * ldq, k, v, ldk, nk, D, scale, P + i * nk, o);
        row_dS(P + i * nk, o, dout + i * lddo, v, ldk, nk, D, dS + i * nk);
    }
    for (int64_t j = 0; j < nk; ++j) {
        for (int64_t i = 0; i < nq; ++i) {
            const double pij = P[i * nk + j], sij = dS[i * nk + j];
            const double* doi = dout + i * lddo;
            const double* qi = q + i * ldq;
            for (int d = 0; d < D; ++d) {
                dv[j * lddk + d] += pij * doi[d];           /* dV = P^T dO */
                dk[j * lddk + d] += scale * sij * qi[d];    /* dK = scale dS^T Q */
            }
        }
    }
    for (int64_t i = 0; i < nq; ++i)
        for (int64_t j = 0; j < nk; ++j) {
            const double sij = dS[i * nk + j];
            const double* kj = k + j * ldk;
            for (int d = 0; d < D; ++d) dq[i * lddq + d] += scale * sij * kj[d];  /* dQ = scale dS K */
        }
    free(P); free(dS); free(o);
}

/* ---- whole problem ------------------------------------------------------ */

static int check_offsets(const int64_t* off, int B)
{
    if (off[0] != 0) return -1;
    for (int b = 0; b < B; ++b) if (off[b + 1] < off[b]) return -1;
    return 0;
}

/* Forward over the packed problem.  q_off == NULL selects broadcast mode
 * (q holds Lq rows shared by every sequence).  o: [n_o, H, D], lse: [H, n_o]
 * with n_o = q_off[B] (self) or B*Lq (broadcast). */
int oracle_fwd(const double* q, const double* k, const double* v,
               const int64_t* kv_off, const int64_t* q_off,
               int B, int H, int64_t Lq, int D, double scale,
               double* o, double* lse)
{
    if (check_offsets(kv_off, B) || (q_off && check_offsets(q_off, B))) return -1;
    const int64_t n_o = q_off ? q_off[B] : (int64_t)B * Lq;
    const int64_t ld = (int64_t)H * D;
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            const int64_t q0 = q_off ? q_off[b] : 0;
            const int64_t nq = q_off ? q_off[b + 1] - q_off[b] : Lq;
            const int64_t o0 = q_off ? q_off[b] : (int64_t)b * Lq;
            const int64_t k0 = kv_off[b], nk = kv_off[b + 1] - kv_off[b];
            oracle_seq_fwd(q + q0 * ld + h * D, ld, nq,
                           k + k0 * ld + h * D, v + k0 * ld + h * D, ld, nk, D, scale,
                           o + o0 * ld + h * D, ld, lse + (int64_t)h * n_o + o0, 1);
        }
    return 0;
}

/* Backward over the packed problem.  dq: [Lq, H, D] (broadcast, summed over
 * the batch) or [q_off[B], H, D] (self); dk, dv: [kv_off[B], H, D]. */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
               const int64_t* kv_off, const int64_t* q_off,
               int B, int H, int64_t Lq, int D, double scale,
               double* dq, double* dk, double* dv)
{
    if (check_offsets(kv_off, B) || (q_off && check_offsets(q_off, B))) return -1;
    const int64_t ld = (int64_t)H * D;
    const int64_t n_q = q_off ? q_off[B] : Lq;
    memset(dq, 0, (size_t)(n_q * ld) * sizeof(double));
    #pragma omp parallel
    {
        /* broadcast mode: each thread sums its sequences' dQ_b privately,
         * then the partial sums are added together */
        double* dq_part = q_off ? NULL : (double*)calloc((size_t)(n_q * ld), sizeof(double));
        #pragma omp for collapse(2) schedule(dynamic)
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; ++h) {
                const int64_t q0 = q_off ? q_off[b] : 0;
                const int64_t nq = q_off ? q_off[b + 1] - q_off[b] : Lq;
                const int64_t o0 = q_off ? q_off[b] : (int64_t)b * Lq;
                const int64_t k0 = kv_off[b], nk = kv_off[b + 1] - kv_off[b];
                double* dq_dst = q_off ? dq : dq_part;
                oracle_seq_bwd(q + q0 * ld + h * D, ld, nq,
                               k + k0 * ld + h * D, v + k0 * ld + h * D, ld, nk,
                               dout + o0 * ld + h * D, ld, D, scale,
                               dq_dst + q0 * ld + h * D, ld,
                               dk + k0 * ld + h * D, dv + k0 * ld + h * D, ld);
            }
        if (dq_part) {
            #pragma omp critical
            for (int64_t i = 0; i < n_q * ld; ++i) dq[i] += dq_part[i];
            free(dq_part);
        }
    }
    return 0;
}

/* dQ for a few query rows of one head, straight from the definition: row i
 * of dQ only needs row i of every sequence's S, P, O, dP and dS.  rows: the
 * query-row indices (into Q); out: [nrows, D].  k, v, dout are the full
 * packed tensors.  Lets full-size problems be checked row by row. */
int oracle_dq_rows(const double* q, const double* k, const double* v, const double* dout,
                   const int64_t* kv_off, const int64_t* q_off,
                   int B, int H, int64_t Lq, int D, double scale, int h,
                   const int64_t* rows, int nrows, double* out)
{
    if (check_offsets(kv_off, B) || (q_off && check_offsets(q_off, B))) return -1;
    const int64_t ld = (int64_t)H * D;
    int64_t maxk = 1;
    for (int b = 0; b < B; ++b) if (kv_off[b + 1] - kv_off[b] > maxk) maxk = kv_off[b + 1] - kv_off[b];
    #pragma omp parallel
    {
        double* p = (double*)malloc((size_t)maxk * sizeof(double));
        double* ds = (double*)malloc((size_t)maxk * sizeof(double));
        double* o = (double*)malloc((size_t)D * sizeof(double));
        #pragma omp for schedule(dynamic)
        for (int r = 0; r < nrows; ++r) {
            const int64_t i = rows[r];
            double* dst = out + (int64_t)r * D;
            for (int d = 0; d < D; ++d) dst[d] = 0.0;
            for (int b = 0; b < B; ++b) {
                int64_t orow;
                if (q_off) {                      /* self: row i belongs to one sequence */
                    if (i < q_off[b] || i >= q_off[b + 1]) continue;
                    orow = i;
                } else {
                    orow = (int64_t)b * Lq + i;
                }
                const int64_t k0 = kv_off[b], nk = kv_off[b + 1] - kv_off[b];
                if (nk == 0) continue;
                const double* kb = k + k0 * ld + h * D;
                const double* vb = v + k0 * ld + h * D;
                (void)row_forward(q + i * ld + h * D, kb, vb, ld, nk, D, scale, p, o);
                row_dS(p, o, dout + orow * ld + h * D, vb, ld, nk, D, ds);
                for (int64_t j = 0; j < nk; ++j)
                    for (int d = 0; d < D; ++d) dst[d] += scale * ds[j] * kb[j * ld + d];
            }
        }
        free(p); free(ds); free(o);
    }
    return 0;
}

int oracle_num_threads(void)
{
    int n = 1;
    #pragma omp parallel
    {
        #pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
